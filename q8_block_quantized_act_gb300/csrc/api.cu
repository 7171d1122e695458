// api.cu -- the extern "C" boundary of libq8act (declared in include/q8act.h): argument
// checks, per-device setup and dispatch to the kernels.  No call allocates memory or
// synchronizes, except q8act_device_status.
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace {

constexpr int kMaxDevices = 64;

// Device-side status word: kernels OR bits into it when a pipeline wait times out.
__device__ int g_status;

struct DeviceSlot {
    bool ready = false;
    unsigned long long ctx = 0;   // context whose status-word address `info` holds
    int rc = Q8ACT_OK;
    q8::DeviceInfo info{};
};

DeviceSlot g_slots[kMaxDevices];
std::mutex g_mutex;

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? Q8ACT_OK : Q8ACT_ERR_CUDA_BASE + (int)e; }

// Current device's info; checks once per device (and context: the status word's address
// belongs to the context) that it is an sm_103 GPU.
int current_device(const q8::DeviceInfo **out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_rc(e);
    if (dev < 0 || dev >= kMaxDevices) return Q8ACT_ERR_DEVICE;
    const unsigned long long ctx = q8::current_context_id();
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceSlot &s = g_slots[dev];
    if (!s.ready || ctx == 0 || ctx != s.ctx) {
        int major = 0, minor = 0, sms = 0, smem = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
            return cuda_rc(e);
        if (major != 10 || minor != 3) {
            s.rc = Q8ACT_ERR_DEVICE;
        } else {
            void *status = nullptr;
            if ((e = cudaGetSymbolAddress(&status, g_status)) != cudaSuccess) return cuda_rc(e);
            s.info.device = dev;
            s.info.num_sms = sms;
            s.info.max_smem_optin = (size_t)smem;
            s.info.status = static_cast<int *>(status);
            s.rc = Q8ACT_OK;
        }
        s.ctx = ctx;
        s.ready = true;
    }
    *out = &s.info;
    return s.rc;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_k(int64_t k)
{
    return (k > 0 && k % q8::K_ALIGN == 0 && k <= Q8ACT_MAX_K) ? Q8ACT_OK : Q8ACT_ERR_DIMS;
}

// Largest m * k the GEMM accepts (keeps every element index inside 32 bits).
constexpr int64_t kMaxGemmElems = (int64_t)1 << 30;

int check_gemm_dims(int64_t m, int64_t n, int64_t k)
{
    if (check_k(k) != Q8ACT_OK || m < 1 || n < 1) return Q8ACT_ERR_DIMS;
    if (m * k > kMaxGemmElems || n * k > ((int64_t)1 << 34) || m * n > ((int64_t)1 << 31))
        return Q8ACT_ERR_DIMS;
    if (n > INT32_MAX || m > INT32_MAX) return Q8ACT_ERR_DIMS;
    return Q8ACT_OK;
}

}  // namespace

extern "C" {

int q8act_version(void) { return 100; }

const char *q8act_strerror(int rc)
{
    switch (rc) {
    case Q8ACT_OK: return "ok";
    case Q8ACT_ERR_NULL: return "a required pointer is NULL";
    case Q8ACT_ERR_DIMS: return "dimensions out of range (k must be a positive multiple of 256)";
    case Q8ACT_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case Q8ACT_ERR_WORKSPACE: return "workspace missing or too small";
    case Q8ACT_ERR_DEVICE: return "the current device is not an sm_103 (GB300) GPU";
    case Q8ACT_ERR_TIMEOUT: return "a kernel timed out waiting in its pipeline";
    case Q8ACT_ERR_DRAIN_TIMEOUT: return "a kernel timed out waiting for its own copies before exit";
    default:
        if (rc >= Q8ACT_ERR_CUDA_BASE) return cudaGetErrorString((cudaError_t)(rc - Q8ACT_ERR_CUDA_BASE));
        return "unknown error";
    }
}

int64_t q8act_mmq_ldm(int64_t m) { return m < 1 ? 0 : (m + 3) / 4 * 4; }

int q8act_quantize_q8_1(const float *x, int8_t *xq, float *xd, int64_t m, int64_t k, void *stream)
{
    if (!x || !xq || !xd) return Q8ACT_ERR_NULL;
    if (check_k(k) != Q8ACT_OK || m < 1 || m * k > ((int64_t)1 << 34)) return Q8ACT_ERR_DIMS;
    if (!aligned16(x) || !aligned16(xq) || !aligned16(xd)) return Q8ACT_ERR_ALIGN;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    return cuda_rc(q8::launch_quantize_q8_1(*dev, x, xq, xd, m, k, (cudaStream_t)stream));
}

int q8act_quantize_q8_1_mmq(const float *x, uint16_t *xqh, float *xdt, int64_t m, int64_t k, void *stream)
{
    if (!x || !xqh || !xdt) return Q8ACT_ERR_NULL;
    if (check_k(k) != Q8ACT_OK || m < 1 || m * k > kMaxGemmElems) return Q8ACT_ERR_DIMS;
    if (!aligned16(x) || !aligned16(xqh) || !aligned16(xdt)) return Q8ACT_ERR_ALIGN;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    return cuda_rc(q8::launch_quantize_q8_1_mmq(*dev, x, xqh, xdt, m, k, q8act_mmq_ldm(m), (cudaStream_t)stream));
}

int q8act_quantize_q8_0(const float *w, void *wq, int64_t n, int64_t k, void *stream)
{
    if (!w || !wq) return Q8ACT_ERR_NULL;
    if (check_k(k) != Q8ACT_OK || n < 1 || n * k > ((int64_t)1 << 34)) return Q8ACT_ERR_DIMS;
    if (!aligned16(w) || !aligned16(wq)) return Q8ACT_ERR_ALIGN;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    return cuda_rc(q8::launch_quantize_q8_0(*dev, w, static_cast<uint8_t *>(wq), n, k, (cudaStream_t)stream));
}

int q8act_dequant_q8_0_f16(const void *w, void *w16, int64_t n, int64_t k, void *stream)
{
    if (!w || !w16) return Q8ACT_ERR_NULL;
    if (check_k(k) != Q8ACT_OK || n < 1 || n * k > ((int64_t)1 << 34)) return Q8ACT_ERR_DIMS;
    if (!aligned16(w) || !aligned16(w16)) return Q8ACT_ERR_ALIGN;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    return cuda_rc(q8::launch_dequant_q8_0_f16(*dev, static_cast<const uint8_t *>(w), static_cast<uint16_t *>(w16), n, k,
                                               (cudaStream_t)stream));
}

int64_t q8act_repack_ldn(int64_t n) { return n < 1 ? 0 : (n + 3) / 4 * 4; }

int q8act_repack_q8_0(const void *w, uint16_t *wq16, float *wdt, int64_t n, int64_t k, void *stream)
{
    if (!w || !wq16 || !wdt) return Q8ACT_ERR_NULL;
    if (check_k(k) != Q8ACT_OK || n < 1 || n * k > ((int64_t)1 << 34)) return Q8ACT_ERR_DIMS;
    if (!aligned16(w) || !aligned16(wq16) || !aligned16(wdt)) return Q8ACT_ERR_ALIGN;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    return cuda_rc(q8::launch_repack_q8_0(*dev, static_cast<const uint8_t *>(w), wq16, wdt, q8act_repack_ldn(n),
                                          n, k, (cudaStream_t)stream));
}

// pdl: the stream's previous operation is the q8_1 quantizer of the same call; the GEMV is
// then launched as its programmatic dependent.
static int gemv_common(const void *w, const int8_t *xq, const float *xd, float *y, int32_t *dots, int64_t m,
                       int64_t n, int64_t k, void *stream, bool pdl = false)
{
    if (!w || !xq || !xd || (!y && !dots)) return Q8ACT_ERR_NULL;
    if (check_k(k) != Q8ACT_OK || m < 1 || m > Q8ACT_GEMV_MAX_M || n < 1 || n > INT32_MAX / 2 ||
        n * k > ((int64_t)1 << 36))
        return Q8ACT_ERR_DIMS;
    if (!aligned16(w) || !aligned16(xq) || !aligned16(xd) || (y && !aligned16(y)) || (dots && !aligned16(dots)))
        return Q8ACT_ERR_ALIGN;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    if (q8::gemv_mma_supported(*dev, m, k))
        return cuda_rc(q8::launch_gemv_q8_0_mma(*dev, static_cast<const uint8_t *>(w), xq, xd, y, dots, m, n, k,
                                                (cudaStream_t)stream, pdl));
    if (!q8::gemv_supported(*dev, m, k)) return Q8ACT_ERR_DIMS;
    return cuda_rc(q8::launch_gemv_q8_0(*dev, static_cast<const uint8_t *>(w), xq, xd, y, dots, m, n, k,
                                        (cudaStream_t)stream, pdl));
}

int q8act_gemv_q8_0(const void *w, const int8_t *xq, const float *xd, float *y, int64_t m, int64_t n, int64_t k,
                    void *stream)
{
    if (!y) return Q8ACT_ERR_NULL;
    return gemv_common(w, xq, xd, y, nullptr, m, n, k, stream);
}

// Workspace of the fused GEMV: [int8 quants, m * k][f32 scales, m * k / 32], each part
// rounded up to 256 bytes.
size_t q8act_gemv_workspace_bytes(int64_t m, int64_t k)
{
    if (check_k(k) != Q8ACT_OK || m < 1 || m > Q8ACT_GEMV_MAX_M) return 0;
    const size_t quants = (size_t)m * (size_t)k;
    const size_t scales = (size_t)m * (size_t)(k / q8::QK) * 4;
    return ((quants + 255) / 256 * 256) + ((scales + 255) / 256 * 256);
}

int q8act_gemv_q8_0_f32(const void *w, const float *x, float *y, int64_t m, int64_t n, int64_t k, void *ws,
                        size_t ws_bytes, void *stream)
{
    if (!w || !x || !y) return Q8ACT_ERR_NULL;
    if (check_k(k) != Q8ACT_OK || m < 1 || m > Q8ACT_GEMV_MAX_M || n < 1 || n > INT32_MAX / 2 ||
        n * k > ((int64_t)1 << 36))
        return Q8ACT_ERR_DIMS;
    const size_t need = q8act_gemv_workspace_bytes(m, k);
    if (!ws || ws_bytes < need) return Q8ACT_ERR_WORKSPACE;
    if (!aligned16(w) || !aligned16(x) || !aligned16(y) || !aligned16(ws)) return Q8ACT_ERR_ALIGN;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    if (!q8::gemv_mma_supported(*dev, m, k) && !q8::gemv_supported(*dev, m, k)) return Q8ACT_ERR_DIMS;
    int8_t *xq = static_cast<int8_t *>(ws);
    float *xd = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + ((size_t)m * k + 255) / 256 * 256);
    rc = q8act_quantize_q8_1(x, xq, xd, m, k, stream);
    if (rc) return rc;
    return gemv_common(w, xq, xd, y, nullptr, m, n, k, stream, true);
}

int q8act_gemv_q8_0_group(const void *const *w, float *const *y, const int64_t *n, int count, const int8_t *xq,
                          const float *xd, int64_t m, int64_t k, void *stream)
{
    if (!w || !y || !n || !xq || !xd) return Q8ACT_ERR_NULL;
    if (count < 1 || count > Q8ACT_GEMV_MAX_GROUP) return Q8ACT_ERR_DIMS;
    if (check_k(k) != Q8ACT_OK || m < 1 || m > Q8ACT_GEMV_MAX_M) return Q8ACT_ERR_DIMS;
    for (int i = 0; i < count; ++i) {
        if (!w[i] || !y[i]) return Q8ACT_ERR_NULL;
        if (n[i] < 1 || n[i] > INT32_MAX / 2 || n[i] * k > ((int64_t)1 << 36)) return Q8ACT_ERR_DIMS;
        if (!aligned16(w[i]) || !aligned16(y[i])) return Q8ACT_ERR_ALIGN;
    }
    if (!aligned16(xq) || !aligned16(xd)) return Q8ACT_ERR_ALIGN;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    if (q8::gemv_mma_supported(*dev, m, k))
        return cuda_rc(q8::launch_gemv_q8_0_group_mma(*dev, reinterpret_cast<const uint8_t *const *>(w), y, n, count,
                                                      xq, xd, m, k, (cudaStream_t)stream));
    if (!q8::gemv_supported(*dev, m, k)) return Q8ACT_ERR_DIMS;
    return cuda_rc(q8::launch_gemv_q8_0_group(*dev, reinterpret_cast<const uint8_t *const *>(w), y, n, count, xq, xd,
                                              m, k, (cudaStream_t)stream));
}

int q8act_debug_gemv_block_dots(const void *w, const int8_t *xq, int32_t *D, int64_t m, int64_t n, int64_t k,
                                void *stream)
{
    if (!D) return Q8ACT_ERR_NULL;
    // The dot stage needs valid (unused) scales: pass the quants pointer, which is readable.
    return gemv_common(w, xq, reinterpret_cast<const float *>(xq), nullptr, D, m, n, k, stream);
}

// ---- Q4_0 (GGUF 18-byte blocks) ----

int q8act_quantize_q4_0(const float *w, void *wq, int64_t n, int64_t k, void *stream)
{
    if (!w || !wq) return Q8ACT_ERR_NULL;
    if (check_k(k) != Q8ACT_OK || n < 1 || n * k > ((int64_t)1 << 34)) return Q8ACT_ERR_DIMS;
    if (!aligned16(w) || !aligned16(wq)) return Q8ACT_ERR_ALIGN;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    return cuda_rc(q8::launch_quantize_q4_0(*dev, w, static_cast<uint8_t *>(wq), n, k, (cudaStream_t)stream));
}

int q8act_dequant_q4_0_f16(const void *w, void *w16, int64_t n, int64_t k, void *stream)
{
    if (!w || !w16) return Q8ACT_ERR_NULL;
    if (check_k(k) != Q8ACT_OK || n < 1 || n * k > ((int64_t)1 << 34)) return Q8ACT_ERR_DIMS;
    if (!aligned16(w) || !aligned16(w16)) return Q8ACT_ERR_ALIGN;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    return cuda_rc(q8::launch_dequant_q4_0_f16(*dev, static_cast<const uint8_t *>(w), static_cast<uint16_t *>(w16), n, k,
                                               (cudaStream_t)stream));
}

static int gemv_q4_0_common(const void *w, const int8_t *xq, const float *xd, float *y, int32_t *dots, int64_t m,
                            int64_t n, int64_t k, void *stream)
{
    if (!w || !xq || !xd || (!y && !dots)) return Q8ACT_ERR_NULL;
    if (check_k(k) != Q8ACT_OK || m < 1 || m > Q8ACT_GEMV_MAX_M || n < 1 || n > INT32_MAX / 2 ||
        n * k > ((int64_t)1 << 36))
        return Q8ACT_ERR_DIMS;
    if (!aligned16(w) || !aligned16(xq) || !aligned16(xd) || (y && !aligned16(y)) || (dots && !aligned16(dots)))
        return Q8ACT_ERR_ALIGN;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    if (q8::gemv_q4_0_mma_supported(*dev, m, k))
        return cuda_rc(q8::launch_gemv_q4_0_mma(*dev, static_cast<const uint8_t *>(w), xq, xd, y, dots, m, n, k,
                                                (cudaStream_t)stream));
    if (!q8::gemv_q4_0_supported(*dev, m, k)) return Q8ACT_ERR_DIMS;
    return cuda_rc(q8::launch_gemv_q4_0(*dev, static_cast<const uint8_t *>(w), xq, xd, y, dots, m, n, k,
                                        (cudaStream_t)stream));
}

int q8act_gemv_q4_0(const void *w, const int8_t *xq, const float *xd, float *y, int64_t m, int64_t n, int64_t k,
                    void *stream)
{
    if (!y) return Q8ACT_ERR_NULL;
    return gemv_q4_0_common(w, xq, xd, y, nullptr, m, n, k, stream);
}

int q8act_debug_gemv_q4_0_block_dots(const void *w, const int8_t *xq, int32_t *D, int64_t m, int64_t n, int64_t k,
                                     void *stream)
{
    if (!D) return Q8ACT_ERR_NULL;
    // As for Q8_0: the dot stage reads (and ignores) a scale array; the quants are readable.
    return gemv_q4_0_common(w, xq, reinterpret_cast<const float *>(xq), nullptr, D, m, n, k, stream);
}

// ---- K-quant superblocks (GGUF Q6_K 210 B, Q4_K 144 B, Q5_K 176 B; 256 weights each) ----

static int dequant_kq_common(int fmt, const void *w, void *w16, int64_t n, int64_t k, void *stream)
{
    if (!w || !w16) return Q8ACT_ERR_NULL;
    if (check_k(k) != Q8ACT_OK || n < 1 || n > INT32_MAX || n * k > ((int64_t)1 << 34)) return Q8ACT_ERR_DIMS;
    if (!aligned16(w) || !aligned16(w16)) return Q8ACT_ERR_ALIGN;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    return cuda_rc(q8::launch_dequant_kq_f16(*dev, fmt, static_cast<const uint8_t *>(w), static_cast<uint16_t *>(w16),
                                             n, k, (cudaStream_t)stream));
}

int q8act_dequant_q6_k_f16(const void *w, void *w16, int64_t n, int64_t k, void *stream)
{
    return dequant_kq_common(6, w, w16, n, k, stream);
}
int q8act_dequant_q4_k_f16(const void *w, void *w16, int64_t n, int64_t k, void *stream)
{
    return dequant_kq_common(4, w, w16, n, k, stream);
}
int q8act_dequant_q5_k_f16(const void *w, void *w16, int64_t n, int64_t k, void *stream)
{
    return dequant_kq_common(5, w, w16, n, k, stream);
}

static int gemv_kq_common(int fmt, const void *w, const int8_t *xq, const float *xd, float *y, int32_t *dots,
                          int64_t m, int64_t n, int64_t k, void *stream)
{
    if (!w || !xq || !xd || (!y && !dots)) return Q8ACT_ERR_NULL;
    if (check_k(k) != Q8ACT_OK || m < 1 || m > Q8ACT_GEMV_KQ_MAX_M || n < 1 || n > INT32_MAX / 2 ||
        n * k > ((int64_t)1 << 36))
        return Q8ACT_ERR_DIMS;
    if (!aligned16(w) || !aligned16(xq) || !aligned16(xd) || (y && !aligned16(y)) || (dots && !aligned16(dots)))
        return Q8ACT_ERR_ALIGN;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    if (!q8::gemv_kq_supported(*dev, fmt, m, k)) return Q8ACT_ERR_DIMS;
    return cuda_rc(q8::launch_gemv_kq(*dev, fmt, static_cast<const uint8_t *>(w), xq, xd, y, dots, m, n, k,
                                      (cudaStream_t)stream));
}

int q8act_gemv_q6_k(const void *w, const int8_t *xq, const float *xd, float *y, int64_t m, int64_t n, int64_t k,
                    void *stream)
{
    if (!y) return Q8ACT_ERR_NULL;
    return gemv_kq_common(6, w, xq, xd, y, nullptr, m, n, k, stream);
}
int q8act_gemv_q4_k(const void *w, const int8_t *xq, const float *xd, float *y, int64_t m, int64_t n, int64_t k,
                    void *stream)
{
    if (!y) return Q8ACT_ERR_NULL;
    return gemv_kq_common(4, w, xq, xd, y, nullptr, m, n, k, stream);
}
int q8act_gemv_q5_k(const void *w, const int8_t *xq, const float *xd, float *y, int64_t m, int64_t n, int64_t k,
                    void *stream)
{
    if (!y) return Q8ACT_ERR_NULL;
    return gemv_kq_common(5, w, xq, xd, y, nullptr, m, n, k, stream);
}

// The block-integer stage needs a readable scale array; the quants are readable and larger.
int q8act_debug_gemv_q6_k_block_dots(const void *w, const int8_t *xq, int32_t *D, int64_t m, int64_t n, int64_t k,
                                     void *stream)
{
    if (!D) return Q8ACT_ERR_NULL;
    return gemv_kq_common(6, w, xq, reinterpret_cast<const float *>(xq), nullptr, D, m, n, k, stream);
}
int q8act_debug_gemv_q4_k_block_dots(const void *w, const int8_t *xq, int32_t *D, int64_t m, int64_t n, int64_t k,
                                     void *stream)
{
    if (!D) return Q8ACT_ERR_NULL;
    return gemv_kq_common(4, w, xq, reinterpret_cast<const float *>(xq), nullptr, D, m, n, k, stream);
}
int q8act_debug_gemv_q5_k_block_dots(const void *w, const int8_t *xq, int32_t *D, int64_t m, int64_t n, int64_t k,
                                     void *stream)
{
    if (!D) return Q8ACT_ERR_NULL;
    return gemv_kq_common(5, w, xq, reinterpret_cast<const float *>(xq), nullptr, D, m, n, k, stream);
}

// Workspace of the fused GEMMs: [binary16 quants][block-major scales][split region].  The
// first two are required; with the split region as well, a launch may take the balanced
// schedule (equal runs of (tile, k group) units per CTA, tiles cut into k pieces at the runs'
// ends).
static size_t act_bytes(int64_t m, int64_t k)
{
    const size_t quants = (size_t)m * (size_t)k * 2;
    const size_t scales = (size_t)(k / q8::QK) * (size_t)q8act_mmq_ldm(m) * 4;
    return ((quants + 255) / 256 * 256) + ((scales + 255) / 256 * 256);
}

size_t q8act_gemm_workspace_bytes(int64_t m, int64_t k)
{
    if (check_k(k) != Q8ACT_OK || m < 1 || m * k > kMaxGemmElems) return 0;
    return act_bytes(m, k) + Q8ACT_GEMM_SPLIT_BYTES;
}

// pdl: the stream's previous operation is the MMQ quantizer of the same call, enqueued after
// q8::gemm_prepare_split; the GEMM is then launched as its programmatic dependent.
static int gemm_core(const void *w, const uint16_t *xqh, const float *xdt, float *y, int32_t *dots, int64_t m,
                     int64_t n, int64_t k, void *split_ws, size_t split_bytes, bool pdl, void *stream)
{
    if (!w || !xqh || !xdt || (!y && !dots)) return Q8ACT_ERR_NULL;
    if (check_gemm_dims(m, n, k) != Q8ACT_OK) return Q8ACT_ERR_DIMS;
    if (!aligned16(w) || !aligned16(xqh) || !aligned16(xdt) || (y && !aligned16(y)) || (dots && !aligned16(dots)))
        return Q8ACT_ERR_ALIGN;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    return cuda_rc(q8::launch_gemm_q8_0(*dev, static_cast<const uint8_t *>(w), xqh, xdt, y, dots, m, n, k,
                                        q8act_mmq_ldm(m), split_ws, split_bytes, pdl, (cudaStream_t)stream));
}

int q8act_gemm_q8_0(const void *w, const float *x, float *y, int64_t m, int64_t n, int64_t k, void *ws,
                    size_t ws_bytes, void *stream)
{
    if (!w || !x || !y) return Q8ACT_ERR_NULL;
    if (check_gemm_dims(m, n, k) != Q8ACT_OK) return Q8ACT_ERR_DIMS;
    const size_t need = act_bytes(m, k);
    if (!ws || ws_bytes < need) return Q8ACT_ERR_WORKSPACE;
    if (!aligned16(w) || !aligned16(x) || !aligned16(y) || !aligned16(ws)) return Q8ACT_ERR_ALIGN;
    uint16_t *xqh = static_cast<uint16_t *>(ws);
    float *xdt = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + ((size_t)m * k * 2 + 255) / 256 * 256);
    void *split_ws = static_cast<uint8_t *>(ws) + need;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    rc = cuda_rc(q8::gemm_prepare_split(*dev, m, n, k, false, split_ws, ws_bytes - need, (cudaStream_t)stream));
    if (rc) return rc;
    rc = q8act_quantize_q8_1_mmq(x, xqh, xdt, m, k, stream);
    if (rc) return rc;
    return gemm_core(w, xqh, xdt, y, nullptr, m, n, k, split_ws, ws_bytes - need, true, stream);
}

int q8act_gemm_q8_0_preq(const void *w, const uint16_t *xqh, const float *xdt, float *y, int64_t m, int64_t n,
                         int64_t k, void *stream)
{
    if (!y) return Q8ACT_ERR_NULL;
    return gemm_core(w, xqh, xdt, y, nullptr, m, n, k, nullptr, 0, false, stream);
}

static int gemm_repacked_core(const uint16_t *wq16, const float *wdt, const uint16_t *xqh, const float *xdt,
                              float *y, int32_t *dots, int64_t m, int64_t n, int64_t k, void *split_ws,
                              size_t split_bytes, bool pdl, void *stream)
{
    if (!wq16 || !wdt || !xqh || !xdt || (!y && !dots)) return Q8ACT_ERR_NULL;
    if (check_gemm_dims(m, n, k) != Q8ACT_OK) return Q8ACT_ERR_DIMS;
    if (!aligned16(wq16) || !aligned16(wdt) || !aligned16(xqh) || !aligned16(xdt) || (y && !aligned16(y)) ||
        (dots && !aligned16(dots)))
        return Q8ACT_ERR_ALIGN;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    return cuda_rc(q8::launch_gemm_q8_0_repacked(*dev, wq16, wdt, q8act_repack_ldn(n), xqh, xdt, y, dots, m, n, k,
                                                 q8act_mmq_ldm(m), split_ws, split_bytes, pdl, (cudaStream_t)stream));
}

int q8act_gemm_q8_0_repacked(const uint16_t *wq16, const float *wdt, const float *x, float *y, int64_t m,
                             int64_t n, int64_t k, void *ws, size_t ws_bytes, void *stream)
{
    if (!wq16 || !wdt || !x || !y) return Q8ACT_ERR_NULL;
    if (check_gemm_dims(m, n, k) != Q8ACT_OK) return Q8ACT_ERR_DIMS;
    const size_t need = act_bytes(m, k);
    if (!ws || ws_bytes < need) return Q8ACT_ERR_WORKSPACE;
    if (!aligned16(wq16) || !aligned16(wdt) || !aligned16(x) || !aligned16(y) || !aligned16(ws))
        return Q8ACT_ERR_ALIGN;
    uint16_t *xqh = static_cast<uint16_t *>(ws);
    float *xdt = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + ((size_t)m * k * 2 + 255) / 256 * 256);
    void *split_ws = static_cast<uint8_t *>(ws) + need;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    rc = cuda_rc(q8::gemm_prepare_split(*dev, m, n, k, true, split_ws, ws_bytes - need, (cudaStream_t)stream));
    if (rc) return rc;
    rc = q8act_quantize_q8_1_mmq(x, xqh, xdt, m, k, stream);
    if (rc) return rc;
    return gemm_repacked_core(wq16, wdt, xqh, xdt, y, nullptr, m, n, k, split_ws, ws_bytes - need, true, stream);
}

int q8act_debug_gemm_repacked_block_dots(const uint16_t *wq16, const float *wdt, const uint16_t *xqh, int32_t *D,
                                         int64_t m, int64_t n, int64_t k, void *stream)
{
    if (!D) return Q8ACT_ERR_NULL;
    // The dot stage needs a readable (unused) activation-scale array: reuse the quants.
    return gemm_repacked_core(wq16, wdt, xqh, reinterpret_cast<const float *>(xqh), nullptr, D, m, n, k, nullptr, 0,
                              false, stream);
}

int q8act_debug_gemm_block_dots(const void *w, const uint16_t *xqh, int32_t *D, int64_t m, int64_t n, int64_t k,
                                void *stream)
{
    if (!D) return Q8ACT_ERR_NULL;
    // The dot stage needs a readable (unused) scale array of the right shape: reuse the
    // quants, which are larger than the scale array.
    return gemm_core(w, xqh, reinterpret_cast<const float *>(xqh), nullptr, D, m, n, k, nullptr, 0, false, stream);
}

// Test hook: one thread waits on an mbarrier that nothing arrives on, through the pipelines'
// own bounded wait, until limit_ns passes; the wait then records STATUS_TIMEOUT.  Nothing
// else is in flight (no copies, no tensor-core work), so the exit is clean.
__global__ void wait_timeout_kernel(unsigned long long limit_ns, int *status)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        q8::mbar_init(&bar, 1);
        q8::fence_mbar_init();
        q8::mbar_wait_for(&bar, 0, status, limit_ns, q8::STATUS_TIMEOUT);
        asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(q8::smem_u32(&bar)) : "memory");
    }
}

int q8act_debug_wait_timeout(int64_t limit_ns, void *stream)
{
    if (limit_ns < 1000 || limit_ns > 1000000000) return Q8ACT_ERR_DIMS;
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((unsigned long long)limit_ns, dev->status);
    return cuda_rc(cudaGetLastError());
}

int q8act_device_status(void *stream)
{
    const q8::DeviceInfo *dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_rc(e);
    int host = 0;
    const int zero = 0;
    if ((e = cudaMemcpyFromSymbol(&host, g_status, sizeof(int))) != cudaSuccess) return cuda_rc(e);
    if (host && (e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int))) != cudaSuccess) return cuda_rc(e);
    if (host & q8::STATUS_DRAIN_TIMEOUT) return Q8ACT_ERR_DRAIN_TIMEOUT;
    return host ? Q8ACT_ERR_TIMEOUT : Q8ACT_OK;
}

}  // extern "C"
