// noalloc.cu -- q8act_gemm_q8_0_noalloc: the fused-quantize GEMM for callers that must not
// allocate device memory.
//
// Who needs it: code that runs where cudaMalloc (or any allocator) is off limits -- for
// example a custom allocator's own hooks, a real-time serving loop that forbids allocation
// after start-up, or a runtime that hands kernels only the input and output buffers it
// already owns.  q8act_gemm_q8_0 asks such callers for a workspace they cannot provide.
//
// What it does instead: the quantized activation (binary16 quants + transposed scales, the
// same bytes q8act_gemm_q8_0 writes into its caller's workspace) goes into one fixed device
// array declared in this file.  Every GPU that loads the library reserves the whole array
// (Q8ACT_NOALLOC_WS_BYTES) for the life of the process.  The first call on a device looks up
// the array's device address with cudaGetSymbolAddress while that device is current; later
// calls reuse the cached address for as long as the same CUDA context is current (the
// address belongs to the context: after a cudaDeviceReset, or a primary context released
// and created again, the next call looks it up afresh).  The call itself allocates nothing
// and frees nothing.
//
// Size limit: the quantized activation, q8act_gemm_workspace_bytes(m, k) minus
// Q8ACT_GEMM_SPLIT_BYTES bytes, must fit in the array (k = 4096: m <= 2891); larger calls are
// refused before anything is launched.  When the split region fits in the rest of the array
// as well (m * k up to about 2M at k = 4096), the GEMM may take its balanced schedule, as
// q8act_gemm_q8_0 does with a full workspace; otherwise every tile is done by one CTA.
//
// Sharing rules: every call on a device uses the same array, and the array keeps whatever
// the previous call left in it.  Nothing in it has to start at zero: each call rewrites all
// the quants and scales it reads (the scale columns past m are never read), and the split
// counters are zeroed on the stream before the quantizer runs.  Two calls whose work can
// overlap on the GPU -- on different streams without ordering between them -- race on the
// array and may corrupt each other's results; order them on one stream or with events.
#include <mutex>

#include "common.cuh"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_ws[Q8ACT_NOALLOC_WS_BYTES];

struct NoallocSlot {
    unsigned long long ctx = 0;   // the context the cached address belongs to (0: none)
    void *ptr = nullptr;
};

NoallocSlot g_noalloc_slots[kMaxDevices];
std::mutex g_noalloc_mutex;

}  // namespace

extern "C" int q8act_gemm_q8_0_noalloc(const void *w, const float *x, float *y, int64_t m,
                                       int64_t n, int64_t k, void *stream)
{
    if (!w || !x || !y) return Q8ACT_ERR_NULL;
    const size_t full = q8act_gemm_workspace_bytes(m, k);
    if (full == 0 || n < 1) return Q8ACT_ERR_DIMS;
    // The quantized activation must fit; the split region (balanced schedule) is used only when the
    // rest of the array holds it.
    if (full - Q8ACT_GEMM_SPLIT_BYTES > (size_t)Q8ACT_NOALLOC_WS_BYTES) return Q8ACT_ERR_WORKSPACE;

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return Q8ACT_ERR_CUDA_BASE + (int)e;
    if (dev < 0 || dev >= kMaxDevices) return Q8ACT_ERR_DEVICE;
    void *ws = nullptr;
    {
        const unsigned long long ctx = q8::current_context_id();
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        NoallocSlot &s = g_noalloc_slots[dev];
        if (ctx == 0 || ctx != s.ctx) {
            // Device `dev` is current here, so this is the array's address on that device (in
            // its current context).
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_ws);
            if (e != cudaSuccess) return Q8ACT_ERR_CUDA_BASE + (int)e;
            s.ptr = p;
            s.ctx = ctx;
        }
        ws = s.ptr;
    }
    return q8act_gemm_q8_0(w, x, y, m, n, k, ws, (size_t)Q8ACT_NOALLOC_WS_BYTES, stream);
}
