// kquant.cu -- two passes over the GGUF K-quant superblocks (layouts in kquant.cuh):
//   * the fp16 mirror (memra-engine 0.81.0 f16_ffi.rs memra_q6_K / q4_K / q5_K_dequant_f16):
//     every weight's exact value, rounded once to binary16;
//   * the decode GEMV with the q8_1 activation (1 <= m <= 8), exact integer dots per 32-wide
//     activation block and an f32 fold (from m = 2 the tensor-core kernel of gemv_kq_mma.cu
//     takes over where the row layout allows it, with the same bits).
// Both passes stream chunks of whole rows into a shared-memory ring with cp.async.bulk, as
// the Q8_0 kernels do.  Q6_K rows are a 16-byte multiple only when k is a multiple of 2048,
// so a chunk holds a multiple of 8 rows (8 rows always are) and the last chunk's final
// 0..14 bytes are copied by the producer thread itself.
#include "common.cuh"
#include "kquant.cuh"
#include "launch.h"

namespace q8 {
namespace {

constexpr int KMAX_STAGES = 6;

__host__ __device__ constexpr int gcd_int(int a, int b) { return b == 0 ? a : gcd_int(b, a % b); }

// Rows per chunk must make every chunk start (and every stage) 16-byte aligned.
inline int row_align(uint32_t row_bytes) { return 16 / gcd_int((int)(row_bytes % 16 == 0 ? 16 : row_bytes % 16), 16); }

// The superblock at p (2-byte aligned for Q6_K, 16-byte aligned otherwise) as 32-bit words
// of its bytes, read from shared memory.
template <class F>
__device__ __forceinline__ void load_superblock(const uint8_t *p, uint32_t (&w)[F::WORDS])
{
    if constexpr (F::BYTES % 16 == 0) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p);
#pragma unroll
        for (int c = 0; c < F::WORDS / 4; ++c) {
            const uint4 v = src[c];
            w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
        }
    } else {
        // Aligned words from the word below p, funnel-shifted by the 0 or 2 bytes of offset.
        const uintptr_t a = reinterpret_cast<uintptr_t>(p);
        const uint32_t *base = reinterpret_cast<const uint32_t *>(a & ~(uintptr_t)3);
        const uint32_t sh = (uint32_t)(a & 3) * 8;
        uint32_t prev = base[0];
#pragma unroll
        for (int i = 0; i < F::WORDS; ++i) {
            const uint32_t nxt = base[i + 1];
            w[i] = __funnelshift_r(prev, nxt, sh);
            prev = nxt;
        }
    }
}

// Unsigned bytes of a times signed bytes of b, summed into c.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// The codes of 32-wide block j of a superblock, as 8 words of 4 bytes each (element order),
// ready for dp4a: Q6_K gives the signed bytes code - 32 (or, with Q6_UNSIGNED, the codes
// 0..63 themselves); Q4_K / Q5_K the unsigned codes.
template <class F, bool Q6_UNSIGNED = false>
__device__ __forceinline__ void block_codes(const uint32_t (&w)[F::WORDS], int j, uint32_t (&q)[8])
{
    if constexpr (F::BYTES == KQ6::BYTES) {
        const int n = j >> 2, g = j & 3;
        const int qlw = 16 * n + 8 * (g & 1), qhw = 32 + 8 * n;
        const int s1 = 4 * (g >> 1), s2 = 2 * g;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint32_t code = ((w[qlw + c] >> s1) & 0x0F0F0F0Fu) | (((w[qhw + c] >> s2) & 0x03030303u) << 4);
            q[c] = Q6_UNSIGNED ? code : q6_signed_bytes(code);
        }
    } else {
        const int g = j >> 1, u = j & 1;
        constexpr int QS = F::BYTES == KQ4::BYTES ? 4 : 12;   // word of qs[0]
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint32_t code = (w[QS + 8 * g + c] >> (4 * u)) & 0x0F0F0F0Fu;
            if constexpr (F::BYTES == KQ5::BYTES) code |= ((w[4 + c] >> j) & 0x01010101u) << 4;
            q[c] = code;
        }
    }
}

// ---------------------------------------------------------------------------------------
// Streaming plan and producer shared by both passes
// ---------------------------------------------------------------------------------------
struct KPlan {
    int G;              // superblocks per row (k / 256)
    int R;              // rows per chunk (a multiple of the row alignment)
    int U;              // units (superblocks) per chunk
    int stages;
    int ctas_per_sm;
    int warp_reduce;    // 1: a row's units are consecutive lanes of one warp (G divides 32)
    uint32_t row_bytes;
    uint32_t chunk_bytes;
    int64_t nchunks;
    size_t off_x, off_xd, off_xs, off_part, off_bar, smem;
};

// Copy rows [row0, row0 + rows) of w into dst, completing on `bar`: a bulk copy of the
// 16-byte multiple, then (for the last, ragged chunk of a Q6_K matrix) the few bytes after it
// with plain stores, made before the arrival so that they are visible with the copy.
__device__ __forceinline__ void produce_chunk(uint8_t *dst, const uint8_t *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy)
{
    const uint32_t main = bytes & ~15u;
    for (uint32_t i = main; i < bytes; ++i) dst[i] = src[i];
    mbar_arrive_expect_tx(bar, main);
    if (main) bulk_g2s_hint(dst, src, main, bar, policy);
}

// ---------------------------------------------------------------------------------------
// fp16 mirror
// ---------------------------------------------------------------------------------------
constexpr int DQ_WARPS = 16;
constexpr int DQ_THREADS = (DQ_WARPS + 1) * 32;
constexpr int DQ_TARGET_CHUNK = 17408;

// Round-to-odd difference of two f32 values: the truncated difference with its last bit set
// when the difference is inexact.  Rounding that to binary16 (11 bits, far fewer than f32's
// 24) gives the correctly rounded binary16 of the exact difference.  Inexactness is read from
// the directed roundings without a compare: for a positive difference the rounding down is
// the truncation and the rounding up is the next float (encoding + 1) when inexact; for a
// negative one the roles swap.  Either way bit 0 of (up | down) is set exactly when the
// truncation is odd or the difference inexact, which is the round-to-odd bit.
__device__ __forceinline__ float sub_round_odd(float a, float b)
{
    const uint32_t z = __float_as_uint(__fsub_rz(a, b));
    const uint32_t t = __float_as_uint(__fsub_ru(a, b)) | __float_as_uint(__fsub_rd(a, b));
    return __uint_as_float((z & ~1u) | (t & 1u));
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi)
{
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// The bytes lane j needs for weights e0 = 8j .. 8j + 7 of a superblock, read from shared
// memory (load), and those weights' values rounded once to binary16, packed in element order
// (packed).  The codes are unpacked four to a word; each code becomes an exact f32 through
// byte_magic and one exact subtraction, and every product below is exact in f32.
template <class F, bool Q6 = F::BYTES == KQ6::BYTES>
struct KqPiece;

template <class F>
struct KqPiece<F, true> {
    uint32_t ql0, ql1, qh0, qh1, head;   // 8 ql bytes, 8 qh bytes, d and the scale byte
    __device__ void load(const uint8_t *sb, int e0)
    {
        const int h = e0 >> 7, pp = e0 & 127, g = pp >> 5, l0 = pp & 31;
        const uint8_t *ql = sb + 64 * h + 32 * (g & 1) + l0;   // 2-byte aligned
        const uint8_t *qh = sb + 128 + 32 * h + l0;
        const uint16_t *a = reinterpret_cast<const uint16_t *>(ql), *b = reinterpret_cast<const uint16_t *>(qh);
        ql0 = a[0] | ((uint32_t)a[1] << 16);
        ql1 = a[2] | ((uint32_t)a[3] << 16);
        qh0 = b[0] | ((uint32_t)b[1] << 16);
        qh1 = b[2] | ((uint32_t)b[3] << 16);
        head = *reinterpret_cast<const uint16_t *>(sb + 208) | ((uint32_t)sb[192 + (e0 >> 4)] << 16);
    }
    // value = d * scale * (code - 32): 11 + 7 + 5 significant bits, exact in f32.
    __device__ uint4 packed(int e0) const
    {
        const int g = (e0 & 127) >> 5;
        const uint32_t s1 = 4 * (g >> 1), s2 = 2 * g;
        const float d = half_bits_to_float(head & 0xffffu);
        const float ds = __fmul_rn(d, (float)(int8_t)(head >> 16));
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t ql = h ? ql1 : ql0, qh = h ? qh1 : qh0;
            const uint32_t code = ((ql >> s1) & 0x0F0F0F0Fu) | (((qh >> s2) & 0x03030303u) << 4);
            float v[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) v[b] = __fmul_rn(ds, __fsub_rn(byte_magic(code, b), 8388640.0f));   // 2^23 + 32
            o[2 * h] = pack_h2(v[0], v[1]);
            o[2 * h + 1] = pack_h2(v[2], v[3]);
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
};

template <class F>
struct KqPiece<F, false> {
    uint32_t head[4];
    uint2 qv, hv;
    __device__ void load(const uint8_t *sb, int e0)
    {
        const uint4 hd = *reinterpret_cast<const uint4 *>(sb);
        head[0] = hd.x; head[1] = hd.y; head[2] = hd.z; head[3] = hd.w;
        const int g = e0 >> 6, l0 = e0 & 31;
        constexpr int QS = F::BYTES == KQ4::BYTES ? 16 : 48;
        qv = *reinterpret_cast<const uint2 *>(sb + QS + 32 * g + l0);
        hv = make_uint2(0, 0);
        if constexpr (F::BYTES == KQ5::BYTES) hv = *reinterpret_cast<const uint2 *>(sb + 16 + l0);
    }
    // value = d * sc * code - dmin * mn: both products exact in f32 (11 + 6 + 5 and 11 + 6
    // significant bits), their difference rounded once to binary16.  Write a finite binary16
    // h as M * 2^(E - 25) with M < 2048 and E its exponent field as stored (a subnormal,
    // M' * 2^-24 with M' < 1024, is 2M' * 2^(0 - 25)).  The difference is then an integer N
    // times 2^(min(Ed, Em) - 25) with
    // |N| <= 2047 * 63 * 31 * 2^(Ed - min) + 2047 * 63 * 2^(Em - min), below 2^24 whenever
    // -6 <= Ed - Em <= 2: there it is an f32, one FMA yields it exactly, and its binary16
    // rounding is the correctly rounded one.  Other superblocks (wider exponent gaps, an
    // infinite or NaN scale) take the difference rounded to odd first, which gives the same
    // binary16 whenever both apply.  The choice is per superblock, so uniform over a warp.
    __device__ uint4 packed(int e0) const
    {
        const int u2 = (e0 >> 5) & 1, j = e0 >> 5;
        uint32_t sc_lo, mn_lo, sc_hi, mn_hi;
        k4_scales_mins(head[1], head[2], head[3], sc_lo, mn_lo, sc_hi, mn_hi);
        const float scf = __fsub_rn(byte_magic(j < 4 ? sc_lo : sc_hi, j & 3), 8388608.0f);
        const float mnf = __fsub_rn(byte_magic(j < 4 ? mn_lo : mn_hi, j & 3), 8388608.0f);
        const float d = half_bits_to_float(head[0] & 0xffffu), dmin = half_bits_to_float(head[0] >> 16);
        const float dsc = __fmul_rn(d, scf), dmm = __fmul_rn(dmin, mnf);
        uint32_t code[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            code[h] = ((h ? qv.y : qv.x) >> (4 * u2)) & 0x0F0F0F0Fu;
            if constexpr (F::BYTES == KQ5::BYTES) code[h] |= (((h ? hv.y : hv.x) >> j) & 0x01010101u) << 4;
        }
        const int ed = (int)((head[0] >> 10) & 31u), em = (int)((head[0] >> 26) & 31u);
        uint32_t o[4];
        if (ed != 31 && em != 31 && (uint32_t)(ed - em + 6) <= 8u) {
            const float ndmm = -dmm;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v[4];
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    v[b] = __fmaf_rn(dsc, __fsub_rn(byte_magic(code[h], b), 8388608.0f), ndmm);
                o[2 * h] = pack_h2(v[0], v[1]);
                o[2 * h + 1] = pack_h2(v[2], v[3]);
            }
        } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v[4];
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    v[b] = sub_round_odd(__fmul_rn(dsc, __fsub_rn(byte_magic(code[h], b), 8388608.0f)), dmm);
                o[2 * h] = pack_h2(v[0], v[1]);
                o[2 * h + 1] = pack_h2(v[2], v[3]);
            }
        }
        return make_uint4(o[0], o[1], o[2], o[3]);
    }
};

template <class F>
__global__ void __launch_bounds__(DQ_THREADS, 2)
    kq_dequant_kernel(const uint8_t *__restrict__ w, uint4 *__restrict__ out, int n, int k, KPlan p, int *status)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    uint64_t *empty = full + KMAX_STAGES;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], DQ_WARPS);
        }
        fence_mbar_init();
    }
    __syncthreads();
    // launched as a programmatic dependent of the stream's previous kernel
    griddep_enter();
    const int64_t my_chunks = blockIdx.x < p.nchunks ? (p.nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    if (warp == DQ_WARPS) {
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();
            int64_t issued = 0;
            for (int64_t i = 0; i < my_chunks; ++i) {
                const int s = (int)(i % p.stages);
                if (!mbar_wait(&empty[s], (uint32_t)(((i / p.stages) & 1) ^ 1), status)) break;
                const int64_t row0 = (blockIdx.x + i * gridDim.x) * p.R;
                const int64_t rows = (n - row0) < p.R ? (n - row0) : p.R;
                produce_chunk(smem + (size_t)s * p.chunk_bytes, w + row0 * p.row_bytes, (uint32_t)rows * p.row_bytes,
                              &full[s], policy);
                ++issued;
            }
            for (int64_t i = issued - p.stages < 0 ? 0 : issued - p.stages; i < issued; ++i)
                mbar_wait_drain(&full[i % p.stages], (uint32_t)((i / p.stages) & 1), status);
        }
        return;
    }

    // Lane j of a warp converts weights 8j .. 8j + 7 of a superblock (one 16-byte output piece).
    const int e0 = 8 * lane;
    for (int64_t i = 0; i < my_chunks; ++i) {
        const int s = (int)(i % p.stages);
        const bool ok = mbar_wait(&full[s], (uint32_t)((i / p.stages) & 1), status);
        if (__any_sync(0xffffffffu, !ok)) break;
        const int64_t row0 = (blockIdx.x + i * gridDim.x) * p.R;
        const int rows = (int)((n - row0) < p.R ? (n - row0) : p.R);
        const uint8_t *sbase = smem + (size_t)s * p.chunk_bytes;
        const int units = rows * p.G;
        // unit u (row u / G, superblock u % G of the chunk) starts at element row0 * k + 256 u
        // of the output, since k = 256 G
        uint4 *outc = out + row0 * (int64_t)(k / 8) + lane;
        // Two superblocks per warp step: both are read from shared memory before either is
        // converted (more loads in flight per warp).
        constexpr int UNR = 2;
        for (int u0 = warp; u0 < units; u0 += UNR * DQ_WARPS) {
            KqPiece<F> pc[UNR];
#pragma unroll
            for (int e = 0; e < UNR; ++e) {
                const int u = u0 + e * DQ_WARPS;
                pc[e].load(sbase + (size_t)(u < units ? u : u0) * F::BYTES, e0);
            }
#pragma unroll
            for (int e = 0; e < UNR; ++e) {
                const int u = u0 + e * DQ_WARPS;
                if (u >= units) break;
                __stcs(outc + 32 * u, pc[e].packed(e0));
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

KPlan dequant_plan(int64_t n, int64_t k, int sb_bytes, size_t smem_cap)
{
    KPlan p{};
    p.G = (int)(k / QK_K);
    p.row_bytes = (uint32_t)(p.G * sb_bytes);
    const int ra = row_align(p.row_bytes);
    p.R = (int)(DQ_TARGET_CHUNK / p.row_bytes) / ra * ra;
    if (p.R < ra) p.R = ra;
    if ((int64_t)p.R > n) p.R = (int)((n + ra - 1) / ra * ra);
    p.chunk_bytes = (uint32_t)p.R * p.row_bytes;
    p.nchunks = (n + p.R - 1) / p.R;
    const size_t room = smem_cap > 2 * KMAX_STAGES * 8 + 64 ? smem_cap - 2 * KMAX_STAGES * 8 - 64 : 0;
    int64_t st = (int64_t)(room / p.chunk_bytes);
    p.stages = (int)(st > KMAX_STAGES ? KMAX_STAGES : st);
    p.off_bar = (size_t)p.stages * p.chunk_bytes;
    p.smem = p.off_bar + 2 * KMAX_STAGES * 8;
    return p;
}

template <class F>
cudaError_t launch_kq_dequant(const DeviceInfo &dev, const uint8_t *w, uint16_t *w16, int64_t n, int64_t k,
                              cudaStream_t stream)
{
    const size_t half_sm = 113 * 1024;
    KPlan p = dequant_plan(n, k, F::BYTES, half_sm < dev.max_smem_optin ? half_sm : dev.max_smem_optin);
    int per_sm = 2;
    if (p.stages < 3) {
        p = dequant_plan(n, k, F::BYTES, dev.max_smem_optin);
        per_sm = 1;
    }
    if (p.stages < 2) return cudaErrorInvalidValue;
    cudaError_t e = set_kernel_smem<kq_dequant_kernel<F>>(dev.device, p.smem);
    if (e != cudaSuccess) return e;
    const int64_t slots = (int64_t)dev.num_sms * per_sm;
    const int64_t grid = p.nchunks < slots ? p.nchunks : slots;
    return launch_dependent(kq_dequant_kernel<F>, (unsigned)grid, DQ_THREADS, p.smem, stream, w,
                            reinterpret_cast<uint4 *>(w16), (int)n, (int)k, p, dev.status);
}

// ---------------------------------------------------------------------------------------
// GEMV
// ---------------------------------------------------------------------------------------
constexpr int GV_CONSUMERS = 128;
constexpr int XG_WORDS = 68;    // activation quants per (token, 256-group): 64 words + 4 pad
constexpr int XDG_WORDS = 12;   // activation scales per (token, group): 8 + 4 pad

KPlan gemv_plan(int64_t m, int64_t n, int64_t k, int sb_bytes, size_t smem_cap, int r_cap)
{
    KPlan p{};
    p.G = (int)(k / QK_K);
    p.row_bytes = (uint32_t)(p.G * sb_bytes);
    const int ra = row_align(p.row_bytes);
    int R = p.G <= GV_CONSUMERS ? GV_CONSUMERS / p.G : 1;
    if (R > r_cap) R = r_cap;
    R = R / ra * ra;
    if (R < ra) R = ra;
    if ((int64_t)R > n) R = (int)((n + ra - 1) / ra * ra);
    p.R = R;
    p.U = p.R * p.G;
    p.chunk_bytes = (uint32_t)p.R * p.row_bytes;
    p.nchunks = (n + p.R - 1) / p.R;
    const size_t x_bytes = (size_t)m * p.G * XG_WORDS * 4;
    const size_t xd_bytes = (size_t)m * p.G * XDG_WORDS * 4;
    // per (token, 32-wide block): the quant sum as an f32 (Q4_K / Q5_K), or for Q6_K at m = 1
    // the two 16-wide halves' sums times -32 as int32
    const size_t xs_bytes = (size_t)m * p.G * 8 * (sb_bytes == KQ6::BYTES && m == 1 ? 8 : 4);
    const size_t part_bytes = 2 * (size_t)p.U * m * 4;
    const size_t fixed = 16 + x_bytes + xd_bytes + xs_bytes + part_bytes + 2 * KMAX_STAGES * 8 + 64;
    const size_t room = smem_cap > fixed ? smem_cap - fixed : 0;
    int64_t st = (int64_t)(room / p.chunk_bytes);
    p.stages = (int)(st > KMAX_STAGES ? KMAX_STAGES : st);
    // 16 bytes after the ring: the Q6_K word loads read up to 6 bytes past a superblock.
    p.off_x = (size_t)p.stages * p.chunk_bytes + 16;
    p.off_xd = p.off_x + x_bytes;
    p.off_xs = p.off_xd + xd_bytes;
    p.off_part = p.off_xs + xs_bytes;
    p.off_bar = (p.off_part + part_bytes + 7) & ~(size_t)7;
    p.smem = p.off_bar + 2 * KMAX_STAGES * 8;
    p.ctas_per_sm = 1;
    p.warp_reduce = (p.G <= 32 && 32 % p.G == 0) ? 1 : 0;
    return p;
}

// MM: the largest token count of the instance; the call's m (<= MM) tokens are folded, each
// with the same operations in the same order for every MM (decode == verify).
template <class F, int MM>
__global__ void __launch_bounds__(GV_CONSUMERS + 32, (MM <= 1 && F::BYTES != KQ6::BYTES) ? 4 : (MM <= 2 ? 3 : 2))
    kq_gemv_kernel(const uint8_t *__restrict__ w, const int8_t *__restrict__ xq, const float *__restrict__ xd,
                   float *__restrict__ y, int32_t *__restrict__ dots, int m, int n, int k, KPlan p, int *status)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    uint32_t *xs = reinterpret_cast<uint32_t *>(smem + p.off_x);
    float *xds = reinterpret_cast<float *>(smem + p.off_xd);
    float *xsum = reinterpret_cast<float *>(smem + p.off_xs);   // exact integers
    float *part = reinterpret_cast<float *>(smem + p.off_part);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    uint64_t *empty = full + KMAX_STAGES;
    const int tid = threadIdx.x;
    const int G = p.G;
    const int nb = k / QK;
    // Q6_K at m = 1: the dots take the codes 0..63 as unsigned bytes and start from -32 times
    // the activation's sum over each 16-wide half, which gives the same integers as the signed
    // codes - 32 without making them signed word by word (4096 -> 64448: 45.4 -> 42.4 us); with
    // more tokens the extra per-token load costs more than it saves.
    constexpr bool Q6U = F::BYTES == KQ6::BYTES && MM == 1;

    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], GV_CONSUMERS / 32);
        }
        fence_mbar_init();
    }
    __syncthreads();
    // launched as a programmatic dependent of the stream's previous kernel
    griddep_enter();
    if (tid < GV_CONSUMERS) {
        // The activation cache: quants [t][group][68 words], scales [t][group][12], and the
        // sum of each 32-wide block's quants (the Q4_K / Q5_K min term).
        for (int idx = tid; idx < m * G * 16; idx += GV_CONSUMERS) {
            const int t = idx / (G * 16), rem = idx - t * G * 16, g = rem >> 4, c = rem & 15;
            const uint4 v = *reinterpret_cast<const uint4 *>(xq + (int64_t)t * k + g * 256 + c * 16);
            *reinterpret_cast<uint4 *>(xs + (t * G + g) * XG_WORDS + c * 4) = v;
        }
        for (int idx = tid; idx < m * G * 2; idx += GV_CONSUMERS) {
            const int t = idx / (G * 2), rem = idx - t * G * 2, g = rem >> 1, c = rem & 1;
            const float4 v = *reinterpret_cast<const float4 *>(xd + (int64_t)t * nb + g * 8 + c * 4);
            *reinterpret_cast<float4 *>(xds + (t * G + g) * XDG_WORDS + c * 4) = v;
        }
        named_bar_sync(2, GV_CONSUMERS);
        for (int idx = tid; idx < m * G * 8; idx += GV_CONSUMERS) {
            const int tg = idx >> 3, j = idx & 7;
            const uint32_t *xv = xs + tg * XG_WORDS + 8 * j;
            if constexpr (Q6U) {
                int s0 = 0, s1 = 0;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    s0 = dp4a(0x01010101u, xv[c], s0);
                    s1 = dp4a(0x01010101u, xv[4 + c], s1);
                }
                reinterpret_cast<int2 *>(xsum)[idx] = make_int2(-32 * s0, -32 * s1);
            } else {
                int sum = 0;
#pragma unroll
                for (int c = 0; c < 8; ++c) sum = dp4a(0x01010101u, xv[c], sum);
                xsum[idx] = __int2float_rn(sum);   // |sum| <= 32 * 127: exact
            }
        }
        named_bar_sync(2, GV_CONSUMERS);
    }

    const int64_t my_chunks = blockIdx.x < p.nchunks ? (p.nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    if (tid >= GV_CONSUMERS) {
        if (tid == GV_CONSUMERS) {
            const uint64_t policy = l2_policy_evict_first();
            int64_t issued = 0;
            for (int64_t i = 0; i < my_chunks; ++i) {
                const int s = (int)(i % p.stages);
                if (!mbar_wait(&empty[s], (uint32_t)(((i / p.stages) & 1) ^ 1), status)) break;
                const int64_t row0 = (blockIdx.x + i * gridDim.x) * p.R;
                const int64_t rows = (n - row0) < p.R ? (n - row0) : p.R;
                produce_chunk(smem + (size_t)s * p.chunk_bytes, w + row0 * p.row_bytes, (uint32_t)rows * p.row_bytes,
                              &full[s], policy);
                ++issued;
            }
            for (int64_t i = issued - p.stages < 0 ? 0 : issued - p.stages; i < issued; ++i)
                mbar_wait_drain(&full[i % p.stages], (uint32_t)((i / p.stages) & 1), status);
        }
        return;
    }

    for (int64_t i = 0; i < my_chunks; ++i) {
        const int s = (int)(i % p.stages);
        const bool ok = mbar_wait(&full[s], (uint32_t)((i / p.stages) & 1), status);
        if (p.warp_reduce ? __any_sync(0xffffffffu, !ok) : bar_red_or(1, GV_CONSUMERS, !ok)) break;
        const int64_t row0 = (blockIdx.x + i * gridDim.x) * p.R;
        const int rows = (int)((n - row0) < p.R ? (n - row0) : p.R);
        const uint8_t *sbase = smem + (size_t)s * p.chunk_bytes;
        float *pbuf = part + (size_t)(i & 1) * p.U * MM;
        const int ulimit = p.warp_reduce ? (p.U + 31) / 32 * 32 : p.U;
        for (int u = tid; u < ulimit; u += GV_CONSUMERS) {
            const int row = u / G;
            const int g = u - row * G;
            float acc[MM];
#pragma unroll
            for (int t = 0; t < MM; ++t) acc[t] = 0.0f;
            if (row < rows) {
                uint32_t wv[F::WORDS];
                load_superblock<F>(sbase + (size_t)row * p.row_bytes + (size_t)g * F::BYTES, wv);
                float d, dmin = 0.0f;
                // Q4_K / Q5_K: the 6-bit scales and mins of all 8 sub-blocks, four to a word
                // (byte j & 3 of the word for sub-block j), unpacked from the 12 scale bytes
                uint32_t sc_lo = 0, mn_lo = 0, sc_hi = 0, mn_hi = 0;
                if constexpr (F::BYTES == KQ6::BYTES) {
                    d = half_bits_to_float(wv[52] & 0xffffu);
                } else {
                    d = half_bits_to_float(wv[0] & 0xffffu);
                    dmin = half_bits_to_float(wv[0] >> 16);
                    k4_scales_mins(wv[1], wv[2], wv[3], sc_lo, mn_lo, sc_hi, mn_hi);
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    uint32_t q[8];
                    block_codes<F, Q6U>(wv, j, q);
                    int sc0 = 0, sc1 = 0;
                    float dsc = 0.0f, dmm = 0.0f;
                    if constexpr (F::BYTES == KQ6::BYTES) {
                        const uint32_t sw = wv[48 + (j >> 1)] >> (16 * (j & 1));
                        sc0 = (int)(int8_t)(sw & 0xFFu);
                        sc1 = (int)(int8_t)((sw >> 8) & 0xFFu);
                    } else {
                        const float scf = __fsub_rn(byte_magic(j < 4 ? sc_lo : sc_hi, j & 3), 8388608.0f);
                        const float mnf = __fsub_rn(byte_magic(j < 4 ? mn_lo : mn_hi, j & 3), 8388608.0f);
                        dsc = __fmul_rn(d, scf);       // exact
                        dmm = __fmul_rn(dmin, mnf);    // exact
                    }
#pragma unroll
                    for (int t = 0; t < MM; ++t) {
                        if (t >= m) break;
                        const uint4 *xv = reinterpret_cast<const uint4 *>(xs + (t * G + g) * XG_WORDS + j * 8);
                        const uint4 a = xv[0], b = xv[1];
                        int D0, D1;
                        if constexpr (Q6U) {
                            // sum (code - 32) * x = sum code * x - 32 * sum x, per 16-wide half
                            const int2 nx = reinterpret_cast<const int2 *>(xsum)[(t * G + g) * 8 + j];
                            D0 = dp4a_us(q[0], a.x, nx.x);
                            D1 = dp4a_us(q[4], b.x, nx.y);
                            D0 = dp4a_us(q[1], a.y, D0);
                            D1 = dp4a_us(q[5], b.y, D1);
                            D0 = dp4a_us(q[2], a.z, D0);
                            D1 = dp4a_us(q[6], b.z, D1);
                            D0 = dp4a_us(q[3], a.w, D0);
                            D1 = dp4a_us(q[7], b.w, D1);
                        } else {
                            D0 = dp4a(q[0], a.x, 0);
                            D1 = dp4a(q[4], b.x, 0);
                            D0 = dp4a(q[1], a.y, D0);
                            D1 = dp4a(q[5], b.y, D1);
                            D0 = dp4a(q[2], a.z, D0);
                            D1 = dp4a(q[6], b.z, D1);
                            D0 = dp4a(q[3], a.w, D0);
                            D1 = dp4a(q[7], b.w, D1);
                        }
                        const float da = xds[(t * G + g) * XDG_WORDS + j];
                        // exact int -> f32 for |D| < 2^22: the bits of D + bits(1.5 * 2^23) are those
                        // of 1.5 * 2^23 + D, and subtracting 1.5 * 2^23 leaves D
                        auto exact_f = [](int D) { return __fsub_rn(__int_as_float(D + 0x4B400000), 12582912.0f); };
                        if constexpr (F::BYTES == KQ6::BYTES) {
                            const int E = sc0 * D0 + sc1 * D1;   // exact, |E| < 2^24
                            if (dots)
                                dots[((int64_t)t * n + row0 + row) * nb + g * 8 + j] = E;
                            else
                                acc[t] = __fmaf_rn(__fmul_rn(d, da), __int2float_rn(E), acc[t]);
                        } else {
                            const int D = D0 + D1;                                   // exact
                            if (dots) {
                                dots[((int64_t)t * n + row0 + row) * nb + g * 8 + j] = D;
                            } else {
                                const float X = xsum[(t * G + g) * 8 + j];
                                const float v = __fmaf_rn(dsc, exact_f(D), -__fmul_rn(dmm, X));
                                acc[t] = __fmaf_rn(da, v, acc[t]);
                            }
                        }
                    }
                }
            }
            if (dots) continue;
            if (p.warp_reduce) {
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    if (o >= G) break;
#pragma unroll
                    for (int t = 0; t < MM; ++t) acc[t] = __fadd_rn(acc[t], __shfl_xor_sync(0xffffffffu, acc[t], o));
                }
                if (g == 0 && row < rows) {
#pragma unroll
                    for (int t = 0; t < MM; ++t)
                        if (t < m) y[(int64_t)t * n + row0 + row] = acc[t];
                }
            } else {
#pragma unroll
                for (int t = 0; t < MM; ++t) pbuf[u * MM + t] = acc[t];
            }
        }
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(&empty[s]);
        if (dots || p.warp_reduce) continue;
        named_bar_sync(1, GV_CONSUMERS);
        for (int idx = tid; idx < rows * m; idx += GV_CONSUMERS) {
            const int t = idx / rows, r = idx - t * rows;
            const float *pr = pbuf + (size_t)r * G * MM + t;
            float sum = pr[0];
            for (int g = 1; g < G; ++g) sum = __fadd_rn(sum, pr[g * MM]);
            y[(int64_t)t * n + row0 + r] = sum;
        }
    }
}

// Q4_K / Q5_K at m = 1: four CTAs per SM, two 18-22 KB stages each in a quarter of shared
// memory (4096 -> 64448: Q4_K 29.8 -> 27.7 us, Q5_K 32.4 -> 30.9 us against three CTAs; Q6_K,
// whose 27 KB chunks leave room for one stage there, stays at three).  Otherwise three CTAs per
// SM when three stages (two for Q6_K) fit in a third of shared memory -- the consumers of these
// formats work harder per streamed byte than Q8_0's, so more of them pay -- else two when three
// stages fit in half, else one CTA with as many stages as fit.
template <class F>
KPlan choose_gemv_plan(int64_t m, int64_t n, int64_t k, size_t smem_optin, int *per_sm)
{
    const size_t third_sm = 74 * 1024, half_sm = 113 * 1024, quarter_sm = 56 * 1024;
    if (m <= 1 && F::BYTES != KQ6::BYTES) {
        KPlan p4 = gemv_plan(m, n, k, F::BYTES, quarter_sm < smem_optin ? quarter_sm : smem_optin, GV_CONSUMERS);
        if (p4.stages >= 2) {
            *per_sm = 4;
            return p4;
        }
    }
    if (m <= 2) {
        KPlan p3 = gemv_plan(m, n, k, F::BYTES, third_sm < smem_optin ? third_sm : smem_optin, GV_CONSUMERS);
        if (p3.stages >= (F::BYTES == KQ6::BYTES ? 2 : 3)) {
            *per_sm = 3;
            return p3;
        }
    }
    KPlan p = gemv_plan(m, n, k, F::BYTES, half_sm < smem_optin ? half_sm : smem_optin, GV_CONSUMERS);
    if (p.stages >= 3) {
        *per_sm = 2;
        return p;
    }
    *per_sm = 1;
    p = gemv_plan(m, n, k, F::BYTES, smem_optin, GV_CONSUMERS);
    for (int r_cap = p.R / 2; p.stages < 2 && r_cap >= 1; r_cap /= 2)
        p = gemv_plan(m, n, k, F::BYTES, smem_optin, r_cap);
    return p;
}

template <class F, int MM>
cudaError_t launch_kq_gemv_m(const DeviceInfo &dev, const uint8_t *w, const int8_t *xq, const float *xd, float *y,
                             int32_t *dots, int64_t m, int64_t n, int64_t k, cudaStream_t stream)
{
    int per_sm = 1;
    KPlan p = choose_gemv_plan<F>(MM, n, k, dev.max_smem_optin, &per_sm);
    if (p.stages < 2) return cudaErrorInvalidValue;
    cudaError_t e = set_kernel_smem<kq_gemv_kernel<F, MM>>(dev.device, p.smem);
    if (e != cudaSuccess) return e;
    // never more CTAs than are resident at once (registers may allow fewer than the plan)
    int resident = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, kq_gemv_kernel<F, MM>, GV_CONSUMERS + 32, p.smem) ==
            cudaSuccess &&
        resident >= 1 && resident < per_sm)
        per_sm = resident;
    const int64_t slots = (int64_t)dev.num_sms * per_sm;
    const int64_t grid = p.nchunks < slots ? p.nchunks : slots;
    return launch_dependent(kq_gemv_kernel<F, MM>, (unsigned)grid, GV_CONSUMERS + 32, p.smem, stream, w, xq, xd, y,
                            dots, (int)m, (int)n, (int)k, p, dev.status);
}

template <class F>
cudaError_t launch_kq_gemv(const DeviceInfo &dev, const uint8_t *w, const int8_t *xq, const float *xd, float *y,
                           int32_t *dots, int64_t m, int64_t n, int64_t k, cudaStream_t stream)
{
    if (m <= 1) return launch_kq_gemv_m<F, 1>(dev, w, xq, xd, y, dots, m, n, k, stream);
    if (m <= 2) return launch_kq_gemv_m<F, 2>(dev, w, xq, xd, y, dots, m, n, k, stream);
    if (m <= 4) return launch_kq_gemv_m<F, 4>(dev, w, xq, xd, y, dots, m, n, k, stream);
    if (m <= 8) return launch_kq_gemv_m<F, 8>(dev, w, xq, xd, y, dots, m, n, k, stream);
    return cudaErrorInvalidValue;
}

template <class F>
bool kq_gemv_fits(const DeviceInfo &dev, int64_t m, int64_t k)
{
    int per_sm = 1;
    const int mm = m <= 1 ? 1 : m <= 2 ? 2 : m <= 4 ? 4 : 8;
    return choose_gemv_plan<F>(mm, 1 << 20, k, dev.max_smem_optin, &per_sm).stages >= 2;
}

}  // namespace

cudaError_t launch_dequant_kq_f16(const DeviceInfo &dev, int fmt, const uint8_t *w, uint16_t *w16, int64_t n,
                                  int64_t k, cudaStream_t stream)
{
    switch (fmt) {
    case 6: return launch_kq_dequant<KQ6>(dev, w, w16, n, k, stream);
    case 4: return launch_kq_dequant<KQ4>(dev, w, w16, n, k, stream);
    case 5: return launch_kq_dequant<KQ5>(dev, w, w16, n, k, stream);
    default: return cudaErrorInvalidValue;
    }
}

bool gemv_kq_supported(const DeviceInfo &dev, int fmt, int64_t m, int64_t k)
{
    if (m < 1 || m > 8) return false;
    switch (fmt) {
    case 6: return kq_gemv_fits<KQ6>(dev, m, k);
    case 4: return kq_gemv_fits<KQ4>(dev, m, k);
    case 5: return kq_gemv_fits<KQ5>(dev, m, k);
    default: return false;
    }
}

cudaError_t launch_gemv_kq(const DeviceInfo &dev, int fmt, const uint8_t *w, const int8_t *xq, const float *xd,
                           float *y, int32_t *dots, int64_t m, int64_t n, int64_t k, cudaStream_t stream)
{
    // from m = 2 on, the tensor-core kernel (same bits) where the row layout allows it
    if (m >= 2 && gemv_kq_mma_supported(dev, fmt, m, k))
        return launch_gemv_kq_mma(dev, fmt, w, xq, xd, y, dots, m, n, k, stream);
    switch (fmt) {
    case 6: return launch_kq_gemv<KQ6>(dev, w, xq, xd, y, dots, m, n, k, stream);
    case 4: return launch_kq_gemv<KQ4>(dev, w, xq, xd, y, dots, m, n, k, stream);
    case 5: return launch_kq_gemv<KQ5>(dev, w, xq, xd, y, dots, m, n, k, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace q8
