// gemv_kq_mma.cu -- the multi-token GEMV (2 <= m <= 8) over the GGUF K-quant superblocks
// (Q6_K 210 bytes, Q4_K 144 bytes, Q5_K 176 bytes per 256 weights; memra-engine 0.81.0
// f16_ffi.rs names them beside Q8_0) on the warp-level int8 tensor-core MMA.
//
// The dp4a K-quant GEMV spends 64 dp4a per superblock on every token, so from m = 2 on the
// integer dots set its pace.  Here a warp computes the dots of a 16-row x 8-token tile of one
// 32-wide sub-block with mma.sync: Q4_K / Q5_K take one m16n8k32 per sub-block (the unsigned
// 4- or 5-bit codes against the signed activation quants: D exact in int32), Q6_K takes two
// m16n8k16, one per 16-wide half, because each half has its own int8 scale (E = s0 * D_a +
// s1 * D_b, exact).  The superblock layouts are the GGUF formats' (kquant.cuh).
//
// Per (row, token) the fold is the dp4a K-quant kernel's, operation for operation: per
// superblock acc = 0, then over its 8 sub-blocks in order
//   Q6_K:         acc = fma(d * d_a, E, acc)
//   Q4_K / Q5_K:  acc = fma(d_a, fma(d*sc, D, -(dmin*mn*X)), acc)   (X: the activation block's quant sum)
// and the superblock sums of a row combined by the same fixed tree (pairwise when the
// superblock count divides 32, else left to right).  Token t's result is therefore bitwise
// the same for every m, and the same as the m = 1 kernel's (the pages' decode == verify law).
//
// Layout and hand-offs are those of the Q8_0 tensor-core GEMV: persistent CTAs, a producer
// warp copying each weight row of a chunk with one cp.async.bulk into a row slot padded to 16
// (mod 128) bytes, 16 MMA warps each owning (16-row tile, superblock) items, 3 reducer warps
// combining a chunk's per-superblock sums while the MMA warps go on; every hand-off is an
// mbarrier with a bounded wait.  Rows must be a multiple of 16 bytes (Q4_K, Q5_K always; Q6_K
// when k is a multiple of 2048); other shapes stay on the dp4a kernel.
#include <type_traits>

#include "common.cuh"
#include "kquant.cuh"
#include "launch.h"

namespace q8 {
namespace {

constexpr int NW = 16;                   // MMA warps
constexpr int NR = 3;                    // reducer warps
constexpr int PRODUCER = NW + NR;        // bulk-copy producer warp
constexpr int THREADS = (NW + NR + 1) * 32;
constexpr int MAX_STAGES = 3;
constexpr int MAX_ITEMS = 4;             // (16-row tile, superblock) items per warp and chunk
constexpr int SUB_BLOCKS = 8;            // 32-wide sub-blocks per superblock

struct KMPlan {
    int G;              // superblocks per row
    int RT;             // 16-row tiles per chunk
    int R;              // rows per chunk (16 * RT)
    int items;          // RT * G
    int stages;
    int warp_tree;      // 1: combine superblocks pairwise (G divides 32), else left to right
    int nparts;         // partial slots (1 or 2)
    uint32_t row_bytes; // weight bytes per row
    uint32_t rs;        // padded row slot in shared memory (16 mod 128)
    uint32_t xs;        // padded activation row of the cache
    uint32_t stage_bytes;
    uint32_t part_bytes; // one partial slot: [G][8 tokens][R] f32
    int64_t nchunks;     // set at launch
    size_t off_x, off_xd, off_xsum, off_part, off_bar, smem;
};

KMPlan make_plan(int64_t k, size_t smem_cap, int sb_bytes, int rt_cap)
{
    KMPlan p{};
    p.G = (int)(k / 256);
    p.RT = (NW + p.G - 1) / p.G;
    if (p.RT > rt_cap) p.RT = rt_cap;
    if (p.RT < 1) p.RT = 1;
    p.R = 16 * p.RT;
    p.items = p.RT * p.G;
    p.row_bytes = (uint32_t)(p.G * sb_bytes);
    p.rs = p.row_bytes + (uint32_t)((16 - (int64_t)(p.row_bytes % 128) + 128) % 128);
    p.xs = (uint32_t)k + 16;   // k is a multiple of 256: activation rows 16 (mod 128) apart
    p.stage_bytes = (uint32_t)p.R * p.rs;
    p.warp_tree = (p.G <= 32 && 32 % p.G == 0) ? 1 : 0;
    p.part_bytes = (uint32_t)((size_t)p.G * 8 * p.R * 4);
    const size_t x_bytes = (size_t)8 * p.xs;
    const size_t xd_bytes = (size_t)(k / QK) * 8 * 4;
    const size_t xsum_bytes = (size_t)(k / QK) * 8 * 4;
    const size_t bars = 2 * (MAX_STAGES + 2) * 8 + 64;
    // two stages and one partial slot at least; then a second slot, then a third stage
    p.stages = 2;
    p.nparts = 1;
    auto total = [&]() {
        return (size_t)p.stages * p.stage_bytes + x_bytes + xd_bytes + xsum_bytes + (size_t)p.nparts * p.part_bytes +
               bars;
    };
    if (total() > smem_cap) p.stages = 0;
    if (p.stages) {
        p.nparts = 2;
        if (total() > smem_cap) p.nparts = 1;
        ++p.stages;
        if (total() > smem_cap) --p.stages;
    }
    p.off_x = (size_t)p.stages * p.stage_bytes;   // multiple of 16
    p.off_xd = p.off_x + x_bytes;
    p.off_xsum = p.off_xd + xd_bytes;
    p.off_part = (p.off_xsum + xsum_bytes + 15) & ~(size_t)15;
    p.off_bar = p.off_part + (size_t)p.nparts * p.part_bytes;
    p.smem = p.off_bar + 2 * (MAX_STAGES + 2) * 8;
    return p;
}

bool plan_ok(const KMPlan &p) { return p.stages >= 2 && (p.items + NW - 1) / NW <= MAX_ITEMS; }

// Weight formats.  codes(sb, j, c, lo, hi): the two words of sub-block j of the superblock at
// sb that lane column c feeds to the MMA, elements 4c..4c+3 (lo) and 16+4c..16+4c+3 (hi) of
// the sub-block as bytes.
//
// Q4_K / Q5_K: 16-byte aligned superblocks (144 and 176 are multiples of 16).  Element l of
// sub-block j = 2g + u is nibble u of qs[32g + l] (Q5_K: plus bit j of qh[l] as the fifth bit).
template <int B>
struct MK45 {
    static constexpr int BYTES = B;
    static constexpr bool Q6 = false;
    static constexpr bool Q5 = B == 176;
    static constexpr int QS = Q5 ? 48 : 16;
    template <bool ALIGNED>
    __device__ static void codes(const uint8_t *sb, int j, int c, uint32_t &lo, uint32_t &hi)
    {
        const int g = j >> 1, u = j & 1;
        const uint8_t *q = sb + QS + 32 * g + 4 * c;
        lo = (lds32(q) >> (4 * u)) & 0x0F0F0F0Fu;
        hi = (lds32(q + 16) >> (4 * u)) & 0x0F0F0F0Fu;
        if constexpr (Q5) {
            const uint8_t *h = sb + 16 + 4 * c;
            lo |= ((lds32(h) >> j) & 0x01010101u) << 4;
            hi |= ((lds32(h + 16) >> j) & 0x01010101u) << 4;
        }
    }
};

// Q6_K: 2-byte aligned superblocks (their offset within a row is g * 210).  Element l of
// sub-block j = 4n + g: low 4 bits from ql[64n + 32(g & 1) + l] (low nibble for g < 2, high
// for g >= 2), high 2 bits from qh[32n + l] >> 2g; the MMA takes code - 32 as a signed byte.
struct MK6 {
    static constexpr int BYTES = 210;
    static constexpr bool Q6 = true;
    // the 4 bytes at p: one word when the superblock is 4-byte aligned, else (2 mod 4) the
    // two aligned words around them, funnel-shifted by 16 bits
    template <bool ALIGNED>
    __device__ static uint32_t word(const uint8_t *p)
    {
        if constexpr (ALIGNED) return lds32(p);
        return __funnelshift_r(lds32(p - 2), lds32(p + 2), 16u);
    }
    __device__ static uint32_t signed_code(uint32_t ql, uint32_t qh, int s1, int s2)
    {
        return q6_signed_bytes(((ql >> s1) & 0x0F0F0F0Fu) | (((qh >> s2) & 0x03030303u) << 4));
    }
    template <bool ALIGNED>
    __device__ static void codes(const uint8_t *sb, int j, int c, uint32_t &lo, uint32_t &hi)
    {
        const int n = j >> 2, g = j & 3;
        const uint8_t *ql = sb + 64 * n + 32 * (g & 1) + 4 * c;
        const uint8_t *qh = sb + 128 + 32 * n + 4 * c;
        lo = signed_code(word<ALIGNED>(ql), word<ALIGNED>(qh), 4 * (g >> 1), 2 * g);
        hi = signed_code(word<ALIGNED>(ql + 16), word<ALIGNED>(qh + 16), 4 * (g >> 1), 2 * g);
    }
};

template <class F, bool DOTS>
__global__ void __launch_bounds__(THREADS, 1)
    kq_mma_kernel(const uint8_t *__restrict__ w, float *__restrict__ y, const int8_t *__restrict__ xq,
                  const float *__restrict__ xd, int32_t *__restrict__ dots, int m, int n, int k, KMPlan p,
                  int *status)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *xs8 = smem + p.off_x;                                          // int8 [8][xs]
    float *xds = reinterpret_cast<float *>(smem + p.off_xd);                // f32 [k/32][8]
    float *xsum = reinterpret_cast<float *>(smem + p.off_xsum);             // f32 [k/32][8], exact integers
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    uint64_t *empty = full + MAX_STAGES;
    uint64_t *pfull = empty + MAX_STAGES;
    uint64_t *pempty = pfull + 2;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int G = p.G;
    const int nb = k / QK;

    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        for (int s = 0; s < p.nparts; ++s) {
            mbar_init(&pfull[s], NW);
            mbar_init(&pempty[s], NR);
        }
        fence_mbar_init();
    }
    __syncthreads();

    const int64_t my_chunks = blockIdx.x < p.nchunks ? (p.nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    if (warp == PRODUCER) {
        // ---------------- producer: one bulk copy per weight row into its padded slot ----------
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();   // the weights are read once
            griddep_wait();   // after the stream's previous kernel (a programmatic dependent)
            int64_t issued = 0;
            for (int64_t i = 0; i < my_chunks; ++i) {
                const int s = (int)(i % p.stages);
                if (!mbar_wait(&empty[s], (uint32_t)(((i / p.stages) & 1) ^ 1), status)) break;
                const int64_t row0 = (blockIdx.x + i * gridDim.x) * p.R;
                const int rows = (int)((n - row0) < p.R ? (n - row0) : p.R);
                mbar_arrive_expect_tx(&full[s], (uint32_t)rows * p.row_bytes);
                uint8_t *dst = smem + (size_t)s * p.stage_bytes;
                for (int r = 0; r < rows; ++r)
                    bulk_g2s_hint(dst + (size_t)r * p.rs, w + (row0 + r) * (int64_t)p.row_bytes, p.row_bytes,
                                  &full[s], policy);
                ++issued;
            }
            for (int64_t i = issued - p.stages < 0 ? 0 : issued - p.stages; i < issued; ++i)
                mbar_wait_drain(&full[i % p.stages], (uint32_t)((i / p.stages) & 1), status);
        }
        return;
    }

    if (warp >= NW) {
        // ---------------- reducers: combine the superblock sums of each chunk in the fixed order
        if (DOTS) return;
        const int rtid = tid - NW * 32;
        for (int64_t i = 0; i < my_chunks; ++i) {
            const int ps = (int)(i % p.nparts);
            const bool ok = mbar_wait(&pfull[ps], (uint32_t)((i / p.nparts) & 1), status);
            if (__any_sync(0xffffffffu, !ok)) break;
            const int64_t row0 = (blockIdx.x + i * gridDim.x) * p.R;
            const int rows = (int)((n - row0) < p.R ? (n - row0) : p.R);
            const float *part = reinterpret_cast<const float *>(smem + p.off_part + (size_t)ps * p.part_bytes);
            const size_t gstride = (size_t)8 * p.R;
            for (int idx = rtid; idx < rows * m; idx += NR * 32) {
                const int t = idx / rows, r = idx - t * rows;   // rows fastest: consecutive addresses
                const float *pr = part + (size_t)t * p.R + r;
                float sum;
                if (p.warp_tree) {
                    // pairwise: ((p0 + p1) + (p2 + p3)) + ..., the dp4a kernel's butterfly order
                    float v[32];
#pragma unroll
                    for (int gg = 0; gg < 32; ++gg) v[gg] = gg < G ? pr[gg * gstride] : 0.0f;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        if (o >= G) break;
#pragma unroll
                        for (int gg = 0; gg < 32; gg += 2 * o)
                            if (gg < G) v[gg] = __fadd_rn(v[gg], v[gg + o]);
                    }
                    sum = v[0];
                } else {
                    sum = pr[0];
                    for (int gg = 1; gg < G; ++gg) sum = __fadd_rn(sum, pr[gg * gstride]);
                }
                y[(int64_t)t * n + row0 + r] = sum;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&pempty[ps]);
        }
        return;
    }

    // ---------------- MMA warps: the activation cache (tokens >= m read as zero) -------------
    griddep_wait();
    griddep_launch_dependents();
    for (int idx = tid; idx < 8 * (k / 16); idx += NW * 32) {
        const int t = idx / (k / 16), c16 = idx - t * (k / 16);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (t < m) v = *reinterpret_cast<const uint4 *>(xq + (int64_t)t * k + c16 * 16);
        *reinterpret_cast<uint4 *>(xs8 + (size_t)t * p.xs + c16 * 16) = v;
    }
    for (int idx = tid; idx < nb * 8; idx += NW * 32) {
        const int b = idx >> 3, t = idx & 7;
        xds[idx] = t < m ? xd[(int64_t)t * nb + b] : 0.0f;
    }
    named_bar_sync(1, NW * 32);
    if constexpr (!F::Q6) {
        // each activation block's quant sum (the min term of Q4_K / Q5_K), exact
        for (int idx = tid; idx < nb * 8; idx += NW * 32) {
            const int b = idx >> 3, t = idx & 7;
            const uint8_t *xp = xs8 + (size_t)t * p.xs + 32 * b;
            int sum = 0;
#pragma unroll
            for (int c = 0; c < 8; ++c) sum = dp4a(0x01010101u, lds32(xp + 4 * c), sum);
            xsum[idx] = __int2float_rn(sum);   // |sum| <= 32 * 127: exact
        }
        named_bar_sync(1, NW * 32);
    }

    const int gl = lane >> 2;     // fragment group: row within an 8-row half, token within 8
    const int c = lane & 3;       // fragment column pair
    for (int64_t i = 0; i < my_chunks; ++i) {
        const int s = (int)(i % p.stages);
        const bool ok = mbar_wait(&full[s], (uint32_t)((i / p.stages) & 1), status);
        if (__any_sync(0xffffffffu, !ok)) break;
        const int64_t row0 = (blockIdx.x + i * gridDim.x) * p.R;
        const int rows = (int)((n - row0) < p.R ? (n - row0) : p.R);
        const uint8_t *stage = smem + (size_t)s * p.stage_bytes;

        float acc[MAX_ITEMS][4];
#pragma unroll
        for (int q = 0; q < MAX_ITEMS; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[q][e] = 0.0f;

#pragma unroll
        for (int q = 0; q < MAX_ITEMS; ++q) {
            const int it = warp + q * NW;
            if (it >= p.items) break;
            const int rt = it / G, g = it - rt * G;
            // this lane's two rows (gl, gl + 8 of the tile) and their superblock g
            const uint8_t *sb0 = stage + (size_t)(16 * rt + gl) * p.rs + (size_t)g * F::BYTES;
            const uint8_t *sb1 = sb0 + (size_t)8 * p.rs;
            float d0, d1, dmin0 = 0.0f, dmin1 = 0.0f;
            // Q4_K / Q5_K: each row's 8 scales and mins, four to a word (scales of sub-blocks
            // 0..3, mins 0..3, scales 4..7, mins 4..7)
            uint32_t s0[4] = {0u, 0u, 0u, 0u}, s1[4] = {0u, 0u, 0u, 0u};
            if constexpr (F::Q6) {
                d0 = half_bits_to_float(lds16(sb0 + 208));
                d1 = half_bits_to_float(lds16(sb1 + 208));
            } else {
                const uint4 a = *reinterpret_cast<const uint4 *>(sb0);
                const uint4 b = *reinterpret_cast<const uint4 *>(sb1);
                d0 = half_bits_to_float(a.x & 0xffffu);
                dmin0 = half_bits_to_float(a.x >> 16);
                d1 = half_bits_to_float(b.x & 0xffffu);
                dmin1 = half_bits_to_float(b.x >> 16);
                k4_scales_mins(a.y, a.z, a.w, s0[0], s0[1], s0[2], s0[3]);
                k4_scales_mins(b.y, b.z, b.w, s1[0], s1[1], s1[2], s1[3]);
            }
            auto fold_superblock = [&](auto aligned) {
                constexpr bool AL = decltype(aligned)::value;
#pragma unroll
                for (int j = 0; j < SUB_BLOCKS; ++j) {
                    uint32_t w0lo, w0hi, w1lo, w1hi;
                    F::template codes<AL>(sb0, j, c, w0lo, w0hi);
                    F::template codes<AL>(sb1, j, c, w1lo, w1hi);
                    const int b = g * SUB_BLOCKS + j;
                    const uint8_t *xp = xs8 + (size_t)gl * p.xs + 32 * b + 4 * c;
                    const float2 da = *reinterpret_cast<const float2 *>(xds + b * 8 + 2 * c);
                    // the exact integers of the block dots as f32 (E, or D for Q4_K / Q5_K)
                    float Ef[4];
                    int E[4];
                    if constexpr (F::Q6) {
                        // two 16-wide halves, each with its own int8 scale
                        int Da[4], Db[4];
                        mma_s8_16816(Da, w0lo, w1lo, lds32(xp));
                        mma_s8_16816(Db, w0hi, w1hi, lds32(xp + 16));
                        const uint32_t s0 = lds16(sb0 + 192 + 2 * j), s1 = lds16(sb1 + 192 + 2 * j);
                        const int s0a = (int)(int8_t)(s0 & 0xFFu), s0b = (int)(int8_t)(s0 >> 8);
                        const int s1a = (int)(int8_t)(s1 & 0xFFu), s1b = (int)(int8_t)(s1 >> 8);
                        E[0] = s0a * Da[0] + s0b * Db[0];
                        E[1] = s0a * Da[1] + s0b * Db[1];
                        E[2] = s1a * Da[2] + s1b * Db[2];
                        E[3] = s1a * Da[3] + s1b * Db[3];
                        // |E| < 2^24: exact in f32, but beyond the magic conversion's 2^22
#pragma unroll
                        for (int e = 0; e < 4; ++e) Ef[e] = __int2float_rn(E[e]);
                    } else {
                        const uint32_t a[4] = {w0lo, w1lo, w0hi, w1hi};
                        mma_s8_16832(E, a, lds32(xp), lds32(xp + 16));
                        // |D| < 2^22: the f32 with the bits of D + bits(1.5 * 2^23) is exactly
                        // 1.5 * 2^23 + D, and subtracting 1.5 * 2^23 leaves D
#pragma unroll
                        for (int e = 0; e < 4; ++e) Ef[e] = __fsub_rn(__int_as_float(E[e] + 0x4B400000), 12582912.0f);
                    }
                    // E[0]: (row gl, token 2c), E[1]: (gl, 2c+1), E[2]: (gl+8, 2c), E[3]: (gl+8, 2c+1)
                    if (DOTS) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int r = 16 * rt + gl + 8 * (e >> 1);
                            const int t = 2 * c + (e & 1);
                            if (r < rows && t < m) dots[((int64_t)t * n + row0 + r) * nb + b] = E[e];
                        }
                        continue;
                    }
                    if constexpr (F::Q6) {
                        const float s00 = __fmul_rn(d0, da.x), s01 = __fmul_rn(d0, da.y);
                        const float s10 = __fmul_rn(d1, da.x), s11 = __fmul_rn(d1, da.y);
                        acc[q][0] = __fmaf_rn(s00, Ef[0], acc[q][0]);
                        acc[q][1] = __fmaf_rn(s01, Ef[1], acc[q][1]);
                        acc[q][2] = __fmaf_rn(s10, Ef[2], acc[q][2]);
                        acc[q][3] = __fmaf_rn(s11, Ef[3], acc[q][3]);
                    } else {
                        // the 6-bit scale and min as exact f32 (byte under 2^23, one exact subtraction)
                        const int hi = j < 4 ? 0 : 2;
                        const float sc0 = __fsub_rn(byte_magic(s0[hi], j & 3), 8388608.0f);
                        const float mn0 = __fsub_rn(byte_magic(s0[hi + 1], j & 3), 8388608.0f);
                        const float sc1 = __fsub_rn(byte_magic(s1[hi], j & 3), 8388608.0f);
                        const float mn1 = __fsub_rn(byte_magic(s1[hi + 1], j & 3), 8388608.0f);
                        const float dsc0 = __fmul_rn(d0, sc0), dmm0 = __fmul_rn(dmin0, mn0);   // exact
                        const float dsc1 = __fmul_rn(d1, sc1), dmm1 = __fmul_rn(dmin1, mn1);
                        const float2 X = *reinterpret_cast<const float2 *>(xsum + b * 8 + 2 * c);
                        const float v0 = __fmaf_rn(dsc0, Ef[0], -__fmul_rn(dmm0, X.x));
                        const float v1 = __fmaf_rn(dsc0, Ef[1], -__fmul_rn(dmm0, X.y));
                        const float v2 = __fmaf_rn(dsc1, Ef[2], -__fmul_rn(dmm1, X.x));
                        const float v3 = __fmaf_rn(dsc1, Ef[3], -__fmul_rn(dmm1, X.y));
                        acc[q][0] = __fmaf_rn(da.x, v0, acc[q][0]);
                        acc[q][1] = __fmaf_rn(da.y, v1, acc[q][1]);
                        acc[q][2] = __fmaf_rn(da.x, v2, acc[q][2]);
                        acc[q][3] = __fmaf_rn(da.y, v3, acc[q][3]);
                    }
                }
            };
            // Q6_K superblocks sit 2 (mod 4) bytes into the row slot for odd g (the same for
            // every row of the tile: row slots are 16-byte multiples apart)
            if (!F::Q6 || (g & 1) == 0)
                fold_superblock(std::integral_constant<bool, true>{});
            else
                fold_superblock(std::integral_constant<bool, false>{});
        }
        // this warp's reads of the stage are done
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (DOTS) continue;

        // park the superblock sums in partial slot ps ([superblock][token][row]) once the
        // reducers are done with the slot's previous chunk
        const int ps = (int)(i % p.nparts);
        const bool free_ok = i < p.nparts ||
                             mbar_wait(&pempty[ps], (uint32_t)(((i / p.nparts) & 1) ^ 1), status);
        if (__any_sync(0xffffffffu, !free_ok)) break;
        float *part = reinterpret_cast<float *>(smem + p.off_part + (size_t)ps * p.part_bytes);
#pragma unroll
        for (int q = 0; q < MAX_ITEMS; ++q) {
            const int it = warp + q * NW;
            if (it >= p.items) break;
            const int rt = it / G, g = it - rt * G;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = 16 * rt + gl + 8 * (e >> 1);
                const int t = 2 * c + (e & 1);
                part[((size_t)g * 8 + t) * p.R + r] = acc[q][e];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[ps]);
    }
}

int sb_bytes_of(int fmt) { return fmt == 6 ? 210 : fmt == 4 ? 144 : fmt == 5 ? 176 : 0; }

// 16-row tiles per chunk: the count that minimises waves of chunks over the SMs times rounds
// of items per MMA warp, ties to fewer (more SMs streaming).
int rt_cap_for(const DeviceInfo &dev, int64_t n, int64_t k)
{
    const int64_t tiles = (n + 15) / 16;
    const int g = (int)(k / 256), rt0 = (NW + g - 1) / g > 1 ? (NW + g - 1) / g : 1;
    int cap = 1;
    int64_t best = -1;
    for (int rt = 1; rt <= rt0; ++rt) {
        const int64_t waves = ((tiles + rt - 1) / rt + dev.num_sms - 1) / dev.num_sms;
        const int64_t cost = waves * ((rt * g + NW - 1) / NW);
        if (best < 0 || cost < best) {
            best = cost;
            cap = rt;
        }
    }
    return cap;
}

template <class F, bool DOTS>
cudaError_t launch_f(const DeviceInfo &dev, const uint8_t *w, const int8_t *xq, const float *xd, float *y,
                     int32_t *dots, int64_t m, int64_t n, int64_t k, cudaStream_t stream)
{
    KMPlan p = make_plan(k, dev.max_smem_optin, F::BYTES, rt_cap_for(dev, n, k));
    if (!plan_ok(p) || p.row_bytes % 16 != 0) return cudaErrorInvalidValue;
    p.nchunks = (n + p.R - 1) / p.R;
    cudaError_t e = set_kernel_smem<kq_mma_kernel<F, DOTS>>(dev.device, p.smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = p.nchunks < dev.num_sms ? p.nchunks : dev.num_sms;
    return launch_dependent(kq_mma_kernel<F, DOTS>, (unsigned)grid, THREADS, p.smem, stream, w, y, xq, xd, dots,
                            (int)m, (int)n, (int)k, p, dev.status);
}

template <class F>
cudaError_t launch_fmt(const DeviceInfo &dev, const uint8_t *w, const int8_t *xq, const float *xd, float *y,
                       int32_t *dots, int64_t m, int64_t n, int64_t k, cudaStream_t stream)
{
    return dots ? launch_f<F, true>(dev, w, xq, xd, y, dots, m, n, k, stream)
                : launch_f<F, false>(dev, w, xq, xd, y, dots, m, n, k, stream);
}

}  // namespace

bool gemv_kq_mma_supported(const DeviceInfo &dev, int fmt, int64_t m, int64_t k)
{
    const int sb = sb_bytes_of(fmt);
    if (!sb || m < 2 || m > 8 || k % 256 != 0) return false;
    const KMPlan p = make_plan(k, dev.max_smem_optin, sb, 1 << 20);
    return plan_ok(p) && p.row_bytes % 16 == 0;
}

cudaError_t launch_gemv_kq_mma(const DeviceInfo &dev, int fmt, const uint8_t *w, const int8_t *xq, const float *xd,
                               float *y, int32_t *dots, int64_t m, int64_t n, int64_t k, cudaStream_t stream)
{
    switch (fmt) {
    case 6: return launch_fmt<MK6>(dev, w, xq, xd, y, dots, m, n, k, stream);
    case 4: return launch_fmt<MK45<144>>(dev, w, xq, xd, y, dots, m, n, k, stream);
    case 5: return launch_fmt<MK45<176>>(dev, w, xq, xd, y, dots, m, n, k, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace q8
