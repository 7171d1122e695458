// gemv_mma.cu -- the multi-token GEMV (speculative verify and small batches, m <= 16) on the
// warp-level tensor-core MMA, over Q8_0 (from m = 2) or Q4_0 (from m = 5) weights.
//
// The dp4a GEMV re-reads the activation from shared memory for every row it folds, so above
// m = 1 it is bound by shared-memory bandwidth.  Here a warp computes a 16-row x 8-token tile
// of block dots on the tensor cores: each row fragment is read once for 8 tokens, each token
// fragment once for 16 rows.  One token group (m <= 8) takes one mma.sync m16n8k32 (s8 in,
// s32 out) per block: the block dot itself, converted exactly to f32 (|D| < 2^19).  Two token
// groups take two mma.sync m16n8k16 per block and group on exact binary16 integers (f32
// accumulation; every partial sum is an integer below 2^19, exact), so each weight fragment
// is converted once and serves both groups: the int8 MMA runs at a third of the f16 rate on
// this part, and two of them per block would bound the kernel.
//
// Per (row, token) the fold is the dp4a kernel's, operation for operation: acc = 0, then
// acc = fma(d_w * d_a, D, acc) over the 8 blocks of each 256-wide group in order, then the
// groups' sums combined by the same fixed tree (pairwise when the group count divides 32, else
// left to right).  Token t's result is therefore bitwise the same for every m, and the same as
// the m = 1 kernel's (the pages' decode == verify law, fp8_ffi.rs and f16_ffi.rs module docs).
//
// Layout: persistent CTAs; a producer warp copies R weight rows per chunk with one
// cp.async.bulk per row into row slots padded to 16 (mod 128) bytes, so that the 8 rows a
// warp reads at once fall in distinct banks.  The activation (int8) and its scales sit in
// shared memory for the whole kernel, padded the same way.  Each MMA warp hands its weight
// stage back once it has finished the chunk's items (handing it back right after the fragment
// reads, before the MMAs, measured no faster) and parks its per-group partial sums in a partial
// slot ([group][token][row]); reducer warps combine a chunk's partials in the fixed order and
// store y while the MMA warps go on with the next chunk.  Every hand-off is an mbarrier with
// a bounded wait; there is no CTA-wide barrier in the loop.
#include "common.cuh"
#include "launch.h"

namespace q8 {
namespace {

constexpr int NW = 16;                   // MMA warps
constexpr int NR = 3;                    // reducer warps
constexpr int PRODUCER = NW + NR;        // bulk-copy producer warp
constexpr int THREADS = (NW + NR + 1) * 32;
constexpr int MAX_STAGES = 3;
constexpr int MAX_ITEMS = 4;             // (16-row tile, group) items per warp and chunk

struct MPlan {
    int G;              // 256-wide groups per row
    int RT;             // 16-row tiles per chunk
    int R;              // rows per chunk (16 * RT)
    int items;          // RT * G
    int stages;
    int warp_tree;      // 1: combine groups pairwise (G divides 32), else left to right
    uint32_t row_bytes; // weight bytes per row
    uint32_t rs;        // padded row slot in shared memory (16 mod 128)
    uint32_t xs;        // padded activation row of the cache
    uint32_t stage_bytes;
    uint32_t part_bytes; // one partial slot: [G][8 mt][R] f32
    int nparts;          // partial slots (1 or 2)
    int wait_weights;    // 1: the producer waits for the stream's previous kernel before streaming
    int64_t nchunks;    // chunks of the whole group (set at launch)
    size_t off_x, off_xd, off_part, off_bar, smem;
};

// rt_cap: at most this many 16-row tiles per chunk.  A chunk takes up to enough tiles to give
// each MMA warp an item (16 / G of them); the launch picks the count that minimises waves of
// chunks over the SMs times rounds of items per warp (k = 1280, five groups per row: two tiles
// per chunk at 4096 rows -- one wave of 128 chunks, 10 items each -- and three at 20480 rows,
// where four would give 20 items to 16 warps).
MPlan make_mplan(int mt, int64_t k, size_t smem_cap, int block_bytes, int rt_cap = 1 << 20)
{
    MPlan p{};
    p.G = (int)(k / 256);
    p.RT = (NW + p.G - 1) / p.G;
    if (p.RT > rt_cap) p.RT = rt_cap;
    if (p.RT < 1) p.RT = 1;
    p.R = 16 * p.RT;
    p.items = p.RT * p.G;
    p.row_bytes = (uint32_t)(k / QK * block_bytes);
    p.rs = p.row_bytes + (uint32_t)((16 - (int64_t)(p.row_bytes % 128) + 128) % 128);
    // int8 activation cache, rows 16 (mod 128) bytes apart
    p.xs = (uint32_t)k + 16;
    p.stage_bytes = (uint32_t)p.R * p.rs;
    p.warp_tree = (p.G <= 32 && 32 % p.G == 0) ? 1 : 0;
    p.part_bytes = (uint32_t)((size_t)p.G * 8 * mt * p.R * 4);
    const size_t x_bytes = (size_t)8 * mt * p.xs;
    const size_t xd_bytes = (size_t)(k / QK) * 8 * mt * 4;
    const size_t bars = 2 * (MAX_STAGES + 2) * 8 + 64;
    // two stages and one partial slot at least; then a second slot, then a third stage
    p.stages = 2;
    p.nparts = 1;
    auto total = [&]() {
        return (size_t)p.stages * p.stage_bytes + x_bytes + xd_bytes + (size_t)p.nparts * p.part_bytes + bars;
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
    p.off_part = (p.off_xd + xd_bytes + 15) & ~(size_t)15;
    p.off_bar = p.off_part + (size_t)p.nparts * p.part_bytes;
    p.smem = p.off_bar + 2 * (MAX_STAGES + 2) * 8;
    return p;
}

bool mplan_ok(const MPlan &p, int)
{
    return p.stages >= 2 && (p.items + NW - 1) / NW <= MAX_ITEMS;
}

// Four signed bytes -> two f16x2 words holding the same integers (exact): (b ^ 0x80) is q + 128,
// the binary16 pattern 0x64uu is 1024 + uu, and 1152 is subtracted.
__device__ __forceinline__ void s8x4_to_f16x2x2(uint32_t q4, uint32_t &lo, uint32_t &hi)
{
    const uint32_t u = q4 ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x5140);
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x5342);
    const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
    lo = *reinterpret_cast<const uint32_t *>(&ha);
    hi = *reinterpret_cast<const uint32_t *>(&hb);
}

// Weight formats.  quants(): the two words of block j of group g of a row (in its slot) that
// this lane feeds to the int8 MMA: lo holds elements 4c..4c+3 and hi elements 16+4c..16+4c+3
// of the block, as signed bytes.  The int8 MMA then sums 2^SHIFT * D exactly.
//
// Q8_0 (34-byte blocks): the quants themselves, bytes 4c..4c+3 and 16+4c..16+4c+3.
struct MQ8_0 {
    static constexpr int BLOCK_BYTES = Q8_0_BYTES;
    static constexpr int GROUP = GROUP_BYTES;
    static constexpr int SHIFT = 0;
    // From m = 2 on this kernel beats the dp4a GEMV (4096 -> 64448: 58.5 vs 61.6 us at m = 2).
    static constexpr int MIN_M = 2;
    __device__ static void quants(const uint8_t *rowp, int g, int j, int c, uint32_t &lo, uint32_t &hi)
    {
        const int bo = g * GROUP + j * BLOCK_BYTES;   // block start (2 mod 4 when j is odd)
        if ((j & 1) == 0) {
            // quants start at bo + 2, 2 mod 4: two aligned words each, bytes 2..5 of the pair
            const uint8_t *q = rowp + bo + 4 * c;
            lo = __byte_perm(lds32(q), lds32(q + 4), 0x5432);
            hi = __byte_perm(lds32(q + 16), lds32(q + 20), 0x5432);
        } else {
            const uint8_t *q = rowp + bo + 2 + 4 * c;       // word aligned
            lo = lds32(q);
            hi = lds32(q + 16);
        }
    }
};

// Q4_0 (GGUF 18-byte blocks): element i < 16 in the low nibble of quant byte i, element i + 16
// in its high nibble, value d * (nibble - 8).  Quant bytes 4c..4c+3 hold both of this lane's
// element sets; each nibble is moved to the top of its byte and the byte's sign bit flipped,
// which is the signed byte 16 * (nibble - 8).
struct MQ4_0 {
    static constexpr int BLOCK_BYTES = Q4_0_BYTES;
    static constexpr int GROUP = Q4_GROUP_BYTES;
    static constexpr int SHIFT = 4;
    // Half the bytes of Q8_0 for the same MMA work: the dp4a GEMV stays ahead up to m = 3 and
    // ties at m = 4 (4096 -> 64448: 36.1 / 45.5 / 59.7 us at m = 2 / 3 / 4 against ~57.5 here,
    // ahead at 4096 x 4096); 95.3 against 57.7 at m = 8, 229.8 against ~84 at m = 15.
    static constexpr int MIN_M = 5;
    __device__ static void quants(const uint8_t *rowp, int g, int j, int c, uint32_t &lo, uint32_t &hi)
    {
        const int bo = g * GROUP + j * BLOCK_BYTES;   // block start (2 mod 4 when j is odd)
        uint32_t q4;
        if ((j & 1) == 0) {
            const uint8_t *q = rowp + bo + 4 * c;     // quant bytes 4c.. start 2 bytes in
            q4 = __byte_perm(lds32(q), lds32(q + 4), 0x5432);
        } else {
            q4 = lds32(rowp + bo + 2 + 4 * c);        // word aligned
        }
        lo = ((q4 << 4) & 0xF0F0F0F0u) ^ 0x80808080u;
        hi = (q4 & 0xF0F0F0F0u) ^ 0x80808080u;
    }
};

template <class F, int MT, bool DOTS>
__global__ void __launch_bounds__(THREADS, 1)
    gemv_mma_kernel(const __grid_constant__ Group grp, const int8_t *__restrict__ xq,
                    const float *__restrict__ xd, int32_t *__restrict__ dots, int m, int k, MPlan p,
                    int *status)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    // activation cache [8 MT][xs], int8
    uint8_t *xs8 = smem + p.off_x;
    // one token group: one int8 MMA per block; two: the weight fragment converted to binary16
    // once and fed to the f16 MMA for both groups
    constexpr bool I8 = MT == 1;
    float *xds = reinterpret_cast<float *>(smem + p.off_xd);         // f32 [k/32][8 MT]
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    uint64_t *empty = full + MAX_STAGES;
    uint64_t *pfull = empty + MAX_STAGES;
    uint64_t *pempty = pfull + 2;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int G = p.G;
    const int nb = k / QK;
    constexpr int TOK = 8 * MT;

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

    const int64_t my_chunks =
        blockIdx.x < p.nchunks ? (p.nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    if (warp == PRODUCER) {
        // ---------------- producer: one bulk copy per weight row into its padded slot ----------
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();   // the weights are read once
            if (p.wait_weights) griddep_wait();
            int64_t issued = 0;
            for (int64_t i = 0; i < my_chunks; ++i) {
                const int s = (int)(i % p.stages);
                if (!mbar_wait(&empty[s], (uint32_t)(((i / p.stages) & 1) ^ 1), status)) break;
                const ChunkRef cr = chunk_ref(grp, blockIdx.x + i * gridDim.x, p.R);
                const int64_t row0 = cr.row0;
                const int rows = cr.rows;
                mbar_arrive_expect_tx(&full[s], (uint32_t)rows * p.row_bytes);
                uint8_t *dst = smem + (size_t)s * p.stage_bytes;
                for (int r = 0; r < rows; ++r)
                    bulk_g2s_hint(dst + (size_t)r * p.rs, cr.w + (row0 + r) * (int64_t)p.row_bytes, p.row_bytes,
                                  &full[s], policy);
                ++issued;
            }
            for (int64_t i = issued - p.stages < 0 ? 0 : issued - p.stages; i < issued; ++i)
                mbar_wait_drain(&full[i % p.stages], (uint32_t)((i / p.stages) & 1), status);
        }
        return;
    }

    if (warp >= NW) {
        // ---------------- reducers: combine the groups of each chunk in the fixed order -------
        if (DOTS) return;
        const int rtid = tid - NW * 32;
        for (int64_t i = 0; i < my_chunks; ++i) {
            const int ps = (int)(i % p.nparts);
            const bool ok = mbar_wait(&pfull[ps], (uint32_t)((i / p.nparts) & 1), status);
            if (__any_sync(0xffffffffu, !ok)) break;
            const ChunkRef cr = chunk_ref(grp, blockIdx.x + i * gridDim.x, p.R);
            const int64_t row0 = cr.row0;
            const int rows = cr.rows;
            const float *part = reinterpret_cast<const float *>(smem + p.off_part + (size_t)ps * p.part_bytes);
            const size_t gstride = (size_t)TOK * p.R;
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
                cr.y[(int64_t)t * cr.n + row0 + r] = sum;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&pempty[ps]);
        }
        return;
    }

    // ---------------- MMA warps: the activation cache (tokens >= m read as zero) -------------
    // (after the stream's previous kernel: this kernel is launched as its programmatic
    // dependent; in a fused call that is the call's own quantizer, and the weight stream does
    // not wait for it)
    griddep_wait();
    griddep_launch_dependents();
    for (int idx = tid; idx < TOK * (k / 16); idx += NW * 32) {
        const int t = idx / (k / 16), c16 = idx - t * (k / 16);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (t < m) v = *reinterpret_cast<const uint4 *>(xq + (int64_t)t * k + c16 * 16);
        *reinterpret_cast<uint4 *>(xs8 + (size_t)t * p.xs + c16 * 16) = v;
    }
    for (int idx = tid; idx < nb * TOK; idx += NW * 32) {
        const int b = idx / TOK, t = idx - b * TOK;
        xds[idx] = t < m ? xd[(int64_t)t * nb + b] : 0.0f;
    }
    named_bar_sync(1, NW * 32);

    const int gl = lane >> 2;     // fragment group: row within an 8-row half, token within 8
    const int c = lane & 3;       // fragment column pair
    for (int64_t i = 0; i < my_chunks; ++i) {
        const int s = (int)(i % p.stages);
        const bool ok = mbar_wait(&full[s], (uint32_t)((i / p.stages) & 1), status);
        if (__any_sync(0xffffffffu, !ok)) break;
        // (the block-dot export serves a group of one)
        const int64_t row0 = (blockIdx.x + i * gridDim.x) * p.R;
        const int n = grp.n[0];
        const int rows = (int)((n - row0) < p.R ? (n - row0) : p.R);
        const uint8_t *stage = smem + (size_t)s * p.stage_bytes;

        float acc[MAX_ITEMS][MT][4];
#pragma unroll
        for (int q = 0; q < MAX_ITEMS; ++q)
#pragma unroll
            for (int tg = 0; tg < MT; ++tg)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[q][tg][e] = 0.0f;

#pragma unroll
        for (int q = 0; q < MAX_ITEMS; ++q) {
            const int it = warp + q * NW;
            if (it >= p.items) break;
            const int rt = it / G, g = it - rt * G;
            const uint8_t *r0p = stage + (size_t)(16 * rt + gl) * p.rs;
            const uint8_t *r1p = r0p + (size_t)8 * p.rs;
            // the group's 8 blocks unrolled (2 -> 8: Q4_0 m = 8 60.8 -> 57.7 us, Q8_0 m = 12
            // 86.2 -> 81.4 us at 4096 -> 64448)
#pragma unroll
            for (int j = 0; j < GROUP_BLOCKS; ++j) {
                uint32_t w0lo, w0hi, w1lo, w1hi;
                F::quants(r0p, g, j, c, w0lo, w0hi);
                F::quants(r1p, g, j, c, w1lo, w1hi);
                // f16 A fragments: k16 step 0 takes bytes 4c..4c+3, step 1 bytes 16+4c..16+4c+3;
                // the int8 m16n8k32 fragment takes the same words as they are
                uint32_t a0[4], a1[4];
                if constexpr (I8) {
                    a0[0] = w0lo; a0[1] = w1lo; a0[2] = w0hi; a0[3] = w1hi;
                } else {
                    s8x4_to_f16x2x2(w0lo, a0[0], a0[2]);
                    s8x4_to_f16x2x2(w1lo, a0[1], a0[3]);
                    s8x4_to_f16x2x2(w0hi, a1[0], a1[2]);
                    s8x4_to_f16x2x2(w1hi, a1[1], a1[3]);
                }
                const int bo = g * F::GROUP + j * F::BLOCK_BYTES;
                const float dw0 = half_bits_to_float(*reinterpret_cast<const uint16_t *>(r0p + bo));
                const float dw1 = half_bits_to_float(*reinterpret_cast<const uint16_t *>(r1p + bo));
                const int b = g * GROUP_BLOCKS + j;
#pragma unroll
                for (int tg = 0; tg < MT; ++tg) {
                    const uint8_t *xp = xs8 + (size_t)(8 * tg + gl) * p.xs + 32 * b + 4 * c;
                    float D[4];
                    if constexpr (I8) {
                        // the exact int32 block dot (|D| < 2^19, a multiple of 2^SHIFT before
                        // the shift), converted exactly
                        int di[4];
                        mma_s8_16832(di, a0, lds32(xp), lds32(xp + 16));
                        // int -> f32 without the conversion pipe: for |D| < 2^22 the f32 with
                        // the bits of D + bits(1.5 * 2^23) is exactly 1.5 * 2^23 + D (unit
                        // spacing there), and subtracting 1.5 * 2^23 leaves D exactly
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            D[e] = __fsub_rn(__int_as_float((di[e] >> F::SHIFT) + 0x4B400000), 12582912.0f);
                    } else {
                        uint32_t b0lo, b0hi, b1lo, b1hi;
                        s8x4_to_f16x2x2(lds32(xp), b0lo, b0hi);
                        s8x4_to_f16x2x2(lds32(xp + 16), b1lo, b1hi);
                        const float zero[4] = {0.f, 0.f, 0.f, 0.f};
                        float d[4];
                        mma_f16_16816(d, a0, b0lo, b0hi, zero);
                        mma_f16_16816(D, a1, b1lo, b1hi, d);
                        // 2^SHIFT * D is an integer below 2^24 (exact in f32); the scaling by a
                        // power of two is exact
                        if (F::SHIFT)
#pragma unroll
                            for (int e = 0; e < 4; ++e) D[e] *= 1.0f / (float)(1 << F::SHIFT);
                    }
                    // D[0]: (row gl, token 2c), D[1]: (gl, 2c+1), D[2]: (gl+8, 2c), D[3]: (gl+8, 2c+1)
                    if (DOTS) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int r = 16 * rt + gl + 8 * (e >> 1);
                            const int t = 8 * tg + 2 * c + (e & 1);
                            if (r < rows && t < m)
                                dots[((int64_t)t * n + row0 + r) * nb + b] = __float2int_rn(D[e]);
                        }
                    } else {
                        // acc = fma(d_w * d_a, D, acc) per lane
                        const float2 da = *reinterpret_cast<const float2 *>(xds + b * TOK + 8 * tg + 2 * c);
                        if constexpr (I8 && F::SHIFT == 0) {
                            // Q8_0, one token group: one lane per instruction (m = 2..8, 4096 ->
                            // 64448: 55.3 -> 54.3 us; the packed form below is faster for two
                            // token groups and for Q4_0)
                            acc[q][tg][0] = __fmaf_rn(__fmul_rn(dw0, da.x), D[0], acc[q][tg][0]);
                            acc[q][tg][1] = __fmaf_rn(__fmul_rn(dw0, da.y), D[1], acc[q][tg][1]);
                            acc[q][tg][2] = __fmaf_rn(__fmul_rn(dw1, da.x), D[2], acc[q][tg][2]);
                            acc[q][tg][3] = __fmaf_rn(__fmul_rn(dw1, da.y), D[3], acc[q][tg][3]);
                        } else {
                            // two lanes per instruction
                            const float2 s0 = __fmul2_rn(make_float2(dw0, dw0), da);
                            const float2 s1 = __fmul2_rn(make_float2(dw1, dw1), da);
                            const float2 r0 = __ffma2_rn(s0, make_float2(D[0], D[1]), make_float2(acc[q][tg][0], acc[q][tg][1]));
                            const float2 r1 = __ffma2_rn(s1, make_float2(D[2], D[3]), make_float2(acc[q][tg][2], acc[q][tg][3]));
                            acc[q][tg][0] = r0.x; acc[q][tg][1] = r0.y;
                            acc[q][tg][2] = r1.x; acc[q][tg][3] = r1.y;
                        }
                    }
                }
            }
        }
        // this warp's reads of the stage are done
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (DOTS) continue;

        // park the group sums in partial slot ps ([group][token][row]) once the reducers are
        // done with the slot's previous chunk
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
            for (int tg = 0; tg < MT; ++tg)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = 16 * rt + gl + 8 * (e >> 1);
                    const int t = 8 * tg + 2 * c + (e & 1);
                    part[((size_t)g * TOK + t) * p.R + r] = acc[q][tg][e];
                }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[ps]);
    }
}

template <class F, int MT, bool DOTS>
cudaError_t launch_mt(const DeviceInfo &dev, Group grp, const int8_t *xq, const float *xd, int32_t *dots, int64_t m,
                      int64_t k, cudaStream_t stream, bool pdl)
{
    // 16-row tiles of the whole group
    int64_t tiles = 0;
    for (int i = 0; i < grp.count; ++i) tiles += (grp.n[i] + 15) / 16;
    // 16-row tiles per chunk: the fewest (waves of chunks over the SMs) x (rounds of items per
    // MMA warp), ties to fewer tiles per chunk (more SMs streaming)
    int rt_cap = 1;
    {
        const int g = (int)(k / 256), rt0 = (NW + g - 1) / g > 1 ? (NW + g - 1) / g : 1;
        int64_t best = -1;
        for (int rt = 1; rt <= rt0; ++rt) {
            const int64_t waves = ((tiles + rt - 1) / rt + dev.num_sms - 1) / dev.num_sms;
            const int64_t cost = waves * ((rt * g + NW - 1) / NW);
            if (best < 0 || cost < best) {
                best = cost;
                rt_cap = rt;
            }
        }
    }
    MPlan p = make_mplan(MT, k, dev.max_smem_optin, F::BLOCK_BYTES, rt_cap);
    if (!mplan_ok(p, MT)) return cudaErrorInvalidValue;
    if (DOTS && grp.count != 1) return cudaErrorInvalidValue;   // the export serves one matrix
    grp.first_chunk[0] = 0;
    for (int i = 0; i < grp.count; ++i) grp.first_chunk[i + 1] = grp.first_chunk[i] + (grp.n[i] + p.R - 1) / p.R;
    p.nchunks = grp.first_chunk[grp.count];
    auto kern = gemv_mma_kernel<F, MT, DOTS>;
    cudaError_t e = set_kernel_smem<gemv_mma_kernel<F, MT, DOTS>>(dev.device, p.smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = p.nchunks < dev.num_sms ? p.nchunks : dev.num_sms;
    // pdl: the previous kernel is this call's quantizer, which does not write the weights
    p.wait_weights = pdl ? 0 : 1;
    return launch_dependent(kern, (unsigned)grid, THREADS, p.smem, stream, grp, xq, xd, dots, (int)m, (int)k, p,
                            dev.status);
}

template <class F>
bool supported(const DeviceInfo &dev, int64_t m, int64_t k)
{
    // where this kernel is the faster one (both give the same bits)
    if (m < F::MIN_M || m > 16) return false;
    const int mt = m > 8 ? 2 : 1;
    return mplan_ok(make_mplan(mt, k, dev.max_smem_optin, F::BLOCK_BYTES), mt);
}

template <class F>
cudaError_t launch(const DeviceInfo &dev, const Group &grp, const int8_t *xq, const float *xd, int32_t *dots,
                   int64_t m, int64_t k, cudaStream_t stream, bool pdl)
{
    if (m > 8)
        return dots ? launch_mt<F, 2, true>(dev, grp, xq, xd, dots, m, k, stream, pdl)
                    : launch_mt<F, 2, false>(dev, grp, xq, xd, dots, m, k, stream, pdl);
    return dots ? launch_mt<F, 1, true>(dev, grp, xq, xd, dots, m, k, stream, pdl)
                : launch_mt<F, 1, false>(dev, grp, xq, xd, dots, m, k, stream, pdl);
}

Group group_of_one(const uint8_t *w, float *y, int64_t n)
{
    Group grp{};
    grp.count = 1;
    grp.w[0] = w;
    grp.y[0] = y;
    grp.n[0] = (int)n;
    return grp;
}

}  // namespace

bool gemv_mma_supported(const DeviceInfo &dev, int64_t m, int64_t k) { return supported<MQ8_0>(dev, m, k); }

cudaError_t launch_gemv_q8_0_mma(const DeviceInfo &dev, const uint8_t *w, const int8_t *xq, const float *xd,
                                 float *y, int32_t *dots, int64_t m, int64_t n, int64_t k, cudaStream_t stream,
                                 bool pdl)
{
    return launch<MQ8_0>(dev, group_of_one(w, y, n), xq, xd, dots, m, k, stream, pdl);
}

cudaError_t launch_gemv_q8_0_group_mma(const DeviceInfo &dev, const uint8_t *const *w, float *const *y,
                                       const int64_t *n, int count, const int8_t *xq, const float *xd,
                                       int64_t m, int64_t k, cudaStream_t stream)
{
    if (count < 1 || count > Q8ACT_GEMV_MAX_GROUP) return cudaErrorInvalidValue;
    Group grp{};
    grp.count = count;
    for (int i = 0; i < count; ++i) {
        grp.w[i] = w[i];
        grp.y[i] = y[i];
        grp.n[i] = (int)n[i];
    }
    return launch<MQ8_0>(dev, grp, xq, xd, nullptr, m, k, stream, false);
}

bool gemv_q4_0_mma_supported(const DeviceInfo &dev, int64_t m, int64_t k) { return supported<MQ4_0>(dev, m, k); }

cudaError_t launch_gemv_q4_0_mma(const DeviceInfo &dev, const uint8_t *w, const int8_t *xq, const float *xd,
                                 float *y, int32_t *dots, int64_t m, int64_t n, int64_t k, cudaStream_t stream)
{
    return launch<MQ4_0>(dev, group_of_one(w, y, n), xq, xd, dots, m, k, stream, false);
}

}  // namespace q8
