// gemv.cu -- Q8_0 x q8_1 GEMV for decode and speculative verify (m = 1..15): the "mmvq"
// regime of memra-engine 0.113.0 decode_kernel_census.rs (fn q8 -> qmatvec_mmvq_into); and
// the same kernel over Q4_0 weights (the GGUF 18-byte block of f16_ffi.rs).
//
// The weight stream (34 or 18 bytes per 32 weights) is read exactly once, so the kernel is
// bound by HBM bandwidth.  Design (persistent CTAs, two per SM):
//   * a producer warp streams "chunks" of R consecutive rows (contiguous in memory) into a
//     ring of shared-memory stages with cp.async.bulk, completing on mbarriers -- coalesced,
//     16-byte aligned, no per-thread address math;
//   * 128 consumer threads split each chunk into "units" of 8 blocks (272 = 17 x 16 or 144 = 9 x 16 bytes,
//     the period at which the blocks realign to 16 bytes); a unit is read with conflict-free
//     16-byte shared loads, its 8 blocks are dotted with the activation (8 dp4a per block
//     per token) and folded as acc += (d_w * d_a) * D;
//   * the activation (m x k int8 + scales) sits in shared memory for the whole kernel, padded
//     so that neighbouring units hit different banks;
//   * the per-row sum over units uses a fixed order -- a butterfly of warp shuffles when a
//     row's units are consecutive lanes of one warp, else a shared-memory pass -- so token
//     t's result is the same sequence of operations for every m (the pages' decode == verify
//     law, fp8_ffi.rs and f16_ffi.rs module docs).
#include "common.cuh"
#include "launch.h"

namespace q8 {
namespace {

constexpr int MAX_STAGES = 6;
constexpr int XG_WORDS = 68;   // per (token, group): 64 quant words + 4 pad
constexpr int XDG_WORDS = 12;  // per (token, group): 8 scales + 4 pad

// Block formats.  A unit is 8 blocks (272 bytes of Q8_0, 144 of Q4_0: multiples of 16).
// block(): the scale bits of block j of a unit and its 32 quants as signed bytes scaled by
// 2^SHIFT, ready for dp4a with the activation (the exact dot is the dp4a sum >> SHIFT).
struct GQ8_0 {
    static constexpr int BLOCK_BYTES = Q8_0_BYTES;
    static constexpr int UNIT_BYTES = GROUP_BYTES;
    static constexpr int UNIT_WORDS = UNIT_BYTES / 4;   // 68
    static constexpr int SHIFT = 0;
    static constexpr int CONSUMERS = 128;    // consumer threads per CTA
    static constexpr int CHUNK_UNITS = 128;  // units per chunk: one per consumer
    __device__ static void block(const uint32_t (&wv)[UNIT_WORDS], int j, uint32_t (&q)[8], uint32_t &dbits)
    {
        // Block j starts at byte 34j: even j at word 17(j/2) (scale in the low half, quants
        // straddle words), odd j with its scale in the high half of word 17(j/2)+8 and
        // word-aligned quants after it.
        if ((j & 1) == 0) {
            const int w0 = 17 * (j >> 1);
            dbits = wv[w0] & 0xffffu;
#pragma unroll
            for (int e = 0; e < 8; ++e) q[e] = __byte_perm(wv[w0 + e], wv[w0 + e + 1], 0x5432);
        } else {
            const int w1 = 17 * (j >> 1) + 8;
            dbits = wv[w1] >> 16;
#pragma unroll
            for (int e = 0; e < 8; ++e) q[e] = wv[w1 + 1 + e];
        }
    }
};

// Q4_0 (the GGUF 18-byte block): element i < 16 in the low nibble of quant byte i, element
// i + 16 in its high nibble, value nibble - 8.  Moving a nibble n to the top of its byte and
// flipping the sign bit gives the signed byte 16 (n - 8), so dp4a sums 16 D exactly.
struct GQ4_0 {
    static constexpr int BLOCK_BYTES = Q4_0_BYTES;
    static constexpr int UNIT_BYTES = Q4_GROUP_BYTES;
    static constexpr int UNIT_WORDS = UNIT_BYTES / 4;   // 36
    static constexpr int SHIFT = 4;
    static constexpr int CONSUMERS = 128;
    static constexpr int CHUNK_UNITS = 128;
    __device__ static void block(const uint32_t (&wv)[UNIT_WORDS], int j, uint32_t (&q)[8], uint32_t &dbits)
    {
        // Block j starts at byte 18j: even j at word 9(j/2) (scale in the low half, the 16
        // quant bytes straddle words), odd j with its scale in the high half of word
        // 9(j/2)+4 and word-aligned quant bytes after it.
        uint32_t b[4];
        if ((j & 1) == 0) {
            const int w0 = 9 * (j >> 1);
            dbits = wv[w0] & 0xffffu;
#pragma unroll
            for (int e = 0; e < 4; ++e) b[e] = __byte_perm(wv[w0 + e], wv[w0 + e + 1], 0x5432);
        } else {
            const int w1 = 9 * (j >> 1) + 4;
            dbits = wv[w1] >> 16;
#pragma unroll
            for (int e = 0; e < 4; ++e) b[e] = wv[w1 + 1 + e];
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            q[e] = ((b[e] << 4) & 0xF0F0F0F0u) ^ 0x80808080u;   // elements 4e .. 4e+3
            q[4 + e] = (b[e] & 0xF0F0F0F0u) ^ 0x80808080u;      // elements 16+4e .. 16+4e+3
        }
    }
};

struct Plan {
    int G;              // groups of 8 blocks per row (k / 256)
    int R;              // rows per chunk
    int U;              // units per chunk (R * G)
    int stages;
    int ctas_per_sm;    // resident CTAs per SM the shared-memory plan allows
    int warp_reduce;    // 1: a row's units are consecutive lanes of one warp (G divides 32)
    int wait_weights;   // 1: the producer waits for the stream's previous kernel before streaming
    uint32_t row_bytes;
    uint32_t chunk_bytes;
    int64_t nchunks;
    size_t off_x, off_xd, off_part, off_bar, smem;
};

Plan make_plan(int64_t m, int64_t n, int64_t k, size_t smem_cap, int r_cap, int block_bytes, int chunk_units)
{
    Plan p{};
    p.G = (int)(k / 256);
    p.R = p.G <= chunk_units ? chunk_units / p.G : 1;
    if (p.R > r_cap) p.R = r_cap;
    if ((int64_t)p.R > n) p.R = (int)n;
    p.U = p.R * p.G;
    p.row_bytes = (uint32_t)(k / QK * block_bytes);
    p.chunk_bytes = (uint32_t)p.R * p.row_bytes;
    p.nchunks = (n + p.R - 1) / p.R;
    const size_t x_bytes = (size_t)m * p.G * XG_WORDS * 4;
    const size_t xd_bytes = (size_t)m * p.G * XDG_WORDS * 4;
    const size_t part_bytes = 2 * (size_t)p.U * m * 4;
    const size_t fixed = x_bytes + xd_bytes + part_bytes + 2 * MAX_STAGES * 8 + 64;
    const size_t room = smem_cap > fixed ? smem_cap - fixed : 0;
    int64_t st = (int64_t)(room / p.chunk_bytes);
    if (st > MAX_STAGES) st = MAX_STAGES;
    p.stages = (int)st;
    p.off_x = (size_t)p.stages * p.chunk_bytes;            // multiple of 16
    p.off_xd = p.off_x + x_bytes;
    p.off_part = p.off_xd + xd_bytes;
    p.off_bar = (p.off_part + part_bytes + 7) & ~(size_t)7;
    p.smem = p.off_bar + 2 * MAX_STAGES * 8;
    p.ctas_per_sm = 1;
    p.warp_reduce = (p.G <= 32 && 32 % p.G == 0) ? 1 : 0;
    return p;
}

// Q4_0 at m = 1: four CTAs per SM with two 18.4 KB stages each in a quarter of the shared
// memory (its consumers do twice the work per streamed byte of Q8_0's and need the warps:
// 4096 -> 64448 26.0 -> 24.5 us against three CTAs, 33.1 us with two).  Otherwise three CTAs per
// SM when rings of at least 3 stages fit in a third of the shared memory, else two when 3-stage
// rings fit in half, else one CTA with up to 6 stages.
// When a large activation leaves room for fewer than 2 full-size stages, the chunk shrinks
// (fewer rows per chunk) until two fit.
template <class F>
Plan choose_plan(int64_t m, int64_t n, int64_t k, size_t smem_optin)
{
    const size_t third = 74 * 1024, quarter = 56 * 1024;
    if (m == 1 && F::BLOCK_BYTES == Q4_0_BYTES) {
        Plan p4 = make_plan(m, n, k, quarter < smem_optin ? quarter : smem_optin, F::CHUNK_UNITS, F::BLOCK_BYTES,
                            F::CHUNK_UNITS);
        if (p4.stages >= 2) {
            p4.ctas_per_sm = 4;
            return p4;
        }
    }
    Plan p = make_plan(m, n, k, third < smem_optin ? third : smem_optin, F::CHUNK_UNITS, F::BLOCK_BYTES, F::CHUNK_UNITS);
    if (p.stages >= 3) {
        p.ctas_per_sm = 3;
        return p;
    }
    const size_t half = 113 * 1024;
    p = make_plan(m, n, k, half < smem_optin ? half : smem_optin, F::CHUNK_UNITS, F::BLOCK_BYTES, F::CHUNK_UNITS);
    if (p.stages >= 3) {
        p.ctas_per_sm = 2;
        return p;
    }
    p = make_plan(m, n, k, smem_optin, F::CHUNK_UNITS, F::BLOCK_BYTES, F::CHUNK_UNITS);
    for (int r_cap = p.R / 2; p.stages < 2 && r_cap >= 1; r_cap /= 2)
        p = make_plan(m, n, k, smem_optin, r_cap, F::BLOCK_BYTES, F::CHUNK_UNITS);
    return p;
}

template <class F, int M, bool DOTS>
__global__ void __launch_bounds__(F::CONSUMERS + 32, 2)
    gemv_kernel(const __grid_constant__ Group grp, const int8_t *__restrict__ xq,
                     const float *__restrict__ xd, int32_t *__restrict__ dots, int k, Plan p,
                     int *status)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    uint32_t *xs = reinterpret_cast<uint32_t *>(smem + p.off_x);
    float *xds = reinterpret_cast<float *>(smem + p.off_xd);
    float *part = reinterpret_cast<float *>(smem + p.off_part);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    uint64_t *empty = full + MAX_STAGES;

    constexpr int CONSUMERS = F::CONSUMERS;
    const int tid = threadIdx.x;
    const int G = p.G;
    const int nb = k / QK;

    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CONSUMERS / 32);
        }
        fence_mbar_init();
    }
    __syncthreads();
    // The producer starts streaming weights right away; the consumers meanwhile load the
    // activation cache -- quants [token][group][68 words], scales [token][group][12 words] --
    // and meet at a named barrier before their first chunk.
    if (tid < CONSUMERS) {
        // The activation may come from the kernel just before this one in the stream (this
        // kernel is launched as its programmatic dependent); in a fused call that is the
        // call's own quantizer, and the weight stream does not wait for it.
        griddep_wait();
        griddep_launch_dependents();
        for (int idx = tid; idx < M * G * 16; idx += CONSUMERS) {
            const int t = idx / (G * 16), rem = idx - t * G * 16, g = rem >> 4, c = rem & 15;
            const uint4 v = *reinterpret_cast<const uint4 *>(xq + (int64_t)t * k + g * 256 + c * 16);
            *reinterpret_cast<uint4 *>(xs + (t * G + g) * XG_WORDS + c * 4) = v;
        }
        for (int idx = tid; idx < M * G * 2; idx += CONSUMERS) {
            const int t = idx / (G * 2), rem = idx - t * G * 2, g = rem >> 1, c = rem & 1;
            const float4 v = *reinterpret_cast<const float4 *>(xd + (int64_t)t * nb + g * 8 + c * 4);
            *reinterpret_cast<float4 *>(xds + (t * G + g) * XDG_WORDS + c * 4) = v;
        }
        named_bar_sync(2, CONSUMERS);
    }

    const int64_t my_chunks =
        blockIdx.x < p.nchunks ? (p.nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    if (tid >= CONSUMERS) {
        // ---------------- producer warp: one lane issues the bulk copies ----------------
        if (tid == CONSUMERS) {
            const uint64_t policy = l2_policy_evict_first();   // the weights are read once
            if (p.wait_weights) griddep_wait();
            int64_t issued = 0;
            for (int64_t i = 0; i < my_chunks; ++i) {
                const int s = (int)(i % p.stages);
                const uint32_t ph = (uint32_t)((i / p.stages) & 1);
                if (!mbar_wait(&empty[s], ph ^ 1, status)) break;
                const ChunkRef cr = chunk_ref(grp, blockIdx.x + i * gridDim.x, p.R);
                const uint32_t bytes = (uint32_t)cr.rows * p.row_bytes;
                mbar_arrive_expect_tx(&full[s], bytes);
                bulk_g2s_hint(smem + (size_t)s * p.chunk_bytes, cr.w + cr.row0 * p.row_bytes, bytes, &full[s],
                              policy);
                ++issued;
            }
            // Do not leave while copies into this CTA's shared memory may be in flight.
            for (int64_t i = issued - p.stages < 0 ? 0 : issued - p.stages; i < issued; ++i)
                mbar_wait_drain(&full[i % p.stages], (uint32_t)((i / p.stages) & 1), status);
        }
        return;
    }

    // -------------------------------- consumers --------------------------------
    for (int64_t i = 0; i < my_chunks; ++i) {
        const int s = (int)(i % p.stages);
        const uint32_t ph = (uint32_t)((i / p.stages) & 1);
        const bool ok = mbar_wait(&full[s], ph, status);
        // Leave together: the whole CTA when rows are reduced through shared memory, the
        // whole warp when they are reduced with shuffles.
        if (p.warp_reduce ? __any_sync(0xffffffffu, !ok) : bar_red_or(1, CONSUMERS, !ok)) break;

        const ChunkRef cr = chunk_ref(grp, blockIdx.x + i * gridDim.x, p.R);
        const int64_t row0 = cr.row0;
        const int rows = cr.rows;
        const int n = cr.n;
        float *__restrict__ y = cr.y;
        const uint8_t *sbase = smem + (size_t)s * p.chunk_bytes;
        float *pbuf = part + (size_t)(i & 1) * p.U * M;

        // In shuffle mode every lane of a warp takes part (lanes past the last unit act as
        // empty units of rows beyond `rows`).
        const int ulimit = p.warp_reduce ? (p.U + 31) / 32 * 32 : p.U;
        for (int u = tid; u < ulimit; u += CONSUMERS) {
            const int row = u / G;
            const int g = u - row * G;
            float acc[M];
#pragma unroll
            for (int t = 0; t < M; ++t) acc[t] = 0.0f;
            if (row < rows) {
                const uint4 *src = reinterpret_cast<const uint4 *>(sbase + (size_t)row * p.row_bytes +
                                                                   g * F::UNIT_BYTES);
                uint32_t wv[F::UNIT_WORDS];
#pragma unroll
                for (int c = 0; c < F::UNIT_WORDS / 4; ++c) {
                    const uint4 v = src[c];
                    wv[4 * c + 0] = v.x;
                    wv[4 * c + 1] = v.y;
                    wv[4 * c + 2] = v.z;
                    wv[4 * c + 3] = v.w;
                }
                const uint32_t *xg = xs + g * XG_WORDS;
                const float *xdg = xds + g * XDG_WORDS;
#pragma unroll
                for (int j = 0; j < GROUP_BLOCKS; ++j) {
                    uint32_t q[8];
                    uint32_t dbits;
                    F::block(wv, j, q, dbits);
                    const float dw = half_bits_to_float(dbits);
#pragma unroll
                    for (int t = 0; t < M; ++t) {
                        const uint4 *xv = reinterpret_cast<const uint4 *>(xg + t * G * XG_WORDS + j * 8);
                        const uint4 a = xv[0], b = xv[1];
                        // Two independent chains of 4 (integer sums: exact in any order).
                        int D0 = dp4a(q[0], a.x, 0);
                        int D1 = dp4a(q[4], b.x, 0);
                        D0 = dp4a(q[1], a.y, D0);
                        D1 = dp4a(q[5], b.y, D1);
                        D0 = dp4a(q[2], a.z, D0);
                        D1 = dp4a(q[6], b.z, D1);
                        D0 = dp4a(q[3], a.w, D0);
                        D1 = dp4a(q[7], b.w, D1);
                        const int D = (D0 + D1) >> F::SHIFT;   // exact: a multiple of 2^SHIFT
                        if (DOTS) {
                            dots[((int64_t)t * n + row0 + row) * nb + g * GROUP_BLOCKS + j] = D;
                        } else {
                            const float da = xdg[t * G * XDG_WORDS + j];
                            acc[t] = __fmaf_rn(__fmul_rn(dw, da), __int2float_rn(D), acc[t]);
                        }
                    }
                }
            }
            if (DOTS) continue;
            if (p.warp_reduce) {
                // The row's G units sit in G consecutive lanes (G divides 32): butterfly sum,
                // the same fixed sequence of additions for every m.
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    if (o >= G) break;
#pragma unroll
                    for (int t = 0; t < M; ++t) acc[t] = __fadd_rn(acc[t], __shfl_xor_sync(0xffffffffu, acc[t], o));
                }
                if (g == 0 && row < rows) {
#pragma unroll
                    for (int t = 0; t < M; ++t) y[(int64_t)t * n + row0 + row] = acc[t];
                }
            } else {
#pragma unroll
                for (int t = 0; t < M; ++t) pbuf[u * M + t] = acc[t];
            }
        }
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage's bytes
        if (DOTS || p.warp_reduce) continue;
        named_bar_sync(1, CONSUMERS);
        for (int idx = tid; idx < rows * M; idx += CONSUMERS) {
            const int t = idx / rows, r = idx - t * rows;
            const float *pr = pbuf + (size_t)r * G * M + t;
            float sum = pr[0];
            for (int g = 1; g < G; ++g) sum = __fadd_rn(sum, pr[g * M]);
            y[(int64_t)t * n + row0 + r] = sum;
        }
    }
}

template <class F, int M, bool DOTS>
cudaError_t launch_m(const DeviceInfo &dev, Group grp, const int8_t *xq, const float *xd,
                     int32_t *dots, int64_t k, bool pdl, cudaStream_t stream)
{
    int64_t nmax = 0;
    for (int i = 0; i < grp.count; ++i) nmax = grp.n[i] > nmax ? grp.n[i] : nmax;
    Plan p = choose_plan<F>(M, nmax, k, dev.max_smem_optin);
    if (p.stages < 2) return cudaErrorInvalidValue;
    grp.first_chunk[0] = 0;
    for (int i = 0; i < grp.count; ++i) grp.first_chunk[i + 1] = grp.first_chunk[i] + (grp.n[i] + p.R - 1) / p.R;
    p.nchunks = grp.first_chunk[grp.count];
    auto kern = gemv_kernel<F, M, DOTS>;
    cudaError_t e = set_kernel_smem<gemv_kernel<F, M, DOTS>>(dev.device, p.smem);
    if (e != cudaSuccess) return e;
    const int64_t slots = (int64_t)dev.num_sms * p.ctas_per_sm;
    int64_t grid = p.nchunks < slots ? p.nchunks : slots;
    // fused: the previous kernel is this call's quantizer, which does not write the weights
    p.wait_weights = pdl ? 0 : 1;
    return launch_dependent(kern, (unsigned)grid, F::CONSUMERS + 32, p.smem, stream, grp, xq, xd, dots, (int)k, p,
                            dev.status);
}

template <class F, bool DOTS>
cudaError_t dispatch(const DeviceInfo &dev, const Group &grp, const int8_t *xq, const float *xd,
                     int32_t *dots, int64_t m, int64_t k, cudaStream_t stream, bool pdl = false)
{
    switch (m) {
    case 1: return launch_m<F, 1, DOTS>(dev, grp, xq, xd, dots, k, pdl, stream);
    case 2: return launch_m<F, 2, DOTS>(dev, grp, xq, xd, dots, k, pdl, stream);
    case 3: return launch_m<F, 3, DOTS>(dev, grp, xq, xd, dots, k, pdl, stream);
    case 4: return launch_m<F, 4, DOTS>(dev, grp, xq, xd, dots, k, pdl, stream);
    case 5: return launch_m<F, 5, DOTS>(dev, grp, xq, xd, dots, k, pdl, stream);
    case 6: return launch_m<F, 6, DOTS>(dev, grp, xq, xd, dots, k, pdl, stream);
    case 7: return launch_m<F, 7, DOTS>(dev, grp, xq, xd, dots, k, pdl, stream);
    case 8: return launch_m<F, 8, DOTS>(dev, grp, xq, xd, dots, k, pdl, stream);
    case 9: return launch_m<F, 9, DOTS>(dev, grp, xq, xd, dots, k, pdl, stream);
    case 10: return launch_m<F, 10, DOTS>(dev, grp, xq, xd, dots, k, pdl, stream);
    case 11: return launch_m<F, 11, DOTS>(dev, grp, xq, xd, dots, k, pdl, stream);
    case 12: return launch_m<F, 12, DOTS>(dev, grp, xq, xd, dots, k, pdl, stream);
    case 13: return launch_m<F, 13, DOTS>(dev, grp, xq, xd, dots, k, pdl, stream);
    case 14: return launch_m<F, 14, DOTS>(dev, grp, xq, xd, dots, k, pdl, stream);
    case 15: return launch_m<F, 15, DOTS>(dev, grp, xq, xd, dots, k, pdl, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool gemv_supported(const DeviceInfo &dev, int64_t m, int64_t k)
{
    if (m < 1 || m > Q8ACT_GEMV_MAX_M) return false;
    return choose_plan<GQ8_0>(m, 1 << 20, k, dev.max_smem_optin).stages >= 2;
}

cudaError_t launch_gemv_q8_0(const DeviceInfo &dev, const uint8_t *w, const int8_t *xq,
                             const float *xd, float *y, int32_t *dots, int64_t m, int64_t n,
                             int64_t k, cudaStream_t stream, bool pdl)
{
    Group grp{};
    grp.count = 1;
    grp.w[0] = w;
    grp.y[0] = y;
    grp.n[0] = (int)n;
    if (dots) return dispatch<GQ8_0, true>(dev, grp, xq, xd, dots, m, k, stream, pdl);
    return dispatch<GQ8_0, false>(dev, grp, xq, xd, dots, m, k, stream, pdl);
}

bool gemv_q4_0_supported(const DeviceInfo &dev, int64_t m, int64_t k)
{
    if (m < 1 || m > Q8ACT_GEMV_MAX_M) return false;
    return choose_plan<GQ4_0>(m, 1 << 20, k, dev.max_smem_optin).stages >= 2;
}

cudaError_t launch_gemv_q4_0(const DeviceInfo &dev, const uint8_t *w, const int8_t *xq,
                             const float *xd, float *y, int32_t *dots, int64_t m, int64_t n,
                             int64_t k, cudaStream_t stream)
{
    Group grp{};
    grp.count = 1;
    grp.w[0] = w;
    grp.y[0] = y;
    grp.n[0] = (int)n;
    if (dots) return dispatch<GQ4_0, true>(dev, grp, xq, xd, dots, m, k, stream);
    return dispatch<GQ4_0, false>(dev, grp, xq, xd, dots, m, k, stream);
}

cudaError_t launch_gemv_q8_0_group(const DeviceInfo &dev, const uint8_t *const *w, float *const *y,
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
    return dispatch<GQ8_0, false>(dev, grp, xq, xd, nullptr, m, k, stream);
}

}  // namespace q8
