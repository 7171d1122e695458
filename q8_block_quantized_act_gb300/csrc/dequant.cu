// dequant.cu -- Q8_0 and Q4_0 -> row-major binary16 (memra-engine 0.81.0 f16_ffi.rs,
// memra_q8_0_dequant_f16 and memra_q4_0_dequant_f16: w16[r][32b+i] = fp16(d_w * q)), and the
// load-time repack of Q8_0 for the tensor-core GEMM (the same stream; it stores the exact
// binary16 quants wq16[r][32b+i] = q and the scale plane wdt[b][r] = f32(d_w) instead of
// their rounded product).
//
// HBM-bound: 34 (Q8_0) or 18 (Q4_0) bytes in and 64 bytes out per block.  Persistent CTAs
// stream chunks of whole rows (contiguous, 16-byte aligned) into a shared-memory ring with
// cp.async.bulk.  A warp converts one unit of 8 blocks (256 values: 272 or 144 bytes, both
// multiples of 16) at a time: lane j builds the 16-byte output piece j (8 values of block
// j/4) from shared memory and the warp stores the unit's 512 output bytes with one fully
// coalesced 16-byte-per-lane store.
//
// Arithmetic: the quants become binary16 exactly (|q| <= 127), and the binary16 multiplier
// rounds the exact product d_w * q once, to nearest even -- the same value as rounding the
// (exact) f32 product, which is how the formats' dequant is defined.
#include "common.cuh"
#include "launch.h"

namespace q8 {
namespace {

constexpr int CONV_WARPS = 16;
constexpr int THREADS = (CONV_WARPS + 1) * 32;   // + one bulk-copy producer warp
constexpr int MAX_STAGES = 6;
constexpr size_t TWO_PER_SM_SMEM = 113 * 1024;   // two CTAs per SM when 3 stages fit in this
constexpr int TARGET_CHUNK = 17408;               // bytes of raw rows per stage (<= 64 units)

struct Plan {
    int G;               // units (groups of 8 blocks) per row
    int R;               // rows per chunk
    int stages;
    uint32_t row_bytes;
    uint32_t chunk_bytes;
    int64_t nchunks;
    size_t off_bar, smem;
};

Plan make_plan(int64_t n, int64_t k, int block_bytes, size_t smem_cap)
{
    Plan p{};
    p.G = (int)(k / 256);
    p.row_bytes = (uint32_t)(k / QK * block_bytes);
    p.R = (int)(TARGET_CHUNK / p.row_bytes);
    if (p.R < 1) p.R = 1;
    if ((int64_t)p.R > n) p.R = (int)n;
    p.chunk_bytes = (uint32_t)p.R * p.row_bytes;
    p.nchunks = (n + p.R - 1) / p.R;
    const size_t room = smem_cap > 2 * MAX_STAGES * 8 + 64 ? smem_cap - 2 * MAX_STAGES * 8 - 64 : 0;
    int64_t st = (int64_t)(room / p.chunk_bytes);
    p.stages = (int)(st > MAX_STAGES ? MAX_STAGES : st);
    p.off_bar = (size_t)p.stages * p.chunk_bytes;
    p.smem = p.off_bar + 2 * MAX_STAGES * 8;
    return p;
}

__device__ __forceinline__ uint32_t lds_u16(const uint8_t *p)
{
    return *reinterpret_cast<const uint16_t *>(p);
}

// Four signed bytes (packed in a 32-bit word) -> two half2 with the same integer values.
// (b ^ 0x80) is q + 128 in 0..255; the binary16 pattern 0x6400 | u is 1024 + u, so
// subtracting 1152 leaves q exactly.
__device__ __forceinline__ void bytes_to_half2x2(uint32_t q4, __half2 &lo, __half2 &hi)
{
    const uint32_t u = q4 ^ 0x80808080u;
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x5140);  // bytes 0,1 -> 0x64uu pairs
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x5342);  // bytes 2,3
    const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));  // 1152
    lo = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);
    hi = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
}

// Four 4-bit values (one per byte, 0..15) -> two half2 holding value - 8 exactly: the
// binary16 pattern 0x6400 | v is 1024 + v, and subtracting 1032 leaves v - 8.
__device__ __forceinline__ void nibbles_to_half2x2(uint32_t n4, __half2 &lo, __half2 &hi)
{
    const uint32_t a = __byte_perm(n4, 0x64646464u, 0x5140);
    const uint32_t b = __byte_perm(n4, 0x64646464u, 0x5342);
    const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6408));  // 1032
    lo = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);
    hi = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
}

// Block formats.  load(): the raw words of lane (jb, sub)'s piece -- values 8 sub .. 8 sub + 7
// of block jb of a unit; convert(): those 8 values as exact binary16 integers.
struct FmtQ8_0 {
    static constexpr int BLOCK_BYTES = Q8_0_BYTES;
    static constexpr int UNIT_BYTES = GROUP_BYTES;
    __device__ static void load(const uint8_t *unit, int jb, int sub, uint32_t &dbits, uint32_t &w0, uint32_t &w1)
    {
        const uint8_t *blk = unit + jb * Q8_0_BYTES;
        const uint8_t *qp = blk + 2 + 8 * sub;
        dbits = lds_u16(blk);
        w0 = lds_u16(qp) | (lds_u16(qp + 2) << 16);
        w1 = lds_u16(qp + 4) | (lds_u16(qp + 6) << 16);
    }
    __device__ static void convert(uint32_t w0, uint32_t w1, int, __half2 (&h)[4])
    {
        bytes_to_half2x2(w0, h[0], h[1]);
        bytes_to_half2x2(w1, h[2], h[3]);
    }
};

// Q4_0 (the GGUF 18-byte block): element i < 16 in the low nibble of quant byte i, element
// i + 16 in its high nibble, value d * (nibble - 8).  Pieces 0 and 1 are the low nibbles of
// bytes 0-7 and 8-15, pieces 2 and 3 their high nibbles.
struct FmtQ4_0 {
    static constexpr int BLOCK_BYTES = Q4_0_BYTES;
    static constexpr int UNIT_BYTES = Q4_GROUP_BYTES;
    __device__ static void load(const uint8_t *unit, int jb, int sub, uint32_t &dbits, uint32_t &w0, uint32_t &w1)
    {
        const uint8_t *blk = unit + jb * Q4_0_BYTES;
        const uint8_t *qp = blk + 2 + 8 * (sub & 1);
        dbits = lds_u16(blk);
        w0 = lds_u16(qp) | (lds_u16(qp + 2) << 16);
        w1 = lds_u16(qp + 4) | (lds_u16(qp + 6) << 16);
    }
    __device__ static void convert(uint32_t w0, uint32_t w1, int sub, __half2 (&h)[4])
    {
        const int sh = (sub & 2) ? 4 : 0;
        nibbles_to_half2x2((w0 >> sh) & 0x0F0F0F0Fu, h[0], h[1]);
        nibbles_to_half2x2((w1 >> sh) & 0x0F0F0F0Fu, h[2], h[3]);
    }
};

// REPACK (Q8_0 only): store the exact quants and the transposed f32 scale plane instead of
// the rounded products.
template <class F, bool REPACK>
__global__ void __launch_bounds__(THREADS, 2)
    dequant_f16_kernel(const uint8_t *__restrict__ w, uint4 *__restrict__ out,
                       float *__restrict__ wdt, int64_t ldn, int n, int k, Plan p, int *status)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    uint64_t *empty = full + MAX_STAGES;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], CONV_WARPS);
        }
        fence_mbar_init();
    }
    __syncthreads();
    // launched as a programmatic dependent of the stream's previous kernel
    griddep_enter();

    const int64_t my_chunks =
        blockIdx.x < p.nchunks ? (p.nchunks - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    if (warp == CONV_WARPS) {
        if (lane == 0) {
            const uint64_t policy = l2_policy_evict_first();   // the weights are read once
            int64_t issued = 0;
            for (int64_t i = 0; i < my_chunks; ++i) {
                const int s = (int)(i % p.stages);
                if (!mbar_wait(&empty[s], (uint32_t)(((i / p.stages) & 1) ^ 1), status)) break;
                const int64_t row0 = (blockIdx.x + i * gridDim.x) * p.R;
                const int64_t rows = (n - row0) < p.R ? (n - row0) : p.R;
                const uint32_t bytes = (uint32_t)rows * p.row_bytes;
                mbar_arrive_expect_tx(&full[s], bytes);
                bulk_g2s_hint(smem + (size_t)s * p.chunk_bytes, w + row0 * p.row_bytes, bytes, &full[s],
                              policy);
                ++issued;
            }
            for (int64_t i = issued - p.stages < 0 ? 0 : issued - p.stages; i < issued; ++i)
                mbar_wait_drain(&full[i % p.stages], (uint32_t)((i / p.stages) & 1), status);
        }
        return;
    }

    const int jb = lane >> 2;           // block within the unit
    const int sub = lane & 3;           // 8-value piece within the block
    for (int64_t i = 0; i < my_chunks; ++i) {
        const int s = (int)(i % p.stages);
        const bool ok = mbar_wait(&full[s], (uint32_t)((i / p.stages) & 1), status);
        if (__any_sync(0xffffffffu, !ok)) break;
        const int64_t row0 = (blockIdx.x + i * gridDim.x) * p.R;
        const int rows = (int)((n - row0) < p.R ? (n - row0) : p.R);
        const uint8_t *sbase = smem + (size_t)s * p.chunk_bytes;
        const int units = rows * p.G;
        // unit u (row u / G, group u % G of the chunk) starts at element row0 * k + 256 u of
        // the output, since k = 256 G
        uint4 *outc = out + row0 * (int64_t)(k / 8) + lane;
        // Four units per warp step: their shared-memory reads are issued together.
        constexpr int UNR = 4;
        for (int u0 = warp; u0 < units; u0 += UNR * CONV_WARPS) {
            uint32_t dbits[UNR], q01[UNR], q23[UNR];
#pragma unroll
            for (int e = 0; e < UNR; ++e) {
                const int u = u0 + e * CONV_WARPS;
                const int uu = u < units ? u : u0;   // an in-range unit; its result is not stored
                F::load(sbase + (size_t)uu * F::UNIT_BYTES, jb, sub, dbits[e], q01[e], q23[e]);
            }
#pragma unroll
            for (int e = 0; e < UNR; ++e) {
                const int u = u0 + e * CONV_WARPS;
                if (u >= units) break;
                const __half2 d2 = __half2half2(__ushort_as_half((unsigned short)dbits[e]));
                __half2 h[4];
                F::convert(q01[e], q23[e], sub, h);
                uint4 o;
                uint32_t *ow = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __half2 prod = REPACK ? h[j] : __hmul2_rn(h[j], d2);
                    ow[j] = *reinterpret_cast<const uint32_t *>(&prod);
                }
                if (REPACK && sub == 0) {
                    const int row = u / p.G, g = u - row * p.G;
                    wdt[(int64_t)(g * GROUP_BLOCKS + jb) * ldn + row0 + row] = half_bits_to_float(dbits[e]);
                }
                // 256 outputs of the unit = 32 pieces of 16 bytes: piece `lane`.
                __stcs(outc + 32 * u, o);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

template <class F, bool REPACK>
cudaError_t launch_stream(const DeviceInfo &dev, const uint8_t *w, uint16_t *w16, float *wdt,
                          int64_t ldn, int64_t n, int64_t k, cudaStream_t stream)
{
    Plan p = make_plan(n, k, F::BLOCK_BYTES,
                       TWO_PER_SM_SMEM < dev.max_smem_optin ? TWO_PER_SM_SMEM : dev.max_smem_optin);
    int per_sm = 2;
    if (p.stages < 3) {
        p = make_plan(n, k, F::BLOCK_BYTES, dev.max_smem_optin);
        per_sm = 1;
    }
    if (p.stages < 2) return cudaErrorInvalidValue;
    auto kern = dequant_f16_kernel<F, REPACK>;
    cudaError_t e = set_kernel_smem<dequant_f16_kernel<F, REPACK>>(dev.device, p.smem);
    if (e != cudaSuccess) return e;
    const int64_t slots = (int64_t)dev.num_sms * per_sm;
    const int64_t grid = p.nchunks < slots ? p.nchunks : slots;
    return launch_dependent(kern, (unsigned)grid, THREADS, p.smem, stream, w, reinterpret_cast<uint4 *>(w16), wdt,
                            ldn, (int)n, (int)k, p, dev.status);
}

}  // namespace

cudaError_t launch_dequant_q8_0_f16(const DeviceInfo &dev, const uint8_t *w, uint16_t *w16,
                                    int64_t n, int64_t k, cudaStream_t stream)
{
    return launch_stream<FmtQ8_0, false>(dev, w, w16, nullptr, 0, n, k, stream);
}

cudaError_t launch_dequant_q4_0_f16(const DeviceInfo &dev, const uint8_t *w, uint16_t *w16,
                                    int64_t n, int64_t k, cudaStream_t stream)
{
    return launch_stream<FmtQ4_0, false>(dev, w, w16, nullptr, 0, n, k, stream);
}

cudaError_t launch_repack_q8_0(const DeviceInfo &dev, const uint8_t *w, uint16_t *wq16, float *wdt,
                               int64_t ldn, int64_t n, int64_t k, cudaStream_t stream)
{
    return launch_stream<FmtQ8_0, true>(dev, w, wq16, wdt, ldn, n, k, stream);
}

}  // namespace q8
