// gemm.cu -- Q8_0 x q8_1 GEMM for prefill (the "MMQ" regime: m >= 16 in the pages'
// dispatch, memra-engine 0.70.0 fp8_ffi.rs module doc), on the sm_103a tensor cores.
//
//   y[t][r] = sum_b d_w[r][b] * d_a[t][b] * D[t][r][b],  D = exact int32 32-wide block dot.
//
// sm_103a has no int8 tcgen05 MMA (ptxas rejects .kind::i8 for this target), so the exact
// integer dot runs on the f16 pipe: every quant |q| <= 127 is an exact binary16 value, every
// product |wq * xq| <= 16129 is exact in the f32 accumulator, and so is every partial sum of
// a 32-wide block (|D| <= 516128 < 2^24).  Each block gets a fresh accumulator in tensor
// memory (two K=16 MMAs), and fold warps apply the block's scales on the CUDA cores -- the
// per-32 fold of the pages' MMQ floor (accprobe_bench.rs module doc), scheduled so that the
// tensor pipe runs ahead into other accumulator buffers while a block is being folded.
//
// Tile: 128 weight rows (MMA M, TMEM lanes) x 128 tokens (MMA N, TMEM columns), full k.
// Warp roles, raw Q8_0 weights (640 threads, 20 warps: a multiple of 4, so registers are not
// rounded away):
//   warps 0-1   converters: raw Q8_0 rows (TMA, 272-byte groups) -> binary16 A tiles in the
//               128-byte-swizzled K-major layout + f32 weight scales (two rows per thread)
//   warps 2-17  fold: each owns 32 TMEM lanes (its warp index mod 4) x 32 columns;
//               tcgen05.ld (16x256b) of a block's D, acc += (d_w * d_a) * D in packed f32x2
//   warp 18     producer: TMA of activation tiles, activation scales and raw weight groups
//   warp 19     TMEM allocator + single-thread MMA issuer
// Repacked weights (608 threads): no converters; warps 0-15 fold, 16 producer (TMA of both
// operand tiles and both scale vectors), 17 allocator + issuer of even chunks, 18 issuer of
// odd chunks; six operand stages instead of four.
#include "common.cuh"
#include "launch.h"

namespace q8 {
namespace {

constexpr int BM = 128;            // weight rows per tile
constexpr int KC = 64;             // k per chunk (one 128-byte swizzle row of binary16)
constexpr int CHUNKS_PER_GROUP = 4;  // a 256-wide raw weight group feeds 4 chunks

constexpr int MAX_STAGES = 6;      // k chunks in flight: activation tile + weight tile
constexpr int RAW_STAGES = 2;
constexpr int SC_STAGES = 8;
constexpr int D_PAIRS = 2;         // TMEM accumulator buffers, handed over in pairs (one chunk)
constexpr int A_TILE_BYTES = BM * KC * 2;          // 16384
constexpr int RAW_TILE_BYTES = BM * GROUP_BYTES;   // 34816
constexpr int NUM_BARS = 2 * (MAX_STAGES + RAW_STAGES + SC_STAGES + D_PAIRS) + 1;
constexpr int FOLD_COLS = 32;                      // columns per fold warp
constexpr int RP_BN = 128;                         // tokens per tile of the repacked GEMM

// Tile shapes.  128 tokens per tile, one CTA per SM: with 2 converter warps for raw Q8_0
// input, without them for repacked weights; 16 fold warps.  Narrower tiles (64 tokens, two CTAs
// per SM, 8 fold warps) are expressible but measured slower: half the work per MMA instruction
// and twice the weight-tile traffic outweigh the overlap of the two CTAs' folds.
template <int BN_, bool CONV>
struct Cfg {
    static constexpr int BN = BN_;                               // tokens per tile
    // Operand stages: the raw path's shared memory also holds the raw weight groups; the
    // repacked path spends it on a deeper ring, which two MMA issuers need to stay fed.
    static constexpr int STAGES = CONV ? 4 : 6;
    static_assert(STAGES <= MAX_STAGES && STAGES % D_PAIRS == 0,
                  "a stage must always belong to the same accumulator pair");
    static constexpr int TMEM_COLS = 2 * D_PAIRS * BN;           // four accumulator buffers
    static constexpr int ACT_TILE_BYTES = BN * KC * 2;
    static constexpr int SC_SLOT_BYTES = 2 * BN * 4 + 2 * BM * 4;  // act scales [2][BN], weight scales [2][BM]
    static constexpr int RAW_ST = CONV ? RAW_STAGES : 0;
    static constexpr int OFF_ACT = 0;
    static constexpr int OFF_A = OFF_ACT + STAGES * ACT_TILE_BYTES;
    static constexpr int OFF_RAW = OFF_A + STAGES * A_TILE_BYTES;
    static constexpr int OFF_SC = OFF_RAW + RAW_ST * RAW_TILE_BYTES;
    static constexpr int OFF_BAR = OFF_SC + SC_STAGES * SC_SLOT_BYTES;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;   // + slack for 1024-byte base alignment
    static constexpr int NUM_CONV_WARPS = CONV ? 2 : 0;
    static constexpr int NUM_FOLD_WARPS = 4 * BN / FOLD_COLS;
    static constexpr int PRODUCER_WARP = NUM_CONV_WARPS + NUM_FOLD_WARPS;
    static constexpr int MMA_WARP = PRODUCER_WARP + 1;          // TMEM allocator, issues even chunks
    // One MMA issuer per accumulator pair; with converter warps a second issuer would push the
    // CTA to 21 warps and the register budget below 96.
    static constexpr int NUM_MMA_WARPS = CONV ? 1 : D_PAIRS;
    static constexpr int THREADS = (MMA_WARP + NUM_MMA_WARPS) * 32;
    static constexpr int CTAS_PER_SM = BN == 128 ? 1 : 2;
    // Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A and B binary16 (bits 7-9,
    // 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
    static constexpr uint32_t IDESC = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
    static_assert(OFF_A % 1024 == 0 && OFF_RAW % 1024 == 0 && OFF_SC % 128 == 0, "alignment");
};

// Shared-memory matrix descriptor for a K-major operand stored in 128-byte swizzled rows
// (8-row atoms of 1024 bytes): start address >> 4 (bits 0-13), leading byte offset
// (unused for this layout, bits 16-29), stride byte offset = 1024 >> 4 (bits 32-45),
// descriptor version 1 (bits 46-47), swizzle mode 2 = 128-byte (bits 61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
        ::"r"(smem_u32(bar))
        : "memory");
}

// 16 lanes x 256 bits, repeated 4 times along the columns (16 registers), asynchronous:
// the registers are valid only after tc_wait_ld_bind16.
__device__ __forceinline__ void tc_ld_16x256b_x4_async(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

template <bool WAIT>
__device__ __forceinline__ void tc_wait_ld_bind16(uint32_t (&r)[16])
{
    if (WAIT) asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// Packed f32x2 arithmetic (two f32 lanes per instruction, each rounded to nearest even
// exactly like the scalar mul.rn / fma.rn), through the compiler's builtins so that the
// operand pairs are allocated as register pairs.
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// Four signed bytes -> two half2 holding the same integers (exact).
__device__ __forceinline__ uint2 bytes_to_f16x4(uint32_t q4)
{
    const uint32_t u = q4 ^ 0x80808080u;                   // q + 128 in 0..255
    const uint32_t a = __byte_perm(u, 0x64646464u, 0x5140); // 0x64uu = 1024 + u
    const uint32_t b = __byte_perm(u, 0x64646464u, 0x5342);
    const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));  // 1152
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
    return make_uint2(*reinterpret_cast<const uint32_t *>(&ha),
                      *reinterpret_cast<const uint32_t *>(&hb));
}

// Barriers.  stage_full[s] completes when chunk s's activation tile has landed (TMA bytes)
// and the converters have written its weight tile; stage_empty[s] when the MMAs reading
// both have completed.  pair_full[p] / pair_empty[p] hand the two accumulator buffers of
// one chunk between the MMA issuer and the fold warps.
struct Bars {
    uint64_t *stage_full, *stage_empty, *raw_full, *raw_empty, *sc_full, *sc_empty,
        *pair_full, *pair_empty, *mma_done;
};

__device__ __forceinline__ Bars carve_bars(uint8_t *base)
{
    uint64_t *b = reinterpret_cast<uint64_t *>(base);
    Bars r;
    r.stage_full = b; b += MAX_STAGES;
    r.stage_empty = b; b += MAX_STAGES;
    r.raw_full = b; b += RAW_STAGES;
    r.raw_empty = b; b += RAW_STAGES;
    r.sc_full = b; b += SC_STAGES;
    r.sc_empty = b; b += SC_STAGES;
    r.pair_full = b; b += D_PAIRS;
    r.pair_empty = b; b += D_PAIRS;
    r.mma_done = b;
    return r;
}

// A wait that also gives up as soon as another role of this CTA has given up.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, int *status,
                                              volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
#pragma unroll 1
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, WAIT_HINT_NS)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > WAIT_TIMEOUT_NS) {
            atomicOr(status, STATUS_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}

// Work schedule of one launch.  The work is the sequence of units (tile, 256-wide k group),
// tile-major; tiles are 128 weight rows x BN tokens, row tile fastest.  Plain: CTA c does tile
// c over the whole of k.  Balanced: CTA c does the contiguous units [c U / C, (c + 1) U / C),
// whole tiles in the middle and pieces of at most one tile at each end, so every CTA has the
// same work to within one group whatever the tile count.  A piece parks each fold warp's
// 32 x 32 slice of its partial sums in slot 2c (the CTA's first tile) or 2c + 1 (its last);
// for every slice, the warp that completes the count of the tile's pieces (counters[first CTA
// of the tile][warp]) adds the pieces' slices in CTA order and stores them, so the output does
// not depend on which piece finishes first, and no warp ever waits for another.
struct Sched {
    int ntn;             // tiles along n
    int G;               // 256-wide k groups per tile
    long long units;     // tiles * G
    int ctas;            // C = gridDim.x in balanced mode
    int balanced;
    float *partial;      // float4 [2 C][8][512 fold threads]
    unsigned *counters;  // [C][16 fold warps], zero on entry, zero again on exit
};

__host__ __device__ __forceinline__ long long sched_start(const Sched &s, long long c)
{
    return c * s.units / s.ctas;
}

// The CTA whose range holds unit u.
__host__ __device__ __forceinline__ int sched_owner(const Sched &s, long long u)
{
    return (int)(((u + 1) * s.ctas - 1) / s.units);
}

// REPACKED: the weights come as the load-time repacked planes (binary16 quants [n][k] and
// f32 scales [k/32][ldn]) and are loaded by TMA exactly like the activation; the converter
// warps have nothing to do.
template <bool DOTS, bool REPACKED, int BN_T>
__global__ void __launch_bounds__(Cfg<BN_T, !REPACKED>::THREADS, Cfg<BN_T, !REPACKED>::CTAS_PER_SM)
    gemm_q8_0_kernel(const __grid_constant__ CUtensorMap tm_w,
                     const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_xd,
                     const __grid_constant__ CUtensorMap tm_wd, float *__restrict__ y,
                     int32_t *__restrict__ dots, int m, int n, int k, Sched sp, int *status)
{
    using C = Cfg<BN_T, !REPACKED>;
    constexpr int BN = C::BN, TMEM_COLS = C::TMEM_COLS, ACT_TILE_BYTES = C::ACT_TILE_BYTES;
    constexpr int SC_SLOT_BYTES = C::SC_SLOT_BYTES, OFF_ACT = C::OFF_ACT, OFF_A = C::OFF_A, OFF_RAW = C::OFF_RAW;
    constexpr int OFF_SC = C::OFF_SC, OFF_BAR = C::OFF_BAR, OFF_MISC = C::OFF_MISC;
    constexpr int NUM_CONV_WARPS = C::NUM_CONV_WARPS, NUM_FOLD_WARPS = C::NUM_FOLD_WARPS;
    constexpr int PRODUCER_WARP = C::PRODUCER_WARP, MMA_WARP = C::MMA_WARP, NUM_MMA_WARPS = C::NUM_MMA_WARPS;
    constexpr int STAGES = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    Bars bars = carve_bars(smem + OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // This CTA's units [u0, u1); kc below counts the CTA's own chunks (unit u0 + kc / 4).
    const int G = sp.G;
    long long u0, u1;
    if (sp.balanced) {
        u0 = sched_start(sp, blockIdx.x);
        u1 = sched_start(sp, (long long)blockIdx.x + 1);
    } else {
        u0 = (long long)blockIdx.x * G;
        u1 = u0 + G;
    }
    const int nkc = (int)(u1 - u0) * CHUNKS_PER_GROUP;
    const int tile_first = (int)(u0 / G), kg_first = (int)(u0 % G);   // the CTA's first unit
    const int nb = k / QK;

    if (threadIdx.x == 0) {
        constexpr uint32_t conv_arrivals = REPACKED ? 0 : NUM_CONV_WARPS;     // one lane per converter warp
        for (int s = 0; s < STAGES; ++s) { mbar_init(&bars.stage_full[s], 1 + conv_arrivals); mbar_init(&bars.stage_empty[s], 1); }
        for (int s = 0; s < RAW_STAGES; ++s) { mbar_init(&bars.raw_full[s], 1); mbar_init(&bars.raw_empty[s], REPACKED ? 1 : NUM_CONV_WARPS); }
        for (int s = 0; s < SC_STAGES; ++s) { mbar_init(&bars.sc_full[s], 1 + conv_arrivals); mbar_init(&bars.sc_empty[s], NUM_FOLD_WARPS); }
        for (int s = 0; s < D_PAIRS; ++s) { mbar_init(&bars.pair_full[s], 1); mbar_init(&bars.pair_empty[s], NUM_FOLD_WARPS); }
        mbar_init(bars.mma_done, NUM_MMA_WARPS);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(tmem_slot)), "r"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == PRODUCER_WARP && lane == 0) {
        prefetch_tensormap(&tm_w);
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_xd);
        if (REPACKED) prefetch_tensormap(&tm_wd);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;


    if (warp == PRODUCER_WARP) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            int issued_raw = 0, issued_act = 0, issued_sc = 0;
            // The chunk's k group and tile (row tile rt, token tile tt), advanced without
            // divisions: this thread's issue latency paces the repacked kernel.
            int kg = kg_first, rt = tile_first % sp.ntn, tt = tile_first / sp.ntn;
            int row0 = rt * BM, tok0 = tt * BN;
            for (int kc = 0; kc < nkc; ++kc) {
                if (kc > 0 && (kc & (CHUNKS_PER_GROUP - 1)) == 0 && ++kg == G) {
                    kg = 0;
                    if (++rt == sp.ntn) {
                        rt = 0;
                        ++tt;
                    }
                    row0 = rt * BM;
                    tok0 = tt * BN;
                }
                const int kch = kg * CHUNKS_PER_GROUP + (kc & (CHUNKS_PER_GROUP - 1));
                if (!REPACKED && (kc & (CHUNKS_PER_GROUP - 1)) == 0) {
                    const int g = kc / CHUNKS_PER_GROUP;       // local group (ring position)
                    const int rs = g % RAW_STAGES;
                    if (!wait_or_abort(&bars.raw_empty[rs], ((g / RAW_STAGES) & 1) ^ 1, status, abort_flag)) break;
                    mbar_arrive_expect_tx(&bars.raw_full[rs], RAW_TILE_BYTES);
                    tma_load_2d(smem + OFF_RAW + rs * RAW_TILE_BYTES, &tm_w, kg * (GROUP_BYTES / 2), row0,
                                &bars.raw_full[rs]);
                    ++issued_raw;
                }
                const int st = kc % STAGES;
                if (!wait_or_abort(&bars.stage_empty[st], ((kc / STAGES) & 1) ^ 1, status, abort_flag)) break;
                // The activation may come from the kernel just before this one in the stream
                // (launched as its programmatic dependent): everything above -- barriers, TMEM,
                // the first raw weight group -- overlaps that kernel's tail.  After the wait the
                // next kernel of the stream may become resident in turn.
                if (kc == 0) {
                    griddep_wait();
                    griddep_launch_dependents();
                }
                mbar_arrive_expect_tx(&bars.stage_full[st], ACT_TILE_BYTES + (REPACKED ? A_TILE_BYTES : 0));
                tma_load_2d(smem + OFF_ACT + st * ACT_TILE_BYTES, &tm_x, kch * KC, tok0, &bars.stage_full[st]);
                if (REPACKED)
                    tma_load_2d(smem + OFF_A + st * A_TILE_BYTES, &tm_w, kch * KC, row0, &bars.stage_full[st]);
                ++issued_act;
                const int ss = kc % SC_STAGES;
                if (!wait_or_abort(&bars.sc_empty[ss], ((kc / SC_STAGES) & 1) ^ 1, status, abort_flag)) break;
                mbar_arrive_expect_tx(&bars.sc_full[ss], 2 * BN * 4 + (REPACKED ? 2 * BM * 4 : 0));
                tma_load_2d(smem + OFF_SC + ss * SC_SLOT_BYTES, &tm_xd, tok0, 2 * kch, &bars.sc_full[ss]);
                if (REPACKED)
                    tma_load_2d(smem + OFF_SC + ss * SC_SLOT_BYTES + 2 * BN * 4, &tm_wd, row0, 2 * kch, &bars.sc_full[ss]);
                ++issued_sc;
            }
            // Drain: never leave with a copy into this CTA's shared memory in flight.
            for (int i = issued_raw > RAW_STAGES ? issued_raw - RAW_STAGES : 0; i < issued_raw; ++i)
                mbar_wait_drain(&bars.raw_full[i % RAW_STAGES], (i / RAW_STAGES) & 1, status);
            for (int i = issued_act > STAGES ? issued_act - STAGES : 0; i < issued_act; ++i)
                mbar_wait_drain(&bars.stage_full[i % STAGES], (i / STAGES) & 1, status);
            for (int i = issued_sc > SC_STAGES ? issued_sc - SC_STAGES : 0; i < issued_sc; ++i)
                mbar_wait_drain(&bars.sc_full[i % SC_STAGES], (i / SC_STAGES) & 1, status);
        }
    } else if (warp >= MMA_WARP) {
        // ------------------------------ MMA issuers ------------------------------
        // With two issuers, chunk kc goes to the issuer of accumulator pair kc & 1, so one
        // issuer's waits and commits overlap the other's MMAs and the tensor pipe stays fed.
        // A commit tracks the MMAs of its own thread only, which is all that the pair's and
        // the stage's barriers need (a stage, like a pair, is only ever used by one issuer).
        if (lane == 0) {
            // Descriptors of stage 0; a stage or a k step inside the 128-byte row only moves
            // the 14-bit start-address field (all of shared memory is below 256 KB).
            const uint64_t adesc0 = smem_desc_sw128(smem_u32(smem + OFF_A));
            const uint64_t bdesc0 = smem_desc_sw128(smem_u32(smem + OFF_ACT));
            for (int kc = warp - MMA_WARP; kc < nkc; kc += NUM_MMA_WARPS) {
                const int st = kc % STAGES;
                const int pr = kc & 1;
                if (!wait_or_abort(&bars.stage_full[st], (kc / STAGES) & 1, status, abort_flag)) break;
                if (!wait_or_abort(&bars.pair_empty[pr], ((kc >> 1) & 1) ^ 1, status, abort_flag)) break;
                tc_fence_after();
                const uint64_t ad = adesc0 + (uint64_t)(st * (A_TILE_BYTES >> 4));
                const uint64_t bd = bdesc0 + (uint64_t)(st * (ACT_TILE_BYTES >> 4));
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // block 2kc+h -> accumulator buffer 2*pr+h
                    const uint32_t d_tmem = tmem_base + (uint32_t)((2 * pr + h) * BN);
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const uint64_t off = (uint64_t)((h * 64 + kk * 32) >> 4);
                        tc_mma_f16(d_tmem, ad + off, bd + off, C::IDESC, kk);
                    }
                }
                tc_commit(&bars.pair_full[pr]);
                tc_commit(&bars.stage_empty[st]);
            }
            // All MMAs of both issuers have completed once this phase completes.
            tc_commit(bars.mma_done);
            mbar_wait_drain(bars.mma_done, 0, status);
        }
    } else if (warp < NUM_CONV_WARPS) {
        if (REPACKED) {
            // nothing to convert: the producer loads the binary16 weight tiles directly
        } else {
        // ------------------------------ converters ------------------------------
        // Thread t converts rows t and t + 64 of the tile.  For chunk `part` of a raw group,
        // the 68 bytes of its two blocks start at byte 68*part; the five 16-byte words from
        // byte 64*part cover them, the data starting at word `part` of that window.  Both
        // rows' words are read before the waits for the destination slots, and each warp
        // reports a finished chunk with one arrival (after every lane's proxy fence).
        const int ngroups = nkc / CHUNKS_PER_GROUP;
        for (int g = 0; g < ngroups; ++g) {
            const int rs = g % RAW_STAGES;
            if (!wait_or_abort(&bars.raw_full[rs], (g / RAW_STAGES) & 1, status, abort_flag)) break;
            bool ok = true;
#pragma unroll
            for (int part = 0; part < CHUNKS_PER_GROUP; ++part) {
                const int kc = g * CHUNKS_PER_GROUP + part;
                const int aslot = kc % STAGES;
                const int ss = kc % SC_STAGES;
                uint32_t wv[2][20];
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        smem + OFF_RAW + rs * RAW_TILE_BYTES + (threadIdx.x + 64 * rr) * GROUP_BYTES + 64 * part);
#pragma unroll
                    for (int c = 0; c < 5; ++c) {
                        const uint4 v = src[c];
                        wv[rr][4 * c + 0] = v.x; wv[rr][4 * c + 1] = v.y; wv[rr][4 * c + 2] = v.z; wv[rr][4 * c + 3] = v.w;
                    }
                }
                if (!wait_or_abort(&bars.stage_empty[aslot], ((kc / STAGES) & 1) ^ 1, status, abort_flag) ||
                    !wait_or_abort(&bars.sc_empty[ss], ((kc / SC_STAGES) & 1) ^ 1, status, abort_flag)) {
                    ok = false;
                    break;
                }
                float *wsc = reinterpret_cast<float *>(smem + OFF_SC + ss * SC_SLOT_BYTES + 2 * BN * 4);
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int r = threadIdx.x + 64 * rr;
                    // block 2*part: scale in the low half of data word 0, quants straddle words;
                    // block 2*part+1: scale in the high half of data word 8, quants in words 9..16.
                    const int w0 = part;
                    const int w1 = part + 8;
                    uint8_t *arow = smem + OFF_A + aslot * A_TILE_BYTES + r * 128;
                    const int sw = r & 7;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t q0 = __byte_perm(wv[rr][w0 + 2 * c], wv[rr][w0 + 2 * c + 1], 0x5432);
                        const uint32_t q1 = __byte_perm(wv[rr][w0 + 2 * c + 1], wv[rr][w0 + 2 * c + 2], 0x5432);
                        const uint2 lo = bytes_to_f16x4(q0), hi = bytes_to_f16x4(q1);
                        *reinterpret_cast<uint4 *>(arow + ((c ^ sw) << 4)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint2 lo = bytes_to_f16x4(wv[rr][w1 + 1 + 2 * c]);
                        const uint2 hi = bytes_to_f16x4(wv[rr][w1 + 2 + 2 * c]);
                        *reinterpret_cast<uint4 *>(arow + (((c + 4) ^ sw) << 4)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
                    }
                    wsc[r] = half_bits_to_float(wv[rr][w0] & 0xffffu);
                    wsc[BM + r] = half_bits_to_float(wv[rr][w1] >> 16);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars.stage_full[aslot]);
                    mbar_arrive(&bars.sc_full[ss]);
                    if (part == CHUNKS_PER_GROUP - 1) mbar_arrive(&bars.raw_empty[rs]);
                }
            }
            if (!ok) break;
        }
        }
    } else {
        // ------------------------------ fold warps ------------------------------
        const int fw = warp - NUM_CONV_WARPS;      // 0..15
        const int quarter = warp & 3;              // TMEM lanes 32*quarter .. +31
        const int cq = fw >> 2;                    // columns FOLD_COLS*cq .. +FOLD_COLS-1
        const int tr = lane >> 2;                  // row within a 16-lane group (and +8)
        const int tc = 2 * (lane & 3);             // column pair within each 8 columns
        constexpr int NJ = FOLD_COLS / 8;
        // acc[hl][j][e]: rows tr + 8e of the 16-lane half hl, columns (8j+tc, 8j+tc+1).
        float2 acc[2][NJ][2];
#pragma unroll
        for (int hl = 0; hl < 2; ++hl)
#pragma unroll
            for (int j = 0; j < NJ; ++j) { acc[hl][j][0] = make_float2(0.f, 0.f); acc[hl][j][1] = make_float2(0.f, 0.f); }

        constexpr int FT = NUM_FOLD_WARPS * 32;
        // Segments: runs of this CTA's chunks within one tile.  The chunk loop inside is the
        // hot loop; a segment's epilogue stores or parks its accumulators.
        bool ok = true;
        int kc = 0;
        for (int tile = tile_first, seg_kg = kg_first; ok && kc < nkc; ++tile, seg_kg = 0) {
            const int seg_groups = (G - seg_kg) < (nkc - kc) / CHUNKS_PER_GROUP ? (G - seg_kg) : (nkc - kc) / CHUNKS_PER_GROUP;
            const int seg_end = kc + seg_groups * CHUNKS_PER_GROUP;
            const int kch0 = seg_kg * CHUNKS_PER_GROUP - kc;    // + kc: the chunk's place in k
            const int row0 = (tile % sp.ntn) * BM, tok0 = (tile / sp.ntn) * BN;
        for (; kc < seg_end; ++kc) {
            const int ss = kc % SC_STAGES;
            const int pr = kc & 1;
            if (!wait_or_abort(&bars.pair_full[pr], (kc >> 1) & 1, status, abort_flag) ||
                !wait_or_abort(&bars.sc_full[ss], (kc / SC_STAGES) & 1, status, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
                const int b = 2 * (kch0 + kc) + blk;
                // Both 16-lane halves of this warp's 32 x 32 slice of the block's accumulator.
                uint32_t d0[16], d1[16];
                const uint32_t tcol = (uint32_t)((2 * pr + blk) * BN + FOLD_COLS * cq);
                tc_ld_16x256b_x4_async(tmem_base + ((uint32_t)(32 * quarter) << 16) + tcol, d0);
                tc_ld_16x256b_x4_async(tmem_base + ((uint32_t)(32 * quarter + 16) << 16) + tcol, d1);
                tc_wait_ld_bind16<true>(d0);
                tc_wait_ld_bind16<false>(d1);
                if (blk == 1) {
                    // Both buffers of the pair sit in registers (or are folded): hand them back.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars.pair_empty[pr]);
                }

                const float *asc = reinterpret_cast<const float *>(smem + OFF_SC + ss * SC_SLOT_BYTES) + blk * BN + FOLD_COLS * cq + tc;
                const float *wsc = reinterpret_cast<const float *>(smem + OFF_SC + ss * SC_SLOT_BYTES + 2 * BN * 4) + blk * BM + 32 * quarter + tr;
                if (DOTS) {
#pragma unroll
                    for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                        for (int j = 0; j < NJ; ++j)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int r_e = row0 + 32 * quarter + 16 * hl + tr + 8 * (e >> 1);
                                const int t_e = tok0 + FOLD_COLS * cq + 8 * j + tc + (e & 1);
                                const uint32_t v = hl ? d1[4 * j + e] : d0[4 * j + e];
                                if (r_e < n && t_e < m)
                                    dots[((int64_t)t_e * n + r_e) * nb + b] = __float2int_rn(__uint_as_float(v));
                            }
                } else {
                    const float dw00 = wsc[0], dw01 = wsc[8], dw10 = wsc[16], dw11 = wsc[24];
                    const float2 w00 = make_float2(dw00, dw00), w01 = make_float2(dw01, dw01);
                    const float2 w10 = make_float2(dw10, dw10), w11 = make_float2(dw11, dw11);
#pragma unroll
                    for (int j = 0; j < NJ; ++j) {
                        const float2 da = *reinterpret_cast<const float2 *>(asc + 8 * j);
                        const float2 a0 = make_float2(__uint_as_float(d0[4 * j + 0]), __uint_as_float(d0[4 * j + 1]));
                        const float2 a1 = make_float2(__uint_as_float(d0[4 * j + 2]), __uint_as_float(d0[4 * j + 3]));
                        const float2 b0 = make_float2(__uint_as_float(d1[4 * j + 0]), __uint_as_float(d1[4 * j + 1]));
                        const float2 b1 = make_float2(__uint_as_float(d1[4 * j + 2]), __uint_as_float(d1[4 * j + 3]));
                        acc[0][j][0] = fma2_rn(mul2_rn(w00, da), a0, acc[0][j][0]);
                        acc[0][j][1] = fma2_rn(mul2_rn(w01, da), a1, acc[0][j][1]);
                        acc[1][j][0] = fma2_rn(mul2_rn(w10, da), b0, acc[1][j][0]);
                        acc[1][j][1] = fma2_rn(mul2_rn(w11, da), b1, acc[1][j][1]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.sc_empty[ss]);
        }
            // ---- end of the segment ----
            if (!ok) break;
            if (!DOTS && !*abort_flag) {
                bool store = seg_kg == 0 && seg_groups == G;   // the whole tile
                if (!store) {
                    // A piece: park this warp's slice, thread index fastest (every warp store is
                    // one contiguous 512-byte run), then count it.
                    const int slot = 2 * (int)blockIdx.x + (tile == tile_first ? 0 : 1);
                    float4 *dst = reinterpret_cast<float4 *>(sp.partial) + (int64_t)slot * (2 * NJ * FT) + fw * 32 + lane;
#pragma unroll
                    for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                        for (int j = 0; j < NJ; ++j)
                            __stcg(dst + (hl * NJ + j) * FT,
                                   make_float4(acc[hl][j][0].x, acc[hl][j][0].y, acc[hl][j][1].x, acc[hl][j][1].y));
                    __threadfence();
                    __syncwarp();
                    const int c0 = sched_owner(sp, (long long)tile * G);
                    const int cl = sched_owner(sp, (long long)tile * G + G - 1);
                    uint32_t last = 0;
                    if (lane == 0) {
                        unsigned *ctr = sp.counters + (size_t)c0 * NUM_FOLD_WARPS + fw;
                        const unsigned before = atomicAdd(ctr, 1u);
                        last = before == (unsigned)(cl - c0) ? 1u : 0u;
                        if (last) *ctr = 0;   // ready for the next launch
                        __threadfence();
                    }
                    store = __shfl_sync(0xffffffffu, last, 0) != 0;
                    if (store) {
                        // This warp's slice is complete: the pieces' sum, in CTA order.
                        __threadfence();
                        for (int cc = c0; cc <= cl; ++cc) {
                            const int sl = 2 * cc + (tile == (int)(sched_start(sp, cc) / G) ? 0 : 1);
                            const float4 *src = reinterpret_cast<const float4 *>(sp.partial) + (int64_t)sl * (2 * NJ * FT) +
                                                fw * 32 + lane;
#pragma unroll
                            for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                                for (int j = 0; j < NJ; ++j) {
                                    const float4 v = __ldcg(src + (hl * NJ + j) * FT);
                                    if (cc == c0) {
                                        acc[hl][j][0] = make_float2(v.x, v.y);
                                        acc[hl][j][1] = make_float2(v.z, v.w);
                                    } else {
                                        acc[hl][j][0].x = __fadd_rn(acc[hl][j][0].x, v.x);
                                        acc[hl][j][0].y = __fadd_rn(acc[hl][j][0].y, v.y);
                                        acc[hl][j][1].x = __fadd_rn(acc[hl][j][1].x, v.z);
                                        acc[hl][j][1].y = __fadd_rn(acc[hl][j][1].y, v.w);
                                    }
                                }
                        }
                    }
                }
                if (store) {
#pragma unroll
                    for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                        for (int j = 0; j < NJ; ++j)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int r_e = row0 + 32 * quarter + 16 * hl + tr + 8 * (e >> 1);
                                const int t_e = tok0 + FOLD_COLS * cq + 8 * j + tc + (e & 1);
                                const float2 v = acc[hl][j][e >> 1];
                                if (r_e < n && t_e < m) y[(int64_t)t_e * n + r_e] = (e & 1) ? v.y : v.x;
                            }
                }
            }
#pragma unroll
            for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                for (int j = 0; j < NJ; ++j) { acc[hl][j][0] = make_float2(0.f, 0.f); acc[hl][j][1] = make_float2(0.f, 0.f); }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(TMEM_COLS) : "memory");
    }
}

// ---------------------------------------------------------------------------------------
// Host: tensor maps through the driver entry point (no libcuda link dependency).
// ---------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

bool encode_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t dim0,
               uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
               CUtensorMapSwizzle swz)
{
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {dim0, dim1};
    const cuuint64_t strides[1] = {stride1_bytes};
    const cuuint32_t box[2] = {box0, box1};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {

}  // namespace

size_t gemm_split_bytes();

namespace {

constexpr int kMaxCtas = 160;   // CTAs of a balanced launch (>= the SM count)
constexpr int kFoldWarps = 16;
constexpr size_t kPartialBytes = (size_t)2 * kMaxCtas * BM * 128 * 4;   // two 128 x 128 f32 tiles per CTA
constexpr size_t kCounterBytes = (size_t)kMaxCtas * kFoldWarps * sizeof(unsigned);

// Plain (one CTA per tile over the whole of k) or balanced, whichever a simple cost model in
// k groups on the longest-running SM favours: plain takes waves * G plus one group of set-up
// per extra wave; balanced takes ceil(U / C) groups plus two for parking and counting pieces
// plus one per piece of the most-cut tile (the completing warp reads every piece).  Measured
// on GB300: at m = 512, 4096 x 4096 (128 tiles on 152 SMs, every tile cut) plain wins, 54 vs
// 62 us per call; at 164, 640, 2016 and 2560 tiles balanced wins by 3-30 %.  The block-dot
// export and calls without the split region are always plain.
Sched plan_sched(const DeviceInfo &dev, int64_t m, int64_t n, int64_t k, int BN, int ctas_per_sm, void *split_ws,
                 size_t split_bytes, bool zero_counters, int64_t *grid, cudaStream_t stream, cudaError_t *err)
{
    Sched sp{};
    const int64_t ntn = (n + BM - 1) / BM, ntm = (m + BN - 1) / BN, tiles = ntn * ntm;
    sp.ntn = (int)ntn;
    sp.G = (int)(k / (KC * CHUNKS_PER_GROUP));
    sp.units = tiles * sp.G;
    sp.ctas = (int)tiles;
    sp.balanced = 0;
    *grid = tiles;
    *err = cudaSuccess;
    const int64_t cap = (int64_t)dev.num_sms * ctas_per_sm;
    const int64_t slots = cap < kMaxCtas ? cap : kMaxCtas;
    if (!split_ws || split_bytes < gemm_split_bytes() || tiles % slots == 0) return sp;
    const int64_t C = slots < sp.units ? slots : sp.units;
    const int64_t waves = (tiles + slots - 1) / slots;
    const int64_t plain_cost = waves * sp.G + (waves - 1);
    const int64_t per = sp.units / C;
    const int64_t most_pieces = (sp.G + per - 1) / per + 1;
    const int64_t balanced_cost = (sp.units + C - 1) / C + 2 + most_pieces;
    if (balanced_cost >= plain_cost) return sp;
    sp.balanced = 1;
    sp.ctas = (int)C;
    sp.partial = static_cast<float *>(split_ws);
    sp.counters = reinterpret_cast<unsigned *>(static_cast<uint8_t *>(split_ws) + kPartialBytes);
    *grid = C;
    if (zero_counters) *err = cudaMemsetAsync(sp.counters, 0, (size_t)C * kFoldWarps * sizeof(unsigned), stream);
    return sp;
}

// pdl: launch as a programmatic dependent of the stream's previous kernel (the activation
// quantizer of the same call); the split counters were then zeroed before that kernel.
template <bool DOTS, bool REPACKED, int BN_T>
cudaError_t launch_kernel(const DeviceInfo &dev, const CUtensorMap &tm_w, const CUtensorMap &tm_x,
                          const CUtensorMap &tm_xd, const CUtensorMap &tm_wd, float *y, int32_t *dots,
                          int64_t m, int64_t n, int64_t k, void *split_ws, size_t split_bytes, bool pdl,
                          cudaStream_t stream)
{
    using C = Cfg<BN_T, !REPACKED>;
    auto kern = gemm_q8_0_kernel<DOTS, REPACKED, BN_T>;
    cudaError_t e = set_kernel_smem<gemm_q8_0_kernel<DOTS, REPACKED, BN_T>>(dev.device, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    int64_t grid = 0;
    static_assert(C::NUM_FOLD_WARPS == kFoldWarps, "counter layout");
    const Sched sp = plan_sched(dev, m, n, k, BN_T, C::CTAS_PER_SM, DOTS ? nullptr : split_ws, split_bytes, !pdl,
                                &grid, stream, &e);
    if (e != cudaSuccess) return e;
    if (!pdl) {
        kern<<<(unsigned)grid, C::THREADS, C::SMEM_BYTES, stream>>>(tm_w, tm_x, tm_xd, tm_wd, y, dots, (int)m,
                                                              (int)n, (int)k, sp, dev.status);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tm_w, tm_x, tm_xd, tm_wd, y, dots, (int)m, (int)n, (int)k, sp, dev.status);
}

bool encode_activation(CUtensorMap *tm_x, CUtensorMap *tm_xd, const uint16_t *xqh, const float *xdt,
                       int64_t m, int64_t k, int64_t ldm, int bn)
{
    return encode_2d(tm_x, CU_TENSOR_MAP_DATA_TYPE_UINT16, xqh, (uint64_t)k, (uint64_t)m, (uint64_t)k * 2,
                     KC, bn, CU_TENSOR_MAP_SWIZZLE_128B) &&
           encode_2d(tm_xd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, xdt, (uint64_t)m, (uint64_t)(k / QK),
                     (uint64_t)ldm * 4, bn, 2, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace

size_t gemm_split_bytes()
{
    static_assert(kPartialBytes + kCounterBytes == Q8ACT_GEMM_SPLIT_BYTES,
                  "split region size");
    return Q8ACT_GEMM_SPLIT_BYTES;
}

cudaError_t gemm_prepare_split(const DeviceInfo &dev, int64_t m, int64_t n, int64_t k, bool repacked,
                               void *split_ws, size_t split_bytes, cudaStream_t stream)
{
    int64_t grid = 0;
    cudaError_t e = cudaSuccess;
    const int ctas = repacked ? Cfg<RP_BN, false>::CTAS_PER_SM : Cfg<128, true>::CTAS_PER_SM;
    plan_sched(dev, m, n, k, repacked ? RP_BN : 128, ctas, split_ws, split_bytes, true, &grid, stream, &e);
    return e;
}

cudaError_t launch_gemm_q8_0(const DeviceInfo &dev, const uint8_t *w, const uint16_t *xqh,
                             const float *xdt, float *y, int32_t *dots, int64_t m, int64_t n,
                             int64_t k, int64_t ldm, void *split_ws, size_t split_bytes, bool pdl,
                             cudaStream_t stream)
{
    CUtensorMap tm_w, tm_x, tm_xd;
    const uint64_t row_bytes = (uint64_t)k / QK * Q8_0_BYTES;
    // Raw weights viewed as uint16 elements: a 272-byte group is 136 elements (16-byte multiple).
    if (!encode_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT16, w, row_bytes / 2, (uint64_t)n, row_bytes,
                   GROUP_BYTES / 2, BM, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_activation(&tm_x, &tm_xd, xqh, xdt, m, k, ldm, 128))
        return cudaErrorInvalidValue;
    return dots ? launch_kernel<true, false, 128>(dev, tm_w, tm_x, tm_xd, tm_xd, y, dots, m, n, k, nullptr, 0, pdl,
                                                  stream)
                : launch_kernel<false, false, 128>(dev, tm_w, tm_x, tm_xd, tm_xd, y, dots, m, n, k, split_ws,
                                                   split_bytes, pdl, stream);
}

cudaError_t launch_gemm_q8_0_repacked(const DeviceInfo &dev, const uint16_t *wq16, const float *wdt,
                                      int64_t ldn, const uint16_t *xqh, const float *xdt, float *y,
                                      int32_t *dots, int64_t m, int64_t n, int64_t k, int64_t ldm,
                                      void *split_ws, size_t split_bytes, bool pdl, cudaStream_t stream)
{
    CUtensorMap tm_w, tm_x, tm_xd, tm_wd;
    // The weight planes have the activation's layouts: binary16 [n][k] tiles of 64 k x 128
    // rows with the 128-byte swizzle, and f32 scales [k/32][ldn] in boxes of 128 rows x 2 blocks.
    if (!encode_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT16, wq16, (uint64_t)k, (uint64_t)n, (uint64_t)k * 2,
                   KC, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tm_wd, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, wdt, (uint64_t)n, (uint64_t)(k / QK),
                   (uint64_t)ldn * 4, BM, 2, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_activation(&tm_x, &tm_xd, xqh, xdt, m, k, ldm, RP_BN))
        return cudaErrorInvalidValue;
    return dots ? launch_kernel<true, true, RP_BN>(dev, tm_w, tm_x, tm_xd, tm_wd, y, dots, m, n, k, nullptr, 0, pdl,
                                                   stream)
                : launch_kernel<false, true, RP_BN>(dev, tm_w, tm_x, tm_xd, tm_wd, y, dots, m, n, k, split_ws,
                                                    split_bytes, pdl, stream);
}

}  // namespace q8
