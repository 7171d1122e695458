// common.cuh -- shared device helpers of libq8act (sm_103a): constants, PTX wrappers for
// mbarriers, bulk/TMA copies and tcgen05, and bounded pipeline waits.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "q8act.h"

namespace q8 {

constexpr int QK = 32;            // values per block
constexpr int Q8_0_BYTES = 34;    // binary16 scale + 32 int8 quants
constexpr int GROUP_BLOCKS = 8;   // 8 blocks = 272 bytes = 17 x 16 B (lcm of 34 and 16)
constexpr int GROUP_BYTES = GROUP_BLOCKS * Q8_0_BYTES;
constexpr int Q4_0_BYTES = 18;    // binary16 scale + 16 bytes of 4-bit quants (GGUF Q4_0)
constexpr int Q4_GROUP_BYTES = GROUP_BLOCKS * Q4_0_BYTES;   // 144 = 9 x 16 B
constexpr int K_ALIGN = 256;      // k must be a multiple of this (row start 16 B aligned)

// Device status word bits (read back by q8act_device_status).
constexpr int STATUS_TIMEOUT = 1;        // a pipeline wait gave up; the kernel left its loop
constexpr int STATUS_DRAIN_TIMEOUT = 2;  // a wait for the CTA's own copies in flight gave up

// A pipeline wait gives up after this long (the kernel then records STATUS_TIMEOUT and
// leaves its loop instead of hanging the GPU).
constexpr unsigned long long WAIT_TIMEOUT_NS = 2000000000ull;

__device__ __forceinline__ unsigned long long globaltimer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: the waiting thread is parked by the hardware until the
// phase completes or about `hint_ns` nanoseconds pass, instead of spinning on the issue slots
// that the working warps of the same SM sub-partition need.
// Programmatic dependent launch.  The GEMVs, dequants and K-quant kernels are launched with
// programmatic stream serialization, so they may become resident while the previous kernel
// of the stream still runs; each passes griddep_wait() before touching global memory (the
// wait returns once that grid has completed and its writes are visible; without a
// prerequisite grid it returns at once), and only then calls griddep_launch_dependents(),
// which lets the next kernel become resident in turn.  So a dependent that starts early knows
// that everything before its predecessor has completed.  The quantizers are ordinary launches
// (grids of many small CTAs, beside which waiting dependents would take issue slots) that
// trigger their dependents at entry; the second kernel of a fused call (the GEMV or GEMM
// after the call's own quantizer) streams weights before its wait, which the quantizer does
// not write.  Resident dependents cannot starve their predecessor: they launch only once every
// CTA of it has started.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// The entry of a kernel with nothing to do before its predecessor completes.
__device__ __forceinline__ void griddep_enter()
{
    griddep_wait();
    griddep_launch_dependents();
}

// Host: launch `kern` as a programmatic dependent of the stream's previous kernel.
template <typename Kern, typename... Args>
cudaError_t launch_dependent(Kern kern, dim3 grid, unsigned block, size_t smem, cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

constexpr uint32_t WAIT_HINT_NS = 200000;

// Wait until the phase with the given parity has completed.  Returns false (after OR-ing
// `bit` into *status) if that takes longer than limit_ns nanoseconds.
__device__ __forceinline__ bool mbar_wait_for(uint64_t *bar, uint32_t parity, int *status,
                                              unsigned long long limit_ns, int bit)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    const uint32_t hint = limit_ns < WAIT_HINT_NS ? (uint32_t)limit_ns : WAIT_HINT_NS;
#pragma unroll 1
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, hint)) return true;
        if (globaltimer() - t0 > limit_ns) {
            atomicOr(status, bit);
            return false;
        }
    }
}

// A pipeline wait: gives up (STATUS_TIMEOUT) after WAIT_TIMEOUT_NS.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *status)
{
    return mbar_wait_for(bar, parity, status, WAIT_TIMEOUT_NS, STATUS_TIMEOUT);
}

// A producer's final wait for its own copies into shared memory before the CTA exits: gives
// up (STATUS_DRAIN_TIMEOUT, the more serious condition -- a copy may then still land in
// shared memory after the CTA is gone) after WAIT_TIMEOUT_NS.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t *bar, uint32_t parity, int *status)
{
    return mbar_wait_for(bar, parity, status, WAIT_TIMEOUT_NS, STATUS_DRAIN_TIMEOUT);
}

// ---------------------------------------------------------------------------------------
// Bulk (non-tensor) and tensor (TMA) copies global -> shared, completing on an mbarrier.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                         uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// The same copy with an L2 cache policy (e.g. evict-first for a stream read exactly once).
__device__ __forceinline__ void bulk_g2s_hint(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// An L2 policy that evicts the lines it covers first.
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}

__device__ __forceinline__ void tma_load_2d(void *dst_smem, const CUtensorMap *map, int32_t x,
                                            int32_t y, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst_smem)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
        "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Generic-proxy shared-memory writes -> visible to the async proxy (tensor core reads).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------------------
// Small arithmetic helpers
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float half_bits_to_float(uint32_t h16)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h16)));
}

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c)
{
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// Shared-memory words at byte addresses (4- and 2-byte aligned).
__device__ __forceinline__ uint32_t lds32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }
__device__ __forceinline__ uint32_t lds16(const uint8_t *p) { return *reinterpret_cast<const uint16_t *>(p); }

// A CTA barrier over `nthreads` threads that also ORs a predicate across them.
__device__ __forceinline__ bool bar_red_or(int id, int nthreads, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------------------------------
// Warp-level tensor-core MMA (mma.sync): A 16 x K row-major, B K x 8 column-major, fragments
// as the PTX ISA lays them out (lane = 4 * group + column pair).
// ---------------------------------------------------------------------------------------
// int8 x int8 -> int32, K = 32: a[0..3] = rows (g, g+8) x k (4c..4c+3, 16+4c..16+4c+3)
__device__ __forceinline__ void mma_s8_16832(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(0));
}

// int8 x int8 -> int32, K = 16: a0 = row g, a1 = row g + 8, k 4c..4c+3
__device__ __forceinline__ void mma_s8_16816(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%7,%7,%7,%7};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(b0), "r"(0));
}

// binary16 x binary16 -> f32, K = 16, accumulating onto c
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                              const float (&c)[4])
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

// ---------------------------------------------------------------------------------------
// Host: a kernel's dynamic shared-memory limit and the largest carveout, set once per device
// (and again when a launch needs more), not on every call -- the driver calls cost microseconds
// of host time, as much as a small kernel runs.
// ---------------------------------------------------------------------------------------
constexpr int kAttrDevices = 16;

template <auto Kern>
cudaError_t set_kernel_smem(int device, size_t smem)
{
    static std::atomic<size_t> done[kAttrDevices];
    const bool cache = device >= 0 && device < kAttrDevices;
    if (cache && done[device].load(std::memory_order_relaxed) >= smem && smem > 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaFuncSetAttribute(Kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (cache) done[device].store(smem, std::memory_order_relaxed);
    return cudaSuccess;
}

// ---------------------------------------------------------------------------------------
// Host: a process-unique id of the calling thread's current CUDA context (0 when there is
// none yet or the driver entry points are unavailable).  Addresses of __device__ variables
// belong to a context: a per-device cache of such an address is keyed on this id, so that a
// context torn down and created again (cudaDeviceReset, a primary context released and
// retained) gets its addresses looked up afresh.
// ---------------------------------------------------------------------------------------
inline unsigned long long current_context_id()
{
    typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
    typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr, *q = nullptr;
        cudaDriverEntryPointQueryResult r1, r2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &r1) == cudaSuccess &&
            r1 == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) == cudaSuccess &&
            r2 == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
            get_id = reinterpret_cast<CtxGetIdFn>(q);
        }
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Several weight matrices that share the activation, streamed by one launch (the census's
// stacked expert gate+up and the fused qkv shapes, as separate buffers): chunk c belongs to
// matrix i when first_chunk[i] <= c < first_chunk[i + 1].  A single GEMV is a group of one.
struct Group {
    int count;
    const uint8_t *w[Q8ACT_GEMV_MAX_GROUP];
    float *y[Q8ACT_GEMV_MAX_GROUP];
    int n[Q8ACT_GEMV_MAX_GROUP];
    int64_t first_chunk[Q8ACT_GEMV_MAX_GROUP + 1];
};

struct ChunkRef {
    const uint8_t *w;
    float *y;
    int n;
    int64_t row0;
    int rows;
};

__device__ __forceinline__ ChunkRef chunk_ref(const Group &grp, int64_t chunk, int R)
{
    int mi = 0;
    while (mi + 1 < grp.count && chunk >= grp.first_chunk[mi + 1]) ++mi;
    ChunkRef c;
    c.w = grp.w[mi];
    c.y = grp.y[mi];
    c.n = grp.n[mi];
    c.row0 = (chunk - grp.first_chunk[mi]) * R;
    c.rows = (int)((c.n - c.row0) < R ? (c.n - c.row0) : R);
    return c;
}

}  // namespace q8
