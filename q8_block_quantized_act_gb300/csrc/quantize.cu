// quantize.cu -- the per-32-block quantizers: q8_1 activations (int8 and MMQ layouts), and
// Q8_0 and Q4_0 weights (data preparation).  All three are HBM-bound elementwise passes: one thread owns 4 consecutive
// values (one 16-byte load), 8 consecutive lanes own one block and find its amax with three
// shuffles.
//
// The arithmetic is the per-block formula of memra-engine 0.81.0 f16_ffi.rs (try_f16_gemm,
// W8A8 pilot): amax = max|v|, d = amax / 127, q = clamp(round(v / d), -127, 127), guarded
// by amax > 0.  The division is IEEE (this file must not be built with fast-math or
// -prec-div=false) and roundf rounds half away from zero, as Rust's f32::round does.
#include "common.cuh"
#include "launch.h"

namespace q8 {
namespace {

constexpr unsigned FULL = 0xffffffffu;

struct Block4 {
    int q[4];
    float d;
};

// Quantize this thread's 4 values of a block whose 32 values are spread over 8 lanes.
__device__ __forceinline__ Block4 quantize4(float4 v)
{
    // Start from 0 so that a block of NaNs behaves like the scalar loop's "a > amax".
    float a = fmaxf(fmaxf(fmaxf(0.0f, fabsf(v.x)), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 1));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 2));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 4));
    Block4 r;
    r.d = __fdiv_rn(a, 127.0f);
    // round(fl(v / d)) without a division per value: q' = v * rcp_rn(d) differs from
    // fl(v / d) by at most ~2.3e-5 (|v / d| <= 127, each of rcp, the product and the quotient
    // is within 2^-24 relative), so unless q' lies within 1e-3 of a half-integer -- or is not
    // finite -- it rounds to the same integer.  Those rare cases take the IEEE division.
    const float rc = __frcp_rn(r.d);
    const float vals[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (r.d == 0.0f) {
            r.q[i] = 0;
        } else {
            const float qa = __fmul_rn(vals[i], rc);
            const float aq = fabsf(qa);
            const float fr = aq - floorf(aq);
            float t = (fabsf(fr - 0.5f) > 1e-3f) ? roundf(qa) : roundf(__fdiv_rn(vals[i], r.d));
            if (t > 127.0f) t = 127.0f;
            if (t < -127.0f) t = -127.0f;
            r.q[i] = __float2int_rz(t);  // NaN converts to 0
        }
    }
    return r;
}

// The q8_1 activation quantizer's form of the same arithmetic, with the quants returned as
// integer-valued floats (+0 for zero).  For a value whose approximate quotient qa = v * (1/d)
// lies farther than 1e-3 from every half-integer, rint(qa) is round-half-away(fl(v / d)): qa
// differs from v / d by under 4e-5 (|v / d| <= 127; the reciprocal's relative error is at most
// 2^-23, the product's 2^-24) and fl(v / d) from v / d by under 8e-6, so all three round to the
// same integer, and no tie is involved.  The test |qa - rint(qa)| < 0.499 selects exactly those
// values; the rest (near a half-integer, or qa not finite) take the IEEE division and the
// rounding of the scalar formula, as in quantize4.  A block whose amax is 0 gives q = 0.
struct Block4f {
    float t[4];
    float d;
};

__device__ __forceinline__ float rcp_approx(float x)
{
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// amax / 127 correctly rounded, for amax >= 0: Markstein's correction for a division by a
// known divisor (a quotient q0 = amax * RN(1/127), its exact residual amax - 127 q0 by one FMA,
// and q0 + residual * RN(1/127) by another).  Checked against IEEE division on the host for
// every non-negative binary32 value: all agree except amax = +inf (the residual is then NaN),
// which is selected separately.
__device__ __forceinline__ float div127(float a)
{
    const float c = 1.0f / 127.0f;
    const float q0 = __fmul_rn(a, c);
    const float q1 = __fmaf_rn(__fmaf_rn(-q0, 127.0f, a), c, q0);
    return a == __int_as_float(0x7f800000) ? a : q1;
}

__device__ __forceinline__ Block4f quantize4f(float4 v)
{
    float a = fmaxf(fmaxf(fmaxf(0.0f, fabsf(v.x)), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 1));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 2));
    a = fmaxf(a, __shfl_xor_sync(FULL, a, 4));
    Block4f r;
    r.d = div127(a);
    const float rc = rcp_approx(r.d);
    const float vals[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float qa = __fmul_rn(vals[i], rc);
        float t = rintf(qa);
        if (r.d == 0.0f) {
            t = 0.0f;
        } else if (fabsf(__fsub_rn(qa, t)) < 0.499f) {
            t = fminf(fmaxf(t, -127.0f), 127.0f);
        } else {
            t = roundf(__fdiv_rn(vals[i], r.d));
            if (t > 127.0f) t = 127.0f;
            if (t < -127.0f) t = -127.0f;
            if (!(t == t)) t = 0.0f;       // NaN quantizes to 0
        }
        r.t[i] = __fadd_rn(t, 0.0f);       // -0 -> +0
    }
    return r;
}

// An integer-valued float t, |t| <= 127, as its int8 byte: the bits of t + 1.5 * 2^23 are
// those of 1.5 * 2^23 plus t (unit spacing there), so the low byte is t's two's complement.
__device__ __forceinline__ uint32_t byte_of(float t)
{
    return (uint32_t)__float_as_int(__fadd_rn(t, 12582912.0f)) & 0xFFu;
}

__device__ __forceinline__ float4 load_stream(const float4 *p)
{
    return __ldcs(p);
}

// x [m][k] f32 -> xq [m][k] int8, xd [m][k/32] f32.
__global__ void __launch_bounds__(256) quantize_q8_1_kernel(const float4 *__restrict__ x,
                                                            uint32_t *__restrict__ xq,
                                                            float *__restrict__ xd,
                                                            int64_t nchunks)
{
    // An ordinary launch (it starts once everything before it in the stream has completed);
    // the GEMV that consumes this activation is launched as its programmatic dependent and may
    // start streaming its weights now (it waits for this grid before reading the activation).
    griddep_launch_dependents();
    // Two independent chunks per step (more loads in flight).  nchunks is a multiple of 64
    // and the stride of 32, so both halves are warp-uniform, as the shuffles need.
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nchunks; i += 2 * stride) {
        const bool two = i + stride < nchunks;
        const float4 v0 = load_stream(x + i);
        const float4 v1 = two ? load_stream(x + i + stride) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (h == 1 && !two) break;
            const int64_t c = i + h * stride;
            const Block4f b = quantize4f(h ? v1 : v0);
            xq[c] = byte_of(b.t[0]) | (byte_of(b.t[1]) << 8) | (byte_of(b.t[2]) << 16) | (byte_of(b.t[3]) << 24);
            if ((c & 7) == 0) xd[c >> 3] = b.d;
        }
    }
}

// x [m][k] f32 -> xqh [m][k] binary16 (exact small integers), xdt [k/32][ldm] f32.
// Grid: (ceil(k/4 / 256), min(ceil(m / MMQ_TPT), 65535)); thread (chunk c of the row of each
// of its tokens t = blockIdx.y + (i * MMQ_TPT + j) * gridDim.y).  A thread loads its MMQ_TPT
// tokens' chunks before quantizing any of them (loads in flight); k/4 is a multiple of 64 and
// the token test is the same for every lane of a warp, so every warp is either fully inside
// a row or fully past its end, as the block's shuffles need.
constexpr int MMQ_TPT = 4;
__global__ void __launch_bounds__(256) quantize_q8_1_mmq_kernel(const float4 *__restrict__ x,
                                                                uint2 *__restrict__ xqh,
                                                                float *__restrict__ xdt,
                                                                int64_t m, int chunks_per_row,
                                                                int64_t ldm)
{
    // An ordinary launch (it starts once everything before it in the stream has completed);
    // the GEMM that consumes this layout is launched as its programmatic dependent and may
    // start its prologue now (it waits for this grid before reading the activation).
    griddep_launch_dependents();
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= chunks_per_row) return;
    const int64_t ys = gridDim.y;
    for (int64_t t0 = blockIdx.y; t0 < m; t0 += ys * MMQ_TPT) {
        float4 v[MMQ_TPT];
#pragma unroll
        for (int j = 0; j < MMQ_TPT; ++j) {
            const int64_t t = t0 + j * ys;
            v[j] = t < m ? load_stream(x + t * chunks_per_row + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < MMQ_TPT; ++j) {
            const int64_t t = t0 + j * ys;
            if (t >= m) break;
            const int64_t g = t * chunks_per_row + c;
            const Block4f b = quantize4f(v[j]);
            // the quants are small integers: exact in binary16
            const __half2 h01 = __floats2half2_rn(b.t[0], b.t[1]);
            const __half2 h23 = __floats2half2_rn(b.t[2], b.t[3]);
            xqh[g] = make_uint2(*reinterpret_cast<const uint32_t *>(&h01), *reinterpret_cast<const uint32_t *>(&h23));
            if ((c & 7) == 0) xdt[(int64_t)(c >> 3) * ldm + t] = b.d;
        }
    }
}

// w [n][k] f32 -> Q8_0 blocks (34 B: binary16 scale of the f32 d, then 32 int8 quants).
__global__ void __launch_bounds__(256) quantize_q8_0_kernel(const float4 *__restrict__ w,
                                                            uint8_t *__restrict__ out,
                                                            int64_t nchunks)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nchunks; i += stride) {
        Block4 b = quantize4(load_stream(w + i));
        uint8_t *blk = out + (i >> 3) * Q8_0_BYTES;
        const int j = (int)(i & 7);
        // quants of this thread start at byte 2 + 4j: 2-byte aligned
        uint16_t *q16 = reinterpret_cast<uint16_t *>(blk + 2 + 4 * j);
        q16[0] = (uint16_t)((b.q[0] & 0xff) | ((b.q[1] & 0xff) << 8));
        q16[1] = (uint16_t)((b.q[2] & 0xff) | ((b.q[3] & 0xff) << 8));
        if (j == 0)
            *reinterpret_cast<uint16_t *>(blk) = __half_as_ushort(__float2half_rn(b.d));
    }
}

// w [n][k] f32 -> Q4_0 blocks (18 B: binary16 scale of the f32 d = amax / 7, then 16 bytes,
// element i < 16 in the low nibble of byte i and element i + 16 in its high nibble, each
// stored as q + 8 with q = clamp(round(v / d), -8, 7)).  Data preparation for the Q4_0 path.
// nchunks is a multiple of 64 and the stride of 32, so the loop and its shuffles are
// warp-uniform; lanes 0-3 of a block's 8 write its bytes, merging lane j + 4's nibbles.
__global__ void __launch_bounds__(256) quantize_q4_0_kernel(const float4 *__restrict__ w,
                                                            uint8_t *__restrict__ out,
                                                            int64_t nchunks)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nchunks; i += stride) {
        const float4 v = load_stream(w + i);
        float a = fmaxf(fmaxf(fmaxf(0.0f, fabsf(v.x)), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
        a = fmaxf(a, __shfl_xor_sync(FULL, a, 1));
        a = fmaxf(a, __shfl_xor_sync(FULL, a, 2));
        a = fmaxf(a, __shfl_xor_sync(FULL, a, 4));
        const float d = __fdiv_rn(a, 7.0f);
        const float vals[4] = {v.x, v.y, v.z, v.w};
        uint32_t nib4 = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            int q = 0;
            if (d != 0.0f) {
                float t = roundf(__fdiv_rn(vals[e], d));
                if (t > 7.0f) t = 7.0f;
                if (t < -8.0f) t = -8.0f;
                q = __float2int_rz(t);   // NaN converts to 0
            }
            nib4 |= (uint32_t)(q + 8) << (8 * e);
        }
        const uint32_t hi = __shfl_down_sync(FULL, nib4, 4);
        const int j = (int)(i & 7);
        if (j < 4) {
            uint8_t *blk = out + (i >> 3) * Q4_0_BYTES;
            const uint32_t bytes = nib4 | (hi << 4);
            uint16_t *q16 = reinterpret_cast<uint16_t *>(blk + 2 + 4 * j);   // 2-byte aligned
            q16[0] = (uint16_t)(bytes & 0xffffu);
            q16[1] = (uint16_t)(bytes >> 16);
            if (j == 0) *reinterpret_cast<uint16_t *>(blk) = __half_as_ushort(__float2half_rn(d));
        }
    }
}

// Every kernel of the library asks for the largest shared-memory carveout, so that moving
// between these smem-free passes and the shared-memory-heavy GEMV/GEMM/dequant never forces
// the SM to re-partition its L1/shared memory between launches.
template <typename K>
void set_max_carveout(K kern)
{
    static bool done = false;
    if (!done) {
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
        done = true;
    }
}

int grid_for(const DeviceInfo &dev, int64_t nchunks, int threads)
{
    int64_t want = (nchunks + threads - 1) / threads;
    int64_t cap = (int64_t)dev.num_sms * 8;
    return (int)(want < cap ? want : cap);
}

}  // namespace

cudaError_t launch_quantize_q8_1(const DeviceInfo &dev, const float *x, int8_t *xq, float *xd,
                                 int64_t m, int64_t k, cudaStream_t stream)
{
    const int64_t nchunks = m * k / 4;
    set_max_carveout(quantize_q8_1_kernel);
    quantize_q8_1_kernel<<<grid_for(dev, nchunks, 256), 256, 0, stream>>>(
        reinterpret_cast<const float4 *>(x), reinterpret_cast<uint32_t *>(xq), xd, nchunks);
    return cudaGetLastError();
}

cudaError_t launch_quantize_q8_1_mmq(const DeviceInfo &dev, const float *x, uint16_t *xqh,
                                     float *xdt, int64_t m, int64_t k, int64_t ldm,
                                     cudaStream_t stream)
{
    const int cpr = (int)(k / 4);
    set_max_carveout(quantize_q8_1_mmq_kernel);
    const int64_t gy = (m + MMQ_TPT - 1) / MMQ_TPT;
    const dim3 grid((unsigned)((cpr + 255) / 256), (unsigned)(gy < 65535 ? gy : 65535));
    quantize_q8_1_mmq_kernel<<<grid, 256, 0, stream>>>(
        reinterpret_cast<const float4 *>(x), reinterpret_cast<uint2 *>(xqh), xdt, m, cpr, ldm);
    return cudaGetLastError();
}

cudaError_t launch_quantize_q8_0(const DeviceInfo &dev, const float *w, uint8_t *wq, int64_t n,
                                 int64_t k, cudaStream_t stream)
{
    const int64_t nchunks = n * k / 4;
    set_max_carveout(quantize_q8_0_kernel);
    quantize_q8_0_kernel<<<grid_for(dev, nchunks, 256), 256, 0, stream>>>(
        reinterpret_cast<const float4 *>(w), wq, nchunks);
    return cudaGetLastError();
}

cudaError_t launch_quantize_q4_0(const DeviceInfo &dev, const float *w, uint8_t *wq, int64_t n,
                                 int64_t k, cudaStream_t stream)
{
    const int64_t nchunks = n * k / 4;
    set_max_carveout(quantize_q4_0_kernel);
    quantize_q4_0_kernel<<<grid_for(dev, nchunks, 256), 256, 0, stream>>>(
        reinterpret_cast<const float4 *>(w), wq, nchunks);
    return cudaGetLastError();
}

}  // namespace q8
