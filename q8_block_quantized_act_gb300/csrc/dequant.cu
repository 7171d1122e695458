// dequant.cu -- Q8_0 -> row-major binary16 (memra-engine 0.81.0 f16_ffi.rs,
// memra_q8_0_dequant_f16: w16[r][32b+i] = fp16(d_w * q)).
//
// HBM-bound: 34 bytes in and 64 bytes out per block.  One lane produces one 16-byte output
// chunk (8 values), so a warp writes 512 contiguous bytes per step and reads the 272
// contiguous bytes of 8 blocks.  The int8 quants become binary16 exactly (|q| <= 127), and
// the product d_w * q is formed by the binary16 multiplier, which rounds the exact product
// once to nearest even -- the same value as rounding the (exact) f32 product.
#include "common.cuh"
#include "launch.h"

namespace q8 {
namespace {

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

__global__ void __launch_bounds__(256) dequant_q8_0_f16_kernel(const uint8_t *__restrict__ w,
                                                               uint4 *__restrict__ out,
                                                               int64_t nchunks)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < nchunks; c += stride) {
        const uint8_t *blk = w + (c >> 2) * Q8_0_BYTES;
        const int sub = (int)(c & 3);
        const uint16_t *p = reinterpret_cast<const uint16_t *>(blk);  // 2-byte aligned
        const uint32_t dbits = __ldg(p);
        const uint16_t *qp = reinterpret_cast<const uint16_t *>(blk + 2 + 8 * sub);
        const uint32_t q01 = (uint32_t)__ldg(qp + 0) | ((uint32_t)__ldg(qp + 1) << 16);
        const uint32_t q23 = (uint32_t)__ldg(qp + 2) | ((uint32_t)__ldg(qp + 3) << 16);
        const __half2 d2 = __half2half2(__ushort_as_half((unsigned short)dbits));
        __half2 h[4];
        bytes_to_half2x2(q01, h[0], h[1]);
        bytes_to_half2x2(q23, h[2], h[3]);
        uint4 o;
        uint32_t *ow = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half2 prod = __hmul2_rn(h[j], d2);
            ow[j] = *reinterpret_cast<const uint32_t *>(&prod);
        }
        __stcs(out + c, o);
    }
}

}  // namespace

cudaError_t launch_dequant_q8_0_f16(const DeviceInfo &dev, const uint8_t *w, uint16_t *w16,
                                    int64_t n, int64_t k, cudaStream_t stream)
{
    const int64_t nchunks = n * k / 8;
    int64_t grid = (nchunks + 255) / 256;
    const int64_t cap = (int64_t)dev.num_sms * 8;
    if (grid > cap) grid = cap;
    dequant_q8_0_f16_kernel<<<(int)grid, 256, 0, stream>>>(w, reinterpret_cast<uint4 *>(w16),
                                                           nchunks);
    return cudaGetLastError();
}

}  // namespace q8
