// launch.h -- internal launchers of libq8act (host side).  Arguments are validated by the
// C-ABI layer (api.cu) before any of these is called; each returns the launch status.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace q8 {

struct DeviceInfo {
    int device;
    int num_sms;
    size_t max_smem_optin;
    int *status;  // device address of the status word
};

cudaError_t launch_quantize_q8_1(const DeviceInfo &dev, const float *x, int8_t *xq, float *xd,
                                 int64_t m, int64_t k, cudaStream_t stream);
cudaError_t launch_quantize_q8_1_mmq(const DeviceInfo &dev, const float *x, uint16_t *xqh,
                                     float *xdt, int64_t m, int64_t k, int64_t ldm,
                                     cudaStream_t stream);
cudaError_t launch_quantize_q8_0(const DeviceInfo &dev, const float *w, uint8_t *wq, int64_t n,
                                 int64_t k, cudaStream_t stream);
cudaError_t launch_dequant_q8_0_f16(const DeviceInfo &dev, const uint8_t *w, uint16_t *w16,
                                    int64_t n, int64_t k, cudaStream_t stream);
cudaError_t launch_repack_q8_0(const DeviceInfo &dev, const uint8_t *w, uint16_t *wq16, float *wdt,
                               int64_t ldn, int64_t n, int64_t k, cudaStream_t stream);
// Q4_0 (GGUF 18-byte blocks): the writer (data preparation), the fp16 dequant, the GEMV.
cudaError_t launch_quantize_q4_0(const DeviceInfo &dev, const float *w, uint8_t *wq, int64_t n,
                                 int64_t k, cudaStream_t stream);
cudaError_t launch_dequant_q4_0_f16(const DeviceInfo &dev, const uint8_t *w, uint16_t *w16,
                                    int64_t n, int64_t k, cudaStream_t stream);
bool gemv_q4_0_supported(const DeviceInfo &dev, int64_t m, int64_t k);
cudaError_t launch_gemv_q4_0(const DeviceInfo &dev, const uint8_t *w, const int8_t *xq,
                             const float *xd, float *y, int32_t *dots, int64_t m, int64_t n,
                             int64_t k, cudaStream_t stream);
// The tensor-core Q4_0 GEMV for 5 <= m <= 16 (bitwise the same results as launch_gemv_q4_0).
bool gemv_q4_0_mma_supported(const DeviceInfo &dev, int64_t m, int64_t k);
cudaError_t launch_gemv_q4_0_mma(const DeviceInfo &dev, const uint8_t *w, const int8_t *xq,
                                 const float *xd, float *y, int32_t *dots, int64_t m, int64_t n,
                                 int64_t k, cudaStream_t stream);

// K-quant superblocks (fmt 6: Q6_K, 4: Q4_K, 5: Q5_K): the fp16 mirror and the GEMV
// (1 <= m <= 8; dots != nullptr stores the exact per-32-block integers instead of folding).
cudaError_t launch_dequant_kq_f16(const DeviceInfo &dev, int fmt, const uint8_t *w, uint16_t *w16, int64_t n,
                                  int64_t k, cudaStream_t stream);
bool gemv_kq_supported(const DeviceInfo &dev, int fmt, int64_t m, int64_t k);
// The tensor-core K-quant GEMV (2 <= m <= 8, rows a multiple of 16 bytes); the same bits as
// the dp4a kernel, which launch_gemv_kq routes to otherwise.
bool gemv_kq_mma_supported(const DeviceInfo &dev, int fmt, int64_t m, int64_t k);
cudaError_t launch_gemv_kq_mma(const DeviceInfo &dev, int fmt, const uint8_t *w, const int8_t *xq, const float *xd,
                               float *y, int32_t *dots, int64_t m, int64_t n, int64_t k, cudaStream_t stream);
cudaError_t launch_gemv_kq(const DeviceInfo &dev, int fmt, const uint8_t *w, const int8_t *xq, const float *xd,
                           float *y, int32_t *dots, int64_t m, int64_t n, int64_t k, cudaStream_t stream);

// GEMV: returns cudaErrorInvalidValue when m*k is too large for the shared-memory plan.
bool gemv_supported(const DeviceInfo &dev, int64_t m, int64_t k);
cudaError_t launch_gemv_q8_0_group(const DeviceInfo &dev, const uint8_t *const *w, float *const *y,
                                   const int64_t *n, int count, const int8_t *xq, const float *xd,
                                   int64_t m, int64_t k, cudaStream_t stream);
// The tensor-core GEMV for 2 <= m <= 16 (bitwise the same results as launch_gemv_q8_0).
bool gemv_mma_supported(const DeviceInfo &dev, int64_t m, int64_t k);
// Every GEMV launch is a programmatic dependent of the stream's previous kernel.  pdl: that
// kernel is the call's own q8_1 quantizer producing xq / xd, and the GEMV streams weights
// while it finishes; otherwise the GEMV waits for it before touching memory.
cudaError_t launch_gemv_q8_0_mma(const DeviceInfo &dev, const uint8_t *w, const int8_t *xq, const float *xd,
                                 float *y, int32_t *dots, int64_t m, int64_t n, int64_t k, cudaStream_t stream,
                                 bool pdl = false);
// The grouped GEMV (several weight matrices, one activation) on the tensor-core kernel, for the
// m that gemv_mma_supported accepts (bitwise the same results as launch_gemv_q8_0_group).
cudaError_t launch_gemv_q8_0_group_mma(const DeviceInfo &dev, const uint8_t *const *w, float *const *y,
                                       const int64_t *n, int count, const int8_t *xq, const float *xd,
                                       int64_t m, int64_t k, cudaStream_t stream);
cudaError_t launch_gemv_q8_0(const DeviceInfo &dev, const uint8_t *w, const int8_t *xq,
                             const float *xd, float *y, int32_t *dots, int64_t m, int64_t n,
                             int64_t k, cudaStream_t stream, bool pdl = false);

// GEMM on MMQ-layout activations (xqh binary16 quants [m][k], xdt f32 scales [k/32][ldm]).
// With dots != nullptr the fold is replaced by a store of the block dots D[m][n][k/32].
// Bytes of the optional workspace region that lets a GEMM take the balanced schedule (tiles
// cut into k pieces at the ends of equal per-CTA runs of work).
size_t gemm_split_bytes();
// pdl: launch as a programmatic dependent of the stream's previous kernel, which must be the
// MMQ quantizer producing xqh / xdt (it lets the GEMM start early; the GEMM waits for it
// before reading them), with gemm_prepare_split already enqueued before that quantizer.
// Without pdl the launch is ordinary and zeroes the split counters itself.
cudaError_t gemm_prepare_split(const DeviceInfo &dev, int64_t m, int64_t n, int64_t k, bool repacked,
                               void *split_ws, size_t split_bytes, cudaStream_t stream);
cudaError_t launch_gemm_q8_0(const DeviceInfo &dev, const uint8_t *w, const uint16_t *xqh,
                             const float *xdt, float *y, int32_t *dots, int64_t m, int64_t n,
                             int64_t k, int64_t ldm, void *split_ws, size_t split_bytes, bool pdl,
                             cudaStream_t stream);
cudaError_t launch_gemm_q8_0_repacked(const DeviceInfo &dev, const uint16_t *wq16, const float *wdt,
                                      int64_t ldn, const uint16_t *xqh, const float *xdt, float *y,
                                      int32_t *dots, int64_t m, int64_t n, int64_t k, int64_t ldm,
                                      void *split_ws, size_t split_bytes, bool pdl, cudaStream_t stream);

}  // namespace q8
