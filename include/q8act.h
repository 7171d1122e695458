/*
 * q8act.h -- C ABI of libq8act.so: a GB300 (sm_103a) implementation of the Q8_0 weight x
 * q8_1 activation block-quantized matmul of an LLM decoder.
 *
 * The operation, with the notation used throughout:
 *   W   Q8_0 weights, n rows ("out_f") of k/32 blocks ("in_f" = k).  A block is 34 bytes:
 *       a little-endian IEEE binary16 scale d_w at byte 0, then 32 int8 quants wq at bytes
 *       2..33.  Row r occupies bytes [r*row_bytes, (r+1)*row_bytes), row_bytes = k/32*34.
 *       (memra-engine 0.124.1 accprobe_bench.rs, synth_w_q8_0; memra-engine 0.113.0
 *       decode_kernel_census.rs, fn q8: row_bytes = in_f/32*(32+2).)
 *   x   f32 activations, m tokens x k, row-major.
 *   q8_1 quantization of x, per token t and block b of 32 values:
 *       amax = max|x|, d_a = amax/127 (f32, IEEE division), q = clamp(round(x/d_a), -127,
 *       127) with round half away from zero; a block with d_a == 0 gets q = 0.
 *       (memra-engine 0.81.0 f16_ffi.rs, try_f16_gemm / f16_act: the per-block formula
 *       amax/127, (v/d).round().clamp(-127,127), guarded by amax > 0; decode_kernel_census.rs
 *       fn q8: one i8 per column plus a per-32-block f32 scale.)
 *   y   f32 output, m x n, row-major:
 *       y[t][r] = sum_b d_w[r][b] * d_a[t][b] * D[t][r][b],
 *       D[t][r][b] = sum_{i<32} wq[r][32b+i] * xq[t][32b+i]   (exact int32, |D| <= 516128)
 *       with the scale fold in f32 (memra-engine 0.70.0 fp8_ffi.rs, try_fp8_gemm doc:
 *       y[m,out] = x[m,in] @ W^T; accprobe_bench.rs module doc: the MMQ floor folds the
 *       scales once per 32-wide k block).
 *
 * Conventions (as in the pages' extern "C" blocks, fp8_ffi.rs and f16_ffi.rs):
 *   - every pointer is a DEVICE pointer unless stated otherwise; the caller owns all memory;
 *   - `stream` is a cudaStream_t (NULL = legacy default stream); every call only enqueues
 *     work on it and returns without synchronizing (q8act_device_status excepted);
 *   - the return value is 0 on success, a negative Q8ACT_ERR_* code when the arguments are
 *     refused (nothing is launched), or Q8ACT_ERR_CUDA_BASE + cudaError_t when a CUDA call
 *     fails;
 *   - dimensions: k must be a positive multiple of 256 (every row then starts 16-byte
 *     aligned, which the bulk/TMA copies need); n >= 1; m as stated per call;
 *   - alignment: every pointer must be 16-byte aligned.
 *   - stream order: the calls keep the stream's order.  Most of their kernels are launched
 *     as programmatic dependents of the stream's previous kernel (they become resident early
 *     and wait for it to complete before touching memory), and every kernel lets the next
 *     one start early; a kernel that the caller launches after a call with programmatic
 *     stream serialization must therefore wait on its grid dependency (griddepcontrol.wait /
 *     cudaGridDependencySynchronize) before reading the call's outputs, as any such kernel
 *     must.  Ordinary launches, copies and events need nothing.
 *
 * Kernels time out instead of hanging: a pipeline wait that exceeds about two seconds makes
 * the kernel record an error in a device-side status word and return early.
 * q8act_device_status() reads and clears that word.  Before a CTA exits, its producer waits
 * (with the same limit) for every copy it issued into its shared memory; those copies are
 * built from tensor maps and sizes checked on the host, so they always complete, and a
 * timeout there is reported separately (Q8ACT_ERR_DRAIN_TIMEOUT).
 */
#ifndef Q8ACT_H
#define Q8ACT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define Q8ACT_OK 0
#define Q8ACT_ERR_NULL (-1)       /* a required pointer is NULL                        */
#define Q8ACT_ERR_DIMS (-2)       /* m, n or k out of range                            */
#define Q8ACT_ERR_ALIGN (-3)      /* a pointer is not 16-byte aligned                  */
#define Q8ACT_ERR_WORKSPACE (-4)  /* workspace missing or smaller than required        */
#define Q8ACT_ERR_DEVICE (-5)     /* current device is not an sm_103 (GB300) GPU       */
#define Q8ACT_ERR_TIMEOUT (-6)    /* a kernel gave up waiting (see q8act_device_status) */
#define Q8ACT_ERR_DRAIN_TIMEOUT (-7) /* a kernel gave up waiting for its own copies
                                        before exiting (see q8act_device_status)       */
#define Q8ACT_ERR_CUDA_BASE 1000  /* 1000 + cudaError_t                                */

/* Largest supported k (values per row). */
#define Q8ACT_MAX_K 65536
/* Largest token count of the GEMV: decode m = 1 and the m = K + 1 speculative-verify tier,
   i.e. the whole m < 16 range that the pages keep on the dp4a/MMVQ chain (fp8_ffi.rs and
   f16_ffi.rs module docs; m >= 16 is prefill). */
#define Q8ACT_GEMV_MAX_M 15
/* Largest number of weight matrices in one grouped GEMV call. */
#define Q8ACT_GEMV_MAX_GROUP 8

/* Library version, major*10000 + minor*100 + patch. */
int q8act_version(void);

/* Human-readable text for a return code (static storage, never NULL). */
const char *q8act_strerror(int rc);

/*
 * q8_1 activation quantizer (the decode-side activation form of decode_kernel_census.rs
 * fn q8: aq = one int8 per column, ad = per-32-block f32 scale).
 *   x   [m][k] f32 (input)          xq [m][k] int8 (output)      xd [m][k/32] f32 (output)
 *   m >= 1.  Bit-exact to the formula above (IEEE division, round half away from zero).
 */
int q8act_quantize_q8_1(const float *x, int8_t *xq, float *xd, int64_t m, int64_t k,
                        void *stream);

/*
 * q8_1 activation quantizer, MMQ (GEMM operand) layout.  Same quants and scales as
 * q8act_quantize_q8_1, laid out for the tensor-core GEMM, playing the role of the pages'
 * block_q8_1_mmq activation stream (accprobe_bench.rs, synth_act_q8_1):
 *   xqh [m][k] uint16: each quant stored as the IEEE binary16 encoding of the same integer
 *       (exact: |q| <= 127), the operand format of the f16 tensor-core pipe;
 *   xdt [k/32][ldm] f32: the scales transposed (block-major), ldm = q8act_mmq_ldm(m).
 */
int q8act_quantize_q8_1_mmq(const float *x, uint16_t *xqh, float *xdt, int64_t m, int64_t k,
                            void *stream);

/* Leading dimension (in floats) of the transposed scale array of the MMQ layout: m rounded
   up to a multiple of 4.  Returns 0 when m < 1. */
int64_t q8act_mmq_ldm(int64_t m);

/*
 * Q8_0 weight quantizer (load-time data preparation, the writer of the block format of
 * accprobe_bench.rs synth_w_q8_0):
 *   w  [n][k] f32 (input)      wq  n*k/32*34 bytes (output, Q8_0 blocks)
 *   per block: d = amax/127 (f32), quants q = clamp(round(w/d), -127, 127) computed with
 *   the f32 d, stored scale = binary16(d) rounded to nearest even; d == 0 gives q = 0.
 */
int q8act_quantize_q8_0(const float *w, void *wq, int64_t n, int64_t k, void *stream);

/*
 * Q8_0 x q8_1 GEMV, the decode ("mmvq") regime: Engine::qmatvec_mmvq_into in
 * decode_kernel_census.rs fn q8 (weights w, pre-quantized activation aq/ad, m tokens).
 *   w [n rows of Q8_0 blocks], xq [m][k] int8, xd [m][k/32] f32, y [m][n] f32 (overwritten)
 *   1 <= m <= Q8ACT_GEMV_MAX_M.  The m-token activation (1.25 * m * k bytes) is cached in
 *   shared memory beside at least two weight stages, which bounds k: 65536 at m = 1,
 *   18688 at m = 8, 10752 at m = 15; beyond that the call returns Q8ACT_ERR_DIMS.  The result for token t
 *   does not depend on m (the same
 *   operations in the same order for every m: the pages' decode == verify law,
 *   fp8_ffi.rs module doc and f16_ffi.rs module doc).
 */
int q8act_gemv_q8_0(const void *w, const int8_t *xq, const float *xd, float *y, int64_t m,
                    int64_t n, int64_t k, void *stream);

/*
 * Grouped GEMV: count (1..Q8ACT_GEMV_MAX_GROUP) Q8_0 weight matrices that share one
 * activation, streamed by one launch (the pages' fused multi-matrix decode GEMVs -- qkv with
 * gate, the stacked experts' gate+up -- for weights kept in separate buffers; decode_kernel_
 * census.rs).  w[i] is n[i] rows of Q8_0 blocks, y[i] [m][n[i]] f32 (overwritten); xq, xd,
 * m, k as for q8act_gemv_q8_0.  w, y and n are HOST arrays of count entries; each y[i] is
 * bitwise what q8act_gemv_q8_0 gives for w[i].
 */
int q8act_gemv_q8_0_group(const void *const *w, float *const *y, const int64_t *n, int count,
                          const int8_t *xq, const float *xd, int64_t m, int64_t k, void *stream);

/*
 * Bytes of the workspace region that lets a fused GEMM balance its work: when the 128 x 128
 * output tiles do not fill whole waves of the GPU's SMs, every CTA (one per SM) takes an
 * equal contiguous run of (tile, 256-wide k group) units, so that tiles at the runs' ends are
 * cut into k pieces; the pieces park partial tiles here, and the last piece to finish adds
 * them in a fixed order (the result does not depend on timing).  Room for two partial tiles
 * of 64 KiB per CTA for up to 160 CTAs, plus 160 x 16 counters.
 */
#define Q8ACT_GEMM_SPLIT_BYTES ((size_t)320 * 65536 + 160 * 64)

/*
 * Workspace bytes for the fused GEMMs on an m x k activation: the MMQ-layout quants and
 * scales plus Q8ACT_GEMM_SPLIT_BYTES.  A workspace of at least
 * q8act_gemm_workspace_bytes(m, k) - Q8ACT_GEMM_SPLIT_BYTES is accepted (every tile is
 * then done by one CTA over the whole of k).  Returns 0 when the dimensions are invalid (as
 * memra_fp8_blk_q8_0_bytes in fp8_ffi.rs returns 0 on bad dims).
 */
size_t q8act_gemm_workspace_bytes(int64_t m, int64_t k);

/*
 * Q8_0 x q8_1 GEMM, the prefill ("MMQ") regime, activation quantization fused into the call
 * (fp8_ffi.rs memra_fp8_pp_gemm: one C-ABI call, quantize + GEMM on one stream, caller-owned
 * workspace):
 *   w [n rows of Q8_0 blocks], x [m][k] f32, y [m][n] f32 (overwritten),
 *   ws: device workspace of q8act_gemm_workspace_bytes(m, k) bytes (at least that minus
 *   Q8ACT_GEMM_SPLIT_BYTES; see there).
 *   m >= 1 (the pages route m >= 16 here; smaller m is accepted).
 * Enqueued on `stream`: at most one memset of the split counters, the quantizer kernel, then
 * the GEMM kernel as a programmatic dependent of the quantizer (it starts its set-up while
 * the quantizer finishes and waits for it before reading the activation).  The call is
 * ordered after everything earlier on the stream, and later work on the stream is ordered
 * after the GEMM, exactly as for plain launches.  q8act_gemm_q8_0_repacked and
 * q8act_gemm_q8_0_noalloc do the same.
 */
int q8act_gemm_q8_0(const void *w, const float *x, float *y, int64_t m, int64_t n, int64_t k,
                    void *ws, size_t ws_bytes, void *stream);

/*
 * The GEMM on an activation already quantized by q8act_quantize_q8_1_mmq, so that one
 * quantization feeds several GEMMs (the grouped dispatch of f16_ffi.rs f16_act /
 * try_f16_gemm_pre, where a single activation conversion serves every GEMM of a group).
 *   xqh [m][k] binary16 quants, xdt [k/32][q8act_mmq_ldm(m)] f32 scales.
 */
int q8act_gemm_q8_0_preq(const void *w, const uint16_t *xqh, const float *xdt, float *y,
                         int64_t m, int64_t n, int64_t k, void *stream);

/*
 * The fused GEMM above for callers that cannot allocate device memory (an allocator's own
 * hooks, a serving loop that forbids allocation after start-up, a runtime that passes only
 * the buffers it owns).  No counterpart in the pages: it is an addition of this library.
 *   w, x, y, m, n, k, stream: as for q8act_gemm_q8_0; no workspace argument.
 * The activation quants and scales go into one fixed device array of Q8ACT_NOALLOC_WS_BYTES
 * that the library reserves on every GPU that loads it, until the process exits.  Returns
 * Q8ACT_ERR_WORKSPACE (nothing launched) when the quantized activation,
 * q8act_gemm_workspace_bytes(m, k) - Q8ACT_GEMM_SPLIT_BYTES bytes, exceeds that size (for
 * k = 4096: m up to 2891).  The split region is optional: when it fits in the rest of the
 * array too (m * k up to about 2M at k = 4096) the GEMM may take its balanced schedule,
 * otherwise every tile is done by one CTA.  The call never allocates or frees memory.  Its
 * first call on a device (and the first after that device's CUDA context was torn down and
 * created again) looks up the array's address (cudaGetSymbolAddress, with that device
 * current); make that first call before any stream capture.  All calls on a device share
 * the array and it keeps the previous call's contents; nothing in it needs to start at zero.
 * Calls that can overlap on the GPU (unordered streams) race on the array.
 */
#define Q8ACT_NOALLOC_WS_BYTES (24u << 20)
int q8act_gemm_q8_0_noalloc(const void *w, const float *x, float *y, int64_t m, int64_t n,
                            int64_t k, void *stream);

/*
 * Q8_0 -> row-major binary16 dequant (f16_ffi.rs memra_q8_0_dequant_f16, which takes out_f
 * and blocks per row; this call takes k = 32 * blocks per row):
 *   w [n rows of Q8_0 blocks] -> w16 [n][k] binary16, w16 = fp16_rn(f32(d_w) * q).
 *   The int8 part is exact in fp16; the only rounding is that of the product (f16_ffi.rs
 *   module doc, numeric-config paragraph).
 */
int q8act_dequant_q8_0_f16(const void *w, void *w16, int64_t n, int64_t k, void *stream);

/*
 * Load-time repack of Q8_0 weights for the tensor-core GEMM (the pages name such a repack,
 * build_q8_rp4 in the hybrid loader, without defining it; this one keeps the method exact):
 *   w [n rows of Q8_0 blocks] -> wq16 [n][k] binary16, wq16[r][32b+i] = q (exact, |q| <= 127),
 *                                wdt [k/32][ldn] f32, wdt[b][r] = f32(d_w[r][b]),
 *   ldn = q8act_repack_ldn(n); columns n..ldn-1 of wdt are not written.
 *   Output: 2 n k + 4 ldn k/32 bytes (2.125 bytes per weight, twice the Q8_0 bytes, like the
 *   pages' resident fp16 mirror, which however rounds d_w * q).  Caller-owned buffers,
 *   16-byte aligned.
 */
int q8act_repack_q8_0(const void *w, uint16_t *wq16, float *wdt, int64_t n, int64_t k,
                      void *stream);

/* Leading dimension (in floats) of the repacked scale plane: n rounded up to a multiple of 4
   (16-byte rows for the tensor-memory copies).  Returns 0 when n < 1. */
int64_t q8act_repack_ldn(int64_t n);

/*
 * The fused GEMM of q8act_gemm_q8_0 on repacked weights (q8act_repack_q8_0): the same
 * quantization, exact int32 block dots and f32 fold, with the weight tiles loaded by the
 * tensor-memory copy engine instead of being converted from 34-byte blocks in every call.
 *   wq16, wdt: the repack of an n-row weight; x, y, m, n, k, ws, ws_bytes, stream: as for
 *   q8act_gemm_q8_0.
 */
int q8act_gemm_q8_0_repacked(const uint16_t *wq16, const float *wdt, const float *x, float *y,
                             int64_t m, int64_t n, int64_t k, void *ws, size_t ws_bytes,
                             void *stream);

/*
 * Test hooks: export the exact per-block integer dots D[t][r][b] (int32, [m][n][k/32]) as
 * computed by the block-dot stage of the GEMV (1 <= m <= 15, routed exactly as
 * q8act_gemv_q8_0 routes: the tensor-core GEMV -- int8 mma.sync for m <= 8, binary16
 * mma.sync for m = 9..15 -- where its shared-memory plan fits, else the dp4a GEMV) or of the
 * GEMM (its tensor-core path; m >= 1, activation in the MMQ layout).  The fold is replaced by
 * a store of D; everything before it is the production code path.
 */
int q8act_debug_gemv_block_dots(const void *w, const int8_t *xq, int32_t *D, int64_t m,
                                int64_t n, int64_t k, void *stream);
int q8act_debug_gemm_block_dots(const void *w, const uint16_t *xqh, int32_t *D, int64_t m,
                                int64_t n, int64_t k, void *stream);

/* The repacked GEMM's block dots (same contract as q8act_debug_gemm_block_dots). */
int q8act_debug_gemm_repacked_block_dots(const uint16_t *wq16, const float *wdt,
                                         const uint16_t *xqh, int32_t *D, int64_t m, int64_t n,
                                         int64_t k, void *stream);

/*
 * The decode GEMV with the q8_1 quantization fused into the call (f32 activation in), like the
 * fused GEMM: the quantizer writes xq and xd into `ws`, then the GEMV of q8act_gemv_q8_0 runs
 * as a programmatic dependent of the quantizer, streaming its weights while the quantizer
 * finishes and waiting for it before reading the activation.  Bitwise the same y as
 * q8act_quantize_q8_1 followed by q8act_gemv_q8_0.  No counterpart in the pages (their decode
 * census passes a pre-quantized activation): an addition of this library for the decode path.
 *   w, y, m, n, k, stream: as for q8act_gemv_q8_0 (1 <= m <= 15); x [m][k] f32;
 *   ws: device workspace of at least q8act_gemv_workspace_bytes(m, k) bytes (16-byte aligned).
 * q8act_gemv_workspace_bytes returns 0 for invalid m or k.
 */
size_t q8act_gemv_workspace_bytes(int64_t m, int64_t k);
int q8act_gemv_q8_0_f32(const void *w, const float *x, float *y, int64_t m, int64_t n, int64_t k,
                        void *ws, size_t ws_bytes, void *stream);

/*
 * Q4_0 weights -- the GGUF Q4_0 block named by memra-engine 0.81.0 f16_ffi.rs
 * (memra_q4_0_dequant_f16: "GGUF Q4_0 18B blocks -> row-major fp16 mirror").  A row of k
 * weights is k/32 blocks of 18 bytes: the binary16 scale d (little endian), then 16 bytes
 * holding element i (i < 16) in the low nibble of byte i and element i + 16 in its high
 * nibble, each as q + 8; the weight is d * q with q in -8..7.  k: a positive multiple of 256
 * (rows are then 16-byte multiples); pointers 16-byte aligned; errors as for the Q8_0 calls.
 *
 * q8act_quantize_q4_0: data preparation (the pages give no Q4_0 quantizer): per block
 *   d = amax / 7 (f32), q = clamp(round_half_away(v / d), -8, 7), fp16(d) stored; a block
 *   whose d is 0 stores d = 0 and q = 0.  w [n][k] f32 -> wq, n * k / 32 * 18 bytes.
 * q8act_dequant_q4_0_f16: w16[r][32b+i] = fp16_rn(f32(d) * q) (the exact product, rounded
 *   once), row-major [n][k]; the f16_ffi.rs memra_q4_0_dequant_f16 call.
 * q8act_gemv_q4_0: y[t][r] = sum_b d_w * d_a * D with D the exact int32 dot of block b's
 *   4-bit values with the q8_1 quants, folded in f32 exactly as q8act_gemv_q8_0 folds
 *   (ascending blocks within each 256-wide group, then the fixed group order), so token t's
 *   result is bitwise the same for every m.  Arguments as q8act_gemv_q8_0; 1 <= m <= 15.
 * q8act_debug_gemv_q4_0_block_dots: that GEMV's exact block dots D[t][r][b] (test hook).
 */
int q8act_quantize_q4_0(const float *w, void *wq, int64_t n, int64_t k, void *stream);
int q8act_dequant_q4_0_f16(const void *w, void *w16, int64_t n, int64_t k, void *stream);
int q8act_gemv_q4_0(const void *w, const int8_t *xq, const float *xd, float *y, int64_t m,
                    int64_t n, int64_t k, void *stream);
int q8act_debug_gemv_q4_0_block_dots(const void *w, const int8_t *xq, int32_t *D, int64_t m,
                                     int64_t n, int64_t k, void *stream);

/*
 * K-quant weights -- the GGUF superblocks named by memra-engine 0.81.0 f16_ffi.rs
 * (memra_q6_K_dequant_f16: "GGUF Q6_K 210B superblocks", memra_q4_K_dequant_f16: "Q4_K 144B",
 * memra_q5_K_dequant_f16: "Q5_K 176B", each "-> row-major fp16 mirror").  A row of k weights
 * is k/256 superblocks; weight e (0..255) of a superblock:
 *   Q6_K (210 bytes): ql[128] at +0, qh[64] at +128, int8 scales[16] at +192, binary16 d at
 *     +208.  With e = 128h + 32g + l, its 6-bit code is the low (g < 2) or high (g >= 2) nibble
 *     of ql[64h + 32(g%2) + l] plus 16 times bits 2g..2g+1 of qh[32h + l]; its value is
 *     d * scales[e/16] * (code - 32).
 *   Q4_K (144 bytes): binary16 d at +0, binary16 dmin at +2, 12 scale bytes s at +4, qs[128]
 *     at +16.  Sub-block j = e/32 has a 6-bit scale and min: j < 4: s[j] & 63, s[j+4] & 63;
 *     j >= 4: (s[j+4] & 15) | (s[j-4] >> 6) << 4 and (s[j+4] >> 4) | (s[j] >> 6) << 4.  With
 *     e = 64g + 32u + l the code is nibble u of qs[32g + l]; the value is
 *     d * scale_j * code - dmin * min_j.
 *   Q5_K (176 bytes): as Q4_K with qh[32] at +16 and qs[128] at +48; bit j of qh[l] is the
 *     code's fifth bit (code += 16).
 * k: a positive multiple of 256; pointers 16-byte aligned; errors as for the Q8_0 calls.
 *
 * q8act_dequant_q{6,4,5}_k_f16: w16[r][e] = the binary16 nearest to the weight's exact value
 *   (ties to even), row-major [n][k].
 * q8act_gemv_q{6,4,5}_k: the decode GEMV on the q8_1 activation (xq [m][k] int8, xd [m][k/32]
 *   f32, y [m][n] f32 overwritten), 1 <= m <= Q8ACT_GEMV_KQ_MAX_M.  Per 32-wide activation
 *   block b (sub-block j of a superblock) exact integers and an f32 fold:
 *     Q6_K:        E_b = scales[2i] * sum_{16} (code - 32) xq + scales[2i+1] * sum_{16} (code - 32) xq,
 *                  y += (d * d_a) * E_b;
 *     Q4_K, Q5_K:  D_b = sum code * xq,  X_b = sum xq,
 *                  y += d_a * ((d * scale_j) * D_b - (dmin * min_j) * X_b);
 *   blocks ascending within a superblock, superblocks summed in a fixed order, so token t's
 *   result does not depend on m.  k is bounded by shared memory as for q8act_gemv_q8_0
 *   (Q8ACT_ERR_DIMS beyond it).
 * q8act_debug_gemv_q{6,4,5}_k_block_dots: that GEMV's exact integers per block, [m][n][k/32]
 *   int32 (E_b for Q6_K, D_b for Q4_K / Q5_K) (test hook).
 */
#define Q8ACT_GEMV_KQ_MAX_M 8
int q8act_dequant_q6_k_f16(const void *w, void *w16, int64_t n, int64_t k, void *stream);
int q8act_dequant_q4_k_f16(const void *w, void *w16, int64_t n, int64_t k, void *stream);
int q8act_dequant_q5_k_f16(const void *w, void *w16, int64_t n, int64_t k, void *stream);
int q8act_gemv_q6_k(const void *w, const int8_t *xq, const float *xd, float *y, int64_t m,
                    int64_t n, int64_t k, void *stream);
int q8act_gemv_q4_k(const void *w, const int8_t *xq, const float *xd, float *y, int64_t m,
                    int64_t n, int64_t k, void *stream);
int q8act_gemv_q5_k(const void *w, const int8_t *xq, const float *xd, float *y, int64_t m,
                    int64_t n, int64_t k, void *stream);
int q8act_debug_gemv_q6_k_block_dots(const void *w, const int8_t *xq, int32_t *D, int64_t m,
                                     int64_t n, int64_t k, void *stream);
int q8act_debug_gemv_q4_k_block_dots(const void *w, const int8_t *xq, int32_t *D, int64_t m,
                                     int64_t n, int64_t k, void *stream);
int q8act_debug_gemv_q5_k_block_dots(const void *w, const int8_t *xq, int32_t *D, int64_t m,
                                     int64_t n, int64_t k, void *stream);

/*
 * Synchronizes `stream`, then reads and clears the device-side status word that kernels set
 * when a pipeline wait times out.  Returns Q8ACT_OK, Q8ACT_ERR_DRAIN_TIMEOUT (a producer gave
 * up waiting for its own copies before its CTA exited), Q8ACT_ERR_TIMEOUT (a pipeline wait
 * gave up and the kernel returned early; its outputs are incomplete), or a CUDA error code.
 */
int q8act_device_status(void *stream);

/*
 * Test hook for the timeout path: launches one thread that waits, through the same bounded
 * mbarrier wait the pipelines use, on a barrier that nothing ever arrives on, with a limit of
 * limit_ns nanoseconds (1e3 .. 1e9) instead of the pipelines' two seconds.  The wait runs
 * out, records a pipeline timeout in the status word (q8act_device_status then returns
 * Q8ACT_ERR_TIMEOUT) and the kernel exits; nothing else is in flight, so the device stays
 * usable.  Returns Q8ACT_ERR_DIMS for a limit out of range.
 */
int q8act_debug_wait_timeout(int64_t limit_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* Q8ACT_H */
