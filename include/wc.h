/*
 * wc.h -- C ABI of the GB300 quantized-gradient communication kernels.
 *
 * The hot path of ZeRO++ quantized gradient reduction (qgZ) with LoCo error
 * feedback, plus qwZ weight quantization and ZeRO-2 stochastic-rounding
 * gradient accumulation, as sm_103a CUDA kernels.  Several data-parallel
 * ranks are simulated as slices of one device allocation: the all-to-all of
 * the real system becomes the address arithmetic by which each reducing
 * kernel reads its chunks.
 *
 * Sources:
 *   "Merge LoCo with Zero++" (DeepSpeed PR #6730), Overview: error-feedback
 *     compensation of the 4-bit gradients before communication; review
 *     thread: two LoCo parameters, one error buffer per parameter.
 *   "ZeROPlusPlus.md" (notes on ZeRO++), §1.2 ZeRO++: qgZ -- block-based int4
 *     gradients exchanged by all-to-all in place of reduce-scatter, reduced
 *     in full precision, intra-node first and inter-node second; qwZ --
 *     block-based int8 weights for the forward all-gather.
 *   "Zero 2 #593" (llm.c), review of vector_add and of zero.cuh: bf16
 *     gradient accumulation summed in fp32 with stochastic rounding, and the
 *     zeroing of the source fused into the same kernel.
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers to memory the caller allocated and owns;
 *     the library allocates nothing, frees nothing and never synchronizes
 *     the host (the debugging call wc_checked_violations excepted).  Every
 *     call is asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and reads/writes its buffers only in stream order.
 *   - Kernels launch on the calling thread's current device: the pointers
 *     and the stream must belong to it.
 *   - bf16 values are passed as uint16_t bit patterns.
 *   - Every device pointer must be 16-byte aligned (WC_EALIGN otherwise).
 *   - Buffers must not overlap unless an entry point says so.
 *   - Inputs must be finite (not checked).
 *   - Return value: WC_OK, or a negative WC_E* code with nothing launched
 *     (argument errors) or with the launch failed (WC_ECUDA).  The message
 *     of the calling thread's last failure is returned by wc_last_error().
 *   - A size of zero elements is a valid call that launches nothing.
 *
 * Arithmetic (shared with the reference definitions): IEEE binary32 with one
 * rounding per operation (no contraction into fused multiply-adds, no flush
 * to zero); bf16 results are rounded to nearest even unless stated.
 */
#ifndef WC_H
#define WC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define WC_API __attribute__((visibility("default")))
#else
#define WC_API
#endif

/* status codes */
#define WC_OK 0
#define WC_EINVAL (-1)   /* null pointer, bad size or divisibility, bad block */
#define WC_EALIGN (-2)   /* a pointer is not 16-byte aligned */
#define WC_ERANGE (-3)   /* a size exceeds what the kernel indexes */
#define WC_ECUDA (-4)    /* the kernel launch failed; see wc_last_error() */

/* output element types for the reductions */
#define WC_F32 0
#define WC_BF16 1

/*
 * wc_ef_quant_int4 -- error-feedback compensation and int4 quantization of
 * every simulated rank's gradient (LoCo on qgZ).
 *
 * For each rank r in [0, R) and element x of its gradient g_r (N elements):
 *   c = g + s * e                               (fp32; e = ef[r][x])
 * then per block of B consecutive elements of c, m = max |c|:
 *   m <  7 * 2^-126: scale = 0, q = 0           (scale would not be normal)
 *   else:            scale = m / 7, inv = 7 / m, q = clamp(rint(c*inv), -7, 7)
 * and, when ef != NULL,
 *   e <- beta * e + (1 - beta) * (c - q * scale)
 * with 1 - beta formed once in fp32.  ef == NULL quantizes g alone (s and
 * beta are ignored, no error is stored).
 *
 * Send order.  Each rank's N elements are R slices of S = N / R; slice k is
 * reduced on rank k.  With G groups of L = R / G ranks (rank k = g*L + l) the
 * codes of slice g'*L + l are written at chunk position l*G + g', so the
 * chunk bound for local rank l of the first (intra-group) hop is one run of
 * G*S elements.  G = 1 is the identity (flat all-to-all).
 *
 * g      : [R][N] bf16, read.
 * ef     : [R][N] fp32, read and written in place, gradient order; or NULL.
 * codes  : [R][N/2] bytes, written, send order.  Code of position p is a
 *          4-bit two's-complement nibble: low nibble of byte p/2 for even p,
 *          high nibble for odd p.  Values in [-7, 7].
 * scales : [R][N/B] fp32, written, send order (one per block of codes).
 * Requires R >= 1, G >= 1, G | R, R | N, B | N/R, and
 * B in {32, 64, 128, 256, 512, 1024}.  R*N < 2^32 (WC_ERANGE otherwise).
 */
WC_API int wc_ef_quant_int4(const uint16_t *g, float *ef, uint8_t *codes,
                            float *scales, int64_t N, int R, int G, int B,
                            float err_scale, float err_beta, void *stream);

/*
 * wc_ef_quant_int4_bf16ef -- wc_ef_quant_int4 with the error buffer stored in
 * bf16 instead of fp32, halving the extra memory LoCo costs ("Merge LoCo with
 * Zero++", Overview) and the buffer's share of the traffic (6.5 instead of
 * 10.5 bytes per element at B = 256).  The stored error is widened exactly,
 * all arithmetic is the fp32 chain of wc_ef_quant_int4, and only the new
 * error is rounded to the nearest bf16 (ties to even) when stored.
 * ef16 : [R][N] bf16 bit patterns, read and written in place (not NULL).
 * Everything else as wc_ef_quant_int4.
 */
WC_API int wc_ef_quant_int4_bf16ef(const uint16_t *g, uint16_t *ef16,
                                   uint8_t *codes, float *scales, int64_t N,
                                   int R, int G, int B, float err_scale,
                                   float err_beta, void *stream);

/*
 * wc_ef_quant_int4_int8ef -- wc_ef_quant_int4 with the error buffer stored in
 * int8, a quarter of the fp32 buffer's memory ("Merge LoCo with Zero++",
 * Overview: LoCo's cost is the buffer's extra memory): 4.5 instead of 10.5
 * bytes per element at B = 256.  The error of each block of B gradient
 * elements (gradient order) is B int8 codes and one fp32 scale, written by
 * the block rule of wc_qwz_quant_int8 (scale = m / 127, codes
 * rint(e * 127 / m), zero block when m < 127 * 2^-126) applied to the new
 * error, and read back as code * scale (one rounding); all other arithmetic
 * is the fp32 chain of wc_ef_quant_int4.
 * ef8        : [R][N] int8 codes, read and written in place (not NULL).
 * ef8_scales : [R][N/B] fp32, read and written in place (not NULL).
 * A zero buffer is all-zero codes and scales.  Everything else as
 * wc_ef_quant_int4.
 */
WC_API int wc_ef_quant_int4_int8ef(const uint16_t *g, int8_t *ef8,
                                   float *ef8_scales, uint8_t *codes,
                                   float *scales, int64_t N, int R, int G,
                                   int B, float err_scale, float err_beta,
                                   void *stream);

/*
 * wc_dequant_reduce -- dequantize and reduce in full precision: the flat
 * reduce after the all-to-all, or the second hop of the hierarchical reduce.
 *
 * Every destination k in [0, R) computes S = N / R outputs
 *   out[k][i] = out_scale * (d_0 + d_1 + ... + d_{n-1})   (fp32, left to right
 *                                                          from +0)
 * where d_j = code * scale of source j, and then stores it as fp32
 * (out_dtype WC_F32) or rounds it to bf16 (WC_BF16).  out_scale = 1 gives the
 * sum, 1/R the average.
 *   G == 1 (flat): the sources are the R ranks' send buffers produced by
 *     wc_ef_quant_int4 ([R][N/2] codes, [R][N/B] scales); source j of
 *     destination k is chunk k of rank j (n = R).
 *   G > 1 (second hop): the sources are the first hop's outputs produced by
 *     wc_dequant_reduce_requant ([R][G*S/2] codes, [R][G*S/B] scales; unit
 *     u = g*L + l); destination k = g*L + l adds sub-slice g of units
 *     (j, l) for j = 0..G-1 (n = G).
 * out : [R][S] fp32 or bf16, written, destination order (shard k of the
 *       ZeRO partition is out[k]).
 * Requires the same sizes as wc_ef_quant_int4.
 */
WC_API int wc_dequant_reduce(const uint8_t *codes, const float *scales,
                             int64_t N, int R, int G, int B, float out_scale,
                             void *out, int out_dtype, void *stream);

/*
 * wc_dequant_reduce_requant -- first (intra-group) hop of the hierarchical
 * reduce, with the partial sums requantized to int4.
 *
 * Unit (g, l), local rank l of group g, receives from the L ranks g*L + l'
 * of its group their chunk l (send positions l*G .. l*G+G-1: G sub-slices of
 * S).  For each sub-slice g' and element i it adds the L dequantized values
 * in the order l' = 0..L-1 (fp32 from +0), then requantizes each block of B
 * partial sums with the rule of wc_ef_quant_int4 (no error feedback).
 * codes, scales : the send buffers of wc_ef_quant_int4 with the same
 *                 (N, R, G, B), read.
 * out_codes     : [R][G*S/2] bytes, written; unit u = g*L + l holds its G
 *                 sub-slices in order g' = 0..G-1 (sub-slice g' is bound for
 *                 rank g'*L + l).
 * out_scales    : [R][G*S/B] fp32, written, same order.
 * Requires the sizes of wc_ef_quant_int4 and G*N < 2^32.  G = 1 is allowed:
 * it requantizes the flat reduce.
 */
WC_API int wc_dequant_reduce_requant(const uint8_t *codes, const float *scales,
                                     int64_t N, int R, int G, int B,
                                     uint8_t *out_codes, float *out_scales,
                                     void *stream);

/*
 * wc_dequant_reduce_requant_ef -- the first hop with error feedback on its
 * requantization.  "Merge LoCo with Zero++" (review thread) keeps the error
 * buffers on each parameter as `inter_ef_buf`, the buffer of the inter-node
 * message; here every requantized value p keeps an fp32 error e1:
 *   c = p + s * e1;  q, scale = Q4(c) per block;
 *   e1 <- beta * e1 + (1 - beta) * (c - q * scale)   (1 - beta formed in fp32)
 * ef1 : [R][G*S] fp32 in the layout of out_codes (unit u = g*L + l holds G*S
 *       values), read and written in place, not NULL.  Start it at zero.
 * Everything else as wc_dequant_reduce_requant.
 */
WC_API int wc_dequant_reduce_requant_ef(const uint8_t *codes, const float *scales,
                                        int64_t N, int R, int G, int B,
                                        uint8_t *out_codes, float *out_scales,
                                        float *ef1, float err_scale,
                                        float err_beta, void *stream);

/*
 * wc_qgz_step_fused -- the whole flat step (G = 1) in one kernel: for every
 * destination block it runs wc_ef_quant_int4's arithmetic on the R ranks in
 * rank order and adds their dequantized values as wc_dequant_reduce does, so
 * out, ef, codes and scales are bit-identical to calling the two in
 * sequence, while the codes never have to be read back from memory.
 * ("ZeROPlusPlus.md" §1.2: qgZ with CUDA kernel fusion; with every rank in
 * one GPU's memory the fusion can span the all-to-all.)
 * g, ef    : as wc_ef_quant_int4 (ef may be NULL).
 * codes, scales : the send buffers as wc_ef_quant_int4 writes them with G = 1,
 *           or both NULL to skip writing them.
 * out      : [R][S] fp32 or bf16 (out_dtype), destination order.
 * Requires the sizes of wc_ef_quant_int4 with G = 1 and B >= 128.
 */
WC_API int wc_qgz_step_fused(const uint16_t *g, float *ef, uint8_t *codes,
                             float *scales, int64_t N, int R, int B,
                             float err_scale, float err_beta, float out_scale,
                             void *out, int out_dtype, void *stream);

/*
 * wc_qgz_step_fused_bf16ef / _int8ef -- wc_qgz_step_fused with the error
 * buffer of wc_ef_quant_int4_bf16ef (ef16: [R][N] bf16, in place) or of
 * wc_ef_quant_int4_int8ef (ef8: [R][N] int8 codes, ef8_scales: [R][N/B]
 * fp32, gradient order, in place): out, codes, scales and the buffer are
 * bit-identical to calling that quantization and wc_dequant_reduce in
 * sequence ("Merge LoCo with Zero++", Overview: the error buffer's memory is
 * LoCo's cost).  The buffer is required (no NULL); the other arguments and
 * requirements are wc_qgz_step_fused's.
 */
WC_API int wc_qgz_step_fused_bf16ef(const uint16_t *g, uint16_t *ef16, uint8_t *codes,
                                    float *scales, int64_t N, int R, int B,
                                    float err_scale, float err_beta, float out_scale,
                                    void *out, int out_dtype, void *stream);
WC_API int wc_qgz_step_fused_int8ef(const uint16_t *g, int8_t *ef8, float *ef8_scales,
                                    uint8_t *codes, float *scales, int64_t N, int R,
                                    int B, float err_scale, float err_beta,
                                    float out_scale, void *out, int out_dtype,
                                    void *stream);

/*
 * wc_qgz_first_hop_fused -- the hierarchical step's first stage in one
 * kernel: every rank's error-feedback quantization (wc_ef_quant_int4 with
 * G groups) and the first, intra-group hop (wc_dequant_reduce_requant)
 * together.  For every block of the first hop's output it runs
 * wc_ef_quant_int4's arithmetic on the L ranks of the unit's group, in
 * local-rank order, on the blocks those ranks send to the unit, and adds
 * their dequantized values from +0 as the first hop does before
 * requantizing; so out_codes, out_scales, ef, codes and scales are
 * bit-identical to calling the two in sequence, while the ranks' codes are
 * never read back from memory.  ("ZeROPlusPlus.md" §1.2: qgZ reduces
 * intra-node first, with CUDA kernel fusion; with every rank in one GPU's
 * memory the fusion can span the intra-group all-to-all.)  The second hop is
 * wc_dequant_reduce with G groups on out_codes and out_scales.
 * g, ef    : as wc_ef_quant_int4 (ef may be NULL).
 * codes, scales : the ranks' send buffers as wc_ef_quant_int4 writes them,
 *           or both NULL to skip writing them.
 * out_codes, out_scales : the first hop's output, as
 *           wc_dequant_reduce_requant writes it.
 * ef1      : NULL, or the first hop's own error buffer [G*N] fp32 (in
 *           place, output order), applied to the requantization as
 *           wc_dequant_reduce_requant_ef does, with the same err_scale and
 *           err_beta as the ranks' buffers ("Merge LoCo with Zero++",
 *           review thread: the inter-node message's error buffer).
 * Requires the sizes of wc_dequant_reduce_requant and B >= 128; every
 * pointer 16-byte aligned.
 */
WC_API int wc_qgz_first_hop_fused(const uint16_t *g, float *ef, uint8_t *codes,
                                  float *scales, int64_t N, int R, int G, int B,
                                  float err_scale, float err_beta,
                                  uint8_t *out_codes, float *out_scales,
                                  float *ef1, void *stream);

/*
 * wc_qgz_first_hop_fused_bf16ef / _int8ef -- wc_qgz_first_hop_fused with the
 * ranks' error buffer of wc_ef_quant_int4_bf16ef (ef16) or of
 * wc_ef_quant_int4_int8ef (ef8, ef8_scales), as in wc_qgz_step_fused_bf16ef
 * / _int8ef; bit-identical to that quantization followed by
 * wc_dequant_reduce_requant (or wc_dequant_reduce_requant_ef with ef1).  The
 * buffer is required; the other arguments are wc_qgz_first_hop_fused's.
 */
WC_API int wc_qgz_first_hop_fused_bf16ef(const uint16_t *g, uint16_t *ef16,
                                         uint8_t *codes, float *scales, int64_t N,
                                         int R, int G, int B, float err_scale,
                                         float err_beta, uint8_t *out_codes,
                                         float *out_scales, float *ef1, void *stream);
WC_API int wc_qgz_first_hop_fused_int8ef(const uint16_t *g, int8_t *ef8,
                                         float *ef8_scales, uint8_t *codes,
                                         float *scales, int64_t N, int R, int G, int B,
                                         float err_scale, float err_beta,
                                         uint8_t *out_codes, float *out_scales,
                                         float *ef1, void *stream);

/*
 * wc_qwz_quant_int8 -- qwZ block weight quantization.
 * Per block of B weights (bf16 widened exactly to fp32), m = max |w|:
 *   m < 127 * 2^-126: scale = 0, q = 0
 *   else: scale = m / 127, inv = 127 / m, q = clamp(rint(w * inv), -127, 127)
 * w : [n] bf16, read.  codes : [n] int8, written.  scales : [n/B] fp32.
 * Requires B | n and B in {32, 64, ..., 4096} (powers of two).  n < 2^32.
 */
WC_API int wc_qwz_quant_int8(const uint16_t *w, int8_t *codes, float *scales,
                             int64_t n, int B, void *stream);

/*
 * wc_qwz_quant_replica_int8 -- wc_qwz_quant_int8 that also writes, in the same
 * pass, the bf16 weights the codes stand for: replica = bf16_rn(q * scale),
 * exactly what wc_qwz_dequant_int8 returns for these codes.  This is the
 * copy a node keeps after the quantized forward all-gather ("ZeROPlusPlus.md"
 * §1.2: the hierarchical partition keeps a full model copy inside each node),
 * written without re-reading the codes: 5 bytes per weight instead of 6.
 * replica : [n] bf16, written.  Everything else as wc_qwz_quant_int8.
 */
WC_API int wc_qwz_quant_replica_int8(const uint16_t *w, int8_t *codes,
                                     float *scales, uint16_t *replica,
                                     int64_t n, int B, void *stream);

/*
 * wc_qwz_dequant_int8 -- back to bf16: w' = bf16_rn(q * scale).
 * codes : [n] int8, scales : [n/B] fp32, read.  w_out : [n] bf16, written.
 * Same size rules as wc_qwz_quant_int8.
 */
WC_API int wc_qwz_dequant_int8(const int8_t *codes, const float *scales,
                               uint16_t *w_out, int64_t n, int B, void *stream);

/*
 * wc_sr_accumulate_bf16 -- ZeRO-2 gradient accumulation with stochastic
 * rounding and the source zeroed in the same kernel.
 * For i in [0, n):
 *   x = f32(dst[i]) + f32(src[i])                       (fp32)
 *   r = mix(key ^ i) & 0xFFFF,  key = mix(mix(seed) ^ step),
 *       mix(z) = fmix32(z + 0x9E3779B9)  (MurmurHash3's 32-bit finalizer)
 *   dst[i] = upper half of (bits(x) + r)                 (rounds the
 *            magnitude up with probability (low 16 bits of x) / 65536)
 *   src[i] = 0
 * Unbiased: the mean over r is exactly x.  Infinities pass through; sums
 * within one bf16 step of the largest finite value may round to infinity.
 * dst, src : [n] bf16, read and written in place; they must not overlap.
 * Requires n < 2^32 (the index is 32-bit).
 */
WC_API int wc_sr_accumulate_bf16(uint16_t *dst, uint16_t *src, int64_t n,
                                 uint32_t seed, uint32_t step, void *stream);

/*
 * wc_checked_violations -- a debugging aid with no counterpart on the pages.
 * A library built with WC_CHECKED=1 compares every global load and store of
 * every kernel with the extent of its buffer, as the call's sizes define it,
 * and skips any access that would fall outside (it never traps).  This call
 * returns the number of accesses skipped since the last reset, summed over
 * the kernel files: 0 means every launch stayed inside its buffers.  When it
 * is not 0, wc_last_error() names the source file and line of one of them.
 * flags: WC_CHECK_RESET clears the records after reading them;
 *        WC_CHECK_PROBE first launches, in each kernel file, a one-thread
 *        kernel that fails one comparison without touching memory, so the
 *        count includes one violation per kernel file (a self-test).
 * Reads device memory synchronously: call it once the launches it should
 * cover have completed (synchronize their streams first).
 * Returns WC_EINVAL in an ordinary build or for unknown flags, WC_ECUDA if
 * the read fails.
 */
#define WC_CHECK_RESET 1
#define WC_CHECK_PROBE 2
WC_API int wc_checked_violations(int flags);

/* Message describing the calling thread's last failed call ("" if none). */
WC_API const char *wc_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
WC_API int wc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* WC_H */
