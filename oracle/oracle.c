/*
 * oracle.c -- plain, slow, single-threaded CPU statement of what the
 * quantized-gradient hot path computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library or its
 * Python binding) links, loads or calls this file.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg use it, as the independent
 * reference the GPU kernels are compared against.
 *
 * Sources of the definitions:
 *   [LoCo]  "Merge LoCo with Zero++" (DeepSpeed pull request #6730), Overview:
 *           error-feedback compensation is applied to the 4-bit gradients
 *           before they are communicated; it costs extra GPU memory (the
 *           error buffer) and no extra time.  Review thread: LoCo takes two
 *           parameters and keeps one error buffer per parameter.
 *   [qgZ]   "ZeROPlusPlus.md" (notes on the ZeRO++ paper), §1.2 ZeRO++, third
 *           item (quantized gradient communication): block-based int4
 *           quantization, an all-to-all in place of reduce-scatter, the
 *           reduction itself in full precision, intra-node before inter-node.
 *   [qwZ]   same page, §1.2, first item: block-based fp16 -> int8 weight
 *           quantization before the forward all-gather.
 *   [SR]    "Zero 2 #593" (llm.c pull request), review of llmc/cuda_utils.cuh
 *           (vector_add): dst and src are summed in fp32 and rounded back to
 *           bf16 stochastically so the accumulation stays correct in
 *           expectation; review of llmc/zero.cuh: the memset that zeroes src
 *           after the add belongs inside the same kernel.
 *
 * Where the pages leave a step open the reading taken is stated at that step.
 *
 * Arithmetic: IEEE-754 binary32, one rounding per operation, round to nearest
 * even, no fused multiply-add (build with -ffp-contract=off), no flush to
 * zero.  binary32 is the precision the method's own decisions are made in
 * (which integer code a value gets), so the oracle takes those decisions in
 * the same precision; fp64 appears nowhere in here.
 *
 * Parity status of every function: pinned by the CPU tests (closed forms,
 * exhaustive small cases, exact-rational brute force, invariants).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_EXPORT __attribute__((visibility("default")))

/*
 * Per-block scratch.  The functions that quantize a block at a time keep the
 * block's values on the stack in arrays of ORC_MAX_BLOCK elements, so each
 * of them first checks B itself: a block size outside [1, ORC_MAX_BLOCK] is
 * refused with ORC_EBLOCK before anything is written.  They return 0 on
 * success.
 */
#define ORC_MAX_BLOCK 8192
#define ORC_EBLOCK (-1)

static int orc_block_ok(int B) { return B >= 1 && B <= ORC_MAX_BLOCK; }

ORC_EXPORT int orc_max_block(void) { return ORC_MAX_BLOCK; }

/* ------------------------------------------------------------------------ */
/* bfloat16 <-> binary32                                                      */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float bits_f32(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

/* A bfloat16 is the upper half of a binary32, so widening is exact. */
ORC_EXPORT float orc_bf16_to_f32(uint16_t h)
{
    return bits_f32((uint32_t)h << 16);
}

/* Round a binary32 to the nearest bfloat16, ties to even (the IEEE default
 * rounding, applied at bit 16).  NaN stays NaN: its upper half is kept and
 * the quiet bit is set, so the payload can never round into an infinity. */
ORC_EXPORT uint16_t orc_f32_to_bf16_rne(float x)
{
    uint32_t u = f32_bits(x);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
        upper += 1u;              /* a carry into the exponent is correct */
    return (uint16_t)upper;
}

/* ------------------------------------------------------------------------ */
/* Symmetric absmax block quantization                                        */
/* ------------------------------------------------------------------------ */

/*
 * Quantize one block x[0..B) to integers in [-qmax, qmax] with one binary32
 * scale, the block-based quantization of [qgZ] (qmax = 7, int4) and [qwZ]
 * (qmax = 127, int8):
 *   m     = max |x_i|
 *   scale = m / qmax                (IEEE division)
 *   inv   = qmax / m                (IEEE division)
 *   q_i   = clamp(rint(x_i * inv), -qmax, qmax)   (rint: ties to even)
 * Readings: a block whose scale would not be a normal binary32, i.e.
 * m < qmax * 2^-126 (this includes all-zero and subnormal blocks), gets scale
 * 0 and all-zero codes; above that bound scale is normal and inv = qmax / m
 * <= 2^126 is finite (with the bound at 2^-126 itself, qmax / m overflows to
 * infinity for m just above 2^-126).  The code is x_i * inv rounded once,
 * never x_i / scale; -qmax-1 is never produced.
 */
ORC_EXPORT void orc_quant_block(const float *x, int B, int qmax,
                                int8_t *q, float *scale_out)
{
    float m = 0.0f;
    for (int i = 0; i < B; ++i) {
        float a = fabsf(x[i]);
        if (a > m) m = a;
    }
    float fq = (float)qmax;
    if (m < fq * FLT_MIN) {          /* qmax * 2^-126 is exact */
        for (int i = 0; i < B; ++i) q[i] = 0;
        *scale_out = 0.0f;
        return;
    }
    float scale = m / fq;
    float inv = fq / m;
    for (int i = 0; i < B; ++i) {
        float t = x[i] * inv;
        float r = rintf(t);
        if (r > fq) r = fq;
        if (r < -fq) r = -fq;
        q[i] = (int8_t)r;
    }
    *scale_out = scale;
}

/* Dequantized value of one code: the code times the block scale, one
 * rounding.  Sender (error update) and receiver (reduction) use this same
 * value. */
ORC_EXPORT float orc_dequant(int q, float scale)
{
    return (float)q * scale;
}

/* ------------------------------------------------------------------------ */
/* int4 packing                                                               */
/* ------------------------------------------------------------------------ */

/* Reading (the pages give no wire format): codes are 4-bit two's complement;
 * element 2k sits in the low nibble of byte k and element 2k+1 in the high
 * nibble. */
static void put_nibble(uint8_t *codes, int64_t pos, int q)
{
    uint8_t nib = (uint8_t)(q & 0xF);
    uint8_t *byte = &codes[pos >> 1];
    if ((pos & 1) == 0) *byte = (uint8_t)((*byte & 0xF0) | nib);
    else                *byte = (uint8_t)((*byte & 0x0F) | (nib << 4));
}

ORC_EXPORT int orc_get_nibble(const uint8_t *codes, int64_t pos)
{
    int v = (pos & 1) ? (codes[pos >> 1] >> 4) : (codes[pos >> 1] & 0xF);
    return v >= 8 ? v - 16 : v;
}

/* ------------------------------------------------------------------------ */
/* All-to-all send order                                                      */
/* ------------------------------------------------------------------------ */

/*
 * A rank's N elements are R contiguous slices of S = N/R; slice k is reduced
 * on, and finally owned by, rank k (the ZeRO partition).  With G groups of
 * L = R/G ranks (rank k = g*L + l), the first all-to-all stays inside a group
 * and sends to local rank l everything that ends on ranks {g'*L + l}; [qgZ]
 * reduces intra-node first, then inter-node.  Reading: a sender lays out
 * chunk position p = l*G + g' holding slice g'*L + l, so each destination's
 * data is one contiguous run of G*S elements; with G = 1 this is the identity.
 * Returns the chunk position of slice `slice`.
 */
ORC_EXPORT int64_t orc_send_position(int64_t slice, int R, int G)
{
    int L = R / G;
    int64_t gq = slice / L;     /* destination group g' */
    int64_t l = slice % L;      /* destination local rank l */
    return l * G + gq;
}

/* ------------------------------------------------------------------------ */
/* Error-feedback compensation + int4 quantization, one rank                   */
/* ------------------------------------------------------------------------ */

/*
 * One rank's step of [LoCo] on [qgZ]:
 *   c = g + s * e                             (error compensation)
 *   q, scale = Q4(c) per block of B           (block int4, absmax / 7)
 *   d = q * scale                             (what the receivers will see)
 *   e <- beta * e + (1 - beta) * (c - d)      (error update)
 * Reading for the update (the page names two LoCo parameters without giving
 * them): s scales the stored error when it is added back, beta is a moving
 * average that keeps part of the old error; s = 1, beta = 0 is plain error
 * feedback.  1 - beta is formed once in binary32.  e == NULL quantizes g
 * alone and stores no error.
 *
 * g: N bf16 bit patterns; e: N floats (in place) or NULL; codes: N/2 bytes;
 * scales: N/B floats.  Codes and scales come out in send order (above); the
 * error buffer stays in gradient order.
 */
ORC_EXPORT int orc_ef_quant_int4_rank(const uint16_t *g, float *e,
                                       uint8_t *codes, float *scales,
                                       int64_t N, int R, int G, int B,
                                       float s, float beta)
{
    if (!orc_block_ok(B)) return ORC_EBLOCK;
    int64_t S = N / R;
    float one_minus_beta = 1.0f - beta;
    float c[ORC_MAX_BLOCK];
    int8_t q[ORC_MAX_BLOCK];
    for (int64_t slice = 0; slice < R; ++slice) {
        int64_t p = orc_send_position(slice, R, G);
        for (int64_t b0 = 0; b0 < S; b0 += B) {
            int64_t in0 = slice * S + b0;
            int64_t out0 = p * S + b0;
            for (int i = 0; i < B; ++i) {
                float gi = orc_bf16_to_f32(g[in0 + i]);
                if (e) {
                    float se = s * e[in0 + i];
                    c[i] = gi + se;
                } else {
                    c[i] = gi;
                }
            }
            float scale;
            orc_quant_block(c, B, 7, q, &scale);
            scales[out0 / B] = scale;
            for (int i = 0; i < B; ++i)
                put_nibble(codes, out0 + i, q[i]);
            if (e) {
                for (int i = 0; i < B; ++i) {
                    float d = orc_dequant(q[i], scale);
                    float resid = c[i] - d;
                    float kept = beta * e[in0 + i];
                    float added = one_minus_beta * resid;
                    e[in0 + i] = kept + added;
                }
            }
        }
    }
    return 0;
}

/* All R ranks: g and e are [R][N], codes [R][N/2], scales [R][N/B]. */
ORC_EXPORT int orc_ef_quant_int4(const uint16_t *g, float *e,
                                  uint8_t *codes, float *scales,
                                  int64_t N, int R, int G, int B,
                                  float s, float beta)
{
    if (!orc_block_ok(B)) return ORC_EBLOCK;
    for (int r = 0; r < R; ++r)
        orc_ef_quant_int4_rank(g + (int64_t)r * N,
                               e ? e + (int64_t)r * N : 0,
                               codes + (int64_t)r * (N / 2),
                               scales + (int64_t)r * (N / B),
                               N, R, G, B, s, beta);
    return 0;
}

/*
 * The same step with a bf16 error buffer.  LoCo's cost is the extra memory of
 * the error buffer ("Merge LoCo with Zero++", Overview); storing it in bf16
 * halves that memory and its traffic.  Reading: the stored error is widened
 * exactly, every operation is the binary32 chain of orc_ef_quant_int4_rank,
 * and only the new error is rounded to the nearest bf16 (ties to even) when
 * it is stored.  e16: N bf16 bit patterns, in place (not NULL).
 */
ORC_EXPORT int orc_ef_quant_int4_rank_bf16ef(const uint16_t *g, uint16_t *e16,
                                              uint8_t *codes, float *scales,
                                              int64_t N, int R, int G, int B,
                                              float s, float beta)
{
    if (!orc_block_ok(B)) return ORC_EBLOCK;
    int64_t S = N / R;
    float omb = 1.0f - beta;
    float c[ORC_MAX_BLOCK];
    int8_t q[ORC_MAX_BLOCK];
    for (int64_t slice = 0; slice < R; ++slice) {
        int64_t p = orc_send_position(slice, R, G);
        for (int64_t b0 = 0; b0 < S; b0 += B) {
            int64_t in0 = slice * S + b0;
            int64_t out0 = p * S + b0;
            for (int i = 0; i < B; ++i) {
                float gh = orc_bf16_to_f32(g[in0 + i]);
                float eh = orc_bf16_to_f32(e16[in0 + i]);
                float seh = s * eh;
                c[i] = gh + seh;
            }
            float scale;
            orc_quant_block(c, B, 7, q, &scale);
            scales[out0 / B] = scale;
            for (int i = 0; i < B; ++i)
                put_nibble(codes, out0 + i, q[i]);
            for (int i = 0; i < B; ++i) {
                float eh = orc_bf16_to_f32(e16[in0 + i]);
                float dh = orc_dequant(q[i], scale);
                float rh = c[i] - dh;
                float kh = beta * eh;
                float ah = omb * rh;
                e16[in0 + i] = orc_f32_to_bf16_rne(kh + ah);
            }
        }
    }
    return 0;
}

ORC_EXPORT int orc_ef_quant_int4_bf16ef(const uint16_t *g, uint16_t *e16,
                                         uint8_t *codes, float *scales,
                                         int64_t N, int R, int G, int B,
                                         float s, float beta)
{
    if (!orc_block_ok(B)) return ORC_EBLOCK;
    for (int r = 0; r < R; ++r)
        orc_ef_quant_int4_rank_bf16ef(g + (int64_t)r * N, e16 + (int64_t)r * N,
                                      codes + (int64_t)r * (N / 2),
                                      scales + (int64_t)r * (N / B),
                                      N, R, G, B, s, beta);
    return 0;
}

/*
 * The same step with an int8 error buffer: a quarter of the fp32 buffer's
 * memory and traffic ("Merge LoCo with Zero++", Overview: LoCo's cost is the
 * extra memory of the error buffer).  Reading: the error of each gradient
 * block (B elements, gradient order) is stored as B int8 codes and one fp32
 * scale by the block quantizer with qmax = 127 (the qwZ rule: scale = m/127,
 * codes rint(e * 127/m), zero block below 127 * 2^-126); it is read back as
 * code * scale, one rounding; every other operation is the binary32 chain of
 * orc_ef_quant_int4_rank.  e8: N codes and e8s: N/B scales of one rank, in
 * place (a zero buffer is all-zero codes and scales).
 */
ORC_EXPORT int orc_ef_quant_int4_rank_int8ef(const uint16_t *g, int8_t *e8, float *e8s,
                                              uint8_t *codes, float *scales,
                                              int64_t N, int R, int G, int B,
                                              float s, float beta)
{
    if (!orc_block_ok(B)) return ORC_EBLOCK;
    int64_t S = N / R;
    float one_mb = 1.0f - beta;
    float c8[ORC_MAX_BLOCK];
    float ev8[ORC_MAX_BLOCK];
    float en8[ORC_MAX_BLOCK];
    int8_t q8[ORC_MAX_BLOCK];
    for (int64_t slice = 0; slice < R; ++slice) {
        int64_t p = orc_send_position(slice, R, G);
        for (int64_t b0 = 0; b0 < S; b0 += B) {
            int64_t in0 = slice * S + b0;
            int64_t out0 = p * S + b0;
            float es8 = e8s[in0 / B];
            for (int i = 0; i < B; ++i) {
                ev8[i] = orc_dequant(e8[in0 + i], es8);
                float g8 = orc_bf16_to_f32(g[in0 + i]);
                float se8 = s * ev8[i];
                c8[i] = g8 + se8;
            }
            float scale;
            orc_quant_block(c8, B, 7, q8, &scale);
            scales[out0 / B] = scale;
            for (int i = 0; i < B; ++i)
                put_nibble(codes, out0 + i, q8[i]);
            for (int i = 0; i < B; ++i) {
                float d8 = orc_dequant(q8[i], scale);
                float r8 = c8[i] - d8;
                float k8 = beta * ev8[i];
                float a8 = one_mb * r8;
                en8[i] = k8 + a8;
            }
            orc_quant_block(en8, B, 127, e8 + in0, &e8s[in0 / B]);
        }
    }
    return 0;
}

ORC_EXPORT int orc_ef_quant_int4_int8ef(const uint16_t *g, int8_t *e8, float *e8s,
                                         uint8_t *codes, float *scales,
                                         int64_t N, int R, int G, int B,
                                         float s, float beta)
{
    if (!orc_block_ok(B)) return ORC_EBLOCK;
    for (int r = 0; r < R; ++r)
        orc_ef_quant_int4_rank_int8ef(g + (int64_t)r * N, e8 + (int64_t)r * N,
                                      e8s + (int64_t)r * (N / B),
                                      codes + (int64_t)r * (N / 2),
                                      scales + (int64_t)r * (N / B),
                                      N, R, G, B, s, beta);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* a6-a7 / a9: dequantize and reduce in full precision                        */
/* ------------------------------------------------------------------------ */

/* Dequantized value at global code position pos of a code/scale buffer. */
static float dq_at(const uint8_t *codes, const float *scales, int64_t pos, int B)
{
    return orc_dequant(orc_get_nibble(codes, pos), scales[pos / B]);
}

/*
 * Destination k of a reduction.  [qgZ]: after the all-to-all, each receiver
 * dequantizes what it got and reduces in full precision (binary32 here, the
 * sources added in a fixed order starting from +0).  The result is then
 * multiplied by out_scale (1 gives the sum, 1/R the average) and stored as
 * binary32 (out_bf16 = 0) or rounded to bf16 (out_bf16 = 1).
 *
 * G == 1, the flat reduce: the buffers are the R ranks' send buffers ([R][N]
 *   codes in send order); destination k adds chunk k of ranks 0..R-1.
 * G > 1, the second (inter-group) hop: the buffers are the first hop's
 *   outputs, unit (g, l) at index g*L + l, each [G][S] (below); destination
 *   k = g*L + l adds sub-slice g of units (0, l), (1, l), ..., (G-1, l).
 * In both cases out holds S values.
 */
ORC_EXPORT void orc_dequant_reduce_dest_range(const uint8_t *codes,
                                              const float *scales,
                                              int64_t N, int R, int G, int B, int k,
                                              int64_t i0, int64_t i1,
                                              float out_scale, void *out,
                                              int out_bf16);

ORC_EXPORT void orc_dequant_reduce_dest(const uint8_t *codes,
                                        const float *scales,
                                        int64_t N, int R, int G, int B, int k,
                                        float out_scale, void *out,
                                        int out_bf16)
{
    orc_dequant_reduce_dest_range(codes, scales, N, R, G, B, k, 0, N / R,
                                  out_scale, out, out_bf16);
}

/* Outputs [i0, i1) of destination k, written to out[0 .. i1-i0): every
 * output is its own sum, so a range is exactly that part of the whole. */
ORC_EXPORT void orc_dequant_reduce_dest_range(const uint8_t *codes,
                                              const float *scales,
                                              int64_t N, int R, int G, int B, int k,
                                              int64_t i0, int64_t i1,
                                              float out_scale, void *out,
                                              int out_bf16)
{
    int64_t S = N / R;
    int L = R / G;
    for (int64_t i = i0; i < i1; ++i) {
        float acc = 0.0f;
        if (G == 1) {
            for (int r = 0; r < R; ++r) {
                int64_t pos = (int64_t)r * N + (int64_t)k * S + i;
                acc = acc + dq_at(codes, scales, pos, B);
            }
        } else {
            int g = k / L, l = k % L;
            for (int gq = 0; gq < G; ++gq) {
                int64_t unit = (int64_t)gq * L + l;
                int64_t pos = unit * G * S + (int64_t)g * S + i;
                acc = acc + dq_at(codes, scales, pos, B);
            }
        }
        float v = acc * out_scale;
        if (out_bf16) ((uint16_t *)out)[i - i0] = orc_f32_to_bf16_rne(v);
        else          ((float *)out)[i - i0] = v;
    }
}

/* Every destination: out is [R][S] in destination order. */
ORC_EXPORT void orc_dequant_reduce(const uint8_t *codes, const float *scales,
                                   int64_t N, int R, int G, int B,
                                   float out_scale, void *out, int out_bf16)
{
    int64_t S = N / R;
    for (int k = 0; k < R; ++k) {
        void *o = out_bf16 ? (void *)((uint16_t *)out + (int64_t)k * S)
                           : (void *)((float *)out + (int64_t)k * S);
        orc_dequant_reduce_dest(codes, scales, N, R, G, B, k, out_scale, o,
                                out_bf16);
    }
}

/* ------------------------------------------------------------------------ */
/* a8: first hop of the hierarchical reduce, with requantization              */
/* ------------------------------------------------------------------------ */

/*
 * Unit (g, l) -- local rank l of group g -- receives from the L ranks of its
 * group their chunk l (send positions l*G .. l*G+G-1, G sub-slices of S),
 * reduces them in full precision in local-rank order, and requantizes each
 * block of B of the partial sums to int4 for the inter-group hop [qgZ].  No
 * error feedback on this hop.  Output: G*S codes (G*S/2 bytes) and G*S/B
 * scales, sub-slice g' first-to-last; sub-slice g' is bound for rank g'*L + l.
 */
ORC_EXPORT int orc_dequant_reduce_requant_unit_ef(const uint8_t *codes,
                                                   const float *scales,
                                                   int64_t N, int R, int G, int B,
                                                   int g, int l,
                                                   uint8_t *out_codes,
                                                   float *out_scales,
                                                   float *e1, float s, float beta);

ORC_EXPORT int orc_dequant_reduce_requant_unit(const uint8_t *codes,
                                                const float *scales,
                                                int64_t N, int R, int G, int B,
                                                int g, int l,
                                                uint8_t *out_codes,
                                                float *out_scales)
{
    return orc_dequant_reduce_requant_unit_ef(codes, scales, N, R, G, B, g, l,
                                              out_codes, out_scales, 0, 0.0f, 0.0f);
}

/*
 * The same first hop with error feedback on the requantization ("Merge LoCo
 * with Zero++", review thread: the error buffers hang off each parameter as
 * `inter_ef_buf`, the buffer of the inter-node message).  Reading: the unit
 * keeps one fp32 error per requantized value, e1 [G*S] in output order, and
 * applies the update of orc_ef_quant_int4_rank to the partial sums:
 *   c = p + s * e1;  q, scale = Q4(c);  e1 <- beta * e1 + (1 - beta) * (c - d).
 * e1 == NULL is the plain first hop.
 */
ORC_EXPORT int orc_dequant_reduce_requant_unit_ef(const uint8_t *codes,
                                                   const float *scales,
                                                   int64_t N, int R, int G, int B,
                                                   int g, int l,
                                                   uint8_t *out_codes,
                                                   float *out_scales,
                                                   float *e1, float s, float beta)
{
    if (!orc_block_ok(B)) return ORC_EBLOCK;
    int64_t S = N / R;
    int L = R / G;
    float one_minus_beta = 1.0f - beta;
    float part[ORC_MAX_BLOCK];
    int8_t q[ORC_MAX_BLOCK];
    for (int gq = 0; gq < G; ++gq) {
        for (int64_t b0 = 0; b0 < S; b0 += B) {
            int64_t out0 = (int64_t)gq * S + b0;
            for (int i = 0; i < B; ++i) {
                float acc = 0.0f;
                for (int lq = 0; lq < L; ++lq) {
                    int64_t r = (int64_t)g * L + lq;
                    int64_t pos = r * N + ((int64_t)l * G + gq) * S + b0 + i;
                    acc = acc + dq_at(codes, scales, pos, B);
                }
                if (e1) {
                    float se1 = s * e1[out0 + i];
                    acc = acc + se1;
                }
                part[i] = acc;
            }
            float scale;
            orc_quant_block(part, B, 7, q, &scale);
            out_scales[out0 / B] = scale;
            for (int i = 0; i < B; ++i)
                put_nibble(out_codes, out0 + i, q[i]);
            if (e1) {
                for (int i = 0; i < B; ++i) {
                    float d1 = orc_dequant(q[i], scale);
                    float resid1 = part[i] - d1;
                    float kept1 = beta * e1[out0 + i];
                    float added1 = one_minus_beta * resid1;
                    e1[out0 + i] = kept1 + added1;
                }
            }
        }
    }
    return 0;
}

/* Every unit: out_codes is [R][G*S/2], out_scales [R][G*S/B], unit g*L + l;
 * e1 (or NULL) is [R][G*S] in the same unit order. */
ORC_EXPORT int orc_dequant_reduce_requant_ef(const uint8_t *codes,
                                              const float *scales,
                                              int64_t N, int R, int G, int B,
                                              uint8_t *out_codes,
                                              float *out_scales,
                                              float *e1, float s, float beta)
{
    if (!orc_block_ok(B)) return ORC_EBLOCK;
    int64_t S = N / R;
    int L = R / G;
    for (int g = 0; g < G; ++g)
        for (int l = 0; l < L; ++l) {
            int64_t unit = (int64_t)g * L + l;
            orc_dequant_reduce_requant_unit_ef(codes, scales, N, R, G, B, g, l,
                                               out_codes + unit * (G * S / 2),
                                               out_scales + unit * (G * S / B),
                                               e1 ? e1 + unit * (G * S) : 0,
                                               s, beta);
        }
    return 0;
}

ORC_EXPORT int orc_dequant_reduce_requant(const uint8_t *codes,
                                           const float *scales,
                                           int64_t N, int R, int G, int B,
                                           uint8_t *out_codes,
                                           float *out_scales)
{
    return orc_dequant_reduce_requant_ef(codes, scales, N, R, G, B, out_codes,
                                         out_scales, 0, 0.0f, 0.0f);
}

/* ------------------------------------------------------------------------ */
/* a10-a11: qwZ int8 block weight quantization                               */
/* ------------------------------------------------------------------------ */

/* [qwZ]: per block of B weights, symmetric int8 with scale absmax / 127. */
ORC_EXPORT int orc_qwz_quant_int8(const uint16_t *w, int8_t *codes,
                                   float *scales, int64_t n, int B)
{
    if (!orc_block_ok(B)) return ORC_EBLOCK;
    float x[ORC_MAX_BLOCK];
    for (int64_t b0 = 0; b0 < n; b0 += B) {
        for (int i = 0; i < B; ++i) x[i] = orc_bf16_to_f32(w[b0 + i]);
        orc_quant_block(x, B, 127, codes + b0, &scales[b0 / B]);
    }
    return 0;
}

/* Back to bf16: code times scale (one rounding), then rounded to bf16. */
ORC_EXPORT void orc_qwz_dequant_int8(const int8_t *codes, const float *scales,
                                     uint16_t *w_out, int64_t n, int B)
{
    for (int64_t i = 0; i < n; ++i)
        w_out[i] = orc_f32_to_bf16_rne(orc_dequant(codes[i], scales[i / B]));
}

/* qwZ quantization that also writes the bf16 weights the codes stand for:
 * the copy a node keeps after the forward all-gather (the hierarchical
 * partition of "ZeROPlusPlus.md" §1.2 keeps a full model copy in each node).
 * Exactly orc_qwz_quant_int8 followed by orc_qwz_dequant_int8. */
ORC_EXPORT int orc_qwz_quant_replica_int8(const uint16_t *w, int8_t *codes,
                                           float *scales, uint16_t *replica,
                                           int64_t n, int B)
{
    if (orc_qwz_quant_int8(w, codes, scales, n, B) != 0) return ORC_EBLOCK;
    orc_qwz_dequant_int8(codes, scales, replica, n, B);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* a12: stochastic-rounding accumulate with the source zeroed                 */
/* ------------------------------------------------------------------------ */

/* MurmurHash3's 32-bit finalizer (Austin Appleby, public domain). */
ORC_EXPORT uint32_t orc_fmix32(uint32_t h)
{
    h ^= h >> 16;
    h *= 0x85EBCA6Bu;
    h ^= h >> 13;
    h *= 0xC2B2AE35u;
    h ^= h >> 16;
    return h;
}

/* Reading of "a splitmix32 hash of (seed, step, index)": add the 32-bit
 * golden-ratio increment, then finalize. */
ORC_EXPORT uint32_t orc_mix32(uint32_t z)
{
    return orc_fmix32(z + 0x9E3779B9u);
}

/* The 16 random bits used for element i of call (seed, step). */
ORC_EXPORT uint32_t orc_sr_bits(uint32_t seed, uint32_t step, uint32_t i)
{
    uint32_t key = orc_mix32(orc_mix32(seed) ^ step);
    return orc_mix32(key ^ i) & 0xFFFFu;
}

/*
 * Stochastic rounding of a binary32 to bf16 with 16 uniform bits r: add r
 * below the kept half and truncate.  The magnitude is rounded up exactly when
 * the carry reaches bit 16, i.e. with probability (low 16 bits) / 65536, so
 * the expected result is x [SR].  Infinities pass through; magnitudes within
 * one bf16 step of FLT_MAX can round to infinity.  Inputs are finite sums.
 */
ORC_EXPORT uint16_t orc_sr_round(float x, uint32_t r)
{
    uint32_t u = f32_bits(x);
    return (uint16_t)((u + r) >> 16);
}

/* [SR]: dst_i <- SR(f32(dst_i) + f32(src_i)); src_i <- 0. */
ORC_EXPORT void orc_sr_accumulate_bf16(uint16_t *dst, uint16_t *src, int64_t n,
                                       uint32_t seed, uint32_t step)
{
    for (int64_t i = 0; i < n; ++i) {
        float sum = orc_bf16_to_f32(dst[i]) + orc_bf16_to_f32(src[i]);
        dst[i] = orc_sr_round(sum, orc_sr_bits(seed, step, (uint32_t)i));
        src[i] = 0;
    }
}
