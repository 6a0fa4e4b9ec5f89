// int8_error_block.cuh -- one block of the error-feedback int4 quantization
// with the int8 error buffer, in packed exact arithmetic: shared by the
// stand-alone quantization (qgz_quant.cu) and the fused steps (qgz_fused.cu),
// so both run the same operations.
//
// "Merge LoCo with Zero++" (DeepSpeed PR #6730), Overview: error feedback on
// the 4-bit gradients, at the cost of the error buffer's memory (here one
// byte per element plus one fp32 scale per block).
#pragma once

#include "wc_device.cuh"

namespace wc {

// The int8 error buffer's step for whole-warp blocks (B >= 128), in packed
// exact arithmetic (wc_device.cuh): the same operations as the EF = kEfInt8
// case of ef_quant_int4_warp, two elements per instruction, with the codes of
// both quantizations packed through biased rounding (q + 8 and q + 128 in the
// low byte).  Every code, scale and stored error is the one the scalar chain
// gives, bit for bit.  Lane t holds elements 128k + 4t + j of the block as
// pairs (j = 0, 1) and (2, 3); the block's loads (gv: bf16 gradients, e8w:
// stored error codes, es: stored error scale) are already in registers.
// S1: the error scale s is 1, so s*e is e itself (exact for every finite e,
// signed zeros included) and its multiply is left out.  tile0 is the block's
// first gradient element, out0 its send position; total = R*N bounds every
// access.  WRITE_CODES: store the int4 codes and the block scale (a fused
// step may skip them).  ACC: add the dequantized values into acc (lane t's
// elements 128k + 4t + j in acc[k][j], one IEEE addition each), the running
// sums of a fused reduce.
template <int B, bool S1, bool WRITE_CODES, bool ACC>
__device__ __forceinline__ void int8ef_block(const uint2 (&gv)[B / 128],
                                             const uint32_t (&e8w)[B / 128], float es,
                                             int8_t *__restrict__ ef8,
                                             float *__restrict__ ef_scales,
                                             uint8_t *__restrict__ codes,
                                             float *__restrict__ scales, uint32_t total,
                                             uint32_t tile0, uint32_t out0, int lane, float s,
                                             float beta, float one_minus_beta, const Ops2 &ops,
                                             float (*acc)[4]) {
    constexpr int K = B / 128;
    const uint32_t eblk = tile0 / B;
    const f32x2 es2 = pack2(es, es), s2 = pack2(s, s);
    const f32x2 unbias8 = pack2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
    f32x2 c[K][2], e[K][2];
    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const uint32_t u = e8w[k] ^ 0x80808080u;  // stored error codes + 128
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const f32x2 f = pack2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7440u + 2 * h)),
                                  __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7441u + 2 * h)));
            e[k][h] = ops.mul(ops.add(f, unbias8), es2);  // stored error: code (exact) * scale
            const uint32_t gw = h ? gv[k].y : gv[k].x;
            const f32x2 gf = pack2(__uint_as_float(gw << 16), __uint_as_float(gw & 0xFFFF0000u));
            c[k][h] = ops.add(gf, S1 ? e[k][h] : ops.mul(s2, e[k][h]));
            float a, b;
            unpack2(c[k][h], a, b);
            m = max3(m, fabsf(a), fabsf(b));
        }
    }
    m = group_max<kWarp>(m);
    const BlockScale bs = block_scale<7>(m);
    const f32x2 inv2 = pack2(bs.inv, bs.inv), sc2 = pack2(bs.scale, bs.scale);
    const f32x2 shift4 = pack2(kRoundShift4, kRoundShift4);
    const f32x2 unshift4 = pack2(-kRoundShift4, -kRoundShift4);
    const f32x2 beta2 = pack2(beta, beta), omb2 = pack2(one_minus_beta, one_minus_beta);
    f32x2 en[K][2];
    float m8 = 0.0f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        uint32_t pr[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const f32x2 rq = ops.add(ops.mul(c[k][h], inv2), shift4);
            float r0, r1;
            unpack2(rq, r0, r1);
            pr[h] = __float_as_uint(r0) + (__float_as_uint(r1) << 4);  // (q0 + 8) + 16 (q1 + 8)
            const f32x2 d = ops.mul(ops.add(rq, unshift4), sc2);       // the code (exact) * scale
            if (ACC) {
                f32x2 a2 = pack2(acc[k][2 * h], acc[k][2 * h + 1]);
                a2 = ops.add(a2, d);
                unpack2(a2, acc[k][2 * h], acc[k][2 * h + 1]);
            }
            en[k][h] = ops.add(ops.mul(beta2, e[k][h]), ops.mul(omb2, ops.sub(c[k][h], d)));
            float a, b;
            unpack2(en[k][h], a, b);
            m8 = max3(m8, fabsf(a), fabsf(b));
        }
        const uint32_t pos = out0 + 128u * k + 4u * lane;
        if (WRITE_CODES && WC_IN_BOUNDS(uint64_t(pos) + 4 <= total))
            __stcs(reinterpret_cast<unsigned short *>(codes + pos / 2),
                   (unsigned short)(__byte_perm(pr[0], pr[1], 0x0040u) ^ 0x8888u));
    }
    if (WRITE_CODES && lane == 0 && WC_IN_BOUNDS(out0 / B < total / B))
        __stcs(scales + out0 / B, bs.scale);
    // the new error of the block, quantized by the int8 absmax rule
    m8 = group_max<kWarp>(m8);
    const BlockScale bse = block_scale<127>(m8);
    const f32x2 inv8 = pack2(bse.inv, bse.inv), shift8 = pack2(kRoundShift8, kRoundShift8);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        uint32_t rb[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float r0, r1;
            unpack2(ops.add(ops.mul(en[k][h], inv8), shift8), r0, r1);
            rb[2 * h] = __float_as_uint(r0);
            rb[2 * h + 1] = __float_as_uint(r1);
        }
        const uint32_t x = tile0 + 128u * k + 4u * lane;
        if (WC_IN_BOUNDS(uint64_t(x) + 4 <= total))
            __stcs(reinterpret_cast<unsigned int *>(ef8 + x), pack_int8_quad(rb[0], rb[1], rb[2], rb[3]));
    }
    if (lane == 0 && WC_IN_BOUNDS(eblk < total / B)) __stcs(ef_scales + eblk, bse.scale);
}

}  // namespace wc
