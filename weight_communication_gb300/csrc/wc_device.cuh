// wc_device.cuh -- device helpers shared by the kernels.
//
// Every rounding-relevant operation goes through an explicitly rounded
// intrinsic (__fadd_rn, __fmul_rn, __fsub_rn, __fdiv_rn, __float2int_rn),
// so the compiler can neither contract a multiply and an add into one fused
// operation nor replace a division by a reciprocal: the kernels compute the
// same binary32 chain of operations that the method defines.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "wc_internal.h"

namespace wc {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr float kMinNormal = 1.17549435082228750797e-38f;  // 2^-126

// Checked builds (compiled with -DWC_CHECKED=1): before every global load or
// store a kernel compares the access with the extent of its buffer, as the
// call's sizes define it.  WC_IN_BOUNDS(ok) is that comparison.  A failure
// counts one violation in this source file's record, keeps the first failing
// line, and skips the access, so a checked kernel never touches memory
// outside its buffers and never traps.  The host reads and clears the records
// through wc_checked_violations().  In ordinary builds WC_IN_BOUNDS(ok) is
// the constant true and the comparison is not compiled.
#ifndef WC_CHECKED
#define WC_CHECKED 0
#endif

#if WC_CHECKED
static __device__ CheckRecord g_check_record;

__device__ __forceinline__ bool in_bounds(bool ok, unsigned int line) {
    if (!ok) {
        atomicAdd(&g_check_record.count, 1u);
        atomicCAS(&g_check_record.first_line, 0u, line);
    }
    return ok;
}
#define WC_IN_BOUNDS(ok) ::wc::in_bounds((ok), __LINE__)

// Host reader of this source file's record (one per file: the record is
// file-local device memory).  probe first launches a one-thread kernel of
// this file that fails one comparison and touches no memory, to show that a
// violation reaches the host.
#define WC_CHECK_RECORD_READER(name)                                                    \
    __global__ void name##_probe() { (void)WC_IN_BOUNDS(false); }                       \
    cudaError_t name(CheckRecord *out, bool reset, bool probe) {                        \
        if (probe) {                                                                     \
            name##_probe<<<1, 1>>>();                                                    \
            const cudaError_t p = cudaGetLastError();                                    \
            if (p != cudaSuccess) return p;                                              \
        }                                                                                \
        cudaError_t e = cudaMemcpyFromSymbol(out, g_check_record, sizeof(CheckRecord));  \
        if (e == cudaSuccess && reset) {                                                 \
            const CheckRecord zero = {0u, 0u};                                           \
            e = cudaMemcpyToSymbol(g_check_record, &zero, sizeof(CheckRecord));          \
        }                                                                                \
        return e;                                                                        \
    }
#else
#define WC_IN_BOUNDS(ok) true
#define WC_CHECK_RECORD_READER(name)
#endif

// bf16 bit pattern -> fp32 (exact: a bf16 is the upper half of a binary32).
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) {
    return __uint_as_float(h << 16);
}

// fp32 -> bf16 bit pattern, round to nearest even.
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Two fp32 -> two bf16 bit patterns in one word (lo in the low half), each
// rounded to nearest even: one paired conversion instead of two single ones
// and the shift and or that join them.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2_bits(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    uint32_t bits;
    memcpy(&bits, &v, sizeof(bits));  // .x is the low half
    return bits;
}

// Max over the `width` lanes of an aligned lane group (width a power of two)
// of values v >= +0 that are not NaN -- every caller reduces absolute values.
// For such floats the order of the encodings, read as unsigned integers, is
// the order of the values, so a whole warp reduces with one integer max
// (redux.sync); narrower groups use shuffles.
template <int WIDTH>
__device__ __forceinline__ float group_max(float v) {
    if constexpr (WIDTH == kWarp) {
        return __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(v)));
    } else {
#pragma unroll
        for (int off = WIDTH / 2; off > 0; off >>= 1)
            v = fmaxf(v, __shfl_xor_sync(kFull, v, off));
        return v;
    }
}

// Scale and reciprocal of a symmetric block: a block whose scale m / qmax
// would not be a normal binary32 (m < qmax * 2^-126) is a zero block, with
// scale 0 and inv 0 -- every finite value then quantizes to the code 0.
struct BlockScale {
    float scale;
    float inv;
};

template <int QMAX>
__device__ __forceinline__ BlockScale block_scale(float m) {
    BlockScale s;
    if (m < float(QMAX) * kMinNormal) {  // exact product
        s.scale = 0.0f;
        s.inv = 0.0f;
    } else {
        s.scale = __fdiv_rn(m, float(QMAX));
        s.inv = __fdiv_rn(float(QMAX), m);
    }
    return s;
}

// Integer conversions without the (slow) conversion pipe.
//
// Rounding: for |x| < 2^22, x + 1.5*2^23 lies in [2^23, 2^24) where the spacing
// of binary32 is exactly 1, so the IEEE addition rounds x to the nearest
// integer, ties to even (1.5*2^23 is even); subtracting the constant again is
// exact.  The low bits of the sum's encoding are the integer's low bits in
// two's complement, because the constant's low 22 bits are zero.
constexpr float kRoundShift = 12582912.0f;  // 1.5 * 2^23

// Code of one value of a block: q = clamp(rint(x * inv), -QMAX, QMAX), as an
// exact integer-valued float together with its two's-complement bits (the
// caller masks the low 4 or 8), both from the one rounding addition.
// No clamp is executed because none can be active: every |x| of the block
// is at most m, inv = fl(QMAX / m) <= (QMAX / m)(1 + 2^-24), so
// |x * inv| <= QMAX (1 + 2^-24)^2 < QMAX + 1/2 after its own rounding, and
// rint returns at most QMAX; a zero block has inv = 0 and gives q = 0.
struct QCode {
    float q;
    uint32_t bits;
};

template <int QMAX>
__device__ __forceinline__ QCode quant_code(float x, const BlockScale &s) {
    const float r = __fadd_rn(__fmul_rn(x, s.inv), kRoundShift);
    QCode c;
    c.bits = __float_as_uint(r);
    c.q = __fsub_rn(r, kRoundShift);
    return c;
}

// Dequantized value: code * scale, one rounding.
__device__ __forceinline__ float dequant(float q, float scale) { return __fmul_rn(q, scale); }

// First term of a sum that starts at +0: (+0) + fl(q * scale), two roundings,
// equals fma(q, scale, +0), one rounding, for every integer-valued q and
// every scale.  If q * scale is exactly zero, both sums are +0 (a sum of
// zeros of opposite sign rounds to +0).  Otherwise |q * scale| >= |scale| is
// at least the smallest subnormal, so it rounds to a nonzero r.  Adding +0
// to r is exact, and the fma rounds q * scale + 0 = q * scale once, to r.
// One instruction instead of two.
__device__ __forceinline__ float dequant_first(float q, float scale) {
    return __fmaf_rn(q, scale, 0.0f);
}

// Unpacking: a biased code u in [0, 2^k) placed in the mantissa of 2^23 reads
// as 2^23 + u exactly; subtracting 2^23 + bias leaves the signed code, exact.
// PRMT (byte permute) moves byte `b` of x under the exponent byte 0x4B.
__device__ __forceinline__ float biased_byte_to_float(uint32_t x, int b, float offset) {
    return __fsub_rn(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7440u + b)), offset);
}

// The 8 signed int4 codes of a packed word (element 2k in the low nibble of
// byte k), as exact floats.
__device__ __forceinline__ void unpack_int4x8(uint32_t w, float f[8]) {
    const uint32_t lo = (w ^ 0x88888888u) & 0x0F0F0F0Fu;         // nibble + 8, even elements
    const uint32_t hi = ((w >> 4) ^ 0x08080808u) & 0x0F0F0F0Fu;  // nibble + 8, odd elements
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        f[2 * b] = biased_byte_to_float(lo, b, 8388616.0f);      // 2^23 + 8
        f[2 * b + 1] = biased_byte_to_float(hi, b, 8388616.0f);
    }
}

// The 4 signed int8 codes of a packed word, as exact floats.
__device__ __forceinline__ void unpack_int8x4(uint32_t w, float f[4]) {
    const uint32_t u = w ^ 0x80808080u;                            // byte + 128
#pragma unroll
    for (int b = 0; b < 4; ++b) f[b] = biased_byte_to_float(u, b, 8388736.0f);  // 2^23 + 128
}

// ---------------------------------------------------------------------------
// Packed pairs (f32x2): two independent binary32 lanes per instruction
// ---------------------------------------------------------------------------
//
// sm_100-class GPUs execute fma.rn.f32x2 -- two fused multiply-adds, each
// rounded once -- in one instruction.  The kernels whose exact fp32 chains
// are issue-bound run them two values at a time with it, and every packed
// operation is an fma whose third or second operand makes it exact:
//   x * y  = fma(x, y, -0)   (one rounding of the product; -0 keeps the sign
//                             of a zero product, and x*y + (-0) = x*y)
//   x + y  = fma(x, 1, y)    (one rounding of the sum)
//   x - y  = fma(y, -1, x)   (negation is exact; one rounding of x - y)
// The constants 1, -0 and -1 reach the kernels as launch arguments
// (Exact2), not as literals, so no compiler pass can recognise a product
// feeding a sum and contract the two into one fma with a single rounding.
struct Exact2 {
    float one, mzero, mone;  // 1, -0, -1
};
inline Exact2 exact2_constants() { return Exact2{1.0f, -0.0f, -1.0f}; }

typedef unsigned long long f32x2;  // .x in the low half

__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(f32x2 v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 fma2_rn(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

struct Ops2 {
    f32x2 one, mzero, mone;
    __device__ __forceinline__ explicit Ops2(const Exact2 &k)
        : one(pack2(k.one, k.one)), mzero(pack2(k.mzero, k.mzero)), mone(pack2(k.mone, k.mone)) {}
    __device__ __forceinline__ f32x2 mul(f32x2 x, f32x2 y) const { return fma2_rn(x, y, mzero); }
    __device__ __forceinline__ f32x2 add(f32x2 x, f32x2 y) const { return fma2_rn(x, one, y); }
    __device__ __forceinline__ f32x2 sub(f32x2 x, f32x2 y) const { return fma2_rn(y, mone, x); }
};

// max(a, b, c) of non-NaN values in one instruction.
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Biased rounding for packing.  For |x| < 2^22, fl(x + (1.5*2^23 + bias)) is
// rint(x) + 1.5*2^23 + bias, ties to even (the constants are even integers in
// [2^23, 2^24), where binary32 spacing is 1), so it rounds exactly as
// kRoundShift does, and the low byte of its encoding is rint(x) + bias.  With
// bias = 8 (int4) and 128 (int8) a code in [-7, 7] or [-127, 127] becomes the
// non-negative byte q + bias, so bytes can be combined by adds and byte
// permutes without masking; an xor with 8 (0x80) per field at the end turns
// q + bias into q's two's complement.
constexpr float kRoundShift4 = 12582920.0f;  // 1.5 * 2^23 + 8
constexpr float kRoundShift8 = 12583040.0f;  // 1.5 * 2^23 + 128

// Four biased int4 pairs -> one word of 8 two's-complement codes.  pairs[j]
// has (q_{2j} + 8) + 16 (q_{2j+1} + 8) in its low byte.
__device__ __forceinline__ uint32_t pack_int4_pairs(const uint32_t pairs[4]) {
    return __byte_perm(__byte_perm(pairs[0], pairs[1], 0x0040u),
                       __byte_perm(pairs[2], pairs[3], 0x0040u), 0x5410u) ^ 0x88888888u;
}
// Low bytes of four biased int8 codes -> one word of 4 two's-complement codes.
__device__ __forceinline__ uint32_t pack_int8_quad(uint32_t b0, uint32_t b1, uint32_t b2,
                                                   uint32_t b3) {
    return __byte_perm(__byte_perm(b0, b1, 0x0040u), __byte_perm(b2, b3, 0x0040u), 0x5410u) ^
           0x80808080u;
}

// ---------------------------------------------------------------------------
// Dequantization through a per-block product table
// ---------------------------------------------------------------------------
//
// Every int4 code of a (source, block) pair dequantizes to one of 16 values
// fl(q * scale), q = -8 .. 7.  A reducing warp whose lanes all read the same
// block of a source (or, for 16-wide tables, whose half-warps each read one
// block) forms those 16 products once -- lane l holds the product for the
// nibble l & 15 -- and fetches each code's product with one shuffle indexed
// by the code's nibble.  The shuffle reads only the low 4 (16-wide) or 5
// (32-wide) bits of its lane index, and lanes l and l + 16 hold the same
// product, so the index needs no mask: a shift that brings the nibble to bit
// 0 is enough.  The value fetched is the very product R3 defines, bit for
// bit, so the sums are unchanged; the unpack, the unbias and the multiply
// leave the per-code path.  FIRST: the table of a sum's first source holds
// fma(q, scale, +0) (dequant_first), so the fetched value is already the sum
// after its first add to the +0 start.
template <bool FIRST>
__device__ __forceinline__ float product_table(float scale, int lane) {
    const float q = float(int((lane & 15) ^ 8) - 8);  // the nibble's two's-complement code
    return FIRST ? dequant_first(q, scale) : dequant(q, scale);
}

// The product of nibble j of x (bits 4j .. 4j+3) from the table.
template <int WIDTH>
__device__ __forceinline__ float table_lookup(float table, uint32_t x, int j, unsigned mask) {
    return __shfl_sync(mask, table, int(x >> (4 * j)), WIDTH);
}

// The 8 codes of word x (element 2k in the low nibble of byte k) added into
// four packed pair sums: acc[j] holds elements 2j, 2j+1.  TABLE: products
// from this lane's table (product_table, fetched with WIDTH-wide shuffles
// over the lanes in mask); else the byte-permute path in packed form -- the
// biased code under exponent 2^23 minus (2^23 + 8) (exact), times the scale
// s2 (one rounding).  FIRST: acc is the sums' +0 start; the table then holds
// fma(q, scale, +0) and the byte-permute path forms the same value.
template <bool FIRST, bool TABLE, int WIDTH>
__device__ __forceinline__ void accumulate_word(uint32_t x, float table, f32x2 s2, f32x2 acc[4],
                                                unsigned mask, const Ops2 &ops) {
    if (TABLE) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const f32x2 d = pack2(table_lookup<WIDTH>(table, x, 2 * j, mask),
                                  table_lookup<WIDTH>(table, x, 2 * j + 1, mask));
            acc[j] = FIRST ? d : ops.add(acc[j], d);
        }
    } else {
        const f32x2 unbias = pack2(-8388616.0f, -8388616.0f);        // -(2^23 + 8)
        const uint32_t lo = (x ^ 0x88888888u) & 0x0F0F0F0Fu;         // even elements + 8
        const uint32_t hi = ((x >> 4) ^ 0x08080808u) & 0x0F0F0F0Fu;  // odd elements + 8
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const f32x2 f = pack2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7440u + j)),
                                  __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7440u + j)));
            const f32x2 q = ops.add(f, unbias);
            const f32x2 d = FIRST ? fma2_rn(q, s2, pack2(0.0f, 0.0f)) : ops.mul(q, s2);
            acc[j] = FIRST ? d : ops.add(acc[j], d);
        }
    }
}

// Streaming (read-once) and plain vector accesses.
__device__ __forceinline__ float4 ld_stream_f4(const float *p) {
    return __ldcs(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ uint2 ld_stream_u2(const void *p) {
    return __ldcs(reinterpret_cast<const uint2 *>(p));
}
__device__ __forceinline__ uint4 ld_stream_u4(const void *p) {
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}

}  // namespace wc
