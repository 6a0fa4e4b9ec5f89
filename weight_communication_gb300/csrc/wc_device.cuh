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

namespace wc {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr float kMinNormal = 1.17549435082228750797e-38f;  // 2^-126

// bf16 bit pattern -> fp32 (exact: a bf16 is the upper half of a binary32).
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) {
    return __uint_as_float(h << 16);
}

// fp32 -> bf16 bit pattern, round to nearest even.
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Max over the `width` lanes of an aligned lane group (width a power of two).
template <int WIDTH>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
    for (int off = WIDTH / 2; off > 0; off >>= 1)
        v = fmaxf(v, __shfl_xor_sync(kFull, v, off));
    return v;
}

// Scale and reciprocal of a symmetric block: a block whose scale m / qmax
// would not be a normal binary32 (m < qmax * 2^-126) is a zero block.
struct BlockScale {
    float scale;
    float inv;
    bool zero;
};

template <int QMAX>
__device__ __forceinline__ BlockScale block_scale(float m) {
    BlockScale s;
    s.zero = m < float(QMAX) * kMinNormal;  // exact product
    if (s.zero) {
        s.scale = 0.0f;
        s.inv = 0.0f;
    } else {
        s.scale = __fdiv_rn(m, float(QMAX));
        s.inv = __fdiv_rn(float(QMAX), m);
    }
    return s;
}

// Code of one value: clamp(rint(x * inv), -QMAX, QMAX), ties to even.
template <int QMAX>
__device__ __forceinline__ int quant_code(float x, const BlockScale &s) {
    if (s.zero) return 0;
    int q = __float2int_rn(__fmul_rn(x, s.inv));
    return min(max(q, -QMAX), QMAX);
}

// Dequantized value: code * scale, one rounding.
__device__ __forceinline__ float dequant(int q, float scale) {
    return __fmul_rn(__int2float_rn(q), scale);
}

// Signed value of nibble j (0..7) of a packed 32-bit word (element 2k in the
// low nibble of byte k).
__device__ __forceinline__ int nibble(uint32_t w, int j) {
    return int(w << (28 - 4 * j)) >> 28;  // arithmetic shift sign-extends
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
