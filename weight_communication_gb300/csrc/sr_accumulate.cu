// sr_accumulate.cu -- ZeRO-2 bf16 gradient accumulation with stochastic
// rounding, the source zeroed in the same pass.
//
// "Zero 2 #593" (llm.c), review of llmc/cuda_utils.cuh: vector_add adds the
// incoming bf16 gradient to the accumulated one in fp32 and rounds the sum
// back to bf16 stochastically, so that many small additions stay correct in
// expectation instead of being rounded away; review of llmc/zero.cuh: the
// memset that clears the source after the add is a separate tiny launch and
// should be fused into it.
//
// Random bits: a counter-based hash of (seed, step, element index), so the
// result does not depend on the launch shape.  mix(z) = fmix32(z + golden
// ratio increment), fmix32 being MurmurHash3's 32-bit finalizer; the per-call
// key mix(mix(seed) ^ step) is formed on the host.
//
// One thread per 8 elements: 16-byte loads of dst and src, a 16-byte store of
// each (the zeros for src); 8 bytes of HBM traffic per element in all.
#include "wc_device.cuh"
#include "wc_internal.h"

namespace wc {

__host__ __device__ __forceinline__ uint32_t fmix32(uint32_t h) {
    h ^= h >> 16;
    h *= 0x85EBCA6Bu;
    h ^= h >> 13;
    h *= 0xC2B2AE35u;
    h ^= h >> 16;
    return h;
}

__host__ __device__ __forceinline__ uint32_t mix32(uint32_t z) {
    return fmix32(z + 0x9E3779B9u);
}

uint32_t sr_key(uint32_t seed, uint32_t step) { return mix32(mix32(seed) ^ step); }

// Stochastic rounding of an fp32 to bf16 with 16 random bits: add them below
// the kept half; the carry into bit 16 happens with probability
// (low 16 bits) / 65536.
__device__ __forceinline__ uint32_t sr_round(float x, uint32_t r16) {
    return (__float_as_uint(x) + r16) >> 16;
}

__device__ __forceinline__ uint32_t sr_one(uint32_t d, uint32_t s, uint32_t key, uint32_t i) {
    const float x = __fadd_rn(bf16_bits_to_f32(d), bf16_bits_to_f32(s));
    return sr_round(x, mix32(key ^ i) & 0xFFFFu);
}

__global__ void __launch_bounds__(256)
sr_accumulate_kernel(uint16_t *__restrict__ dst, uint16_t *__restrict__ src, uint32_t n,
                     uint32_t key) {
    const uint32_t v = blockIdx.x * blockDim.x + threadIdx.x;
    if (uint64_t(v) * 8u >= n) return;
    const uint32_t x = v * 8u;
    if (uint64_t(x) + 8u <= n) {
        const uint4 dv = ld_stream_u4(dst + x);
        const uint4 sv = ld_stream_u4(src + x);
        const uint32_t dw[4] = {dv.x, dv.y, dv.z, dv.w};
        const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
        uint32_t ow[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t lo = sr_one(dw[j] & 0xFFFFu, sw[j] & 0xFFFFu, key, x + 2 * j);
            const uint32_t hi = sr_one(dw[j] >> 16, sw[j] >> 16, key, x + 2 * j + 1);
            ow[j] = (lo & 0xFFFFu) | (hi << 16);
        }
        __stcs(reinterpret_cast<uint4 *>(dst + x), make_uint4(ow[0], ow[1], ow[2], ow[3]));
        __stcs(reinterpret_cast<uint4 *>(src + x), make_uint4(0u, 0u, 0u, 0u));
    } else {
        for (uint32_t i = x; i < n; ++i) {
            dst[i] = uint16_t(sr_one(dst[i], src[i], key, i));
            src[i] = 0;
        }
    }
}

cudaError_t launch_sr_accumulate(uint16_t *dst, uint16_t *src, uint32_t n, uint32_t seed,
                                 uint32_t step, cudaStream_t stream) {
    const uint32_t threads = 256;
    const uint32_t nvec = uint32_t((uint64_t(n) + 7) / 8);  // n + 7 would wrap at n = 2^32 - 1
    const uint32_t grid = (nvec + threads - 1) / threads;
    sr_accumulate_kernel<<<grid, threads, 0, stream>>>(dst, src, n, sr_key(seed, step));
    return cudaPeekAtLastError();
}

}  // namespace wc
