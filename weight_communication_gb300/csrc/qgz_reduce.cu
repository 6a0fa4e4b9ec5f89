// qgz_reduce.cu -- dequantize the chunks every destination receives and
// reduce them in full precision.
//
// "ZeROPlusPlus.md", §1.2 ZeRO++ (quantized gradient communication): the
// int4 gradients are exchanged by an all-to-all instead of a reduce-scatter
// and the reduction itself runs in full precision; with two hops the second
// (inter-node) hop reduces the first hop's requantized partial sums.
//
// With the ranks simulated in one allocation the all-to-all is pure address
// arithmetic: destination k reads chunk c(k) of every source buffer, where
// the sources sit N elements apart.  Flat (G = 1): R sources (the ranks'
// send buffers), c(k) = k.  Second hop (G > 1): G sources (one per group:
// the first-hop outputs of its L units, N elements in all), c(k) = l*G + g
// for k = g*L + l.
//
// Grid: y = destination, x = 8-output groups of its shard.  One thread makes
// 8 consecutive outputs: per source one 32-bit word of codes (coalesced,
// 128 B per warp instruction) and one scale, then the 8 sums in source
// order.  Sources are fetched 8 at a time before any add, so that enough
// loads are in flight per thread; the codes are unpacked with byte permutes
// and exact fp32 subtractions (wc_device.cuh), keeping the conversion pipe
// idle -- the per-code work is one permute, one subtract, one multiply and
// one add.
#include "wc_device.cuh"
#include "wc_internal.h"

namespace wc {

template <bool OUT_BF16>
__global__ void __launch_bounds__(256)
dequant_reduce_kernel(const uint8_t *__restrict__ codes, const float *__restrict__ scales,
                      QgzGeometry geo, uint32_t nsrc, uint32_t log2_b, float out_scale,
                      void *__restrict__ out) {
    const uint32_t k = blockIdx.y;  // destination
    const uint32_t v = blockIdx.x * blockDim.x + threadIdx.x;
    if (uint64_t(v) * 8u >= geo.S) return;
    const uint32_t i = v * 8u;  // offset in the shard
    uint32_t chunk = k;
    if (geo.G > 1) {
        const uint32_t grp = k / geo.L;
        chunk = (k - grp * geo.L) * geo.G + grp;
    }
    const uint32_t base = chunk * geo.S + i;
    const uint8_t *cp = codes + base / 2;
    const float *sp = scales + (base >> log2_b);
    const uint32_t cstride = geo.N / 2;         // bytes between sources
    const uint32_t sstride = geo.N >> log2_b;   // scales between sources

    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (uint32_t s0 = 0; s0 < nsrc; s0 += 8) {
        uint32_t w[8];
        float sc[8];
        const uint32_t nb = min(8u, nsrc - s0);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            if (t < nb) {
                w[t] = __ldcs(reinterpret_cast<const unsigned int *>(cp + (s0 + t) * cstride));
                sc[t] = __ldg(sp + (s0 + t) * sstride);
            }
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            if (t < nb) {
                float f[8];
                unpack_int4x8(w[t], f);
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], dequant(f[j], sc[t]));
            }
        }
    }

    const uint32_t o = k * geo.S + i;
    if (OUT_BF16) {
        uint32_t h[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) h[j] = f32_to_bf16_bits(__fmul_rn(acc[j], out_scale));
        uint4 pk = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                              h[6] | (h[7] << 16));
        __stcs(reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + o), pk);
    } else {
        float *dst = static_cast<float *>(out) + o;
        __stcs(reinterpret_cast<float4 *>(dst),
               make_float4(__fmul_rn(acc[0], out_scale), __fmul_rn(acc[1], out_scale),
                           __fmul_rn(acc[2], out_scale), __fmul_rn(acc[3], out_scale)));
        __stcs(reinterpret_cast<float4 *>(dst + 4),
               make_float4(__fmul_rn(acc[4], out_scale), __fmul_rn(acc[5], out_scale),
                           __fmul_rn(acc[6], out_scale), __fmul_rn(acc[7], out_scale)));
    }
}

cudaError_t launch_dequant_reduce(const uint8_t *codes, const float *scales,
                                  const QgzGeometry &geo, int B, float out_scale, void *out,
                                  bool out_bf16, cudaStream_t stream) {
    uint32_t log2_b = 0;
    while ((1u << log2_b) < uint32_t(B)) ++log2_b;
    const uint32_t nsrc = geo.G > 1 ? geo.G : geo.R;
    const uint32_t threads = 256;
    const dim3 grid((geo.S / 8 + threads - 1) / threads, geo.R);
    if (out_bf16)
        dequant_reduce_kernel<true><<<grid, threads, 0, stream>>>(codes, scales, geo, nsrc,
                                                                   log2_b, out_scale, out);
    else
        dequant_reduce_kernel<false><<<grid, threads, 0, stream>>>(codes, scales, geo, nsrc,
                                                                    log2_b, out_scale, out);
    return cudaPeekAtLastError();
}

}  // namespace wc
