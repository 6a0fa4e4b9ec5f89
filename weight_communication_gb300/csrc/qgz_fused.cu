// qgz_fused.cu -- the whole flat qgZ step in one kernel: error-feedback
// compensation and int4 quantization of every rank, and the full-precision
// reduce of every destination, without the codes round-tripping through HBM.
//
// "ZeROPlusPlus.md", §1.2 ZeRO++ (quantized gradient communication): block
// int4 quantization, all-to-all, full-precision reduce, and CUDA kernel
// fusion to cut latency; "Merge LoCo with Zero++" (DeepSpeed PR #6730),
// Overview: error feedback on the 4-bit gradients before communication.
//
// With every simulated rank in the same HBM, one warp can own one block of
// one destination shard for all ranks at once: for r = 0..R-1 it compensates
// and quantizes rank r's block (same arithmetic as wc_ef_quant_int4), updates
// rank r's error buffer, optionally writes the codes and the scale (the wire
// message), and adds the dequantized values to the running fp32 sum in rank
// order (same arithmetic as wc_dequant_reduce).  Per gradient element this
// moves 10 bytes (bf16 g, fp32 e read and written) instead of 10.5 + the
// reduce's re-read of the codes.  The next rank's block is loaded while the
// current one is processed.
#include "wc_device.cuh"
#include "wc_internal.h"

namespace wc {

template <int B, bool HAS_EF, bool WRITE_CODES, bool OUT_BF16>
__global__ void __launch_bounds__(256)
qgz_fused_step_kernel(const uint16_t *__restrict__ g, float *__restrict__ ef,
                      uint8_t *__restrict__ codes, float *__restrict__ scales, QgzGeometry geo,
                      float s, float beta, float one_minus_beta, float out_scale,
                      void *__restrict__ out) {
    static_assert(B >= 128 && B % 128 == 0, "one warp per block");
    constexpr int K = B / 128;
    const int lane = threadIdx.x & (kWarp - 1);
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) / kWarp;
    if (uint64_t(warp) * B >= geo.N) return;  // one item per block of a rank's N
    const uint32_t x0 = warp * uint32_t(B);     // element offset inside every rank

    float acc[K][4];
    uint2 gv[K];
    float4 ev[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[k][j] = 0.0f;
        const uint32_t x = x0 + 128u * k + 4u * lane;  // rank 0
        gv[k] = make_uint2(0u, 0u);
        ev[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (WC_IN_BOUNDS(uint64_t(x) + 4 <= geo.total)) {
            gv[k] = ld_stream_u2(g + x);
            if (HAS_EF) ev[k] = ld_stream_f4(ef + x);
        }
    }

    for (uint32_t r = 0; r < geo.R; ++r) {
        const uint32_t xr = r * geo.N + x0;
        // prefetch rank r + 1
        uint2 gn[K];
        float4 en[K];
        if (r + 1 < geo.R) {
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const uint32_t x = xr + geo.N + 128u * k + 4u * lane;
                gn[k] = make_uint2(0u, 0u);
                en[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (WC_IN_BOUNDS(uint64_t(x) + 4 <= geo.total)) {
                    gn[k] = ld_stream_u2(g + x);
                    if (HAS_EF) en[k] = ld_stream_f4(ef + x);
                }
            }
        }
        float c[K][4];
        float e[K][4];
        float m = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const float gf[4] = {bf16_bits_to_f32(gv[k].x & 0xFFFFu), bf16_bits_to_f32(gv[k].x >> 16),
                                 bf16_bits_to_f32(gv[k].y & 0xFFFFu), bf16_bits_to_f32(gv[k].y >> 16)};
            e[k][0] = ev[k].x; e[k][1] = ev[k].y; e[k][2] = ev[k].z; e[k][3] = ev[k].w;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                c[k][j] = HAS_EF ? __fadd_rn(gf[j], __fmul_rn(s, e[k][j])) : gf[j];
                m = fmaxf(m, fabsf(c[k][j]));
            }
        }
        m = group_max<kWarp>(m);
        const BlockScale bs = block_scale<7>(m);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const uint32_t x = xr + 128u * k + 4u * lane;
            uint32_t packed = 0;
            float4 eo;
            float *o = &eo.x;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const QCode qc = quant_code<7>(c[k][j], bs);
                const float q = qc.q;
                const float d = dequant(q, bs.scale);
                acc[k][j] = __fadd_rn(acc[k][j], d);
                if (WRITE_CODES) packed |= (qc.bits & 15u) << (4 * j);
                if (HAS_EF)
                    o[j] = __fadd_rn(__fmul_rn(beta, e[k][j]),
                                     __fmul_rn(one_minus_beta, __fsub_rn(c[k][j], d)));
            }
            if (!WC_IN_BOUNDS(uint64_t(x) + 4 <= geo.total)) continue;
            if (HAS_EF) __stcs(reinterpret_cast<float4 *>(ef + x), eo);
            if (WRITE_CODES)
                __stcs(reinterpret_cast<unsigned short *>(codes + x / 2), (unsigned short)packed);
        }
        if (WRITE_CODES && lane == 0 && WC_IN_BOUNDS(xr / B < geo.total / B))
            __stcs(scales + xr / B, bs.scale);
        if (r + 1 < geo.R) {
#pragma unroll
            for (int k = 0; k < K; ++k) {
                gv[k] = gn[k];
                ev[k] = en[k];
            }
        }
    }

#pragma unroll
    for (int k = 0; k < K; ++k) {
        const uint32_t x = x0 + 128u * k + 4u * lane;  // destination-major output = slice order
        if (!WC_IN_BOUNDS(uint64_t(x) + 4 <= geo.N)) continue;
        if (OUT_BF16) {
            __stcs(reinterpret_cast<uint2 *>(static_cast<uint16_t *>(out) + x),
                   make_uint2(f32x2_to_bf16x2_bits(__fmul_rn(acc[k][0], out_scale),
                                                   __fmul_rn(acc[k][1], out_scale)),
                              f32x2_to_bf16x2_bits(__fmul_rn(acc[k][2], out_scale),
                                                   __fmul_rn(acc[k][3], out_scale))));
        } else {
            __stcs(reinterpret_cast<float4 *>(static_cast<float *>(out) + x),
                   make_float4(__fmul_rn(acc[k][0], out_scale), __fmul_rn(acc[k][1], out_scale),
                               __fmul_rn(acc[k][2], out_scale), __fmul_rn(acc[k][3], out_scale)));
        }
    }
}

template <int B, bool HAS_EF, bool WRITE_CODES>
static cudaError_t launch_fused_3(const uint16_t *g, float *ef, uint8_t *codes, float *scales,
                                  const QgzGeometry &geo, float s, float beta, float out_scale,
                                  void *out, bool out_bf16, cudaStream_t stream) {
    const uint32_t items = geo.N / B;
    const uint32_t threads = 256;
    const uint32_t grid = (items + threads / kWarp - 1) / (threads / kWarp);
    const float omb = 1.0f - beta;
    if (out_bf16)
        qgz_fused_step_kernel<B, HAS_EF, WRITE_CODES, true><<<grid, threads, 0, stream>>>(
            g, ef, codes, scales, geo, s, beta, omb, out_scale, out);
    else
        qgz_fused_step_kernel<B, HAS_EF, WRITE_CODES, false><<<grid, threads, 0, stream>>>(
            g, ef, codes, scales, geo, s, beta, omb, out_scale, out);
    return cudaPeekAtLastError();
}

template <int B>
static cudaError_t launch_fused_b(const uint16_t *g, float *ef, uint8_t *codes, float *scales,
                                  const QgzGeometry &geo, float s, float beta, float out_scale,
                                  void *out, bool out_bf16, cudaStream_t stream) {
    if (ef) {
        if (codes)
            return launch_fused_3<B, true, true>(g, ef, codes, scales, geo, s, beta, out_scale,
                                                 out, out_bf16, stream);
        return launch_fused_3<B, true, false>(g, ef, codes, scales, geo, s, beta, out_scale, out,
                                              out_bf16, stream);
    }
    if (codes)
        return launch_fused_3<B, false, true>(g, ef, codes, scales, geo, s, beta, out_scale, out,
                                              out_bf16, stream);
    return launch_fused_3<B, false, false>(g, ef, codes, scales, geo, s, beta, out_scale, out,
                                           out_bf16, stream);
}

WC_CHECK_RECORD_READER(check_record_qgz_fused)

cudaError_t launch_qgz_fused_step(const uint16_t *g, float *ef, uint8_t *codes, float *scales,
                                  const QgzGeometry &geo, int B, float s, float beta,
                                  float out_scale, void *out, bool out_bf16,
                                  cudaStream_t stream) {
    switch (B) {
        case 128: return launch_fused_b<128>(g, ef, codes, scales, geo, s, beta, out_scale, out, out_bf16, stream);
        case 256: return launch_fused_b<256>(g, ef, codes, scales, geo, s, beta, out_scale, out, out_bf16, stream);
        case 512: return launch_fused_b<512>(g, ef, codes, scales, geo, s, beta, out_scale, out, out_bf16, stream);
        case 1024: return launch_fused_b<1024>(g, ef, codes, scales, geo, s, beta, out_scale, out, out_bf16, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace wc
