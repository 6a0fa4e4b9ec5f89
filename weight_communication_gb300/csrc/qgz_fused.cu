// qgz_fused.cu -- the whole flat qgZ step in one kernel (error-feedback
// compensation and int4 quantization of every rank, and the full-precision
// reduce of every destination), and the hierarchical step's first stage in
// one kernel (the same quantization fused with the intra-group reduce and its
// requantization), without the codes round-tripping through HBM.
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

// ---------------------------------------------------------------------------
// The hierarchical first stage in one kernel: every rank's EF-quant fused
// with the first (intra-group) hop
// ---------------------------------------------------------------------------
//
// One warp per first-hop output block: unit u = g*L + l (grid z), sub-slice
// g' (grid y), block j of the sub-slice (grid x).  The unit's sum takes, from
// each local rank l' of group g (rank g*L + l'), block j of gradient slice
// g'*L + l: the block that rank sends to local rank l for sub-slice g' (send
// position l*G + g').  For l' = 0..L-1 in order the warp runs that rank's
// error-feedback quantization of the block (the arithmetic of
// wc_ef_quant_int4), writes its codes and scale at the send position when
// asked to, and adds the dequantized values to the running fp32 sum (from
// +0, in local-rank order); then it requantizes the sum to the first hop's
// output (the arithmetic of wc_dequant_reduce_requant, or with HAS_EF1 that
// of wc_dequant_reduce_requant_ef: the sum compensated with the first hop's
// own error buffer, which is then updated).  Every (rank, slice,
// block) belongs to exactly one output block, so every gradient block is
// quantized once, and the codes are never read back from memory.  The next
// rank's block is loaded while the current one is processed.  Up to B = 512
// a register budget for three CTAs of 256 threads per SM (80 registers, a
// 12-byte spill with EF and codes) keeps more loads in flight than the
// compiler's own choice of 122 registers: about 1 % faster at B = 512.
template <int B, bool HAS_EF, bool WRITE_CODES, bool HAS_EF1>
__global__ void __launch_bounds__(256, B <= 512 ? 3 : 1)
qgz_first_hop_fused_kernel(const uint16_t *__restrict__ g, float *__restrict__ ef,
                           uint8_t *__restrict__ codes, float *__restrict__ scales,
                           QgzGeometry geo, float s, float beta, float one_minus_beta,
                           uint8_t *__restrict__ out_codes, float *__restrict__ out_scales,
                           float *__restrict__ ef1) {
    static_assert(B >= 128 && B % 128 == 0, "one warp per block");
    constexpr int K = B / 128;
    const int lane = threadIdx.x & (kWarp - 1);
    const uint32_t off = (blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp) * B;
    if (off >= geo.S) return;  // whole warp: the grid's x is rounded up
    const uint32_t gq = blockIdx.y, u = blockIdx.z;
    const uint32_t grp = u / geo.L, l = u - grp * geo.L;
    // local rank l' reads gradient elements xbase + l'*N + 128k + 4*lane and
    // writes its codes at send position cbase + l'*N + ...
    const uint32_t xbase = grp * geo.L * geo.N + (gq * geo.L + l) * geo.S + off;
    const uint32_t cbase = grp * geo.L * geo.N + (l * geo.G + gq) * geo.S + off;
    const uint32_t o0 = (u * geo.G + gq) * geo.S + off;  // first output of the block
    const uint64_t total_out = uint64_t(geo.G) * geo.N;

    float acc[K][4];
    uint2 gv[K];
    float4 ev[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[k][j] = 0.0f;
        const uint32_t x = xbase + 128u * k + 4u * lane;  // local rank 0
        gv[k] = make_uint2(0u, 0u);
        ev[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (WC_IN_BOUNDS(uint64_t(x) + 4 <= geo.total)) {
            gv[k] = ld_stream_u2(g + x);
            if (HAS_EF) ev[k] = ld_stream_f4(ef + x);
        }
    }

    for (uint32_t lq = 0; lq < geo.L; ++lq) {
        const uint32_t xr = xbase + lq * geo.N;
        uint2 gn[K];
        float4 en[K];
        if (lq + 1 < geo.L) {  // prefetch the next local rank's block
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
        const uint32_t cr = cbase + lq * geo.N;  // this rank's send position
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const uint32_t x = xr + 128u * k + 4u * lane;
            uint32_t packed = 0;
            float4 eo;
            float *o = &eo.x;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const QCode qc = quant_code<7>(c[k][j], bs);
                const float d = dequant(qc.q, bs.scale);
                acc[k][j] = __fadd_rn(acc[k][j], d);
                if (WRITE_CODES) packed |= (qc.bits & 15u) << (4 * j);
                if (HAS_EF)
                    o[j] = __fadd_rn(__fmul_rn(beta, e[k][j]),
                                     __fmul_rn(one_minus_beta, __fsub_rn(c[k][j], d)));
            }
            if (HAS_EF && WC_IN_BOUNDS(uint64_t(x) + 4 <= geo.total))
                __stcs(reinterpret_cast<float4 *>(ef + x), eo);
            const uint32_t pos = cr + 128u * k + 4u * lane;
            if (WRITE_CODES && WC_IN_BOUNDS(uint64_t(pos) + 4 <= geo.total))
                __stcs(reinterpret_cast<unsigned short *>(codes + pos / 2), (unsigned short)packed);
        }
        if (WRITE_CODES && lane == 0 && WC_IN_BOUNDS(cr / B < geo.total / B))
            __stcs(scales + cr / B, bs.scale);
        if (lq + 1 < geo.L) {
#pragma unroll
            for (int k = 0; k < K; ++k) {
                gv[k] = gn[k];
                ev[k] = en[k];
            }
        }
    }

    // requantize the block's sums for the second hop (compensated with the
    // first hop's error buffer, in output order, when it has one)
    float e1[K][4];
    if (HAS_EF1) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const uint32_t o = o0 + 128u * k + 4u * lane;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (WC_IN_BOUNDS(uint64_t(o) + 4 <= total_out)) v = ld_stream_f4(ef1 + o);
            e1[k][0] = v.x; e1[k][1] = v.y; e1[k][2] = v.z; e1[k][3] = v.w;
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[k][j] = __fadd_rn(acc[k][j], __fmul_rn(s, e1[k][j]));
        }
    }
    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
        for (int j = 0; j < 4; ++j) m = fmaxf(m, fabsf(acc[k][j]));
    m = group_max<kWarp>(m);
    const BlockScale bs = block_scale<7>(m);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        uint32_t packed = 0;
        float4 eo;
        float *eout = &eo.x;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const QCode qc = quant_code<7>(acc[k][j], bs);
            packed |= (qc.bits & 15u) << (4 * j);
            if (HAS_EF1)
                eout[j] = __fadd_rn(__fmul_rn(beta, e1[k][j]),
                                    __fmul_rn(one_minus_beta,
                                              __fsub_rn(acc[k][j], dequant(qc.q, bs.scale))));
        }
        const uint32_t o = o0 + 128u * k + 4u * lane;
        if (!WC_IN_BOUNDS(uint64_t(o) + 4 <= total_out)) continue;
        __stcs(reinterpret_cast<unsigned short *>(out_codes + o / 2), (unsigned short)packed);
        if (HAS_EF1) __stcs(reinterpret_cast<float4 *>(ef1 + o), eo);
    }
    if (lane == 0 && WC_IN_BOUNDS(uint64_t(o0 / B) < total_out / B)) __stcs(out_scales + o0 / B, bs.scale);
}

template <int B, bool HAS_EF, bool WRITE_CODES, bool HAS_EF1>
static cudaError_t launch_first_hop_fused_4(const uint16_t *g, float *ef, uint8_t *codes,
                                            float *scales, const QgzGeometry &geo, float s,
                                            float beta, uint8_t *out_codes, float *out_scales,
                                            float *ef1, cudaStream_t stream) {
    const uint32_t threads = 256;
    const uint32_t warps = geo.S / B;  // blocks per sub-slice
    const dim3 grid((warps + threads / kWarp - 1) / (threads / kWarp), geo.G, geo.R);
    qgz_first_hop_fused_kernel<B, HAS_EF, WRITE_CODES, HAS_EF1><<<grid, threads, 0, stream>>>(
        g, ef, codes, scales, geo, s, beta, 1.0f - beta, out_codes, out_scales, ef1);
    return cudaPeekAtLastError();
}

template <int B, bool HAS_EF, bool WRITE_CODES>
static cudaError_t launch_first_hop_fused_3(const uint16_t *g, float *ef, uint8_t *codes,
                                            float *scales, const QgzGeometry &geo, float s,
                                            float beta, uint8_t *out_codes, float *out_scales,
                                            float *ef1, cudaStream_t stream) {
    if (ef1)
        return launch_first_hop_fused_4<B, HAS_EF, WRITE_CODES, true>(
            g, ef, codes, scales, geo, s, beta, out_codes, out_scales, ef1, stream);
    return launch_first_hop_fused_4<B, HAS_EF, WRITE_CODES, false>(
        g, ef, codes, scales, geo, s, beta, out_codes, out_scales, ef1, stream);
}

template <int B>
static cudaError_t launch_first_hop_fused_b(const uint16_t *g, float *ef, uint8_t *codes,
                                            float *scales, const QgzGeometry &geo, float s,
                                            float beta, uint8_t *out_codes, float *out_scales,
                                            float *ef1, cudaStream_t stream) {
    if (ef) {
        if (codes)
            return launch_first_hop_fused_3<B, true, true>(g, ef, codes, scales, geo, s, beta,
                                                           out_codes, out_scales, ef1, stream);
        return launch_first_hop_fused_3<B, true, false>(g, ef, codes, scales, geo, s, beta,
                                                        out_codes, out_scales, ef1, stream);
    }
    if (codes)
        return launch_first_hop_fused_3<B, false, true>(g, ef, codes, scales, geo, s, beta,
                                                        out_codes, out_scales, ef1, stream);
    return launch_first_hop_fused_3<B, false, false>(g, ef, codes, scales, geo, s, beta,
                                                     out_codes, out_scales, ef1, stream);
}

cudaError_t launch_qgz_first_hop_fused(const uint16_t *g, float *ef, uint8_t *codes,
                                       float *scales, const QgzGeometry &geo, int B, float s,
                                       float beta, uint8_t *out_codes, float *out_scales,
                                       float *ef1, cudaStream_t stream) {
    switch (B) {
        case 128: return launch_first_hop_fused_b<128>(g, ef, codes, scales, geo, s, beta, out_codes, out_scales, ef1, stream);
        case 256: return launch_first_hop_fused_b<256>(g, ef, codes, scales, geo, s, beta, out_codes, out_scales, ef1, stream);
        case 512: return launch_first_hop_fused_b<512>(g, ef, codes, scales, geo, s, beta, out_codes, out_scales, ef1, stream);
        case 1024: return launch_first_hop_fused_b<1024>(g, ef, codes, scales, geo, s, beta, out_codes, out_scales, ef1, stream);
        default: return cudaErrorInvalidValue;
    }
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
