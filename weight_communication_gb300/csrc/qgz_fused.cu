// qgz_fused.cu -- the whole flat qgZ step in one kernel (error-feedback
// compensation and int4 quantization of every rank, and the full-precision
// reduce of every destination), and the hierarchical step's first stage in
// one kernel (the same quantization fused with the intra-group reduce and its
// requantization), without the codes round-tripping through HBM.
//
// "ZeROPlusPlus.md", §1.2 ZeRO++ (quantized gradient communication): block
// int4 quantization, all-to-all, full-precision reduce, and CUDA kernel
// fusion to cut latency; "Merge LoCo with Zero++" (DeepSpeed PR #6730),
// Overview: error feedback on the 4-bit gradients before communication, at
// the cost of the error buffer's memory (kept here in fp32, bf16, or int8
// with one fp32 scale per block).
//
// With every simulated rank in the same HBM, one warp can own one block of
// one destination shard for all ranks at once: for r = 0..R-1 it compensates
// and quantizes rank r's block (same arithmetic as wc_ef_quant_int4 and its
// bf16 and int8 error-buffer forms), updates rank r's error buffer,
// optionally writes the codes and the scale (the wire message), and adds the
// dequantized values to the running fp32 sum in rank order (same arithmetic
// as wc_dequant_reduce).  Per gradient element this moves 10 bytes with the
// fp32 buffer (bf16 g, fp32 e read and written), 6 with bf16 and 4 plus the
// block scales with int8, instead of those + 0.5 + the reduce's re-read of
// the codes.  The next rank's block is loaded while the current one is
// processed.
#include "int8_error_block.cuh"
#include "wc_device.cuh"
#include "wc_internal.h"

namespace wc {

constexpr int kEfModeNone = 0;

// The stored error of a lane's 4 consecutive elements at element x, as raw
// bits (fp32: 4 values; bf16: 2 words; int8: 1 word of codes).
template <int EF>
__device__ __forceinline__ float4 load_error_raw(const void *ef, uint32_t x) {
    if (EF == kEfModeF32) return ld_stream_f4(static_cast<const float *>(ef) + x);
    if (EF == kEfModeBf16) {
        const uint2 v = ld_stream_u2(static_cast<const uint16_t *>(ef) + x);
        return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), 0.f, 0.f);
    }
    if (EF == kEfModeInt8) {
        const uint32_t v =
            __ldcs(reinterpret_cast<const unsigned int *>(static_cast<const int8_t *>(ef) + x));
        return make_float4(__uint_as_float(v), 0.f, 0.f, 0.f);
    }
    return make_float4(0.f, 0.f, 0.f, 0.f);
}

// The 4 stored errors as fp32: fp32 as is, bf16 widened exactly.
template <int EF>
__device__ __forceinline__ void decode_error(const float4 &raw, float e[4]) {
    if (EF == kEfModeF32) {
        e[0] = raw.x; e[1] = raw.y; e[2] = raw.z; e[3] = raw.w;
    } else if (EF == kEfModeBf16) {
        const uint32_t a = __float_as_uint(raw.x), b = __float_as_uint(raw.y);
        e[0] = bf16_bits_to_f32(a & 0xFFFFu); e[1] = bf16_bits_to_f32(a >> 16);
        e[2] = bf16_bits_to_f32(b & 0xFFFFu); e[3] = bf16_bits_to_f32(b >> 16);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) e[j] = 0.0f;
    }
}

// Loads of a rank's block into registers (zeros outside the buffers): gv the
// bf16 gradients, er the raw stored errors, es the stored int8 block scale.
template <int B, int EF>
__device__ __forceinline__ void load_rank_block(const uint16_t *__restrict__ g,
                                                const void *__restrict__ ef,
                                                const float *__restrict__ ef_scales, uint32_t xr,
                                                uint32_t total, int lane, uint2 (&gv)[B / 128],
                                                float4 (&er)[B / 128], float &es) {
#pragma unroll
    for (int k = 0; k < B / 128; ++k) {
        const uint32_t x = xr + 128u * k + 4u * lane;
        gv[k] = make_uint2(0u, 0u);
        er[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (WC_IN_BOUNDS(uint64_t(x) + 4 <= total)) {
            gv[k] = ld_stream_u2(g + x);
            if (EF != kEfModeNone) er[k] = load_error_raw<EF>(ef, x);
        }
    }
    es = 0.0f;
    if (EF == kEfModeInt8 && WC_IN_BOUNDS(xr / B < total / B)) es = __ldg(ef_scales + xr / B);
}

// A rank's block (B elements, a whole warp; lane t holds elements
// 128k + 4t + j) in registers, as load_rank_block leaves it.  Runs the
// rank's error-feedback quantization (compensation, block absmax, scale,
// int4 codes, error update in the buffer's form), writes the codes at send
// position cr and the scale when WRITE_CODES, and adds the dequantized
// values into acc (from +0, in the order the caller visits the ranks).  xr
// is the block's first gradient element; total = R*N bounds every access.
// The int8 buffer takes the packed routine of the stand-alone quantization
// (int8ef_block), the other forms the scalar chain of wc_ef_quant_int4.  S1:
// the error scale s is 1, so s*e is e itself (exact for every finite e) and
// its multiply is left out.
template <int B, int EF, bool WRITE_CODES, bool S1>
__device__ __forceinline__ void quantize_rank_block(
    const uint2 (&gv)[B / 128], const float4 (&er)[B / 128], float es, float (&acc)[B / 128][4],
    void *__restrict__ ef, float *__restrict__ ef_scales, uint8_t *__restrict__ codes,
    float *__restrict__ scales, uint32_t xr, uint32_t cr, uint32_t total, int lane, float s,
    float beta, float one_minus_beta, const Ops2 &ops) {
    constexpr int K = B / 128;
    if constexpr (EF == kEfModeInt8) {
        uint32_t e8w[K];
#pragma unroll
        for (int k = 0; k < K; ++k) e8w[k] = __float_as_uint(er[k].x);
        int8ef_block<B, S1, WRITE_CODES, true>(gv, e8w, es, static_cast<int8_t *>(ef),
                                                  ef_scales, codes, scales, total, xr, cr, lane,
                                                  s, beta, one_minus_beta, ops, acc);
    } else {
        constexpr bool HAS_EF = EF != kEfModeNone;
        float c[K][4];
        float e[K][4];
        float m = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const float gf[4] = {bf16_bits_to_f32(gv[k].x & 0xFFFFu),
                                 bf16_bits_to_f32(gv[k].x >> 16),
                                 bf16_bits_to_f32(gv[k].y & 0xFFFFu),
                                 bf16_bits_to_f32(gv[k].y >> 16)};
            decode_error<EF>(er[k], e[k]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                c[k][j] = HAS_EF ? __fadd_rn(gf[j], S1 ? e[k][j] : __fmul_rn(s, e[k][j])) : gf[j];
                m = fmaxf(m, fabsf(c[k][j]));
            }
        }
        m = group_max<kWarp>(m);
        const BlockScale bs = block_scale<7>(m);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const uint32_t x = xr + 128u * k + 4u * lane;
            uint32_t packed = 0;
            float o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const QCode qc = quant_code<7>(c[k][j], bs);
                const float d = dequant(qc.q, bs.scale);
                acc[k][j] = __fadd_rn(acc[k][j], d);
                if (WRITE_CODES) packed |= (qc.bits & 15u) << (4 * j);
                o[j] = HAS_EF ? __fadd_rn(__fmul_rn(beta, e[k][j]),
                                          __fmul_rn(one_minus_beta, __fsub_rn(c[k][j], d)))
                              : 0.0f;
            }
            if (WC_IN_BOUNDS(uint64_t(x) + 4 <= total)) {
                if (EF == kEfModeF32)
                    __stcs(reinterpret_cast<float4 *>(static_cast<float *>(ef) + x),
                           make_float4(o[0], o[1], o[2], o[3]));
                if (EF == kEfModeBf16)
                    __stcs(reinterpret_cast<uint2 *>(static_cast<uint16_t *>(ef) + x),
                           make_uint2(f32x2_to_bf16x2_bits(o[0], o[1]),
                                      f32x2_to_bf16x2_bits(o[2], o[3])));
            }
            const uint32_t pos = cr + 128u * k + 4u * lane;
            if (WRITE_CODES && WC_IN_BOUNDS(uint64_t(pos) + 4 <= total))
                __stcs(reinterpret_cast<unsigned short *>(codes + pos / 2),
                       (unsigned short)packed);
        }
        if (WRITE_CODES && lane == 0 && WC_IN_BOUNDS(cr / B < total / B))
            __stcs(scales + cr / B, bs.scale);
    }
}

// Launch bounds: the low-precision buffers move fewer bytes per element, so a
// warp has fewer in flight, and more resident warps pay.  At B <= 256, on the
// single-hop workload, bit-identical: bf16 under a register budget for 6 CTAs
// per SM (40 registers, no spill) 0.442-0.456 -> 0.407-0.418 ms; int8 for 4
// (64 registers, no spill) 0.423 -> 0.383 ms, where 5 spills and prefetching
// two or three ranks ahead was slower.  The fp32 form (10.5 bytes per
// element) measured the same under every budget.
template <int B, int EF>
constexpr int fused_step_min_ctas() {
    return B > 256 ? 1 : EF == kEfModeBf16 ? 6 : EF == kEfModeInt8 ? 4 : 1;
}

template <int B, int EF, bool WRITE_CODES, bool OUT_BF16, bool S1>
__global__ void __launch_bounds__(256, fused_step_min_ctas<B, EF>())
qgz_fused_step_kernel(const uint16_t *__restrict__ g, void *__restrict__ ef,
                      float *__restrict__ ef_scales, uint8_t *__restrict__ codes,
                      float *__restrict__ scales, QgzGeometry geo, float s, float beta,
                      float one_minus_beta, float out_scale, void *__restrict__ out,
                      Exact2 kc) {
    static_assert(B >= 128 && B % 128 == 0, "one warp per block");
    constexpr int K = B / 128;
    const int lane = threadIdx.x & (kWarp - 1);
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) / kWarp;
    if (uint64_t(warp) * B >= geo.N) return;  // one item per block of a rank's N
    const uint32_t x0 = warp * uint32_t(B);     // element offset inside every rank
    const Ops2 ops(kc);

    float acc[K][4];
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[k][j] = 0.0f;
    uint2 gv[K];
    float4 er[K];
    float es;
    load_rank_block<B, EF>(g, ef, ef_scales, x0, geo.total, lane, gv, er, es);

    for (uint32_t r = 0; r < geo.R; ++r) {
        const uint32_t xr = r * geo.N + x0;  // with G = 1 the send position is xr too
        uint2 gn[K];
        float4 en[K];
        float esn = 0.0f;
        if (r + 1 < geo.R)  // prefetch rank r + 1
            load_rank_block<B, EF>(g, ef, ef_scales, xr + geo.N, geo.total, lane, gn, en, esn);
        quantize_rank_block<B, EF, WRITE_CODES, S1>(gv, er, es, acc, ef, ef_scales, codes, scales,
                                                    xr, xr, geo.total, lane, s, beta,
                                                    one_minus_beta, ops);
        if (r + 1 < geo.R) {
#pragma unroll
            for (int k = 0; k < K; ++k) {
                gv[k] = gn[k];
                er[k] = en[k];
            }
            es = esn;
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

template <int B, int EF, bool WRITE_CODES, bool S1>
static cudaError_t launch_fused_3(const uint16_t *g, void *ef, float *ef_scales, uint8_t *codes,
                                  float *scales, const QgzGeometry &geo, float s, float beta,
                                  float out_scale, void *out, bool out_bf16, cudaStream_t stream) {
    const uint32_t items = geo.N / B;
    const uint32_t threads = 256;
    const uint32_t grid = (items + threads / kWarp - 1) / (threads / kWarp);
    const float omb = 1.0f - beta;
    if (out_bf16)
        qgz_fused_step_kernel<B, EF, WRITE_CODES, true, S1><<<grid, threads, 0, stream>>>(
            g, ef, ef_scales, codes, scales, geo, s, beta, omb, out_scale, out,
            exact2_constants());
    else
        qgz_fused_step_kernel<B, EF, WRITE_CODES, false, S1><<<grid, threads, 0, stream>>>(
            g, ef, ef_scales, codes, scales, geo, s, beta, omb, out_scale, out,
            exact2_constants());
    return cudaPeekAtLastError();
}

// The low-precision buffers' forms are issue-bound, so they also come in a
// form for s = 1; the fp32 form is HBM-bound and takes the general one.
template <int EF>
constexpr bool has_s1_form() {
    return EF == kEfModeBf16 || EF == kEfModeInt8;
}

template <int B, int EF, bool S1>
static cudaError_t launch_fused_s(const uint16_t *g, void *ef, float *ef_scales, uint8_t *codes,
                                  float *scales, const QgzGeometry &geo, float s, float beta,
                                  float out_scale, void *out, bool out_bf16, cudaStream_t stream) {
    if (codes)
        return launch_fused_3<B, EF, true, S1>(g, ef, ef_scales, codes, scales, geo, s, beta,
                                               out_scale, out, out_bf16, stream);
    return launch_fused_3<B, EF, false, S1>(g, ef, ef_scales, codes, scales, geo, s, beta,
                                            out_scale, out, out_bf16, stream);
}

template <int B, int EF>
static cudaError_t launch_fused_2(const uint16_t *g, void *ef, float *ef_scales, uint8_t *codes,
                                  float *scales, const QgzGeometry &geo, float s, float beta,
                                  float out_scale, void *out, bool out_bf16, cudaStream_t stream) {
    if constexpr (has_s1_form<EF>()) {
        if (s == 1.0f)
            return launch_fused_s<B, EF, true>(g, ef, ef_scales, codes, scales, geo, s, beta,
                                               out_scale, out, out_bf16, stream);
    }
    return launch_fused_s<B, EF, false>(g, ef, ef_scales, codes, scales, geo, s, beta, out_scale,
                                        out, out_bf16, stream);
}

template <int B>
static cudaError_t launch_fused_b(const uint16_t *g, void *ef, int ef_mode, float *ef_scales,
                                  uint8_t *codes, float *scales, const QgzGeometry &geo, float s,
                                  float beta, float out_scale, void *out, bool out_bf16,
                                  cudaStream_t stream) {
    if (ef == nullptr)
        return launch_fused_2<B, kEfModeNone>(g, ef, ef_scales, codes, scales, geo, s, beta,
                                              out_scale, out, out_bf16, stream);
    switch (ef_mode) {
        case kEfModeF32:
            return launch_fused_2<B, kEfModeF32>(g, ef, ef_scales, codes, scales, geo, s, beta,
                                                 out_scale, out, out_bf16, stream);
        case kEfModeBf16:
            return launch_fused_2<B, kEfModeBf16>(g, ef, ef_scales, codes, scales, geo, s, beta,
                                                  out_scale, out, out_bf16, stream);
        case kEfModeInt8:
            return launch_fused_2<B, kEfModeInt8>(g, ef, ef_scales, codes, scales, geo, s, beta,
                                                  out_scale, out, out_bf16, stream);
        default: return cudaErrorInvalidValue;
    }
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
// wc_ef_quant_int4 or its bf16 and int8 error-buffer forms), writes its codes
// and scale at the send position when asked to, and adds the dequantized
// values to the running fp32 sum (from +0, in local-rank order); then it
// requantizes the sum to the first hop's output (the arithmetic of
// wc_dequant_reduce_requant, or with HAS_EF1 that of
// wc_dequant_reduce_requant_ef: the sum compensated with the first hop's own
// error buffer, which is then updated).  Every (rank, slice, block) belongs
// to exactly one output block, so every gradient block is quantized once,
// and the codes are never read back from memory.  The next rank's block is
// loaded while the current one is processed.  Up to B = 512 a register
// budget for three CTAs of 256 threads per SM (80 registers, a 12-byte spill
// with the fp32 error buffer and codes) keeps more loads in flight than the
// compiler's own choice of 122 registers: about 1 % faster at B = 512.
template <int B, int EF, bool WRITE_CODES, bool HAS_EF1, bool S1>
__global__ void __launch_bounds__(256, B <= 512 ? 3 : 1)
qgz_first_hop_fused_kernel(const uint16_t *__restrict__ g, void *__restrict__ ef,
                           float *__restrict__ ef_scales, uint8_t *__restrict__ codes,
                           float *__restrict__ scales, QgzGeometry geo, float s, float beta,
                           float one_minus_beta, uint8_t *__restrict__ out_codes,
                           float *__restrict__ out_scales, float *__restrict__ ef1, Exact2 kc) {
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
    [[maybe_unused]] const uint64_t total_out = uint64_t(geo.G) * geo.N;
    const Ops2 ops(kc);

    float acc[K][4];
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[k][j] = 0.0f;
    uint2 gv[K];
    float4 er[K];
    float es;
    load_rank_block<B, EF>(g, ef, ef_scales, xbase, geo.total, lane, gv, er, es);

    for (uint32_t lq = 0; lq < geo.L; ++lq) {
        const uint32_t xr = xbase + lq * geo.N;
        uint2 gn[K];
        float4 en[K];
        float esn = 0.0f;
        if (lq + 1 < geo.L)  // prefetch the next local rank's block
            load_rank_block<B, EF>(g, ef, ef_scales, xr + geo.N, geo.total, lane, gn, en, esn);
        quantize_rank_block<B, EF, WRITE_CODES, S1>(gv, er, es, acc, ef, ef_scales, codes, scales,
                                                    xr, cbase + lq * geo.N, geo.total, lane, s,
                                                    beta, one_minus_beta, ops);
        if (lq + 1 < geo.L) {
#pragma unroll
            for (int k = 0; k < K; ++k) {
                gv[k] = gn[k];
                er[k] = en[k];
            }
            es = esn;
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

template <int B, int EF, bool WRITE_CODES, bool HAS_EF1, bool S1>
static cudaError_t launch_first_hop_fused_4(const uint16_t *g, void *ef, float *ef_scales,
                                            uint8_t *codes, float *scales, const QgzGeometry &geo,
                                            float s, float beta, uint8_t *out_codes,
                                            float *out_scales, float *ef1, cudaStream_t stream) {
    const uint32_t threads = 256;
    const uint32_t warps = geo.S / B;  // blocks per sub-slice
    const dim3 grid((warps + threads / kWarp - 1) / (threads / kWarp), geo.G, geo.R);
    qgz_first_hop_fused_kernel<B, EF, WRITE_CODES, HAS_EF1, S1><<<grid, threads, 0, stream>>>(
        g, ef, ef_scales, codes, scales, geo, s, beta, 1.0f - beta, out_codes, out_scales, ef1,
        exact2_constants());
    return cudaPeekAtLastError();
}

template <int B, int EF, bool S1>
static cudaError_t launch_first_hop_fused_s(const uint16_t *g, void *ef, float *ef_scales,
                                            uint8_t *codes, float *scales, const QgzGeometry &geo,
                                            float s, float beta, uint8_t *out_codes,
                                            float *out_scales, float *ef1, cudaStream_t stream) {
    if (codes) {
        if (ef1)
            return launch_first_hop_fused_4<B, EF, true, true, S1>(
                g, ef, ef_scales, codes, scales, geo, s, beta, out_codes, out_scales, ef1, stream);
        return launch_first_hop_fused_4<B, EF, true, false, S1>(
            g, ef, ef_scales, codes, scales, geo, s, beta, out_codes, out_scales, ef1, stream);
    }
    if (ef1)
        return launch_first_hop_fused_4<B, EF, false, true, S1>(
            g, ef, ef_scales, codes, scales, geo, s, beta, out_codes, out_scales, ef1, stream);
    return launch_first_hop_fused_4<B, EF, false, false, S1>(
        g, ef, ef_scales, codes, scales, geo, s, beta, out_codes, out_scales, ef1, stream);
}

template <int B, int EF>
static cudaError_t launch_first_hop_fused_2(const uint16_t *g, void *ef, float *ef_scales,
                                            uint8_t *codes, float *scales, const QgzGeometry &geo,
                                            float s, float beta, uint8_t *out_codes,
                                            float *out_scales, float *ef1, cudaStream_t stream) {
    if constexpr (has_s1_form<EF>()) {
        if (s == 1.0f)
            return launch_first_hop_fused_s<B, EF, true>(g, ef, ef_scales, codes, scales, geo, s,
                                                         beta, out_codes, out_scales, ef1, stream);
    }
    return launch_first_hop_fused_s<B, EF, false>(g, ef, ef_scales, codes, scales, geo, s, beta,
                                                  out_codes, out_scales, ef1, stream);
}

template <int B>
static cudaError_t launch_first_hop_fused_b(const uint16_t *g, void *ef, int ef_mode,
                                            float *ef_scales, uint8_t *codes, float *scales,
                                            const QgzGeometry &geo, float s, float beta,
                                            uint8_t *out_codes, float *out_scales, float *ef1,
                                            cudaStream_t stream) {
    if (ef == nullptr)
        return launch_first_hop_fused_2<B, kEfModeNone>(g, ef, ef_scales, codes, scales, geo, s,
                                                        beta, out_codes, out_scales, ef1, stream);
    switch (ef_mode) {
        case kEfModeF32:
            return launch_first_hop_fused_2<B, kEfModeF32>(g, ef, ef_scales, codes, scales, geo,
                                                           s, beta, out_codes, out_scales, ef1,
                                                           stream);
        case kEfModeBf16:
            return launch_first_hop_fused_2<B, kEfModeBf16>(g, ef, ef_scales, codes, scales, geo,
                                                            s, beta, out_codes, out_scales, ef1,
                                                            stream);
        case kEfModeInt8:
            return launch_first_hop_fused_2<B, kEfModeInt8>(g, ef, ef_scales, codes, scales, geo,
                                                            s, beta, out_codes, out_scales, ef1,
                                                            stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_qgz_first_hop_fused(const uint16_t *g, void *ef, int ef_mode,
                                       float *ef_scales, uint8_t *codes, float *scales,
                                       const QgzGeometry &geo, int B, float s, float beta,
                                       uint8_t *out_codes, float *out_scales, float *ef1,
                                       cudaStream_t stream) {
#define WC_FH_B(BB)                                                                         \
    case BB:                                                                                \
        return launch_first_hop_fused_b<BB>(g, ef, ef_mode, ef_scales, codes, scales, geo, s, \
                                            beta, out_codes, out_scales, ef1, stream);
    switch (B) {
        WC_FH_B(128)
        WC_FH_B(256)
        WC_FH_B(512)
        WC_FH_B(1024)
        default: return cudaErrorInvalidValue;
    }
#undef WC_FH_B
}

WC_CHECK_RECORD_READER(check_record_qgz_fused)

cudaError_t launch_qgz_fused_step(const uint16_t *g, void *ef, int ef_mode, float *ef_scales,
                                  uint8_t *codes, float *scales, const QgzGeometry &geo, int B,
                                  float s, float beta, float out_scale, void *out, bool out_bf16,
                                  cudaStream_t stream) {
#define WC_FS_B(BB)                                                                          \
    case BB:                                                                                 \
        return launch_fused_b<BB>(g, ef, ef_mode, ef_scales, codes, scales, geo, s, beta,     \
                                  out_scale, out, out_bf16, stream);
    switch (B) {
        WC_FS_B(128)
        WC_FS_B(256)
        WC_FS_B(512)
        WC_FS_B(1024)
        default: return cudaErrorInvalidValue;
    }
#undef WC_FS_B
}

}  // namespace wc
