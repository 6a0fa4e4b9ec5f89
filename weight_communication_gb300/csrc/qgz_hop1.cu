// qgz_hop1.cu -- first (intra-group) hop of the hierarchical qgZ reduce:
// dequantize the L chunks a unit receives from its group, add them in fp32 in
// local-rank order, and requantize the partial sums to int4 for the second
// hop -- optionally compensating the requantization with an error buffer.
//
// "ZeROPlusPlus.md", §1.2 ZeRO++ (quantized gradient communication): reduce
// intra-node first, then inter-node, in full precision, with the data on the
// wire block-quantized to int4.  "Merge LoCo with Zero++" (DeepSpeed PR
// #6730), review thread: the error-feedback buffers live on each parameter as
// `inter_ef_buf`, the buffer of the inter-node message -- here the optional
// fp32 error e1 of each requantized value: c = p + s*e1, q = Q4(c),
// e1 <- beta*e1 + (1 - beta)*(c - q*scale).
//
// Output element o (over all R units, G*S each) belongs to unit u = g*L + l,
// sub-slice g' and offset i; its inputs are the codes at position
// (g*L + l')*N + (l*G + g')*S + i for l' = 0..L-1.  Per output the kernel
// reads L codes and scales (L/2 + 4L/B bytes) and writes half a byte, so it
// is bound by instruction issue, not bytes, and the work goes into the
// instructions per code.
//
// Fast path (B = 256, 512, 1024 and L a power of two up to 16): one warp per
// output block, lane t owning outputs t*B/32 .. t*B/32 + B/32 - 1, the source
// count a template parameter so that all L loads are issued before the adds,
// and a 3-D grid (block, sub-slice, unit) that spares the index divisions.
// The warp's outputs are one block of every source, so a source's codes take
// only 16 distinct products: each lane forms one of them, and a code's
// product is fetched by one shuffle indexed by its nibble (product_table in
// wc_device.cuh) -- a shift, a shuffle and half a packed add per code, in
// place of an unpack, an unbias, a multiply and an add.  The shuffles run on
// the load/store pipe, so the last source takes the byte-permute path, in
// packed form, on the ALU and FMA pipes.  The requantization is packed as
// well (requantize_pairs).  With its error buffer the hop is bound by HBM,
// and the shuffles would compete with the error traffic for the load/store
// pipe, so that form keeps the scalar byte-permute path.  Other shapes: a
// general kernel (lane groups of 8 consecutive outputs, sources fetched 8 at
// a time, scalar arithmetic).
#include "wc_device.cuh"
#include "wc_internal.h"

namespace wc {

// Code position, in a rank's buffer of the first source (local rank 0 of the
// group), of output element o; consecutive sources are N codes apart.
__device__ __forceinline__ uint32_t hop1_source(const QgzGeometry &geo, uint32_t o) {
    const uint32_t unit_len = geo.G * geo.S;
    const uint32_t u = o / unit_len;
    const uint32_t rem = o - u * unit_len;
    const uint32_t gq = rem / geo.S;
    const uint32_t i = rem - gq * geo.S;
    const uint32_t grp = u / geo.L;
    const uint32_t l = u - grp * geo.L;
    return grp * geo.L * geo.N + (l * geo.G + gq) * geo.S + i;
}

// W consecutive 32-bit code words (8 codes each) from p.
template <int W>
__device__ __forceinline__ void load_words(const uint8_t *p, uint32_t w[W]) {
    if (W == 1) {
        w[0] = __ldcs(reinterpret_cast<const unsigned int *>(p));
    } else if (W == 2) {
        const uint2 v = __ldcs(reinterpret_cast<const uint2 *>(p));
        w[0] = v.x;
        w[1] = v.y;
    } else {
#pragma unroll
        for (int q = 0; q < W; q += 4) {
            const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(p) + q / 4);
            w[q] = v.x;
            w[q + 1] = v.y;
            w[q + 2] = v.z;
            w[q + 3] = v.w;
        }
    }
}

template <int W>
__device__ __forceinline__ void store_words(uint8_t *p, const uint32_t w[W]) {
    if (W == 1) {
        __stcs(reinterpret_cast<unsigned int *>(p), w[0]);
    } else if (W == 2) {
        __stcs(reinterpret_cast<uint2 *>(p), make_uint2(w[0], w[1]));
    } else {
#pragma unroll
        for (int q = 0; q < W; q += 4)
            __stcs(reinterpret_cast<uint4 *>(p) + q / 4, make_uint4(w[q], w[q + 1], w[q + 2], w[q + 3]));
    }
}

// E (a multiple of 8) consecutive values of one lane, in place: compensation
// c = p + s*e1 (HAS_EF), absmax over the LPB-lane group that holds the block,
// int4 codes to out_codes at code position o, the error update, the scale.
// out_ok (false only in a checked build, for a lane whose outputs would lie
// outside the G*N outputs) skips every access of the lane.
template <int E, int LPB, bool HAS_EF, int B>
__device__ __forceinline__ void requantize_lane(float p[E], uint32_t o, bool out_ok, int lane,
                                                uint8_t *__restrict__ out_codes,
                                                float *__restrict__ out_scales,
                                                float *__restrict__ ef1, float s, float beta,
                                                float one_minus_beta) {
    float e[E];
    if (HAS_EF) {
#pragma unroll
        for (int q = 0; q < E / 4; ++q) {
            const float4 v = out_ok ? ld_stream_f4(ef1 + o + 4 * q) : make_float4(0.f, 0.f, 0.f, 0.f);
            e[4 * q] = v.x;
            e[4 * q + 1] = v.y;
            e[4 * q + 2] = v.z;
            e[4 * q + 3] = v.w;
        }
#pragma unroll
        for (int j = 0; j < E; ++j) p[j] = __fadd_rn(p[j], __fmul_rn(s, e[j]));
    }
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < E; ++j) m = fmaxf(m, fabsf(p[j]));
    m = group_max<LPB>(m);
    const BlockScale bs = block_scale<7>(m);
    uint32_t words[E / 8];
    float q[E];
#pragma unroll
    for (int wq = 0; wq < E / 8; ++wq) {
        uint32_t packed = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const QCode qc = quant_code<7>(p[8 * wq + j], bs);
            q[8 * wq + j] = qc.q;
            packed |= (qc.bits & 15u) << (4 * j);
        }
        words[wq] = packed;
    }
    if (out_ok) store_words<E / 8>(out_codes + o / 2, words);
    if (HAS_EF && out_ok) {
#pragma unroll
        for (int qd = 0; qd < E / 4; ++qd) {
            float4 v;
            float *vo = &v.x;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int x = 4 * qd + j;
                const float d = dequant(q[x], bs.scale);
                vo[j] = __fadd_rn(__fmul_rn(beta, e[x]),
                                  __fmul_rn(one_minus_beta, __fsub_rn(p[x], d)));
            }
            __stcs(reinterpret_cast<float4 *>(ef1 + o + 4 * qd), v);
        }
    }
    if (out_ok && (lane & (LPB - 1)) == 0) __stcs(out_scales + o / B, bs.scale);
}

// requantize_lane (without error feedback) on the E values of a lane held as
// E/2 packed pairs (p[j]: values 2j, 2j+1), in packed exact arithmetic, with
// the codes packed through the biased rounding of kRoundShift4: the same
// codes and scale bit for bit.  The whole warp holds one block.
template <int E, int B>
__device__ __forceinline__ void requantize_pairs(const f32x2 p[E / 2], uint32_t o, bool out_ok,
                                                 int lane, uint8_t *__restrict__ out_codes,
                                                 float *__restrict__ out_scales, const Ops2 &ops) {
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < E / 2; ++j) {
        float a, b;
        unpack2(p[j], a, b);
        m = max3(m, fabsf(a), fabsf(b));
    }
    m = group_max<kWarp>(m);
    const BlockScale bs = block_scale<7>(m);
    const f32x2 inv2 = pack2(bs.inv, bs.inv);
    const f32x2 shift = pack2(kRoundShift4, kRoundShift4);
    uint32_t words[E / 8];
#pragma unroll
    for (int wq = 0; wq < E / 8; ++wq) {
        uint32_t pairs[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            float r0, r1;
            unpack2(ops.add(ops.mul(p[4 * wq + jj], inv2), shift), r0, r1);
            pairs[jj] = __float_as_uint(r0) + (__float_as_uint(r1) << 4);  // (q0 + 8) + 16 (q1 + 8)
        }
        words[wq] = pack_int4_pairs(pairs);
    }
    if (out_ok) store_words<E / 8>(out_codes + o / 2, words);
    if (out_ok && lane == 0) __stcs(out_scales + o / B, bs.scale);
}

// Sources of the fixed kernel that read their products from a table (the
// lookups run on the load/store pipe; the last source takes the packed
// byte-permute path on the ALU and FMA pipes instead).
__host__ __device__ constexpr int hop1_table_sources(int L) { return L - (L + 7) / 8; }

// Launch bounds: a budget for 1280 threads per SM (at most 51 registers) at B <= 512
// measured faster than the compiler's unbounded choice -- at B = 512, L = 8,
// 0.594 -> 0.574 ms without error feedback (48 registers instead of 40) and
// 0.815 -> 0.773 ms with it (48 with 4 bytes of spills, instead of 55 and 4
// CTAs of 256 threads).  A budget for 6 such CTAs was slower with error
// feedback.  B = 1024 needs about 110 registers and takes no budget.
// CTAs of 128 threads: with the same register budget (10 CTAs of 128
// threads per SM) they measured 0.447 -> 0.441 ms against 256-thread CTAs,
// bit-identical (more CTAs per SM start and stall at different times).
constexpr int kHop1Threads = 128;

template <int B, int L, bool HAS_EF>
__global__ void __launch_bounds__(kHop1Threads, B <= 512 ? 10 : 1)
hop1_fixed_kernel(const uint8_t *__restrict__ codes, const float *__restrict__ scales,
                  uint8_t *__restrict__ out_codes, float *__restrict__ out_scales,
                  QgzGeometry geo, float *__restrict__ ef1, float s, float beta,
                  float one_minus_beta, Exact2 kc) {
    constexpr int E = B / kWarp;  // outputs per lane
    constexpr int W = E / 8;      // code words per lane and source
    const int lane = threadIdx.x & (kWarp - 1);
    // Grid x: blocks of one sub-slice (a warp each), y: sub-slice g', z: unit
    // u = g*L + l -- the positions need no division (L is a power of two).
    const uint32_t off = (blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp) * B;
    if (off >= geo.S) return;  // whole warp: the grid's x is rounded up
    const uint32_t gq = blockIdx.y, u = blockIdx.z;
    const uint32_t grp = u / L, l = u - grp * L;
    const uint32_t i = off + uint32_t(E) * lane;
    const uint32_t o = (u * geo.G + gq) * geo.S + i;  // output element
    const uint32_t pos0 = grp * L * geo.N + (l * geo.G + gq) * geo.S + i;
    const uint8_t *cp = codes + pos0 / 2;
    const float *sp = scales + pos0 / B;
    const uint32_t cstride = geo.N / 2;
    const uint32_t sstride = geo.N / B;

    uint32_t w[L][W];
    float sc[L];
#pragma unroll
    for (int t = 0; t < L; ++t) {
#pragma unroll
        for (int q = 0; q < W; ++q) w[t][q] = 0u;
        sc[t] = 0.0f;
        // source t's E codes lie inside the R ranks' N codes each
        if (WC_IN_BOUNDS(uint64_t(pos0) + uint64_t(t) * geo.N + E <= geo.total)) {
            load_words<W>(cp + size_t(t) * cstride, w[t]);
            sc[t] = __ldg(sp + size_t(t) * sstride);
        }
    }
    const bool out_ok = WC_IN_BOUNDS(uint64_t(o) + E <= uint64_t(geo.G) * geo.N);
    if (HAS_EF) {
        // With its error buffer the hop moves 8 more bytes per output and is
        // bound by HBM; shuffles there compete with the error loads and
        // stores for the load/store pipe and measured slower (0.77 -> 0.82 ms
        // at B = 512, L = 8), so this form keeps the scalar byte-permute path.
        float p[E];
#pragma unroll
        for (int t = 0; t < L; ++t) {
#pragma unroll
            for (int wq = 0; wq < W; ++wq) {
                float f[8];
                unpack_int4x8(w[t][wq], f);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    p[8 * wq + j] = t == 0 ? dequant_first(f[j], sc[t])
                                           : __fadd_rn(p[8 * wq + j], dequant(f[j], sc[t]));
            }
        }
        requantize_lane<E, kWarp, HAS_EF, B>(p, o, out_ok, lane, out_codes, out_scales, ef1, s,
                                             beta, one_minus_beta);
        return;
    }
    // The warp's E * 32 outputs are one block of every source, so each
    // source's products come from one warp-wide table.
    constexpr int NT = hop1_table_sources(L);
    const Ops2 ops(kc);
    f32x2 p[E / 2];
#pragma unroll
    for (int t = 0; t < L; ++t) {
        const f32x2 s2 = pack2(sc[t], sc[t]);
        const float table = t >= NT ? 0.0f
                            : t == 0 ? product_table<true>(sc[t], lane)
                                     : product_table<false>(sc[t], lane);
#pragma unroll
        for (int wq = 0; wq < W; ++wq) {
            f32x2 *pw = p + 4 * wq;
            if (t == 0 && t < NT) accumulate_word<true, true, kWarp>(w[t][wq], table, s2, pw, kFull, ops);
            else if (t == 0) accumulate_word<true, false, kWarp>(w[t][wq], table, s2, pw, kFull, ops);
            else if (t < NT) accumulate_word<false, true, kWarp>(w[t][wq], table, s2, pw, kFull, ops);
            else accumulate_word<false, false, kWarp>(w[t][wq], table, s2, pw, kFull, ops);
        }
    }
    requantize_pairs<E, B>(p, o, out_ok, lane, out_codes, out_scales, ops);
}

// General shapes: warp tile T = max(B, 256) outputs, lane t holds outputs
// 256*k + 8*t + j (one code word per source and k); blocks shorter than 256
// belong to aligned groups of B/8 lanes.
template <int B, bool HAS_EF>
__global__ void __launch_bounds__(256)
hop1_general_kernel(const uint8_t *__restrict__ codes, const float *__restrict__ scales,
                    uint8_t *__restrict__ out_codes, float *__restrict__ out_scales,
                    QgzGeometry geo, float *__restrict__ ef1, float s, float beta,
                    float one_minus_beta) {
    constexpr int T = B >= 256 ? B : 256;
    constexpr int K = T / 256;
    constexpr int LPB = B >= 256 ? 32 : B / 8;
    const int lane = threadIdx.x & (kWarp - 1);
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) / kWarp;
    const uint32_t total_out = geo.G * geo.N;
    if (uint64_t(warp) * T >= total_out) return;
    const uint32_t tile0 = warp * uint32_t(T);
    const uint32_t cstride = geo.N / 2;
    const uint32_t sstride = geo.N / B;

    float p[K][8];
    float e[K][8];
    bool active[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const uint32_t o = tile0 + 256u * k + 8u * lane;
        active[k] = o < total_out;  // only blocks shorter than 256 leave lanes idle
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            p[k][j] = 0.0f;
            e[k][j] = 0.0f;
        }
        if (!active[k]) continue;
        if (!WC_IN_BOUNDS(uint64_t(o) + 8 <= total_out)) {
            active[k] = false;  // checked builds: the lane's outputs are not all there
            continue;
        }
        const uint32_t pos0 = hop1_source(geo, o);
        const uint8_t *cp = codes + pos0 / 2;
        const float *sp = scales + pos0 / B;
        for (uint32_t l0 = 0; l0 < geo.L; l0 += 8) {
            uint32_t w[8];
            float sc[8];
            const uint32_t nb = min(8u, geo.L - l0);
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                w[t] = 0u;
                sc[t] = 0.0f;
                if (t < nb &&
                    WC_IN_BOUNDS(uint64_t(pos0) + uint64_t(l0 + t) * geo.N + 8 <= geo.total)) {
                    w[t] = __ldcs(reinterpret_cast<const unsigned int *>(cp + size_t(l0 + t) * cstride));
                    sc[t] = __ldg(sp + size_t(l0 + t) * sstride);
                }
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                if (t < nb) {
                    float f[8];
                    unpack_int4x8(w[t], f);
#pragma unroll
                    for (int j = 0; j < 8; ++j) p[k][j] = __fadd_rn(p[k][j], dequant(f[j], sc[t]));
                }
            }
        }
        if (HAS_EF) {
            const float4 a = ld_stream_f4(ef1 + o);
            const float4 b = ld_stream_f4(ef1 + o + 4);
            e[k][0] = a.x; e[k][1] = a.y; e[k][2] = a.z; e[k][3] = a.w;
            e[k][4] = b.x; e[k][5] = b.y; e[k][6] = b.z; e[k][7] = b.w;
#pragma unroll
            for (int j = 0; j < 8; ++j) p[k][j] = __fadd_rn(p[k][j], __fmul_rn(s, e[k][j]));
        }
    }

    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
        for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(p[k][j]));
    m = group_max<LPB>(m);
    const BlockScale bs = block_scale<7>(m);

#pragma unroll
    for (int k = 0; k < K; ++k) {
        if (!active[k]) continue;
        const uint32_t o = tile0 + 256u * k + 8u * lane;
        uint32_t packed = 0;
        float q[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const QCode qc = quant_code<7>(p[k][j], bs);
            q[j] = qc.q;
            packed |= (qc.bits & 15u) << (4 * j);
        }
        __stcs(reinterpret_cast<unsigned int *>(out_codes + o / 2), packed);
        if (HAS_EF) {
            float v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = __fadd_rn(__fmul_rn(beta, e[k][j]),
                                 __fmul_rn(one_minus_beta, __fsub_rn(p[k][j], dequant(q[j], bs.scale))));
            __stcs(reinterpret_cast<float4 *>(ef1 + o), make_float4(v[0], v[1], v[2], v[3]));
            __stcs(reinterpret_cast<float4 *>(ef1 + o + 4), make_float4(v[4], v[5], v[6], v[7]));
        }
        if (k == 0 && (lane & (LPB - 1)) == 0) __stcs(out_scales + o / B, bs.scale);
    }
}

template <int B, bool HAS_EF>
static bool launch_fixed_b(const uint8_t *codes, const float *scales, uint8_t *out_codes,
                           float *out_scales, const QgzGeometry &geo, float *ef1, float s,
                           float beta, cudaStream_t stream) {
    const uint32_t warps = geo.S / B;  // per sub-slice
    constexpr uint32_t kWarpsPerCta = kHop1Threads / kWarp;
    const dim3 grid((warps + kWarpsPerCta - 1) / kWarpsPerCta, geo.G, geo.R);
    const float omb = 1.0f - beta;
    const Exact2 kc = exact2_constants();
#define WC_HOP1(LL)                                                                           \
    case LL:                                                                                  \
        hop1_fixed_kernel<B, LL, HAS_EF><<<grid, kHop1Threads, 0, stream>>>(codes, scales, out_codes,  \
                                                                   out_scales, geo, ef1, s,   \
                                                                   beta, omb, kc);            \
        return true;
    switch (geo.L) {
        WC_HOP1(1) WC_HOP1(2) WC_HOP1(4) WC_HOP1(8)
        case 16:
            if (B > 512) return false;  // 16 sources x 4 words would not fit in registers
            hop1_fixed_kernel<B, (B > 512 ? 8 : 16), HAS_EF><<<grid, kHop1Threads, 0, stream>>>(
                codes, scales, out_codes, out_scales, geo, ef1, s, beta, omb, kc);
            return true;
        default:
            return false;
    }
#undef WC_HOP1
}

template <int B, bool HAS_EF>
static void launch_general_b(const uint8_t *codes, const float *scales, uint8_t *out_codes,
                             float *out_scales, const QgzGeometry &geo, float *ef1, float s,
                             float beta, cudaStream_t stream) {
    constexpr int T = B >= 256 ? B : 256;
    const uint32_t total_out = geo.G * geo.N;
    const uint32_t tiles = uint32_t((uint64_t(total_out) + T - 1) / T);  // no wrap near 2^32
    const uint32_t grid = (tiles + 7) / 8;
    hop1_general_kernel<B, HAS_EF><<<grid, 256, 0, stream>>>(codes, scales, out_codes, out_scales,
                                                             geo, ef1, s, beta, 1.0f - beta);
}

template <int B, bool HAS_EF>
static void launch_b(const uint8_t *codes, const float *scales, uint8_t *out_codes,
                     float *out_scales, const QgzGeometry &geo, float *ef1, float s, float beta,
                     cudaStream_t stream) {
    if (B >= 256 && launch_fixed_b<(B >= 256 ? B : 256), HAS_EF>(codes, scales, out_codes,
                                                                   out_scales, geo, ef1, s,
                                                                   beta, stream))
        return;
    launch_general_b<B, HAS_EF>(codes, scales, out_codes, out_scales, geo, ef1, s, beta, stream);
}

template <bool HAS_EF>
static cudaError_t launch_ef(const uint8_t *codes, const float *scales, uint8_t *out_codes,
                             float *out_scales, const QgzGeometry &geo, int B, float *ef1,
                             float s, float beta, cudaStream_t stream) {
    switch (B) {
        case 32: launch_b<32, HAS_EF>(codes, scales, out_codes, out_scales, geo, ef1, s, beta, stream); break;
        case 64: launch_b<64, HAS_EF>(codes, scales, out_codes, out_scales, geo, ef1, s, beta, stream); break;
        case 128: launch_b<128, HAS_EF>(codes, scales, out_codes, out_scales, geo, ef1, s, beta, stream); break;
        case 256: launch_b<256, HAS_EF>(codes, scales, out_codes, out_scales, geo, ef1, s, beta, stream); break;
        case 512: launch_b<512, HAS_EF>(codes, scales, out_codes, out_scales, geo, ef1, s, beta, stream); break;
        case 1024: launch_b<1024, HAS_EF>(codes, scales, out_codes, out_scales, geo, ef1, s, beta, stream); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaPeekAtLastError();
}

WC_CHECK_RECORD_READER(check_record_qgz_hop1)

cudaError_t launch_dequant_reduce_requant(const uint8_t *codes, const float *scales,
                                          uint8_t *out_codes, float *out_scales,
                                          const QgzGeometry &geo, int B, float *ef1, float s,
                                          float beta, cudaStream_t stream) {
    if (ef1 != nullptr)
        return launch_ef<true>(codes, scales, out_codes, out_scales, geo, B, ef1, s, beta, stream);
    return launch_ef<false>(codes, scales, out_codes, out_scales, geo, B, ef1, s, beta, stream);
}

}  // namespace wc
