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
// The per-code work -- unpack, multiply by the scale, add in source order --
// is all the kernel does besides moving bytes, so it runs issue-bound unless
// the instructions per code stay few.  Hence: the source count is a template
// parameter (no loop bounds, no guards, every load hoisted ahead of the
// adds), each thread makes 16 consecutive outputs from one 8-byte code word
// per source (so the per-source address and scale work is amortized over 16
// codes), the destination comes from the grid's y index (no division), and
// codes are unpacked with byte permutes and exact subtractions
// (wc_device.cuh), never on the conversion pipe.  For 3 to 8 sources and
// blocks of 256 or more the sums run two outputs per packed instruction
// (byte permute, then an exact packed unbias, multiply and add per pair of
// codes), and the first source's products come from a half-warp product
// table instead (each half-warp's 256 outputs lie in one block of every
// source); that kernel takes CTAs of 128 threads and a register budget for
// 10 of them per SM.  Source
// counts above kMaxFixedSources take a loop over batches of eight.
#include "wc_device.cuh"
#include "wc_internal.h"

namespace wc {

constexpr int kMaxFixedSources = 16;
constexpr uint32_t kOutPerThread = 16;

// The 16 sums times out_scale, to fp32 or (rounded to nearest even) bf16.
// SCALED = false (out_scale == 1) skips the multiplies: x * 1 is exactly x
// for every float.
template <bool OUT_BF16, bool SCALED>
__device__ __forceinline__ void store16(void *out, uint32_t o, const float acc[16],
                                           float out_scale) {
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = SCALED ? __fmul_rn(acc[j], out_scale) : acc[j];
    if (OUT_BF16) {
        uint32_t h[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) h[j] = f32x2_to_bf16x2_bits(v[2 * j], v[2 * j + 1]);
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + o);
        __stcs(dst, make_uint4(h[0], h[1], h[2], h[3]));
        __stcs(dst + 1, make_uint4(h[4], h[5], h[6], h[7]));
    } else {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(out) + o);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            __stcs(dst + q, make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
    }
}

// acc[0..16) += the 16 codes of w (element 2k in the low nibble of byte k) * sc;
// FIRST: acc is +0 (the sums' start), so the add folds into one fma.
template <bool FIRST = false>
__device__ __forceinline__ void accumulate16(uint2 w, float sc, float acc[16]) {
    float f[8];
    unpack_int4x8(w.x, f);
#pragma unroll
    for (int j = 0; j < 8; ++j)
        acc[j] = FIRST ? dequant_first(f[j], sc) : __fadd_rn(acc[j], dequant(f[j], sc));
    unpack_int4x8(w.y, f);
#pragma unroll
    for (int j = 0; j < 8; ++j)
        acc[8 + j] = FIRST ? dequant_first(f[j], sc) : __fadd_rn(acc[8 + j], dequant(f[j], sc));
}

// First code position and scale index of destination k's 16 outputs at i.
__device__ __forceinline__ uint32_t source_base(const QgzGeometry &geo, uint32_t k, uint32_t i) {
    uint32_t chunk = k;
    if (geo.G > 1) {
        const uint32_t grp = k / geo.L;
        chunk = (k - grp * geo.L) * geo.G + grp;
    }
    return chunk * geo.S + i;
}

// Checked builds: source t's 16 codes (and so its scale) lie inside the
// source buffers, R of N codes each for the flat reduce, G for the second hop.
__device__ __forceinline__ bool source_in_bounds(const QgzGeometry &geo, uint32_t base,
                                                 uint32_t t) {
    const uint64_t ncodes = uint64_t(geo.G > 1 ? geo.G : geo.R) * geo.N;
    return uint64_t(base) + uint64_t(t) * geo.N + kOutPerThread <= ncodes;
}

__device__ __forceinline__ bool output_in_bounds(const QgzGeometry &geo, uint32_t k, uint32_t i) {
    return uint64_t(k) * geo.S + i + kOutPerThread <= geo.N;
}

// The same sums two outputs at a time (acc[j]: outputs 2j, 2j+1), for 3..8
// sources and B >= 256.  S is then a multiple of 256, so every half-warp is
// wholly inside the shard or wholly past it, and the 256 outputs of a
// half-warp lie in one block of every source: the first source's products
// come from the half-warp's product table (one 16-wide shuffle per code),
// the others from the packed byte-permute path (accumulate_word).  Measured
// at 8 sources and B = 256: 0.0758 -> 0.0695 ms.  The register budget (1280
// threads per SM) matters: unbounded, the compiler's allocation took it to
// 0.164 ms.  CTAs of 128 threads (10 per SM) in place of 256 (5 per SM):
// 0.0689 -> 0.0670 ms, bit-identical.
constexpr uint32_t kPairsThreads = 128;

template <int NSRC, bool OUT_BF16, bool SCALED>
__global__ void __launch_bounds__(kPairsThreads, 10)
dequant_reduce_pairs_kernel(const uint8_t *__restrict__ codes, const float *__restrict__ scales,
                            QgzGeometry geo, uint32_t log2_b, float out_scale,
                            void *__restrict__ out, Exact2 kc) {
    const uint32_t k = blockIdx.y;  // destination
    const uint32_t v = blockIdx.x * blockDim.x + threadIdx.x;
    if (uint64_t(v) * kOutPerThread >= geo.S) return;  // whole half-warps
    const uint32_t i = v * kOutPerThread;
    const uint32_t base = source_base(geo, k, i);
    const uint8_t *cp = codes + base / 2;
    const float *sp = scales + (base >> log2_b);
    const uint32_t cstride = geo.N / 2;
    const uint32_t sstride = geo.N >> log2_b;
    uint2 w[NSRC];
    float sc[NSRC];
#pragma unroll
    for (int t = 0; t < NSRC; ++t) {
        w[t] = make_uint2(0u, 0u);
        sc[t] = 0.0f;
        if (WC_IN_BOUNDS(source_in_bounds(geo, base, t))) {
            w[t] = __ldcs(reinterpret_cast<const uint2 *>(cp + size_t(t) * cstride));
            sc[t] = __ldg(sp + size_t(t) * sstride);
        }
    }
    const Ops2 ops(kc);
    const int lane = threadIdx.x & (kWarp - 1);
    const unsigned hmask = 0xFFFFu << (lane & 16);
    f32x2 a2[8];
    {
        const float table = product_table<true>(sc[0], lane);
        accumulate_word<true, true, 16>(w[0].x, table, pack2(0.0f, 0.0f), a2, hmask, ops);
        accumulate_word<true, true, 16>(w[0].y, table, pack2(0.0f, 0.0f), a2 + 4, hmask, ops);
    }
#pragma unroll
    for (int t = 1; t < NSRC; ++t) {
        const f32x2 s2 = pack2(sc[t], sc[t]);
        accumulate_word<false, false, 16>(w[t].x, 0.0f, s2, a2, hmask, ops);
        accumulate_word<false, false, 16>(w[t].y, 0.0f, s2, a2 + 4, hmask, ops);
    }
    float acc[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) unpack2(a2[j], acc[2 * j], acc[2 * j + 1]);
    if (WC_IN_BOUNDS(output_in_bounds(geo, k, i)))
        store16<OUT_BF16, SCALED>(out, k * geo.S + i, acc, out_scale);
}

template <int NSRC, bool OUT_BF16, bool SCALED>
__global__ void __launch_bounds__(256)
dequant_reduce_fixed_kernel(const uint8_t *__restrict__ codes, const float *__restrict__ scales,
                            QgzGeometry geo, uint32_t log2_b, float out_scale,
                            void *__restrict__ out) {
    const uint32_t k = blockIdx.y;  // destination
    const uint32_t v = blockIdx.x * blockDim.x + threadIdx.x;
    if (uint64_t(v) * kOutPerThread >= geo.S) return;
    const uint32_t i = v * kOutPerThread;  // offset in the shard
    const uint32_t base = source_base(geo, k, i);
    const uint8_t *cp = codes + base / 2;
    const float *sp = scales + (base >> log2_b);
    const uint32_t cstride = geo.N / 2;        // bytes between sources
    const uint32_t sstride = geo.N >> log2_b;  // scales between sources

    uint2 w[NSRC];
    float sc[NSRC];
#pragma unroll
    for (int t = 0; t < NSRC; ++t) {
        w[t] = make_uint2(0u, 0u);
        sc[t] = 0.0f;
        if (WC_IN_BOUNDS(source_in_bounds(geo, base, t))) {
            w[t] = __ldcs(reinterpret_cast<const uint2 *>(cp + size_t(t) * cstride));
            sc[t] = __ldg(sp + size_t(t) * sstride);
        }
    }
    float acc[16];
    accumulate16<true>(w[0], sc[0], acc);
#pragma unroll
    for (int t = 1; t < NSRC; ++t) accumulate16(w[t], sc[t], acc);
    if (WC_IN_BOUNDS(output_in_bounds(geo, k, i)))
        store16<OUT_BF16, SCALED>(out, k * geo.S + i, acc, out_scale);
}

template <bool OUT_BF16, bool SCALED>
__global__ void __launch_bounds__(256)
dequant_reduce_loop_kernel(const uint8_t *__restrict__ codes, const float *__restrict__ scales,
                           QgzGeometry geo, uint32_t nsrc, uint32_t log2_b, float out_scale,
                           void *__restrict__ out) {
    const uint32_t k = blockIdx.y;
    const uint32_t v = blockIdx.x * blockDim.x + threadIdx.x;
    if (uint64_t(v) * kOutPerThread >= geo.S) return;
    const uint32_t i = v * kOutPerThread;
    const uint32_t base = source_base(geo, k, i);
    const uint8_t *cp = codes + base / 2;
    const float *sp = scales + (base >> log2_b);
    const uint32_t cstride = geo.N / 2;
    const uint32_t sstride = geo.N >> log2_b;

    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
    uint32_t t = 0;
    for (; t + 8 <= nsrc; t += 8) {
        uint2 w[8];
        float sc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            w[u] = make_uint2(0u, 0u);
            sc[u] = 0.0f;
            if (WC_IN_BOUNDS(source_in_bounds(geo, base, t + u))) {
                w[u] = __ldcs(reinterpret_cast<const uint2 *>(cp + size_t(t + u) * cstride));
                sc[u] = __ldg(sp + size_t(t + u) * sstride);
            }
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) accumulate16(w[u], sc[u], acc);
    }
    for (; t < nsrc; ++t)
        if (WC_IN_BOUNDS(source_in_bounds(geo, base, t)))
            accumulate16(__ldcs(reinterpret_cast<const uint2 *>(cp + size_t(t) * cstride)),
                         __ldg(sp + size_t(t) * sstride), acc);
    if (WC_IN_BOUNDS(output_in_bounds(geo, k, i)))
        store16<OUT_BF16, SCALED>(out, k * geo.S + i, acc, out_scale);
}

template <int NSRC, bool OUT_BF16, bool SCALED>
static void launch_fixed(const uint8_t *codes, const float *scales, const QgzGeometry &geo,
                         uint32_t log2_b, float out_scale, void *out, dim3 grid,
                         cudaStream_t stream) {
    if (NSRC >= 3 && NSRC <= 8 && log2_b >= 8) {  // B >= 256
        const dim3 pgrid((geo.S / kOutPerThread + kPairsThreads - 1) / kPairsThreads, grid.y);
        dequant_reduce_pairs_kernel<(NSRC >= 3 && NSRC <= 8 ? NSRC : 3), OUT_BF16, SCALED>
            <<<pgrid, kPairsThreads, 0, stream>>>(codes, scales, geo, log2_b, out_scale, out,
                                                  exact2_constants());
    } else {
        dequant_reduce_fixed_kernel<NSRC, OUT_BF16, SCALED><<<grid, 256, 0, stream>>>(
            codes, scales, geo, log2_b, out_scale, out);
    }
}

template <bool OUT_BF16, bool SCALED>
static void launch_any(const uint8_t *codes, const float *scales, const QgzGeometry &geo,
                       uint32_t nsrc, uint32_t log2_b, float out_scale, void *out, dim3 grid,
                       cudaStream_t stream) {
#define WC_FIXED(n)                                                                        \
    case n:                                                                                \
        launch_fixed<n, OUT_BF16, SCALED>(codes, scales, geo, log2_b, out_scale, out, grid, \
                                          stream);                                         \
        return;
    switch (nsrc) {
        WC_FIXED(1) WC_FIXED(2) WC_FIXED(3) WC_FIXED(4) WC_FIXED(5) WC_FIXED(6) WC_FIXED(7)
        WC_FIXED(8) WC_FIXED(9) WC_FIXED(10) WC_FIXED(11) WC_FIXED(12) WC_FIXED(13)
        WC_FIXED(14) WC_FIXED(15) WC_FIXED(16)
        default:
            dequant_reduce_loop_kernel<OUT_BF16, SCALED><<<grid, 256, 0, stream>>>(
                codes, scales, geo, nsrc, log2_b, out_scale, out);
    }
#undef WC_FIXED
}

WC_CHECK_RECORD_READER(check_record_qgz_reduce)

cudaError_t launch_dequant_reduce(const uint8_t *codes, const float *scales,
                                  const QgzGeometry &geo, int B, float out_scale, void *out,
                                  bool out_bf16, cudaStream_t stream) {
    static_assert(kMaxFixedSources == 16, "dispatch table covers 1..16");
    uint32_t log2_b = 0;
    while ((1u << log2_b) < uint32_t(B)) ++log2_b;
    const uint32_t nsrc = geo.G > 1 ? geo.G : geo.R;
    const uint32_t threads = 256;
    // S is a multiple of B >= 32, hence of the 16 outputs a thread makes
    const dim3 grid((geo.S / kOutPerThread + threads - 1) / threads, geo.R);
    // out_scale == 1 takes the kernels without the final multiplies
    const bool scaled = out_scale != 1.0f;
    if (out_bf16 && scaled)
        launch_any<true, true>(codes, scales, geo, nsrc, log2_b, out_scale, out, grid, stream);
    else if (out_bf16)
        launch_any<true, false>(codes, scales, geo, nsrc, log2_b, out_scale, out, grid, stream);
    else if (scaled)
        launch_any<false, true>(codes, scales, geo, nsrc, log2_b, out_scale, out, grid, stream);
    else
        launch_any<false, false>(codes, scales, geo, nsrc, log2_b, out_scale, out, grid, stream);
    return cudaPeekAtLastError();
}

}  // namespace wc
