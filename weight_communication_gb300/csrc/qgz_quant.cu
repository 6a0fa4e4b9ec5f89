// qgz_quant.cu -- the kernel that produces the int4 send buffers:
//   * error-feedback compensation + int4 block quantization of every rank's
//     gradient, written in all-to-all send order (LoCo on qgZ);
//   (the first hop of the hierarchical reduce, which requantizes, is in
//   qgz_hop1.cu).
//
// "Merge LoCo with Zero++" (DeepSpeed PR #6730), Overview: the 4-bit
// gradients are compensated with an error-feedback buffer before they are
// communicated.  "ZeROPlusPlus.md", §1.2 ZeRO++ (quantized gradient
// communication): block-based int4 quantization, all-to-all in place of the
// reduce-scatter, reduction in full precision, intra-node before inter-node,
// with kernel fusion.
//
// One warp owns one quantization block (or, for blocks shorter than the warp
// tile, each aligned group of lanes owns one block), so the absmax is a warp
// reduction and codes, scales and the error update are produced
// in the same pass that loads the block -- no second read, no shared memory,
// no block barrier.  Codes are rounded and unpacked with exact fp32
// arithmetic (wc_device.cuh), never on the conversion pipe.
#include "wc_device.cuh"
#include "wc_internal.h"
#include "int8_error_block.cuh"

namespace wc {

// ---------------------------------------------------------------------------
// EF compensation + int4 quantization (HBM-bound: 10.5 bytes per element)
// ---------------------------------------------------------------------------
//
// Lane layout: a warp tile is T = max(B, 128) consecutive gradient elements;
// lane t holds elements 128*k + 4*t + j (k < T/128, j < 4).  Every access is
// then fully coalesced: 8-byte bf16 loads (256 B per warp instruction),
// 16-byte fp32 error loads and stores (512 B), 2-byte code stores (64 B).
//
// EF selects the error buffer: none, fp32 (4 bytes per element each way),
// bf16 (2 bytes; the new error is rounded to the nearest bf16 when stored) or
// int8 (1 byte, plus one fp32 scale per block: the new error of a block is
// quantized by the int8 absmax rule once the whole block is known, so it is
// kept in registers until a second warp reduction has found its maximum).
enum EfMode { kEfNone = 0, kEfF32 = 1, kEfBf16 = 2, kEfInt8 = 3 };

// int8 error buffer, B >= 128: each warp takes NB consecutive blocks of a
// slice and issues the loads of all of them before it computes the first.
// A warp reads only 12 bytes per lane and block here, so with one block per
// warp too few bytes are in flight to cover DRAM latency.  At B = 256, timed
// back to back: one block per warp under a budget of 8 CTAs per SM 0.388 ms,
// two blocks with 4 CTAs 0.367-0.380 ms, three blocks with 3 CTAs 0.353 ms,
// four blocks with 2 or 3 CTAs 0.365 ms.
template <int B, int NB, int MINB, bool S1>
__global__ void __launch_bounds__(256, MINB)
ef_quant_int8ef_kernel(const uint16_t *__restrict__ g, int8_t *__restrict__ ef8,
                       float *__restrict__ ef_scales, uint8_t *__restrict__ codes,
                       float *__restrict__ scales, QgzGeometry geo, float s, float beta,
                       float one_minus_beta, Exact2 kc) {
    static_assert(B >= 128 && B % 128 == 0, "one warp per block");
    constexpr int K = B / 128;
    const int lane = threadIdx.x & (kWarp - 1);
    const uint32_t off0 = (blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp) * (B * NB);
    if (off0 >= geo.S) return;  // whole warp
    const uint32_t slice = blockIdx.y, r = blockIdx.z;
    uint32_t p = slice;
    if (geo.G > 1) {
        const uint32_t gq = slice / geo.L;
        p = (slice - gq * geo.L) * geo.G + gq;
    }
    const Ops2 ops(kc);
    uint2 gv[NB][K];
    uint32_t e8w[NB][K];
    float es[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const uint32_t tile0 = r * geo.N + slice * geo.S + off0 + b * B;
        es[b] = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            gv[b][k] = make_uint2(0u, 0u);
            e8w[b][k] = 0u;
        }
        if (off0 + b * B >= geo.S) continue;  // past the slice's last block (whole warp)
        if (WC_IN_BOUNDS(tile0 / B < geo.total / B)) es[b] = __ldg(ef_scales + tile0 / B);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const uint32_t x = tile0 + 128u * k + 4u * lane;
            if (WC_IN_BOUNDS(uint64_t(x) + 4 <= geo.total)) {
                gv[b][k] = ld_stream_u2(g + x);
                e8w[b][k] = __ldcs(reinterpret_cast<const unsigned int *>(ef8 + x));
            }
        }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        if (off0 + b * B >= geo.S) break;
        const uint32_t tile0 = r * geo.N + slice * geo.S + off0 + b * B;
        const uint32_t out0 = r * geo.N + p * geo.S + off0 + b * B;
        int8ef_block<B, S1, true, false>(gv[b], e8w[b], es[b], ef8, ef_scales, codes, scales,
                                         geo.total, tile0, out0, lane, s, beta, one_minus_beta,
                                         ops, nullptr);
    }
}

template <int B, int EF, bool S1 = false>
__device__ __forceinline__ void ef_quant_int4_warp(const uint16_t *__restrict__ g,
                                                   void *__restrict__ ef_v,
                                                   float *__restrict__ ef_scales,
                                                   uint8_t *__restrict__ codes,
                                                   float *__restrict__ scales, QgzGeometry geo,
                                                   float s, float beta, float one_minus_beta) {
    constexpr bool HAS_EF = EF != kEfNone;
    float *__restrict__ ef = static_cast<float *>(ef_v);
    uint16_t *__restrict__ ef16 = static_cast<uint16_t *>(ef_v);
    int8_t *__restrict__ ef8 = static_cast<int8_t *>(ef_v);
    constexpr int T = B >= 128 ? B : 128;
    constexpr int K = T / 128;
    constexpr int LPB = B >= 128 ? 32 : B / 4;  // lanes per block
    const int lane = threadIdx.x & (kWarp - 1);
    uint32_t tile0;  // first gradient element of the warp's tile
    uint32_t out0;   // code position of the first element of the lane's block
    uint32_t eblk;   // the lane's block in gradient order (int8 error scales)
    bool active;
    if (B >= 128) {
        // Grid x: blocks of one slice (a warp each), y: slice, z: rank -- the
        // send position needs no division except slice -> (group, local rank).
        const uint32_t off = (blockIdx.x * (blockDim.x / kWarp) + threadIdx.x / kWarp) * B;
        if (off >= geo.S) return;  // whole warp: the grid's x is rounded up
        const uint32_t slice = blockIdx.y, r = blockIdx.z;
        uint32_t p = slice;
        if (geo.G > 1) {
            const uint32_t gq = slice / geo.L;
            p = (slice - gq * geo.L) * geo.G + gq;
        }
        tile0 = r * geo.N + slice * geo.S + off;
        out0 = r * geo.N + p * geo.S + off;
        eblk = tile0 / B;
        active = true;
    } else {
        // 1-D grid of 128-element tiles holding 128/B blocks each.
        const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) / kWarp;
        // Warps past the end leave at once; the comparison is 64-bit so a tile
        // start cannot wrap around 2^32.
        if (uint64_t(warp) * T >= geo.total) return;
        tile0 = warp * uint32_t(T);
        const uint32_t first = tile0 + 4u * lane;
        active = first < geo.total;
        const uint32_t blk = first / B;
        eblk = blk;
        const uint32_t r = blk / geo.blocks_per_rank;
        const uint32_t x0 = (blk - r * geo.blocks_per_rank) * B;  // element in rank
        const uint32_t slice = x0 / geo.S;
        const uint32_t off = x0 - slice * geo.S;
        const uint32_t gq = slice / geo.L;
        const uint32_t l = slice - gq * geo.L;
        out0 = r * geo.N + (l * geo.G + gq) * geo.S + off;
    }

    float c[K][4];
    float e[K][4];
    float es = 0.0f;  // int8 error: the block's stored scale
    if (EF == kEfInt8 && active && WC_IN_BOUNDS(eblk < geo.total / B)) es = __ldg(ef_scales + eblk);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const uint32_t x = tile0 + 128u * k + 4u * lane;
        uint2 gv = make_uint2(0u, 0u);
        float4 ev = make_float4(0.f, 0.f, 0.f, 0.f);
        if (active && WC_IN_BOUNDS(uint64_t(x) + 4 <= geo.total)) {
            gv = ld_stream_u2(g + x);
            if (EF == kEfF32) ev = ld_stream_f4(ef + x);
            if (EF == kEfBf16) {
                const uint2 eh = ld_stream_u2(ef16 + x);
                ev = make_float4(bf16_bits_to_f32(eh.x & 0xFFFFu), bf16_bits_to_f32(eh.x >> 16),
                                 bf16_bits_to_f32(eh.y & 0xFFFFu), bf16_bits_to_f32(eh.y >> 16));
            }
            if (EF == kEfInt8) {
                float f[4];
                unpack_int8x4(__ldcs(reinterpret_cast<const unsigned int *>(ef8 + x)), f);
                ev = make_float4(dequant(f[0], es), dequant(f[1], es), dequant(f[2], es),
                                 dequant(f[3], es));
            }
        }
        const float gf[4] = {bf16_bits_to_f32(gv.x & 0xFFFFu), bf16_bits_to_f32(gv.x >> 16),
                             bf16_bits_to_f32(gv.y & 0xFFFFu), bf16_bits_to_f32(gv.y >> 16)};
        e[k][0] = ev.x; e[k][1] = ev.y; e[k][2] = ev.z; e[k][3] = ev.w;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            // S1: s = 1, and s*e is e itself (exact for every finite e)
            c[k][j] = HAS_EF ? __fadd_rn(gf[j], S1 ? e[k][j] : __fmul_rn(s, e[k][j])) : gf[j];
    }

    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
        for (int j = 0; j < 4; ++j) m = fmaxf(m, fabsf(c[k][j]));
    m = group_max<LPB>(m);
    const BlockScale bs = block_scale<7>(m);
    // int8 error: every lane takes part in the second reduction below
    if (EF != kEfInt8 && !active) return;
    float en[EF == kEfInt8 ? K : 1][4];  // int8 error: the new error, until stored

#pragma unroll
    for (int k = 0; k < K; ++k) {
        float q[4];
        uint32_t packed = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const QCode qc = quant_code<7>(c[k][j], bs);
            q[j] = qc.q;
            packed |= (qc.bits & 15u) << (4 * j);
        }
        const uint32_t in_blk = B >= 128 ? 128u * k + 4u * lane : (4u * lane) % B;
        const uint32_t pos = out0 + in_blk;
        if (active && WC_IN_BOUNDS(uint64_t(pos) + 4 <= geo.total))
            __stcs(reinterpret_cast<unsigned short *>(codes + pos / 2), (unsigned short)packed);
        if (HAS_EF) {
            float4 ev;
            float *o = &ev.x;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float d = dequant(q[j], bs.scale);
                o[j] = __fadd_rn(__fmul_rn(beta, e[k][j]),
                                 __fmul_rn(one_minus_beta, __fsub_rn(c[k][j], d)));
            }
            if (EF == kEfInt8) {
#pragma unroll
                for (int j = 0; j < 4; ++j) en[EF == kEfInt8 ? k : 0][j] = o[j];
                continue;
            }
            const uint32_t x = tile0 + 128u * k + 4u * lane;
            if (!WC_IN_BOUNDS(uint64_t(x) + 4 <= geo.total)) continue;
            if (EF == kEfF32) __stcs(reinterpret_cast<float4 *>(ef + x), ev);
            if (EF == kEfBf16)
                __stcs(reinterpret_cast<uint2 *>(ef16 + x),
                       make_uint2(f32x2_to_bf16x2_bits(ev.x, ev.y), f32x2_to_bf16x2_bits(ev.z, ev.w)));
        }
    }
    if (active && (lane & (LPB - 1)) == 0 && WC_IN_BOUNDS(out0 / B < geo.total / B))
        __stcs(scales + out0 / B, bs.scale);

    if (EF == kEfInt8) {
        // the new error of the block, quantized by the int8 absmax rule
        float m8 = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k)
#pragma unroll
            for (int j = 0; j < 4; ++j) m8 = fmaxf(m8, fabsf(en[EF == kEfInt8 ? k : 0][j]));
        m8 = group_max<LPB>(m8);
        const BlockScale bse = block_scale<127>(m8);
        if (!active) return;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                word |= (quant_code<127>(en[EF == kEfInt8 ? k : 0][j], bse).bits & 0xFFu) << (8 * j);
            const uint32_t x = tile0 + 128u * k + 4u * lane;
            if (WC_IN_BOUNDS(uint64_t(x) + 4 <= geo.total))
                __stcs(reinterpret_cast<unsigned int *>(ef8 + x), word);
        }
        if ((lane & (LPB - 1)) == 0 && WC_IN_BOUNDS(eblk < geo.total / B))
            __stcs(ef_scales + eblk, bse.scale);
    }
}

template <int B, int EF>
__global__ void __launch_bounds__(256)
ef_quant_int4_kernel(const uint16_t *__restrict__ g, void *__restrict__ ef_v,
                     float *__restrict__ ef_scales, uint8_t *__restrict__ codes,
                     float *__restrict__ scales, QgzGeometry geo, float s, float beta,
                     float one_minus_beta) {
    ef_quant_int4_warp<B, EF>(g, ef_v, ef_scales, codes, scales, geo, s, beta, one_minus_beta);
}

// The bf16 and int8 error buffers move 2 and 1 bytes per element each way
// instead of 4, so a warp has fewer bytes in flight; at B = 128 and 256 the
// same code under a register budget for 8 CTAs (64 warps) per SM keeps more
// of them resident.  (The fp32 buffer already saturates DRAM at 6 CTAs per
// SM, and larger blocks would spill.)  S1: the error scale s is 1 (the
// multiply by s is left out).
template <int B, int EF, bool S1>
__global__ void __launch_bounds__(256, 8)
ef_quant_int4_resident8_kernel(const uint16_t *__restrict__ g, void *__restrict__ ef_v,
                               float *__restrict__ ef_scales, uint8_t *__restrict__ codes,
                               float *__restrict__ scales, QgzGeometry geo, float s, float beta,
                               float one_minus_beta) {
    ef_quant_int4_warp<B, EF, S1>(g, ef_v, ef_scales, codes, scales, geo, s, beta,
                                  one_minus_beta);
}

template <int B>
static cudaError_t launch_ef_quant_b(const uint16_t *g, void *ef, int ef_mode, float *ef_scales,
                                     uint8_t *codes, float *scales, const QgzGeometry &geo,
                                     float s, float beta, cudaStream_t stream) {
    constexpr int T = B >= 128 ? B : 128;
    const uint32_t threads = 256;
    dim3 grid;
    if (B >= 128) {
        // one warp per block: x covers the S / B blocks of a slice, y the
        // slices, z the ranks
        const uint32_t blocks = geo.S / B;
        grid = dim3((blocks + threads / kWarp - 1) / (threads / kWarp), geo.R, geo.R);
    } else {
        const uint32_t tiles = uint32_t((uint64_t(geo.total) + T - 1) / T);  // no wrap near 2^32
        grid = dim3((tiles + threads / kWarp - 1) / (threads / kWarp));
    }
    const float omb = 1.0f - beta;
    constexpr bool kResident8 = B == 128 || B == 256;
    if constexpr (B >= 128) {
        if (ef != nullptr && ef_mode == kEfInt8) {
            // three blocks per warp at B = 128 and 256 (see ef_quant_int8ef_kernel)
            constexpr int NB = kResident8 ? 3 : 1;
            const uint32_t warps = (geo.S / B + NB - 1) / NB;
            const dim3 g8((warps + threads / kWarp - 1) / (threads / kWarp), geo.R, geo.R);
            constexpr int MINB = kResident8 ? 3 : 1;
            if (s == 1.0f)
                ef_quant_int8ef_kernel<B, NB, MINB, true><<<g8, threads, 0, stream>>>(
                    g, static_cast<int8_t *>(ef), ef_scales, codes, scales, geo, s, beta, omb,
                    exact2_constants());
            else
                ef_quant_int8ef_kernel<B, NB, MINB, false><<<g8, threads, 0, stream>>>(
                    g, static_cast<int8_t *>(ef), ef_scales, codes, scales, geo, s, beta, omb,
                    exact2_constants());
            return cudaPeekAtLastError();
        }
    }
#define WC_EFQ(KERNEL, MODE)                                                                   \
    KERNEL<B, MODE><<<grid, threads, 0, stream>>>(g, ef, ef_scales, codes, scales, geo, s, beta, \
                                                   omb)
    if (ef == nullptr) {
        WC_EFQ(ef_quant_int4_kernel, kEfNone);
    } else if (ef_mode == kEfBf16) {
        if constexpr (kResident8) {
            if (s == 1.0f)
                ef_quant_int4_resident8_kernel<B, kEfBf16, true><<<grid, threads, 0, stream>>>(
                    g, ef, ef_scales, codes, scales, geo, s, beta, omb);
            else
                ef_quant_int4_resident8_kernel<B, kEfBf16, false><<<grid, threads, 0, stream>>>(
                    g, ef, ef_scales, codes, scales, geo, s, beta, omb);
        } else {
            WC_EFQ(ef_quant_int4_kernel, kEfBf16);
        }
    } else if (ef_mode == kEfInt8) {
        WC_EFQ(ef_quant_int4_kernel, kEfInt8);
    } else {
        WC_EFQ(ef_quant_int4_kernel, kEfF32);
    }
#undef WC_EFQ
    return cudaPeekAtLastError();
}

WC_CHECK_RECORD_READER(check_record_qgz_quant)

cudaError_t launch_ef_quant_int4(const uint16_t *g, void *ef, int ef_mode, float *ef_scales,
                                 uint8_t *codes, float *scales, const QgzGeometry &geo, int B,
                                 float s, float beta, cudaStream_t stream) {
#define WC_EFQ_B(BB)                                                                       \
    case BB:                                                                               \
        return launch_ef_quant_b<BB>(g, ef, ef_mode, ef_scales, codes, scales, geo, s, beta, \
                                     stream);
    switch (B) {
        WC_EFQ_B(32) WC_EFQ_B(64) WC_EFQ_B(128) WC_EFQ_B(256) WC_EFQ_B(512) WC_EFQ_B(1024)
        default: return cudaErrorInvalidValue;
    }
#undef WC_EFQ_B
}

}  // namespace wc
