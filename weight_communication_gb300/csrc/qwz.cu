// qwz.cu -- qwZ int8 block weight quantization and dequantization.
//
// "ZeROPlusPlus.md", §1.2 ZeRO++ (quantized weight communication): the
// weights are quantized fp16 -> int8 before the forward all-gather, halving
// its volume, with block-based quantization (an independent scale per block
// of weights) to keep accuracy.  Here the weights are bf16.
//
// Quantization: one warp per block (a lane group per block for blocks shorter
// than the warp tile); lane t holds weights 256*k + 8*t + j, i.e. 16-byte
// bf16 loads and 8-byte code stores, both fully coalesced.  The raw bf16
// words stay in registers between the absmax pass and the code pass.
// Dequantization: a warp per 1024 weights, 32 per lane from two 16-byte code
// loads issued together, and 16-byte stores.
// Codes are rounded and unpacked with exact fp32 arithmetic (wc_device.cuh).
#include "wc_device.cuh"
#include "wc_internal.h"

namespace wc {

// REPLICA also writes the bf16 weights the codes stand for, bf16_rn(q*scale),
// in the same pass (the dequantized copy a node keeps).
template <int B, bool REPLICA>
__global__ void __launch_bounds__(256)
qwz_quant_int8_kernel(const uint16_t *__restrict__ w, int8_t *__restrict__ codes,
                      float *__restrict__ scales, uint16_t *__restrict__ replica, uint32_t n) {
    constexpr int T = B >= 256 ? B : 256;
    constexpr int K = T / 256;
    constexpr int LPB = B >= 256 ? 32 : B / 8;
    const int lane = threadIdx.x & (kWarp - 1);
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) / kWarp;
    if (uint64_t(warp) * T >= n) return;
    const uint32_t tile0 = warp * uint32_t(T);

    uint4 raw[K];
    bool active[K];
    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const uint32_t x = tile0 + 256u * k + 8u * lane;
        active[k] = x < n && WC_IN_BOUNDS(uint64_t(x) + 8 <= n);
        raw[k] = active[k] ? ld_stream_u4(w + x) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t *h = &raw[k].x;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            m = fmaxf(m, fabsf(bf16_bits_to_f32(h[j] & 0xFFFFu)));
            m = fmaxf(m, fabsf(bf16_bits_to_f32(h[j] >> 16)));
        }
    }
    m = group_max<LPB>(m);
    const BlockScale bs = block_scale<127>(m);

#pragma unroll
    for (int k = 0; k < K; ++k) {
        if (!active[k]) continue;
        const uint32_t x = tile0 + 256u * k + 8u * lane;
        const uint32_t *h = &raw[k].x;
        uint32_t word[2] = {0u, 0u};
        float d[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t half = (j & 1) ? (h[j / 2] >> 16) : (h[j / 2] & 0xFFFFu);
            const QCode qc = quant_code<127>(bf16_bits_to_f32(half), bs);
            word[j / 4] |= (qc.bits & 0xFFu) << (8 * (j % 4));
            d[j] = dequant(qc.q, bs.scale);
        }
        uint32_t rep[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) rep[j] = f32x2_to_bf16x2_bits(d[2 * j], d[2 * j + 1]);
        __stcs(reinterpret_cast<uint2 *>(codes + x), make_uint2(word[0], word[1]));
        if (REPLICA)
            __stcs(reinterpret_cast<uint4 *>(replica + x), make_uint4(rep[0], rep[1], rep[2], rep[3]));
        if (k == 0 && (lane & (LPB - 1)) == 0 && WC_IN_BOUNDS(x / B < n / B))
            __stcs(scales + x / B, bs.scale);
    }
}

// Warp tile of 1024 weights; lane t handles weights 512*k + 16*t + j (k < 2,
// j < 16): a 16-byte code load per k (512 B per warp instruction), both loads
// issued before any work so that each lane keeps 32 bytes in flight, and two
// 16-byte bf16 stores per k.  16 consecutive weights never straddle a block
// (B >= 32).
__global__ void __launch_bounds__(256)
qwz_dequant_int8_kernel(const int8_t *__restrict__ codes, const float *__restrict__ scales,
                        uint16_t *__restrict__ w_out, uint32_t n, uint32_t log2_b) {
    const uint32_t warp = (blockIdx.x * blockDim.x + threadIdx.x) / kWarp;
    const int lane = threadIdx.x & (kWarp - 1);
    if (uint64_t(warp) * 1024u >= n) return;
    const uint32_t tile0 = warp * 1024u;
    uint4 q[2];
    float sc[2];
    bool active[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint32_t x = tile0 + 512u * k + 16u * lane;
        // n is a multiple of 32, so 16 weights are all in or all out
        active[k] = x < n && WC_IN_BOUNDS(uint64_t(x) + 16 <= n) &&
                    WC_IN_BOUNDS((x >> log2_b) < (n >> log2_b));
        if (active[k]) {
            q[k] = ld_stream_u4(codes + x);
            sc[k] = __ldg(scales + (x >> log2_b));
        }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        if (!active[k]) continue;
        const uint32_t x = tile0 + 512u * k + 16u * lane;
        const uint32_t qw[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
        uint32_t h[8];
#pragma unroll
        for (int wq = 0; wq < 4; ++wq) {
            float f[4];
            unpack_int8x4(qw[wq], f);
            h[2 * wq] = f32x2_to_bf16x2_bits(dequant(f[0], sc[k]), dequant(f[1], sc[k]));
            h[2 * wq + 1] = f32x2_to_bf16x2_bits(dequant(f[2], sc[k]), dequant(f[3], sc[k]));
        }
        uint4 *dst = reinterpret_cast<uint4 *>(w_out + x);
        __stcs(dst, make_uint4(h[0], h[1], h[2], h[3]));
        __stcs(dst + 1, make_uint4(h[4], h[5], h[6], h[7]));
    }
}

template <int B>
static cudaError_t launch_qwz_quant_b(const uint16_t *w, int8_t *codes, float *scales,
                                      uint16_t *replica, uint32_t n, cudaStream_t stream) {
    constexpr int T = B >= 256 ? B : 256;
    const uint32_t tiles = uint32_t((uint64_t(n) + T - 1) / T);  // no wrap near 2^32
    const uint32_t threads = 256;
    const uint32_t grid = (tiles + threads / kWarp - 1) / (threads / kWarp);
    if (replica)
        qwz_quant_int8_kernel<B, true><<<grid, threads, 0, stream>>>(w, codes, scales, replica, n);
    else
        qwz_quant_int8_kernel<B, false><<<grid, threads, 0, stream>>>(w, codes, scales, replica, n);
    return cudaPeekAtLastError();
}

WC_CHECK_RECORD_READER(check_record_qwz)

cudaError_t launch_qwz_quant_int8(const uint16_t *w, int8_t *codes, float *scales,
                                  uint16_t *replica, uint32_t n, int B, cudaStream_t stream) {
    switch (B) {
        case 32: return launch_qwz_quant_b<32>(w, codes, scales, replica, n, stream);
        case 64: return launch_qwz_quant_b<64>(w, codes, scales, replica, n, stream);
        case 128: return launch_qwz_quant_b<128>(w, codes, scales, replica, n, stream);
        case 256: return launch_qwz_quant_b<256>(w, codes, scales, replica, n, stream);
        case 512: return launch_qwz_quant_b<512>(w, codes, scales, replica, n, stream);
        case 1024: return launch_qwz_quant_b<1024>(w, codes, scales, replica, n, stream);
        case 2048: return launch_qwz_quant_b<2048>(w, codes, scales, replica, n, stream);
        case 4096: return launch_qwz_quant_b<4096>(w, codes, scales, replica, n, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_qwz_dequant_int8(const int8_t *codes, const float *scales, uint16_t *w_out,
                                    uint32_t n, int B, cudaStream_t stream) {
    uint32_t log2_b = 0;
    while ((1u << log2_b) < uint32_t(B)) ++log2_b;
    const uint32_t threads = 256;
    const uint32_t warps = uint32_t((uint64_t(n) + 1023) / 1024);  // no wrap near 2^32
    const uint32_t grid = (warps + threads / kWarp - 1) / (threads / kWarp);
    qwz_dequant_int8_kernel<<<grid, threads, 0, stream>>>(codes, scales, w_out, n, log2_b);
    return cudaPeekAtLastError();
}

}  // namespace wc
