// wc_internal.h -- launchers shared between the kernel files and the C ABI.
// Arguments reaching these have been validated by the ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace wc {

// Sizes of one qgZ problem.  All element indices fit in 32 bits: the ABI
// rejects R*N >= 2^32.
struct QgzGeometry {
    uint32_t N;                // elements per rank
    uint32_t S;                // slice (shard) length, N / R
    uint32_t R;                // ranks
    uint32_t G;                // groups
    uint32_t L;                // ranks per group, R / G
    uint32_t blocks_per_rank;  // N / B
    uint32_t total;            // R * N
};

// ef: NULL, or the error buffer [R][N] in the form ef_mode names: 1 fp32,
// 2 bf16, 3 int8 codes with ef_scales [R][N/B] fp32 (gradient order).
constexpr int kEfModeF32 = 1, kEfModeBf16 = 2, kEfModeInt8 = 3;
cudaError_t launch_ef_quant_int4(const uint16_t *g, void *ef, int ef_mode, float *ef_scales,
                                 uint8_t *codes, float *scales, const QgzGeometry &geo, int B,
                                 float s, float beta, cudaStream_t stream);
cudaError_t launch_dequant_reduce(const uint8_t *codes, const float *scales,
                                  const QgzGeometry &geo, int B, float out_scale, void *out,
                                  bool out_bf16, cudaStream_t stream);
// ef1: fp32 [G*N] error of every requantized value (unit order), or NULL.
cudaError_t launch_dequant_reduce_requant(const uint8_t *codes, const float *scales,
                                          uint8_t *out_codes, float *out_scales,
                                          const QgzGeometry &geo, int B, float *ef1, float s,
                                          float beta, cudaStream_t stream);
// ef, ef_mode, ef_scales as in launch_ef_quant_int4; codes/scales: the
// ranks' send buffers, or both NULL.
cudaError_t launch_qgz_fused_step(const uint16_t *g, void *ef, int ef_mode, float *ef_scales,
                                  uint8_t *codes, float *scales, const QgzGeometry &geo, int B,
                                  float s, float beta, float out_scale, void *out, bool out_bf16,
                                  cudaStream_t stream);
// The same, with out_codes/out_scales the first hop's output as
// launch_dequant_reduce_requant writes it and ef1 its error buffer or NULL.
cudaError_t launch_qgz_first_hop_fused(const uint16_t *g, void *ef, int ef_mode,
                                       float *ef_scales, uint8_t *codes, float *scales,
                                       const QgzGeometry &geo, int B, float s, float beta,
                                       uint8_t *out_codes, float *out_scales, float *ef1,
                                       cudaStream_t stream);
// replica: bf16 [n] written with the dequantized weights, or NULL.
cudaError_t launch_qwz_quant_int8(const uint16_t *w, int8_t *codes, float *scales,
                                  uint16_t *replica, uint32_t n, int B, cudaStream_t stream);
cudaError_t launch_qwz_dequant_int8(const int8_t *codes, const float *scales, uint16_t *w_out,
                                    uint32_t n, int B, cudaStream_t stream);
cudaError_t launch_sr_accumulate(uint16_t *dst, uint16_t *src, uint32_t n, uint32_t seed,
                                 uint32_t step, cudaStream_t stream);
uint32_t sr_key(uint32_t seed, uint32_t step);

// Violation record of one source file's kernels in a checked build (see
// WC_IN_BOUNDS in wc_device.cuh).  sr_accumulate.cu has none: its kernel
// tests every access against the element count as part of its own logic.
struct CheckRecord {
    unsigned int count;       // accesses skipped since the last reset
    unsigned int first_line;  // source line of the first one (0: none)
};

#if defined(WC_CHECKED) && WC_CHECKED
cudaError_t check_record_qgz_quant(CheckRecord *out, bool reset, bool probe);
cudaError_t check_record_qgz_reduce(CheckRecord *out, bool reset, bool probe);
cudaError_t check_record_qgz_hop1(CheckRecord *out, bool reset, bool probe);
cudaError_t check_record_qgz_fused(CheckRecord *out, bool reset, bool probe);
cudaError_t check_record_qwz(CheckRecord *out, bool reset, bool probe);
#endif

}  // namespace wc
