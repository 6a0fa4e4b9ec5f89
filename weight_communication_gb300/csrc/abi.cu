// abi.cu -- the extern "C" entry points declared in include/wc.h: argument
// validation on the host, then exactly one kernel launch per call.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "../../include/wc.h"
#include "wc_internal.h"

namespace {

thread_local char g_last_error[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return code;
}

int from_cuda(cudaError_t err, const char *what) {
    if (err == cudaSuccess) return WC_OK;
    return fail(WC_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool pow2_in(int64_t b, int64_t lo, int64_t hi) {
    return b >= lo && b <= hi && (b & (b - 1)) == 0;
}

// Validates the sizes shared by the qgZ entry points and fills `geo`.
// Returns WC_OK, or an error code with the message set.
int qgz_geometry(const char *fn, int64_t N, int R, int G, int B, wc::QgzGeometry *geo) {
    if (N < 0) return fail(WC_EINVAL, "%s: N = %lld is negative", fn, (long long)N);
    if (R < 1 || G < 1) return fail(WC_EINVAL, "%s: need R >= 1 and G >= 1 (R=%d, G=%d)", fn, R, G);
    if (R % G) return fail(WC_EINVAL, "%s: G=%d does not divide R=%d", fn, G, R);
    if (!pow2_in(B, 32, 1024))
        return fail(WC_EINVAL, "%s: block B=%d must be a power of two in [32, 1024]", fn, B);
    if (N % R) return fail(WC_EINVAL, "%s: R=%d does not divide N=%lld", fn, R, (long long)N);
    const int64_t S = N / R;
    if (S % B) return fail(WC_EINVAL, "%s: B=%d does not divide the shard N/R=%lld", fn, B, (long long)S);
    // (R*N < 2^32 with B >= 32 dividing N/R also keeps R below 65536, the
    // grid's y limit that the reduce uses for destinations.)
    if (N >= (int64_t(1) << 32) || N * (int64_t)R >= (int64_t(1) << 32))
        return fail(WC_ERANGE, "%s: R*N = %lld must be below 2^32", fn, (long long)(N * R));
    geo->N = uint32_t(N);
    geo->S = uint32_t(S);
    geo->R = uint32_t(R);
    geo->G = uint32_t(G);
    geo->L = uint32_t(R / G);
    geo->blocks_per_rank = uint32_t(N / B);
    geo->total = uint32_t(N * R);
    return WC_OK;
}

#define WC_REQUIRE_PTR(fn, p)                                                        \
    do {                                                                             \
        if ((p) == nullptr) return fail(WC_EINVAL, "%s: %s is NULL", fn, #p);        \
        if (!aligned16(p)) return fail(WC_EALIGN, "%s: %s is not 16-byte aligned", fn, #p); \
    } while (0)

}  // namespace

extern "C" {

WC_API const char *wc_last_error(void) { return g_last_error; }

WC_API int wc_version(void) { return 1 * 10000 + 0 * 100 + 0; }

WC_API int wc_ef_quant_int4(const uint16_t *g, float *ef, uint8_t *codes, float *scales,
                            int64_t N, int R, int G, int B, float err_scale, float err_beta,
                            void *stream) {
    static const char *fn = "wc_ef_quant_int4";
    wc::QgzGeometry geo;
    int rc = qgz_geometry(fn, N, R, G, B, &geo);
    if (rc != WC_OK) return rc;
    if (N == 0) return WC_OK;
    WC_REQUIRE_PTR(fn, g);
    WC_REQUIRE_PTR(fn, codes);
    WC_REQUIRE_PTR(fn, scales);
    if (ef != nullptr && !aligned16(ef)) return fail(WC_EALIGN, "%s: ef is not 16-byte aligned", fn);
    return from_cuda(wc::launch_ef_quant_int4(g, ef, wc::kEfModeF32, nullptr, codes, scales, geo,
                                              B, err_scale, err_beta,
                                              static_cast<cudaStream_t>(stream)),
                     fn);
}

WC_API int wc_ef_quant_int4_bf16ef(const uint16_t *g, uint16_t *ef16, uint8_t *codes,
                                   float *scales, int64_t N, int R, int G, int B,
                                   float err_scale, float err_beta, void *stream) {
    static const char *fn = "wc_ef_quant_int4_bf16ef";
    wc::QgzGeometry geo;
    int rc = qgz_geometry(fn, N, R, G, B, &geo);
    if (rc != WC_OK) return rc;
    if (N == 0) return WC_OK;
    WC_REQUIRE_PTR(fn, g);
    WC_REQUIRE_PTR(fn, ef16);
    WC_REQUIRE_PTR(fn, codes);
    WC_REQUIRE_PTR(fn, scales);
    return from_cuda(wc::launch_ef_quant_int4(g, ef16, wc::kEfModeBf16, nullptr, codes, scales,
                                              geo, B, err_scale, err_beta,
                                              static_cast<cudaStream_t>(stream)),
                     fn);
}

WC_API int wc_ef_quant_int4_int8ef(const uint16_t *g, int8_t *ef8, float *ef8_scales,
                                   uint8_t *codes, float *scales, int64_t N, int R, int G,
                                   int B, float err_scale, float err_beta, void *stream) {
    static const char *fn = "wc_ef_quant_int4_int8ef";
    wc::QgzGeometry geo;
    int rc = qgz_geometry(fn, N, R, G, B, &geo);
    if (rc != WC_OK) return rc;
    if (N == 0) return WC_OK;
    WC_REQUIRE_PTR(fn, g);
    WC_REQUIRE_PTR(fn, ef8);
    WC_REQUIRE_PTR(fn, ef8_scales);
    WC_REQUIRE_PTR(fn, codes);
    WC_REQUIRE_PTR(fn, scales);
    return from_cuda(wc::launch_ef_quant_int4(g, ef8, wc::kEfModeInt8, ef8_scales, codes, scales,
                                              geo, B, err_scale, err_beta,
                                              static_cast<cudaStream_t>(stream)),
                     fn);
}

WC_API int wc_dequant_reduce(const uint8_t *codes, const float *scales, int64_t N, int R,
                             int G, int B, float out_scale, void *out, int out_dtype,
                             void *stream) {
    static const char *fn = "wc_dequant_reduce";
    wc::QgzGeometry geo;
    int rc = qgz_geometry(fn, N, R, G, B, &geo);
    if (rc != WC_OK) return rc;
    if (out_dtype != WC_F32 && out_dtype != WC_BF16)
        return fail(WC_EINVAL, "%s: out_dtype %d is neither WC_F32 nor WC_BF16", fn, out_dtype);
    if (N == 0) return WC_OK;
    WC_REQUIRE_PTR(fn, codes);
    WC_REQUIRE_PTR(fn, scales);
    WC_REQUIRE_PTR(fn, out);
    return from_cuda(wc::launch_dequant_reduce(codes, scales, geo, B, out_scale, out,
                                               out_dtype == WC_BF16,
                                               static_cast<cudaStream_t>(stream)),
                     fn);
}

WC_API int wc_dequant_reduce_requant(const uint8_t *codes, const float *scales, int64_t N,
                                     int R, int G, int B, uint8_t *out_codes,
                                     float *out_scales, void *stream) {
    static const char *fn = "wc_dequant_reduce_requant";
    wc::QgzGeometry geo;
    int rc = qgz_geometry(fn, N, R, G, B, &geo);
    if (rc != WC_OK) return rc;
    if (N * (int64_t)G >= (int64_t(1) << 32))
        return fail(WC_ERANGE, "%s: G*N must be below 2^32", fn);
    if (N == 0) return WC_OK;
    WC_REQUIRE_PTR(fn, codes);
    WC_REQUIRE_PTR(fn, scales);
    WC_REQUIRE_PTR(fn, out_codes);
    WC_REQUIRE_PTR(fn, out_scales);
    return from_cuda(wc::launch_dequant_reduce_requant(codes, scales, out_codes, out_scales, geo,
                                                       B, nullptr, 0.0f, 0.0f,
                                                       static_cast<cudaStream_t>(stream)),
                     fn);
}

WC_API int wc_dequant_reduce_requant_ef(const uint8_t *codes, const float *scales, int64_t N,
                                        int R, int G, int B, uint8_t *out_codes,
                                        float *out_scales, float *ef1, float err_scale,
                                        float err_beta, void *stream) {
    static const char *fn = "wc_dequant_reduce_requant_ef";
    wc::QgzGeometry geo;
    int rc = qgz_geometry(fn, N, R, G, B, &geo);
    if (rc != WC_OK) return rc;
    if (N * (int64_t)G >= (int64_t(1) << 32))
        return fail(WC_ERANGE, "%s: G*N must be below 2^32", fn);
    if (N == 0) return WC_OK;
    WC_REQUIRE_PTR(fn, codes);
    WC_REQUIRE_PTR(fn, scales);
    WC_REQUIRE_PTR(fn, out_codes);
    WC_REQUIRE_PTR(fn, out_scales);
    WC_REQUIRE_PTR(fn, ef1);
    return from_cuda(wc::launch_dequant_reduce_requant(codes, scales, out_codes, out_scales, geo,
                                                       B, ef1, err_scale, err_beta,
                                                       static_cast<cudaStream_t>(stream)),
                     fn);
}

// The fused step's checks and launch for every error-buffer form (ef_mode:
// the buffer's form; ef_needed: the entry point takes no NULL buffer).
static int fused_step(const char *fn, const uint16_t *g, void *ef, int ef_mode, bool ef_needed,
                      float *ef_scales, uint8_t *codes, float *scales, int64_t N, int R, int B,
                      float err_scale, float err_beta, float out_scale, void *out, int out_dtype,
                      void *stream) {
    wc::QgzGeometry geo;
    int rc = qgz_geometry(fn, N, R, 1, B, &geo);
    if (rc != WC_OK) return rc;
    if (B < 128) return fail(WC_EINVAL, "%s: block B=%d must be at least 128", fn, B);
    if (out_dtype != WC_F32 && out_dtype != WC_BF16)
        return fail(WC_EINVAL, "%s: out_dtype %d is neither WC_F32 nor WC_BF16", fn, out_dtype);
    if ((codes == nullptr) != (scales == nullptr))
        return fail(WC_EINVAL, "%s: codes and scales must both be given or both be NULL", fn);
    if (N == 0) return WC_OK;
    WC_REQUIRE_PTR(fn, g);
    WC_REQUIRE_PTR(fn, out);
    if (ef_needed) WC_REQUIRE_PTR(fn, ef);
    if (ef != nullptr && !aligned16(ef)) return fail(WC_EALIGN, "%s: ef is not 16-byte aligned", fn);
    if (ef_mode == wc::kEfModeInt8) WC_REQUIRE_PTR(fn, ef_scales);
    if (codes != nullptr && (!aligned16(codes) || !aligned16(scales)))
        return fail(WC_EALIGN, "%s: codes or scales is not 16-byte aligned", fn);
    return from_cuda(wc::launch_qgz_fused_step(g, ef, ef_mode, ef_scales, codes, scales, geo, B,
                                               err_scale, err_beta, out_scale, out,
                                               out_dtype == WC_BF16,
                                               static_cast<cudaStream_t>(stream)),
                     fn);
}

WC_API int wc_qgz_step_fused(const uint16_t *g, float *ef, uint8_t *codes, float *scales,
                             int64_t N, int R, int B, float err_scale, float err_beta,
                             float out_scale, void *out, int out_dtype, void *stream) {
    return fused_step("wc_qgz_step_fused", g, ef, wc::kEfModeF32, false, nullptr, codes, scales,
                      N, R, B, err_scale, err_beta, out_scale, out, out_dtype, stream);
}

WC_API int wc_qgz_step_fused_bf16ef(const uint16_t *g, uint16_t *ef16, uint8_t *codes,
                                    float *scales, int64_t N, int R, int B, float err_scale,
                                    float err_beta, float out_scale, void *out, int out_dtype,
                                    void *stream) {
    return fused_step("wc_qgz_step_fused_bf16ef", g, ef16, wc::kEfModeBf16, true, nullptr, codes,
                      scales, N, R, B, err_scale, err_beta, out_scale, out, out_dtype, stream);
}

WC_API int wc_qgz_step_fused_int8ef(const uint16_t *g, int8_t *ef8, float *ef8_scales,
                                    uint8_t *codes, float *scales, int64_t N, int R, int B,
                                    float err_scale, float err_beta, float out_scale, void *out,
                                    int out_dtype, void *stream) {
    return fused_step("wc_qgz_step_fused_int8ef", g, ef8, wc::kEfModeInt8, true, ef8_scales,
                      codes, scales, N, R, B, err_scale, err_beta, out_scale, out, out_dtype,
                      stream);
}

// The fused first stage's checks and launch for every error-buffer form.
static int first_hop_fused(const char *fn, const uint16_t *g, void *ef, int ef_mode,
                           bool ef_needed, float *ef_scales, uint8_t *codes, float *scales,
                           int64_t N, int R, int G, int B, float err_scale, float err_beta,
                           uint8_t *out_codes, float *out_scales, float *ef1, void *stream) {
    wc::QgzGeometry geo;
    int rc = qgz_geometry(fn, N, R, G, B, &geo);
    if (rc != WC_OK) return rc;
    if (B < 128) return fail(WC_EINVAL, "%s: block B=%d must be at least 128", fn, B);
    if (N * (int64_t)G >= (int64_t(1) << 32))
        return fail(WC_ERANGE, "%s: G*N must be below 2^32", fn);
    if ((codes == nullptr) != (scales == nullptr))
        return fail(WC_EINVAL, "%s: codes and scales must both be given or both be NULL", fn);
    if (N == 0) return WC_OK;
    WC_REQUIRE_PTR(fn, g);
    WC_REQUIRE_PTR(fn, out_codes);
    WC_REQUIRE_PTR(fn, out_scales);
    if (ef_needed) WC_REQUIRE_PTR(fn, ef);
    if (ef != nullptr && !aligned16(ef)) return fail(WC_EALIGN, "%s: ef is not 16-byte aligned", fn);
    if (ef_mode == wc::kEfModeInt8) WC_REQUIRE_PTR(fn, ef_scales);
    if (codes != nullptr && (!aligned16(codes) || !aligned16(scales)))
        return fail(WC_EALIGN, "%s: codes or scales is not 16-byte aligned", fn);
    if (!aligned16(out_codes) || !aligned16(out_scales))
        return fail(WC_EALIGN, "%s: out_codes or out_scales is not 16-byte aligned", fn);
    if (ef1 != nullptr && !aligned16(ef1)) return fail(WC_EALIGN, "%s: ef1 is not 16-byte aligned", fn);
    return from_cuda(wc::launch_qgz_first_hop_fused(g, ef, ef_mode, ef_scales, codes, scales, geo,
                                                    B, err_scale, err_beta, out_codes, out_scales,
                                                    ef1, static_cast<cudaStream_t>(stream)),
                     fn);
}

WC_API int wc_qgz_first_hop_fused(const uint16_t *g, float *ef, uint8_t *codes, float *scales,
                                  int64_t N, int R, int G, int B, float err_scale,
                                  float err_beta, uint8_t *out_codes, float *out_scales,
                                  float *ef1, void *stream) {
    return first_hop_fused("wc_qgz_first_hop_fused", g, ef, wc::kEfModeF32, false, nullptr, codes,
                           scales, N, R, G, B, err_scale, err_beta, out_codes, out_scales, ef1,
                           stream);
}

WC_API int wc_qgz_first_hop_fused_bf16ef(const uint16_t *g, uint16_t *ef16, uint8_t *codes,
                                         float *scales, int64_t N, int R, int G, int B,
                                         float err_scale, float err_beta, uint8_t *out_codes,
                                         float *out_scales, float *ef1, void *stream) {
    return first_hop_fused("wc_qgz_first_hop_fused_bf16ef", g, ef16, wc::kEfModeBf16, true,
                           nullptr, codes, scales, N, R, G, B, err_scale, err_beta, out_codes,
                           out_scales, ef1, stream);
}

WC_API int wc_qgz_first_hop_fused_int8ef(const uint16_t *g, int8_t *ef8, float *ef8_scales,
                                         uint8_t *codes, float *scales, int64_t N, int R, int G,
                                         int B, float err_scale, float err_beta,
                                         uint8_t *out_codes, float *out_scales, float *ef1,
                                         void *stream) {
    return first_hop_fused("wc_qgz_first_hop_fused_int8ef", g, ef8, wc::kEfModeInt8, true,
                           ef8_scales, codes, scales, N, R, G, B, err_scale, err_beta, out_codes,
                           out_scales, ef1, stream);
}

static int qwz_sizes(const char *fn, int64_t n, int B) {
    if (n < 0) return fail(WC_EINVAL, "%s: n = %lld is negative", fn, (long long)n);
    if (!pow2_in(B, 32, 4096))
        return fail(WC_EINVAL, "%s: block B=%d must be a power of two in [32, 4096]", fn, B);
    if (n % B) return fail(WC_EINVAL, "%s: B=%d does not divide n=%lld", fn, B, (long long)n);
    if (n >= (int64_t(1) << 32)) return fail(WC_ERANGE, "%s: n must be below 2^32", fn);
    return WC_OK;
}

WC_API int wc_qwz_quant_int8(const uint16_t *w, int8_t *codes, float *scales, int64_t n, int B,
                             void *stream) {
    static const char *fn = "wc_qwz_quant_int8";
    int rc = qwz_sizes(fn, n, B);
    if (rc != WC_OK) return rc;
    if (n == 0) return WC_OK;
    WC_REQUIRE_PTR(fn, w);
    WC_REQUIRE_PTR(fn, codes);
    WC_REQUIRE_PTR(fn, scales);
    return from_cuda(wc::launch_qwz_quant_int8(w, codes, scales, nullptr, uint32_t(n), B,
                                               static_cast<cudaStream_t>(stream)),
                     fn);
}

WC_API int wc_qwz_quant_replica_int8(const uint16_t *w, int8_t *codes, float *scales,
                                     uint16_t *replica, int64_t n, int B, void *stream) {
    static const char *fn = "wc_qwz_quant_replica_int8";
    int rc = qwz_sizes(fn, n, B);
    if (rc != WC_OK) return rc;
    if (n == 0) return WC_OK;
    WC_REQUIRE_PTR(fn, w);
    WC_REQUIRE_PTR(fn, codes);
    WC_REQUIRE_PTR(fn, scales);
    WC_REQUIRE_PTR(fn, replica);
    return from_cuda(wc::launch_qwz_quant_int8(w, codes, scales, replica, uint32_t(n), B,
                                               static_cast<cudaStream_t>(stream)),
                     fn);
}

WC_API int wc_qwz_dequant_int8(const int8_t *codes, const float *scales, uint16_t *w_out,
                               int64_t n, int B, void *stream) {
    static const char *fn = "wc_qwz_dequant_int8";
    int rc = qwz_sizes(fn, n, B);
    if (rc != WC_OK) return rc;
    if (n == 0) return WC_OK;
    WC_REQUIRE_PTR(fn, codes);
    WC_REQUIRE_PTR(fn, scales);
    WC_REQUIRE_PTR(fn, w_out);
    return from_cuda(wc::launch_qwz_dequant_int8(codes, scales, w_out, uint32_t(n), B,
                                                 static_cast<cudaStream_t>(stream)),
                     fn);
}

WC_API int wc_sr_accumulate_bf16(uint16_t *dst, uint16_t *src, int64_t n, uint32_t seed,
                                 uint32_t step, void *stream) {
    static const char *fn = "wc_sr_accumulate_bf16";
    if (n < 0) return fail(WC_EINVAL, "%s: n = %lld is negative", fn, (long long)n);
    if (n >= (int64_t(1) << 32)) return fail(WC_ERANGE, "%s: n must be below 2^32", fn);
    if (n == 0) return WC_OK;
    WC_REQUIRE_PTR(fn, dst);
    WC_REQUIRE_PTR(fn, src);
    const uintptr_t a = reinterpret_cast<uintptr_t>(dst), b = reinterpret_cast<uintptr_t>(src);
    const uintptr_t bytes = uintptr_t(n) * 2u;
    if (a < b + bytes && b < a + bytes) return fail(WC_EINVAL, "%s: dst and src overlap", fn);
    return from_cuda(wc::launch_sr_accumulate(dst, src, uint32_t(n), seed, step,
                                              static_cast<cudaStream_t>(stream)),
                     fn);
}

WC_API int wc_checked_violations(int flags) {
    static const char *fn = "wc_checked_violations";
    if (flags & ~(WC_CHECK_RESET | WC_CHECK_PROBE))
        return fail(WC_EINVAL, "%s: unknown flags 0x%x", fn, unsigned(flags));
#if defined(WC_CHECKED) && WC_CHECKED
    struct Reader {
        const char *file;
        cudaError_t (*read)(wc::CheckRecord *, bool, bool);
    };
    static const Reader readers[] = {
        {"qgz_quant.cu", wc::check_record_qgz_quant}, {"qgz_reduce.cu", wc::check_record_qgz_reduce},
        {"qgz_hop1.cu", wc::check_record_qgz_hop1},   {"qgz_fused.cu", wc::check_record_qgz_fused},
        {"qwz.cu", wc::check_record_qwz},
    };
    uint64_t total = 0;
    const char *first_file = nullptr;
    unsigned int first_line = 0;
    for (const Reader &r : readers) {
        wc::CheckRecord rec = {0u, 0u};
        const cudaError_t e = r.read(&rec, (flags & WC_CHECK_RESET) != 0,
                                     (flags & WC_CHECK_PROBE) != 0);
        if (e != cudaSuccess) return from_cuda(e, fn);
        if (rec.count != 0 && first_file == nullptr) {
            first_file = r.file;
            first_line = rec.first_line;
        }
        total += rec.count;
    }
    if (total == 0) return 0;
    fail(WC_OK, "%s: %llu accesses skipped, one of them in %s line %u", fn,
         (unsigned long long)total, first_file, first_line);
    return total > 0x7FFFFFFFull ? 0x7FFFFFFF : int(total);
#else
    return fail(WC_EINVAL, "%s: this library was built without checks (WC_CHECKED=1)", fn);
#endif
}

}  // extern "C"
