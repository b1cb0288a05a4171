// fa_api.cu -- the C ABI (include/fa.h): argument validation, status
// mapping and dispatch to the fp32 SIMT kernel or the bf16 tcgen05 kernel.
//
// Validation follows the interface of "FlashAttention forward in C"
// (section 4): every error is returned before any launch and before anything
// is written.  There is no CPU fallback: a configuration the GPU kernels do
// not cover is rejected with FA_EUNSUPPORTED.
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <limits>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

thread_local char g_last_error[512] = "";

fa_status fail(fa_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

bool mul_ok(int64_t a, int64_t b, int64_t &out) {
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > std::numeric_limits<int64_t>::max() / a) return false;
    out = a * b;
    return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int64_t kMaxLen = int64_t(1) << 30;

}  // namespace

extern "C" const char *fa_last_error(void) { return g_last_error; }

extern "C" int fa_version(void) { return 100; }

extern "C" fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                            int64_t Hq, int64_t Hkv, int64_t Tq, int64_t Tk, int64_t d, float scale,
                            int64_t q_offset, int causal, int64_t window, const float *sinks, const float *mask,
                            int64_t mask_sb, int64_t mask_sh, int64_t mask_sq, int64_t mask_sk, int dtype,
                            void *stream) {
    g_last_error[0] = '\0';
    if (dtype != FA_DTYPE_F32 && dtype != FA_DTYPE_BF16) return fail(FA_EINVAL, "unknown dtype %d", dtype);
    if (B < 0 || Hq < 0 || Hkv < 0 || Tq < 0 || Tk < 0 || d < 0)
        return fail(FA_EINVAL, "negative size (B=%lld Hq=%lld Hkv=%lld Tq=%lld Tk=%lld d=%lld)", (long long)B,
                    (long long)Hq, (long long)Hkv, (long long)Tq, (long long)Tk, (long long)d);
    if (q_offset < 0) return fail(FA_EINVAL, "negative q_offset %lld", (long long)q_offset);
    if (!std::isfinite(scale)) return fail(FA_EINVAL, "scale is not finite");
    if (mask && (mask_sb < 0 || mask_sh < 0 || mask_sq < 0 || mask_sk < 0))
        return fail(FA_EINVAL, "negative mask stride");
    if (Hkv == 0 ? Hq > 0 : (Hkv > Hq || Hq % Hkv != 0))
        return fail(FA_ESHAPE, "Hq=%lld is not a multiple of Hkv=%lld (or Hkv > Hq)", (long long)Hq,
                    (long long)Hkv);

    int64_t rows = 0, q_elems = 0, kv_rows = 0, kv_elems = 0;
    if (!mul_ok(B, Hq, rows) || !mul_ok(rows, Tq, rows) || !mul_ok(rows, d, q_elems) ||
        !mul_ok(B, Hkv, kv_rows) || !mul_ok(kv_rows, Tk, kv_rows) || !mul_ok(kv_rows, d, kv_elems) ||
        q_elems > (std::numeric_limits<int64_t>::max() >> 3) || kv_elems > (std::numeric_limits<int64_t>::max() >> 3))
        return fail(FA_EINVAL, "element counts overflow");
    if (rows == 0) return FA_OK;  // nothing to compute, nothing to write

    if (!q || !o) return fail(FA_EINVAL, "q or o is NULL");
    if (Tk > 0 && (!k || !v)) return fail(FA_EINVAL, "k or v is NULL with Tk > 0");

    if (d == 0 || (d & 1)) return fail(FA_EUNSUPPORTED, "d=%lld: d must be even and positive", (long long)d);
    if (dtype == FA_DTYPE_F32 && d > 256)
        return fail(FA_EUNSUPPORTED, "fp32 path supports d <= 256 (got %lld)", (long long)d);
    if (dtype == FA_DTYPE_BF16 && (d % 8 != 0 || d > 128))
        return fail(FA_EUNSUPPORTED, "bf16 path supports d a multiple of 8 up to 128 (got %lld)", (long long)d);
    if (Tq >= kMaxLen || Tk >= kMaxLen || q_offset >= kMaxLen)
        return fail(FA_EUNSUPPORTED, "Tq, Tk and q_offset must be below 2^30");
    if (B * Hq >= (int64_t(1) << 24)) return fail(FA_EUNSUPPORTED, "B*Hq must be below 2^24");
    if (!aligned16(q) || !aligned16(o) || (Tk > 0 && (!aligned16(k) || !aligned16(v))))
        return fail(FA_EUNSUPPORTED, "q, k, v and o must be 16-byte aligned");

    fa::Params P;
    std::memset(&P, 0, sizeof P);
    P.q = q;
    P.k = k;
    P.v = v;
    P.o = o;
    P.lse = lse;
    P.sinks = sinks;
    P.mask = mask;
    P.msb = mask_sb;
    P.msh = mask_sh;
    P.msq = mask_sq;
    P.msk = mask_sk;
    P.B = (int)B;
    P.Hq = (int)Hq;
    P.Hkv = (int)Hkv;
    P.Tq = (int)Tq;
    P.Tk = (int)Tk;
    P.d = (int)d;
    P.group = (int)(Hq / Hkv);
    P.splits = 1;
    P.q_offset = (int)q_offset;
    P.causal = causal ? 1 : 0;
    // A window wider than every possible distance is no window.
    P.window = window <= 0 ? 0 : (window >= 2 * kMaxLen ? 0 : (int)window);
    P.scale = scale;
    P.scale_log2 = (float)((double)scale * 1.4426950408889634);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = dtype == FA_DTYPE_F32 ? fa::launch_f32(P, s) : fa::launch_bf16(P, s);
    if (e != cudaSuccess) return fail(FA_ECUDA, "CUDA error: %s", cudaGetErrorString(e));
    return FA_OK;
}
