// fa_api.cu -- the C ABI (include/fa.h): argument validation, status
// mapping and dispatch to the fp32 SIMT kernel or the bf16 tcgen05 kernel.
//
// Validation follows the interface of "FlashAttention forward in C"
// (section 4): every error is returned before any launch and before anything
// is written.  There is no CPU fallback: a configuration the GPU kernels do
// not cover is rejected with FA_EUNSUPPORTED.
#include <algorithm>
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

extern "C" int fa_version(void) { return 101; }

extern "C" fa_status fa_device_status(void *stream) {
    g_last_error[0] = '\0';
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int tc5 = 0, tf32 = 0;
    cudaError_t e = fa::bf16_watchdog(s, &tc5);
    if (e == cudaSuccess) e = fa::f32tc_watchdog(s, &tf32);
    if (e != cudaSuccess) return fail(FA_ECUDA, "CUDA error: %s", cudaGetErrorString(e));
    if (tc5 != 0 || tf32 != 0)
        return fail(FA_ETIMEOUT, "a bounded wait ran out in the %s kernel since the last check; outputs of the calls "
                                 "in between are not valid",
                    tc5 != 0 && tf32 != 0 ? "bf16/e4m3 and fp32 tensor-core" : tc5 != 0 ? "bf16/e4m3" : "fp32 tensor-core");
    return FA_OK;
}

namespace fa {
int g_test_max_ctas = 0;
}

extern "C" fa_status fa_test_max_ctas(int64_t n) {
    g_last_error[0] = '\0';
    if (n < 0) return fail(FA_EINVAL, "fa_test_max_ctas: n = %lld is negative", (long long)n);
    fa::g_test_max_ctas = n > (int64_t)1 << 30 ? 1 << 30 : (int)n;
    return FA_OK;
}

extern "C" fa_status fa_test_drop_arrive(int enable) {
    g_last_error[0] = '\0';
    const int on = enable ? 1 : 0;
    cudaError_t e = fa::bf16_set_drop_arrive(on);
    if (e == cudaSuccess) e = fa::f32tc_set_drop_arrive(on);
    if (e != cudaSuccess) return fail(FA_ECUDA, "CUDA error: %s", cudaGetErrorString(e));
    return FA_OK;
}

namespace {

// Row spans of a [B, H, T, d] view with strides (sb, sh, st), d contiguous:
// false if a dimension of extent > 1 has a negative stride, or if two rows
// share memory under the sufficient rule "each stride (in increasing order)
// covers the span of the dimensions inside it".  `bytes_last` is the offset
// of the last element + 1 (in elements).
bool layout_ok(int64_t B, int64_t H, int64_t T, int64_t d, int64_t sb, int64_t sh, int64_t st, bool distinct,
               int64_t &span) {
    span = 0;
    if (B == 0 || H == 0 || T == 0) return true;  // an empty tensor has no rows
    struct Dim { int64_t n, s; } dims[3] = {{B, sb}, {H, sh}, {T, st}};
    for (auto &x : dims)
        if (x.n > 1 && x.s < 0) return false;
    // sort by stride
    for (int i = 0; i < 3; ++i)
        for (int j = i + 1; j < 3; ++j)
            if (dims[j].s < dims[i].s) std::swap(dims[i], dims[j]);
    span = d;
    for (auto &x : dims) {
        if (x.n <= 1) continue;
        if (distinct && x.s < span) return false;
        int64_t ext = 0;
        if (!mul_ok(x.s, x.n - 1, ext) || ext > std::numeric_limits<int64_t>::max() - span) return false;
        span = distinct ? ext + span : std::max(span, ext + d);
    }
    return true;
}

bool known_dtype(int dtype) {
    return dtype == FA_DTYPE_F32 || dtype == FA_DTYPE_BF16 || dtype == FA_DTYPE_F32_TC || dtype == FA_DTYPE_FP8_E4M3;
}

// Every stride of a dimension with extent > 1 is a multiple of `m` elements.
bool strides_multiple(int64_t B, int64_t H, int64_t T, int64_t sb, int64_t sh, int64_t st, int64_t m) {
    return (B <= 1 || sb % m == 0) && (H <= 1 || sh % m == 0) && (T <= 1 || st % m == 0);
}

fa_status fwd_impl(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B, int64_t Hq,
                   int64_t Hkv, int64_t Tq, int64_t Tk, int64_t d, const int64_t *qs, const int64_t *ks,
                   const int64_t *vs, const int64_t *os, float scale, int64_t q_offset, int causal, int64_t window,
                   const float *sinks, const float *mask, int64_t mask_sb, int64_t mask_sh, int64_t mask_sq,
                   int64_t mask_sk, int dtype, void *stream, bool splitkv = false, void *workspace = nullptr,
                   size_t workspace_bytes = 0, bool noalloc = false) {
    g_last_error[0] = '\0';
    if (!known_dtype(dtype)) return fail(FA_EINVAL, "unknown dtype %d", dtype);
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
    int64_t span = 0;
    if (!layout_ok(B, Hq, Tq, d, qs[0], qs[1], qs[2], false, span) ||
        !layout_ok(B, Hkv, Tk, d, ks[0], ks[1], ks[2], false, span) ||
        !layout_ok(B, Hkv, Tk, d, vs[0], vs[1], vs[2], false, span))
        return fail(FA_EINVAL, "q, k or v strides are negative or their extents overflow");
    if (!layout_ok(B, Hq, Tq, d, os[0], os[1], os[2], true, span))
        return fail(FA_EINVAL, "o strides are negative or make two output rows overlap");
    if (rows == 0) return FA_OK;  // nothing to compute, nothing to write

    if (!q || !o) return fail(FA_EINVAL, "q or o is NULL");
    if (Tk > 0 && (!k || !v)) return fail(FA_EINVAL, "k or v is NULL with Tk > 0");

    if (d == 0 || (d & 1)) return fail(FA_EUNSUPPORTED, "d=%lld: d must be even and positive", (long long)d);
    if (dtype == FA_DTYPE_F32 && d > 256)
        return fail(FA_EUNSUPPORTED, "fp32 path supports d <= 256 (got %lld)", (long long)d);
    if (dtype == FA_DTYPE_BF16 && (d % 8 != 0 || d > 128))
        return fail(FA_EUNSUPPORTED, "bf16 path supports d a multiple of 8 up to 128 (got %lld)", (long long)d);
    if (dtype == FA_DTYPE_F32_TC && (d % 4 != 0 || d > 128))
        return fail(FA_EUNSUPPORTED, "tensor-core fp32 path supports d a multiple of 4 up to 128 (got %lld)",
                    (long long)d);
    if (dtype == FA_DTYPE_FP8_E4M3 && (d % 16 != 0 || d > 128))
        return fail(FA_EUNSUPPORTED, "e4m3 path supports d a multiple of 16 up to 128 (got %lld)", (long long)d);
    if (Tq >= kMaxLen || Tk >= kMaxLen || q_offset >= kMaxLen)
        return fail(FA_EUNSUPPORTED, "Tq, Tk and q_offset must be below 2^30");
    if (B * Hq >= (int64_t(1) << 24)) return fail(FA_EUNSUPPORTED, "B*Hq must be below 2^24");
    if (!aligned16(q) || !aligned16(o) || (Tk > 0 && (!aligned16(k) || !aligned16(v))))
        return fail(FA_EUNSUPPORTED, "q, k, v and o must be 16-byte aligned");
    // bf16, e4m3 and fp32 on the tensor cores: tensor-map strides are
    // 16-byte multiples below 2^40 bytes (o is bf16 with e4m3 inputs).  fp32
    // on the SIMT cores: rows start on 8-byte boundaries (16-byte copies when
    // all do).
    const bool tma = dtype != FA_DTYPE_F32;
    const int64_t in_bytes = dtype == FA_DTYPE_FP8_E4M3 ? 1 : (dtype == FA_DTYPE_BF16 ? 2 : 4);
    const int64_t out_bytes = dtype == FA_DTYPE_FP8_E4M3 ? 2 : in_bytes;
    const int64_t m = tma ? 16 / in_bytes : 2, mo = tma ? 16 / out_bytes : 2;
    const bool kv = Tk > 0;
    if (!strides_multiple(B, Hq, Tq, qs[0], qs[1], qs[2], m) || !strides_multiple(B, Hq, Tq, os[0], os[1], os[2], mo) ||
        (kv && (!strides_multiple(B, Hkv, Tk, ks[0], ks[1], ks[2], m) ||
                !strides_multiple(B, Hkv, Tk, vs[0], vs[1], vs[2], m))))
        return fail(FA_EUNSUPPORTED, "strides must be multiples of %lld elements (o: %lld) for this dtype",
                    (long long)m, (long long)mo);
    if (tma) {
        const int64_t ext[4][3] = {{B, Hq, Tq}, {B, Hkv, Tk}, {B, Hkv, Tk}, {B, Hq, Tq}};
        const int64_t *all[4] = {qs, ks, vs, os};
        for (int t = 0; t < 4; ++t)
            for (int i = 0; i < 3; ++i) {
                const int64_t lim = ((int64_t(1) << 40) / (t == 3 ? out_bytes : in_bytes)) - 1;  // elements
                if (all[t][i] > lim) return fail(FA_EUNSUPPORTED, "a stride reaches 2^40 bytes");
                if (ext[t][i] > 1 && all[t][i] <= 0 && (t == 0 || t == 3 || kv))
                    return fail(FA_EUNSUPPORTED, "strides must be positive for this dtype (tensor maps)");
            }
        if (B > 0x7fffffff || Hq > 0x7fffffff) return fail(FA_EUNSUPPORTED, "B and H must fit 31 bits");
    }
    // The kernels index the query tiles of each (batch, head) as 31-bit
    // block or unit numbers: 128-row tiles on the tensor cores, 64 on SIMT.
    if (tma && ((Tq + 127) / 128) * B * Hq > 0x7fffffff)
        return fail(FA_EUNSUPPORTED, "tensor-core paths: B*Hq*ceil(Tq/128) must be below 2^31");
    if (!tma && ((Tq + 63) / 64) * B * Hq > 0x7fffffff)
        return fail(FA_EUNSUPPORTED, "fp32 path: B*Hq*ceil(Tq/64) must be below 2^31");

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
    P.q_sb = qs[0], P.q_sh = qs[1], P.q_st = qs[2];
    P.k_sb = ks[0], P.k_sh = ks[1], P.k_st = ks[2];
    P.v_sb = vs[0], P.v_sh = vs[1], P.v_st = vs[2];
    P.o_sb = os[0], P.o_sh = os[1], P.o_st = os[2];
    P.vec16 = (d % 4 == 0) && strides_multiple(B, Hq, Tq, qs[0], qs[1], qs[2], 4) &&
              (!kv || (strides_multiple(B, Hkv, Tk, ks[0], ks[1], ks[2], 4) &&
                       strides_multiple(B, Hkv, Tk, vs[0], vs[1], vs[2], 4)));
    P.q_offset = (int)q_offset;
    P.causal = causal ? 1 : 0;
    // A window wider than every possible distance is no window.
    P.window = window <= 0 ? 0 : (window >= 2 * kMaxLen ? 0 : (int)window);
    P.scale = scale;
    P.scale_log2 = (float)((double)scale * 1.4426950408889634);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (noalloc && dtype == FA_DTYPE_BF16) {
        // The split-KV call of fa_fwd_splitkv with the library's static
        // scratch array as its workspace; calls that need none run as fa_fwd.
        const size_t need = fa::splitkv_workspace_bytes(P.B, P.Hkv, P.group, P.Tq, P.d);
        if (need > 0) {
            if (need > fa::kNoAllocScratchBytes)
                return fail(FA_EUNSUPPORTED,
                            "fa_fwd_splitkv_noalloc: this call needs %zu bytes of scratch, more than the %zu bytes "
                            "the library holds per GPU; use fa_fwd_splitkv with a workspace of that size",
                            need, fa::kNoAllocScratchBytes);
            const cudaError_t e = fa::launch_bf16_splitkv_noalloc(P, s);
            if (e != cudaSuccess) return fail(FA_ECUDA, "CUDA error: %s", cudaGetErrorString(e));
            return FA_OK;
        }
    }
    if (splitkv && dtype == FA_DTYPE_BF16) {
        const size_t need = fa::splitkv_workspace_bytes(P.B, P.Hkv, P.group, P.Tq, P.d);
        if (need > 0) {
            if (workspace == nullptr || workspace_bytes < need)
                return fail(FA_EINVAL, "fa_fwd_splitkv: the workspace needs %zu bytes (got %zu%s)", need,
                            workspace_bytes, workspace == nullptr ? ", NULL" : "");
            if (!aligned16(workspace)) return fail(FA_EINVAL, "fa_fwd_splitkv: the workspace must be 16-byte aligned");
            const cudaError_t e = fa::launch_bf16_splitkv(P, workspace, s);
            if (e != cudaSuccess) return fail(FA_ECUDA, "CUDA error: %s", cudaGetErrorString(e));
            return FA_OK;
        }
    }
    cudaError_t e = dtype == FA_DTYPE_F32      ? fa::launch_f32(P, s)
                    : dtype == FA_DTYPE_BF16   ? fa::launch_bf16(P, s)
                    : dtype == FA_DTYPE_F32_TC ? fa::launch_f32_tc(P, s)
                                               : fa::launch_fp8(P, s);
    if (e != cudaSuccess) return fail(FA_ECUDA, "CUDA error: %s", cudaGetErrorString(e));
    return FA_OK;
}

}  // namespace

extern "C" fa_status fa_splitkv_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t Tq, int64_t d,
                                                int dtype, size_t *bytes) {
    g_last_error[0] = '\0';
    if (bytes == nullptr) return fail(FA_EINVAL, "fa_splitkv_workspace_bytes: bytes is NULL");
    *bytes = 0;
    if (!known_dtype(dtype)) return fail(FA_EINVAL, "unknown dtype %d", dtype);
    if (B < 0 || Hq < 0 || Hkv < 0 || Tq < 0 || d < 0) return fail(FA_EINVAL, "negative size");
    if (Hkv == 0 ? Hq > 0 : (Hkv > Hq || Hq % Hkv != 0))
        return fail(FA_ESHAPE, "Hq=%lld is not a multiple of Hkv=%lld (or Hkv > Hq)", (long long)Hq,
                    (long long)Hkv);
    if (dtype != FA_DTYPE_BF16 || B == 0 || Hq == 0 || Tq == 0 || d == 0) return FA_OK;  // no workspace
    if (Tq >= kMaxLen || d > 128) return FA_OK;  // not a call fa_fwd_splitkv accepts
    if (B > 0x7fffffff / Hq) return fail(FA_EUNSUPPORTED, "B*Hq must be below 2^31");
    *bytes = fa::splitkv_workspace_bytes((int)B, (int)Hkv, (int)(Hq / Hkv), (int)Tq, (int)d);
    return FA_OK;
}

extern "C" fa_status fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                                    int64_t Hq, int64_t Hkv, int64_t Tq, int64_t Tk, int64_t d, float scale,
                                    int64_t q_offset, int causal, int64_t window, const float *sinks,
                                    const float *mask, int64_t mask_sb, int64_t mask_sh, int64_t mask_sq,
                                    int64_t mask_sk, void *workspace, size_t workspace_bytes, int dtype,
                                    void *stream) {
    // Contiguous [B, H, T, d], as in fa_fwd.
    const uint64_t uq = (uint64_t)(Tq < 0 ? 0 : Tq) * (uint64_t)(d < 0 ? 0 : d);
    const uint64_t uk = (uint64_t)(Tk < 0 ? 0 : Tk) * (uint64_t)(d < 0 ? 0 : d);
    const int64_t qs[3] = {(int64_t)(uq * (uint64_t)(Hq < 0 ? 0 : Hq)), (int64_t)uq, d},
                  ks[3] = {(int64_t)(uk * (uint64_t)(Hkv < 0 ? 0 : Hkv)), (int64_t)uk, d};
    return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, qs, ks, ks, qs, scale, q_offset, causal, window, sinks,
                    mask, mask_sb, mask_sh, mask_sq, mask_sk, dtype, stream, true, workspace, workspace_bytes);
}

static_assert(FA_SPLITKV_NOALLOC_MAX_SCRATCH == fa::kNoAllocScratchBytes, "the header states the array's size");

extern "C" fa_status fa_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                                            int64_t B, int64_t Hq, int64_t Hkv, int64_t Tq, int64_t Tk, int64_t d,
                                            float scale, int64_t q_offset, int causal, int64_t window,
                                            const float *sinks, const float *mask, int64_t mask_sb, int64_t mask_sh,
                                            int64_t mask_sq, int64_t mask_sk, int dtype, void *stream) {
    // Contiguous [B, H, T, d], as in fa_fwd.
    const uint64_t uq = (uint64_t)(Tq < 0 ? 0 : Tq) * (uint64_t)(d < 0 ? 0 : d);
    const uint64_t uk = (uint64_t)(Tk < 0 ? 0 : Tk) * (uint64_t)(d < 0 ? 0 : d);
    const int64_t qs[3] = {(int64_t)(uq * (uint64_t)(Hq < 0 ? 0 : Hq)), (int64_t)uq, d},
                  ks[3] = {(int64_t)(uk * (uint64_t)(Hkv < 0 ? 0 : Hkv)), (int64_t)uk, d};
    return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, qs, ks, ks, qs, scale, q_offset, causal, window, sinks,
                    mask, mask_sb, mask_sh, mask_sq, mask_sk, dtype, stream, false, nullptr, 0, true);
}

extern "C" fa_status fa_fwd_strided(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                                    int64_t Hq, int64_t Hkv, int64_t Tq, int64_t Tk, int64_t d, int64_t q_sb,
                                    int64_t q_sh, int64_t q_st, int64_t k_sb, int64_t k_sh, int64_t k_st,
                                    int64_t v_sb, int64_t v_sh, int64_t v_st, int64_t o_sb, int64_t o_sh,
                                    int64_t o_st, float scale, int64_t q_offset, int causal, int64_t window,
                                    const float *sinks, const float *mask, int64_t mask_sb, int64_t mask_sh,
                                    int64_t mask_sq, int64_t mask_sk, int dtype, void *stream) {
    const int64_t qs[3] = {q_sb, q_sh, q_st}, ks[3] = {k_sb, k_sh, k_st}, vs[3] = {v_sb, v_sh, v_st},
                  os[3] = {o_sb, o_sh, o_st};
    return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, qs, ks, vs, os, scale, q_offset, causal, window, sinks,
                    mask, mask_sb, mask_sh, mask_sq, mask_sk, dtype, stream);
}

extern "C" fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                            int64_t Hq, int64_t Hkv, int64_t Tq, int64_t Tk, int64_t d, float scale,
                            int64_t q_offset, int causal, int64_t window, const float *sinks, const float *mask,
                            int64_t mask_sb, int64_t mask_sh, int64_t mask_sq, int64_t mask_sk, int dtype,
                            void *stream) {
    // Contiguous [B, H, T, d]; products are checked for overflow in fwd_impl
    // through the element counts, so wrapped strides only reach it when those
    // counts are rejected first.
    const uint64_t uq = (uint64_t)(Tq < 0 ? 0 : Tq) * (uint64_t)(d < 0 ? 0 : d);
    const uint64_t uk = (uint64_t)(Tk < 0 ? 0 : Tk) * (uint64_t)(d < 0 ? 0 : d);
    const int64_t qs[3] = {(int64_t)(uq * (uint64_t)(Hq < 0 ? 0 : Hq)), (int64_t)uq, d},
                  ks[3] = {(int64_t)(uk * (uint64_t)(Hkv < 0 ? 0 : Hkv)), (int64_t)uk, d};
    return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, qs, ks, ks, qs, scale, q_offset, causal, window, sinks,
                    mask, mask_sb, mask_sh, mask_sq, mask_sk, dtype, stream);
}

extern "C" fa_status fa_fwd_paged(const void *q, const void *k_cache, const void *v_cache, void *o, float *lse,
                                  int64_t B, int64_t Hq, int64_t Hkv, int64_t Tq, int64_t d, const int32_t *seq_lens,
                                  int64_t max_seq_len, const int32_t *block_table, int64_t max_blocks,
                                  int64_t page_size, int64_t num_pages, float scale, int causal, int64_t window,
                                  const float *sinks, int dtype, void *stream) {
    g_last_error[0] = '\0';
    if (!known_dtype(dtype)) return fail(FA_EINVAL, "unknown dtype %d", dtype);
    if (B < 0 || Hq < 0 || Hkv < 0 || Tq < 0 || d < 0 || max_seq_len < 0 || max_blocks < 0 || page_size < 0 ||
        num_pages < 0)
        return fail(FA_EINVAL, "negative size");
    if (!std::isfinite(scale)) return fail(FA_EINVAL, "scale is not finite");
    if (Hkv == 0 ? Hq > 0 : (Hkv > Hq || Hq % Hkv != 0))
        return fail(FA_ESHAPE, "Hq=%lld is not a multiple of Hkv=%lld (or Hkv > Hq)", (long long)Hq,
                    (long long)Hkv);
    int64_t rows = 0, elems = 0, cache = 0;
    if (!mul_ok(B, Hq, rows) || !mul_ok(rows, Tq, rows) || !mul_ok(rows, d, elems) || !mul_ok(num_pages, page_size, cache) ||
        !mul_ok(cache, Hkv, cache) || !mul_ok(cache, d, cache) || elems > (std::numeric_limits<int64_t>::max() >> 3) ||
        cache > (std::numeric_limits<int64_t>::max() >> 3))
        return fail(FA_EINVAL, "element counts overflow");
    if (rows == 0) return FA_OK;
    if (!q || !o || !seq_lens) return fail(FA_EINVAL, "q, o or seq_lens is NULL");
    if (max_seq_len > 0 && (!k_cache || !v_cache || !block_table))
        return fail(FA_EINVAL, "k_cache, v_cache or block_table is NULL");
    if (dtype != FA_DTYPE_BF16) return fail(FA_EUNSUPPORTED, "the paged path is bf16 only");
    if (d % 8 != 0 || d == 0 || d > 128)
        return fail(FA_EUNSUPPORTED, "bf16 path supports d a multiple of 8 up to 128 (got %lld)", (long long)d);
    if (Hq / Hkv * Tq > 128)
        return fail(FA_EUNSUPPORTED, "paged path: (Hq / Hkv) * Tq must be at most 128 (decode steps)");
    if (max_seq_len > 0) {
        if (page_size < 8 || (page_size <= 128 ? (128 % page_size != 0) : (page_size % 128 != 0)))
            return fail(FA_EUNSUPPORTED, "page_size must divide 128 (and be >= 8) or be a multiple of 128");
        int64_t capacity = 0;  // keys the table can address (a product too large for int64 addresses them all)
        if (max_blocks == 0 || (mul_ok(max_blocks, page_size, capacity) && max_seq_len > capacity))
            return fail(FA_EINVAL, "max_seq_len exceeds max_blocks * page_size");
        if (num_pages == 0 || num_pages > 0x7fffffff || max_blocks > 0x7fffffff || page_size > 0x7fffffff)
            return fail(FA_EUNSUPPORTED, "num_pages and max_blocks must be in [1, 2^31), page_size below 2^31");
    }
    if (max_seq_len >= kMaxLen || Tq >= kMaxLen) return fail(FA_EUNSUPPORTED, "lengths must be below 2^30");
    if (B * Hq >= (int64_t(1) << 24)) return fail(FA_EUNSUPPORTED, "B*Hq must be below 2^24");
    if (!aligned16(q) || !aligned16(o) || (max_seq_len > 0 && (!aligned16(k_cache) || !aligned16(v_cache))))
        return fail(FA_EUNSUPPORTED, "q, o and the caches must be 16-byte aligned");

    fa::Params P;
    std::memset(&P, 0, sizeof P);
    P.q = q;
    P.k = k_cache;
    P.v = v_cache;
    P.o = o;
    P.lse = lse;
    P.sinks = sinks;
    P.B = (int)B;
    P.Hq = (int)Hq;
    P.Hkv = (int)Hkv;
    P.Tq = (int)Tq;
    P.Tk = (int)max_seq_len;
    P.d = (int)d;
    P.group = (int)(Hq / Hkv);
    P.splits = 1;
    P.q_sb = Hq * Tq * d, P.q_sh = Tq * d, P.q_st = d;
    P.o_sb = P.q_sb, P.o_sh = P.q_sh, P.o_st = P.q_st;
    P.causal = causal ? 1 : 0;
    P.window = window <= 0 ? 0 : (window >= 2 * kMaxLen ? 0 : (int)window);
    P.scale = scale;
    P.scale_log2 = (float)((double)scale * 1.4426950408889634);
    P.seq_lens = seq_lens;
    P.block_table = block_table;
    P.max_blocks = (int)max_blocks;
    P.page_size = (int)(page_size > 0 ? page_size : 128);
    P.num_pages = (int)(num_pages > 0 ? num_pages : 1);
    P.max_seq_len = (int)max_seq_len;
    cudaError_t e = fa::launch_bf16_paged(P, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(FA_ECUDA, "CUDA error: %s", cudaGetErrorString(e));
    return FA_OK;
}

extern "C" fa_status fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse, int64_t B,
                                   int64_t Hq, int64_t Hkv, int64_t d, const int32_t *cu_seqlens_q,
                                   const int32_t *cu_seqlens_k, int64_t total_q, int64_t total_k,
                                   int64_t max_seqlen_q, int64_t max_seqlen_k, int64_t q_sh, int64_t q_st,
                                   int64_t k_sh, int64_t k_st, int64_t v_sh, int64_t v_st, int64_t o_sh,
                                   int64_t o_st, float scale, int causal, int64_t window, const float *sinks,
                                   int dtype, void *stream) {
    g_last_error[0] = '\0';
    if (!known_dtype(dtype)) return fail(FA_EINVAL, "unknown dtype %d", dtype);
    if (B < 0 || Hq < 0 || Hkv < 0 || d < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0)
        return fail(FA_EINVAL, "negative size");
    if (!std::isfinite(scale)) return fail(FA_EINVAL, "scale is not finite");
    if (Hkv == 0 ? Hq > 0 : (Hkv > Hq || Hq % Hkv != 0))
        return fail(FA_ESHAPE, "Hq=%lld is not a multiple of Hkv=%lld (or Hkv > Hq)", (long long)Hq,
                    (long long)Hkv);
    int64_t span = 0;
    if (!layout_ok(1, Hq, total_q, d, 0, q_sh, q_st, false, span) ||
        !layout_ok(1, Hkv, total_k, d, 0, k_sh, k_st, false, span) ||
        !layout_ok(1, Hkv, total_k, d, 0, v_sh, v_st, false, span))
        return fail(FA_EINVAL, "q, k or v strides are negative or their extents overflow");
    if (!layout_ok(1, Hq, total_q, d, 0, o_sh, o_st, true, span))
        return fail(FA_EINVAL, "o strides are negative or make two output rows overlap");
    if (B == 0 || Hq == 0 || total_q == 0 || max_seqlen_q == 0) return FA_OK;  // no query row
    if (!q || !o || !cu_seqlens_q || !cu_seqlens_k) return fail(FA_EINVAL, "q, o or a cu_seqlens table is NULL");
    if (total_k > 0 && (!k || !v)) return fail(FA_EINVAL, "k or v is NULL with total_k > 0");
    if (dtype == FA_DTYPE_F32_TC)
        return fail(FA_EUNSUPPORTED, "the varlen path is fp32 (SIMT), bf16 or e4m3 only");
    if (d == 0 || (d & 1)) return fail(FA_EUNSUPPORTED, "d=%lld: d must be even and positive", (long long)d);
    if (dtype == FA_DTYPE_F32 && d > 256)
        return fail(FA_EUNSUPPORTED, "fp32 path supports d <= 256 (got %lld)", (long long)d);
    if (dtype == FA_DTYPE_FP8_E4M3 && (d % 16 != 0 || d > 128))
        return fail(FA_EUNSUPPORTED, "e4m3 path supports d a multiple of 16 up to 128 (got %lld)", (long long)d);
    if (dtype == FA_DTYPE_BF16 && (d % 8 != 0 || d > 128))
        return fail(FA_EUNSUPPORTED, "bf16 path supports d a multiple of 8 up to 128 (got %lld)", (long long)d);
    if (total_q >= kMaxLen || total_k >= kMaxLen || max_seqlen_q > total_q)
        return fail(FA_EUNSUPPORTED, "totals must be below 2^30 and max_seqlen_q <= total_q");
    int64_t bh = 0;
    if (B >= (int64_t(1) << 24) || !mul_ok(B, Hq, bh) || bh >= (int64_t(1) << 31))
        return fail(FA_EUNSUPPORTED, "too many sequences");
    // Query tiles of every (sequence, head) as 31-bit block or unit numbers:
    // 128 rows on the tensor cores, 64 on SIMT.
    const int64_t tile_rows = dtype == FA_DTYPE_F32 ? 64 : 128;
    if (((max_seqlen_q + tile_rows - 1) / tile_rows) * bh > 0x7fffffff)
        return fail(FA_EUNSUPPORTED, "B*Hq*ceil(max_seqlen_q/%lld) must be below 2^31", (long long)tile_rows);
    if (!aligned16(q) || !aligned16(o) || (total_k > 0 && (!aligned16(k) || !aligned16(v))))
        return fail(FA_EUNSUPPORTED, "q, k, v and o must be 16-byte aligned");
    // Tensor maps: 16-byte stride multiples (o is bf16 with e4m3 inputs).
    const bool tma = dtype != FA_DTYPE_F32;
    const int64_t in_bytes = dtype == FA_DTYPE_FP8_E4M3 ? 1 : (dtype == FA_DTYPE_BF16 ? 2 : 4);
    const int64_t m = tma ? 16 / in_bytes : 2, mo = tma ? 8 : 2;
    const bool kv = total_k > 0;
    if (!strides_multiple(1, Hq, total_q, 0, q_sh, q_st, m) || !strides_multiple(1, Hq, total_q, 0, o_sh, o_st, mo) ||
        (kv && (!strides_multiple(1, Hkv, total_k, 0, k_sh, k_st, m) ||
                !strides_multiple(1, Hkv, total_k, 0, v_sh, v_st, m))))
        return fail(FA_EUNSUPPORTED, "strides must be multiples of %lld elements for this dtype", (long long)m);
    if (tma) {
        const int64_t st[8] = {q_sh, q_st, k_sh, k_st, v_sh, v_st, o_sh, o_st};
        const int64_t ext[8] = {Hq, total_q, Hkv, total_k, Hkv, total_k, Hq, total_q};
        for (int i = 0; i < 8; ++i) {
            const int64_t lim = ((int64_t(1) << 40) / (i >= 6 ? 2 : in_bytes)) - 1;  // elements; o is bf16
            if (st[i] > lim) return fail(FA_EUNSUPPORTED, "a stride reaches 2^40 bytes");
            if (ext[i] > 1 && st[i] <= 0)
                return fail(FA_EUNSUPPORTED, "strides must be positive for this dtype (tensor maps)");
        }
    }

    fa::Params P;
    std::memset(&P, 0, sizeof P);
    P.q = q;
    P.k = k;
    P.v = v;
    P.o = o;
    P.lse = lse;
    P.sinks = sinks;
    P.B = (int)B;
    P.Hq = (int)Hq;
    P.Hkv = (int)Hkv;
    P.Tq = (int)max_seqlen_q;
    P.Tk = (int)(max_seqlen_k < kMaxLen ? max_seqlen_k : kMaxLen - 1);
    P.d = (int)d;
    P.group = (int)(Hq / Hkv);
    P.splits = 1;
    P.q_sh = q_sh, P.q_st = q_st, P.k_sh = k_sh, P.k_st = k_st;
    P.v_sh = v_sh, P.v_st = v_st, P.o_sh = o_sh, P.o_st = o_st;
    P.vec16 = (d % 4 == 0) && strides_multiple(1, Hq, total_q, 0, q_sh, q_st, 4) &&
              (!kv || (strides_multiple(1, Hkv, total_k, 0, k_sh, k_st, 4) &&
                       strides_multiple(1, Hkv, total_k, 0, v_sh, v_st, 4)));
    P.causal = causal ? 1 : 0;
    P.window = window <= 0 ? 0 : (window >= 2 * kMaxLen ? 0 : (int)window);
    P.scale = scale;
    P.scale_log2 = (float)((double)scale * 1.4426950408889634);
    P.cu_q = cu_seqlens_q;
    P.cu_k = cu_seqlens_k;
    P.total_q = (int)total_q;
    P.total_k = (int)total_k;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = dtype == FA_DTYPE_F32    ? fa::launch_f32_varlen(P, s)
                    : dtype == FA_DTYPE_BF16 ? fa::launch_bf16_varlen(P, s)
                                             : fa::launch_fp8_varlen(P, s);
    if (e != cudaSuccess) return fail(FA_ECUDA, "CUDA error: %s", cudaGetErrorString(e));
    return FA_OK;
}
