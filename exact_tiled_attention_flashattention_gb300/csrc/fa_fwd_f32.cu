// fa_fwd_f32.cu -- fp32 exact tiled attention on the SIMT cores (FFMA).
//
// One CTA of 256 threads owns one (batch, query head, 64-row query tile) and
// walks the key tiles any of its rows can see, 64 keys at a time, under the
// online softmax of "FlashAttention forward in C" (section 2.2): per row a
// running max m, denominator l and output accumulator, rescaled by
// 2^(m_old - m_new) when the max grows.  Scores live in the log2 domain
// (scale * log2 e folded into one multiply) so every exponential is one ex2.
//
// Key tiles sit at absolute positions [64t, 64t + 64) and a row adds its keys
// in increasing j within a tile, so a row's bits do not depend on the query
// tile, the chunking through q_offset or the batch ("FlashAttention forward in
// C", section 2.4).  A tile that a row cannot see leaves that row's state bit
// for bit unchanged (alpha = 1, p = 0), so rows need no per-row skip branch.
//
// The rescale guard follows "Fused attention and softmax: fast and exact"
// (the exact definition, steps 2 and 5): shift = 0 while the max is -inf and
// alpha = 1 when the max did not move, which avoids -inf - (-inf).
//
// Thread layout: tx = tid % 16, ty = tid / 16.  S: thread (ty, tx) owns rows
// 4ty..4ty+3 and keys tx + 16b (b < 4); row reductions are 16-lane shuffles.
// O: the same rows, columns 2tx + 32m (float2 pairs, m < DT/32).
// Memory: K, V tiles staged by cp.async (zero-filled past Tk and past d), V
// in flight while S and the softmax run, the next K in flight during P.V.
#include <cmath>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kBr = 64;
constexpr int kBc = 64;
constexpr int kThreads = 256;
constexpr int kPLd = kBr + 4;  // P stored transposed: Pt[key][row]
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, int src_bytes) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes));
}

__device__ __forceinline__ void cp_async8(void *smem, const void *gmem, int src_bytes) {
    const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(s), "l"(gmem), "r"(src_bytes));
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }

// Programmatic dependent launch: wait for the previous grid in the stream
// (its writes visible), and let the next grid start launching.
__device__ __forceinline__ void grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Stage rows [row0, row0 + 64) of a [T, d] fp32 matrix with row stride `ld`
// (elements) into dst[64][DT + 4], zero-filling rows outside [0, T) and
// columns [d, DT).  vec16: every row starts on a 16-byte boundary and d is a
// multiple of 4 (16-byte copies); otherwise rows start on 8-byte boundaries.
template <int DT>
__device__ __forceinline__ void stage_rows(float *dst, const float *src, int row0, int T, int d, int64_t ld,
                                           bool vec16) {
    constexpr int LD = DT + 4;
    if (vec16) {
        constexpr int kChunks = DT / 4;
#pragma unroll 4
        for (int c = threadIdx.x; c < kBr * kChunks; c += kThreads) {
            const int r = c / kChunks, col = (c % kChunks) * 4;
            const int row = row0 + r;
            const bool ok = row < T && col < d;
            const float *g = ok ? src + (int64_t)row * ld + col : src;
            cp_async16(dst + r * LD + col, g, ok ? 16 : 0);
        }
    } else {
        constexpr int kChunks = DT / 2;
#pragma unroll 4
        for (int c = threadIdx.x; c < kBr * kChunks; c += kThreads) {
            const int r = c / kChunks, col = (c % kChunks) * 2;
            const int row = row0 + r;
            const bool ok = row < T && col < d;
            const float *g = ok ? src + (int64_t)row * ld + col : src;
            cp_async8(dst + r * LD + col, g, ok ? 8 : 0);
        }
    }
}

// Registers: at d >= 128 shared memory holds one CTA per SM, so the kernel
// declares one resident CTA and the compiler may use what it needs (no
// spills); smaller d keeps the compiler's own choice.
template <int DT, bool VARLEN>
__global__ void __launch_bounds__(kThreads, DT >= 128 ? 1 : 0) fa_fwd_f32_kernel(const Params P) {
    constexpr int LD = DT + 4;
    constexpr int NC = DT / 32;  // float2 column pairs per thread
    extern __shared__ float4 smem_f4[];
    float *Qs = reinterpret_cast<float *>(smem_f4);
    float *Ks = Qs + kBr * LD;
    float *Vs = Ks + kBc * LD;
    float *Pt = Vs + kBc * LD;

    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int BH = P.B * P.Hq;
    const int nqt = (P.Tq + kBr - 1) / kBr;
    // Heaviest query tiles first: under a causal rule the last tiles see most keys.
    const int qt = nqt - 1 - (int)(blockIdx.x / BH);
    const int bh = (int)(blockIdx.x % BH);
    const int b = bh / P.Hq, h = bh % P.Hq;
    const int g = h / P.group;
    const int r0 = qt * kBr;

    // The sequence's rows, keys and the position of its row 0: the call's,
    // or (variable-length batch) sequence b's, whose queries are its last
    // positions, with its rows and keys starting at tensor rows qrow / krow.
    int Tq = P.Tq, Tk = P.Tk, qoff = P.q_offset;
    int64_t qrow = 0, krow = 0;
    // Everything above reads kernel parameters only and runs while the
    // previous grid finishes; the call's tensors (and, in a variable-length
    // batch, its offsets) are read after the dependency wait.
    grid_wait();
    grid_launch_next();
    if constexpr (VARLEN) {
        // offsets clamped into the tensors: a malformed table cannot reach outside them
        const int q0 = min(max(__ldg(P.cu_q + b), 0), P.total_q), k0 = min(max(__ldg(P.cu_k + b), 0), P.total_k);
        Tq = min(max(__ldg(P.cu_q + b + 1), q0), P.total_q) - q0;
        Tk = min(max(__ldg(P.cu_k + b + 1), k0), P.total_k) - k0;
        qoff = Tk - Tq;
        qrow = q0;
        krow = k0;
        if (r0 >= Tq) return;  // a tile past the sequence's rows (the whole block leaves)
    }
    const float *qh = static_cast<const float *>(P.q) + (VARLEN ? 0 : b * P.q_sb) + h * P.q_sh + qrow * P.q_st;
    const float *kh = static_cast<const float *>(P.k) + (VARLEN ? 0 : b * P.k_sb) + g * P.k_sh + krow * P.k_st;
    const float *vh = static_cast<const float *>(P.v) + (VARLEN ? 0 : b * P.v_sb) + g * P.v_sh + krow * P.v_st;

    // Key tiles any row of this query tile can see.
    const int64_t p_first = (int64_t)qoff + r0;
    const int64_t p_last = (int64_t)qoff + min(r0 + kBr, Tq) - 1;
    int64_t lo_a, hi_a, lo_b, hi_b;
    visible_range_tk(P, Tk, p_first, lo_a, hi_a);
    visible_range_tk(P, Tk, p_last, lo_b, hi_b);
    const int64_t klo = lo_a, khi = hi_b > hi_a ? hi_b : hi_a;
    const int t_begin = (int)(klo / kBc);
    const int t_end = khi > klo ? (int)((khi + kBc - 1) / kBc) : t_begin;

    // Per-row state, log2 domain.  A sink starts the row at m = z log2 e, l = 1.
    float m[4], l[4];
    float2 acc[4][NC];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const bool sink = P.sinks != nullptr;
        m[a] = sink ? __ldg(P.sinks + h) * kLog2e : -INFINITY;
        l[a] = sink ? 1.f : 0.f;
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[a][c] = make_float2(0.f, 0.f);
    }

    stage_rows<DT>(Qs, qh, r0, Tq, P.d, P.q_st, P.vec16 != 0);
    if (t_begin < t_end) stage_rows<DT>(Ks, kh, t_begin * kBc, Tk, P.d, P.k_st, P.vec16 != 0);
    cp_async_commit();

    for (int t = t_begin; t < t_end; ++t) {
        cp_async_wait<0>();
        __syncthreads();  // Q and K_t landed; every thread finished the previous P.V
        stage_rows<DT>(Vs, vh, t * kBc, Tk, P.d, P.v_st, P.vec16 != 0);
        cp_async_commit();

        // S = Q K_t^T for rows 4ty+a, keys tx+16b.
        float s[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) s[a][bb] = 0.f;
#pragma unroll 4
        for (int x = 0; x < DT; x += 4) {
            float4 qa[4], kb[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) qa[a] = *reinterpret_cast<const float4 *>(Qs + (4 * ty + a) * LD + x);
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) kb[bb] = *reinterpret_cast<const float4 *>(Ks + (tx + 16 * bb) * LD + x);
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) {
                    float r = s[a][bb];
                    r = fmaf(qa[a].x, kb[bb].x, r);
                    r = fmaf(qa[a].y, kb[bb].y, r);
                    r = fmaf(qa[a].z, kb[bb].z, r);
                    r = fmaf(qa[a].w, kb[bb].w, r);
                    s[a][bb] = r;
                }
        }

        // Scale, additive mask, visibility.  Interior tiles (every key visible
        // to every row of the tile) skip the per-element rule.
        const int j0 = t * kBc;
        const bool full = (j0 + kBc <= Tk) && (!P.causal || (int64_t)(j0 + kBc - 1) <= p_first) &&
                          (P.window <= 0 || (int64_t)j0 > p_last - P.window);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = r0 + 4 * ty + a;
            const int64_t p = (int64_t)qoff + i;
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
                const int j = j0 + tx + 16 * bb;
                float v = s[a][bb] * P.scale_log2;
                if (!VARLEN && P.mask != nullptr && i < Tq && j < Tk)
                    v = fmaf(__ldg(P.mask + b * P.msb + h * P.msh + (int64_t)i * P.msq + (int64_t)j * P.msk),
                             kLog2e, v);
                if (!full) {
                    const bool vis = j < Tk && (!P.causal || (int64_t)j <= p) &&
                                     (P.window <= 0 || (int64_t)j > p - P.window);
                    if (!vis) v = -INFINITY;
                }
                s[a][bb] = v;
            }
        }

        // Online softmax update per row.
        float alpha[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            float bm = fmaxf(fmaxf(s[a][0], s[a][1]), fmaxf(s[a][2], s[a][3]));
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
            const float mnew = fmaxf(m[a], bm);
            const float shift = (mnew == -INFINITY) ? 0.f : mnew;
            alpha[a] = (m[a] == shift) ? 1.f : ex2(m[a] - shift);
            float rs = 0.f;
#pragma unroll
            for (int bb = 0; bb < 4; ++bb) {
                const float pj = ex2(s[a][bb] - shift);
                s[a][bb] = pj;
                rs += pj;
            }
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
            l[a] = fmaf(alpha[a], l[a], rs);
            m[a] = mnew;
        }
#pragma unroll
        for (int bb = 0; bb < 4; ++bb)
            *reinterpret_cast<float4 *>(Pt + (tx + 16 * bb) * kPLd + 4 * ty) =
                make_float4(s[0][bb], s[1][bb], s[2][bb], s[3][bb]);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                acc[a][c].x *= alpha[a];
                acc[a][c].y *= alpha[a];
            }

        __syncthreads();  // Pt complete; every thread done with Ks
        if (t + 1 < t_end) {
            stage_rows<DT>(Ks, kh, (t + 1) * kBc, Tk, P.d, P.k_st, P.vec16 != 0);
            cp_async_commit();
            cp_async_wait<1>();  // V_t landed; K_{t+1} may still be in flight
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();

        // O += P V_t, keys in increasing order.
#pragma unroll 4
        for (int j = 0; j < kBc; ++j) {
            const float4 pr = *reinterpret_cast<const float4 *>(Pt + j * kPLd + 4 * ty);
            const float pa[4] = {pr.x, pr.y, pr.z, pr.w};
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const float2 vv = *reinterpret_cast<const float2 *>(Vs + j * LD + 2 * tx + 32 * c);
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    acc[a][c].x = fmaf(pa[a], vv.x, acc[a][c].x);
                    acc[a][c].y = fmaf(pa[a], vv.y, acc[a][c].y);
                }
            }
        }
    }
    cp_async_wait<0>();

    // Epilogue: o = acc / l; lse = (m + log2 l) ln 2; empty rows give 0 and -inf.
    float *oh = static_cast<float *>(P.o) + (VARLEN ? 0 : b * P.o_sb) + h * P.o_sh + qrow * P.o_st;
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int i = r0 + 4 * ty + a;
        if (i >= Tq) continue;
        const float inv = l[a] > 0.f ? 1.f / l[a] : 0.f;
        float *orow = oh + (int64_t)i * P.o_st;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const int col = 2 * tx + 32 * c;
            if (col < P.d) *reinterpret_cast<float2 *>(orow + col) = make_float2(acc[a][c].x * inv, acc[a][c].y * inv);
        }
        if (tx == 0 && P.lse != nullptr)
            P.lse[VARLEN ? (int64_t)h * P.total_q + qrow + i : (int64_t)bh * P.Tq + i] =
                l[a] > 0.f ? (m[a] + log2f(l[a])) * kLn2 : -INFINITY;
    }
}

template <int DT, bool VARLEN>
cudaError_t launch_dt(const Params &P, cudaStream_t stream) {
    constexpr int LD = DT + 4;
    const size_t smem = (size_t)(kBr * LD + 2 * kBc * LD + kBc * kPLd) * sizeof(float);
    static DeviceOnce configured;  // one attribute call per instantiation and device
    int dev = -1;
    if (!configured.done(dev)) {
        if (dev < 0) return cudaErrorInvalidDevice;
        cudaError_t e = cudaFuncSetAttribute(fa_fwd_f32_kernel<DT, VARLEN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        configured.mark(dev);
    }
    const int nqt = (P.Tq + kBr - 1) / kBr;
    const unsigned grid = (unsigned)nqt * (unsigned)(P.B * P.Hq);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fa_fwd_f32_kernel<DT, VARLEN>, P);
}

}  // namespace

template <bool VARLEN>
cudaError_t launch_f32_v(const Params &P, cudaStream_t stream) {
    if (P.d <= 64) return launch_dt<64, VARLEN>(P, stream);
    if (P.d <= 96) return launch_dt<96, VARLEN>(P, stream);
    if (P.d <= 128) return launch_dt<128, VARLEN>(P, stream);
    return launch_dt<256, VARLEN>(P, stream);
}

cudaError_t launch_f32(const Params &P, cudaStream_t stream) { return launch_f32_v<false>(P, stream); }

cudaError_t launch_f32_varlen(const Params &P, cudaStream_t stream) { return launch_f32_v<true>(P, stream); }

}  // namespace fa
