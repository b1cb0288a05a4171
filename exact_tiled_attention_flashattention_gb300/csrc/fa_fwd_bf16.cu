// fa_fwd_bf16.cu -- bf16 exact tiled attention on the tcgen05 tensor cores.
//
// One CTA owns one (batch, query head, 128-row query tile).  The score tile
// S = Q K_t^T (128 x 128, fp32) and the output accumulator O (128 x d, fp32)
// live in tensor memory; Q, K_t and V_t are staged in shared memory by TMA
// with the 128-byte swizzle that tcgen05.mma reads directly.  Each query row
// keeps a running max m and denominator l in registers and the online softmax
// of "FlashAttention forward in C" (section 2.2) rescales O in tensor memory
// by 2^(m_old - m_new) when the max grows.  P = 2^(s - m) is rounded to bf16
// and written back to tensor memory, where it is the A operand of O += P V_t.
//
// Warp roles (192 threads):
//   warps 0-3  softmax: thread t owns query row t = tensor-memory lane t;
//              scale, mask, row max, exponentials, P, O rescale, epilogue
//   warp 4     TMA producer: Q once, then K_t / V_t into a 2-stage ring
//   warp 5     MMA issuer (one lane) and tensor-memory owner
// The issuer runs one tile ahead: S_{t+1} = Q K_{t+1}^T is computed (into the
// second S buffer) while the softmax warps work on S_t, then O += P_t V_t.
//
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O [256, 256+d),
// P [384, 448) as bf16 pairs.
//
// Key tiles sit at absolute positions [128t, 128t + 128); keys a row cannot
// see get p = 0 and leave its m, l and O unchanged, so a row's bits do not
// depend on its query tile or on chunking through q_offset ("FlashAttention
// forward in C", section 2.4).  The rescale guard follows "Fused attention
// and softmax: fast and exact" (the exact definition, steps 2 and 5).
//
// Every mbarrier wait is bounded (two seconds of wall time); a wait that runs
// out sets a CTA-wide abort flag and the device watchdog word, all roles leave
// their loops, in-flight copies and MMAs are drained with bounded waits, and
// tensor memory is released before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "fa_internal.h"
#include "sm100_ptx.cuh"

namespace fa {

__device__ unsigned int g_watchdog = 0;

namespace {

using namespace sm100;

constexpr int kBM = 128;  // query rows per tile = tensor-memory lanes
constexpr int kBN = 128;  // keys per tile
constexpr int kStages = 2;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColP = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kSwRowBytes = 128;  // one swizzled row: 64 bf16

template <int D>
struct SmemLayout {
    static constexpr int kBoxes = D / 64;                       // 64-column TMA boxes per tile
    static constexpr uint32_t kQBytes = kBM * D * 2;
    static constexpr uint32_t kKVBytes = kBN * D * 2;
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kQ + kQBytes;
    static constexpr uint32_t kV = kK + kStages * kKVBytes;
    static constexpr uint32_t kBar = kV + kStages * kKVBytes;  // barriers after the tiles
    static constexpr uint32_t kTotal = kBar + 256;
};

struct Barriers {
    uint64_t q_full;
    uint64_t k_full[kStages];
    uint64_t v_full[kStages];
    uint64_t kv_empty[kStages];
    uint64_t s_full[2];
    uint64_t s_free[2];
    uint64_t p_full;
    uint64_t o_ready;
    uint64_t mma_drain;
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const Params P) {
    using L = SmemLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Barriers &bar = *reinterpret_cast<Barriers *>(smem + L::kBar);
    volatile int *abort = &bar.abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Work unit: heaviest query tiles first (under a causal rule the last
    // tiles see the most keys).
    const int BH = P.B * P.Hq;
    const int nqt = (P.Tq + kBM - 1) / kBM;
    const int qt = nqt - 1 - (int)(blockIdx.x / BH);
    const int bh = (int)(blockIdx.x % BH);
    const int b = bh / P.Hq, h = bh % P.Hq, g = h / P.group;
    const int r0 = qt * kBM;
    const int64_t p_first = (int64_t)P.q_offset + r0;
    const int64_t p_last = (int64_t)P.q_offset + min(r0 + kBM, P.Tq) - 1;
    int64_t lo_a, hi_a, lo_b, hi_b;
    visible_range(P, p_first, lo_a, hi_a);
    visible_range(P, p_last, lo_b, hi_b);
    const int64_t klo = lo_a, khi = hi_b > hi_a ? hi_b : hi_a;
    const int t_begin = (int)(klo / kBN);
    const int n_tiles = khi > klo ? (int)((khi + kBN - 1) / kBN) - t_begin : 0;

    if (threadIdx.x == 0) {
        mbar_init(&bar.q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bar.k_full[s], 1);
            mbar_init(&bar.v_full[s], 1);
            mbar_init(&bar.kv_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar.s_full[s], 1);
            mbar_init(&bar.s_free[s], kBM);
        }
        mbar_init(&bar.p_full, kBM);
        mbar_init(&bar.o_ready, 1);
        mbar_init(&bar.mma_drain, 1);
        bar.abort = 0;
        mbar_init_fence();
    }
    if (warp == 5) {
        tmem_alloc(&bar.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = bar.tmem_base;

    if (warp == 4) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0 && n_tiles > 0) {
            const int kv_head = b * P.Hkv + g;
            mbar_arrive_expect_tx(&bar.q_full, L::kQBytes);
#pragma unroll
            for (int c = 0; c < L::kBoxes; ++c)
                tma_load_3d(smem + L::kQ + c * (kBM * kSwRowBytes), &tmQ, &bar.q_full, c * 64, r0, bh);
            int issued[kStages] = {};
            for (int jj = 0; jj < n_tiles; ++jj) {
                const int st = jj % kStages, u = jj / kStages;
                if (u > 0 && !mbar_wait(&bar.kv_empty[st], (u - 1) & 1, abort)) break;
                const int key0 = (t_begin + jj) * kBN;
                mbar_arrive_expect_tx(&bar.k_full[st], L::kKVBytes);
#pragma unroll
                for (int c = 0; c < L::kBoxes; ++c)
                    tma_load_3d(smem + L::kK + st * L::kKVBytes + c * (kBN * kSwRowBytes), &tmK, &bar.k_full[st],
                                c * 64, key0, kv_head);
                mbar_arrive_expect_tx(&bar.v_full[st], L::kKVBytes);
#pragma unroll
                for (int c = 0; c < L::kBoxes; ++c)
                    tma_load_3d(smem + L::kV + st * L::kKVBytes + c * (kBN * kSwRowBytes), &tmV, &bar.v_full[st],
                                c * 64, key0, kv_head);
                ++issued[st];
            }
            if (*abort) {
                // Drain: let every copy this thread issued land before the
                // CTA (and its shared memory) goes away.
                int never = 0;
                mbar_wait(&bar.q_full, 0, &never, 200000000ull);
                for (int s = 0; s < kStages; ++s)
                    if (issued[s] > 0) {
                        mbar_wait(&bar.k_full[s], (issued[s] - 1) & 1, &never, 200000000ull);
                        mbar_wait(&bar.v_full[s], (issued[s] - 1) & 1, &never, 200000000ull);
                    }
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0 && n_tiles > 0) {
            constexpr uint32_t kIdS = idesc_bf16_f32(kBM, kBN, 0, 0);  // Q, K both K-major
            constexpr uint32_t kIdO = idesc_bf16_f32(kBM, D, 0, 1);    // P from TMEM, V MN-major
            const uint32_t q_addr = smem_u32(smem + L::kQ);
            if (mbar_wait(&bar.q_full, 0, abort)) {
                for (int jj = 0; jj <= n_tiles; ++jj) {
                    if (jj < n_tiles) {
                        const int st = jj % kStages, sb = jj & 1;
                        if (!mbar_wait(&bar.k_full[st], (jj / kStages) & 1, abort)) break;
                        if (jj >= 2 && !mbar_wait(&bar.s_free[sb], ((jj - 2) >> 1) & 1, abort)) break;
                        tc_fence_after();
                        const uint32_t k_addr = smem_u32(smem + L::kK + st * L::kKVBytes);
                        const uint32_t d_tmem = tbase + (sb ? kColS1 : kColS0);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = (kk >> 2) * (kBM * kSwRowBytes) + (kk & 3) * 32;
                            const uint64_t a = smem_desc_sw128(q_addr + off, 16, 1024);
                            const uint64_t bd = smem_desc_sw128(k_addr + (kk >> 2) * (kBN * kSwRowBytes) + (kk & 3) * 32,
                                                                16, 1024);
                            mma_ss(d_tmem, a, bd, kIdS, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(&bar.s_full[sb]);
                    }
                    if (jj >= 1) {
                        const int pj = jj - 1, st = pj % kStages;
                        if (!mbar_wait(&bar.p_full, pj & 1, abort)) break;
                        if (!mbar_wait(&bar.v_full[st], (pj / kStages) & 1, abort)) break;
                        tc_fence_after();
                        const uint32_t v_addr = smem_u32(smem + L::kV + st * L::kKVBytes);
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk) {
                            // 16 keys = two 8-row swizzle atoms; the next 64
                            // value columns sit one TMA box further on.
                            const uint64_t bd = smem_desc_sw128(v_addr + kk * 16 * kSwRowBytes,
                                                                kBN * kSwRowBytes, 1024);
                            mma_ts(tbase + kColO, tbase + kColP + kk * 8, bd, kIdO, (pj > 0 || kk > 0) ? 1u : 0u);
                        }
                        mma_commit(&bar.o_ready);
                        mma_commit(&bar.kv_empty[st]);
                    }
                }
            }
            // Every MMA issued above completes before tensor memory is freed.
            mma_commit(&bar.mma_drain);
            int never = 0;
            mbar_wait(&bar.mma_drain, 0, &never, 200000000ull);
        }
    } else {
        // ------------------------------------------------- softmax warps 0-3
        const int row = threadIdx.x;  // query row within the tile = TMEM lane
        const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
        const int i = r0 + row;
        const int64_t p = (int64_t)P.q_offset + i;
        const bool has_sink = P.sinks != nullptr;
        float m = has_sink ? __ldg(P.sinks + h) * kLog2e : -INFINITY;
        float l = has_sink ? 1.f : 0.f;
        const float *mrow = P.mask ? P.mask + b * P.msb + h * P.msh + (int64_t)i * P.msq : nullptr;
        bool ok = true;

        for (int jj = 0; jj < n_tiles && ok; ++jj) {
            const int sb = jj & 1;
            // warp-uniform outcome: the tcgen05.ld/st below are warp-collective
            if (!__all_sync(0xffffffffu, mbar_wait(&bar.s_full[sb], (jj >> 1) & 1, abort))) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[kBN];
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) {
                uint32_t r[32];
                tmem_load32(lane_addr + (sb ? kColS1 : kColS0) + c * 32, r);
#pragma unroll
                for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(r[e]);
            }
            tc_fence_before();
            mbar_arrive(&bar.s_free[sb]);

            const int j0 = (t_begin + jj) * kBN;
            const bool full = (j0 + kBN <= P.Tk) && (!P.causal || (int64_t)(j0 + kBN - 1) <= p_first) &&
                              (P.window <= 0 || (int64_t)j0 > p_last - P.window);
            float bm = -INFINITY;
#pragma unroll
            for (int e = 0; e < kBN; ++e) {
                float v = s[e] * P.scale_log2;
                if (mrow != nullptr && i < P.Tq && j0 + e < P.Tk)
                    v = fmaf(__ldg(mrow + (int64_t)(j0 + e) * P.msk), kLog2e, v);
                if (!full) {
                    const int64_t j = j0 + e;
                    const bool vis = j < P.Tk && (!P.causal || j <= p) && (P.window <= 0 || j > p - P.window);
                    if (!vis) v = -INFINITY;
                }
                s[e] = v;
                bm = fmaxf(bm, v);
            }
            const float mnew = fmaxf(m, bm);
            const float shift = (mnew == -INFINITY) ? 0.f : mnew;
            const float alpha = (m == shift) ? 1.f : ex2(m - shift);

            uint32_t pk[kBN / 2];
            float rs = 0.f;
#pragma unroll
            for (int e = 0; e < kBN; e += 2) {
                const float p0 = ex2(s[e] - shift), p1 = ex2(s[e + 1] - shift);
                rs += p0 + p1;
                pk[e / 2] = pack_bf16x2(p0, p1);
            }

            if (jj >= 1) {  // P_{t-1} consumed and O final for t-1
                if (!__all_sync(0xffffffffu, mbar_wait(&bar.o_ready, (jj - 1) & 1, abort))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
#pragma unroll
            for (int c = 0; c < kBN / 64; ++c) {
                uint32_t r[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = pk[c * 32 + e];
                tmem_store32(lane_addr + kColP + c * 32, r);
            }
            if (jj >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[32];
                    tmem_load32(lane_addr + kColO + c * 32, r);
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                    tmem_store32(lane_addr + kColO + c * 32, r);
                }
            }
            tc_fence_before();
            mbar_arrive(&bar.p_full);
            l = fmaf(alpha, l, rs);
            m = mnew;
        }

        if (ok && n_tiles > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bar.o_ready, (n_tiles - 1) & 1, abort));
            tc_fence_after();
        }
        if (ok) {
            // Epilogue: o = O / l (0 for an empty row), lse = (m + log2 l) ln 2.
            const float inv = l > 0.f ? 1.f / l : 0.f;
            __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(P.o) + ((int64_t)bh * P.Tq + i) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                if (n_tiles > 0) {
                    tmem_load32(lane_addr + kColO + c * 32, r);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) r[e] = 0u;
                }
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * inv, __uint_as_float(r[2 * e + 1]) * inv);
                if (i < P.Tq) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                    for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
                }
            }
            if (P.lse != nullptr && i < P.Tq)
                P.lse[(int64_t)bh * P.Tq + i] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort && threadIdx.x == 0) atomicOr(&g_watchdog, 1u);
    if (warp == 5) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

// ------------------------------------------------------------------ host

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (fn == nullptr) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// [heads, rows, d] bf16 viewed as a 3-D tensor; boxes of 64 columns x 128 rows
// with the 128-byte swizzle; rows past `rows` read as zero.
bool make_map(EncodeTiledFn enc, CUtensorMap *map, const void *base, int d, int rows, int heads) {
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)heads};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows * d * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_d(const Params &P, cudaStream_t stream) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    CUtensorMap tq, tk, tv;
    // With Tk == 0 no key tile is ever loaded; the K/V maps only need to be valid.
    const void *kb = P.Tk > 0 ? P.k : P.q;
    const void *vb = P.Tk > 0 ? P.v : P.q;
    const int krows = P.Tk > 0 ? P.Tk : 1;
    const int kheads = P.Tk > 0 ? P.B * P.Hkv : 1;
    if (!make_map(enc, &tq, P.q, D, P.Tq, P.B * P.Hq) || !make_map(enc, &tk, kb, D, krows, kheads) ||
        !make_map(enc, &tv, vb, D, krows, kheads))
        return cudaErrorInvalidValue;
    // At least 116 KB so that one CTA holds an SM: the CTA takes all 512
    // tensor-memory columns, and a second resident CTA would only wait in
    // tcgen05.alloc.
    const size_t smem = SmemLayout<D>::kTotal + 1024 > 116 * 1024 ? SmemLayout<D>::kTotal + 1024 : 116 * 1024;
    static bool configured = false;
    if (!configured) {
        cudaError_t e =
            cudaFuncSetAttribute(fa_fwd_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int nqt = (P.Tq + kBM - 1) / kBM;
    const unsigned grid = (unsigned)nqt * (unsigned)(P.B * P.Hq);
    fa_fwd_bf16_kernel<D><<<grid, kThreads, smem, stream>>>(tq, tk, tv, P);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bf16(const Params &P, cudaStream_t stream) {
    if (P.d == 64) return launch_d<64>(P, stream);
    return launch_d<128>(P, stream);
}

}  // namespace fa
