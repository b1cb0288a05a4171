// fa_fwd_f32tc.cu -- fp32 exact tiled attention on the tcgen05 tensor cores
// with three TF32 products per matrix product.
//
// The tensor core's TF32 mode keeps the top 19 bits of each fp32 operand (the
// low 13 mantissa bits are dropped, not rounded).  With x = x_hi + x_lo,
// x_hi = x with those bits cleared and x_lo = x - x_hi (exact in fp32),
//
//   a . b  ~  a_hi b_hi + a_hi b_lo + a_lo b_hi        (the a_lo b_lo term,
//                                                      ~2^-20 relative, dropped)
//
// where the tensor core itself truncates raw fp32 to x_hi, so only the lo
// parts are materialised.  Same method as "FlashAttention forward in C"
// (sections 2.2-2.4): the online softmax over absolute key tiles, in base 2
// with a lazy maximum; per key tile t of 32 keys:
//
//   S_t = Q K_t^T       3 x (d / 8) MMAs 128 x 32 x 8, A = Q_hi / Q_lo from
//                       tensor memory, B = raw K_t / K_t,lo from shared memory
//   P_t = 2^(S_t c - m) softmax warps; P_t and P_t,lo written to tensor memory
//   O  += P_t V_t       3 x 4 MMAs 128 x d x 8, A = P_t / P_t,lo (tensor
//                       memory), B = V_t^T hi / lo (shared memory, K-major)
//
// Work unit: one 128-row query tile of one (batch, head); one unit per CTA.
// Warp roles (448 threads):
//   warps 0-7   softmax, Q split into tensor memory, epilogue: two threads per
//               row (paired-lane TMEM access), each half of the keys and of O
//   warps 8-11  splitters: K_lo next to the raw K tile; V transposed into
//               V^T hi / lo (every B operand is K-major)
//   warp 12     TMA producer (one lane): raw K and V tiles
//   warp 13     MMA issuer (one lane) and tensor-memory owner
// Tensor memory (512 columns): Q_hi [0,128) Q_lo [128,256) O [256,384)
// S_b / P_b [384 + 64b, +32) P_b,lo [416 + 64b, +32), b = 0, 1.
//
// Every mbarrier wait is bounded; a wait that runs out sets the CTA abort
// flag and the device watchdog word, the roles leave their loops and drain
// their copies and MMAs with bounded waits, and tensor memory is freed.
#include <cuda.h>

#include <cstdint>

#include "fa_internal.h"
#include "sm100_ptx.cuh"

namespace fa {

// Set when a bounded wait of this kernel ran out.
__device__ unsigned int g_watchdog_tc = 0;

namespace {

using namespace sm100;

constexpr int kBM = 128;  // query rows per unit
constexpr int kBN = 32;   // keys per tile
constexpr int kThreads = 448;
constexpr int kSoftmaxWarps = 8, kSplitWarps = 4;
constexpr int kWarpSplit = 8, kWarpTma = 12, kWarpMma = 13;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQh = 0, kColQl = 128, kColO = 256;
__host__ __device__ constexpr uint32_t col_s(int b) { return 384u + 64u * b; }
__host__ __device__ constexpr uint32_t col_plo(int b) { return 416u + 64u * b; }
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kKStages = 3, kVRawStages = 2, kVTStages = 3;

template <int D>
struct Layout {
    static constexpr int kBoxes = D / 32;                        // 32-column (128-byte) boxes per K/V tile
    static constexpr uint32_t kTileBytes = kBN * D * 4;          // raw K or V tile, K_lo tile
    static constexpr uint32_t kVTBytes = D * kBN * 4;            // V^T tile: D rows x 32 keys
    static constexpr uint32_t kKRaw = 0;
    static constexpr uint32_t kKLo = kKRaw + kKStages * kTileBytes;
    static constexpr uint32_t kVRaw = kKLo + kKStages * kTileBytes;
    static constexpr uint32_t kVHiT = kVRaw + kVRawStages * kTileBytes;
    static constexpr uint32_t kVLoT = kVHiT + kVTStages * kVTBytes;
    static constexpr uint32_t kBar = kVLoT + kVTStages * kVTBytes;
    static constexpr uint32_t kTotal = kBar + 512;
};

struct Barriers {
    uint64_t k_full[kKStages], k_empty[kKStages], ks_full[kKStages];  // raw K landed / free; K_lo written
    uint64_t vr_full[kVRawStages], vr_empty[kVRawStages];             // raw V landed / read by the splitters
    uint64_t vt_full[kVTStages], vt_empty[kVTStages];                 // V^T hi/lo written / free
    uint64_t q_ready;                                                  // Q_hi / Q_lo in tensor memory
    uint64_t s_full[2], p_full[2];
    uint64_t o_done, o_final, drain;
    uint32_t tmem_base;
    int abort;
};

struct Pos {
    int st = 0;
    uint32_t ph = 0;
    template <int N>
    __device__ __forceinline__ void advance() {
        if (++st == N) {
            st = 0;
            ph ^= 1u;
        }
    }
};

// Drop the 13 mantissa bits the TF32 mode ignores.
__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xffffe000u); }

struct Unit {
    int b, h, g, r0, t_begin, n_tiles;
};

// Unit = blockIdx.x: heaviest query tiles first.
__device__ __forceinline__ Unit make_unit(const Params &P) {
    Unit U;
    const int BH = P.B * P.Hq;
    const int nqt = (P.Tq + kBM - 1) / kBM;
    const int qt = nqt - 1 - (int)(blockIdx.x / BH);
    const int bh = (int)(blockIdx.x % BH);
    U.b = bh / P.Hq;
    U.h = bh % P.Hq;
    U.g = U.h / P.group;
    U.r0 = qt * kBM;
    int64_t lo_a, hi_a, lo_b, hi_b;
    visible_range(P, (int64_t)P.q_offset + U.r0, lo_a, hi_a);
    visible_range(P, (int64_t)P.q_offset + min(U.r0 + kBM, P.Tq) - 1, lo_b, hi_b);
    const int64_t klo = lo_a, khi = hi_b > hi_a ? hi_b : hi_a;
    U.t_begin = khi > klo ? (int)(klo / kBN) : 0;
    U.n_tiles = khi > klo ? (int)((khi + kBN - 1) / kBN) - U.t_begin : 0;
    return U;
}

// TMA producer: raw K_j and V_j in turn.
template <int D>
__device__ __forceinline__ void producer_role(const CUtensorMap &tmK, const CUtensorMap &tmV, const Params &P,
                                              const Unit &U, uint8_t *smem, Barriers &bar) {
    using L = Layout<D>;
    volatile int *abort = &bar.abort;
    int k_issued[kKStages] = {}, v_issued[kVRawStages] = {};
    Pos kp, vp;
    bool ok = true;
    for (int j = 0; j < U.n_tiles && ok; ++j) {
        const int key0 = (U.t_begin + j) * kBN;
        if (k_issued[kp.st] > 0 && !(ok = mbar_wait(&bar.k_empty[kp.st], kp.ph ^ 1u, abort))) break;
        mbar_arrive_expect_tx(&bar.k_full[kp.st], L::kTileBytes);
#pragma unroll
        for (int c = 0; c < L::kBoxes; ++c)
            tma_load_4d(smem + L::kKRaw + kp.st * L::kTileBytes + c * (kBN * 128), &tmK, &bar.k_full[kp.st], c * 32,
                        key0, U.g, U.b);
        ++k_issued[kp.st];
        kp.template advance<kKStages>();
        if (v_issued[vp.st] > 0 && !(ok = mbar_wait(&bar.vr_empty[vp.st], vp.ph ^ 1u, abort))) break;
        mbar_arrive_expect_tx(&bar.vr_full[vp.st], L::kTileBytes);
#pragma unroll
        for (int c = 0; c < L::kBoxes; ++c)
            tma_load_4d(smem + L::kVRaw + vp.st * L::kTileBytes + c * (kBN * 128), &tmV, &bar.vr_full[vp.st], c * 32,
                        key0, U.g, U.b);
        ++v_issued[vp.st];
        vp.template advance<kVRawStages>();
    }
    // Every copy issued lands before shared memory goes away.
    int never = 0;
    for (int s = 0; s < kKStages; ++s)
        if (k_issued[s] > 0) mbar_wait(&bar.k_full[s], (k_issued[s] - 1) & 1, &never, 200000000ull);
    for (int s = 0; s < kVRawStages; ++s)
        if (v_issued[s] > 0) mbar_wait(&bar.vr_full[s], (v_issued[s] - 1) & 1, &never, 200000000ull);
}

// Splitters (128 threads).  Raw tiles are [D/32 boxes][32 rows][128 bytes]
// with the 128-byte swizzle (16-byte chunk c of row r at c ^ (r % 8)).
//   K_lo: the same layout, element-wise lo part.
//   V^T hi / lo: [D rows (columns of V)][32 keys = 128 bytes], swizzled the
//   same way, so that P V reads V^T as a K-major operand.
template <int D>
__device__ __forceinline__ void split_role(const Params &P, const Unit &U, uint8_t *smem, Barriers &bar, int t,
                                           int lane) {
    using L = Layout<D>;
    volatile int *abort = &bar.abort;
    Pos kp, vrp, vtp;
    bool ok = true;
    for (int j = 0; j < U.n_tiles && ok; ++j) {
        // K_lo
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.k_full[kp.st], kp.ph, abort)))) break;
        {
            const float4 *src = reinterpret_cast<const float4 *>(smem + L::kKRaw + kp.st * L::kTileBytes);
            float4 *dst = reinterpret_cast<float4 *>(smem + L::kKLo + kp.st * L::kTileBytes);
#pragma unroll
            for (int e = t; e < (int)(L::kTileBytes / 16); e += kSplitWarps * 32) {
                const float4 x = src[e];
                dst[e] = make_float4(x.x - tf32_hi(x.x), x.y - tf32_hi(x.y), x.z - tf32_hi(x.z), x.w - tf32_hi(x.w));
            }
        }
        fence_proxy_async_smem();  // the MMAs read K_lo through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.ks_full[kp.st]);
        kp.template advance<kKStages>();

        // V^T hi / lo: thread t owns column x = t of V (row x of V^T)
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.vr_full[vrp.st], vrp.ph, abort)))) break;
        if (j >= kVTStages && !(ok = __all_sync(0xffffffffu, mbar_wait(&bar.vt_empty[vtp.st], vtp.ph ^ 1u, abort))))
            break;
        if (t < D) {
            const int x = t;
            const uint8_t *raw = smem + L::kVRaw + vrp.st * L::kTileBytes + (x / 32) * (kBN * 128);
            const int cx = (x % 32) / 4, wx = (x % 4) * 4;
            float v[kBN];
#pragma unroll
            for (int r = 0; r < kBN; ++r) v[r] = *reinterpret_cast<const float *>(raw + r * 128 + ((cx ^ (r & 7)) * 16) + wx);
            uint8_t *hi = smem + L::kVHiT + vtp.st * L::kVTBytes + x * 128;
            uint8_t *lo = smem + L::kVLoT + vtp.st * L::kVTBytes + x * 128;
#pragma unroll
            for (int c = 0; c < kBN / 4; ++c) {
                const float4 a = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                const float4 ah = make_float4(tf32_hi(a.x), tf32_hi(a.y), tf32_hi(a.z), tf32_hi(a.w));
                *reinterpret_cast<float4 *>(hi + ((c ^ (x & 7)) * 16)) = ah;
                *reinterpret_cast<float4 *>(lo + ((c ^ (x & 7)) * 16)) =
                    make_float4(a.x - ah.x, a.y - ah.y, a.z - ah.z, a.w - ah.w);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.vr_empty[vrp.st]);  // raw V read
        vrp.template advance<kVRawStages>();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.vt_full[vtp.st]);
        vtp.template advance<kVTStages>();
    }
}

// Shared-memory descriptor (128-byte swizzle, K-major, 8-row atoms of 1 KB).
__device__ __forceinline__ uint64_t desc(uint32_t saddr) { return smem_desc_sw128(saddr, 16, 1024); }

// S_b = Q K^T: per 8-column step of d, Q_hi K + Q_hi K_lo + Q_lo K.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t tbase, int b, uint32_t kraw, uint32_t klo) {
    constexpr uint32_t id = idesc_tf32_f32(kBM, kBN);
#pragma unroll
    for (int kk = 0; kk < D / 8; ++kk) {
        const uint32_t off = (kk >> 2) * (kBN * 128) + (kk & 3) * 32;  // box, then 32 bytes per 8 fp32
        const uint64_t dk = desc(kraw + off), dl = desc(klo + off);
        mma_ts_tf32(tbase + col_s(b), tbase + kColQh + kk * 8, (uint32_t)dk, (uint32_t)(dk >> 32), id, kk > 0);
        mma_ts_tf32(tbase + col_s(b), tbase + kColQh + kk * 8, (uint32_t)dl, (uint32_t)(dl >> 32), id, 1u);
        mma_ts_tf32(tbase + col_s(b), tbase + kColQl + kk * 8, (uint32_t)dk, (uint32_t)(dk >> 32), id, 1u);
    }
}

// O += P_b V: per 8 keys, P V_hi^T + P V_lo^T + P_lo V_hi^T.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tbase, int b, uint32_t vhi, uint32_t vlo, uint32_t accumulate) {
    constexpr uint32_t id = idesc_tf32_f32(kBM, D);
#pragma unroll
    for (int kk = 0; kk < kBN / 8; ++kk) {
        const uint64_t dh = desc(vhi + kk * 32), dl = desc(vlo + kk * 32);
        mma_ts_tf32(tbase + kColO, tbase + col_s(b) + kk * 8, (uint32_t)dh, (uint32_t)(dh >> 32), id,
                    (kk > 0 || accumulate) ? 1u : 0u);
        mma_ts_tf32(tbase + kColO, tbase + col_s(b) + kk * 8, (uint32_t)dl, (uint32_t)(dl >> 32), id, 1u);
        mma_ts_tf32(tbase + kColO, tbase + col_plo(b) + kk * 8, (uint32_t)dh, (uint32_t)(dh >> 32), id, 1u);
    }
}

// MMA issuer: S_0, S_1 up front; per tile j: wait P_j, O += P_j V_j, then
// S_{j+2} into the buffer P_j came from (tcgen05 MMAs of one thread execute
// in order).
template <int D>
__device__ __forceinline__ void mma_role(const Unit &U, uint8_t *smem, Barriers &bar, uint32_t tbase) {
    using L = Layout<D>;
    volatile int *abort = &bar.abort;
    const int n = U.n_tiles;
    bool ok = true;
    Pos kp, vtp;
    auto issue_s = [&](int j) -> bool {
        if (!mbar_wait(&bar.ks_full[kp.st], kp.ph, abort)) return false;  // raw K and K_lo
        tc_fence_after();
        issue_qk<D>(tbase, j & 1, smem_u32(smem + L::kKRaw + kp.st * L::kTileBytes),
                    smem_u32(smem + L::kKLo + kp.st * L::kTileBytes));
        mma_commit(&bar.s_full[j & 1]);
        mma_commit(&bar.k_empty[kp.st]);
        kp.template advance<kKStages>();
        return true;
    };
    if (n > 0) {
        ok = mbar_wait(&bar.q_ready, 0, abort);
        if (ok) ok = issue_s(0);
        if (ok && n > 1) ok = issue_s(1);
        for (int j = 0; j < n && ok; ++j) {
            if (!(ok = mbar_wait(&bar.p_full[j & 1], (j >> 1) & 1, abort))) break;
            if (!(ok = mbar_wait(&bar.vt_full[vtp.st], vtp.ph, abort))) break;
            tc_fence_after();
            issue_pv<D>(tbase, j & 1, smem_u32(smem + L::kVHiT + vtp.st * L::kVTBytes),
                        smem_u32(smem + L::kVLoT + vtp.st * L::kVTBytes), j > 0 ? 1u : 0u);
            mma_commit(&bar.o_done);
            mma_commit(&bar.vt_empty[vtp.st]);
            vtp.template advance<kVTStages>();
            if (j + 2 < n && !(ok = issue_s(j + 2))) break;
        }
        mma_commit(&bar.o_final);
    }
    mma_commit(&bar.drain);
    int never = 0;
    mbar_wait(&bar.drain, 0, &never, 200000000ull);
}

// Softmax warps 0-7: Q split into tensor memory, the online softmax, the
// epilogue.  Warp w covers TMEM lanes 32 (w % 4) + 16 (w / 4) .. +16; lanes
// l and l + 16 share a row (keys [0, 16) and [16, 32) of a tile; columns
// [0, D/2) and [D/2, D) of Q and O).
template <int D>
__device__ __forceinline__ void softmax_role(const Params &P, const Unit &U, Barriers &bar, uint32_t tbase, int warp,
                                             int lane) {
    constexpr int kHK = kBN / 2;  // keys per thread
    constexpr int kHD = D / 2;    // columns of Q / O per thread
    volatile int *abort = &bar.abort;
    const int half = lane >> 4;
    const int lane0 = 32 * (warp & 3) + 16 * (warp >> 2);
    const int row = lane0 + (lane & 15);
    const uint32_t lane_off = (uint32_t)lane0 << 16;
    const int i = U.r0 + row;
    const bool live = i < P.Tq;
    const float c = P.scale_log2;
    const int n = U.n_tiles;
    bool ok = true;

    // Q row i, this thread's half of the columns: hi and lo into tensor memory.
    {
        const float *qrow = static_cast<const float *>(P.q) + U.b * P.q_sb + U.h * P.q_sh + (int64_t)i * P.q_st;
#pragma unroll
        for (int cc = 0; cc < kHD; cc += 32) {
            uint32_t hi[32], lo[32];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                const int col = half * kHD + cc + e;
                float2 x = make_float2(0.f, 0.f);
                if (live && col < P.d) x = *reinterpret_cast<const float2 *>(qrow + col);
                const float hx = tf32_hi(x.x), hy = tf32_hi(x.y);
                hi[e] = __float_as_uint(hx);
                hi[e + 1] = __float_as_uint(hy);
                lo[e] = __float_as_uint(x.x - hx);
                lo[e + 1] = __float_as_uint(x.y - hy);
            }
            tmem_store_pair32<kHD>(tbase + lane_off + kColQh + cc, hi);
            tmem_store_pair32<kHD>(tbase + lane_off + kColQl + cc, lo);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.q_ready);
    }

    const int64_t p = (int64_t)P.q_offset + i;
    const int64_t p_first = (int64_t)P.q_offset + U.r0;
    const int64_t p_last = (int64_t)P.q_offset + min(U.r0 + kBM, P.Tq) - 1;
    int vlo, vhi;
    {
        int64_t lo64, hi64;
        visible_range(P, p, lo64, hi64);
        vlo = (int)lo64;
        vhi = (int)hi64;
    }
    const bool has_sink = P.sinks != nullptr;
    float m = has_sink ? __ldg(P.sinks + U.h) * kLog2e : -INFINITY;
    float l = (has_sink && half == 0) ? 1.f : 0.f;
    const float *mrow =
        (P.mask != nullptr && live) ? P.mask + U.b * P.msb + U.h * P.msh + (int64_t)i * P.msq : nullptr;
    int ti_lo = 0, ti_hi = 0;  // interior tiles: every key visible to every row, no mask
    if (P.mask == nullptr && c > 0.f) {
        int64_t hi_key = P.Tk;
        if (P.causal && p_first + 1 < hi_key) hi_key = p_first + 1;
        int64_t lo_key = 0;
        if (P.window > 0 && p_last - P.window + 1 > 0) lo_key = p_last - P.window + 1;
        ti_lo = (int)((lo_key + kBN - 1) / kBN - U.t_begin);
        ti_hi = (int)(hi_key / kBN - U.t_begin);
    }

    for (int j = 0; j < n; ++j) {
        const int b = j & 1;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.s_full[b], (j >> 1) & 1, abort)))) break;
        tc_fence_after();
        uint32_t sr[kHK];
        tmem_load_pair16<kHK>(tbase + lane_off + col_s(b), sr);
        float *s = reinterpret_cast<float *>(sr);
        float cs = c;
        if (j < ti_lo || j >= ti_hi) {
            const int k0 = (U.t_begin + j) * kBN + half * kHK;
            const int elo = min(max(vlo - k0, 0), kHK), ehi = min(max(vhi - k0, 0), kHK);
            if (mrow != nullptr) {
#pragma unroll
                for (int e = 0; e < kHK; ++e) {
                    const int jj = min(k0 + e, P.Tk - 1);
                    const float x = fmaf(__ldg(mrow + (int64_t)jj * P.msk), kLog2e, s[e] * c);
                    s[e] = (e >= elo && e < ehi) ? x : -INFINITY;
                }
                cs = 1.f;
            } else if (c <= 0.f) {
#pragma unroll
                for (int e = 0; e < kHK; ++e) s[e] = (e >= elo && e < ehi) ? s[e] * c : -INFINITY;
                cs = 1.f;
            } else {
#pragma unroll
                for (int e = 0; e < kHK; ++e) s[e] = (e >= elo && e < ehi) ? s[e] : -INFINITY;
            }
        }
        float bm = s[0];
#pragma unroll
        for (int e = 1; e < kHK; ++e) bm = fmaxf(bm, s[e]);
        bm *= cs;
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
        float alpha = 1.f;
        if (bm > m + kRescaleThreshold) {
            alpha = ex2_approx(m - bm);
            m = bm;
        }
        const float shift = (m == -INFINITY) ? 0.f : m;
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
            // O must hold P_{j-1} V_{j-1} before it is rescaled.
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.o_done, (uint32_t)((j - 1) & 1), abort)))) break;
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < kHD; cc += 32) {
                uint32_t orr[32];
                tmem_load_pair32<kHD>(tbase + lane_off + kColO + cc, orr);
#pragma unroll
                for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
                tmem_store_pair32<kHD>(tbase + lane_off + kColO + cc, orr);
            }
        }
        // p in fp32: P = p (the tensor core drops its low bits), P_lo = p - P_hi.
        uint32_t ph[kHK], pl[kHK];
        float sum = 0.f;
#pragma unroll
        for (int e = 0; e < kHK; ++e) {
            const float pe = ex2_approx(fmaf(s[e], cs, -shift));
            sum += pe;
            ph[e] = __float_as_uint(pe);
            pl[e] = __float_as_uint(pe - tf32_hi(pe));
        }
        tmem_store_pair16<kHK>(tbase + lane_off + col_s(b), ph);
        tmem_store_pair16<kHK>(tbase + lane_off + col_plo(b), pl);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.p_full[b]);
        l = fmaf(alpha, l, sum);
    }
    if (!ok) return;

    // Epilogue: o = O / l (0 for an empty row), lse = (m + log2 l) ln 2.
    const float lt = l + __shfl_xor_sync(0xffffffffu, l, 16);
    const float inv = lt > 0.f ? 1.f / lt : 0.f;
    if (n > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(&bar.o_final, 0, abort))) return;
        tc_fence_after();
    }
    float *orow = static_cast<float *>(P.o) + U.b * P.o_sb + U.h * P.o_sh + (int64_t)i * P.o_st;
#pragma unroll
    for (int cc = 0; cc < kHD; cc += 32) {
        uint32_t ov[32];
        if (n > 0) {
            tmem_load_pair32<kHD>(tbase + lane_off + kColO + cc, ov);
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = 0u;
        }
        if (live) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                const int col = half * kHD + cc + e;
                if (col < P.d)
                    *reinterpret_cast<float2 *>(orow + col) =
                        make_float2(__uint_as_float(ov[e]) * inv, __uint_as_float(ov[e + 1]) * inv);
            }
        }
    }
    if (n > 0) tc_fence_before();
    if (live && P.lse != nullptr && half == 0)
        P.lse[((int64_t)U.b * P.Hq + U.h) * P.Tq + i] = lt > 0.f ? (m + log2f(lt)) * kLn2 : -INFINITY;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_f32tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const Params P) {
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Barriers &bar = *reinterpret_cast<Barriers *>(smem + L::kBar);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&bar.k_full[s], 1);
            mbar_init(&bar.k_empty[s], 1);
            mbar_init(&bar.ks_full[s], kSplitWarps);
        }
        for (int s = 0; s < kVRawStages; ++s) {
            mbar_init(&bar.vr_full[s], 1);
            mbar_init(&bar.vr_empty[s], kSplitWarps);
        }
        for (int s = 0; s < kVTStages; ++s) {
            mbar_init(&bar.vt_full[s], kSplitWarps);
            mbar_init(&bar.vt_empty[s], 1);
        }
        mbar_init(&bar.q_ready, kSoftmaxWarps);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar.s_full[s], 1);
            mbar_init(&bar.p_full[s], kSoftmaxWarps);
        }
        mbar_init(&bar.o_done, 1);
        mbar_init(&bar.o_final, 1);
        mbar_init(&bar.drain, 1);
        bar.abort = 0;
        mbar_init_fence();
    }
    if (warp == kWarpMma) {
        tmem_alloc(&bar.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kWarpTma && lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = bar.tmem_base;
    grid_dependency_wait();
    grid_launch_dependents();
    const Unit U = make_unit(P);

    if (warp == kWarpTma) {
        if (lane == 0) producer_role<D>(tmK, tmV, P, U, smem, bar);
    } else if (warp == kWarpMma) {
        if (lane == 0) mma_role<D>(U, smem, bar, tbase);
    } else if (warp >= kWarpSplit) {
        split_role<D>(P, U, smem, bar, threadIdx.x - kWarpSplit * 32, lane);
    } else {
        softmax_role<D>(P, U, bar, tbase, warp, lane);
    }

    tc_fence_before();
    __syncthreads();
    if (bar.abort && threadIdx.x == 0) atomicOr(&g_watchdog_tc, 1u);
    if (warp == kWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

// ------------------------------------------------------------------ host

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn32() {
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

// [B, H, T, d] fp32 with element strides as the 4-D map (d, T, H, B); boxes of
// 32 columns (128 bytes) x 32 rows, 128-byte swizzle; rows and columns past
// the tensor read as zero.  Extent-1 dimensions get a packed stride.
bool make_map32(EncodeTiledFn enc, CUtensorMap *map, const void *base, int d, int T, int H, int B, int64_t st,
                int64_t sh, int64_t sb) {
    const int64_t dims[4] = {d, T, H, B}, strides[4] = {1, st, sh, sb};
    cuuint64_t gd[4], gs[3];
    cuuint32_t bx[4] = {32, (cuuint32_t)kBN, 1, 1}, es[4] = {1, 1, 1, 1};
    uint64_t packed = (uint64_t)d * 4;
    for (int i = 0; i < 4; ++i) {
        gd[i] = (cuuint64_t)dims[i];
        if (i > 0) {
            gs[i - 1] = dims[i] > 1 ? (cuuint64_t)strides[i] * 4 : (cuuint64_t)packed;
            packed = (uint64_t)gs[i - 1] * (uint64_t)dims[i];
        }
    }
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void *>(base), gd, gs, bx, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_tc(const Params &P, cudaStream_t stream) {
    EncodeTiledFn enc = encode_fn32();
    if (enc == nullptr) return cudaErrorNotSupported;
    CUtensorMap tk, tv;
    const bool kv = P.Tk > 0;
    if (!make_map32(enc, &tk, kv ? P.k : P.q, P.d, kv ? P.Tk : 1, kv ? P.Hkv : 1, kv ? P.B : 1, kv ? P.k_st : P.q_st,
                    kv ? P.k_sh : P.q_sh, kv ? P.k_sb : P.q_sb) ||
        !make_map32(enc, &tv, kv ? P.v : P.q, P.d, kv ? P.Tk : 1, kv ? P.Hkv : 1, kv ? P.B : 1, kv ? P.v_st : P.q_st,
                    kv ? P.v_sh : P.q_sh, kv ? P.v_sb : P.q_sb))
        return cudaErrorInvalidValue;
    constexpr size_t kSmem = Layout<D>::kTotal + 1024;
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(fa_fwd_f32tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int nqt = (P.Tq + kBM - 1) / kBM;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((long long)nqt * P.B * P.Hq));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fa_fwd_f32tc_kernel<D>, tk, tv, P);
}

}  // namespace

cudaError_t launch_f32_tc(const Params &P, cudaStream_t stream) {
    return P.d <= 64 ? launch_tc<64>(P, stream) : launch_tc<128>(P, stream);
}

}  // namespace fa
