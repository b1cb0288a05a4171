// fa_fwd_bf16.cu -- bf16 exact tiled attention on the tcgen05 tensor cores.
//
// Work unit: one 128-row query tile of one (batch, query head).  A unit walks
// the key tiles its rows can see, 128 keys at absolute positions
// [128t, 128t + 128) each, under the online softmax of "FlashAttention forward
// in C" (section 2.2), in base 2 (c = scale * log2 e):
//
//   S_t = Q K_t^T          tcgen05.mma, Q and K_t from shared memory (TMA,
//                          128-byte swizzle), fp32 accumulator in TMEM
//   P_t = 2^(S_t c - m)    softmax warps: tcgen05.ld of S_t (with the row max
//                          from the load on interior tiles), ex2, row sum; P
//                          rounded to bf16 and tcgen05.st back into the first
//                          64 columns of S_t's buffer
//   O  += P_t V_t          tcgen05.mma, A = P_t from TMEM, B = V_t (MN-major)
//
// S has three buffers in tensor memory and two threads issue the MMAs: one
// computes S_{t+1}, S_{t+2} while the softmax warps work on S_t, the other
// accumulates O += P_t V_t.  S_{t+3} reuses the buffer of P_t and waits for
// the completion of O += P_t V_t.
//
// The running max m of a row is raised lazily: only when a tile's max
// exceeds it by more than 8 (log2 units) is O rescaled in TMEM by
// 2^(m_old - m_new); otherwise the row keeps the old m, its weights stay
// below 2^8 and the final O / l is the same quantity.  The rescale guard
// follows "Fused attention and softmax: fast and exact" (the exact
// definition, steps 2 and 5).
//
// Persistent schedule: one CTA (or CTA pair) per SM walks a list of units
// sorted heaviest first (under a causal rule the last query tiles see the
// most keys), taking them in snake order (round r takes group g, the next
// round group G-1-g), so heavy and light units balance across SMs.  The K/V
// rings, the S buffers and every barrier run on across units: the next unit's
// K_0, K_1 and Q load while the current unit finishes, its first S tiles run
// while the softmax warps write the current unit's output.
//
// K and V tiles have rings of their own, each read by one issuing thread.
// Every CTA loads its own tiles (no cluster multicast): the K/V tiles a GQA
// group shares come from L2.
//
// Warp roles (384 threads in prefill, 352 for the other mappings):
//   warps 0-7   softmax and epilogue: two threads per query row (= TMEM
//               lane), each with half of the row's keys and of O's columns
//   warp 8      TMA producer (one lane)
//   warp 9      S = Q K^T issuer (one lane) and tensor-memory owner
//   warp 10     O += P V issuer (one lane)
//   warp 11     prefill only, idle: it completes warps 8-11 as a warpgroup,
//               which gives registers to the softmax warpgroups
// Tensor memory (512 columns allocated): S_0 [0,128) S_1 [128,256)
// S_2 [256,384) O [384, 384+d).
//
// A row's arithmetic does not depend on its query tile, its unit's place in
// the schedule or on chunking through q_offset: key tiles are absolute, a key
// the row cannot see gets weight 0 and leaves m, l and O unchanged
// ("FlashAttention forward in C", section 2.4).
//
// Launch: programmatic dependent launch lets the CTA prologue overlap the
// previous kernel in the stream; griddepcontrol.wait orders every global
// access after it.  The producer looks up its first unit (kernel parameters
// only) before that wait, so its first loads issue as soon as it returns.
//
// Every mbarrier wait is bounded (two seconds of wall time); a wait that runs
// out sets a CTA-wide abort flag and the device watchdog word, every role
// leaves its loop, in-flight copies and MMAs are drained with bounded waits,
// and tensor memory is released before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>
#include <mutex>

#include "fa_internal.h"
#include "fa_tma_host.h"
#include "sm100_ptx.cuh"

namespace fa {

__device__ unsigned int g_watchdog = 0;
// Test hook, zero unless a test sets it: CTA 0 then skips its first Q load,
// so that the QK issuer's bounded wait runs out and the abort path runs.
__device__ int g_drop_arrive = 0;

namespace {

using namespace sm100;

constexpr int kBM = 128;  // query rows per unit = tensor-memory lanes
constexpr int kBN = 128;  // keys per tile
constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = 352;
constexpr int kWarpTma = 8, kWarpQk = 9, kWarpPv = 10;
// Prefill mappings add an idle warp 11, so that warps 8-11 form a whole
// warpgroup: it gives registers back (setmaxnreg) and the two softmax
// warpgroups take them, so the softmax keeps every value in registers.
// 384 threads x 168 at launch (three warps per scheduler partition);
// softmax 2 x 128 x 216 + issuers 128 x 64 <= 384 x 168.
constexpr int kThreadsPrefill = 384;
constexpr int kRegsLaunchPrefill = 168, kRegsSoftmaxPrefill = 216, kRegsIssuePrefill = 64;
static_assert(256 * kRegsSoftmaxPrefill + 128 * kRegsIssuePrefill <= kThreadsPrefill * kRegsLaunchPrefill,
              "the register split fits the launch allocation");
static_assert(2 * kRegsSoftmaxPrefill + kRegsIssuePrefill <= 512, "per scheduler partition: two softmax warps and one issuer");
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufs = 3;                                                     // S (and P) buffers
__host__ __device__ constexpr uint32_t col_s(int buf) { return 128u * buf; }  // S_0, S_1, S_2
constexpr uint32_t kColO = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: weights stay below 2^8
constexpr int kPrefetchTiles = 4;          // K and V tiles of the first unit requested into L2 early
constexpr uint32_t kSwRowBytes = 128;      // one swizzled row: 64 bf16
constexpr int kMaxStages = 6;

// The two ways rows are mapped onto 128-row tiles.
//   kPrefill  a unit is one 128-row query tile of one (batch, query head);
//             persistent grid, heaviest units first.
//   kDecode   all group * Tq query rows of a KV head form one tile (row
//             r = i * group + hl: query head g * group + hl, its row i), so K
//             and V are read once per KV head; the unit's key range is split
//             over the CTAs of a cluster, which merge their partial (m, l, O)
//             through distributed shared memory.
//   kPaged    kDecode on paged K/V caches with a key count per sequence:
//             key tiles are gathered page by page through a block table.
//   kVarlen   kPrefill over a batch of sequences packed along the rows
//             ([total, H, d] tensors, cu_seqlens offsets), each with its own
//             row and key counts; O is written with predicated stores.
//   kPrefill8 kPrefill with e4m3 Q, K and V: the MMAs are kind::f8f6f4 (32
//             elements per K step), P is rounded to e4m3 (four per tensor-
//             memory column), O stays bf16.
//   kVarlen8  kVarlen with e4m3 Q, K and V, as kPrefill8.
//   kSplitKv  kDecode without a cluster: the key range of a KV head is split
//             over as many CTAs as fill the SMs, each CTA writes its partial
//             (m, l, O) to a workspace in global memory, and the last CTA of
//             the KV head to finish (a counter per KV head) merges them.
constexpr int kPrefill = 0, kDecode = 1, kPaged = 2, kVarlen = 3, kPrefill8 = 4, kVarlen8 = 5, kSplitKv = 6;
__host__ __device__ constexpr bool is_packed(int mode) { return mode == kDecode || mode == kPaged || mode == kSplitKv; }
// One split's block of the split-KV workspace: R rows of D fp32 (unnormalised
// O), then R (m, l) pairs, padded to a multiple of 4 floats so that every
// block starts on a 16-byte boundary (the rows are written and read as float4).
__host__ __device__ constexpr int64_t ws_block_floats(int R, int D) { return ((int64_t)R * (D + 2) + 3) & ~int64_t(3); }
__host__ __device__ constexpr bool is_prefill(int mode) { return mode == kPrefill || mode == kPrefill8; }
__host__ __device__ constexpr bool is_varlen(int mode) { return mode == kVarlen || mode == kVarlen8; }
__host__ __device__ constexpr int elem_bytes(int mode) {  // Q, K, V
    return (mode == kPrefill8 || mode == kVarlen8) ? 1 : 2;
}
__host__ __device__ constexpr int threads_for(int mode) { return is_prefill(mode) ? kThreadsPrefill : kThreads; }
// bf16 prefill with d = 128 (two 64-column boxes per tile) issues the CTA's
// first S in two halves of d: the first four MMAs need only box 0 of Q and
// K_0, which land on a barrier of their own, while box 1 is still in flight.
// The MMAs and their order are unchanged.
template <int D, int MODE>
__host__ __device__ constexpr bool split_first_s() {
    return is_prefill(MODE) && elem_bytes(MODE) == 2 && D == 128;
}

template <int D, int MODE>
struct SmemLayout {
    static constexpr int kE = elem_bytes(MODE);
    static constexpr int kBoxCols = 128 / kE;  // columns of a 128-byte TMA box
    static constexpr int kBoxes = D / kBoxCols;  // boxes per Q, K or V tile
    static constexpr int kOBoxes = D / 64;       // O is bf16
    static_assert(D % kBoxCols == 0 && kOBoxes * 64 == D, "whole boxes");
    static constexpr uint32_t kQBytes = kBM * D * kE;
    static constexpr uint32_t kKVBytes = kBN * D * kE;                    // one K or V tile (a ring stage)
    static constexpr uint32_t kOBytes = kBM * D * 2;                      // the bf16 O tile
    static constexpr int kStages = (D == 128 && kE == 2) ? 3 : 6;         // K ring: 96 KB
    // V ring: one stage fewer in prefill, where the O tile is staged for its
    // TMA store; packed rows write O from registers and take the full ring.
    static constexpr bool kStaging = is_prefill(MODE);  // O leaves through a TMA store
    static constexpr int kVStages = kStaging ? kStages - 1 : kStages;
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kKRing = kQ + kQBytes;
    static constexpr uint32_t kVRing = kKRing + kStages * kKVBytes;
    static constexpr uint32_t kOStage = kVRing + kVStages * kKVBytes;  // O tile, bf16, for the TMA store
    static constexpr uint32_t kBar = kOStage + (kStaging ? kOBytes : 0u);
    // Packed-row split merge: O partials (fp32, padded rows) over the K ring,
    // (m, l) per row over the V ring.
    static constexpr int kOPartStride = D + 4;
    static_assert(kBM * kOPartStride * 4 <= kStages * kKVBytes, "O partials fit the K ring");
    static constexpr uint32_t kTotal = kBar + 512;
    static_assert(kStages <= kMaxStages && kVStages <= kMaxStages, "ring too deep");
};

struct Barriers {
    uint64_t q_full;                                   // Q of the unit landed
    uint64_t q_empty;                                  // the unit's last S done: Q buffer free
    uint64_t k_full[kMaxStages], k_empty[kMaxStages];  // the K ring
    uint64_t v_full[kMaxStages], v_empty[kMaxStages];  // the V ring
    uint64_t s_full[kSBufs];                           // S written into buffer b
    uint64_t p_full[kSBufs];                           // P written over S in buffer b
    uint64_t o_done[kSBufs];                           // O += P V from buffer b completed
    uint64_t o_final;                                  // the unit's last O += P V completed
    uint64_t ep_free;                                  // the O staging tile may be written
    uint64_t ep_full;                                  // the O staging tile is written
    uint64_t drain[2];                                 // issuers' last MMAs completed
    uint64_t first_lo;  // column box 0 of the CTA's first Q and K_0 landed (first S in halves)
    uint32_t tmem_base;
    int abort;
    int last;  // split-KV through the workspace: this CTA merges its KV head
};


struct Unit {
    int b, h, g, bh;
    int r0;  // first query row of the tile (prefill)
    int t_begin, n_tiles;
    int Tk, q_offset;  // keys of the unit's sequence, position of its query row 0
    int Tq;            // query rows of the unit's sequence
    int qrow, krow;    // tensor rows where the sequence's queries / keys start
};

// Units sorted heaviest first: unit u has query tile nqt-1-u/per_qt, then
// (batch, head).
template <int MODE>
__device__ __forceinline__ Unit make_unit(const Params &P, int u) {
    Unit U;
    const int nqt = (P.Tq + kBM - 1) / kBM;
    // Divisions by launch constants: multiply-high and shift (fast_div.h).
    const int qpos = (int)P.fd_per_qt.div((uint32_t)u);
    const int qt = nqt - 1 - qpos;
    const int r = u - qpos * (int)P.fd_per_qt.d;
    U.b = (int)P.fd_heads.div((uint32_t)r);  // fd_heads: Hq
    U.h = r - U.b * (int)P.fd_heads.d;
    U.bh = U.b * P.Hq + U.h;
    U.g = (int)P.fd_group.div((uint32_t)U.h);
    U.r0 = qt * kBM;
    if constexpr (is_varlen(MODE)) {
        // offsets clamped into the tensors: a malformed table cannot reach outside them
        const int q0 = min(max(__ldg(P.cu_q + U.b), 0), P.total_q);
        const int q1 = min(max(__ldg(P.cu_q + U.b + 1), q0), P.total_q);
        const int k0 = min(max(__ldg(P.cu_k + U.b), 0), P.total_k);
        const int k1 = min(max(__ldg(P.cu_k + U.b + 1), k0), P.total_k);
        U.Tq = q1 - q0;
        U.Tk = k1 - k0;
        U.qrow = q0;
        U.krow = k0;
        U.q_offset = U.Tk - U.Tq;  // the sequence's queries are its last positions
    } else {
        U.Tq = P.Tq;
        U.Tk = P.Tk;
        U.qrow = 0;
        U.krow = 0;
        U.q_offset = P.q_offset;
    }
    U.t_begin = 0;
    U.n_tiles = 0;
    if (U.r0 >= U.Tq) return U;  // a tile past the sequence's rows: nothing to do
    int64_t lo_a, hi_a, lo_b, hi_b;
    visible_range_tk(P, U.Tk, (int64_t)U.q_offset + U.r0, lo_a, hi_a);
    visible_range_tk(P, U.Tk, (int64_t)U.q_offset + min(U.r0 + kBM, U.Tq) - 1, lo_b, hi_b);
    const int64_t klo = lo_a, khi = hi_b > hi_a ? hi_b : hi_a;
    if (khi > klo) {
        U.t_begin = (int)(klo / kBN);
        U.n_tiles = (int)((khi + kBN - 1) / kBN) - U.t_begin;
    } else {
        U.t_begin = 0;
        U.n_tiles = 0;
    }
    return U;
}

// Packed-row unit of this CTA: KV head blockIdx.x / splits of the batch, key
// tiles [t_begin, t_begin + n_tiles) = this CTA's share (cluster rank
// blockIdx.x % splits) of the tiles the rows at positions q_offset ..
// q_offset + Tq - 1 can see.
template <int MODE>
__device__ __forceinline__ Unit decode_unit(const Params &P) {
    Unit U;
    const int cid = (int)P.fd_splits.div(blockIdx.x), rank = (int)blockIdx.x - cid * P.splits;
    U.b = (int)P.fd_hkv.div((uint32_t)cid);
    U.g = cid - U.b * P.Hkv;
    U.h = U.g * P.group;
    U.bh = U.b * P.Hq + U.h;
    U.r0 = 0;
    U.Tq = P.Tq;
    U.qrow = 0;
    U.krow = 0;
    if constexpr (MODE == kPaged) {
        // the sequence's cache length; its Tq queries are its last positions
        U.Tk = min(max(__ldg(P.seq_lens + U.b), 0), P.max_seq_len);
        U.q_offset = U.Tk - P.Tq;  // rows at negative positions see no key
    } else {
        U.Tk = P.Tk;
        U.q_offset = P.q_offset;
    }
    int64_t lo_a, hi_a, lo_b, hi_b;
    visible_range_tk(P, U.Tk, (int64_t)U.q_offset, lo_a, hi_a);
    visible_range_tk(P, U.Tk, (int64_t)U.q_offset + P.Tq - 1, lo_b, hi_b);
    const int64_t klo = lo_a, khi = hi_b > hi_a ? hi_b : hi_a;
    U.t_begin = 0;
    U.n_tiles = 0;
    if (khi > klo) {
        const int tb = (int)(klo / kBN), te = (int)((khi + kBN - 1) / kBN);
        const int chunk = (int)P.fd_splits.div((uint32_t)(te - tb + P.splits - 1));
        const int b0 = tb + rank * chunk, b1 = min(te, b0 + chunk);
        if (b1 > b0) {
            U.t_begin = b0;
            U.n_tiles = b1 - b0;
        }
    }
    return U;
}

template <int MODE>
__device__ __forceinline__ Unit get_unit(const Params &P, int u) {
    if constexpr (is_packed(MODE))
        return decode_unit<MODE>(P);
    else
        return make_unit<MODE>(P, u);
}

// Snake order over groups: round r gives group g unit r*G + g (r even) or
// r*G + G-1-g (r odd); -1 past the end.
struct Schedule {
    int units, groups, group;
    __device__ __forceinline__ int unit_at(int r) const {
        const int u = r * groups + ((r & 1) ? groups - 1 - group : group);
        return u < units ? u : -1;
    }
};

template <int MODE>
__device__ __forceinline__ Schedule make_schedule(const Params &P) {
    if constexpr (is_packed(MODE)) return Schedule{1, 1, 0};  // one unit per CTA
    const int nqt = (P.Tq + kBM - 1) / kBM;
    return Schedule{nqt * P.B * P.Hq, (int)gridDim.x, (int)blockIdx.x};
}

// Position in the K/V ring: stage index and the parity of its current use.
// Stages are produced and consumed strictly in order, so both sides walk the
// ring with a running position.
struct RingPos {
    int st = 0;
    uint32_t ph = 0;
    template <int kStages>
    __device__ __forceinline__ void advance() {
        if (++st == kStages) {
            st = 0;
            ph ^= 1u;
        }
    }
};

// Shared-memory descriptors kept as 32-bit halves: the start-address field
// sits in the low half, and every operand address used here stays below
// 256 KB, so stepping through a tile is a 32-bit add of (offset >> 4).
struct Desc {
    uint32_t lo, hi;
};

__device__ __forceinline__ Desc make_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    const uint64_t d = smem_desc_sw128(saddr, lbo, sbo);
    return Desc{(uint32_t)d, (uint32_t)(d >> 32)};
}

// S = Q K^T over d in 32-byte K steps: D/16 MMAs of 128 x 128 x 16 (bf16) or
// D/32 of 128 x 128 x 32 (e4m3).  Q and K are K-major with the 128-byte
// swizzle: a step advances 32 bytes inside a 128-byte box row, and every
// fourth step jumps to the next box.  issue_qk_steps issues steps [K0, K1)
// (step 0 overwrites the accumulator), so that S can be issued in two halves
// of d.
template <int D, int MODE, int K0, int K1>
__device__ __forceinline__ void issue_qk_steps(uint32_t d_tmem, Desc q, Desc k) {
    constexpr bool kF8 = elem_bytes(MODE) == 1;
    constexpr uint32_t kId = kF8 ? idesc_e4m3_f32(kBM, kBN, 0, 0) : idesc_bf16_f32(kBM, kBN, 0, 0);
#pragma unroll
    for (int kk = K0; kk < K1; ++kk) {
        const uint32_t oq = ((kk >> 2) * (kBM * kSwRowBytes) + (kk & 3) * 32) >> 4;
        const uint32_t ok = ((kk >> 2) * (kBN * kSwRowBytes) + (kk & 3) * 32) >> 4;
        if constexpr (kF8) {
            if (kk == 0)
                mma_ss_f8_c<0>(d_tmem, q.lo + oq, q.hi, k.lo + ok, k.hi, kId);
            else
                mma_ss_f8_c<1>(d_tmem, q.lo + oq, q.hi, k.lo + ok, k.hi, kId);
        } else {
            if (kk == 0)
                mma_ss_c<0>(d_tmem, q.lo + oq, q.hi, k.lo + ok, k.hi, kId);
            else
                mma_ss_c<1>(d_tmem, q.lo + oq, q.hi, k.lo + ok, k.hi, kId);
        }
    }
}

template <int D, int MODE>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, Desc q, Desc k) {
    issue_qk_steps<D, MODE, 0, D * elem_bytes(MODE) / 32>(d_tmem, q, k);
}

// O += P V over the 128 keys of a tile, 32 bytes of keys per step: 8 MMAs of
// 128 x D x 16 (bf16) or 4 of 128 x D x 32 (e4m3), P from tensor memory (8
// columns per step: bf16 pairs or e4m3 quads), V MN-major: a step's keys are
// whole 8-row swizzle atoms, the next 128 bytes of value columns one TMA box
// further on.
template <int D, int MODE>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, Desc v, uint32_t accumulate) {
    constexpr bool kF8 = elem_bytes(MODE) == 1;
    constexpr int kKeys = 32 / elem_bytes(MODE);  // keys per step
    constexpr uint32_t kId = kF8 ? idesc_e4m3_f32(kBM, D, 0, 1) : idesc_bf16_f32(kBM, D, 0, 1);
    if constexpr (kF8) {
        mma_ts_f8_r(o_tmem, p_tmem, v.lo, v.hi, kId, accumulate);
#pragma unroll
        for (int kk = 1; kk < kBN / kKeys; ++kk)
            mma_ts_f8_c<1>(o_tmem, p_tmem + kk * 8, v.lo + ((kk * kKeys * kSwRowBytes) >> 4), v.hi, kId);
    } else {
        mma_ts_r(o_tmem, p_tmem, v.lo, v.hi, kId, accumulate);
#pragma unroll
        for (int kk = 1; kk < kBN / kKeys; ++kk)
            mma_ts_c<1>(o_tmem, p_tmem + kk * 8, v.lo + ((kk * kKeys * kSwRowBytes) >> 4), v.hi, kId);
    }
}

// TMA producer (one thread).  Per unit: K_0 and K_1, then Q once the previous
// unit's last S has released the Q buffer, then V_j and K_{j+2} in turn, each
// into its own ring.
template <int D, int MODE>
__device__ __forceinline__ void producer_role(const CUtensorMap &tmQ, const CUtensorMap &tmK, const CUtensorMap &tmV,
                                              const Params &P, uint8_t *smem, Barriers &bar) {
    using L = SmemLayout<D, MODE>;
    volatile int *abort = &bar.abort;
    const Schedule sched = make_schedule<MODE>(P);
    // The first unit's lookup reads kernel parameters only (not with per-
    // sequence lengths, which are device data), so it runs before the
    // dependency wait: the first loads issue as soon as the previous grid's
    // writes are visible.
    constexpr bool kParamUnits = !is_varlen(MODE) && MODE != kPaged;
    Unit first{};
    if constexpr (kParamUnits) {
        const int u0 = sched.unit_at(0);
        if (u0 >= 0) first = get_unit<MODE>(P, u0);
    }
    // With half the SMs or more left free, a call's CTAs start while the
    // previous grid still runs (programmatic dependent launch) and then wait
    // for it; meanwhile the first unit's Q and first K and V tiles are
    // requested into L2, so that its first loads after the wait hit there.
    // A prefetch changes no value: data the previous grid writes later
    // replaces what L2 holds.
    if constexpr (is_prefill(MODE)) {
        if (P.prefetch_l2 && first.n_tiles > 0) {
#pragma unroll
            for (int c = 0; c < L::kBoxes; ++c) tma_prefetch_l2_4d(&tmQ, c * L::kBoxCols, first.r0, first.h, first.b);
            const int nt = first.n_tiles < kPrefetchTiles ? first.n_tiles : kPrefetchTiles;
            for (int t = 0; t < nt; ++t) {
                const int key0 = (first.t_begin + t) * kBN;
#pragma unroll
                for (int c = 0; c < L::kBoxes; ++c) {
                    tma_prefetch_l2_4d(&tmK, c * L::kBoxCols, key0, first.g, first.b);
                    tma_prefetch_l2_4d(&tmV, c * L::kBoxCols, key0, first.g, first.b);
                }
            }
        }
    }
    // The test hook is set by the host before the launch, not by a kernel.
    const bool drop_first_q = blockIdx.x == 0 && *static_cast<volatile int *>(&g_drop_arrive) != 0;
    grid_dependency_wait();
    grid_launch_dependents();
    // Loads issued into each ring so far: a stage has a previous use once
    // the ring has wrapped (kept as counters, not per-stage arrays, so that
    // nothing here lives in local memory).
    int k_loads = 0, v_loads = 0;
    int q_issued = 0;
    RingPos kput, vput;
    bool ok = true;
    bool first_split = false;  // the first S's box-0 loads went to first_lo
    for (int r = 0; ok; ++r) {
        const int u = sched.unit_at(r);
        if (u < 0) break;
        const Unit U = (kParamUnits && r == 0) ? first : get_unit<MODE>(P, u);
        const int n = U.n_tiles;
        if (n == 0) continue;

        // Tile t of the unit into the next stage of a ring; the stage is
        // refilled once every CTA reading it released its previous use.
        auto load_tile = [&](uint32_t ring, int stages, uint64_t *full, uint64_t *empty, int &loads, RingPos &pos,
                             const CUtensorMap *map, int t) -> bool {
            const int st = pos.st;
            if (loads >= stages && !mbar_wait(&empty[st], pos.ph ^ 1u, abort)) return false;
            mbar_arrive_expect_tx(&full[st], L::kKVBytes);  // halves from both CTAs
            const int key0 = (U.t_begin + t) * kBN;
            const int kvb = is_varlen(MODE) ? 0 : U.b;  // varlen tensors have one batch
            if constexpr (MODE == kPaged) {
                // Runs of min(page_size, 128) keys, each from its page; keys
                // past the sequence (or past the table) read page -1: zeros.
                const int run = P.page_size < kBN ? P.page_size : kBN;
                for (int k0 = 0; k0 < kBN; k0 += run) {
                    const int key = key0 + k0;
                    const int blk = key / P.page_size;
                    const int page = (key < U.Tk && blk < P.max_blocks)
                                         ? __ldg(P.block_table + (int64_t)U.b * P.max_blocks + blk)
                                         : -1;
#pragma unroll
                    for (int c = 0; c < L::kBoxes; ++c)
                        tma_load_4d(smem + ring + st * L::kKVBytes + c * (kBN * kSwRowBytes) + k0 * kSwRowBytes, map,
                                    &full[st], c * L::kBoxCols, key % P.page_size, U.g, page);
                }
            } else {
#pragma unroll
            for (int c = 0; c < L::kBoxes; ++c)
                tma_load_4d(smem + ring + st * L::kKVBytes + c * (kBN * kSwRowBytes), map, &full[st],
                            c * L::kBoxCols, U.krow + key0, U.g, kvb);
            }
            ++loads;
            if (++pos.st == stages) {
                pos.st = 0;
                pos.ph ^= 1u;
            }
            return true;
        };
        auto load_k = [&](int t) {
            return load_tile(L::kKRing, L::kStages, bar.k_full, bar.k_empty, k_loads, kput, &tmK, t);
        };
        auto load_v = [&](int t) {
            return load_tile(L::kVRing, L::kVStages, bar.v_full, bar.v_empty, v_loads, vput, &tmV, t);
        };
        // Q of this unit into the Q buffer (the caller has made sure that the
        // previous unit's S MMAs are done with it).
        auto load_q = [&]() {
            if (q_issued == 0 && drop_first_q) {
                // test hook: no Q load, no arrival on q_full
            } else if constexpr (is_packed(MODE)) {
                // [64 columns] x [group heads] x [Tq rows] boxes: group * Tq rows.
                mbar_arrive_expect_tx(&bar.q_full, (uint32_t)(L::kBoxes * P.group * P.Tq) * kSwRowBytes);
#pragma unroll
                for (int c = 0; c < L::kBoxes; ++c)
                    tma_load_5d(smem + L::kQ + c * (kBM * kSwRowBytes), &tmQ, &bar.q_full, c * L::kBoxCols, 0, 0, U.g,
                                U.b);
            } else {
                mbar_arrive_expect_tx(&bar.q_full, L::kQBytes);
#pragma unroll
                for (int c = 0; c < L::kBoxes; ++c)
                    tma_load_4d(smem + L::kQ + c * (kBM * kSwRowBytes), &tmQ, &bar.q_full, c * L::kBoxCols, U.qrow + U.r0, U.h,
                                is_varlen(MODE) ? 0 : U.b);
            }
            ++q_issued;
        };
        int k_next = 2;  // the unit's next K tile to load
        if (q_issued == 0) {
            // The CTA's first unit: Q first, as its first S needs Q and K_0
            // and all three come from DRAM.  A short unit (up to 16 key
            // tiles) also sends K_2 out before V_0, which is needed only
            // after the first softmax: its S chain is its critical path.
            if constexpr (split_first_s<D, MODE>()) {
              if (!drop_first_q) {
                // Column box 0 of Q and K_0 on first_lo, box 1 on the usual
                // barriers (stage 0 of the K ring, never used before).
                constexpr uint32_t kBox = kBM * kSwRowBytes;
                static_assert(kBN == kBM && L::kBoxes == 2 && L::kQBytes == 2 * kBox && L::kKVBytes == 2 * kBox,
                              "two boxes per Q and K tile");
                const int key0 = U.t_begin * kBN;
                mbar_arrive_expect_tx(&bar.first_lo, 2 * kBox);
                mbar_arrive_expect_tx(&bar.q_full, kBox);
                mbar_arrive_expect_tx(&bar.k_full[0], kBox);
                tma_load_4d(smem + L::kQ, &tmQ, &bar.first_lo, 0, U.r0, U.h, U.b);
                tma_load_4d(smem + L::kKRing, &tmK, &bar.first_lo, 0, key0, U.g, U.b);
                tma_load_4d(smem + L::kQ + kBox, &tmQ, &bar.q_full, L::kBoxCols, U.r0, U.h, U.b);
                tma_load_4d(smem + L::kKRing + kBox, &tmK, &bar.k_full[0], L::kBoxCols, key0, U.g, U.b);
                ++q_issued;
                ++k_loads;
                kput.st = 1;  // stage 0 taken (kStages >= 2)
                first_split = true;
              }
            }
            if (!first_split) {
                load_q();
                if (!(ok = load_k(0))) break;
            }
            if (n > 1 && !(ok = load_k(1))) break;
            if (n > 2 && n <= 16 && L::kStages >= 3) {
                if (!(ok = load_k(2))) break;
                k_next = 3;
            }
        } else {
            // K_0 and K_1 first: Q waits for the previous unit's last S.
            if (!(ok = load_k(0))) break;
            if (n > 1 && !(ok = load_k(1))) break;
            if (!(ok = mbar_wait(&bar.q_empty, (q_issued - 1) & 1, abort))) break;
            load_q();
        }
        for (int j = 0; j < n && ok; ++j) {
            ok = load_v(j);
            if (ok && j + 2 < n && j + 2 >= k_next) ok = load_k(j + 2);
        }
    }
    if (*abort) {
        // Drain: every copy issued above lands before shared memory goes away.
        int never = 0;
        if (q_issued > 0) mbar_wait(&bar.q_full, (q_issued - 1) & 1, &never, 200000000ull);
        if (first_split) mbar_wait(&bar.first_lo, 0, &never, 200000000ull);
        // Stage s of a ring of S stages after n loads was used (n + S - 1 - s) / S times.
        for (int s = 0; s < L::kStages; ++s) {
            const int ku = (k_loads + L::kStages - 1 - s) / L::kStages;
            if (ku > 0) mbar_wait(&bar.k_full[s], (ku - 1) & 1, &never, 200000000ull);
        }
        for (int s = 0; s < L::kVStages; ++s) {
            const int vu = (v_loads + L::kVStages - 1 - s) / L::kVStages;
            if (vu > 0) mbar_wait(&bar.v_full[s], (vu - 1) & 1, &never, 200000000ull);
        }
    }
}

// The tensor core is fed by two issuing threads, so that the barrier work of
// one (waits and commits, a few hundred cycles each, during which a single
// issuer's queue of two or so MMAs runs dry) is covered by the other's MMAs.
// Tile k of the CTA's walk (k counts across units) uses S buffer k % 3:
//   QK issuer   S_k = Q K_k^T into buffer k % 3 once O += P_{k-3} V_{k-3}
//               (the buffer's previous content) has completed
//   PV issuer   O += P_k V_k once the softmax warps have written P_k
// The QK issuer runs up to two tiles ahead, so the softmax warps find the
// next S ready.  Each ring has one reader per CTA, so stage releases cannot
// cross phases.


template <int D, int MODE>
__device__ __forceinline__ void qk_role(const Params &P, uint8_t *smem, Barriers &bar, uint32_t tbase) {
    using L = SmemLayout<D, MODE>;
    volatile int *abort = &bar.abort;
    const Schedule sched = make_schedule<MODE>(P);
    const Desc qd = make_desc(smem_u32(smem + L::kQ), 16, 1024);
    const Desc k0 = make_desc(smem_u32(smem + L::kKRing), 16, 1024);
    constexpr uint32_t kTileUnits = L::kKVBytes >> 4;  // one stage, in descriptor units
    RingPos take;
    RingPos sb;              // S buffer of the next tile and the parity of its use
    bool first_use = true;   // no buffer has been used yet on this pass
    int units = 0;           // non-empty units before this one
    bool ok = true;
    // The producer splits the first S's loads unless the test hook drops
    // that Q (the same host-set value it reads).
    const bool first_split =
        split_first_s<D, MODE>() && !(blockIdx.x == 0 && *static_cast<volatile int *>(&g_drop_arrive) != 0);
    constexpr int kSteps = D * elem_bytes(MODE) / 32;
    for (int r = 0; ok; ++r) {
        const int u = sched.unit_at(r);
        if (u < 0) break;
        const int n = get_unit<MODE>(P, u).n_tiles;
        if (n == 0) continue;
        const bool halves = first_split && units == 0;  // this unit's first S in two halves
        if (!halves && !(ok = mbar_wait(&bar.q_full, units & 1, abort))) break;
        for (int j = 0; j < n; ++j) {
            const int b = sb.st;
            if (halves && j == 0) {
                if (!(ok = mbar_wait(&bar.first_lo, 0, abort))) break;
                tc_fence_after();
                issue_qk_steps<D, MODE, 0, kSteps / 2>(tbase + col_s(b), qd, Desc{k0.lo + take.st * kTileUnits, k0.hi});
                if (!(ok = mbar_wait(&bar.q_full, 0, abort))) break;
            }
            if (!(ok = mbar_wait(&bar.k_full[take.st], take.ph, abort))) break;
            // the buffer's previous use: O += P V from it completed
            if (!first_use && !(ok = mbar_wait(&bar.o_done[b], sb.ph ^ 1u, abort))) break;
            tc_fence_after();
            if (halves && j == 0)
                issue_qk_steps<D, MODE, kSteps / 2, kSteps>(tbase + col_s(b), qd,
                                                             Desc{k0.lo + take.st * kTileUnits, k0.hi});
            else
                issue_qk<D, MODE>(tbase + col_s(b), qd, Desc{k0.lo + take.st * kTileUnits, k0.hi});
            mma_commit(&bar.s_full[b]);
            if (j + 1 == n) mma_commit(&bar.q_empty);  // the unit's last S is issued
            mma_commit(&bar.k_empty[take.st]);
            take.template advance<L::kStages>();
            sb.template advance<kSBufs>();
            if (sb.st == 0) first_use = false;
        }
        ++units;
    }
    // Every MMA issued above completes before tensor memory is freed.
    mma_commit(&bar.drain[0]);
    int never = 0;
    mbar_wait(&bar.drain[0], 0, &never, 200000000ull);
}

// The first O += P_0 V_0 of a unit overwrites O; the softmax warps read the
// previous unit's O before they release P_0, so O is free by then.
template <int D, int MODE>
__device__ __forceinline__ void pv_role(const Params &P, uint8_t *smem, Barriers &bar, uint32_t tbase) {
    using L = SmemLayout<D, MODE>;
    volatile int *abort = &bar.abort;
    const Schedule sched = make_schedule<MODE>(P);
    const Desc v0 = make_desc(smem_u32(smem + L::kVRing), kBN * kSwRowBytes, 1024);
    constexpr uint32_t kTileUnits = L::kKVBytes >> 4;
    RingPos take;
    RingPos sb;  // S buffer holding P of the next tile and the parity of its use
    bool ok = true;
    for (int r = 0; ok; ++r) {
        const int u = sched.unit_at(r);
        if (u < 0) break;
        const int n = get_unit<MODE>(P, u).n_tiles;
        if (n == 0) continue;
        for (int j = 0; j < n; ++j) {
            const int b = sb.st;
            if (!(ok = mbar_wait(&bar.v_full[take.st], take.ph, abort))) break;
            if (!(ok = mbar_wait(&bar.p_full[b], sb.ph, abort))) break;
            tc_fence_after();
            issue_pv<D, MODE>(tbase + kColO, tbase + col_s(b), Desc{v0.lo + take.st * kTileUnits, v0.hi},
                              j > 0 ? 1u : 0u);
            mma_commit(&bar.o_done[b]);
            if (j + 1 == n) mma_commit(&bar.o_final);
            mma_commit(&bar.v_empty[take.st]);
            take.template advance<L::kVStages>();
            sb.template advance<kSBufs>();
        }
    }
    mma_commit(&bar.drain[1]);
    int never = 0;
    mbar_wait(&bar.drain[1], 0, &never, 200000000ull);
}

// Softmax warps 0-7 and epilogue: two threads per query row.  Warp w covers
// the 16 tensor-memory lanes from 32 (w % 4) + 16 (w / 4); in it lanes l and
// l + 16 hold the same row, the first and second half of each tile's keys and
// of O's columns.  Row max and row sum combine through one shuffle, and the
// two warps on a scheduler partition hide each other's latencies.
template <int D, int MODE>
__device__ __forceinline__ void softmax_role(const CUtensorMap &tmO, const Params &P, uint8_t *smem, Barriers &bar,
                                             uint32_t tbase, int warp, int lane) {
    using L = SmemLayout<D, MODE>;
    constexpr int kHK = kBN / 2;  // keys per thread per tile
    constexpr int kHD = D / 2;    // O columns per thread
    static_assert(kHD == 32 || kHD == 64, "a thread's O columns fill half or all of a 64-column box");
    // Prefill-like mappings bound a boundary tile's maximum by the load's
    // (packed rows, whose tiles are nearly all interior, keep the registers).
    constexpr bool kBoundByLoad = !is_packed(MODE);
    volatile int *abort = &bar.abort;
    const Schedule sched = make_schedule<MODE>(P);
    const int half = lane >> 4;
    const int lane0 = 32 * (warp & 3) + 16 * (warp >> 2);  // first tensor-memory lane of the warp
    const int row = lane0 + (lane & 15);
    const uint32_t lane_off = (uint32_t)lane0 << 16;
    const uint32_t o_addr = tbase + lane_off + kColO;
    const float c = P.scale_log2;
    RingPos sb;     // S buffer of the current tile and the parity of its use
    int units = 0;  // non-empty units before this one
    int eps = 0;    // epilogues before this one
    bool ok = true;

    for (int r = 0; ok; ++r) {
        const int u = sched.unit_at(r);
        if (u < 0) break;
        const Unit U = get_unit<MODE>(P, u);
        const int n = U.n_tiles;
        // The row's query head h and its row i in that head.  Prefill: the
        // unit's head, consecutive rows.  Packed rows: row = i * group + hl
        // (h = g * group + hl), and rows from group * Tq on are padding that
        // sees no key.
        int h = U.h, i = U.r0 + row;
        bool live;  // the row holds a query
        // Keys and query position of the unit's sequence: the call's, or the
        // sequence's own with paged K/V (kernel parameters stay in the
        // constant bank otherwise).
        constexpr bool kSeq = MODE == kPaged || is_varlen(MODE);  // per-sequence lengths
        const int uTk = kSeq ? U.Tk : P.Tk;
        const int uq0 = kSeq ? U.q_offset : P.q_offset;
        const int uTq = is_varlen(MODE) ? U.Tq : P.Tq;
        if (is_varlen(MODE) && U.r0 >= uTq) continue;  // a tile past the sequence's rows
        int64_t p_first = (int64_t)uq0 + U.r0, p_last = (int64_t)uq0 + min(U.r0 + kBM, uTq) - 1;
        if constexpr (is_packed(MODE)) {
            live = row < P.group * P.Tq;
            const int iq = (int)P.fd_group.div((uint32_t)row);  // row = i * group + hl
            const int hl = live ? row - iq * P.group : 0;
            h = U.g * P.group + hl;
            i = live ? iq : 0;
            p_first = uq0;
            p_last = (int64_t)uq0 + P.Tq - 1;
        } else {
            live = i < uTq;
        }
        const int64_t p = (int64_t)uq0 + i;
        // Per-row visible key interval [vlo, vhi) before the additive mask.
        int vlo = 0, vhi = 0;  // within [0, Tk]
        if (is_prefill(MODE) || live) {
            int64_t lo64, hi64;
            visible_range_tk(P, uTk, p, lo64, hi64);
            vlo = (int)lo64;
            vhi = (int)hi64;
        }
        const bool has_sink = P.sinks != nullptr;
        // The sink joins the sum once: in the first CTA of a split key range.
        const bool sink_here =
            has_sink && half == 0 && (is_prefill(MODE) || is_varlen(MODE) || P.fd_splits.mod(blockIdx.x) == 0);
        float m = has_sink ? __ldg(P.sinks + h) * kLog2e : -INFINITY;  // log2 units
        float l = sink_here ? 1.f : 0.f;                                // this thread's share of the sum
        const float *mrow = (!kSeq && P.mask != nullptr && live)
                                ? P.mask + U.b * P.msb + h * P.msh + (int64_t)i * P.msq
                                : nullptr;
        // Tiles j in [ti_lo, ti_hi) are interior: every key visible to every
        // row of the unit, and no additive mask.
        int ti_lo = 0, ti_hi = 0;
        if (P.mask == nullptr && c > 0.f) {
            int64_t hi_key = uTk;                                        // j0 + kBN <= Tk
            if (P.causal && p_first + 1 < hi_key) hi_key = p_first + 1;  // j0 + kBN - 1 <= p_first
            int64_t lo_key = 0;                                          // j0 > p_last - window
            if (P.window > 0 && p_last - P.window + 1 > 0) lo_key = p_last - P.window + 1;
            ti_lo = (int)((lo_key + kBN - 1) / kBN - U.t_begin);
            ti_hi = (int)(hi_key / kBN - U.t_begin);
        }

        for (int j = 0; j < n; ++j) {
            const int b = sb.st;
            const uint32_t s_addr = tbase + lane_off + col_s(b);
            // warp-uniform outcome: the tcgen05.ld/st below are warp-collective
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.s_full[b], sb.ph, abort)))) break;
            tc_fence_after();
            uint32_t sr[kHK];
            // The load also gives the maximum of the thread's raw scores: the
            // row maximum of an interior tile, and a bound on a boundary
            // tile's (masked) one.
            const bool interior = j >= ti_lo && j < ti_hi;  // warp-uniform
            float raw_max = 0.f;
            if (kBoundByLoad || interior)
                raw_max = tmem_load_pair64_max<kHK>(s_addr, sr);
            else
                tmem_load_pair64<kHK>(s_addr, sr);
            float *s = reinterpret_cast<float *>(sr);

            float cs = c;  // multiplier from s[] to log2 units for this tile
            if (!interior) {
                const int k0 = (U.t_begin + j) * kBN + half * kHK;  // this thread's first key
                // The row's visible keys among this thread's: [elo, ehi) (clamped).
                const int elo = min(max(vlo - k0, 0), kHK), ehi = min(max(vhi - k0, 0), kHK);
                const KeyBits kb = key_bits(elo, ehi);
                auto visible = [&](int e) { return kb.has(e); };
                if (mrow != nullptr) {
                    // Additive mask: scores in log2 units; keys past Tk read a
                    // clamped (valid) address and are dropped by the interval.
                    if (P.msk == 1 && k0 + kHK <= P.Tk && (reinterpret_cast<uintptr_t>(mrow + k0) & 15) == 0) {
                        // Contiguous keys, all inside the mask row, 16-byte
                        // aligned: 16 vector loads instead of 64 scalar ones.
                        const float4 *m4 = reinterpret_cast<const float4 *>(mrow + k0);
#pragma unroll
                        for (int q4 = 0; q4 < kHK / 4; ++q4) {
                            const float4 mv = __ldg(m4 + q4);
                            const float mvals[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const int e = 4 * q4 + t;
                                const float x = fmaf(mvals[t], kLog2e, s[e] * c);
                                s[e] = visible(e) ? x : -INFINITY;
                            }
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < kHK; ++e) {
                            const int jj = min(k0 + e, P.Tk - 1);  // (no mask with paged K/V)
                            const float x = fmaf(__ldg(mrow + (int64_t)jj * P.msk), kLog2e, s[e] * c);
                            s[e] = visible(e) ? x : -INFINITY;
                        }
                    }
                    cs = 1.f;
                } else if (c <= 0.f) {
                    // A non-positive scale: scale first so that -inf marks the
                    // keys the row cannot see.
#pragma unroll
                    for (int e = 0; e < kHK; ++e) s[e] = visible(e) ? s[e] * c : -INFINITY;
                    cs = 1.f;
                } else {
                    // Boundary tile: keys outside the row's interval drop to -inf.
#pragma unroll
                    for (int e = 0; e < kHK; ++e) s[e] = visible(e) ? s[e] : -INFINITY;
                }
            }
            float bm;  // tile max of s[] * cs over the whole row, in log2 units
            if (interior) {
                bm = raw_max * cs;
                bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));  // the row's other half
            } else {
                // Without an additive mask (and with c > 0) the masked maximum
                // is at most the raw one times c.  When that bound cannot move
                // m past the threshold below, neither can the masked maximum,
                // and m stays as it would have: the maximum is not needed.
                bool exact = true;
                if constexpr (kBoundByLoad) {
                    // every lane shuffles (mrow differs between rows); the
                    // two lanes of a row share mrow and so the outcome
                    float ub = raw_max * c;
                    ub = fmaxf(ub, __shfl_xor_sync(0xffffffffu, ub, 16));
                    exact = mrow != nullptr || c <= 0.f || ub > m + kRescaleThreshold;
                }
                if (!kBoundByLoad || __any_sync(0xffffffffu, exact)) {
                    static_assert(kHK == 64, "max chains assume 64 keys per thread");
                    float mx[8];  // eight independent chains of three-input max
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) mx[c8] = fmax3(s[c8], s[8 + c8], s[16 + c8]);  // keys 0..23
#pragma unroll
                    for (int e = 24; e < 56; e += 16)  // keys 24..55
#pragma unroll
                        for (int c8 = 0; c8 < 8; ++c8) mx[c8] = fmax3(mx[c8], s[e + c8], s[e + 8 + c8]);
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) mx[c8] = fmaxf(mx[c8], s[56 + c8]);  // keys 56..63
                    bm = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * cs;
                    bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));  // the row's other half
                } else {
                    bm = -INFINITY;  // at most m + threshold: m stays
                }
            }

            // Lazy max: move m only when the tile exceeds it by the threshold
            // (with m = -inf any finite tile max does, and 2^(-inf) = 0).
            float alpha = 1.f;
            if (bm > m + kRescaleThreshold) {
                alpha = ex2_approx(m - bm);
                m = bm;
            }
            const float shift = (m == -INFINITY) ? 0.f : m;
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                // O must hold P_{j-1} V_{j-1} (previous buffer) before it is rescaled.
                const int bp = b == 0 ? kSBufs - 1 : b - 1;
                const uint32_t php = b == 0 ? sb.ph ^ 1u : sb.ph;
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.o_done[bp], php, abort)))) break;
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < kHD; cc += 32) {
                    uint32_t orr[32];
                    tmem_load_pair32<kHD>(o_addr + cc, orr);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float2 v = fmul2(make_float2(__uint_as_float(orr[e]), __uint_as_float(orr[e + 1])),
                                               make_float2(alpha, alpha));
                        orr[e] = __float_as_uint(v.x);
                        orr[e + 1] = __float_as_uint(v.y);
                    }
                    tmem_store_pair32<kHD>(o_addr + cc, orr);
                }
            }

            // p = 2^(s cs - shift), rounded to bf16 pairs (e4m3 quads with
            // e4m3 inputs: p <= 2^8 stays below the format's 448); row sum of
            // the unrounded p in fp32.
            const float2 cs2 = make_float2(cs, cs), nsh2 = make_float2(-shift, -shift);
            float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
            constexpr int kPerWord = 4 / elem_bytes(MODE);  // P elements per 32-bit column
            uint32_t pk[kHK / kPerWord];
#pragma unroll
            for (int e = 0; e < kHK; e += 4) {
                const float2 x0 = ffma2(make_float2(s[e], s[e + 1]), cs2, nsh2);
                const float2 x1 = ffma2(make_float2(s[e + 2], s[e + 3]), cs2, nsh2);
                const float2 p0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
                const float2 p1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
                acc0 = fadd2(acc0, p0);
                acc1 = fadd2(acc1, p1);
                if constexpr (kPerWord == 4) {
                    pk[e / 4] = cvt_e4m3x4(p0.x, p0.y, p1.x, p1.y);
                } else {
                    pk[e / 2] = cvt_bf16x2(p0.x, p0.y);
                    pk[e / 2 + 1] = cvt_bf16x2(p1.x, p1.y);
                    // bf16: the first 32 keys' P goes out while the rest
                    // are computed; one wait below covers both stores.
                    if (e + 4 == kHK / 2) tmem_store_pair16_nowait<kHK / 2>(s_addr, pk);
                }
            }
            // P of keys [64 h, 64 h + 64) into columns [32 h, 32 h + 32) (bf16)
            // or [16 h, 16 h + 16) (e4m3) of the buffer.
            if constexpr (kPerWord == 4) {
                tmem_store_pair16<kHK / 4>(s_addr, pk);
            } else {
                tmem_store_pair16_nowait<kHK / 2>(s_addr + 16, pk + 16);
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.p_full[b]);  // one arrival per warp
            const float2 a = fadd2(acc0, acc1);
            l = fmaf(alpha, l, a.x + a.y);
            sb.template advance<kSBufs>();
        }
        if (!ok) break;

        // Epilogue: o = O / l (0 for an empty row), lse = (m + log2 l) ln 2.
        // O goes out through shared memory and a TMA store: the staging tile
        // is [D / 64 boxes][128 rows][128 bytes] with the 128-byte swizzle
        // (16-byte chunk c of row r at chunk c ^ (r % 8)); rows past Tq are
        // clipped by the store.  The previous unit's store must have read the
        // tile before it is rewritten.  O leaves tensor memory before this
        // thread's warp releases the next unit's P_0 (whose P V overwrites O).
        const float lt = l + __shfl_xor_sync(0xffffffffu, l, 16);
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        if (n > 0) {
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.o_final, units & 1, abort)))) break;
            tc_fence_after();
        }
        if constexpr (MODE == kSplitKv) {
            // This CTA's partial result over its share of the keys into its
            // block of the workspace: unnormalised O, [R rows][D] fp32, then
            // (m, l) per row (R = group * Tq).
            const int S = P.splits, cid = (int)P.fd_splits.div(blockIdx.x), rank = (int)blockIdx.x - cid * S;
            const int R = P.group * P.Tq;
            float *blk = P.ws + ((int64_t)cid * S + rank) * ws_block_floats(R, D);
#pragma unroll
            for (int cc = 0; cc < kHD; cc += 32) {
                uint32_t ov[32];
                if (n > 0) {
                    tmem_load_pair32<kHD>(o_addr + cc, ov);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = 0u;
                }
                if (live) {
                    float4 *dst = reinterpret_cast<float4 *>(blk + row * D + half * kHD + cc);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        __stcg(dst + e, make_float4(__uint_as_float(ov[4 * e]), __uint_as_float(ov[4 * e + 1]),
                                                    __uint_as_float(ov[4 * e + 2]), __uint_as_float(ov[4 * e + 3])));
                }
            }
            if (n > 0) tc_fence_before();
            if (live && half == 0) __stcg(reinterpret_cast<float2 *>(blk + R * D) + row, make_float2(m, lt));
        } else if constexpr (MODE == kDecode || MODE == kPaged) {
            // This CTA's partial result over its share of the keys:
            // unnormalised O (fp32, rows of kOPartStride floats) and (m, l) per
            // row, in the K/V ring space (no copy or MMA is in flight any
            // more).  The CTAs of the cluster merge them after the roles end.
            float *opart = reinterpret_cast<float *>(smem + L::kKRing);
            float2 *stats = reinterpret_cast<float2 *>(smem + L::kVRing);
#pragma unroll
            for (int cc = 0; cc < kHD; cc += 32) {
                uint32_t ov[32];
                if (n > 0) {
                    tmem_load_pair32<kHD>(o_addr + cc, ov);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = 0u;
                }
                if (live) {
                    float4 *dst = reinterpret_cast<float4 *>(opart + row * L::kOPartStride + half * kHD + cc);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        dst[e] = make_float4(__uint_as_float(ov[4 * e]), __uint_as_float(ov[4 * e + 1]),
                                             __uint_as_float(ov[4 * e + 2]), __uint_as_float(ov[4 * e + 3]));
                }
            }
            if (n > 0) tc_fence_before();
            if (live && half == 0) stats[row] = make_float2(m, lt);
        } else if constexpr (is_varlen(MODE)) {
            // The sequence's rows only (a 128-row store would reach into the
            // next sequence): this thread's half of the row, 16-byte stores.
#pragma unroll
            for (int cc = 0; cc < kHD; cc += 32) {
                uint32_t ov[32];
                if (n > 0) {
                    tmem_load_pair32<kHD>(o_addr + cc, ov);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = 0u;
                }
                if (live) {
                    const int col0 = half * kHD + cc;  // columns [d, D) are padding: not written
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(P.o) + (int64_t)U.h * P.o_sh +
                                                           (int64_t)(U.qrow + i) * P.o_st + col0);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint32_t w[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            w[k] = cvt_bf16x2(__uint_as_float(ov[8 * e + 2 * k]) * inv,
                                              __uint_as_float(ov[8 * e + 2 * k + 1]) * inv);
                        if (col0 + 8 * e < P.d) dst[e] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            if (n > 0) tc_fence_before();
            if (live && P.lse != nullptr && half == 0)
                P.lse[(int64_t)U.h * P.total_q + U.qrow + i] = lt > 0.f ? (m + lg2_approx(lt)) * kLn2 : -INFINITY;
        } else {
            if (threadIdx.x == 0) {
                bulk_wait_read_all();
                mbar_arrive(&bar.ep_free);
            }
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.ep_free, eps & 1, abort)))) break;
            {
                const int col0 = half * kHD;  // this thread's first O column
                uint8_t *box = smem + L::kOStage + (col0 / 64) * (kBM * kSwRowBytes) + row * kSwRowBytes;
                // All of the thread's O columns in one tensor-memory load.
                uint32_t ov[kHD];
                if (n > 0) {
                    if constexpr (kHD == 64)
                        tmem_load_pair64<kHD>(o_addr, ov);
                    else
                        tmem_load_pair32<kHD>(o_addr, ov);
                    tc_fence_before();
                } else {
#pragma unroll
                    for (int e = 0; e < kHD; ++e) ov[e] = 0u;
                }
#pragma unroll
                for (int e = 0; e < kHD / 8; ++e) {
                    uint32_t w[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        w[k] = cvt_bf16x2(__uint_as_float(ov[8 * e + 2 * k]) * inv,
                                          __uint_as_float(ov[8 * e + 2 * k + 1]) * inv);
                    const int chunk = ((col0 % 64) / 8 + e) ^ (row & 7);
                    *reinterpret_cast<uint4 *>(box + chunk * 16) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_proxy_async_smem();  // the TMA store reads what this thread wrote
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.ep_full);
            if (warp == 0) {
                if (!(ok = __all_sync(0xffffffffu, mbar_wait(&bar.ep_full, eps & 1, abort)))) break;
                if (lane == 0) {
#pragma unroll
                    for (int cb = 0; cb < L::kOBoxes; ++cb)
                        tma_store_4d(&tmO, smem + L::kOStage + cb * (kBM * kSwRowBytes), cb * 64, U.r0, U.h, U.b);
                    bulk_commit_group();
                }
            }
            ++eps;
            if (i < P.Tq && P.lse != nullptr && half == 0)
                P.lse[(int64_t)U.bh * P.Tq + i] = lt > 0.f ? (m + lg2_approx(lt)) * kLn2 : -INFINITY;
        }
        if (n > 0) ++units;
    }
    // The stores have read the staging tile before shared memory goes away
    // (their global writes are complete when the grid is).
    if (threadIdx.x == 0) bulk_wait_read_all();
}

// Packed-row split merge (after every CTA of the cluster wrote its partial):
// for each (row, column), with (m_s, l_s, O_s) the partials of the cluster's
// S CTAs,  M = max m_s,  w_s = 2^(m_s - M),  o = sum w_s O_s / sum w_s l_s,
// lse = (M + log2 sum w_s l_s) ln 2 -- the rescale of the online softmax
// applied across key ranges.  With one CTA (w = 1) this is the plain epilogue,
// bit for bit.  The (row, column) pairs are spread over all threads of the
// cluster; o and lse go straight to global memory.
template <int D>
__device__ __forceinline__ void merge_partials(const Params &P, uint8_t *smem) {
    using L = SmemLayout<D, kDecode>;
    const int S = P.splits, cid = (int)P.fd_splits.div(blockIdx.x), rank = (int)blockIdx.x - cid * S;
    const int R = P.group * P.Tq;
    const uint32_t op0 = smem_u32(smem + L::kKRing), st0 = smem_u32(smem + L::kVRing);
    const int b = (int)P.fd_hkv.div((uint32_t)cid), g = cid - b * P.Hkv;
    for (int e = rank * kThreads + (int)threadIdx.x; e < R * P.d; e += S * kThreads) {
        const int row = (int)P.fd_d.div((uint32_t)e), col = e - row * P.d;
        const int i = (int)P.fd_group.div((uint32_t)row), h = g * P.group + (row - i * P.group);  // row = i * group + (h - g group)
        float M = -INFINITY;
        for (int sp = 0; sp < S; ++sp) M = fmaxf(M, ld_cluster_f32(map_to_rank(st0 + row * 8, sp)));
        float lsum = 0.f, acc = 0.f;
        for (int sp = 0; sp < S; ++sp) {
            const float2 ml = ld_cluster_f32x2(map_to_rank(st0 + row * 8, sp));
            const float w = ml.x == M ? 1.f : ex2_approx(ml.x - M);  // 0 for an empty partial
            const float ov = ld_cluster_f32(map_to_rank(op0 + (row * L::kOPartStride + col) * 4, sp));
            lsum = sp == 0 ? w * ml.y : fmaf(w, ml.y, lsum);
            acc = sp == 0 ? w * ov : fmaf(w, ov, acc);
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        static_cast<__nv_bfloat16 *>(P.o)[b * P.o_sb + h * P.o_sh + i * P.o_st + col] = __float2bfloat16_rn(acc * inv);
        if (col == 0 && P.lse != nullptr)
            P.lse[((int64_t)b * P.Hq + h) * P.Tq + i] = lsum > 0.f ? (M + lg2_approx(lsum)) * kLn2 : -INFINITY;
    }
}

// The split-KV merge through global memory, run by the last CTA of a KV head
// to finish: the same rescale as merge_partials over the S partials of the
// workspace (M = max m_s, w_s = 2^(m_s - M), o = sum w_s O_s / sum w_s l_s,
// lse = (M + log2 sum w_s l_s) ln 2), the partials taken in split order.
// The per-row weights are formed once (the (row, split) pairs spread over
// the threads, the reductions in split order in shared memory, over the K
// ring), then every thread merges 4 columns of a row at a time.  The
// workspace was written by other CTAs of this grid: it is read through L2
// (ld.global.cg), never through L1.
template <int D>
__device__ __forceinline__ void merge_partials_ws(const Params &P, uint8_t *smem) {
    using L = SmemLayout<D, kSplitKv>;
    const int S = P.splits, cid = (int)P.fd_splits.div(blockIdx.x);
    const int R = P.group * P.Tq;
    const int b = (int)P.fd_hkv.div((uint32_t)cid), g = cid - b * P.Hkv;
    const int64_t bstride = ws_block_floats(R, D);
    const float *blk0 = P.ws + (int64_t)cid * S * bstride;
    float *mls = reinterpret_cast<float *>(smem + L::kKRing);  // [S][R] (m, l) pairs, then weights [S][R]
    float *wts = mls + 2 * S * R;
    float *rowM = wts + S * R, *rowL = rowM + R;
    for (int t = (int)threadIdx.x; t < S * R; t += kThreads) {
        const int sp = t / R, row = t - sp * R;
        const float2 ml = __ldcg(reinterpret_cast<const float2 *>(blk0 + sp * bstride + R * D) + row);
        mls[2 * t] = ml.x;
        mls[2 * t + 1] = ml.y;
    }
    __syncthreads();
    for (int row = (int)threadIdx.x; row < R; row += kThreads) {
        float M = -INFINITY;
        for (int sp = 0; sp < S; ++sp) M = fmaxf(M, mls[2 * (sp * R + row)]);
        float lsum = 0.f;
        for (int sp = 0; sp < S; ++sp) {
            const float m = mls[2 * (sp * R + row)], l = mls[2 * (sp * R + row) + 1];
            const float w = m == M ? 1.f : ex2_approx(m - M);  // 0 for an empty partial
            wts[sp * R + row] = w;
            lsum = sp == 0 ? w * l : fmaf(w, l, lsum);
        }
        rowM[row] = M;
        rowL[row] = lsum;
    }
    __syncthreads();
    const int q4 = P.d / 4;  // 4-column groups of a row (d is a multiple of 8)
    for (int e = (int)threadIdx.x; e < R * q4; e += kThreads) {
        const int row = e / q4, col = 4 * (e - row * q4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int sp = 0; sp < S; ++sp) {
            const float w = wts[sp * R + row];
            const float4 ov = __ldcg(reinterpret_cast<const float4 *>(blk0 + sp * bstride + row * D + col));
            acc = sp == 0 ? make_float4(w * ov.x, w * ov.y, w * ov.z, w * ov.w)
                          : make_float4(fmaf(w, ov.x, acc.x), fmaf(w, ov.y, acc.y), fmaf(w, ov.z, acc.z),
                                        fmaf(w, ov.w, acc.w));
        }
        const float lsum = rowL[row];
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        const int i = (int)P.fd_group.div((uint32_t)row), h = g * P.group + (row - i * P.group);
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(P.o) + b * P.o_sb + h * P.o_sh + (int64_t)i * P.o_st + col;
        const uint2 w2 = make_uint2(cvt_bf16x2(acc.x * inv, acc.y * inv), cvt_bf16x2(acc.z * inv, acc.w * inv));
        *reinterpret_cast<uint2 *>(dst) = w2;
        if (col == 0 && P.lse != nullptr)
            P.lse[((int64_t)b * P.Hq + h) * P.Tq + i] = lsum > 0.f ? (rowM[row] + lg2_approx(lsum)) * kLn2 : -INFINITY;
    }
}

template <int D, int MODE>
__global__ void __launch_bounds__(threads_for(MODE), 1)
    fa_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                       const Params P) {
    using L = SmemLayout<D, MODE>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Barriers &bar = *reinterpret_cast<Barriers *>(smem + L::kBar);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&bar.q_full, 1);
        mbar_init(&bar.q_empty, 1);
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(&bar.k_full[s], 1);
            mbar_init(&bar.v_full[s], 1);
            mbar_init(&bar.k_empty[s], 1);
            mbar_init(&bar.v_empty[s], 1);
        }
        for (int s = 0; s < kSBufs; ++s) {
            mbar_init(&bar.s_full[s], 1);
            mbar_init(&bar.p_full[s], kSoftmaxWarps);  // one arrival per softmax warp
            mbar_init(&bar.o_done[s], 1);
        }
        mbar_init(&bar.o_final, 1);
        mbar_init(&bar.ep_free, 1);
        mbar_init(&bar.ep_full, kSoftmaxWarps);
        mbar_init(&bar.drain[0], 1);
        mbar_init(&bar.drain[1], 1);
        mbar_init(&bar.first_lo, 1);
        bar.abort = 0;
        mbar_init_fence();
    }
    if (warp == kWarpQk) {
        tmem_alloc(&bar.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kWarpTma && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmO);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = bar.tmem_base;
    // Inputs may come from the previous kernel in the stream, and outputs may
    // still be read by it: every thread passes the dependency wait before its
    // first global access (the producer inside its role, after the first
    // unit's lookup).
    if (warp >= kWarpTma) {  // warps 8-10 issue (one lane each); warp 11 (prefill) idles
        if constexpr (is_prefill(MODE)) regs_decrease<kRegsIssuePrefill>();
        if (warp == kWarpTma && lane == 0) {
            producer_role<D, MODE>(tmQ, tmK, tmV, P, smem, bar);
        } else {
            grid_dependency_wait();
            grid_launch_dependents();
            if (warp == kWarpQk) {
                if (lane == 0) qk_role<D, MODE>(P, smem, bar, tbase);
            } else if (warp == kWarpPv) {
                if (lane == 0) pv_role<D, MODE>(P, smem, bar, tbase);
            }
        }
    } else {
        if constexpr (is_prefill(MODE)) regs_increase<kRegsSoftmaxPrefill>();
        grid_dependency_wait();
        grid_launch_dependents();
        softmax_role<D, MODE>(tmO, P, smem, bar, tbase, warp, lane);
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (MODE == kDecode || MODE == kPaged) {
        cluster_sync();  // every CTA's partial is written
        if (!bar.abort) merge_partials<D>(P, smem);
        cluster_sync();  // no CTA leaves while a peer reads its partial
    } else if constexpr (MODE == kSplitKv) {
        // Every thread's workspace writes are visible device-wide before the
        // CTA is counted; the CTA that completes its KV head's count merges.
        __threadfence();
        __syncthreads();
        const int cid = (int)P.fd_splits.div(blockIdx.x);
        if (threadIdx.x == 0) bar.last = atomicAdd(P.ws_cnt + cid, 1u) == (unsigned)(P.splits - 1) ? 1 : 0;
        __syncthreads();
        if (bar.last) {
            __threadfence();
            if (!bar.abort) merge_partials_ws<D>(P, smem);
        }
    }
    if (bar.abort && threadIdx.x == 0) atomicOr(&g_watchdog, 1u);
    if (warp == kWarpQk) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

// ------------------------------------------------------------------ host

// The query rows of one KV group as the 5-D map (d, group, Tq, Hkv, B): head
// g * group + hl at row i is coordinate (., hl, i, g, b), and one box of 64
// columns x group x Tq lands in shared memory as rows i * group + hl.
bool make_packed_map(EncodeTiledFn enc, CUtensorMap *map, const void *base, const Params &P, int64_t st, int64_t sh,
                     int64_t sb) {
    const int64_t dims[5] = {P.d, P.group, P.Tq, P.Hkv, P.B}, strides[5] = {1, sh, st, sh * P.group, sb};
    const uint32_t box[5] = {64, (uint32_t)P.group, (uint32_t)P.Tq, 1, 1};
    return encode_map(enc, map, base, 5, dims, strides, box, 2);
}

// The K and V maps; with Tk == 0 no key tile is ever loaded and the maps only
// need to be valid (they then describe q).
bool make_kv_maps(EncodeTiledFn enc, CUtensorMap *tk, CUtensorMap *tv, const Params &P, int box_rows, int elem = 2) {
    if (P.Tk == 0)
        return make_map(enc, tk, P.q, P.d, 1, 1, 1, P.q_st, P.q_sh, P.q_sb, box_rows, elem) &&
               make_map(enc, tv, P.q, P.d, 1, 1, 1, P.q_st, P.q_sh, P.q_sb, box_rows, elem);
    return make_map(enc, tk, P.k, P.d, P.Tk, P.Hkv, P.B, P.k_st, P.k_sh, P.k_sb, box_rows, elem) &&
           make_map(enc, tv, P.v, P.d, P.Tk, P.Hkv, P.B, P.v_st, P.v_sh, P.v_sb, box_rows, elem);
}

template <int D, int MODE>
cudaError_t launch_d(const Params &P0, cudaStream_t stream) {
    Params P = P0;
    P.fd_per_qt = FastDiv::make((uint32_t)(P.B * P.Hq));
    P.fd_heads = FastDiv::make((uint32_t)P.Hq);
    P.fd_group = FastDiv::make((uint32_t)P.group);
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    CUtensorMap tq, tk, tv, to;
    // The maps carry the true head dimension d <= D: columns [d, D) of Q, K
    // and V load as zero (leaving S exact and O's extra columns zero), and the
    // O store drops them.  A variable-length batch is one [total, H, d]
    // tensor (a batch of one) with the sequences along the rows.
    bool ok;
    constexpr int kE = elem_bytes(MODE);  // Q, K and V in bf16 or e4m3; O is bf16
    if (is_varlen(MODE)) {
        ok = make_map(enc, &tq, P.q, P.d, P.total_q, P.Hq, 1, P.q_st, P.q_sh, 0, kBM, kE) &&
             make_map(enc, &to, P.o, P.d, P.total_q, P.Hq, 1, P.o_st, P.o_sh, 0, kBM);
        if (P.total_k > 0)
            ok = ok && make_map(enc, &tk, P.k, P.d, P.total_k, P.Hkv, 1, P.k_st, P.k_sh, 0, kBN, kE) &&
                 make_map(enc, &tv, P.v, P.d, P.total_k, P.Hkv, 1, P.v_st, P.v_sh, 0, kBN, kE);
        else
            ok = ok && make_map(enc, &tk, P.q, P.d, 1, 1, 1, P.q_st, P.q_sh, 0, kBN, kE) &&
                 make_map(enc, &tv, P.q, P.d, 1, 1, 1, P.q_st, P.q_sh, 0, kBN, kE);
    } else {
        ok = make_map(enc, &tq, P.q, P.d, P.Tq, P.Hq, P.B, P.q_st, P.q_sh, P.q_sb, kBM, kE) &&
             make_kv_maps(enc, &tk, &tv, P, kBN, kE) &&
             make_map(enc, &to, P.o, P.d, P.Tq, P.Hq, P.B, P.o_st, P.o_sh, P.o_sb, kBM);
    }
    if (!ok) return cudaErrorInvalidValue;
    // The CTA takes all 512 tensor-memory columns; the shared-memory request
    // (the K/V ring fills it) keeps a second CTA off the SM.
    constexpr size_t kSmem = SmemLayout<D, MODE>::kTotal + 1024;
    static_assert(kSmem <= 227 * 1024 && kSmem > 114 * 1024, "shared memory budget");
    static DeviceOnce configured;
    int dev = -1;
    if (!configured.done(dev)) {
        if (dev < 0) return cudaErrorInvalidDevice;
        cudaError_t e = cudaFuncSetAttribute(fa_fwd_bf16_kernel<D, MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
        if (e != cudaSuccess) return e;
        if constexpr (is_prefill(MODE)) {
            // The warpgroups' register shares come from what the CTA was
            // launched with; with fewer, the softmax warps' increase could
            // never be granted.  Refuse a build that differs.
            cudaFuncAttributes fattr{};
            e = cudaFuncGetAttributes(&fattr, fa_fwd_bf16_kernel<D, MODE>);
            if (e != cudaSuccess) return e;
            if (fattr.numRegs != kRegsLaunchPrefill) return cudaErrorInvalidKernelImage;
        }
        configured.mark(dev);
    }
    // One CTA per SM, no more than there are units (a test may cap the grid).
    const int nqt = (P.Tq + kBM - 1) / kBM;
    const long long units = (long long)nqt * P.B * P.Hq;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    long long grid = units < sms ? units : sms;
    if (g_test_max_ctas > 0 && grid > g_test_max_ctas) grid = g_test_max_ctas;
    // A grid on at most half the SMs leaves room for the next call's CTAs
    // to start early, so its first tiles are worth requesting into L2.
    if constexpr (is_prefill(MODE)) P.prefetch_l2 = 2 * grid <= sms ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(threads_for(MODE));
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fa_fwd_bf16_kernel<D, MODE>, tq, tk, tv, to, P);
}

// Key tiles seen by the rows at positions q_offset .. q_offset + Tq - 1 among
// Tk keys.
int packed_tiles(const Params &P, int Tk, int q_offset) {
    int64_t lo_a, hi_a, lo_b, hi_b;
    visible_range_tk(P, Tk, (int64_t)q_offset, lo_a, hi_a);
    visible_range_tk(P, Tk, (int64_t)q_offset + P.Tq - 1, lo_b, hi_b);
    const int64_t klo = lo_a, khi = hi_b > hi_a ? hi_b : hi_a;
    if (khi <= klo) return 0;
    return (int)((khi + kBN - 1) / kBN - klo / kBN);
}

// Packed rows (group * Tq <= 128): one cluster of `splits` CTAs per (batch,
// KV head).  The split count is the largest that keeps every cluster of the
// call resident at once (a second wave would double the time) with at least
// two key tiles per CTA; a range of fewer than 4 tiles is not split (and then
// matches the prefill kernel bit for bit).  It depends on B * Hkv and on the
// device's cluster capacity, so split rows are not batch-invariant: the
// split trades invariance for parallelism.
template <int D, int MODE>
cudaError_t launch_packed(const Params &P0, cudaStream_t stream) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    Params P = P0;
    // Paged: the longest sequence sizes the split (each cluster splits its own range).
    const int n = MODE == kPaged ? packed_tiles(P, P.max_seq_len, P.max_seq_len > P.Tq ? P.max_seq_len - P.Tq : 0)
                                 : packed_tiles(P, P.Tk, P.q_offset);
    CUtensorMap tq, tk, tv, to;
    bool ok = make_packed_map(enc, &tq, P.q, P, P.q_st, P.q_sh, P.q_sb) &&
              // to is not used by the packed path (O leaves through the merge).
              make_map(enc, &to, P.o, P.d, P.Tq, P.Hq, P.B, P.o_st, P.o_sh, P.o_sb, kBM);
    if (MODE == kPaged) {
        // caches [num_pages, page_size, Hkv, d]: the map (d, page_size, Hkv, num_pages)
        const int run = P.page_size < kBN ? P.page_size : kBN;
        const int64_t st = (int64_t)P.Hkv * P.d, sp = (int64_t)P.page_size * st;
        ok = ok && make_map(enc, &tk, P.k, P.d, P.page_size, P.Hkv, P.num_pages, st, P.d, sp, run) &&
             make_map(enc, &tv, P.v, P.d, P.page_size, P.Hkv, P.num_pages, st, P.d, sp, run);
    } else {
        ok = ok && make_kv_maps(enc, &tk, &tv, P, kBN);
    }
    if (!ok) return cudaErrorInvalidValue;
    constexpr size_t kSmem = SmemLayout<D, MODE>::kTotal + 1024;
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
    auto kernel = fa_fwd_bf16_kernel<D, MODE>;
    constexpr int kMaxSplits = 16;
    static DeviceOnce configured;
    static int capacity[64][kMaxSplits + 1] = {};  // per device: clusters of s CTAs resident at once
    int dev = -1;
    const bool have = configured.done(dev);
    if (dev < 0) return cudaErrorInvalidDevice;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (!have) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        for (int sp = 1; sp <= kMaxSplits; ++sp) {
            int clusters = 0;
            cfg.gridDim = dim3((unsigned)sp);
            attr[1].val.clusterDim.x = (unsigned)sp;
            if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) {
                (void)cudaGetLastError();
                clusters = 0;
            }
            capacity[dev][sp] = clusters;
        }
        if (capacity[dev][1] <= 0) return cudaErrorInvalidConfiguration;
        configured.mark(dev);
    }
    const int units = P.B * P.Hkv;
    int S = 1;
    if (n >= 4)
        for (int sp = n / 2 < kMaxSplits ? n / 2 : kMaxSplits; sp > 1; --sp)
            if (capacity[dev][sp] >= units) {
                S = sp;
                break;
            }
    P.splits = S;
    P.fd_splits = FastDiv::make((uint32_t)S);
    P.fd_hkv = FastDiv::make((uint32_t)P.Hkv);
    P.fd_group = FastDiv::make((uint32_t)P.group);
    P.fd_d = FastDiv::make((uint32_t)P.d);
    cfg.gridDim = dim3((unsigned)(units * S));
    attr[1].val.clusterDim.x = (unsigned)S;
    return cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, to, P);
}

}  // namespace

cudaError_t bf16_watchdog(cudaStream_t stream, unsigned int *flag) {
    unsigned int v = 0;
    const unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_watchdog, sizeof v, 0, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && v != 0)
        e = cudaMemcpyToSymbolAsync(g_watchdog, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    *flag = v;
    return e;
}

cudaError_t bf16_set_drop_arrive(int on) { return cudaMemcpyToSymbol(g_drop_arrive, &on, sizeof on); }

// Split-KV through the workspace: splits per (batch, KV head) so that the
// grid fills the SMs once (at most kMaxSplitsWs, at least two key tiles per
// CTA, at least 1).
constexpr int kMaxSplitsWs = 64;

int splitkv_splits(int units, int sms) {
    int S = units > 0 ? sms / units : 1;
    return S < 1 ? 1 : (S > kMaxSplitsWs ? kMaxSplitsWs : S);
}

size_t counters_bytes(int units) { return ((size_t)units * sizeof(unsigned int) + 255) / 256 * 256; }

template <int D>
cudaError_t launch_splitkv_d(const Params &P0, void *workspace, cudaStream_t stream) {
    constexpr int MODE = kSplitKv;
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return cudaErrorNotSupported;
    Params P = P0;
    const int n = packed_tiles(P, P.Tk, P.q_offset);
    CUtensorMap tq, tk, tv, to;
    bool ok = make_packed_map(enc, &tq, P.q, P, P.q_st, P.q_sh, P.q_sb) &&
              // to is not used by the packed path (O leaves through the merge).
              make_map(enc, &to, P.o, P.d, P.Tq, P.Hq, P.B, P.o_st, P.o_sh, P.o_sb, kBM) &&
              make_kv_maps(enc, &tk, &tv, P, kBN);
    if (!ok) return cudaErrorInvalidValue;
    constexpr size_t kSmem = SmemLayout<D, MODE>::kTotal + 1024;
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
    static_assert((3 * kMaxSplitsWs + 2) * kBM * 4 <= 2 * SmemLayout<D, MODE>::kStages * SmemLayout<D, MODE>::kKVBytes,
                  "the merge's per-row weights fit the K/V rings");
    auto kernel = fa_fwd_bf16_kernel<D, MODE>;
    static DeviceOnce configured;
    int dev = -1;
    if (!configured.done(dev)) {
        if (dev < 0) return cudaErrorInvalidDevice;
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
        if (e != cudaSuccess) return e;
        configured.mark(dev);
    }
    const int units = P.B * P.Hkv;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    int S = splitkv_splits(units, sms);
    if (S > n / 2) S = n / 2 > 1 ? n / 2 : 1;  // at least two key tiles per CTA
    P.splits = S;
    P.fd_splits = FastDiv::make((uint32_t)S);
    P.fd_hkv = FastDiv::make((uint32_t)P.Hkv);
    P.fd_group = FastDiv::make((uint32_t)P.group);
    P.fd_d = FastDiv::make((uint32_t)P.d);
    P.ws_cnt = static_cast<unsigned int *>(workspace);
    P.ws = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + counters_bytes(units));
    cudaError_t e = cudaMemsetAsync(P.ws_cnt, 0, (size_t)units * sizeof(unsigned int), stream);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(units * S));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, to, P);
}

cudaError_t launch_bf16_paged(const Params &P, cudaStream_t stream) {
    return P.d <= 64 ? launch_packed<64, kPaged>(P, stream) : launch_packed<128, kPaged>(P, stream);
}

cudaError_t launch_bf16_varlen(const Params &P, cudaStream_t stream) {
    return P.d <= 64 ? launch_d<64, kVarlen>(P, stream) : launch_d<128, kVarlen>(P, stream);
}

cudaError_t launch_fp8(const Params &P, cudaStream_t stream) {
    // e4m3 rows of d <= 128 bytes: one 128-byte box per row, padded with zeros.
    return launch_d<128, kPrefill8>(P, stream);
}

cudaError_t launch_fp8_varlen(const Params &P, cudaStream_t stream) { return launch_d<128, kVarlen8>(P, stream); }

cudaError_t launch_bf16(const Params &P, cudaStream_t stream) {
    // d is a multiple of 8 up to 128: the 64- or 128-column kernel, padded.
    // All query rows of a KV group in one tile: the packed-row kernel.
    if ((int64_t)P.group * P.Tq <= kBM)
        return P.d <= 64 ? launch_packed<64, kDecode>(P, stream) : launch_packed<128, kDecode>(P, stream);
    return P.d <= 64 ? launch_d<64, kPrefill>(P, stream) : launch_d<128, kPrefill>(P, stream);
}

size_t splitkv_workspace_bytes(int B, int Hkv, int group, int Tq, int d) {
    if ((int64_t)group * Tq > kBM || B <= 0 || Hkv <= 0 || Tq <= 0 || d <= 0) return 0;
    const int units = B * Hkv, D = d <= 64 ? 64 : 128;
    const int S = splitkv_splits(units, sm_count());
    return counters_bytes(units) + (size_t)units * S * (size_t)ws_block_floats(group * Tq, D) * sizeof(float);
}

cudaError_t launch_bf16_splitkv(const Params &P, void *workspace, cudaStream_t stream) {
    if ((int64_t)P.group * P.Tq > kBM) return launch_bf16(P, stream);  // not a packed-row call: no workspace
    return P.d <= 64 ? launch_splitkv_d<64>(P, workspace, stream) : launch_splitkv_d<128>(P, workspace, stream);
}

// Scratch for callers that cannot allocate device memory: the split-KV
// workspace (counters, then the partial blocks) in one array that every GPU
// loading this library holds until the process exits.  All calls on a device
// share it and the last call's contents stay in it; the launcher clears the
// counters before each kernel, and the partial blocks are always written
// before they are read.  Two calls whose kernels overlap on the GPU (other
// streams, other host threads) race on it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
// g_noalloc_scratch names a host-side stand-in in host code, not device
// memory: the kernels get the address that cudaGetSymbolAddress returns on
// the device where they run, looked up once per device with it current.
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kMaxDevices] = {};

cudaError_t noalloc_scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (p == nullptr) return cudaErrorInvalidSymbol;
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return cudaSuccess;
}
}  // namespace

cudaError_t launch_bf16_splitkv_noalloc(const Params &P, cudaStream_t stream) {
    void *scratch = nullptr;
    const cudaError_t e = noalloc_scratch_address(&scratch);
    if (e != cudaSuccess) return e;
    return launch_bf16_splitkv(P, scratch, stream);
}

}  // namespace fa
