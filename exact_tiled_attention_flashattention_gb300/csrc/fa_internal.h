// fa_internal.h -- parameters shared by the host layer and the kernels.
// Not part of the public ABI (include/fa.h is).
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "fast_div.h"

namespace fa {

// One validated call of fa_fwd, in the form the kernels read it.
struct Params {
    const void *q, *k, *v;
    void *o;
    float *lse;           // [B, Hq, Tq] or nullptr
    const float *sinks;   // [Hq] or nullptr
    const float *mask;    // strided, or nullptr
    int64_t msb, msh, msq, msk;
    int B, Hq, Hkv, Tq, Tk, d;
    int group;            // Hq / Hkv
    int q_offset;         // absolute position of query row 0
    int causal;
    int window;           // <= 0: none (clamped to int range by the host)
    float scale;          // scale applied to q.k
    float scale_log2;     // scale * log2(e)
    int splits;           // bf16 packed-row path: CTAs that split a key range (set by its launcher)
    int prefetch_l2;      // bf16 prefill: request the first unit's tiles into L2 before the
                          // dependency wait (set by its launcher)
    // Element strides of q, k, v, o: batch, head, row (the d elements of a
    // row are contiguous).
    int64_t q_sb, q_sh, q_st, k_sb, k_sh, k_st, v_sb, v_sh, v_st, o_sb, o_sh, o_st;
    int vec16;            // fp32: every q/k/v row starts on a 16-byte boundary
    // Paged K/V (bf16 packed rows): k and v are caches [num_pages, page_size,
    // Hkv, d]; key j of sequence b is row j % page_size of page
    // block_table[b * max_blocks + j / page_size]; sequence b has seq_lens[b]
    // keys (at most max_seq_len) and its Tq queries are its last positions.
    const int *seq_lens;
    const int *block_table;
    int max_blocks, page_size, num_pages, max_seq_len;
    // Variable-length batch: sequence b has rows [cu_q[b], cu_q[b+1]) of q
    // and o (tensors [total_q, H, d]) and rows [cu_k[b], cu_k[b+1]) of k and
    // v; its queries are its last positions.  Tq / Tk hold the maxima.
    const int *cu_q, *cu_k;
    int total_q, total_k;
    // Split-KV through a workspace (bf16 packed rows, fa_fwd_splitkv): the
    // partials [B * Hkv][splits][R rows][D + 2] fp32 (R = group * Tq, D = 64
    // or 128: O, then (m, l) per row) and one counter per (batch, KV head).
    float *ws;
    unsigned int *ws_cnt;
    // Divisors of the tcgen05 kernel's index arithmetic, set by its launchers:
    // units per query tile, heads per unit row (Hq, or Hq / 2 with CTA
    // pairs), the GQA group, the split count, Hkv and d.
    FastDiv fd_per_qt, fd_heads, fd_group, fd_splits, fd_hkv, fd_d;
};

// Visible key range [lo, hi) of query position p (absolute) among Tk keys,
// before the mask.
__host__ __device__ inline void visible_range_tk(const Params &P, int64_t Tk, int64_t p, int64_t &lo, int64_t &hi) {
    hi = P.causal ? (p + 1 < Tk ? p + 1 : Tk) : Tk;
    lo = P.window > 0 ? (p - P.window + 1 > 0 ? p - P.window + 1 : 0) : 0;
    if (hi < lo) hi = lo;
}

__host__ __device__ inline void visible_range(const Params &P, int64_t p, int64_t &lo, int64_t &hi) {
    visible_range_tk(P, (int64_t)P.Tk, p, lo, hi);
}

// A thread's visible keys among its (at most 64) keys of a tile, the interval
// [elo, ehi) with 0 <= elo, ehi <= 64, as a bit mask: key e is visible iff
// bit e is set (none when ehi <= elo).  On a boundary tile the kernels test
// one constant bit per key instead of comparing e with both ends.
struct KeyBits {
    uint32_t lo, hi;  // keys 0-31, 32-63
    __host__ __device__ bool has(int e) const { return ((e < 32 ? lo : hi) & (1u << (e & 31))) != 0u; }
};
__host__ __device__ inline KeyBits key_bits(int elo, int ehi) {
    const uint64_t below_hi = ehi >= 64 ? ~0ull : (1ull << ehi) - 1ull;
    const uint64_t below_lo = elo >= 64 ? ~0ull : (1ull << elo) - 1ull;
    const uint64_t v = below_hi & ~below_lo;
    return KeyBits{(uint32_t)v, (uint32_t)(v >> 32)};
}

cudaError_t launch_f32(const Params &P, cudaStream_t stream);
// fp32 with three TF32 tensor-core products per matrix product.
cudaError_t launch_f32_tc(const Params &P, cudaStream_t stream);
cudaError_t launch_bf16(const Params &P, cudaStream_t stream);
// e4m3 Q, K, V (kind::f8f6f4 MMAs, P rounded to e4m3), bf16 O.
cudaError_t launch_fp8(const Params &P, cudaStream_t stream);
cudaError_t launch_fp8_varlen(const Params &P, cudaStream_t stream);
cudaError_t launch_bf16_paged(const Params &P, cudaStream_t stream);
cudaError_t launch_bf16_varlen(const Params &P, cudaStream_t stream);
// Packed-row calls (group * Tq <= 128) with their key ranges split over as
// many CTAs as fill the SMs, merged through a workspace of
// splitkv_workspace_bytes(P) bytes (see fa_fwd_splitkv).  The launcher
// clears the counters on `stream` before the kernel.
cudaError_t launch_bf16_splitkv(const Params &P, void *workspace, cudaStream_t stream);
// Bytes of that workspace for calls of this shape on the current device (0
// if the call does not take the packed-row mapping).
size_t splitkv_workspace_bytes(int B, int Hkv, int group, int Tq, int d);
// The same split-KV call with its workspace in a static device array of
// kNoAllocScratchBytes per GPU instead of caller memory (fa_fwd_splitkv_noalloc):
// the caller checks the size first; the launcher looks up the array's device
// address on the current device (once per device) and launches.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
cudaError_t launch_bf16_splitkv_noalloc(const Params &P, cudaStream_t stream);
cudaError_t launch_f32_varlen(const Params &P, cudaStream_t stream);

// Device watchdog words: nonzero once a bounded wait of the kernel ran out.
// Read (after the stream's work) and cleared.
cudaError_t bf16_watchdog(cudaStream_t stream, unsigned int *flag);
cudaError_t f32tc_watchdog(cudaStream_t stream, unsigned int *flag);
// Test hooks: make CTA 0 of the next launches skip one load (see the kernels).
cudaError_t bf16_set_drop_arrive(int on);

// Launchers set their kernels' function attributes (shared-memory size,
// cluster sizes) once per device: the attributes belong to each device's
// context, so a process that calls on several GPUs sets them on each.  Bit
// `dev` records the device; devices 0..63.
struct DeviceOnce {
    std::atomic<unsigned long long> bits{0};
    // The current device in `dev` (-1 if none or >= 64); true once mark(dev) ran.
    bool done(int &dev) const {
        dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
            dev = -1;
            return false;
        }
        return ((bits.load(std::memory_order_acquire) >> dev) & 1ull) != 0;
    }
    void mark(int dev) {
        if (dev >= 0 && dev < 64) bits.fetch_or(1ull << dev, std::memory_order_release);
    }
};

// Test hook: when positive, the persistent launchers use at most this many
// CTAs (0: one per SM).  Set through fa_test_max_ctas.
extern int g_test_max_ctas;
cudaError_t f32tc_set_drop_arrive(int on);

}  // namespace fa
