// fa8_kernel.cuh -- the fused FP8 attention forward for sm_103a (tcgen05 + TMA + TMEM)
// and the split-KV combine kernel.
//
// One CTA computes one 128-row Q tile: the rows are (query position, q-head) pairs of one
// kv-head group, packed position-major (PackGQA), against the kv-head's keys, for one
// split of the request's key range.  Roles (512 threads, four warpgroups):
//   warps 0-3   softmax, keys [0, 64) of every tile: thread r owns TMEM lane r = row r
//   warps 4-7   softmax, keys [64, 128) of the same rows; the two halves exchange their
//               row maxima once per tile and their row sums once at the end
//   warps 8-11  correction: two-level PV fold into fp32 O, epilogue
//   warp 12     TMA producer (Q once, K/V tiles into S-stage rings)
//   warp 13     MMA issuer (lane 0) and TMEM owner
//   warps 14-15 idle (the control warpgroup gives its registers to the correction)
// Splitting each row over two warps halves the per-warp softmax work per tile, so the
// softmax keeps pace with the tensor core; each half reads its 64 S columns from TMEM in a
// single round trip per tile.
//
// Per 128-key tile t (sources: "[Cute,Fwd,Sm90] Native FP8 (E4M3 Q/K/V) forward for
// Hopper", Design; "tml-fa4 PR #4", Summary and "Correctness fix over #1"):
//   S_t   = Q K_t^T                     tcgen05.mma kind::f8f6f4, fp32 in TMEM
//   m     lazy running max: moved only when the tile max exceeds it by more than
//         tau = 0.75 (log2 units), tau <= log2(448) - 8 so that P never clips
//   P_t   = 2^(s*c - m + 8) -> E4M3 (c = softmax_scale * dq * dk * log2 e), stored in
//         TMEM over S_t: the packed P of keys [32k, 32k+32) goes to column 32k of the S_t
//         buffer (8 columns), after that 32-column slice of S_t has been read
//   O_t   = P_t V_t                     accumulated from zero for every tile
//         (on tiles that need a mask, P_t = P_hi + P_lo with P_lo = e4m3(p - P_hi) and
//          both terms go through the PV MMA: rows with only a few visible keys keep
//          ~2^-8 relative precision instead of the 2^-4 of one E4M3 term)
//   O     = O * alpha + O_t             fp32 fold (two-level accumulation)
// and after the last tile O * dv / rowsum -> bf16/fp16, LSE = ln2*(log2 rowsum + m - 8).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "fa8_ptx.cuh"

namespace fa8 {

constexpr int kTileM = 128;     // Q rows per CTA = TMEM lanes
constexpr int kTileN = 128;     // keys per KV tile
constexpr int kNumThreads = 512;
// registers per thread after setmaxnreg; 256 x 112 + 128 x 240 + 128 x 48 = 512 x 128 (launch)
constexpr int kLaunchRegs = 128;
constexpr int kRegsSoft = 112;
constexpr int kRegsCorr = 240;
constexpr int kRegsCtl = 48;
static_assert(2 * kRegsSoft + kRegsCorr + kRegsCtl == 4 * kLaunchRegs, "register split");
// Lazy-rescale threshold, log2 units: the running max moves only when a tile's max passes it
// by more than this, so it must stay below log2(448) - 8 for P = 2^(s c - m + 8) to fit
// E4M3.  FA8_TAU overrides it only for the negative-control build of the threshold test.
#ifdef FA8_TAU
constexpr float kTau = FA8_TAU;
#else
constexpr float kTau = 0.75f;
#endif
constexpr float kPBias = 8.0f;  // P carries a factor 2^8
// A tile's P goes through the PV MMA as two E4M3 terms (P_hi + P_lo, P_lo = e4m3(p - P_hi))
// when the tile needs a mask, or when, in some row, the tile's largest p is more than this
// share of the row's mass so far (its running sum plus that p).  So every key that keeps one
// E4M3 term holds at most this share of its row's final sum, and the single-term rounding
// (up to 2^-4 relative per weight) stays spread over many keys.
constexpr float kTwoTermShare = 0.125f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum : unsigned { kStatusTimeout = 1u, kStatusBounds = 2u };

// Pipeline event trace (compiled in only with -DFA8_TRACE): clock64() per (CTA, event, tile)
// for the first kTraceCtas CTAs of grid row 0; layout [cta][event][tile].  Events are kept
// in shared memory while the CTA runs (a global store before an mbarrier arrive would
// delay the arrive's release) and copied out at the end.
constexpr int kTraceCtas = 8, kTraceEvents = 16, kTraceTiles = 64;
#ifdef FA8_TRACE
constexpr int kTraceSmemBytes = kTraceEvents * kTraceTiles * 8;
#define FA8_EV(ev, it)                                                                  \
    do {                                                                                \
        if ((it) < kTraceTiles)                                                         \
            reinterpret_cast<unsigned long long *>(smem + C::OFF_TRACE)[(ev) * kTraceTiles + (it)] = clock64(); \
    } while (0)
// records a value instead of a clock
#define FA8_VAL(ev, it, v)                                                              \
    do {                                                                                \
        if ((it) < kTraceTiles)                                                         \
            reinterpret_cast<unsigned long long *>(smem + C::OFF_TRACE)[(ev) * kTraceTiles + (it)] = (v); \
    } while (0)
#else
constexpr int kTraceSmemBytes = 0;
#define FA8_EV(ev, it) \
    do {               \
    } while (0)
#define FA8_VAL(ev, it, v) \
    do {                   \
    } while (0)
#endif

struct FwdParams {
    int B, Hq, Hkv, G, rows_per_tile, pos_per_tile;
    int q_varlen;  // q is (total_q, Hq, D) with cu_q
    int kv_mode;   // 0 batched, 1 varlen, 2 paged
    int Sq, Sk;    // batched lengths
    int total_q, total_k;
    int mblocks_per_batch;  // batched Q: ceil(Sq / pos_per_tile)
    const int *cu_q;
    const int *cu_k;
    const int *block_table;
    long long bt_stride;
    int max_pages, page_size, box_n, boxes_per_tile, num_pages;
    const float *dq, *dk, *dv;
    long long dq_sb, dq_sh, dk_sb, dk_sh, dv_sb, dv_sh;
    const float *sink;
    float scale_log2;  // softmax_scale * log2(e)
    int causal, window_left;
    int num_splits;
    int split_mode;  // write fp32 partials for the combine kernel
    void *o;
    long long o_sb, o_ss, o_sh;
    int out_fp16;
    float *lse;
    long long lse_sb, lse_sh, lse_ss;
    float *o_part, *lse_part;
    unsigned long long timeout_ns;
    unsigned int *status;
    unsigned long long *trace;  // event timestamps (builds with FA8_TRACE only), may be null
    // split mode: CTAs that run at once (for split_tile_cap) and the split cap that
    // split_plan_kernel writes before the forward kernel runs, or, when cap_const > 0, the
    // cap itself (no plan kernel)
    int slots;
    int *split_cap;
    int cap_const;
    int units;  // work units of the persistent prefill kernel (slot, kv-head, split)
};

struct CombineParams {
    int total_q, Hq, num_splits, q_varlen, Sq;
    // what the forward kernels derive each row's split count from (see split_range), and
    // the split cap split_plan_kernel wrote (cap_const > 0: that cap instead)
    int B, pos_per_tile, kv_mode, Sk, causal, window_left;
    const int *cu_q, *cu_k;
    const int *split_cap;
    int cap_const;
    int wpr;  // warps per output row (1, 2, 4 or 8): warp w % wpr takes splits s = w % wpr (mod wpr)
    const float *o_part, *lse_part;
    void *o;
    long long o_sb, o_ss, o_sh;
    int out_fp16;
    float *lse;
    long long lse_sb, lse_sh, lse_ss;
};

// Compile-time tile configuration for head dims (D, DV).
template <int D, int DV>
struct Cfg {
    // Q/K rows are split along D into chunks of CW bytes, each its own swizzled block.
    static constexpr int CW = (D % 128 == 0) ? 128 : ((D % 64 == 0) ? 64 : 32);
    static constexpr int NCK = D / CW;
    // V rows are split along DV into chunks of CWV bytes (MN-major operand of PV).
    static constexpr int CWV = (DV % 128 == 0) ? 128 : ((DV % 64 == 0) ? 64 : 32);
    static constexpr int NCV = DV / CWV;
    // Running O lives in registers when it fits (dv <= 128), else in TMEM.
    static constexpr bool O_REGS = DV <= 128;
    static constexpr int NS = O_REGS ? 2 : 1;  // S/P buffers in TMEM
    static constexpr int OTW = (NS * 128 + DV + (O_REGS ? 0 : DV) <= 512) ? DV : DV / 2;
    static constexpr int NPV = DV / OTW;  // PV MMAs per tile (dv split through one O_tile)
    static constexpr int NOT = O_REGS ? 2 : 1;  // O_tile buffers (double-buffered when O is in registers)
    static constexpr uint32_t TM_S = 0;
    static constexpr uint32_t TM_OT = NS * 128;
    static constexpr uint32_t TM_OR = TM_OT + NOT * OTW;
    static constexpr uint32_t TM_COLS = 512;
    static constexpr int CHUNK_Q = kTileM * CW;
    static constexpr int CHUNK_K = kTileN * CW;
    static constexpr int CHUNK_V = kTileN * CWV;
    static constexpr int Q_BYTES = kTileM * D;
    static constexpr int K_BYTES = kTileN * D;
    static constexpr int V_BYTES = kTileN * DV;
    static constexpr int MISC_BYTES = 6208;
    static constexpr int SMEM_LIMIT = 232448;  // max dynamic smem per block on sm_103
    static constexpr int STAGES_FIT =
        (SMEM_LIMIT - 1024 - MISC_BYTES - kTraceSmemBytes - Q_BYTES) / (K_BYTES + V_BYTES);
    static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = Q_BYTES;
    static constexpr int OFF_V = OFF_K + STAGES * K_BYTES;
    static constexpr int OFF_MISC = OFF_V + STAGES * V_BYTES;
    static constexpr int OFF_TRACE = OFF_MISC + MISC_BYTES;
    static constexpr int SMEM_BYTES = OFF_TRACE + kTraceSmemBytes + 1024;
    // barrier slots
    static constexpr int B_Q = 0;
    static constexpr int B_KF = 1;
    static constexpr int B_KE = B_KF + STAGES;
    static constexpr int B_VF = B_KE + STAGES;
    static constexpr int B_VE = B_VF + STAGES;
    static constexpr int B_SF = B_VE + STAGES;
    static constexpr int B_PF = B_SF + NS;
    static constexpr int B_OF = B_PF + NS;   // NOT slots
    static constexpr int B_OE = B_OF + NOT;  // NOT slots
    // Alpha ring depth (softmax -> correction).  The ring needs no "slot empty" barrier: the
    // softmax writes the slot of tile t only after S(t) is ready, which follows the issue of
    // QK(t), which follows the issue of PV(t - 1) or PV(t - 2), which waits for the fold of
    // an O_tile from tile t - 2 or earlier; the correction reads a tile's alpha before it
    // folds that tile, so the slot's previous tile (t - 4) has been read.
    static constexpr int NA = 4;
    static constexpr int B_AF = B_OE + NOT;  // NA slots
    static constexpr int B_XCH = B_AF + NA;  // 2 slots: row-max exchange between the halves
    static constexpr int B_SUM = B_XCH + 2;  // half 1 -> half 0: final partial row sums
    static constexpr int B_FIN = B_SUM + 1;  // half 0 -> correction: final O scale
    static constexpr int B_DONE = B_FIN + 1;
    static constexpr int NUM_BARS = B_DONE + 1;
    static_assert(STAGES >= 2, "smem too small for two K/V stages");
    static_assert(NUM_BARS * 8 <= 512, "barrier area");
    static_assert(TM_OR + (O_REGS ? 0 : DV) <= TM_COLS, "TMEM budget");
    static_assert(OTW % CWV == 0 && OTW % 32 == 0 && OTW % 16 == 0 && OTW <= 256, "PV shape");
    static_assert(D % 32 == 0 && DV % 32 == 0, "head dims");
};

// UMMA shared-memory descriptor: start >>4 [0,14), LBO >>4 [16,30), SBO >>4 [32,46),
// fixed 0b001 at [46,49), swizzle layout at [61,64) (2 = 128B, 4 = 64B, 6 = 32B).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                          uint32_t layout) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)layout << 61;
    return d;
}
__host__ __device__ constexpr uint32_t swz_layout(int chunk_bytes) {
    return chunk_bytes == 128 ? 2u : (chunk_bytes == 64 ? 4u : 6u);
}
// Instruction descriptor, kind::f8f6f4: D fp32 (bit 4), A/B E4M3 (0), B major at bit 16,
// N>>3 at [17,23), M>>4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, bool b_mn_major) {
    return (1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// Bounded mbarrier waits: give up when another role aborted or after timeout_ns, setting
// the CTA abort flag and the device status word.
__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int *abort,
                                          unsigned long long timeout, unsigned int *status) {
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (ptx::globaltimer() - t0 > timeout) {
            *abort = 1;
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
}

// As Waiter::wait_warp, for roles that keep as few registers as possible live: the abort flag by
// its shared-memory address, the bound and status word read from the kernel parameters only
// on the slow path.
__device__ __forceinline__ bool wait_slow_s(uint32_t bar, uint32_t parity, uint32_t abort_saddr,
                                            unsigned long long timeout, unsigned int *status) {
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        int ab;
        asm volatile("ld.volatile.shared.b32 %0, [%1];" : "=r"(ab) : "r"(abort_saddr));
        if (ab) return false;
        if (ptx::globaltimer() - t0 > timeout) {
            asm volatile("st.volatile.shared.b32 [%0], %1;" ::"r"(abort_saddr), "r"(1));
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
}

struct Waiter {
    volatile int *abort;
    unsigned long long timeout;
    unsigned int *status;
    // fast path first; the bounded spin only when the phase is not complete yet
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        return wait_slow(bar, parity, abort, timeout, status);
    }
    // Whole-warp form: every lane waits, the result is made warp-uniform and the warp is
    // reconverged (needed before the warp-collective tcgen05.ld/st that follow).
    __device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity) const {
        const bool ok = wait(bar, parity);
        return __all_sync(0xffffffffu, ok);
    }
    // Used when draining in-flight async work before exit: ignores the abort flag.
    __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity) const {
        const uint64_t t0 = ptx::globaltimer();
        while (!ptx::mbar_try_wait(bar, parity)) {
            if (ptx::globaltimer() - t0 > timeout) {
                atomicOr(status, kStatusTimeout);
                return false;
            }
        }
        return true;
    }
};

// Whether any row of the tile (keys [k0, k0+128)) needs masking: CTA-uniform; the
// softmax and MMA roles both evaluate it so that they agree on the two-term P.
__device__ __forceinline__ bool tile_needs_mask(int k0, int Lk, int causal, int window_left, int pos0,
                                                int pos_last, int delta) {
    return (k0 + kTileN > Lk) || (causal && k0 + kTileN - 1 > pos0 + delta) ||
           (window_left >= 0 && k0 < pos_last + delta - window_left);
}

// Splits of a tile's key range (graph-safe: the launch fixes an upper bound n from shapes
// only, the device picks what runs).  The visible keys of query positions [pos0, pos_last]
// span KV tiles [tb, te); the tile runs eff = clamp(ceil((te - tb) / cap), 1, n) splits of
// ceil((te - tb) / eff) tiles each, where cap (split_tile_cap) is one per launch.  Splits
// >= eff do nothing and the combine kernel, which evaluates the same function per row with
// the same cap, never reads them; split 0 always runs (it also writes the result of a tile
// without visible keys).
struct SplitRange {
    int t_beg, n_tiles, eff;
};
__device__ __forceinline__ SplitRange split_range(int Lq, int Lk, int pos0, int pos_last, int causal,
                                                  int window_left, int num_splits, int cap, int split) {
    const int delta = Lk - Lq;
    const int kv_end = causal ? min(Lk, pos_last + delta + 1) : Lk;
    const int kv_beg = window_left >= 0 ? max(0, pos0 + delta - window_left) : 0;
    SplitRange r{0, 0, 1};
    if (kv_end > kv_beg) {
        const int tb = kv_beg / kTileN;
        const int te = (kv_end + kTileN - 1) / kTileN;
        const int nt = te - tb;
        r.eff = max(1, min(num_splits, (nt + cap - 1) / cap));
        const int per = (nt + r.eff - 1) / r.eff;
        r.t_beg = tb + split * per;
        r.n_tiles = max(0, min(te, r.t_beg + per) - r.t_beg);
    }
    return r;
}

// The largest number of KV tiles a split may take (the cap above), chosen per launch on the
// device from the requests' key counts, so that it follows the data while the grid stays
// fixed.  For each candidate cap T (2, 4, ..., 512, and ceil(t_max / n), the finest the
// launch allows) it counts the work units (tile of query rows, kv-head, split) N(T) and
// models the run time, in tile times, as
//   single wave (N <= slots):  F + min(T, t_max)
//   otherwise:                  (F N + tiles) / slots + beta (F + min(T, t_max))
// with F the fixed cost of a unit (prologue, pipeline fill and drain, finalize), `tiles` the
// total KV tile count, t_max the longest request and `slots` the CTAs that run at once: the
// first term keeps the machine busy, the second is the last units' tail.  F = 3 and
// beta = 0.4 reproduce the decode kernel's measured times over split counts 1-32 on the
// mixed-length paged workload and pick the measured best split count of every
// served-model decode step shape.  Caps that would need more than the launched n splits are
// skipped.  Each request's tile count is taken from its key count (ceil(Lk / 128)), for
// every tile of its query rows.  The whole warp calls it and gets the same value in every
// lane.
constexpr float kFixedTiles = 3.f, kTailWeight = 0.4f;
__device__ __forceinline__ int split_tile_cap(int B, int Hkv, int kv_mode, int Sk, const int *cu_k, int q_varlen,
                                              int Sq, const int *cu_q, int pos_per_tile, int num_splits,
                                              int slots) {
    constexpr int NC = 10;  // candidates 2^1 .. 2^9 tiles, then ceil(t_max / n)
    const int lane = threadIdx.x & 31;
    // 32-bit counts and fp32 arithmetic only: it runs on the critical path of every split
    // launch, and the part's FP64 rate is far too low for it
    unsigned int units[NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) units[c] = 0u;
    unsigned int tiles = 0u;
    int t_max = 0;
    // every lane loads its requests' lengths at once (up to kPer per lane in registers, the
    // rest re-read), the longest request first: it fixes the last candidate
    constexpr int kPer = 8;
    int lks[kPer], lqs[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int b = lane + 32 * i;
        lks[i] = b < B ? (kv_mode == 0 ? Sk : cu_k[b + 1] - cu_k[b]) : 0;
        lqs[i] = b < B ? (q_varlen ? cu_q[b + 1] - cu_q[b] : Sq) : 0;
    }
    auto add_t = [&](int lk) { t_max = max(t_max, lk > 0 ? (lk + kTileN - 1) / kTileN : 0); };
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        if (32 * i < B) add_t(lks[i]);  // (slots past the batch skipped by the whole warp)
    for (int b = lane + 32 * kPer; b < B; b += 32) add_t(kv_mode == 0 ? Sk : cu_k[b + 1] - cu_k[b]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t_max = max(t_max, __shfl_xor_sync(0xffffffffu, t_max, o));
    const int t_fine = max(2, (t_max + num_splits - 1) / num_splits);
    auto cand = [&](int c) { return c < NC - 1 ? (2 << c) : t_fine; };
    // query tiles per request: one division for batched q, where every request has Sq rows
    const unsigned int mb_batched = Sq > 0 ? (unsigned int)(Sq + pos_per_tile - 1) / pos_per_tile : 0u;
    auto add_units = [&](int lk, int lq) {
        const unsigned int t = lk > 0 ? (unsigned int)(lk + kTileN - 1) / kTileN : 0u;
        const unsigned int mb = !q_varlen ? (lq > 0 ? mb_batched : 0u)
                                          : (lq > 0 ? (unsigned int)(lq + pos_per_tile - 1) / pos_per_tile : 0u);
        tiles += t * mb;
#pragma unroll
        for (int c = 0; c < NC; ++c) units[c] += mb * ((t + (unsigned int)cand(c) - 1u) / (unsigned int)cand(c));
    };
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        if (32 * i < B) add_units(lks[i], lqs[i]);
    for (int b = lane + 32 * kPer; b < B; b += 32)
        add_units(kv_mode == 0 ? Sk : cu_k[b + 1] - cu_k[b], q_varlen ? cu_q[b + 1] - cu_q[b] : Sq);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        tiles += __shfl_xor_sync(0xffffffffu, tiles, o);
#pragma unroll
        for (int c = 0; c < NC; ++c) units[c] += __shfl_xor_sync(0xffffffffu, units[c], o);
    }
    int best_cap = t_fine;  // if no power of two fits n
    float best = 3.0e38f;
    const float inv_slots = 1.f / (float)slots;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const int T = cand(c);
        if (T < t_fine) continue;  // would need more than the launched splits
        const float n_units = (float)units[c] * (float)Hkv;
        const float tail = kFixedTiles + (float)min(T, t_max);
        const float m = n_units <= (float)slots
                            ? tail
                            : (kFixedTiles * n_units + (float)tiles * (float)Hkv) * inv_slots + kTailWeight * tail;
        if (m < best) {
            best = m;
            best_cap = T;
        }
    }
    return best_cap;
}

// One warp: chooses the launch's split cap (split_tile_cap) before the forward kernel runs
// and leaves it in the workspace for the forward and combine kernels.
__global__ void split_plan_kernel(const __grid_constant__ FwdParams p);

// Maps a varlen grid slot to (request, slot within the request): the slots enumerate each
// request's groups of `per_slot` consecutive m-blocks in order; within a request the order
// is reversed so that, with a causal mask, the longer rows start first.  Whole warp must
// call it.
__device__ __forceinline__ bool varlen_slot(const FwdParams &p, int x, int &b, int &mb, int per_slot = 1) {
    const int lane = threadIdx.x & 31;
    const int P = p.pos_per_tile * per_slot;
    int base = 0;
    for (int s0 = 0; s0 < p.B; s0 += 32) {
        const int s = s0 + lane;
        int cnt = 0;
        if (s < p.B) {
            const int len = p.cu_q[s + 1] - p.cu_q[s];
            cnt = len > 0 ? (len + P - 1) / P : 0;
        }
        int inc = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        const int cum = base + inc;
        const unsigned m = __ballot_sync(0xffffffffu, s < p.B && x < cum);
        if (m) {
            const int l = __ffs(m) - 1;
            const int ci = __shfl_sync(0xffffffffu, cum, l);
            const int cn = __shfl_sync(0xffffffffu, cnt, l);
            b = s0 + l;
            mb = cn - 1 - (x - (ci - cn));
            return true;
        }
        base += __shfl_sync(0xffffffffu, inc, 31);
    }
    return false;
}

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

// Writes 8 consecutive output values (one 16-byte store) in bf16 or fp16.
__device__ __forceinline__ void store8(void *dst, const float *v, int fp16) {
    uint4 pk;
    uint32_t *w = reinterpret_cast<uint32_t *>(&pk);
    if (fp16) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
    }
    *reinterpret_cast<uint4 *>(dst) = pk;
}

template <int D, int DV>
__global__ void __launch_bounds__(kNumThreads, 1)
    fwd_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
    using C = Cfg<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // ------------------------------------------------------------ tile schedule
    int cap = p.cap_const > 0 ? p.cap_const : (1 << 20);
    if (p.num_splits > 1 && p.cap_const <= 0) {  // chosen by split_plan_kernel, which may still be running
        ptx::griddep_wait();
        cap = *p.split_cap;
    }
    int b, mb;
    if (!p.q_varlen) {
        const int x = blockIdx.x;
        b = x % p.B;
        mb = p.mblocks_per_batch - 1 - x / p.B;
    } else if (!varlen_slot(p, blockIdx.x, b, mb)) {
        return;  // slot beyond the last request's m-blocks
    }
    const int kvh = blockIdx.y % p.Hkv;
    const int split = blockIdx.y / p.Hkv;
    const int P = p.pos_per_tile;
    const int q_start = p.q_varlen ? p.cu_q[b] : b * p.Sq;
    int Lq = p.q_varlen ? p.cu_q[b + 1] - q_start : p.Sq;
    int Lk, k_start = 0;
    if (p.kv_mode == 0) {
        Lk = p.Sk;
    } else {
        k_start = p.cu_k[b];
        Lk = p.cu_k[b + 1] - k_start;
    }
    // device-side sanity of caller-provided lengths: never index outside the tensors
    bool bad = Lq < 0 || Lk < 0 || q_start < 0 || q_start + Lq > p.total_q;
    if (p.kv_mode == 1) bad |= (k_start < 0 || k_start + Lk > p.total_k);
    if (p.kv_mode == 2) bad |= ((long long)Lk > (long long)p.max_pages * p.page_size);
    if (bad) {
        if (tid == 0) atomicOr(p.status, kStatusBounds);
        return;
    }
    const int pos0 = mb * P;
    if (pos0 >= Lq) return;
    const int pos_last = min(pos0 + P, Lq) - 1;
    const int delta = Lk - Lq;
    const SplitRange sr = split_range(Lq, Lk, pos0, pos_last, p.causal, p.window_left, p.num_splits, cap, split);
    if (split >= sr.eff) return;  // this tile runs fewer splits; the combine skips this one
    const int t_beg = sr.t_beg, n_tiles = sr.n_tiles;

    // ------------------------------------------------------------ per-row facts
    const int r = tid & 127;  // tile row of softmax / correction threads
    const int rpos = pos0 + r / p.G;
    const int hq = kvh * p.G + r % p.G;
    const bool row_ok = r < p.rows_per_tile && rpos < Lq;
    const int tok = q_start + rpos;  // packed query token index
    const long long beta = p.q_varlen ? 0 : b;
    const long long rho = p.q_varlen ? tok : rpos;
    const bool has_sink = p.sink != nullptr && (!p.split_mode || split == 0);

    if (n_tiles == 0) {
        // nothing visible for this CTA: O = 0, LSE = -inf (or the sink logit)
        if (tid < 128 && row_ok) {
            const float lse = has_sink ? p.sink[hq] : -INFINITY;
            if (p.split_mode) {
                const long long row = ((long long)split * p.total_q + tok) * p.Hq + hq;
                p.lse_part[row] = lse;
                float4 *dst = reinterpret_cast<float4 *>(p.o_part + row * DV);
                for (int i = 0; i < DV / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
                if (p.lse) p.lse[beta * p.lse_sb + hq * p.lse_sh + rho * p.lse_ss] = lse;
                uint8_t *dst = reinterpret_cast<uint8_t *>(p.o) +
                               2 * (beta * p.o_sb + rho * p.o_ss + hq * p.o_sh);
                for (int i = 0; i < DV / 8; ++i)
                    *reinterpret_cast<uint4 *>(dst + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        return;
    }

    // ------------------------------------------------------------ shared memory
    uint8_t *misc = smem + C::OFF_MISC;
    const uint32_t bar0 = ptx::smem_u32(misc);
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc + 512);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 516);
    float *alpha_ring = reinterpret_cast<float *>(misc + 1024);  // [NA][128]
    float *row_scale = reinterpret_cast<float *>(misc + 3072);   // [128]
    float *mx_part = reinterpret_cast<float *>(misc + 3584);     // [2 parity][2 half][128]
    float *sum_part = reinterpret_cast<float *>(misc + 5632);    // [128]
    int *two_term_votes = reinterpret_cast<int *>(misc + 6144);   // [NS][8 softmax warps]
    const uint32_t sQ = ptx::smem_u32(smem + C::OFF_Q);
    const uint32_t sK = ptx::smem_u32(smem + C::OFF_K);
    const uint32_t sV = ptx::smem_u32(smem + C::OFF_V);

    if (tid == 0) {
        ptx::mbar_init(BAR(C::B_Q), 1);
        for (int i = 0; i < C::STAGES; ++i) {
            ptx::mbar_init(BAR(C::B_KF + i), 1);
            ptx::mbar_init(BAR(C::B_KE + i), 1);
            ptx::mbar_init(BAR(C::B_VF + i), 1);
            ptx::mbar_init(BAR(C::B_VE + i), 1);
        }
        for (int i = 0; i < C::NS; ++i) {
            ptx::mbar_init(BAR(C::B_SF + i), 1);
            ptx::mbar_init(BAR(C::B_PF + i), 256);
        }
        for (int i = 0; i < C::NOT; ++i) {
            ptx::mbar_init(BAR(C::B_OF + i), 1);
            ptx::mbar_init(BAR(C::B_OE + i), 128);
        }
        for (int i = 0; i < C::NA; ++i) {
            ptx::mbar_init(BAR(C::B_AF + i), 128);
        }
        for (int i = 0; i < 2; ++i) ptx::mbar_init(BAR(C::B_XCH + i), 256);
        ptx::mbar_init(BAR(C::B_SUM), 128);
        ptx::mbar_init(BAR(C::B_FIN), 128);
        ptx::mbar_init(BAR(C::B_DONE), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
#ifdef FA8_TRACE
    for (int i = tid; i < kTraceEvents * kTraceTiles; i += kNumThreads)
        reinterpret_cast<unsigned long long *>(smem + C::OFF_TRACE)[i] = 0ull;
#endif
    if (warp == 12 && lane == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
    }
    if (warp == 13) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::TM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Waiter W{abort_flag, p.timeout_ns, p.status};
    if (tid == 0) FA8_EV(15, 0);

    if (warp >= 12) {
      ptx::setmaxnreg_dec<kRegsCtl>();
      if (warp == 12) {
        // ======================================================== TMA producer
        const bool paged = p.kv_mode == 2;
        int issued_k = 0, issued_v = 0;
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(BAR(C::B_Q), (uint32_t)(D * p.rows_per_tile));
            const int c2 = p.q_varlen ? q_start + pos0 : pos0;
            const int c3 = p.q_varlen ? 0 : b;
#pragma unroll
            for (int c = 0; c < C::NCK; ++c)
                ptx::tma_load_4d(sQ + c * C::CHUNK_Q, &tm_q, BAR(C::B_Q), c * C::CW, kvh * p.G, c2, c3);
        }
        for (int it = 0; it < n_tiles; ++it) {
            const int k0 = (t_beg + it) * kTileN;
            const int st = it % C::STAGES;
            const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
            // paged: lane i looks up the page of box i of this tile
            int page = 0, prow = 0;
            if (paged && lane < p.boxes_per_tile) {
                const int j0 = k0 + lane * p.box_n;
                const int pi = j0 / p.page_size;
                prow = j0 - pi * p.page_size;
                page = p.num_pages;  // past the request's keys: out of range, TMA fills zeros
                if (j0 < Lk) {
                    const int e = p.block_table[(long long)b * p.bt_stride + pi];
                    if (e >= 0 && e < p.num_pages) page = e;
                    else atomicOr(p.status, kStatusBounds);
                }
            }
            const int c2 = p.kv_mode == 1 ? k_start + k0 : k0;
            const int c3 = p.kv_mode == 1 ? 0 : b;
            // K tile
            if (!W.wait_warp(BAR(C::B_KE + st), ph ^ 1u)) break;
            if (lane == 0) ptx::mbar_arrive_expect_tx(BAR(C::B_KF + st), (uint32_t)C::K_BYTES);
            __syncwarp();
            const uint32_t dK = sK + st * C::K_BYTES;
            if (paged) {
                if (lane < p.boxes_per_tile) {
#pragma unroll
                    for (int c = 0; c < C::NCK; ++c)
                        ptx::tma_load_4d(dK + c * C::CHUNK_K + lane * p.box_n * C::CW, &tm_k,
                                         BAR(C::B_KF + st), c * C::CW, kvh, prow, page);
                }
            } else if (lane == 0) {
#pragma unroll
                for (int c = 0; c < C::NCK; ++c)
                    ptx::tma_load_4d(dK + c * C::CHUNK_K, &tm_k, BAR(C::B_KF + st), c * C::CW, kvh, c2, c3);
            }
            issued_k = it + 1;
            // V tile
            if (!W.wait_warp(BAR(C::B_VE + st), ph ^ 1u)) break;
            if (lane == 0) ptx::mbar_arrive_expect_tx(BAR(C::B_VF + st), (uint32_t)C::V_BYTES);
            __syncwarp();
            const uint32_t dV = sV + st * C::V_BYTES;
            if (paged) {
                if (lane < p.boxes_per_tile) {
#pragma unroll
                    for (int c = 0; c < C::NCV; ++c)
                        ptx::tma_load_4d(dV + c * C::CHUNK_V + lane * p.box_n * C::CWV, &tm_v,
                                         BAR(C::B_VF + st), c * C::CWV, kvh, prow, page);
                }
            } else if (lane == 0) {
#pragma unroll
                for (int c = 0; c < C::NCV; ++c)
                    ptx::tma_load_4d(dV + c * C::CHUNK_V, &tm_v, BAR(C::B_VF + st), c * C::CWV, kvh, c2, c3);
            }
            issued_v = it + 1;
        }
        if (*abort_flag) {
            // every load already issued must land before the CTA's smem is released;
            // the newest load of each ring slot is the one that can still be in flight
            W.drain(BAR(C::B_Q), 0);
            for (int i = max(0, issued_k - C::STAGES); i < issued_k; ++i)
                W.drain(BAR(C::B_KF + i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u);
            for (int i = max(0, issued_v - C::STAGES); i < issued_v; ++i)
                W.drain(BAR(C::B_VF + i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u);
        }
        __syncwarp();
    } else if (warp == 13) {
        // ======================================================== MMA issuer
        // The whole warp runs this loop (uniform control flow); one elected lane issues the
        // tcgen05 operations.  Shared-memory descriptors are built once and advanced by
        // compile-time byte offsets (start-address field, units of 16 bytes).
        constexpr uint32_t kIdescQK = idesc_e4m3(kTileM, kTileN, false);
        constexpr uint32_t kIdescPV = idesc_e4m3(kTileM, C::OTW, true);
        const uint64_t dq0 = sdesc(sQ, 16, 8 * C::CW, swz_layout(C::CW));
        const uint64_t dk0 = sdesc(sK, 16, 8 * C::CW, swz_layout(C::CW));
        const uint64_t dv0 = sdesc(sV, C::CHUNK_V, 8 * C::CWV, swz_layout(C::CWV));
        const bool leader = ptx::elect_one();
        int pv_uses = 0;
        bool ok = W.wait_warp(BAR(C::B_Q), 0);
        ptx::tc_fence_after();
        auto do_pv = [&](int j) -> bool {
            const int sb = j % C::NS;
            const int vs = j % C::STAGES;
            if (!W.wait_warp(BAR(C::B_PF + sb), (uint32_t)(j / C::NS) & 1u)) return false;
            FA8_EV(10, j);
            if (!W.wait_warp(BAR(C::B_VF + vs), (uint32_t)(j / C::STAGES) & 1u)) return false;
            FA8_EV(11, j);
            ptx::tc_fence_after();
            // two-term P: every softmax warp wrote its vote before arriving on B_PF
            const volatile int *votes = two_term_votes + sb * 8;
            const bool two_term = tile_needs_mask((t_beg + j) * kTileN, Lk, p.causal, p.window_left, pos0,
                                                  pos_last, delta) ||
                                  (votes[0] | votes[1] | votes[2] | votes[3] | votes[4] | votes[5] | votes[6] |
                                   votes[7]) != 0;
            const uint64_t dv_stage = dv0 + (uint64_t)((vs * C::V_BYTES) >> 4);
            const uint32_t s_col = tmem + C::TM_S + sb * 128;
#pragma unroll
            for (int c = 0; c < C::NPV; ++c) {
                const int ob = pv_uses % C::NOT;
                const uint32_t otile = tmem + C::TM_OT + ob * C::OTW;
                if (!W.wait_warp(BAR(C::B_OE + ob), ((uint32_t)(pv_uses / C::NOT) & 1u) ^ 1u)) return false;
                FA8_EV(12, j);
                ptx::tc_fence_after();
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < kTileN / 32; ++kk) {
                        const uint64_t bd = dv_stage + (uint64_t)(((c * C::OTW / C::CWV) * C::CHUNK_V + kk * 32 * C::CWV) >> 4);
                        ptx::mma_f8_ts(otile, s_col + kk * 32, bd, kIdescPV, kk > 0 ? 1u : 0u);
                    }
                    if (two_term) {  // + P_lo V (P_lo 8 columns after each P_hi slice)
#pragma unroll
                        for (int kk = 0; kk < kTileN / 32; ++kk) {
                            const uint64_t bd = dv_stage + (uint64_t)(((c * C::OTW / C::CWV) * C::CHUNK_V + kk * 32 * C::CWV) >> 4);
                            ptx::mma_f8_ts(otile, s_col + kk * 32 + 8, bd, kIdescPV, 1u);
                        }
                    }
                    ptx::tc_commit(BAR(C::B_OF + ob));
                }
                __syncwarp();
                ++pv_uses;
            }
            if (leader) ptx::tc_commit(BAR(C::B_VE + vs));
            __syncwarp();
            FA8_EV(3, j);
            return true;
        };
        for (int it = 0; ok && it < n_tiles; ++it) {
            const int ks = it % C::STAGES;
            if (!W.wait_warp(BAR(C::B_KF + ks), (uint32_t)(it / C::STAGES) & 1u)) { ok = false; break; }
            FA8_EV(9, it);
            ptx::tc_fence_after();
            if (C::NS == 1 && it > 0 && !do_pv(it - 1)) { ok = false; break; }
            const int sb = it % C::NS;
            const uint64_t dk_stage = dk0 + (uint64_t)((ks * C::K_BYTES) >> 4);
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk) {
                    const uint32_t off = (uint32_t)((((kk * 32) / C::CW) * C::CHUNK_Q + (kk * 32) % C::CW) >> 4);
                    ptx::mma_f8_ss(tmem + C::TM_S + sb * 128, dq0 + off, dk_stage + off, kIdescQK, kk > 0 ? 1u : 0u);
                }
                ptx::tc_commit(BAR(C::B_SF + sb));
                ptx::tc_commit(BAR(C::B_KE + ks));
            }
            __syncwarp();
            FA8_EV(2, it);
            if (C::NS == 2 && it > 0 && !do_pv(it - 1)) { ok = false; break; }
        }
        if (ok) ok = do_pv(n_tiles - 1);
        // all MMAs must finish before TMEM is released
        if (leader) ptx::tc_commit(BAR(C::B_DONE));
        __syncwarp();
        W.drain(BAR(C::B_DONE), 0);
        __syncwarp();
      }
    } else if (warp < 8) {
      ptx::setmaxnreg_dec<kRegsSoft>();
      {
        // ======================================================== softmax (half h of each row)
        const int h = warp >> 2;  // keys [64 h, 64 h + 64) of every tile
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const bool warp_active = __any_sync(0xffffffffu, row_ok);
        const float dqv = p.dq ? p.dq[b * p.dq_sb + kvh * p.dq_sh] : 1.f;
        const float dkv = p.dk ? p.dk[b * p.dk_sb + kvh * p.dk_sh] : 1.f;
        const float c = p.scale_log2 * dqv * dkv;
        const uint64_t c2 = ptx::f2pack(c, c);
        const int hi_row = p.causal ? min(Lk - 1, rpos + delta) : Lk - 1;
        const int lo_row = p.window_left >= 0 ? max(0, rpos + delta - p.window_left) : 0;
        float m_run = -INFINITY, row_sum = 0.f;  // identical m_run in both halves
        for (int it = 0; it < n_tiles; ++it) {
            const int k0 = (t_beg + it) * kTileN;
            const int sb = it % C::NS;
            if (!W.wait_warp(BAR(C::B_SF + sb), (uint32_t)(it / C::NS) & 1u)) break;
            if (tid == 0) FA8_EV(4, it);
            ptx::tc_fence_after();
            const uint32_t scol = tmem + lane_base + C::TM_S + sb * 128 + 64 * h;
            const bool need_mask = tile_needs_mask(k0, Lk, p.causal, p.window_left, pos0, pos_last, delta);
            const int hi = hi_row - k0 - 64 * h, lo = lo_row - k0 - 64 * h;  // visible: [lo, hi]
            uint32_t u[2][32];
            float mh = -INFINITY;
            if (warp_active) {
                ptx::tmem_ld32(scol, u[0]);
                ptx::tmem_ld32(scol + 32, u[1]);
                ptx::tmem_wait_ld();
                ptx::reg_fence32(u[0]);
                ptx::reg_fence32(u[1]);
                if (tid == 0) FA8_EV(0, it);
                if (need_mask) {
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        if (i > hi || i < lo) u[i >> 5][i & 31] = __float_as_uint(-INFINITY);
                }
                float mq[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t *v = &u[q >> 1][(q & 1) * 16];
                    float m = ptx::fmax3(u2f(v[0]), u2f(v[1]), u2f(v[2]));
#pragma unroll
                    for (int i = 3; i < 15; i += 2) m = ptx::fmax3(m, u2f(v[i]), u2f(v[i + 1]));
                    mq[q] = fmaxf(m, u2f(v[15]));
                }
                mh = fmaxf(ptx::fmax3(mq[0], mq[1], mq[2]), mq[3]);
            }
            // exchange the half-row maxima (double-buffered slots, bounded wait)
            mx_part[((it & 1) * 2 + h) * 128 + r] = mh;
            ptx::mbar_arrive(BAR(C::B_XCH + (it & 1)));
            if (!W.wait_warp(BAR(C::B_XCH + (it & 1)), (uint32_t)(it >> 1) & 1u)) break;
            const float mx = fmaxf(mh, mx_part[((it & 1) * 2 + (h ^ 1)) * 128 + r]);
            if (tid == 0) FA8_EV(1, it);
            float alpha = 1.f;
            bool two_term = need_mask;
            if (warp_active) {
                const float mt = mx * c;
                if (mt > m_run + kTau) {
                    alpha = ptx::ex2(m_run - mt);
                    row_sum *= alpha;
                    m_run = mt;
                }
                if (!need_mask) {
                    // a dominant key: the tile's largest p against this half's mass so far (at
                    // most the row's, so the vote errs towards two terms)
                    const float pm = ptx::ex2(mt - m_run + kPBias);
                    two_term = __any_sync(0xffffffffu, row_ok && pm > kTwoTermShare * (row_sum + pm));
                }
                // p = 2^(s c - m) in f16 (MUFU, two values per instruction; the argument is
                // near 0 where p is large, so f16 keeps it to 2^-11), P = e4m3(2^8 p) with the
                // scaling exact in f16; the row sum adds the f16 p in groups of eight, then fp32
                const float nm = m_run == -INFINITY ? 0.f : -m_run;
                const uint64_t nm2 = ptx::f2pack(nm, nm);
                constexpr uint32_t kH2Bias = 0x5C005C00u;  // f16x2 {256, 256}
                uint64_t acc = ptx::f2pack(0.f, 0.f);
                // the packed E4M3 of keys [32q, 32q+32) goes to column 32q of the S buffer
                // (P_lo 8 columns later on masked tiles)
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    uint32_t w[8];
                    uint32_t e4_prev = 0u;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        float y0, y1, y2, y3;
                        ptx::f2unpack(ptx::ffma2(ptx::f2pack(u2f(u[g][4 * k]), u2f(u[g][4 * k + 1])), c2, nm2), y0, y1);
                        ptx::f2unpack(ptx::ffma2(ptx::f2pack(u2f(u[g][4 * k + 2]), u2f(u[g][4 * k + 3])), c2, nm2), y2, y3);
                        const uint32_t e01 = ptx::ex2_h2(ptx::cvt_f16x2(y1, y0));
                        const uint32_t e23 = ptx::ex2_h2(ptx::cvt_f16x2(y3, y2));
                        // the row sum adds groups of eight f16 p (each at most 2^0.75, so a
                        // group's sum stays below 14 with an f16 rounding of at most 2^-8)
                        // and then accumulates in fp32
                        const uint32_t e4 = ptx::hadd2(e01, e23);
                        if (k & 1) {
                            float s0, s1;
                            ptx::h2_to_f32(ptx::hadd2(e4_prev, e4), s0, s1);
                            acc = ptx::fadd2(acc, ptx::f2pack(s0, s1));
                        } else {
                            e4_prev = e4;
                        }
                        const uint32_t q01 = ptx::hmul2(e01, kH2Bias), q23 = ptx::hmul2(e23, kH2Bias);
                        w[k] = ptx::cvt_e4m3x2_h2(q01) | (ptx::cvt_e4m3x2_h2(q23) << 16);
                        u[g][2 * k] = q01;  // kept for the second term
                        u[g][2 * k + 1] = q23;
                    }
                    ptx::tmem_st8(scol + 32 * g, w);
                    if (two_term) {
                        // second E4M3 term on masked tiles: P_lo = e4m3(2^8 p - P_hi), in f16
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const uint32_t d01 = ptx::hsub2(u[g][2 * k], ptx::e4m3x2_to_h2(w[k] & 0xFFFFu));
                            const uint32_t d23 = ptx::hsub2(u[g][2 * k + 1], ptx::e4m3x2_to_h2(w[k] >> 16));
                            w[k] = ptx::cvt_e4m3x2_h2(d01) | (ptx::cvt_e4m3x2_h2(d23) << 16);
                        }
                        ptx::tmem_st8(scol + 32 * g + 8, w);
                    } else {
                        // another warp may vote for two terms: this warp's second term is zero
#pragma unroll
                        for (int k = 0; k < 8; ++k) w[k] = 0u;
                        ptx::tmem_st8(scol + 32 * g + 8, w);
                    }
                }
                if (tid == 0) FA8_EV(13, it);
                ptx::tmem_wait_st();
                float a0, a1;
                ptx::f2unpack(acc, a0, a1);
                // the f16 p carry no 2^8 factor: scale the tile's sum to the biased row sum
                row_sum += (a0 + a1) * 256.f;
            }
            if (lane == 0) two_term_votes[sb * 8 + warp] = two_term ? 1 : 0;
            ptx::tc_fence_before();
            ptx::mbar_arrive(BAR(C::B_PF + sb));
            if (tid == 0) FA8_EV(5, it);
            if (h == 0) {
                const int as = it % C::NA;
                alpha_ring[as * 128 + r] = alpha;
                ptx::mbar_arrive(BAR(C::B_AF + as));
                if (tid == 0) FA8_EV(6, it);
            }
        }
        // combine the two halves' row sums, then finalize: the 2^8 bias cancels between O
        // and row_sum and is removed from the LSE
        if (h == 1) {
            sum_part[r] = row_sum;
            ptx::mbar_arrive(BAR(C::B_SUM));
        } else {
            const bool got = W.wait_warp(BAR(C::B_SUM), 0);
            row_sum += got ? sum_part[r] : 0.f;
            const float dvv = p.dv ? p.dv[b * p.dv_sb + kvh * p.dv_sh] : 1.f;
            float scale_o = 0.f, lse;
            const float sig = has_sink ? p.sink[hq] : 0.f;
            if (m_run == -INFINITY) {
                lse = has_sink ? sig : -INFINITY;
            } else {
                const float sl2 = sig * kLog2e;
                const float m_f = (has_sink && sl2 > m_run) ? sl2 : m_run;
                const float sc = ptx::ex2(m_run - m_f);
                const float rs = row_sum * sc + (has_sink ? ptx::ex2(sl2 - m_f + kPBias) : 0.f);
                scale_o = sc * dvv / rs;
                lse = (ptx::lg2(rs) + m_f - kPBias) * kLn2;
            }
            row_scale[r] = scale_o;
            ptx::mbar_arrive(BAR(C::B_FIN));
            if (row_ok) {
                if (p.split_mode)
                    p.lse_part[((long long)split * p.total_q + tok) * p.Hq + hq] = lse;
                else if (p.lse)
                    p.lse[beta * p.lse_sb + hq * p.lse_sh + rho * p.lse_ss] = lse;
            }
        }
      }
    } else {
      ptx::setmaxnreg_inc<kRegsCorr>();
      {
        // ======================================================== correction (warps 8-11)
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const bool warp_active = __any_sync(0xffffffffu, row_ok);
        float o[C::O_REGS ? DV : 1];
#pragma unroll
        for (int i = 0; i < (C::O_REGS ? DV : 1); ++i) o[i] = 0.f;
        int pv_uses = 0;
        bool ok = true;
        for (int it = 0; ok && it < n_tiles; ++it) {
            const int as = it % C::NA;
            if (!W.wait_warp(BAR(C::B_AF + as), (uint32_t)(it / C::NA) & 1u)) break;
            const float alpha = alpha_ring[as * 128 + r];
#pragma unroll
            for (int c = 0; c < C::NPV; ++c) {
                const int ob = pv_uses % C::NOT;
                if (!W.wait_warp(BAR(C::B_OF + ob), (uint32_t)(pv_uses / C::NOT) & 1u)) { ok = false; break; }
                if (tid == 256 && c == 0) FA8_EV(7, it);
                ptx::tc_fence_after();
                const uint32_t otile = tmem + lane_base + C::TM_OT + ob * C::OTW;
                if (warp_active) {
                    if constexpr (C::O_REGS) {
                        // one 32-column slice at a time, packed fold
                        const uint64_t a2 = ptx::f2pack(alpha, alpha);
#pragma unroll
                        for (int j = 0; j < C::OTW / 32; ++j) {
                            uint32_t u[32];
                            ptx::tmem_ld32(otile + 32 * j, u);
                            ptx::tmem_wait_ld();
                            ptx::reg_fence32(u);
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                // O starts at 0 and the first visible tile has alpha = 0,
                                // so no first-tile special case is needed
                                const int idx = (C::O_REGS ? (32 * j + i) : 0);
                                const uint64_t r2 = ptx::ffma2(ptx::f2pack(o[idx], o[idx + 1]), a2,
                                                               ptx::f2pack(u2f(u[i]), u2f(u[i + 1])));
                                ptx::f2unpack(r2, o[idx], o[idx + 1]);
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < C::OTW / 32; ++j) {
                            uint32_t u[32];
                            ptx::tmem_ld32(otile + 32 * j, u);
                            const uint32_t orun = tmem + lane_base + C::TM_OR + c * C::OTW + 32 * j;
                            uint32_t v[32];
                            if (it > 0) {
                                ptx::tmem_ld32(orun, v);
                                ptx::tmem_wait_ld();
                                ptx::reg_fence32(u);
                                ptx::reg_fence32(v);
#pragma unroll
                                for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(fmaf(u2f(v[i]), alpha, u2f(u[i])));
                            } else {
                                ptx::tmem_wait_ld();
                                ptx::reg_fence32(u);
#pragma unroll
                                for (int i = 0; i < 32; ++i) v[i] = u[i];
                            }
                            ptx::tmem_st32(orun, v);
                            ptx::tmem_wait_st();
                        }
                    }
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(BAR(C::B_OE + ob));
                if (tid == 256 && c == C::NPV - 1) FA8_EV(8, it);
                ++pv_uses;
            }
        }
        const bool fin = W.wait_warp(BAR(C::B_FIN), 0);
        const float sc = fin ? row_scale[r] : 0.f;
        // TMEM loads are warp-collective (.sync.aligned): the whole active warp loads, only
        // the valid rows store.
        if (warp_active) {
            if (p.split_mode) {
                float *dst = p.o_part + (((long long)split * p.total_q + tok) * p.Hq + hq) * DV;
                if constexpr (C::O_REGS) {
                    if (row_ok) {
#pragma unroll
                        for (int i = 0; i < DV; i += 4)
                            *reinterpret_cast<float4 *>(dst + i) =
                                make_float4(o[i] * sc, o[i + 1] * sc, o[i + 2] * sc, o[i + 3] * sc);
                    }
                } else {
#pragma unroll 1
                    for (int j = 0; j < DV / 32; ++j) {
                        uint32_t v[32];
                        ptx::tmem_ld32(tmem + lane_base + C::TM_OR + 32 * j, v);
                        ptx::tmem_wait_ld();
                        ptx::reg_fence32(v);
                        if (row_ok) {
#pragma unroll
                            for (int i = 0; i < 32; i += 4)
                                *reinterpret_cast<float4 *>(dst + 32 * j + i) = make_float4(
                                    u2f(v[i]) * sc, u2f(v[i + 1]) * sc, u2f(v[i + 2]) * sc, u2f(v[i + 3]) * sc);
                        }
                    }
                }
            } else {
                uint8_t *dst = reinterpret_cast<uint8_t *>(p.o) + 2 * (beta * p.o_sb + rho * p.o_ss + hq * p.o_sh);
                if constexpr (C::O_REGS) {
                    if (row_ok) {
#pragma unroll
                        for (int i = 0; i < DV; i += 8) {
                            float t8[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) t8[e] = o[i + e] * sc;
                            store8(dst + 2 * i, t8, p.out_fp16);
                        }
                    }
                } else {
#pragma unroll 1
                    for (int j = 0; j < DV / 32; ++j) {
                        uint32_t v[32];
                        ptx::tmem_ld32(tmem + lane_base + C::TM_OR + 32 * j, v);
                        ptx::tmem_wait_ld();
                        ptx::reg_fence32(v);
                        if (row_ok) {
#pragma unroll
                            for (int i = 0; i < 32; i += 8) {
                                float t8[8];
#pragma unroll
                                for (int e = 0; e < 8; ++e) t8[e] = u2f(v[i + e]) * sc;
                                store8(dst + 2 * (32 * j + i), t8, p.out_fp16);
                            }
                        }
                    }
                }
            }
        }
    }
    }
    // ------------------------------------------------------------ teardown
    ptx::tc_fence_before();
    __syncthreads();
#ifdef FA8_TRACE
    if (tid == 0) FA8_EV(15, 1);
    __syncthreads();
    if (p.trace && blockIdx.y == 0 && blockIdx.x < kTraceCtas) {
        const unsigned long long *src = reinterpret_cast<const unsigned long long *>(smem + C::OFF_TRACE);
        for (int i = tid; i < kTraceEvents * kTraceTiles; i += kNumThreads)
            p.trace[(size_t)blockIdx.x * kTraceEvents * kTraceTiles + i] = src[i];
    }
#endif
    if (warp == 13) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::TM_COLS);
    }
}

// Split-KV merge: one warp per (token, q-head) row.
//   LSE = log sum_s exp(LSE_s),  O = sum_s exp(LSE_s - LSE) O_s
// Splits with LSE_s = -inf contribute nothing (their O_s is zero).
template <int DV>
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ CombineParams p) {
    constexpr int PER = DV / 32;  // output columns per lane
    __shared__ __align__(16) float part[8][DV];
    __shared__ int part_used[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = p.wpr;
    const int sub = warp % W;
    const long long row = (long long)blockIdx.x * (8 / W) + warp / W;
    const long long rows = (long long)p.total_q * p.Hq;
    const bool active = row < rows;
    const long long stride_s = rows;
    const int tok = (int)(row / p.Hq);
    const int hq = (int)(row % p.Hq);
    // this grid may start while the forward kernel ahead of it drains (programmatic
    // dependent launch): its partials are complete and visible past this point
    ptx::griddep_wait();
    // the splits the forward ran for this row's tile (split_range on the same inputs)
    int ns = 1;
    if (active) {
        int b = 0, pos = tok, Lq = p.Sq;
        if (p.q_varlen) {
            int lo = 0, hi = p.B - 1;  // last request whose first token is <= tok
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (p.cu_q[mid] <= tok) lo = mid;
                else hi = mid - 1;
            }
            b = lo;
            pos = tok - p.cu_q[b];
            Lq = p.cu_q[b + 1] - p.cu_q[b];
        } else {
            b = tok / p.Sq;
            pos = tok - b * p.Sq;
        }
        const int Lk = p.kv_mode == 0 ? p.Sk : p.cu_k[b + 1] - p.cu_k[b];
        const int pos0 = pos / p.pos_per_tile * p.pos_per_tile;
        const int pos_last = min(pos0 + p.pos_per_tile, Lq) - 1;
        ns = split_range(Lq, Lk, pos0, pos_last, p.causal, p.window_left, p.num_splits,
                         p.cap_const > 0 ? p.cap_const : *p.split_cap, 0).eff;
    }
    // every warp reads all the row's split LSEs (a few floats) for the max and the sum
    float m = -INFINITY;
    if (active)
        for (int s = lane; s < ns; s += 32) m = fmaxf(m, p.lse_part[s * stride_s + row]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    float lse = -INFINITY;
    bool used = false;
    if (active && m != -INFINITY) {
        float sw = 0.f;
        for (int s = lane; s < ns; s += 32) {
            const float l = p.lse_part[s * stride_s + row];
            if (l != -INFINITY) sw += ptx::ex2((l - m) * kLog2e);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sw += __shfl_xor_sync(0xffffffffu, sw, o);
        lse = m + ptx::lg2(sw) * kLn2;
        const float inv = 1.f / sw;
        // this warp's splits, four loads in flight per lane
        for (int s0 = sub; s0 < ns; s0 += 4 * W) {
            float wgt[4];
            float v[4][PER];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int s = s0 + u * W;
                const float l = s < ns ? p.lse_part[s * stride_s + row] : -INFINITY;
                wgt[u] = l == -INFINITY ? 0.f : ptx::ex2((l - m) * kLog2e) * inv;
                if (wgt[u] != 0.f) {
                    const float *src = p.o_part + (s * stride_s + row) * DV + lane * PER;
                    if constexpr (PER % 4 == 0) {
#pragma unroll
                        for (int i = 0; i < PER; i += 4) {
                            const float4 x = *reinterpret_cast<const float4 *>(src + i);
                            v[u][i] = x.x;
                            v[u][i + 1] = x.y;
                            v[u][i + 2] = x.z;
                            v[u][i + 3] = x.w;
                        }
                    } else if constexpr (PER % 2 == 0) {
#pragma unroll
                        for (int i = 0; i < PER; i += 2) {
                            const float2 x = *reinterpret_cast<const float2 *>(src + i);
                            v[u][i] = x.x;
                            v[u][i + 1] = x.y;
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < PER; ++i) v[u][i] = src[i];
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (wgt[u] == 0.f) continue;
#pragma unroll
                for (int i = 0; i < PER; ++i) acc[i] = used ? fmaf(wgt[u], v[u][i], acc[i]) : wgt[u] * v[u][i];
                used = true;
            }
        }
    }
    // the W warps of a row add their partial sums (only warps that had a split with keys,
    // so that a single contributing split passes through unchanged)
#pragma unroll
    for (int i = 0; i < PER; ++i) part[warp][lane * PER + i] = acc[i];
    if (lane == 0) part_used[warp] = used ? 1 : 0;
    __syncthreads();
    if (!active || sub != 0) return;
    bool any = used;
    for (int w2 = warp + 1; w2 < warp + W; ++w2) {
        if (!part_used[w2]) continue;
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] = any ? acc[i] + part[w2][lane * PER + i] : part[w2][lane * PER + i];
        any = true;
    }
    const long long beta = p.q_varlen ? 0 : tok / p.Sq;
    const long long rho = p.q_varlen ? tok : tok % p.Sq;
    if (lane == 0 && p.lse) p.lse[beta * p.lse_sb + hq * p.lse_sh + rho * p.lse_ss] = lse;
    uint8_t *dst = reinterpret_cast<uint8_t *>(p.o) + 2 * (beta * p.o_sb + rho * p.o_ss + hq * p.o_sh + lane * PER);
    if constexpr (PER % 2 == 0) {
#pragma unroll
        for (int i = 0; i < PER; i += 2) {
            uint32_t w;
            if (p.out_fp16) {
                __half2 h = __floats2half2_rn(acc[i], acc[i + 1]);
                w = *reinterpret_cast<uint32_t *>(&h);
            } else {
                __nv_bfloat162 h = __floats2bfloat162_rn(acc[i], acc[i + 1]);
                w = *reinterpret_cast<uint32_t *>(&h);
            }
            *reinterpret_cast<uint32_t *>(dst + 2 * i) = w;
        }
    } else {  // odd columns per lane (dv = 96): one 16-bit store each
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            uint16_t w;
            if (p.out_fp16) {
                const __half h = __float2half_rn(acc[i]);
                w = *reinterpret_cast<const uint16_t *>(&h);
            } else {
                const __nv_bfloat16 h = __float2bfloat16_rn(acc[i]);
                w = *reinterpret_cast<const uint16_t *>(&h);
            }
            *reinterpret_cast<uint16_t *>(dst + 2 * i) = w;
        }
    }
}

// One CTA, one thread: a bounded wait on a barrier that nothing completes.
__global__ void wait_probe_kernel(unsigned long long timeout_ns, unsigned int *status);

}  // namespace fa8
