// fa8_prefill.cuh -- the forward for many query rows per kv-head (prefill, chunked prefill)
// with dv <= 128: two 128-row Q tiles per CTA that take turns on the tensor core.
//
// Same arithmetic as fwd_kernel ("[Cute,Fwd,Sm90] Native FP8 (E4M3 Q/K/V) forward for
// Hopper", Design; "tml-fa4 PR #4", Summary and "Correctness fix over #1"): S = Q K^T in
// TMEM (tcgen05.mma kind::f8f6f4), lazy running max (tau = 0.75 in log2 units), P =
// e4m3(2^(s c - m + 8)) written over S in TMEM, O_t = P V accumulated from zero for every
// KV tile and folded into an fp32 O as O = O * alpha + O_t (two-level accumulation), and
// O * dv / rowsum, LSE = ln2 * (log2 rowsum + m - 8) at the end; a tile's P takes a second
// E4M3 term (P_lo = e4m3(p - P_hi)) when the tile needs a mask or one key of some row holds
// about an eighth or more of that row's mass so far.
//
// The CTA's rows are 2 x 128 (query position, q-head) pairs of one kv-head group, packed
// position-major (PackGQA): tile A takes the first half of the CTA's positions, tile B the
// second.  Both share every K/V tile.  Roles (384 threads, three warpgroups):
//   warps 0-3   tile A: thread r owns TMEM lane r = row r of A; it runs the row's softmax
//               (two passes over the S columns: the row maximum, then P), keeps the row's
//               running O in 128 registers and folds every O_t into it, and writes the row
//   warps 4-7   the same for tile B
//   warp 8      TMA producer (Q of both tiles once, K/V tiles into an S-stage ring)
//   warp 9      MMA issuer (one elected lane) and TMEM owner
//   warps 10-11 idle (their registers go to the two tile warpgroups)
// TMEM (512 columns): S/P of A at 0, S/P of B at 128, O_t of A at 256, O_t of B at 384.
// A build with -DFA8_TRACE records clock64() per KV tile of the first 8 CTAs (debug only):
// tile A, warp 0: 0 S ready, 1 max pass done, 9 / 10 P pass start / end, 2 P written, 11 the
// tile's path (bit 0 two terms, bit 1 masked; a value, not a clock); 5-7 P written by warps
// 1-3; issuer: 8 iteration start, 12 / 13 tile A / B's PV and next QK issued, 14 both done;
// 15 tile B's S ready.
// The issuer runs, per KV tile j, PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1): while one tile's
// warpgroup turns S into P (and folds the previous O_t), the other tile's MMAs run, so every
// sub-partition has two warps on independent work (one per tile).  FlashAttention-4 pairs
// two Q tiles the same way ("PyTorch ... FlashAttention-4 MXFP8", 2.1 Attention Forward,
// TMEM allocation); here each tile's O_t has its own TMEM columns and the running O lives in
// the registers of the warpgroup that owns the tile, which is what two-level accumulation
// needs and what lets S, O_t of both tiles fill TMEM exactly.
#pragma once

#include "fa8_kernel.cuh"

namespace fa8 {

constexpr int kPfThreads = 384;

// registers per thread: launch 168 (384 x 168 <= 64K); setmaxnreg gives the two tile
// warpgroups 216 each (O in 128 of them) and 72 to the control warpgroup
constexpr int kPfLaunchRegs = 168;
constexpr int kPfRegsTile = 216;
constexpr int kPfRegsCtl = 72;
static_assert(2 * kPfRegsTile + kPfRegsCtl == 3 * kPfLaunchRegs, "register split");

template <int D, int DV>
struct PfCfg {
    static_assert(DV <= 128 && DV % 32 == 0 && D % 32 == 0, "prefill kernel: dv <= 128");
    static constexpr int CW = (D % 128 == 0) ? 128 : ((D % 64 == 0) ? 64 : 32);
    static constexpr int NCK = D / CW;
    static constexpr int CWV = (DV % 128 == 0) ? 128 : ((DV % 64 == 0) ? 64 : 32);
    static constexpr int NCV = DV / CWV;
    static constexpr int CHUNK_Q = kTileM * CW;
    static constexpr int CHUNK_K = kTileN * CW;
    static constexpr int CHUNK_V = kTileN * CWV;
    static constexpr int Q_BYTES = kTileM * D;  // one Q tile
    static constexpr int K_BYTES = kTileN * D;
    static constexpr int V_BYTES = kTileN * DV;
    static constexpr int MISC_BYTES = 1024;
    static constexpr int SMEM_LIMIT = 232448;  // max dynamic smem per block on sm_103
    static constexpr int STAGES_FIT =
        (SMEM_LIMIT - 1024 - MISC_BYTES - kTraceSmemBytes - 2 * Q_BYTES) / (K_BYTES + V_BYTES);
    static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
    static constexpr int OFF_Q = 0;  // tile A, then tile B
    static constexpr int OFF_K = 2 * Q_BYTES;
    static constexpr int OFF_V = OFF_K + STAGES * K_BYTES;
    static constexpr int OFF_MISC = OFF_V + STAGES * V_BYTES;
    static constexpr int OFF_TRACE = OFF_MISC + MISC_BYTES;
    static constexpr int SMEM_BYTES = OFF_TRACE + kTraceSmemBytes + 1024;
    static constexpr uint32_t TM_S = 0;     // S/P of tile x at TM_S + 128 x
    static constexpr uint32_t TM_OT = 256;  // O_t of tile x at TM_OT + 128 x
    static constexpr uint32_t TM_COLS = 512;
    // barriers: Q (2), K/V ring, then per tile S written, P written, O_t written, O_t folded
    static constexpr int B_Q = 0;
    static constexpr int B_KF = 2;
    static constexpr int B_KE = B_KF + STAGES;
    static constexpr int B_VF = B_KE + STAGES;
    static constexpr int B_VE = B_VF + STAGES;
    static constexpr int B_SF = B_VE + STAGES;
    static constexpr int B_PF = B_SF + 2;
    static constexpr int B_OF = B_PF + 2;
    static constexpr int B_OE = B_OF + 2;
    static constexpr int B_DONE = B_OE + 2;
    static constexpr int NUM_BARS = B_DONE + 1;
    static constexpr int OFF_TMEM_SLOT = 512;  // within the misc area
    static constexpr int OFF_ABORT = 516;
    static constexpr int OFF_VOTES = 528;  // [tile][warp] two-term votes
    static_assert(STAGES >= 2, "smem too small for two K/V stages");
    static_assert(NUM_BARS * 8 <= 512, "barrier area");
    static_assert(Q_BYTES % 1024 == 0 && K_BYTES % 1024 == 0 && V_BYTES % 1024 == 0, "swizzle alignment");
};

// Key range [kv_beg, kv_end) visible to query positions [pos_first, pos_last] and its KV
// tiles [tb, te) clipped to the split's tiles [t0, t1); empty when tb >= te.
struct TileSpan {
    int tb, te;
};
__device__ __forceinline__ TileSpan tile_span(int pos_first, int pos_last, int Lk, int delta, int causal,
                                              int window_left, int t0, int t1) {
    TileSpan s{0, 0};
    if (pos_last < pos_first) return s;
    const int kv_end = causal ? min(Lk, pos_last + delta + 1) : Lk;
    const int kv_beg = window_left >= 0 ? max(0, pos_first + delta - window_left) : 0;
    if (kv_end <= kv_beg) return s;
    s.tb = max(t0, kv_beg / kTileN);
    s.te = min(t1, (kv_end + kTileN - 1) / kTileN);
    if (s.te < s.tb) s.te = s.tb;
    return s;
}

// The P pass of one tile row (128 keys, 32 at a time) for the thread that owns the row:
// p = 2^(s c - m) on f16 pairs (one MUFU instruction for two scores; the argument is near 0
// where p is large, so f16 keeps it to 2^-11), P = e4m3(2^8 p) with the scaling exact in f16
// (and P_lo = e4m3(2^8 p - P_hi) when TWO) written into the S columns, and the row sum (of p,
// without the 2^8) over f16 groups of eight, then fp32.  The same steps fold the previous KV
// tile's O_t into the running O (O = O alpha + O_t, 16 columns at a time; zeros before the
// first KV tile), whose FFMAs fill issue slots the MUFU-bound exponentials leave.  The P of keys
// [32 kq, 32 kq + 32) goes to column 32 kq (8 columns), P_lo 8 columns later: both on S columns
// this step has read.  No branch inside: on tiles that need a mask, the max pass has already
// written -inf over the masked S columns.
template <int DV, bool TWO>
__device__ __forceinline__ void p_pass(uint32_t scol, uint32_t ocol, uint64_t c2, uint64_t nm2, uint64_t a2,
                                       uint64_t (&o2)[DV / 2], uint64_t &acc) {
#pragma unroll
    for (int kq = 0; kq < 4; ++kq) {
        uint32_t u[32];
        ptx::tmem_ld32(scol + 32 * kq, u);
        ptx::tmem_wait_ld();
        ptx::reg_fence32(u);
        uint32_t w[8], wl[8];
        uint32_t e4_prev = 0u;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float y0, y1, y2, y3;
            ptx::f2unpack(ptx::ffma2(ptx::f2pack(__uint_as_float(u[4 * k]), __uint_as_float(u[4 * k + 1])), c2, nm2),
                          y0, y1);
            ptx::f2unpack(ptx::ffma2(ptx::f2pack(__uint_as_float(u[4 * k + 2]), __uint_as_float(u[4 * k + 3])), c2, nm2),
                          y2, y3);
            const uint32_t e01 = ptx::ex2_h2(ptx::cvt_f16x2(y1, y0));
            const uint32_t e23 = ptx::ex2_h2(ptx::cvt_f16x2(y3, y2));
            const uint32_t e4 = ptx::hadd2(e01, e23);
            if (k & 1) {
                float s0, s1;
                ptx::h2_to_f32(ptx::hadd2(e4_prev, e4), s0, s1);
                acc = ptx::fadd2(acc, ptx::f2pack(s0, s1));
            } else {
                e4_prev = e4;
            }
            const uint32_t q01 = ptx::hmul2(e01, 0x5C005C00u), q23 = ptx::hmul2(e23, 0x5C005C00u);  // x 2^8, exact
            w[k] = ptx::prmt_lo16(ptx::cvt_e4m3x2_h2(q01), ptx::cvt_e4m3x2_h2(q23));
            if (TWO) {
                const uint32_t d01 = ptx::hsub2(q01, ptx::e4m3x2_to_h2(w[k] & 0xFFFFu));
                const uint32_t d23 = ptx::hsub2(q23, ptx::e4m3x2_to_h2(w[k] >> 16));
                wl[k] = ptx::prmt_lo16(ptx::cvt_e4m3x2_h2(d01), ptx::cvt_e4m3x2_h2(d23));
            } else {
                wl[k] = 0u;  // another warp of this tile may vote for two terms: this warp's is zero
            }
        }
        ptx::tmem_st8(scol + 32 * kq, w);
        ptx::tmem_st8(scol + 32 * kq + 8, wl);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int c0 = 32 * kq + 16 * hh;
            if (c0 < DV) {
                uint32_t v[16];
                ptx::tmem_ld16(ocol + c0, v);
                ptx::tmem_wait_ld();
                ptx::reg_fence16(v);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    o2[c0 / 2 + i] =
                        ptx::ffma2(o2[c0 / 2 + i], a2, ptx::f2pack(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])));
            }
        }
    }
}

// O = O alpha + O_t for the whole row (the last KV tile's fold).
template <int DV>
__device__ __forceinline__ void fold_all(uint32_t ocol, uint64_t a2, uint64_t (&o2)[DV / 2]) {
#pragma unroll
    for (int jc = 0; jc < DV / 32; ++jc) {
        uint32_t u[32];
        ptx::tmem_ld32(ocol + 32 * jc, u);
        ptx::tmem_wait_ld();
        ptx::reg_fence32(u);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            o2[16 * jc + i] = ptx::ffma2(o2[16 * jc + i], a2, ptx::f2pack(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1])));
    }
}

template <int D, int DV>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
    using C = PfCfg<D, DV>;
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
        return;  // slot beyond the last request's position blocks
    }
    const int kvh = blockIdx.y % p.Hkv;
    const int split = blockIdx.y / p.Hkv;
    const int PP = p.pos_per_tile;  // positions per CTA (both tiles)
    const int Pt = PP >> 1;         // positions per tile
    const int q_start = p.q_varlen ? p.cu_q[b] : b * p.Sq;
    const int Lq = p.q_varlen ? p.cu_q[b + 1] - q_start : p.Sq;
    int Lk, k_start = 0;
    if (p.kv_mode == 0) {
        Lk = p.Sk;
    } else {
        k_start = p.cu_k[b];
        Lk = p.cu_k[b + 1] - k_start;
    }
    bool bad = Lq < 0 || Lk < 0 || q_start < 0 || q_start + Lq > p.total_q;
    if (p.kv_mode == 1) bad |= (k_start < 0 || k_start + Lk > p.total_k);
    if (p.kv_mode == 2) bad |= ((long long)Lk > (long long)p.max_pages * p.page_size);
    if (bad) {
        if (tid == 0) atomicOr(p.status, kStatusBounds);
        return;
    }
    const int pos0 = mb * PP;
    if (pos0 >= Lq) return;
    const int pos_last = min(pos0 + PP, Lq) - 1;
    const int delta = Lk - Lq;
    const SplitRange sr = split_range(Lq, Lk, pos0, pos_last, p.causal, p.window_left, p.num_splits, cap, split);
    if (split >= sr.eff) return;  // this CTA's rows run fewer splits; the combine skips this one
    const int t_beg = sr.t_beg, t_end = sr.t_beg + sr.n_tiles;
    // each tile's positions and its KV tiles within this split
    // (selects, not arrays: a role picks its tile's values by a run-time index)
    const int tp0_a = pos0, tp0_b = pos0 + Pt;
    const int tpl_a = min(tp0_a + Pt, Lq) - 1, tpl_b = min(tp0_b + Pt, Lq) - 1;
    const TileSpan span_a = tile_span(tp0_a, tpl_a, Lk, delta, p.causal, p.window_left, t_beg, t_end);
    const TileSpan span_b = tile_span(tp0_b, tpl_b, Lk, delta, p.causal, p.window_left, t_beg, t_end);
    auto tp0_of = [&](int x) { return x ? tp0_b : tp0_a; };
    auto tpl_of = [&](int x) { return x ? tpl_b : tpl_a; };
    auto span_of = [&](int x) { return x ? span_b : span_a; };
    const bool has_sink = p.sink != nullptr && (!p.split_mode || split == 0);

    // per-row facts (tile warpgroups): row r of tile x
    const int side = (warp >> 2) & 1;
    const int r = tid & 127;
    const int rpos = tp0_of(side) + r / p.G;
    const int hq = kvh * p.G + r % p.G;
    const bool row_ok = warp < 8 && r < p.rows_per_tile && rpos < Lq;
    const int tok = q_start + rpos;
    const long long beta = p.q_varlen ? 0 : b;
    const long long rho = p.q_varlen ? tok : rpos;

    // writes a row whose keys in this split are all masked: O = 0, LSE = -inf (or the sink)
    auto write_empty_row = [&]() {
        const float lse = has_sink ? p.sink[hq] : -INFINITY;
        if (p.split_mode) {
            const long long row = ((long long)split * p.total_q + tok) * p.Hq + hq;
            p.lse_part[row] = lse;
            float4 *dst = reinterpret_cast<float4 *>(p.o_part + row * DV);
            for (int i = 0; i < DV / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            if (p.lse) p.lse[beta * p.lse_sb + hq * p.lse_sh + rho * p.lse_ss] = lse;
            uint8_t *dst = reinterpret_cast<uint8_t *>(p.o) + 2 * (beta * p.o_sb + rho * p.o_ss + hq * p.o_sh);
            for (int i = 0; i < DV / 8; ++i) *reinterpret_cast<uint4 *>(dst + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
        }
    };
    if (t_end <= t_beg) {
        if (row_ok) write_empty_row();
        return;
    }

    // ------------------------------------------------------------ shared memory
    uint8_t *misc = smem + C::OFF_MISC;
    const uint32_t bar0 = ptx::smem_u32(misc);
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc + C::OFF_TMEM_SLOT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + C::OFF_ABORT);
    volatile int *votes = reinterpret_cast<volatile int *>(misc + C::OFF_VOTES);
    const uint32_t sQ = ptx::smem_u32(smem + C::OFF_Q);
    const uint32_t sK = ptx::smem_u32(smem + C::OFF_K);
    const uint32_t sV = ptx::smem_u32(smem + C::OFF_V);

#ifdef FA8_TRACE
    for (int i = tid; i < kTraceEvents * kTraceTiles; i += kPfThreads)
        reinterpret_cast<unsigned long long *>(smem + C::OFF_TRACE)[i] = 0ull;
#endif
    if (tid == 0) {
        for (int x = 0; x < 2; ++x) {
            ptx::mbar_init(BAR(C::B_Q + x), 1);
            ptx::mbar_init(BAR(C::B_SF + x), 1);
            ptx::mbar_init(BAR(C::B_PF + x), 128);
            ptx::mbar_init(BAR(C::B_OF + x), 1);
            ptx::mbar_init(BAR(C::B_OE + x), 128);
        }
        for (int i = 0; i < C::STAGES; ++i) {
            ptx::mbar_init(BAR(C::B_KF + i), 1);
            ptx::mbar_init(BAR(C::B_KE + i), 1);
            ptx::mbar_init(BAR(C::B_VF + i), 1);
            ptx::mbar_init(BAR(C::B_VE + i), 1);
        }
        ptx::mbar_init(BAR(C::B_DONE), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == 8 && lane == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
    }
    if (warp == 9) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::TM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Waiter W{abort_flag, p.timeout_ns, p.status};

    if (warp >= 8) {
      ptx::setmaxnreg_dec<kPfRegsCtl>();
      if (warp == 8) {
        // ======================================================== TMA producer
        const bool paged = p.kv_mode == 2;
        int issued_k = 0, issued_v = 0;
        if (lane == 0) {
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                if (span_of(x).te <= span_of(x).tb) continue;  // this tile has no keys in this split
                ptx::mbar_arrive_expect_tx(BAR(C::B_Q + x), (uint32_t)(D * p.rows_per_tile));
                const int c2 = p.q_varlen ? q_start + tp0_of(x) : tp0_of(x);
                const int c3 = p.q_varlen ? 0 : b;
#pragma unroll
                for (int c = 0; c < C::NCK; ++c)
                    ptx::tma_load_4d(sQ + x * C::Q_BYTES + c * C::CHUNK_Q, &tm_q, BAR(C::B_Q + x), c * C::CW,
                                     kvh * p.G, c2, c3);
            }
        }
        for (int j = t_beg; j < t_end; ++j) {
            const int it = j - t_beg;
            const int k0 = j * kTileN;
            const int st = it % C::STAGES;
            const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
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
            if (!W.wait_warp(BAR(C::B_KE + st), ph ^ 1u)) break;
            if (lane == 0) ptx::mbar_arrive_expect_tx(BAR(C::B_KF + st), (uint32_t)C::K_BYTES);
            __syncwarp();
            const uint32_t dK = sK + st * C::K_BYTES;
            if (paged) {
                if (lane < p.boxes_per_tile) {
#pragma unroll
                    for (int c = 0; c < C::NCK; ++c)
                        ptx::tma_load_4d(dK + c * C::CHUNK_K + lane * p.box_n * C::CW, &tm_k, BAR(C::B_KF + st),
                                         c * C::CW, kvh, prow, page);
                }
            } else if (lane == 0) {
#pragma unroll
                for (int c = 0; c < C::NCK; ++c)
                    ptx::tma_load_4d(dK + c * C::CHUNK_K, &tm_k, BAR(C::B_KF + st), c * C::CW, kvh, c2, c3);
            }
            issued_k = it + 1;
            if (!W.wait_warp(BAR(C::B_VE + st), ph ^ 1u)) break;
            if (lane == 0) ptx::mbar_arrive_expect_tx(BAR(C::B_VF + st), (uint32_t)C::V_BYTES);
            __syncwarp();
            const uint32_t dV = sV + st * C::V_BYTES;
            if (paged) {
                if (lane < p.boxes_per_tile) {
#pragma unroll
                    for (int c = 0; c < C::NCV; ++c)
                        ptx::tma_load_4d(dV + c * C::CHUNK_V + lane * p.box_n * C::CWV, &tm_v, BAR(C::B_VF + st),
                                         c * C::CWV, kvh, prow, page);
                }
            } else if (lane == 0) {
#pragma unroll
                for (int c = 0; c < C::NCV; ++c)
                    ptx::tma_load_4d(dV + c * C::CHUNK_V, &tm_v, BAR(C::B_VF + st), c * C::CWV, kvh, c2, c3);
            }
            issued_v = it + 1;
        }
        if (*abort_flag) {
            // every load already issued must land before the CTA's smem is released
#pragma unroll
            for (int x = 0; x < 2; ++x)
                if (span_of(x).te > span_of(x).tb) W.drain(BAR(C::B_Q + x), 0);
            for (int i = max(0, issued_k - C::STAGES); i < issued_k; ++i)
                W.drain(BAR(C::B_KF + i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u);
            for (int i = max(0, issued_v - C::STAGES); i < issued_v; ++i)
                W.drain(BAR(C::B_VF + i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u);
        }
        __syncwarp();
      } else if (warp == 9) {
        // ======================================================== MMA issuer (one elected lane)
        // Per KV tile j: PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1).  The tensor core takes one
        // issuer's MMAs in order and its queue is short (an issue waits for room), so this
        // order keeps tile B one MMA phase behind tile A: B's softmax runs while A's PV and QK
        // run, and the other way round.
        constexpr uint32_t kIdescQK = idesc_e4m3(kTileM, kTileN, false);
        constexpr uint32_t kIdescPV = idesc_e4m3(kTileM, DV, true);
        const uint64_t dk0 = sdesc(sK, 16, 8 * C::CW, swz_layout(C::CW));
        const uint64_t dv0 = sdesc(sV, C::CHUNK_V, 8 * C::CWV, swz_layout(C::CWV));
        const bool leader = ptx::elect_one();
        bool ok = true;
#pragma unroll
        for (int x = 0; x < 2; ++x)
            if (ok && span_of(x).te > span_of(x).tb) ok = W.wait_warp(BAR(C::B_Q + x), 0);
        ptx::tc_fence_after();
        auto in_tile = [&](int x, int j) { return j >= span_of(x).tb && j < span_of(x).te; };
        // S_x = Q_x K_j^T
        auto qk = [&](int x, int j) {
            const int ks = (j - t_beg) % C::STAGES;
            const uint64_t dq = sdesc(sQ + x * C::Q_BYTES, 16, 8 * C::CW, swz_layout(C::CW));
            const uint64_t dk = dk0 + (uint64_t)((ks * C::K_BYTES) >> 4);
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk) {
                    const uint32_t off = (uint32_t)((((kk * 32) / C::CW) * C::CHUNK_Q + (kk * 32) % C::CW) >> 4);
                    ptx::mma_f8_ss(tmem + C::TM_S + x * 128, dq + off, dk + off, kIdescQK, kk > 0 ? 1u : 0u);
                }
                ptx::tc_commit(BAR(C::B_SF + x));
            }
            __syncwarp();
        };
        // O_t,x = P_x V_j (+ P_lo V_j): waits for P and for the fold of the previous O_t
        auto pv = [&](int x, int j) -> bool {
            const int n = j - span_of(x).tb;
            if (!W.wait_warp(BAR(C::B_PF + x), (uint32_t)n & 1u)) return false;
            if (!W.wait_warp(BAR(C::B_OE + x), ((uint32_t)n & 1u) ^ 1u)) return false;
            ptx::tc_fence_after();
            const bool two_term =
                tile_needs_mask(j * kTileN, Lk, p.causal, p.window_left, tp0_of(x), tpl_of(x), delta) ||
                (votes[x * 4 + 0] | votes[x * 4 + 1] | votes[x * 4 + 2] | votes[x * 4 + 3]) != 0;
            const int vs = (j - t_beg) % C::STAGES;
            const uint64_t dv = dv0 + (uint64_t)((vs * C::V_BYTES) >> 4);
            const uint32_t s_col = tmem + C::TM_S + x * 128;
            const uint32_t otile = tmem + C::TM_OT + x * 128;
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < kTileN / 32; ++kk)
                    ptx::mma_f8_ts(otile, s_col + kk * 32, dv + (uint64_t)((kk * 32 * C::CWV) >> 4), kIdescPV,
                                   kk > 0 ? 1u : 0u);
                if (two_term) {  // + P_lo V (P_lo 8 columns after each P_hi slice)
#pragma unroll
                    for (int kk = 0; kk < kTileN / 32; ++kk)
                        ptx::mma_f8_ts(otile, s_col + kk * 32 + 8, dv + (uint64_t)((kk * 32 * C::CWV) >> 4),
                                       kIdescPV, 1u);
                }
                ptx::tc_commit(BAR(C::B_OF + x));
            }
            __syncwarp();
            return true;
        };
        // prologue: S of the first KV tile for each Q tile that starts there
        if (ok) ok = W.wait_warp(BAR(C::B_KF + 0), 0u);
        if (ok) {
            ptx::tc_fence_after();
#pragma unroll
            for (int x = 0; x < 2; ++x)
                if (in_tile(x, t_beg)) qk(x, t_beg);
            if (leader) ptx::tc_commit(BAR(C::B_KE + 0));
            __syncwarp();
        }
        for (int j = t_beg; ok && j < t_end; ++j) {
            const int it = j - t_beg;
            const bool more = j + 1 < t_end;
            if (lane == 0) FA8_EV(8, it);
            if (!W.wait_warp(BAR(C::B_VF + it % C::STAGES), (uint32_t)(it / C::STAGES) & 1u)) { ok = false; break; }
            if (more && !W.wait_warp(BAR(C::B_KF + (it + 1) % C::STAGES), (uint32_t)((it + 1) / C::STAGES) & 1u)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                if (in_tile(x, j) && !pv(x, j)) { ok = false; break; }
                if (lane == 0) FA8_EV(12 + x, it);
                if (more && in_tile(x, j + 1)) qk(x, j + 1);
            }
            if (!ok) break;
            if (lane == 0) FA8_EV(14, it);
            if (leader) {
                ptx::tc_commit(BAR(C::B_VE + it % C::STAGES));
                if (more) ptx::tc_commit(BAR(C::B_KE + (it + 1) % C::STAGES));
            }
            __syncwarp();
        }
        // all MMAs must finish before TMEM is released
        if (leader) ptx::tc_commit(BAR(C::B_DONE));
        __syncwarp();
        W.drain(BAR(C::B_DONE), 0);
        __syncwarp();
      }
    } else {
      ptx::setmaxnreg_inc<kPfRegsTile>();
      {
        // bounded waits that keep no pointer live in registers (the fields come from the
        // parameters and the shared abort flag's address on the slow path)
        const uint32_t abort_saddr = ptx::smem_u32(misc + C::OFF_ABORT);
        auto wait_tile = [&](uint32_t bar, uint32_t parity) -> bool {
            bool okw = ptx::mbar_try_wait(bar, parity);
            if (!okw) okw = wait_slow_s(bar, parity, abort_saddr, p.timeout_ns, p.status);
            return __all_sync(0xffffffffu, okw);
        };
        // ======================================================== tile warpgroup (softmax + fold)
        const int x = side;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t scol = tmem + lane_base + C::TM_S + x * 128;
        const uint32_t ocol = tmem + lane_base + C::TM_OT + x * 128;
        const int tb = span_of(x).tb, nt = span_of(x).te - span_of(x).tb;
        const int xp0 = tp0_of(x), xpl = tpl_of(x);
        const float dqv = p.dq ? p.dq[b * p.dq_sb + kvh * p.dq_sh] : 1.f;
        const float dkv = p.dk ? p.dk[b * p.dk_sb + kvh * p.dk_sh] : 1.f;
        const float c = p.scale_log2 * dqv * dkv;
        const uint64_t c2 = ptx::f2pack(c, c);
        const int hi_row = p.causal ? min(Lk - 1, rpos + delta) : Lk - 1;
        const int lo_row = p.window_left >= 0 ? max(0, rpos + delta - p.window_left) : 0;
        uint64_t o2[DV / 2];  // the row's running O, as packed fp32 pairs (columns 2i, 2i+1)
#pragma unroll
        for (int i = 0; i < DV / 2; ++i) o2[i] = ptx::f2pack(0.f, 0.f);
        float m_run = -INFINITY, row_sum = 0.f;
        float alpha_prev = 0.f;  // rescale of the KV tile whose O_t the next fold adds
        {
            // O_t starts at zero, so the first KV tile's P pass folds zeros
            uint32_t z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0u;
#pragma unroll
            for (int jc = 0; jc < DV / 32; ++jc) ptx::tmem_st32(ocol + 32 * jc, z);
            ptx::tmem_wait_st();
        }
        bool ok = true;
        for (int n = 0; ok && n < nt; ++n) {
            const int k0 = (tb + n) * kTileN;
            if (!wait_tile(BAR(C::B_SF + x), (uint32_t)n & 1u)) { ok = false; break; }
            const bool tr = tid == 0;
            if (tr) FA8_EV(0, n);
            if (tid == 128) FA8_EV(15, n);
            ptx::tc_fence_after();
            const bool need_mask =
                tile_needs_mask(k0, Lk, p.causal, p.window_left, xp0, xpl, delta);
            const int hi = hi_row - k0, lo = lo_row - k0;  // visible columns: [lo, hi]
            // ---- pass 1: the row's maximum over the tile, 32 columns at a time; on tiles that
            // need a mask, the masked columns are written back as -inf for the P pass
            float mx = -INFINITY;
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                uint32_t u[32];
                ptx::tmem_ld32(scol + 32 * q, u);
                ptx::tmem_wait_ld();
                ptx::reg_fence32(u);
                if (need_mask) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int col = 32 * q + i;
                        if (col > hi || col < lo) u[i] = __float_as_uint(-INFINITY);
                    }
                    ptx::tmem_st32(scol + 32 * q, u);
                }
                float ma = ptx::fmax3(u2f(u[0]), u2f(u[1]), u2f(u[2]));
                float mb2 = ptx::fmax3(u2f(u[16]), u2f(u[17]), u2f(u[18]));
#pragma unroll
                for (int i = 3; i < 15; i += 2) {
                    ma = ptx::fmax3(ma, u2f(u[i]), u2f(u[i + 1]));
                    mb2 = ptx::fmax3(mb2, u2f(u[16 + i]), u2f(u[16 + i + 1]));
                }
                mx = ptx::fmax3(mx, ptx::fmax3(ma, mb2, u2f(u[15])), u2f(u[31]));
            }
            if (need_mask) ptx::tmem_wait_st();
            if (tr) FA8_EV(1, n);
            // ---- lazy rescale and the two-term vote
            const float mt = mx * c;
            float alpha = 1.f;
            if (mt > m_run + kTau) {
                alpha = ptx::ex2(m_run - mt);
                row_sum *= alpha;
                m_run = mt;
            }
            bool two_term = need_mask;
            if (!need_mask) {
                // the tile's largest p is 2^(mt - m + 8); it holds more than about 1/8 of the row's
                // mass so far when log2 of it exceeds log2(row_sum) - log2(7).  log2(row_sum) is
                // taken as its fp32 exponent (the floor), without a MUFU instruction, which errs
                // towards two terms (an effective share between 1/15 and 1/8)
                const int e_rs = row_sum > 0.f ? (int)((__float_as_uint(row_sum) >> 23) & 0xFF) - 127 : -1000;
                two_term = __any_sync(0xffffffffu, row_ok && (mt - m_run + kPBias) > (float)e_rs - 2.807f);
            }
            if (lane == 0) votes[x * 4 + (warp & 3)] = two_term ? 1 : 0;
            // ---- pass 2 (P, see p_pass), with the fold of the previous KV tile's O_t: O_t(n - 1)
            // stays in TMEM until this pass, so the fold is off the chain P -> PV -> QK -> S
            if (n > 0) {
                if (!wait_tile(BAR(C::B_OF + x), (uint32_t)(n - 1) & 1u)) { ok = false; break; }
                ptx::tc_fence_after();
            }
            const float nm = m_run == -INFINITY ? 0.f : -m_run;
            const uint64_t nm2 = ptx::f2pack(nm, nm);
            const uint64_t a2 = ptx::f2pack(alpha_prev, alpha_prev);
            uint64_t acc = ptx::f2pack(0.f, 0.f);
            if (tr) FA8_EV(9, n);
            if (two_term) p_pass<DV, true>(scol, ocol, c2, nm2, a2, o2, acc);
            else p_pass<DV, false>(scol, ocol, c2, nm2, a2, o2, acc);
            if (tr) FA8_EV(10, n);
            if (tr) FA8_VAL(11, n, (two_term ? 1ull : 0ull) | (need_mask ? 2ull : 0ull));
            alpha_prev = alpha;
            ptx::tmem_wait_st();
            {
                float a0, a1;
                ptx::f2unpack(acc, a0, a1);
                row_sum += (a0 + a1) * 256.f;  // the f16 p carry no 2^8: scale to the biased row sum
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(BAR(C::B_PF + x));
            if (tr) FA8_EV(2, n);
            if (tid == 32 || tid == 64 || tid == 96) FA8_EV(4 + (tid >> 5), n);
            if (n > 0) ptx::mbar_arrive(BAR(C::B_OE + x));  // O_t(n - 1) folded: PV(n) may overwrite it
        }
        // the last KV tile's O_t
        if (ok && nt > 0) {
            if (wait_tile(BAR(C::B_OF + x), (uint32_t)(nt - 1) & 1u)) {
                ptx::tc_fence_after();
                fold_all<DV>(ocol, ptx::f2pack(alpha_prev, alpha_prev), o2);
            } else {
                ok = false;
            }
        }
        // ---- finalize: the 2^8 bias cancels between O and row_sum and is removed from the LSE
        if (row_ok) {
            if (nt == 0 || !ok) {
                if (nt == 0) write_empty_row();
            } else {
                const float dvv = p.dv ? p.dv[b * p.dv_sb + kvh * p.dv_sh] : 1.f;
                const float sig = has_sink ? p.sink[hq] : 0.f;
                float scale_o = 0.f, lse;
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
                if (p.split_mode) {
                    const long long row = ((long long)split * p.total_q + tok) * p.Hq + hq;
                    p.lse_part[row] = lse;
                    float *dst = p.o_part + row * DV;
#pragma unroll
                    for (int i = 0; i < DV; i += 4) {
                        float v0, v1, v2, v3;
                        ptx::f2unpack(o2[i / 2], v0, v1);
                        ptx::f2unpack(o2[i / 2 + 1], v2, v3);
                        *reinterpret_cast<float4 *>(dst + i) =
                            make_float4(v0 * scale_o, v1 * scale_o, v2 * scale_o, v3 * scale_o);
                    }
                } else {
                    if (p.lse) p.lse[beta * p.lse_sb + hq * p.lse_sh + rho * p.lse_ss] = lse;
                    uint8_t *dst = reinterpret_cast<uint8_t *>(p.o) + 2 * (beta * p.o_sb + rho * p.o_ss + hq * p.o_sh);
#pragma unroll
                    for (int i = 0; i < DV; i += 8) {
                        float t8[8];
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            ptx::f2unpack(o2[(i + e) / 2], t8[e], t8[e + 1]);
                            t8[e] *= scale_o;
                            t8[e + 1] *= scale_o;
                        }
                        store8(dst + 2 * i, t8, p.out_fp16);
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
    if (p.trace && blockIdx.y == 0 && blockIdx.x < kTraceCtas) {
        const unsigned long long *src = reinterpret_cast<const unsigned long long *>(smem + C::OFF_TRACE);
        for (int i = tid; i < kTraceEvents * kTraceTiles; i += kPfThreads)
            p.trace[(size_t)blockIdx.x * kTraceEvents * kTraceTiles + i] = src[i];
    }
#endif
    if (warp == 9) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::TM_COLS);
    }
}

}  // namespace fa8
