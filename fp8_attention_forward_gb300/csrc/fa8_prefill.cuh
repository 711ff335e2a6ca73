// fa8_prefill.cuh -- the forward for many query rows per kv-head (prefill, chunked prefill)
// with dv <= 128: a persistent kernel, one CTA per SM, each CTA walking a list of work units
// (a 128-row Q tile of one kv-head group, one split of its keys) and streaming the units' KV
// tiles through one pipeline, so that a unit's last tiles overlap the next unit's first ones.
//
// Same arithmetic as fwd_kernel ("[Cute,Fwd,Sm90] Native FP8 (E4M3 Q/K/V) forward for
// Hopper", Design; "tml-fa4 PR #4", Summary and "Correctness fix over #1"): S = Q K^T in
// TMEM (tcgen05.mma kind::f8f6f4), lazy running max (tau = 0.75 in log2 units), P =
// e4m3(2^(s c - m + 8)) with the 2^8 bias folded into the packed FMA that applies the scale,
// written over S in TMEM; O_t = P V accumulated from zero for every KV tile and folded into an
// fp32 O as O = O * alpha + O_t (two-level accumulation); O * dv / rowsum and LSE = ln2 *
// (log2 rowsum + m - 8) at the end.  A tile's P takes a second E4M3 term (P_lo = e4m3(p -
// P_hi)) when the tile needs a mask or one key of some row holds about an eighth or more of
// that row's mass so far.
//
// The unit list and the order of the work ("PyTorch ... FlashAttention-4 MXFP8", 2.1.2
// Improved unroll-KV): every CTA takes units k * grid + c (even k) or k * grid + grid - 1 - c
// (odd k) of a list ordered by decreasing key count, so the CTAs' loads even out; within a
// CTA, the tile stream i = 0, 1, ... runs across unit boundaries: QK(i + 2) follows PV(i), so
// the next unit's first QKs run under this unit's last softmax.
//
// Roles (384 threads, three warpgroups):
//   warps 0-3   softmax: thread r owns TMEM lane r = row r of the tile; per tile it loads the
//               row's 128 scores into registers once, takes the maximum, writes P over S
//   warps 4-7   correction: holds the row's running O (dv fp32 registers), folds each tile's
//               O_t into it, and writes the unit's output row
//   warp 8      TMA producer (Q of each unit into a double buffer, K/V tiles into a ring)
//   warp 9      PV issuer (one elected lane) and TMEM owner
//   warp 10     QK issuer (one elected lane)
//   warp 11     idle (its registers go to the other warpgroups)
// TMEM (512 columns): S/P of tiles i even / odd at 0 / 128, O_t of tiles i even / odd at 256 /
// 384.  Hand-offs: S(i) full -> softmax; alpha(i) (4-deep ring) -> correction; P(i) -> MMA;
// O_t(i) full -> correction; O_t(i) folded -> MMA (PV(i + 2)); per unit, the row's output
// scale and LSE (4-deep ring) softmax -> correction.
// A build with -DFA8_TRACE records clock64() per tile i (< 64) of the first CTAs (debug only):
// softmax 0 S ready, 1 row max done, 2 P written; producer 3 / 4 K / V load issued; PV issuer
// 8 waits passed, 9 PV issued; QK issuer 11 PV(i - 2) complete, 10 QK(i) issued; correction 12
// alpha read, 13 O_t complete, 14 fold done.  The ring depths follow from the chain
// PV(i) <- fold(i - 2): the softmax can run at most four tiles ahead of the correction.
#pragma once

#include "fa8_kernel.cuh"

namespace fa8 {

constexpr int kPfThreads = 384;

// registers per thread: launch 168 (384 x 168 <= 64K); setmaxnreg gives the softmax
// warpgroup 184 (the row's 128 scores), the correction warpgroup 216 (the row's O in 128 of
// them) and the control warpgroup 104
constexpr int kPfLaunchRegs = 168;
constexpr int kPfRegsSoft = 184;
constexpr int kPfRegsCorr = 216;
constexpr int kPfRegsCtl = 104;
static_assert(kPfRegsSoft + kPfRegsCorr + kPfRegsCtl == 3 * kPfLaunchRegs, "register split");

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
    static constexpr int Q_BYTES = kTileM * D;  // one Q tile (two buffers)
    static constexpr int K_BYTES = kTileN * D;
    static constexpr int V_BYTES = kTileN * DV;
    static constexpr int MISC_BYTES = 8192;
    static constexpr int SMEM_LIMIT = 232448;  // max dynamic smem per block on sm_103
    static constexpr int STAGES_FIT =
        (SMEM_LIMIT - 1024 - MISC_BYTES - kTraceSmemBytes - 2 * Q_BYTES) / (K_BYTES + V_BYTES);
    static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = 2 * Q_BYTES;
    static constexpr int OFF_V = OFF_K + STAGES * K_BYTES;
    static constexpr int OFF_MISC = OFF_V + STAGES * V_BYTES;
    static constexpr int OFF_TRACE = OFF_MISC + MISC_BYTES;
    static constexpr int SMEM_BYTES = OFF_TRACE + kTraceSmemBytes + 1024;
    static constexpr uint32_t TM_S = 0;     // S/P of tile i at TM_S + 128 (i % 2)
    static constexpr uint32_t TM_OT = 256;  // O_t of tile i at TM_OT + 128 (i % 2)
    static constexpr uint32_t TM_COLS = 512;
    // barriers
    static constexpr int B_QF = 0;              // Q buffer full (2)
    static constexpr int B_QE = 2;              // Q buffer free (2)
    static constexpr int B_KF = 4;              // K/V ring
    static constexpr int B_KE = B_KF + STAGES;
    static constexpr int B_VF = B_KE + STAGES;
    static constexpr int B_VE = B_VF + STAGES;
    static constexpr int B_SF = B_VE + STAGES;  // S(i) written (2)
    static constexpr int B_PF = B_SF + 2;       // P(i) written (2)
    static constexpr int B_OF = B_PF + 2;       // O_t(i) written (2)
    static constexpr int B_OE = B_OF + 2;       // O_t(i) folded (2)
    static constexpr int B_AL = B_OE + 2;       // alpha(i) written (4)
    static constexpr int B_FN = B_AL + 4;       // a unit's output scale and LSE written (4)
    static constexpr int B_DONE = B_FN + 4;     // all MMAs of one issuer complete (2)
    static constexpr int NUM_BARS = B_DONE + 2;
    static constexpr int OFF_ALPHA = 512;               // [4][128] fp32
    static constexpr int OFF_FIN = OFF_ALPHA + 2048;    // [4][2][128] fp32 (scale, LSE)
    static constexpr int OFF_VOTES = OFF_FIN + 4096;    // [2][4] int (16-byte aligned rows)
    static constexpr int OFF_TMEM_SLOT = OFF_VOTES + 32;
    static constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;
    static_assert(STAGES >= 2, "smem too small for two K/V stages");
    static_assert(NUM_BARS * 8 <= 512, "barrier area");
    static_assert(OFF_ABORT + 4 <= MISC_BYTES, "misc area");
    static_assert(Q_BYTES % 1024 == 0 && K_BYTES % 1024 == 0 && V_BYTES % 1024 == 0, "swizzle alignment");
};

// One work unit: a 128-row Q tile (pos_per_tile positions x G q-heads of kv-head kvh) of
// request b, and one split of its keys.  state 0: nothing to do (no such tile, no rows, or a
// split the tile does not run); 1: the tile's rows see no key in this split (their output is
// written directly); 2: KV tiles [t_beg, t_end) to run.  Whole warp must call it (varlen).
struct PfUnit {
    int state, b, kvh, split, q_start, Lq, Lk, k_start, pos0, pos_last, delta, t_beg, t_end;
};
__device__ __forceinline__ PfUnit pf_unit(const FwdParams &p, int u, int cap) {
    PfUnit r;
    r.state = 0;
    const int per_x = p.Hkv * p.num_splits;
    const int x = u / per_x, y = u - x * per_x;
    int b, mb;
    if (!p.q_varlen) {
        b = x % p.B;
        mb = p.mblocks_per_batch - 1 - x / p.B;
    } else if (!varlen_slot(p, x, b, mb)) {
        return r;
    }
    r.b = b;
    r.kvh = y % p.Hkv;
    r.split = y / p.Hkv;
    r.q_start = p.q_varlen ? p.cu_q[b] : b * p.Sq;
    r.Lq = p.q_varlen ? p.cu_q[b + 1] - r.q_start : p.Sq;
    r.k_start = 0;
    if (p.kv_mode == 0) {
        r.Lk = p.Sk;
    } else {
        r.k_start = p.cu_k[b];
        r.Lk = p.cu_k[b + 1] - r.k_start;
    }
    // device-side sanity of caller-provided lengths: never index outside the tensors
    bool bad = r.Lq < 0 || r.Lk < 0 || r.q_start < 0 || r.q_start + r.Lq > p.total_q;
    if (p.kv_mode == 1) bad |= (r.k_start < 0 || r.k_start + r.Lk > p.total_k);
    if (p.kv_mode == 2) bad |= ((long long)r.Lk > (long long)p.max_pages * p.page_size);
    if (bad) {
        if ((threadIdx.x & 31) == 0) atomicOr(p.status, kStatusBounds);
        return r;
    }
    r.pos0 = mb * p.pos_per_tile;
    if (r.pos0 >= r.Lq) return r;
    r.pos_last = min(r.pos0 + p.pos_per_tile, r.Lq) - 1;
    r.delta = r.Lk - r.Lq;
    const SplitRange sr =
        split_range(r.Lq, r.Lk, r.pos0, r.pos_last, p.causal, p.window_left, p.num_splits, cap, r.split);
    if (r.split >= sr.eff) return r;  // the combine kernel skips this split of these rows
    r.t_beg = sr.t_beg;
    r.t_end = sr.t_beg + sr.n_tiles;
    r.state = r.t_end > r.t_beg ? 2 : 1;
    return r;
}

// The unit list: the k-th unit a CTA takes (snake order over the list), or -1 past its end.
__device__ __forceinline__ int pf_unit_index(const FwdParams &p, int k) {
    const int g = (int)gridDim.x, c = (int)blockIdx.x;
    const long long u = (long long)k * g + ((k & 1) ? g - 1 - c : c);
    return u < p.units ? (int)u : -1;
}

// The row maximum over the 128 scores held in registers.
__device__ __forceinline__ float row_max(const uint32_t (&u)[128]) {
    float m0 = ptx::fmax3(u2f(u[0]), u2f(u[1]), u2f(u[2]));
    float m1 = ptx::fmax3(u2f(u[3]), u2f(u[4]), u2f(u[5]));
    float m2 = ptx::fmax3(u2f(u[6]), u2f(u[7]), u2f(u[8]));
    float m3 = ptx::fmax3(u2f(u[9]), u2f(u[10]), u2f(u[11]));
#pragma unroll
    for (int i = 12; i < 124; i += 8) {
        m0 = ptx::fmax3(m0, u2f(u[i]), u2f(u[i + 1]));
        m1 = ptx::fmax3(m1, u2f(u[i + 2]), u2f(u[i + 3]));
        m2 = ptx::fmax3(m2, u2f(u[i + 4]), u2f(u[i + 5]));
        m3 = ptx::fmax3(m3, u2f(u[i + 6]), u2f(u[i + 7]));
    }
    m0 = ptx::fmax3(m0, u2f(u[124]), u2f(u[125]));
    m1 = ptx::fmax3(m1, u2f(u[126]), u2f(u[127]));
    return ptx::fmax3(m0, m1, fmaxf(m2, m3));
}

// All 128 score columns of the thread's lane into registers (one wait).
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&u)[128]) {
    uint32_t(&u0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&u[0]);
    uint32_t(&u1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&u[32]);
    uint32_t(&u2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&u[64]);
    uint32_t(&u3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&u[96]);
    ptx::tmem_ld32(taddr, u0);
    ptx::tmem_ld32(taddr + 32, u1);
    ptx::tmem_ld32(taddr + 64, u2);
    ptx::tmem_ld32(taddr + 96, u3);
    ptx::tmem_wait_ld();
    ptx::reg_fence32(u0);
    ptx::reg_fence32(u1);
    ptx::reg_fence32(u2);
    ptx::reg_fence32(u3);
}

// O = O alpha + O_t for the whole row, 64 columns per TMEM round trip, then one packed FMA per
// column pair.
template <int DV>
__device__ __forceinline__ void fold_pass(uint32_t ocol, uint64_t a2, uint64_t (&o2)[DV / 2]) {
#pragma unroll
    for (int h = 0; h < DV / 64; ++h) {
        uint32_t t0[32], t1[32];
        ptx::tmem_ld32(ocol + 64 * h, t0);
        ptx::tmem_ld32(ocol + 64 * h + 32, t1);
        ptx::tmem_wait_ld();
        ptx::reg_fence32(t0);
        ptx::reg_fence32(t1);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            o2[32 * h + i] = ptx::ffma2(o2[32 * h + i], a2, ptx::f2pack(u2f(t0[2 * i]), u2f(t0[2 * i + 1])));
            o2[32 * h + 16 + i] = ptx::ffma2(o2[32 * h + 16 + i], a2, ptx::f2pack(u2f(t1[2 * i]), u2f(t1[2 * i + 1])));
        }
    }
    if (DV % 64) {  // a last 32 columns (dv = 96)
        uint32_t t0[32];
        ptx::tmem_ld32(ocol + DV - 32, t0);
        ptx::tmem_wait_ld();
        ptx::reg_fence32(t0);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            o2[(DV - 32) / 2 + i] = ptx::ffma2(o2[(DV - 32) / 2 + i], a2, ptx::f2pack(u2f(t0[2 * i]), u2f(t0[2 * i + 1])));
    }
}

// P for one 32-key chunk of the row: p = 2^(s c - m + 8) in fp32, the 2^8 bias folded into the
// same packed FMA that applies the scale and subtracts the running maximum; w = e4m3(p) (round
// to nearest even, saturating) and, when `two`, wl = e4m3(p - P_hi) (zeros otherwise: another
// warp of the tile may have voted for two terms); the unrounded p go into two packed fp32
// row-sum accumulators.  Masked keys hold -inf, so their p is exactly 0.  The p overwrite
// their scores in u, so the P_lo step reads them back without a second copy.
__device__ __forceinline__ void p_chunk(uint32_t (&u)[32], uint64_t c2, uint64_t b2, bool two, uint64_t &acc0,
                                        uint64_t &acc1, uint32_t (&w)[8], uint32_t (&wl)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int o = 4 * k;
        float y0, y1, y2, y3;
        ptx::f2unpack(ptx::ffma2(ptx::f2pack(u2f(u[o]), u2f(u[o + 1])), c2, b2), y0, y1);
        ptx::f2unpack(ptx::ffma2(ptx::f2pack(u2f(u[o + 2]), u2f(u[o + 3])), c2, b2), y2, y3);
        const float e0 = ptx::ex2(y0), e1 = ptx::ex2(y1), e2 = ptx::ex2(y2), e3 = ptx::ex2(y3);
        acc0 = ptx::fadd2(acc0, ptx::f2pack(e0, e1));
        acc1 = ptx::fadd2(acc1, ptx::f2pack(e2, e3));
        w[k] = ptx::prmt_lo16(ptx::cvt_e4m3x2(e1, e0), ptx::cvt_e4m3x2(e3, e2));
        u[o] = __float_as_uint(e0);
        u[o + 1] = __float_as_uint(e1);
        u[o + 2] = __float_as_uint(e2);
        u[o + 3] = __float_as_uint(e3);
    }
    if (two) {
        // the residual in f16 (p < 2^9 holds 11 significant bits there, P_hi is exact in f16)
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int o = 4 * k;
            const uint32_t d01 = ptx::hsub2(ptx::cvt_f16x2(u2f(u[o + 1]), u2f(u[o])), ptx::e4m3x2_to_h2(w[k] & 0xFFFFu));
            const uint32_t d23 = ptx::hsub2(ptx::cvt_f16x2(u2f(u[o + 3]), u2f(u[o + 2])), ptx::e4m3x2_to_h2(w[k] >> 16));
            wl[k] = ptx::prmt_lo16(ptx::cvt_e4m3x2_h2(d01), ptx::cvt_e4m3x2_h2(d23));
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) wl[k] = 0u;
    }
}

// The P pass over the row's 128 keys, re-read from TMEM 32 columns at a time with the next
// chunk's load in flight; a rolled loop of two chunks per iteration keeps the code that every
// tile runs small.  P of keys [32 kq, 32 kq + 32) goes to column 32 kq (P_lo to 32 kq + 8),
// written after the next chunk's scores have landed: columns this pass has already read.
__device__ __forceinline__ void p_pass(uint32_t scol, uint64_t c2, uint64_t b2, bool two, uint64_t &acc0,
                                       uint64_t &acc1) {
    uint32_t ua[32], ub[32], w[8], wl[8];
    ptx::tmem_ld32(scol, ua);
    ptx::tmem_wait_ld();
    ptx::reg_fence32(ua);
#pragma unroll 1
    for (int kq = 0; kq < 4; kq += 2) {
        const uint32_t col = scol + 32u * (uint32_t)kq;
        ptx::tmem_ld32(col + 32, ub);
        p_chunk(ua, c2, b2, two, acc0, acc1, w, wl);
        ptx::tmem_wait_ld();
        ptx::reg_fence32(ub);
        ptx::tmem_st8(col, w);
        ptx::tmem_st8(col + 8, wl);
        if (kq == 0) ptx::tmem_ld32(col + 64, ua);
        p_chunk(ub, c2, b2, two, acc0, acc1, w, wl);
        if (kq == 0) {
            ptx::tmem_wait_ld();
            ptx::reg_fence32(ua);
        }
        ptx::tmem_st8(col + 32, w);
        ptx::tmem_st8(col + 40, wl);
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

    int cap = p.cap_const > 0 ? p.cap_const : (1 << 20);
    if (p.num_splits > 1 && p.cap_const <= 0) {  // chosen by split_plan_kernel, which may still be running
        ptx::griddep_wait();
        cap = *p.split_cap;
    }

    // ------------------------------------------------------------ shared memory
    uint8_t *misc = smem + C::OFF_MISC;
    const uint32_t bar0 = ptx::smem_u32(misc);
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc + C::OFF_TMEM_SLOT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + C::OFF_ABORT);
    volatile int *votes = reinterpret_cast<volatile int *>(misc + C::OFF_VOTES);
    const uint32_t votes_saddr = ptx::smem_u32(misc + C::OFF_VOTES);
    float *alpha_ring = reinterpret_cast<float *>(misc + C::OFF_ALPHA);
    float *fin_ring = reinterpret_cast<float *>(misc + C::OFF_FIN);
    const uint32_t sQ = ptx::smem_u32(smem + C::OFF_Q);
    const uint32_t sK = ptx::smem_u32(smem + C::OFF_K);
    const uint32_t sV = ptx::smem_u32(smem + C::OFF_V);

#ifdef FA8_TRACE
    for (int i = tid; i < kTraceEvents * kTraceTiles; i += kPfThreads)
        reinterpret_cast<unsigned long long *>(smem + C::OFF_TRACE)[i] = 0ull;
#endif
    if (tid == 0) {
        for (int x = 0; x < 2; ++x) {
            ptx::mbar_init(BAR(C::B_QF + x), 1);
            ptx::mbar_init(BAR(C::B_QE + x), 1);
            ptx::mbar_init(BAR(C::B_SF + x), 1);
            ptx::mbar_init(BAR(C::B_PF + x), 4);  // one arrival per softmax warp
            ptx::mbar_init(BAR(C::B_OF + x), 1);
            ptx::mbar_init(BAR(C::B_OE + x), 4);  // one arrival per correction warp
        }
        for (int x = 0; x < 4; ++x) {
            ptx::mbar_init(BAR(C::B_AL + x), 4);
            ptx::mbar_init(BAR(C::B_FN + x), 4);
        }
        for (int i = 0; i < C::STAGES; ++i) {
            ptx::mbar_init(BAR(C::B_KF + i), 1);
            ptx::mbar_init(BAR(C::B_KE + i), 1);
            ptx::mbar_init(BAR(C::B_VF + i), 1);
            ptx::mbar_init(BAR(C::B_VE + i), 1);
        }
        ptx::mbar_init(BAR(C::B_DONE), 1);
        ptx::mbar_init(BAR(C::B_DONE + 1), 1);
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
    // bounded waits of the row warpgroups (no pointer kept live: the abort flag by address)
    const uint32_t abort_saddr = ptx::smem_u32(misc + C::OFF_ABORT);
    auto wait_row = [&](uint32_t bar, uint32_t parity) -> bool {
        bool okw = ptx::mbar_try_wait(bar, parity);
        if (!okw) okw = wait_slow_s(bar, parity, abort_saddr, p.timeout_ns, p.status);
        return __all_sync(0xffffffffu, okw);
    };

    if (warp >= 8) {
      ptx::setmaxnreg_dec<kPfRegsCtl>();
      if (warp == 8) {
        // ======================================================== TMA producer
        const bool paged = p.kv_mode == 2;
        int issued_k = 0, issued_v = 0, issued_q = 0;
        bool ok = true;
        int it = 0, uidx = 0;
        for (int k = 0; ok; ++k) {
            const int u = pf_unit_index(p, k);
            if (u < 0) break;
            const PfUnit un = pf_unit(p, u, cap);
            if (un.state != 2) continue;
            // this unit's Q into buffer uidx % 2, once the unit two back has issued its last QK
            const int qb = uidx & 1;
            if (!W.wait_warp(BAR(C::B_QE + qb), (((uint32_t)uidx >> 1) & 1u) ^ 1u)) { ok = false; break; }
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(BAR(C::B_QF + qb), (uint32_t)(D * p.rows_per_tile));
                const int c2 = p.q_varlen ? un.q_start + un.pos0 : un.pos0;
                const int c3 = p.q_varlen ? 0 : un.b;
#pragma unroll
                for (int c = 0; c < C::NCK; ++c)
                    ptx::tma_load_4d(sQ + qb * C::Q_BYTES + c * C::CHUNK_Q, &tm_q, BAR(C::B_QF + qb), c * C::CW,
                                     un.kvh * p.G, c2, c3);
            }
            __syncwarp();
            issued_q = ++uidx;
            for (int j = un.t_beg; j < un.t_end; ++j, ++it) {
                const int k0 = j * kTileN;
                const int st = it % C::STAGES;
                const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
                int page = 0, prow = 0;
                if (paged && lane < p.boxes_per_tile) {
                    const int j0 = k0 + lane * p.box_n;
                    const int pi = j0 / p.page_size;
                    prow = j0 - pi * p.page_size;
                    page = p.num_pages;  // past the request's keys: out of range, TMA fills zeros
                    if (j0 < un.Lk) {
                        const int e = p.block_table[(long long)un.b * p.bt_stride + pi];
                        if (e >= 0 && e < p.num_pages) page = e;
                        else atomicOr(p.status, kStatusBounds);
                    }
                }
                const int c2 = p.kv_mode == 1 ? un.k_start + k0 : k0;
                const int c3 = p.kv_mode == 1 ? 0 : un.b;
                if (!W.wait_warp(BAR(C::B_KE + st), ph ^ 1u)) { ok = false; break; }
                if (lane == 0) ptx::mbar_arrive_expect_tx(BAR(C::B_KF + st), (uint32_t)C::K_BYTES);
                __syncwarp();
                const uint32_t dK = sK + st * C::K_BYTES;
                if (paged) {
                    if (lane < p.boxes_per_tile) {
#pragma unroll
                        for (int c = 0; c < C::NCK; ++c)
                            ptx::tma_load_4d(dK + c * C::CHUNK_K + lane * p.box_n * C::CW, &tm_k, BAR(C::B_KF + st),
                                             c * C::CW, un.kvh, prow, page);
                    }
                } else if (lane == 0) {
#pragma unroll
                    for (int c = 0; c < C::NCK; ++c)
                        ptx::tma_load_4d(dK + c * C::CHUNK_K, &tm_k, BAR(C::B_KF + st), c * C::CW, un.kvh, c2, c3);
                }
                issued_k = it + 1;
                if (lane == 0) FA8_EV(3, it);
                if (!W.wait_warp(BAR(C::B_VE + st), ph ^ 1u)) { ok = false; break; }
                if (lane == 0) ptx::mbar_arrive_expect_tx(BAR(C::B_VF + st), (uint32_t)C::V_BYTES);
                __syncwarp();
                const uint32_t dV = sV + st * C::V_BYTES;
                if (paged) {
                    if (lane < p.boxes_per_tile) {
#pragma unroll
                        for (int c = 0; c < C::NCV; ++c)
                            ptx::tma_load_4d(dV + c * C::CHUNK_V + lane * p.box_n * C::CWV, &tm_v, BAR(C::B_VF + st),
                                             c * C::CWV, un.kvh, prow, page);
                    }
                } else if (lane == 0) {
#pragma unroll
                    for (int c = 0; c < C::NCV; ++c)
                        ptx::tma_load_4d(dV + c * C::CHUNK_V, &tm_v, BAR(C::B_VF + st), c * C::CWV, un.kvh, c2, c3);
                }
                issued_v = it + 1;
                if (lane == 0) FA8_EV(4, it);
            }
        }
        if (*abort_flag) {
            // every load already issued must land before the CTA's smem is released
            for (int i = max(0, issued_q - 2); i < issued_q; ++i)
                W.drain(BAR(C::B_QF + (i & 1)), (uint32_t)(i >> 1) & 1u);
            for (int i = max(0, issued_k - C::STAGES); i < issued_k; ++i)
                W.drain(BAR(C::B_KF + i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u);
            for (int i = max(0, issued_v - C::STAGES); i < issued_v; ++i)
                W.drain(BAR(C::B_VF + i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u);
        }
        __syncwarp();
      } else if (warp == 9 || warp == 10) {
        // ======================================================== MMA issuers (one elected lane each)
        // warp 9 issues PV(i) for every tile; warp 10 issues QK(i + 2) once PV(i) has completed
        // (QK(i + 2) overwrites the S/P columns PV(i) reads), so neither waits on the other's
        // issue costs.
        constexpr uint32_t kIdescQK = idesc_e4m3(kTileM, kTileN, false);
        constexpr uint32_t kIdescPV = idesc_e4m3(kTileM, DV, true);
        const bool leader = ptx::elect_one();
        bool ok = true;
        const bool is_qk = warp == 10;
        const uint64_t dk0 = sdesc(sK, 16, 8 * C::CW, swz_layout(C::CW));
        const uint64_t dv0 = sdesc(sV, C::CHUNK_V, 8 * C::CWV, swz_layout(C::CWV));
        int i = 0, uidx = 0;
        for (int k = 0; ok; ++k) {
            const int u = pf_unit_index(p, k);
            if (u < 0) break;
            const PfUnit un = pf_unit(p, u, cap);
            if (un.state != 2) continue;
            const int qb = uidx & 1;
            ++uidx;
            for (int j = un.t_beg; j < un.t_end; ++j, ++i) {
                if (is_qk) {
                    // S(i) = Q K_j^T; it overwrites P(i - 2): PV(i - 2) must be complete
                    if (i >= 2 && !W.wait_warp(BAR(C::B_OF + (i & 1)), (((uint32_t)i >> 1) & 1u) ^ 1u)) { ok = false; break; }
                    if (lane == 0) FA8_EV(11, i);
                    if (j == un.t_beg && !W.wait_warp(BAR(C::B_QF + qb), ((uint32_t)(uidx - 1) >> 1) & 1u)) { ok = false; break; }
                    const int ks = i % C::STAGES;
                    if (!W.wait_warp(BAR(C::B_KF + ks), (uint32_t)(i / C::STAGES) & 1u)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint64_t dq = sdesc(sQ + qb * C::Q_BYTES, 16, 8 * C::CW, swz_layout(C::CW));
                    const uint64_t dk = dk0 + (uint64_t)((ks * C::K_BYTES) >> 4);
                    if (leader) {
#pragma unroll
                        for (int kk = 0; kk < D / 32; ++kk) {
                            const uint32_t off = (uint32_t)((((kk * 32) / C::CW) * C::CHUNK_Q + (kk * 32) % C::CW) >> 4);
                            ptx::mma_f8_ss(tmem + C::TM_S + (uint32_t)(i & 1) * 128u, dq + off, dk + off, kIdescQK,
                                           kk > 0 ? 1u : 0u);
                        }
                        ptx::tc_commit(BAR(C::B_SF + (i & 1)));
                        ptx::tc_commit(BAR(C::B_KE + ks));
                        if (j + 1 == un.t_end) ptx::tc_commit(BAR(C::B_QE + qb));  // the unit's last QK
                    }
                    __syncwarp();
                    if (lane == 0) FA8_EV(10, i);
                } else {
                    // O_t(i) = P(i) V_j (+ P_lo V_j): waits for P(i) and for the fold of O_t(i - 2).
                    // The P_hi MMAs go first; the two-term decision (the mask, or any warp's vote) is
                    // read while they run, and the P_lo MMAs (onto the same O_t) follow if needed.
                    const int vs = i % C::STAGES;
                    if (!W.wait_warp(BAR(C::B_VF + vs), (uint32_t)(i / C::STAGES) & 1u)) { ok = false; break; }
                    if (!W.wait_warp(BAR(C::B_PF + (i & 1)), ((uint32_t)i >> 1) & 1u)) { ok = false; break; }
                    if (i >= 2 && !W.wait_warp(BAR(C::B_OE + (i & 1)), (((uint32_t)i >> 1) & 1u) ^ 1u)) { ok = false; break; }
                    if (lane == 0) FA8_EV(8, i);
                    ptx::tc_fence_after();
                    const uint64_t dv = dv0 + (uint64_t)((vs * C::V_BYTES) >> 4);
                    const uint32_t s_col = tmem + C::TM_S + (uint32_t)(i & 1) * 128u;
                    const uint32_t otile = tmem + C::TM_OT + (uint32_t)(i & 1) * 128u;
                    if (leader) {
#pragma unroll
                        for (int kk = 0; kk < kTileN / 32; ++kk)
                            ptx::mma_f8_ts(otile, s_col + kk * 32, dv + (uint64_t)((kk * 32 * C::CWV) >> 4), kIdescPV,
                                           kk > 0 ? 1u : 0u);
                    }
                    bool two_term =
                        tile_needs_mask(j * kTileN, un.Lk, p.causal, p.window_left, un.pos0, un.pos_last, un.delta);
                    if (!two_term) {
                        const int4 vt = ptx::ld_shared_v4_volatile(votes_saddr + 16u * (uint32_t)(i & 1));
                        two_term = (vt.x | vt.y | vt.z | vt.w) != 0;
                    }
                    if (leader) {
                        if (two_term) {  // + P_lo V (P_lo 8 columns after each P_hi slice)
#pragma unroll
                            for (int kk = 0; kk < kTileN / 32; ++kk)
                                ptx::mma_f8_ts(otile, s_col + kk * 32 + 8, dv + (uint64_t)((kk * 32 * C::CWV) >> 4),
                                               kIdescPV, 1u);
                        }
                        ptx::tc_commit(BAR(C::B_OF + (i & 1)));
                        ptx::tc_commit(BAR(C::B_VE + vs));
                    }
                    __syncwarp();
                    if (lane == 0) FA8_EV(9, i);
                }
            }
        }
        // this issuer's MMAs must finish before TMEM is released
        const uint32_t done = BAR(C::B_DONE + (warp - 9));
        if (leader) ptx::tc_commit(done);
        __syncwarp();
        W.drain(done, 0);
        __syncwarp();
      }
    } else if (warp < 4) {
      ptx::setmaxnreg_inc<kPfRegsSoft>();
      // ======================================================== softmax warpgroup
      const int r = tid;  // TMEM lane = row
      const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
      bool ok = true;
      int i = 0, uidx = 0;
      for (int kk = 0; ok; ++kk) {
        const int u = pf_unit_index(p, kk);
        if (u < 0) break;
        const PfUnit un = pf_unit(p, u, cap);
        if (un.state != 2) continue;
        const int rpos = un.pos0 + r / p.G;
        const int hq = un.kvh * p.G + r % p.G;
        const bool row_ok = r < p.rows_per_tile && rpos < un.Lq;
        const float dqv = p.dq ? p.dq[un.b * p.dq_sb + un.kvh * p.dq_sh] : 1.f;
        const float dkv = p.dk ? p.dk[un.b * p.dk_sb + un.kvh * p.dk_sh] : 1.f;
        const float c = p.scale_log2 * dqv * dkv;
        const uint64_t c2 = ptx::f2pack(c, c);
        const int hi_row = p.causal ? min(un.Lk - 1, rpos + un.delta) : un.Lk - 1;
        const int lo_row = p.window_left >= 0 ? max(0, rpos + un.delta - p.window_left) : 0;
        float m_run = -INFINITY, row_sum = 0.f;
        for (int j = un.t_beg; j < un.t_end; ++j, ++i) {
            const int k0 = j * kTileN;
            if (!wait_row(BAR(C::B_SF + (i & 1)), ((uint32_t)i >> 1) & 1u)) { ok = false; break; }
            if (tid == 0) FA8_EV(0, i);
            ptx::tc_fence_after();
            const uint32_t scol = tmem + lane_base + C::TM_S + (uint32_t)(i & 1) * 128u;
            const bool need_mask =
                tile_needs_mask(k0, un.Lk, p.causal, p.window_left, un.pos0, un.pos_last, un.delta);
            float mx = -INFINITY;
            if (!need_mask) {
                uint32_t u[128];
                tmem_ld128(scol, u);
                mx = row_max(u);
            } else {
                // tiles with masked columns: 32 at a time, the masked ones written back as -inf
                // for the P pass (a rolled loop: this path is rare and its code stays small)
                const int lo = lo_row - k0, hi = hi_row - k0;
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    uint32_t v[32];
                    ptx::tmem_ld32(scol + 32 * q, v);
                    ptx::tmem_wait_ld();
                    ptx::reg_fence32(v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int col = 32 * q + e;
                        if (col > hi || col < lo) v[e] = __float_as_uint(-INFINITY);
                        mx = fmaxf(mx, u2f(v[e]));
                    }
                    ptx::tmem_st32(scol + 32 * q, v);
                }
                ptx::tmem_wait_st();
            }
            if (tid == 0) FA8_EV(1, i);
            // lazy rescale; alpha(i) to the correction warpgroup
            const float mt = mx * c;
            float alpha = 1.f;
            if (mt > m_run + kTau) {
                alpha = ptx::ex2(m_run - mt);
                row_sum *= alpha;
                m_run = mt;
            }
            alpha_ring[(i & 3) * 128 + r] = alpha;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(BAR(C::B_AL + (i & 3)));
            // two-term vote: the tile's largest p is 2^(mt - m + 8); it holds more than about 1/8 of
            // the row's mass so far when log2 of it exceeds log2(row_sum) - log2(7).  log2(row_sum)
            // is taken as its fp32 exponent (the floor), without a MUFU instruction, which errs
            // towards two terms (an effective share between 1/15 and 1/8)
            bool two_term = need_mask;
            if (!need_mask) {
                const int e_rs = row_sum > 0.f ? (int)((__float_as_uint(row_sum) >> 23) & 0xFF) - 127 : -1000;
                two_term = __any_sync(0xffffffffu, row_ok && (mt - m_run + kPBias) > (float)e_rs - 2.807f);
            }
            if (lane == 0) votes[(i & 1) * 4 + warp] = two_term ? 1 : 0;
            // P = e4m3(2^(s c + (8 - m)))
            const float b8 = m_run == -INFINITY ? kPBias : kPBias - m_run;
            const uint64_t b2 = ptx::f2pack(b8, b8);
            uint64_t acc0 = ptx::f2pack(0.f, 0.f), acc1 = acc0;
            p_pass(scol, c2, b2, two_term, acc0, acc1);
            {
                float a0, a1, a2, a3;
                ptx::f2unpack(acc0, a0, a1);
                ptx::f2unpack(acc1, a2, a3);
                row_sum += (a0 + a1) + (a2 + a3);  // p carry the 2^8 bias: the biased row sum
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(BAR(C::B_PF + (i & 1)));
            if (tid == 0) FA8_EV(2, i);
        }
        if (!ok) break;
        // the unit's output scale and LSE for the correction warpgroup; the 2^8 bias cancels
        // between O and row_sum and is removed from the LSE
        {
            const bool has_sink = p.sink != nullptr && (!p.split_mode || un.split == 0);
            const float dvv = p.dv ? p.dv[un.b * p.dv_sb + un.kvh * p.dv_sh] : 1.f;
            const float sig = (has_sink && row_ok) ? p.sink[hq] : 0.f;
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
            fin_ring[(uidx & 3) * 256 + r] = scale_o;
            fin_ring[(uidx & 3) * 256 + 128 + r] = lse;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(BAR(C::B_FN + (uidx & 3)));
        }
        ++uidx;
      }
    } else {
      ptx::setmaxnreg_inc<kPfRegsCorr>();
      // ======================================================== correction warpgroup
      const int r = tid - 128;
      const int cw = warp - 4;
      const uint32_t lane_base = (uint32_t)(cw * 32) << 16;
      bool ok = true;
      int item = 0, uidx = 0;
      for (int k = 0; ok; ++k) {
        const int u = pf_unit_index(p, k);
        if (u < 0) break;
        const PfUnit un = pf_unit(p, u, cap);
        if (un.state == 0) continue;
        const int rpos = un.pos0 + r / p.G;
        const int hq = un.kvh * p.G + r % p.G;
        const bool row_ok = r < p.rows_per_tile && rpos < un.Lq;
        const int tok = un.q_start + rpos;
        const long long beta = p.q_varlen ? 0 : un.b;
        const long long rho = p.q_varlen ? tok : rpos;
        const bool has_sink = p.sink != nullptr && (!p.split_mode || un.split == 0);
        if (un.state == 1) {
            // no key of this split is visible to the tile's rows: O = 0, LSE = -inf (or the sink)
            if (row_ok) {
                const float lse = has_sink ? p.sink[hq] : -INFINITY;
                if (p.split_mode) {
                    const long long row = ((long long)un.split * p.total_q + tok) * p.Hq + hq;
                    p.lse_part[row] = lse;
                    float4 *dst = reinterpret_cast<float4 *>(p.o_part + row * DV);
                    for (int i = 0; i < DV / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                } else {
                    if (p.lse) p.lse[beta * p.lse_sb + hq * p.lse_sh + rho * p.lse_ss] = lse;
                    uint8_t *dst = reinterpret_cast<uint8_t *>(p.o) + 2 * (beta * p.o_sb + rho * p.o_ss + hq * p.o_sh);
                    for (int i = 0; i < DV / 8; ++i) *reinterpret_cast<uint4 *>(dst + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            continue;
        }
        uint64_t o2[DV / 2];  // the row's running O, as packed fp32 pairs (columns 2i, 2i+1)
#pragma unroll
        for (int q = 0; q < DV / 2; ++q) o2[q] = ptx::f2pack(0.f, 0.f);
        const int nt = un.t_end - un.t_beg;
        float scale_o = 0.f, lse = 0.f;
        for (int n = 0; n < nt; ++n, ++item) {
            const int i = item;
            if (!wait_row(BAR(C::B_AL + (i & 3)), ((uint32_t)i >> 2) & 1u)) { ok = false; break; }
            const float a = alpha_ring[(i & 3) * 128 + r];
            if (tid == 128) FA8_EV(12, i);
            if (!wait_row(BAR(C::B_OF + (i & 1)), ((uint32_t)i >> 1) & 1u)) { ok = false; break; }
            if (tid == 128) FA8_EV(13, i);
            ptx::tc_fence_after();
            fold_pass<DV>(tmem + lane_base + C::TM_OT + (uint32_t)(i & 1) * 128u, ptx::f2pack(a, a), o2);
            if (n == nt - 1) {
                // the unit's scale and LSE: waited before this last fold is released, so the
                // softmax cannot reach this ring slot's next use before it is read
                if (!wait_row(BAR(C::B_FN + (uidx & 3)), ((uint32_t)uidx >> 2) & 1u)) { ok = false; break; }
                scale_o = fin_ring[(uidx & 3) * 256 + r];
                lse = fin_ring[(uidx & 3) * 256 + 128 + r];
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(BAR(C::B_OE + (i & 1)));
            if (tid == 128) FA8_EV(14, i);
        }
        if (!ok) break;
        ++uidx;
        if (row_ok) {
            if (p.split_mode) {
                const long long row = ((long long)un.split * p.total_q + tok) * p.Hq + hq;
                p.lse_part[row] = lse;
                float *dst = p.o_part + row * DV;
#pragma unroll
                for (int q = 0; q < DV; q += 4) {
                    float v0, v1, v2, v3;
                    ptx::f2unpack(o2[q / 2], v0, v1);
                    ptx::f2unpack(o2[q / 2 + 1], v2, v3);
                    *reinterpret_cast<float4 *>(dst + q) = make_float4(v0 * scale_o, v1 * scale_o, v2 * scale_o, v3 * scale_o);
                }
            } else {
                if (p.lse) p.lse[beta * p.lse_sb + hq * p.lse_sh + rho * p.lse_ss] = lse;
                uint8_t *dst = reinterpret_cast<uint8_t *>(p.o) + 2 * (beta * p.o_sb + rho * p.o_ss + hq * p.o_sh);
#pragma unroll
                for (int q = 0; q < DV; q += 8) {
                    float t8[8];
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        ptx::f2unpack(o2[(q + e) / 2], t8[e], t8[e + 1]);
                        t8[e] *= scale_o;
                        t8[e + 1] *= scale_o;
                    }
                    store8(dst + 2 * q, t8, p.out_fp16);
                }
            }
        }
      }
    }
    // ------------------------------------------------------------ teardown
    ptx::tc_fence_before();
    __syncthreads();
#ifdef FA8_TRACE
    if (p.trace && blockIdx.x < kTraceCtas) {
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
