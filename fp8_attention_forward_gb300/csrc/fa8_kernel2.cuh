// fa8_kernel2.cuh -- the prefill form of the forward kernel (dv <= 128): two 128-row Q tiles
// per CTA that share every K/V tile and take turns on the tensor core.
//
// Roles (384 threads, three warpgroups):
//   warpgroup 0 (warps 0-3)  softmax + two-level fold + epilogue for Q tile 0
//   warpgroup 1 (warps 4-7)  the same for Q tile 1
//   warp 8                   TMA producer (both Q tiles once, K/V tiles into S-stage rings)
//   warp 9                   MMA issuer (lane 0) and TMEM owner
//   warps 10-11              idle; warpgroup 2 gives its registers to warpgroups 0 and 1
// TMEM (512 columns): S0 [0,128), S1 [128,256), O_tile0 [256, 256+dv), O_tile1 after it.
// The running fp32 O of each row lives in the registers of the thread that owns the row.
//
// Tensor-core order per KV tile j (after S0(0), S1(0)):
//   O_tile0 = P0(j) V_j,  S0 = Q0 K_{j+1}^T,  O_tile1 = P1(j) V_j,  S1 = Q1 K_{j+1}^T
// so each warpgroup's softmax of tile j+1 overlaps the other tile's MMAs (the ping-pong of
// two Q tiles described for the FlashAttention-4 forward in "PyTorch ... FlashAttention-4
// MXFP8", section 2.1.1).  Each warpgroup, per KV tile: softmax -> P (E4M3, 2^8 bias, two
// terms on masked tiles) -> fold of the previous tile's O_tile into O (O = O * alpha +
// O_tile, "[Cute,Fwd,Sm90] Native FP8 ... forward for Hopper", Design, two-level PV
// accumulation).
#pragma once

#include "fa8_kernel.cuh"

namespace fa8 {

// register split after setmaxnreg (128 x 48 + 256 x 224 <= 384 x 168 at launch)
constexpr int kRegsMath2 = 224;
constexpr int kRegsCtl2 = 48;

template <int D, int DV>
struct Cfg2 {
    static_assert(DV <= 128, "two-tile kernel keeps O in registers");
    static constexpr int CW = Cfg<D, DV>::CW;
    static constexpr int NCK = D / CW;
    static constexpr int CWV = Cfg<D, DV>::CWV;
    static constexpr int NCV = DV / CWV;
    static constexpr uint32_t TM_S = 0;     // tile i: TM_S + 128 i
    static constexpr uint32_t TM_OT = 256;  // tile i: TM_OT + DV i
    static constexpr uint32_t TM_COLS = 512;
    static constexpr int CHUNK_Q = kTileM * CW;
    static constexpr int CHUNK_K = kTileN * CW;
    static constexpr int CHUNK_V = kTileN * CWV;
    static constexpr int QT_BYTES = kTileM * D;  // one Q tile
    static constexpr int K_BYTES = kTileN * D;
    static constexpr int V_BYTES = kTileN * DV;
    static constexpr int MISC_BYTES = 1024;
    static constexpr int SMEM_LIMIT = 232448;
    static constexpr int STAGES_FIT = (SMEM_LIMIT - 1024 - MISC_BYTES - 2 * QT_BYTES) / (K_BYTES + V_BYTES);
    static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = 2 * QT_BYTES;
    static constexpr int OFF_V = OFF_K + STAGES * K_BYTES;
    static constexpr int OFF_MISC = OFF_V + STAGES * V_BYTES;
    static constexpr int SMEM_BYTES = OFF_MISC + MISC_BYTES + 1024;
    static constexpr int B_Q = 0;
    static constexpr int B_KF = 1;
    static constexpr int B_KE = B_KF + STAGES;
    static constexpr int B_VF = B_KE + STAGES;
    static constexpr int B_VE = B_VF + STAGES;
    static constexpr int B_SF = B_VE + STAGES;  // 2: per Q tile
    static constexpr int B_PF = B_SF + 2;
    static constexpr int B_OF = B_PF + 2;
    static constexpr int B_OE = B_OF + 2;
    static constexpr int B_DONE = B_OE + 2;
    static constexpr int NUM_BARS = B_DONE + 1;
    static_assert(STAGES >= 2, "smem too small for two K/V stages");
    static_assert(NUM_BARS * 8 + 16 <= MISC_BYTES, "barrier area");
    static_assert(TM_OT + 2 * DV <= TM_COLS, "TMEM budget");
};

template <int D, int DV>
__global__ void __launch_bounds__(kNumThreads, 1)
    fwd2_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
    using C = Cfg2<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // ------------------------------------------------------------ tile schedule
    int b, mp;  // request, pair of m-blocks
    if (!p.q_varlen) {
        const int x = blockIdx.x;
        b = x % p.B;
        mp = p.mblocks_per_batch - 1 - x / p.B;
    } else if (!varlen_slot(p, blockIdx.x, b, mp, 2)) {
        return;
    }
    const int kvh = blockIdx.y % p.Hkv;
    const int split = blockIdx.y / p.Hkv;
    const int P = p.pos_per_tile;
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
    const int pos00 = 2 * mp * P;  // first position of Q tile 0
    if (pos00 >= Lq) return;
    const int delta = Lk - Lq;
    const int pos_hi = min(pos00 + 2 * P, Lq) - 1;  // last valid position of the pair
    const int kv_end = p.causal ? min(Lk, pos_hi + delta + 1) : Lk;
    const int kv_beg = p.window_left >= 0 ? max(0, pos00 + delta - p.window_left) : 0;
    int t_beg = 0, n_tiles = 0;
    if (kv_end > kv_beg) {
        const int tb = kv_beg / kTileN;
        const int te = (kv_end + kTileN - 1) / kTileN;
        const int per = (te - tb + p.num_splits - 1) / p.num_splits;
        t_beg = tb + split * per;
        n_tiles = max(0, min(te, t_beg + per) - t_beg);
    }
    // Q tile i covers positions [pos00 + i P, pos00 + (i+1) P)
    auto tile_pos0 = [&](int i) { return pos00 + i * P; };
    auto tile_last = [&](int i) { return min(pos00 + (i + 1) * P, Lq) - 1; };

    // ------------------------------------------------------------ per-row facts (warps 0-7)
    const int wg = (warp < 8) ? (warp >> 2) : 0;  // Q tile of this thread
    const int r = tid & 127;
    const int pos0 = tile_pos0(wg);
    const int pos_last = tile_last(wg);
    const int rpos = pos0 + r / p.G;
    const int hq = kvh * p.G + r % p.G;
    const bool row_ok = warp < 8 && r < p.rows_per_tile && rpos < Lq;
    const int tok = q_start + rpos;
    const long long beta = p.q_varlen ? 0 : b;
    const long long rho = p.q_varlen ? tok : rpos;
    const bool has_sink = p.sink != nullptr && (!p.split_mode || split == 0);

    if (n_tiles == 0) {
        if (row_ok) {
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
        }
        return;
    }

    // ------------------------------------------------------------ shared memory
    uint8_t *misc = smem + C::OFF_MISC;
    const uint32_t bar0 = ptx::smem_u32(misc);
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc + 8 * C::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 8 * C::NUM_BARS + 4);
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
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(BAR(C::B_SF + i), 1);
            ptx::mbar_init(BAR(C::B_PF + i), 128);
            ptx::mbar_init(BAR(C::B_OF + i), 1);
            ptx::mbar_init(BAR(C::B_OE + i), 128);
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
    if (tid == 0) FA8_EV(15, 0);

    if (warp >= 8) {
        ptx::setmaxnreg_dec<kRegsCtl2>();
        if (warp == 8) {
            // ==================================================== TMA producer
            const bool paged = p.kv_mode == 2;
            int issued_k = 0, issued_v = 0;
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(BAR(C::B_Q), (uint32_t)(2 * D * p.rows_per_tile));
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int c2 = p.q_varlen ? q_start + tile_pos0(i) : tile_pos0(i);
                    const int c3 = p.q_varlen ? 0 : b;
#pragma unroll
                    for (int c = 0; c < C::NCK; ++c)
                        ptx::tma_load_4d(sQ + i * C::QT_BYTES + c * C::CHUNK_Q, &tm_q, BAR(C::B_Q), c * C::CW,
                                         kvh * p.G, c2, c3);
                }
            }
            for (int it = 0; it < n_tiles; ++it) {
                const int k0 = (t_beg + it) * kTileN;
                const int st = it % C::STAGES;
                const uint32_t ph = (uint32_t)(it / C::STAGES) & 1u;
                int page = 0, prow = 0;
                if (paged && lane < p.boxes_per_tile) {
                    const int j0 = k0 + lane * p.box_n;
                    const int pi = j0 / p.page_size;
                    prow = j0 - pi * p.page_size;
                    page = p.num_pages;
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
                W.drain(BAR(C::B_Q), 0);
                for (int i = max(0, issued_k - C::STAGES); i < issued_k; ++i)
                    W.drain(BAR(C::B_KF + i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u);
                for (int i = max(0, issued_v - C::STAGES); i < issued_v; ++i)
                    W.drain(BAR(C::B_VF + i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u);
            }
            __syncwarp();
        } else if (warp == 9) {
            // ==================================================== MMA issuer
            if (lane == 0) {
                constexpr uint32_t kIdescQK = idesc_e4m3(kTileM, kTileN, false);
                constexpr uint32_t kIdescPV = idesc_e4m3(kTileM, DV, true);
                bool ok = W.wait(BAR(C::B_Q), 0);
                ptx::tc_fence_after();
                // S_i = Q_i K_j^T (the K wait is done once, before tile 0's product)
                auto qk = [&](int i, int j) -> bool {
                    const int ks = j % C::STAGES;
                    if (i == 0) {
                        if (!W.wait(BAR(C::B_KF + ks), (uint32_t)(j / C::STAGES) & 1u)) return false;
                        ptx::tc_fence_after();
                    }
                    const uint32_t kbase = sK + ks * C::K_BYTES;
                    const uint32_t qbase = sQ + i * C::QT_BYTES;
#pragma unroll
                    for (int kk = 0; kk < D / 32; ++kk) {
                        const int chunk = (kk * 32) / C::CW;
                        const int off = (kk * 32) % C::CW;
                        const uint64_t qd = sdesc(qbase + chunk * C::CHUNK_Q + off, 16, 8 * C::CW, swz_layout(C::CW));
                        const uint64_t kd = sdesc(kbase + chunk * C::CHUNK_K + off, 16, 8 * C::CW, swz_layout(C::CW));
                        ptx::mma_f8_ss(tmem + C::TM_S + 128 * i, qd, kd, kIdescQK, kk > 0 ? 1u : 0u);
                    }
                    ptx::tc_commit(BAR(C::B_SF + i));
                    if (i == 1) ptx::tc_commit(BAR(C::B_KE + ks));
                    return true;
                };
                // O_tile_i = P_i(j) V_j (+ P_lo V_j on masked tiles)
                auto pv = [&](int i, int j) -> bool {
                    const int vs = j % C::STAGES;
                    if (!W.wait(BAR(C::B_PF + i), (uint32_t)j & 1u)) return false;
                    if (i == 0 && !W.wait(BAR(C::B_VF + vs), (uint32_t)(j / C::STAGES) & 1u)) return false;
                    if (!W.wait(BAR(C::B_OE + i), ((uint32_t)j & 1u) ^ 1u)) return false;
                    ptx::tc_fence_after();
                    const int k0 = (t_beg + j) * kTileN;
                    const bool two_term =
                        tile_needs_mask(k0, Lk, p.causal, p.window_left, tile_pos0(i), tile_last(i), delta);
                    const uint32_t vbase = sV + vs * C::V_BYTES;
                    const uint32_t s_col = tmem + C::TM_S + 128 * i;
                    const uint32_t otile = tmem + C::TM_OT + DV * i;
#pragma unroll
                    for (int kk = 0; kk < kTileN / 32; ++kk) {
                        const uint64_t bd = sdesc(vbase + kk * 32 * C::CWV, C::CHUNK_V, 8 * C::CWV, swz_layout(C::CWV));
                        ptx::mma_f8_ts(otile, s_col + 32 * kk, bd, kIdescPV, kk > 0 ? 1u : 0u);
                    }
                    if (two_term) {
#pragma unroll
                        for (int kk = 0; kk < kTileN / 32; ++kk) {
                            const uint64_t bd =
                                sdesc(vbase + kk * 32 * C::CWV, C::CHUNK_V, 8 * C::CWV, swz_layout(C::CWV));
                            ptx::mma_f8_ts(otile, s_col + 32 * kk + 8, bd, kIdescPV, 1u);
                        }
                    }
                    ptx::tc_commit(BAR(C::B_OF + i));
                    if (i == 1) ptx::tc_commit(BAR(C::B_VE + vs));
                    return true;
                };
                if (ok) ok = qk(0, 0) && qk(1, 0);
                for (int j = 0; ok && j < n_tiles; ++j) {
                    FA8_EV(2, j);
                    ok = pv(0, j);
                    if (ok && j + 1 < n_tiles) ok = qk(0, j + 1);
                    if (ok) ok = pv(1, j);
                    if (ok && j + 1 < n_tiles) ok = qk(1, j + 1);
                    FA8_EV(3, j);
                }
                ptx::tc_commit(BAR(C::B_DONE));
                W.drain(BAR(C::B_DONE), 0);
            }
            __syncwarp();
        }
    } else {
        ptx::setmaxnreg_inc<kRegsMath2>();
        // ======================================================== softmax + fold (tile wg)
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const bool warp_active = __any_sync(0xffffffffu, row_ok);
        const float dqv = p.dq ? p.dq[b * p.dq_sb + kvh * p.dq_sh] : 1.f;
        const float dkv = p.dk ? p.dk[b * p.dk_sb + kvh * p.dk_sh] : 1.f;
        const float dvv = p.dv ? p.dv[b * p.dv_sb + kvh * p.dv_sh] : 1.f;
        const float c = p.scale_log2 * dqv * dkv;
        const uint64_t c2 = ptx::f2pack(c, c);
        const int hi_row = p.causal ? min(Lk - 1, rpos + delta) : Lk - 1;
        const int lo_row = p.window_left >= 0 ? max(0, rpos + delta - p.window_left) : 0;
        const uint32_t scol = tmem + lane_base + C::TM_S + 128 * wg;
        const uint32_t ocol = tmem + lane_base + C::TM_OT + DV * wg;
        float o[DV];
#pragma unroll
        for (int i = 0; i < DV; ++i) o[i] = 0.f;
        float m_run = -INFINITY, row_sum = 0.f, alpha_prev = 0.f;
        for (int j = 0; j <= n_tiles; ++j) {
            float alpha = 1.f;
            if (j < n_tiles) {
                // ------------------------------------------------ softmax of tile j
                const int k0 = (t_beg + j) * kTileN;
                if (!W.wait_warp(BAR(C::B_SF + wg), (uint32_t)j & 1u)) break;
                if (tid == 0) FA8_EV(4, j);
                ptx::tc_fence_after();
                if (warp_active) {
                    const bool need_mask = tile_needs_mask(k0, Lk, p.causal, p.window_left, pos0, pos_last, delta);
                    const int hi = hi_row - k0, lo = lo_row - k0;
                    // pass 1: row max, one 32-column slice per TMEM round trip
                    float mx = -INFINITY;
#pragma unroll 1
                    for (int q = 0; q < 4; ++q) {
                        uint32_t u[32];
                        ptx::tmem_ld32(scol + 32 * q, u);
                        ptx::tmem_wait_ld();
                        ptx::reg_fence32(u);
                        float x[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            x[i] = u2f(u[i]);
                            if (need_mask && (32 * q + i > hi || 32 * q + i < lo)) x[i] = -INFINITY;
                        }
                        float m0 = ptx::fmax3(x[0], x[1], x[2]), m1 = ptx::fmax3(x[3], x[4], x[5]);
#pragma unroll
                        for (int i = 6; i < 30; i += 4) {
                            m0 = ptx::fmax3(m0, x[i], x[i + 1]);
                            m1 = ptx::fmax3(m1, x[i + 2], x[i + 3]);
                        }
                        mx = ptx::fmax3(mx, ptx::fmax3(m0, x[30], x[31]), m1);
                    }
                    const float mt = mx * c;
                    if (mt > m_run + kTau) {
                        alpha = ptx::ex2(m_run - mt);
                        row_sum *= alpha;
                        m_run = mt;
                    }
                    const float bias = kPBias - (m_run == -INFINITY ? 0.f : m_run);
                    const uint64_t b2 = ptx::f2pack(bias, bias);
                    uint64_t acc0 = ptx::f2pack(0.f, 0.f), acc1 = acc0;
                    // pass 2: P = 2^(s c - m + 8) for 16 keys per step.  The packed E4M3 of
                    // keys [32q, 32q+32) occupies columns [32q, 32q+8) of the S buffer (P_lo
                    // 8 columns later on masked tiles); every write lands on columns of S
                    // that this thread has already read.
#pragma unroll 1
                    for (int sl = 0; sl < 8; ++sl) {
                        uint32_t u[16];
                        ptx::tmem_ld16(scol + 16 * sl, u);
                        ptx::tmem_wait_ld();
                        ptx::reg_fence16(u);
                        float x[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            x[i] = u2f(u[i]);
                            if (need_mask && (16 * sl + i > hi || 16 * sl + i < lo)) x[i] = -INFINITY;
                        }
                        uint32_t w[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            float x0, x1, x2, x3;
                            ptx::f2unpack(ptx::ffma2(ptx::f2pack(x[4 * k], x[4 * k + 1]), c2, b2), x0, x1);
                            ptx::f2unpack(ptx::ffma2(ptx::f2pack(x[4 * k + 2], x[4 * k + 3]), c2, b2), x2, x3);
                            x[4 * k] = ptx::ex2(x0);
                            x[4 * k + 1] = ptx::ex2(x1);
                            x[4 * k + 2] = ptx::ex2(x2);
                            x[4 * k + 3] = ptx::ex2(x3);
                            acc0 = ptx::fadd2(acc0, ptx::f2pack(x[4 * k], x[4 * k + 1]));
                            acc1 = ptx::fadd2(acc1, ptx::f2pack(x[4 * k + 2], x[4 * k + 3]));
                            w[k] = ptx::cvt_e4m3x2(x[4 * k + 1], x[4 * k]) |
                                   (ptx::cvt_e4m3x2(x[4 * k + 3], x[4 * k + 2]) << 16);
                        }
                        const uint32_t pc = scol + 32 * (sl >> 1) + 4 * (sl & 1);
                        ptx::tmem_st4(pc, w);
                        if (need_mask) {
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                float q0, q1, q2, q3;
                                ptx::e4m3x2_to_f32(w[k] & 0xFFFFu, q0, q1);
                                ptx::e4m3x2_to_f32(w[k] >> 16, q2, q3);
                                w[k] = ptx::cvt_e4m3x2(x[4 * k + 1] - q1, x[4 * k] - q0) |
                                       (ptx::cvt_e4m3x2(x[4 * k + 3] - q3, x[4 * k + 2] - q2) << 16);
                            }
                            ptx::tmem_st4(pc + 8, w);
                        }
                    }
                    ptx::tmem_wait_st();
                    float a0, a1, a2, a3;
                    ptx::f2unpack(acc0, a0, a1);
                    ptx::f2unpack(acc1, a2, a3);
                    row_sum += (a0 + a1) + (a2 + a3);
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(BAR(C::B_PF + wg));
                if (tid == 0) FA8_EV(5, j);
            }
            if (j > 0) {
                // ------------------------------------------------ fold of tile j-1
                if (!W.wait_warp(BAR(C::B_OF + wg), (uint32_t)(j - 1) & 1u)) break;
                if (tid == 0) FA8_EV(7, j - 1);
                ptx::tc_fence_after();
                if (warp_active) {
                    // O starts at 0 and the first visible tile has alpha = 0
                    const uint64_t a2 = ptx::f2pack(alpha_prev, alpha_prev);
#pragma unroll
                    for (int q = 0; q < DV / 32; ++q) {
                        uint32_t u[32];
                        ptx::tmem_ld32(ocol + 32 * q, u);
                        ptx::tmem_wait_ld();
                        ptx::reg_fence32(u);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            const uint64_t r2 = ptx::ffma2(ptx::f2pack(o[32 * q + i], o[32 * q + i + 1]), a2,
                                                           ptx::f2pack(u2f(u[i]), u2f(u[i + 1])));
                            ptx::f2unpack(r2, o[32 * q + i], o[32 * q + i + 1]);
                        }
                    }
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(BAR(C::B_OE + wg));
                if (tid == 0) FA8_EV(8, j - 1);
            }
            alpha_prev = alpha;
        }
        // ---------------------------------------------------- finalize and store
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
        if (row_ok) {
            if (p.split_mode) {
                const long long row = ((long long)split * p.total_q + tok) * p.Hq + hq;
                p.lse_part[row] = lse;
                float *dst = p.o_part + row * DV;
#pragma unroll
                for (int i = 0; i < DV; i += 4)
                    *reinterpret_cast<float4 *>(dst + i) =
                        make_float4(o[i] * scale_o, o[i + 1] * scale_o, o[i + 2] * scale_o, o[i + 3] * scale_o);
            } else {
                if (p.lse) p.lse[beta * p.lse_sb + hq * p.lse_sh + rho * p.lse_ss] = lse;
                uint8_t *dst = reinterpret_cast<uint8_t *>(p.o) + 2 * (beta * p.o_sb + rho * p.o_ss + hq * p.o_sh);
#pragma unroll
                for (int i = 0; i < DV; i += 8) {
                    float t8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) t8[e] = o[i + e] * scale_o;
                    store8(dst + 2 * i, t8, p.out_fp16);
                }
            }
        }
    }
    // ------------------------------------------------------------ teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (tid == 0) FA8_EV(15, 1);
    if (warp == 9) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::TM_COLS);
    }
}

}  // namespace fa8
