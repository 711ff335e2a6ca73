// fa8_decode.cuh -- the forward for few query rows per kv-head (decode): at most 16 rows
// (query positions x q-heads of one kv-head) per CTA.
//
// Same arithmetic as fwd_kernel (online exp2 softmax with the descales folded into the
// scale, P in E4M3 with a 2^8 bias, lazy rescale with tau = 0.75, two-level PV
// accumulation, sink and LSE at finalize), except that every tile's P goes through the PV
// MMA as two E4M3 terms, P_hi + P_lo with P_lo = e4m3(p - P_hi): decode rows often hold a
// few keys that carry most of the softmax mass, where one E4M3 term (up to 2^-4 relative
// rounding of a dominant weight) can put the output past the stated error bar; the second
// term costs one more small PV MMA and the P_lo stores, which this HBM-bound kernel hides.
// The tile is transposed so that the 128 keys of a KV tile lie along the MMA's M dimension
// (TMEM lanes) and the query rows along N = 16:
//
//   S^T (128 keys x 16 rows)  = K (128 x d, K-major smem)  .  Q^T (Q: 16 x d, K-major smem)
//   O^T (dv x 16 rows)       += V^T (V: 128 x dv smem, MN-major A operand) . P^T (16 x 128)
//
// so every softmax thread owns one key and holds that key's scores for the tile's rows (the
// R <= 16 real ones: see decode_kernel), and the MMAs are 8x smaller than a 128-row tile
// would make them: the kernel streams K/V at HBM rate instead of spending a 128-row softmax
// on a handful of rows.  P^T is written to shared memory MN-major (key t's 16 row bytes at
// 16 t, no swizzle; rows past R stay zero), one store per thread and term, and read by the
// PV MMA from there.
//
// Roles (384 threads): warp 0 TMA producer, warp 1 issues the QK MMAs and warp 2 the PV
// MMAs (two issuers, so that neither waits behind the other's barriers), warps 4-7 softmax
// (thread = key of the tile), warps 8-11 fold and epilogue (thread = row of O^T, i.e. a dv
// index).
#pragma once

#include "fa8_kernel.cuh"

namespace fa8 {

constexpr int kDecRows = 16;  // query rows per CTA (MMA N)
constexpr int kDecThreads = 384;

template <int D, int DV>
struct DecCfg {
    static_assert(DV % 128 == 0, "decode kernel: dv must be a multiple of 128");
    static constexpr int CW = (D % 128 == 0) ? 128 : ((D % 64 == 0) ? 64 : 32);
    static constexpr int NCK = D / CW;
    static constexpr int NDV = DV / 128;  // 128-row slices of O^T (one PV MMA each per K step)
    static constexpr int CHUNK_Q = kDecRows * CW;
    static constexpr int CHUNK_K = kTileN * CW;
    static constexpr int CHUNK_V = kTileN * 128;
    static constexpr int Q_BYTES = kDecRows * D;
    static constexpr int K_BYTES = kTileN * D;
    static constexpr int V_BYTES = kTileN * DV;
    static constexpr int P_BYTES = kDecRows * kTileN;  // one P^T buffer (16 x 128 e4m3)
    static constexpr int MISC_BYTES = 4096;
    // two CTAs per SM when three K/V stages fit in half of the shared memory
    static constexpr int HALF = 232448 / 2 - 1024;
    static constexpr int FIXED = 1024 + ((Q_BYTES + 1023) / 1024) * 1024 + 4 * P_BYTES + MISC_BYTES;
    static constexpr int CTAS = (FIXED + 3 * (K_BYTES + V_BYTES) <= HALF) ? 2 : 1;
    static constexpr int STAGES_FIT = ((CTAS == 2 ? HALF : 232448 - 1024) - FIXED) / (K_BYTES + V_BYTES);
    static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_P = ((Q_BYTES + 1023) / 1024) * 1024;  // [2 buffers][hi, lo] x 2 KB, MN-major
    static constexpr int OFF_K = OFF_P + 4 * P_BYTES;
    static constexpr int OFF_V = OFF_K + STAGES * K_BYTES;
    static constexpr int OFF_MISC = OFF_V + STAGES * V_BYTES;
    static constexpr int SMEM_BYTES = OFF_MISC + MISC_BYTES + 1024;
    // TMEM: S^T buffers at columns 0 and 16, O^T tiles at 32 + b * NDV * 16
    static constexpr uint32_t TM_S = 0;
    static constexpr uint32_t TM_OT = 32;
    static constexpr uint32_t TM_COLS = 128;
    // Alpha ring (softmax -> fold).  It needs no "slot free" barrier: the softmax writes the
    // slot of tile t after waiting for PV(t - 2) to complete, and PV(t - 2) was issued after
    // the fold of tile t - 4 (which read the slot's previous contents) released its O^T tile.
    static constexpr int NA = 4;
    // barriers
    static constexpr int B_Q = 0;
    static constexpr int B_KF = 1;
    static constexpr int B_KE = B_KF + STAGES;
    static constexpr int B_VF = B_KE + STAGES;
    static constexpr int B_VE = B_VF + STAGES;
    static constexpr int B_SF = B_VE + STAGES;  // 2: S^T written
    static constexpr int B_SE = B_SF + 2;       // 2: S^T read by the softmax
    static constexpr int B_PF = B_SE + 2;       // 2: P^T written
    static constexpr int B_PE = B_PF + 2;       // 2: P^T read by the PV MMA
    static constexpr int B_OF = B_PE + 2;       // 2: O^T tile written
    static constexpr int B_OE = B_OF + 2;       // 2: O^T tile folded
    static constexpr int B_AF = B_OE + 2;       // NA
    static constexpr int B_MX = B_AF + NA;      // 2: tile maxima of the 4 softmax warps written
    static constexpr int B_SUM = B_MX + 2;      // row-sum shares of the 4 softmax warps written
    static constexpr int B_FIN = B_SUM + 1;     // softmax -> fold: final row scales
    static constexpr int B_DONE = B_FIN + 1;
    static constexpr int NUM_BARS = B_DONE + 1;
    static_assert(STAGES >= 2, "decode kernel: smem too small for two K/V stages");
    static_assert(SMEM_BYTES <= 232448, "decode kernel: smem");
    static_assert(NUM_BARS * 8 <= 512, "barrier area");
    static_assert(TM_OT + 2 * NDV * 16 <= TM_COLS, "TMEM budget");
};

// Bounded mbarrier waits whose try_wait carries a suspend-time hint: a waiting thread
// sleeps until the phase completes (woken at once) or the hint expires, instead of
// returning after a short fixed slice.  Same timeout and abort behaviour as Waiter.
struct HintWaiter {
    static constexpr uint32_t kHintNs = 100000u;
    volatile int *abort;
    unsigned long long timeout;
    unsigned int *status;
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
        if (ptx::mbar_try_wait_sleep(bar, parity, kHintNs)) return true;
        const uint64_t t0 = ptx::globaltimer();
        while (true) {
            if (ptx::mbar_try_wait_sleep(bar, parity, kHintNs)) return true;
            if (*abort) return false;
            if (ptx::globaltimer() - t0 > timeout) {
                *abort = 1;
                atomicOr(status, kStatusTimeout);
                return false;
            }
        }
    }
    __device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity) const {
        const bool ok = wait(bar, parity);
        return __all_sync(0xffffffffu, ok);
    }
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

__device__ __forceinline__ float redux_max(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// R: the rows the softmax and fold carry (4 or 8 when a tile holds at most that many real
// rows, as in one-token decode with 4 or 8 q-heads per kv-head; 16 otherwise).  The MMAs
// always run N = 16: P^T rows R..15 stay zero and the O^T columns beyond R are never read.
template <int D, int DV, int R>
__global__ void __launch_bounds__(kDecThreads, DecCfg<D, DV>::CTAS)
    decode_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
    using C = DecCfg<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // ------------------------------------------------------------ tile schedule (batched q)
    // grid x = kv-head + Hkv * slot (kv-heads fastest), grid y = split: the CTAs of one
    // request run side by side and share the L2 lines of its pages, and the splits a
    // request does not use (split >= its split count) come last and exit at once
    const int kvh = blockIdx.x % p.Hkv;
    const int slot = blockIdx.x / p.Hkv;
    const int b = slot % p.B;
    const int mb = slot / p.B;
    const int split = blockIdx.y;
    const int P = p.pos_per_tile;  // 16 / G positions
    int cap = p.cap_const > 0 ? p.cap_const : (1 << 20);
    if (p.num_splits > 1 && p.cap_const <= 0) {  // chosen by split_plan_kernel, which may still be running
        ptx::griddep_wait();
        cap = *p.split_cap;
    }
    const int q_start = b * p.Sq;
    const int Lq = p.Sq;
    int Lk, k_start = 0;
    if (p.kv_mode == 0) {
        Lk = p.Sk;
    } else {
        k_start = p.cu_k[b];
        Lk = p.cu_k[b + 1] - k_start;
    }
    bool bad = Lk < 0;
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
    const bool has_sink = p.sink != nullptr && (!p.split_mode || split == 0);
    // row q of the tile: position pos0 + q / G, q-head kvh * G + q % G
    auto row_pos = [&](int q) { return pos0 + q / p.G; };
    auto row_ok = [&](int q) { return q < p.rows_per_tile && row_pos(q) < Lq; };

    if (n_tiles == 0) {
        if (tid < kDecRows && row_ok(tid)) {
            const int q = tid, pos = row_pos(q), hq = kvh * p.G + q % p.G, tok = q_start + pos;
            const float lse = has_sink ? p.sink[hq] : -INFINITY;
            if (p.split_mode) {
                const long long row = ((long long)split * p.total_q + tok) * p.Hq + hq;
                p.lse_part[row] = lse;
                float4 *dst = reinterpret_cast<float4 *>(p.o_part + row * DV);
                for (int i = 0; i < DV / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
                if (p.lse) p.lse[(long long)b * p.lse_sb + hq * p.lse_sh + (long long)pos * p.lse_ss] = lse;
                uint8_t *dst = reinterpret_cast<uint8_t *>(p.o) + 2 * ((long long)b * p.o_sb + (long long)pos * p.o_ss + hq * p.o_sh);
                for (int i = 0; i < DV / 8; ++i) *reinterpret_cast<uint4 *>(dst + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
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
    float *mx_s = reinterpret_cast<float *>(misc + 1024);     // [2][16 rows][4 warps]
    float *alpha_s = reinterpret_cast<float *>(misc + 1536);  // [NA][16]
    float *sum_s = reinterpret_cast<float *>(misc + 1792);    // [16 rows][4 warps]
    float *scale_s = reinterpret_cast<float *>(misc + 2048);  // [16]
    const uint32_t sQ = ptx::smem_u32(smem + C::OFF_Q);
    const uint32_t sP = ptx::smem_u32(smem + C::OFF_P);
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
            ptx::mbar_init(BAR(C::B_SE + i), 128);
            ptx::mbar_init(BAR(C::B_PF + i), 128);
            ptx::mbar_init(BAR(C::B_PE + i), 1);
            ptx::mbar_init(BAR(C::B_OF + i), 1);
            ptx::mbar_init(BAR(C::B_OE + i), 128);
        }
        for (int i = 0; i < C::NA; ++i) {
            ptx::mbar_init(BAR(C::B_AF + i), 32);
        }
        ptx::mbar_init(BAR(C::B_MX), 128);
        ptx::mbar_init(BAR(C::B_MX + 1), 128);
        ptx::mbar_init(BAR(C::B_SUM), 128);
        ptx::mbar_init(BAR(C::B_FIN), 32);
        ptx::mbar_init(BAR(C::B_DONE), 2);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (R < kDecRows) {  // P^T rows the softmax never writes read as zero by the PV MMA
        for (int i = tid; i < 4 * C::P_BYTES / 16; i += kDecThreads)
            ptx::st_shared_v4(sP + 16u * (uint32_t)i, 0u, 0u, 0u, 0u);
        ptx::fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tm_q);
        ptx::prefetch_tmap(&tm_k);
        ptx::prefetch_tmap(&tm_v);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::TM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const HintWaiter W{abort_flag, p.timeout_ns, p.status};

    if (warp == 0) {
        // ======================================================== TMA producer
        const bool paged = p.kv_mode == 2;
        int issued_k = 0, issued_v = 0;
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(BAR(C::B_Q), (uint32_t)(D * p.rows_per_tile));
#pragma unroll
            for (int c = 0; c < C::NCK; ++c)
                ptx::tma_load_4d(sQ + c * C::CHUNK_Q, &tm_q, BAR(C::B_Q), c * C::CW, kvh * p.G, pos0, b);
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
                    for (int c = 0; c < C::NDV; ++c)
                        ptx::tma_load_4d(dV + c * C::CHUNK_V + lane * p.box_n * 128, &tm_v, BAR(C::B_VF + st), c * 128,
                                         kvh, prow, page);
                }
            } else if (lane == 0) {
#pragma unroll
                for (int c = 0; c < C::NDV; ++c)
                    ptx::tma_load_4d(dV + c * C::CHUNK_V, &tm_v, BAR(C::B_VF + st), c * 128, kvh, c2, c3);
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
    } else if (warp == 1 || warp == 2) {
        // ======================================================== MMA issuers: warp 1 issues
        // S^T = K Q^T, warp 2 issues O^T = V^T P^T; each commits its own barriers
        constexpr uint32_t kIdescS = idesc_e4m3(kTileN, kDecRows, false);
        constexpr uint32_t kIdescO = idesc_e4m3(128, kDecRows, true) | (1u << 15);  // A (V) and B (P^T) MN-major
        const uint64_t da0 = sdesc(sK, 16, 8 * C::CW, swz_layout(C::CW));
        const uint64_t db0 = sdesc(sQ, 16, 8 * C::CW, swz_layout(C::CW));
        const uint64_t dv0 = sdesc(sV, C::CHUNK_V, 8 * 128, swz_layout(128));
        // P^T MN-major without swizzle: core matrices of 8 keys x 16 row bytes (128 B), the
        // next 8 keys 128 B on; the 16 rows are one core matrix wide, so both strides are 128
        const uint64_t dp0 = sdesc(sP, 128, 128, 0u);
        const bool leader = ptx::elect_one();
        bool ok = W.wait_warp(BAR(C::B_Q), 0);
        ptx::tc_fence_after();
        auto do_qk = [&](int it) -> bool {
            const int ks = it % C::STAGES, sb = it & 1;
            if (!W.wait_warp(BAR(C::B_KF + ks), (uint32_t)(it / C::STAGES) & 1u)) return false;
            ptx::tc_fence_after();
            const uint64_t da = da0 + (uint64_t)((ks * C::K_BYTES) >> 4);
            if (leader) {
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk) {
                    const int ch = (kk * 32) / C::CW, off = (kk * 32) % C::CW;
                    ptx::mma_f8_ss(tmem + C::TM_S + sb * kDecRows, da + (uint64_t)((ch * C::CHUNK_K + off) >> 4),
                                   db0 + (uint64_t)((ch * C::CHUNK_Q + off) >> 4), kIdescS, kk > 0 ? 1u : 0u);
                }
                ptx::tc_commit(BAR(C::B_SF + sb));
                ptx::tc_commit(BAR(C::B_KE + ks));
            }
            __syncwarp();
            return true;
        };
        auto do_pv = [&](int j) -> bool {
            const int vs = j % C::STAGES, pb = j & 1;
            if (!W.wait_warp(BAR(C::B_PF + pb), (uint32_t)(j >> 1) & 1u)) return false;
            if (!W.wait_warp(BAR(C::B_VF + vs), (uint32_t)(j / C::STAGES) & 1u)) return false;
            if (!W.wait_warp(BAR(C::B_OE + pb), ((uint32_t)(j >> 1) & 1u) ^ 1u)) return false;
            ptx::tc_fence_after();
            // every tile takes the second P term (see the softmax)
            constexpr bool two_term = true;
            const uint64_t dv = dv0 + (uint64_t)((vs * C::V_BYTES) >> 4);
            const uint64_t dp = dp0 + (uint64_t)((pb * 2 * C::P_BYTES) >> 4);
            if (leader) {
#pragma unroll
                for (int c = 0; c < C::NDV; ++c) {
                    const uint32_t ot = tmem + C::TM_OT + (pb * C::NDV + c) * kDecRows;
#pragma unroll
                    for (int kk = 0; kk < kTileN / 32; ++kk) {
                        const uint64_t a = dv + (uint64_t)((c * C::CHUNK_V + kk * 32 * 128) >> 4);
                        ptx::mma_f8_ss(ot, a, dp + (uint64_t)((kk * 32 * kDecRows) >> 4), kIdescO, kk > 0 ? 1u : 0u);
                    }
                    if (two_term) {  // + V^T P_lo^T (P_lo buffer follows P_hi)
#pragma unroll
                        for (int kk = 0; kk < kTileN / 32; ++kk) {
                            const uint64_t a = dv + (uint64_t)((c * C::CHUNK_V + kk * 32 * 128) >> 4);
                            ptx::mma_f8_ss(ot, a, dp + (uint64_t)((C::P_BYTES + kk * 32 * kDecRows) >> 4), kIdescO, 1u);
                        }
                    }
                }
                ptx::tc_commit(BAR(C::B_OF + pb));
                ptx::tc_commit(BAR(C::B_VE + vs));
                ptx::tc_commit(BAR(C::B_PE + pb));
            }
            __syncwarp();
            return true;
        };
        // S(j + 2) reuses the S^T buffer of S(j) once the softmax has read it (P has its own
        // buffers), so the QK issuer runs two tiles ahead; the PV issuer follows the softmax
        if (warp == 1) {
            if (ok && n_tiles > 0) ok = do_qk(0);
            if (ok && n_tiles > 1) ok = do_qk(1);
            for (int j = 0; ok && j + 2 < n_tiles; ++j) {
                ok = W.wait_warp(BAR(C::B_SE + (j & 1)), (uint32_t)(j >> 1) & 1u);
                if (ok) ok = do_qk(j + 2);
            }
        } else {
            for (int j = 0; ok && j < n_tiles; ++j) ok = do_pv(j);
        }
        // both issuers' MMAs must finish before TMEM is released (B_DONE counts two commits)
        if (leader) ptx::tc_commit(BAR(C::B_DONE));
        __syncwarp();
        if (warp == 1) W.drain(BAR(C::B_DONE), 0);
        __syncwarp();
    } else if (warp >= 4 && warp < 8) {
        // ======================================================== softmax (thread = key t)
        const int t = tid - 128;
        const int sw = warp - 4;
        const uint32_t lane_base = (uint32_t)(sw * 32) << 16;
        const float dqv = p.dq ? p.dq[b * p.dq_sb + kvh * p.dq_sh] : 1.f;
        const float dkv = p.dk ? p.dk[b * p.dk_sb + kvh * p.dk_sh] : 1.f;
        const float c = p.scale_log2 * dqv * dkv;
        // lane q < R keeps row q's running max (the same in every warp); every thread keeps
        // the rows' P biases 8 - m (8 while m = -inf) and its key's share of the row sums
        float m_lane = -INFINITY;
        float bias[R], rsum[R];
#pragma unroll
        for (int q = 0; q < R; ++q) {
            bias[q] = kPBias;
            rsum[q] = 0.f;
        }
        uint8_t *pbase = smem + C::OFF_P;
        bool ok = true;
        for (int it = 0; ok && it < n_tiles; ++it) {
            const int sb = it & 1;
            const int k0 = (t_beg + it) * kTileN;
            if (!W.wait_warp(BAR(C::B_SF + sb), (uint32_t)(it >> 1) & 1u)) break;
            ptx::tc_fence_after();
            uint32_t u[kDecRows];
            ptx::tmem_ld16(tmem + lane_base + C::TM_S + sb * kDecRows, u);
            ptx::tmem_wait_ld();
            ptx::reg_fence16(u);
            ptx::tc_fence_before();
            ptx::mbar_arrive(BAR(C::B_SE + sb));  // S^T read: the MMA may reuse the buffer
            const bool need_mask = tile_needs_mask(k0, Lk, p.causal, p.window_left, pos0, pos_last, delta);
            if (need_mask) {
                const int kg = k0 + t;
#pragma unroll
                for (int q = 0; q < R; ++q) {
                    const int pos = row_pos(q);
                    const int hi = row_ok(q) ? (p.causal ? min(Lk - 1, pos + delta) : Lk - 1) : -1;
                    const int lo = p.window_left >= 0 ? max(0, pos + delta - p.window_left) : 0;
                    if (kg > hi || kg < lo) u[q] = __float_as_uint(-INFINITY);
                }
            }
            // tile max of every row over the 128 keys: warp reduction, then across the 4 warps
            const uint32_t mx_addr = ptx::smem_u32(mx_s) + (uint32_t)(sb * kDecRows * 4 * 4);
#pragma unroll
            for (int q = 0; q < R; ++q) {
                const float m = redux_max(u2f(u[q]));
                if (lane == q) ptx::st_shared_f32(mx_addr + (uint32_t)((q * 4 + sw) * 4), m);
            }
            ptx::mbar_arrive(BAR(C::B_MX + sb));
            if (!W.wait_warp(BAR(C::B_MX + sb), (uint32_t)(it >> 1) & 1u)) break;
            // lazy rescale, row q in lane q; lane q keeps row q's factor for the hand-off
            float my_alpha = 1.f;
            bool resc = false;
            if (lane < R) {
                const float4 mv = ptx::ld_shared_f4(mx_addr + (uint32_t)(lane * 16));
                const float mt = fmaxf(fmaxf(mv.x, mv.y), fmaxf(mv.z, mv.w)) * c;
                if (mt > m_lane + kTau) {
                    my_alpha = ptx::ex2(m_lane - mt);
                    m_lane = mt;
                    resc = true;
                }
            }
            if (__any_sync(0xffffffffu, resc)) {  // some row's running max moved (rare after the first tiles)
#pragma unroll
                for (int q = 0; q < R; ++q) {
                    rsum[q] *= __shfl_sync(0xffffffffu, my_alpha, q);
                    const float mq = __shfl_sync(0xffffffffu, m_lane, q);
                    bias[q] = kPBias - (mq == -INFINITY ? 0.f : mq);
                }
            }
            // P^T(it) overwrites P^T(it - 2): wait until PV(it - 2) has read it
            if (!W.wait_warp(BAR(C::B_PE + sb), ((uint32_t)(it >> 1) & 1u) ^ 1u)) break;
            // warp 4 hands this tile's rescale factors to the fold warps (the ring slot is free:
            // PV(it - 2) has completed, see NA)
            if (sw == 0) {
                const int as = it % C::NA;
                if (lane < R) ptx::st_shared_f32(ptx::smem_u32(alpha_s) + (uint32_t)((as * kDecRows + lane) * 4), my_alpha);
                ptx::mbar_arrive(BAR(C::B_AF + as));
            }
            // key t's P_hi and P_lo bytes of rows 0..R-1, one R-byte store each (MN-major P^T)
            const uint32_t phi = ptx::smem_u32(pbase) + (uint32_t)(sb * 2 * C::P_BYTES) + 16u * (uint32_t)t;
            const uint64_t c2 = ptx::f2pack(c, c);
            uint32_t hw[R / 4], lw[R / 4];
#pragma unroll
            for (int k = 0; k < R / 4; ++k) {
                const int q = 4 * k;
                uint32_t h[2], l[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int r0 = q + 2 * e;
                    float y0, y1;
                    ptx::f2unpack(ptx::ffma2(ptx::f2pack(u2f(u[r0]), u2f(u[r0 + 1])), c2, ptx::f2pack(bias[r0], bias[r0 + 1])), y0, y1);
                    const float p0 = ptx::ex2(y0), p1 = ptx::ex2(y1);
                    rsum[r0] += p0;
                    rsum[r0 + 1] += p1;
                    h[e] = ptx::cvt_e4m3x2(p1, p0);
                    // second E4M3 term on every tile: P_lo = e4m3(p - P_hi)
                    float q0, q1;
                    ptx::e4m3x2_to_f32(h[e], q0, q1);
                    l[e] = ptx::cvt_e4m3x2(p1 - q1, p0 - q0);
                }
                hw[k] = ptx::prmt_lo16(h[0], h[1]);
                lw[k] = ptx::prmt_lo16(l[0], l[1]);
            }
            if constexpr (R == 16) {
                ptx::st_shared_v4(phi, hw[0], hw[1], hw[2], hw[3]);
                ptx::st_shared_v4(phi + C::P_BYTES, lw[0], lw[1], lw[2], lw[3]);
            } else if constexpr (R == 8) {
                ptx::st_shared_v2(phi, hw[0], hw[1]);
                ptx::st_shared_v2(phi + C::P_BYTES, lw[0], lw[1]);
            } else {
                static_assert(R == 4, "decode kernel: 4, 8 or 16 rows");
                ptx::st_shared_u32(phi, hw[0]);
                ptx::st_shared_u32(phi + C::P_BYTES, lw[0]);
            }
            ptx::fence_proxy_async_smem();  // the PV MMA reads P^T through the async proxy
            ptx::mbar_arrive(BAR(C::B_PF + sb));
        }
        // finalize: row sums over all keys (each thread holds its keys' share relative to
        // the common running max), then per row the output scale and the LSE; the 2^8 bias
        // cancels between O and the row sum and is removed from the LSE
#pragma unroll
        for (int q = 0; q < R; ++q) {
            float v = rsum[q];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == q) sum_s[q * 4 + sw] = v;
        }
        ptx::mbar_arrive(BAR(C::B_SUM));
        if (sw == 0) {
            const bool got = W.wait_warp(BAR(C::B_SUM), 0);
            const float m_q = m_lane;
            if (lane < R) {
                const int q = lane;
                const float4 v = *reinterpret_cast<const float4 *>(sum_s + q * 4);
                const float rs_q = got ? (v.x + v.y) + (v.z + v.w) : 0.f;
                const int pos = row_pos(q), hq = kvh * p.G + q % p.G, tok = q_start + pos;
                const bool ok_row = row_ok(q);
                const float dvv = p.dv ? p.dv[b * p.dv_sb + kvh * p.dv_sh] : 1.f;
                const float sig = (has_sink && ok_row) ? p.sink[hq] : 0.f;
                float scale_o = 0.f, lse;
                if (m_q == -INFINITY) {
                    lse = has_sink ? sig : -INFINITY;
                } else {
                    const float sl2 = sig * kLog2e;
                    const float m_f = (has_sink && sl2 > m_q) ? sl2 : m_q;
                    const float sc = ptx::ex2(m_q - m_f);
                    const float rs = rs_q * sc + (has_sink ? ptx::ex2(sl2 - m_f + kPBias) : 0.f);
                    scale_o = sc * dvv / rs;
                    lse = (ptx::lg2(rs) + m_f - kPBias) * kLn2;
                }
                scale_s[q] = ok_row ? scale_o : 0.f;
                if (ok_row) {
                    if (p.split_mode)
                        p.lse_part[((long long)split * p.total_q + tok) * p.Hq + hq] = lse;
                    else if (p.lse)
                        p.lse[(long long)b * p.lse_sb + hq * p.lse_sh + (long long)pos * p.lse_ss] = lse;
                }
            }
            ptx::mbar_arrive(BAR(C::B_FIN));
        }
    } else if (warp >= 8) {
        // ======================================================== fold + epilogue (thread = dv row)
        const int m = tid - 256;
        const uint32_t lane_base = (uint32_t)((warp - 8) * 32) << 16;
        float o[C::NDV][R];
#pragma unroll
        for (int cc = 0; cc < C::NDV; ++cc)
#pragma unroll
            for (int q = 0; q < R; ++q) o[cc][q] = 0.f;
        for (int it = 0; it < n_tiles; ++it) {
            const int as = it % C::NA, pb = it & 1;
            if (!W.wait_warp(BAR(C::B_AF + as), (uint32_t)(it / C::NA) & 1u)) break;
            float alpha[R];
#pragma unroll
            for (int q = 0; q < R; q += 4) {
                const float4 v = *reinterpret_cast<const float4 *>(alpha_s + as * kDecRows + q);
                alpha[q] = v.x;
                alpha[q + 1] = v.y;
                alpha[q + 2] = v.z;
                alpha[q + 3] = v.w;
            }
            if (!W.wait_warp(BAR(C::B_OF + pb), (uint32_t)(it >> 1) & 1u)) break;
            ptx::tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < C::NDV; ++cc) {
                uint32_t u[kDecRows];
                ptx::tmem_ld16(tmem + lane_base + C::TM_OT + (pb * C::NDV + cc) * kDecRows, u);
                ptx::tmem_wait_ld();
                ptx::reg_fence16(u);
#pragma unroll
                for (int q = 0; q < R; ++q) o[cc][q] = fmaf(o[cc][q], alpha[q], u2f(u[q]));
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(BAR(C::B_OE + pb));
        }
        const bool fin = W.wait_warp(BAR(C::B_FIN), 0);
#pragma unroll
        for (int q = 0; q < R; ++q) {
            if (!row_ok(q)) continue;
            const float sc = fin ? scale_s[q] : 0.f;
            const int pos = row_pos(q), hq = kvh * p.G + q % p.G, tok = q_start + pos;
#pragma unroll
            for (int cc = 0; cc < C::NDV; ++cc) {
                const int col = cc * 128 + m;
                const float v = o[cc][q] * sc;
                if (p.split_mode) {
                    p.o_part[(((long long)split * p.total_q + tok) * p.Hq + hq) * DV + col] = v;
                } else {
                    uint16_t h;
                    if (p.out_fp16) {
                        const __half x = __float2half_rn(v);
                        h = *reinterpret_cast<const uint16_t *>(&x);
                    } else {
                        const __nv_bfloat16 x = __float2bfloat16_rn(v);
                        h = *reinterpret_cast<const uint16_t *>(&x);
                    }
                    reinterpret_cast<uint16_t *>(p.o)[(long long)b * p.o_sb + (long long)pos * p.o_ss + hq * p.o_sh + col] = h;
                }
            }
        }
    }
    // ------------------------------------------------------------ teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, C::TM_COLS);
    }
}

}  // namespace fa8
