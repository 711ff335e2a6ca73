// fa8_launch.h -- internal: typed launchers, one translation unit per head-dim pair so the
// instantiations compile in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa8_decode.cuh"
#include "fa8_kernel.cuh"
#include "fa8_prefill.cuh"

namespace fa8 {

template <int D, int DV>
cudaError_t launch_fwd(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, dim3 grid, cudaStream_t stream);

template <int DV>
cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream);

template <int D, int DV>
cudaError_t launch_prefill(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                           const CUtensorMap &tv, dim3 grid, cudaStream_t stream);

// CTAs of decode_kernel<D, DV> resident per SM (shared memory decides).
inline int decode_ctas_per_sm(int D, int DV) {
    switch (D * 1000 + DV) {
        case 128128: return DecCfg<128, 128>::CTAS;
        case 192128: return DecCfg<192, 128>::CTAS;
        case 256256: return DecCfg<256, 256>::CTAS;
        default: return 1;
    }
}

template <int D, int DV>
cudaError_t launch_decode(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                          const CUtensorMap &tv, dim3 grid, cudaStream_t stream);

// fwd_kernel moves registers between its warpgroups with setmaxnreg, which draws on the
// registers the CTA was launched with: a split planned for a launch count the compiler did
// not give would leave setmaxnreg.inc waiting forever.  Its launcher therefore compares the
// compiled count with the planned one once per function and refuses to launch on a
// mismatch.
template <typename K>
inline cudaError_t check_launch_regs(K *kernel, int expected, int *cached) {
    if (*cached < 0) {
        cudaFuncAttributes a;
        const cudaError_t e = cudaFuncGetAttributes(&a, kernel);
        if (e != cudaSuccess) return e;
        *cached = a.numRegs;
    }
    return *cached == expected ? cudaSuccess : cudaErrorInvalidConfiguration;
}

// Launches a forward kernel.  In split mode split_plan_kernel runs just before it on the
// same stream, and the forward grid is launched with programmatic stream serialization so
// that its CTAs start while the plan kernel still runs; they wait for it (griddep_wait)
// only before reading the split cap it writes.
template <typename K>
inline cudaError_t launch_after_plan(K *kernel, const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                                     const CUtensorMap &tv, dim3 grid, int threads, int smem, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3((unsigned)threads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (p.split_mode && p.cap_const <= 0) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, p, tq, tk, tv);
}

// Defines launch_fwd<D, DV>.  Dynamic shared memory above 48 KB needs an opt-in per
// function and device; it is set on every launch (a cheap host call) so that a first
// launch on a new device needs no extra bookkeeping.
#define FA8_DEFINE_FWD(D_, DV_)                                                              \
    template <>                                                                              \
    cudaError_t launch_fwd<D_, DV_>(const FwdParams &p, const CUtensorMap &tq,               \
                                    const CUtensorMap &tk, const CUtensorMap &tv, dim3 grid, \
                                    cudaStream_t stream) {                                   \
        constexpr int smem = Cfg<D_, DV_>::SMEM_BYTES;                                       \
        static int regs = -1;                                                                \
        cudaError_t e = check_launch_regs(fwd_kernel<D_, DV_>, kLaunchRegs, &regs);          \
        if (e != cudaSuccess) return e;                                                      \
        e = cudaFuncSetAttribute(fwd_kernel<D_, DV_>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                 smem);                                                      \
        if (e != cudaSuccess) return e;                                                      \
        return launch_after_plan(fwd_kernel<D_, DV_>, p, tq, tk, tv, grid, kNumThreads, smem, stream); \
    }

// Defines launch_prefill<D, DV> (persistent, one 128-row Q tile per work unit, dv <= 128);
// like fwd_kernel it re-balances registers with setmaxnreg and checks the compiled count.
#define FA8_DEFINE_PREFILL(D_, DV_)                                                          \
    template <>                                                                              \
    cudaError_t launch_prefill<D_, DV_>(const FwdParams &p, const CUtensorMap &tq,           \
                                        const CUtensorMap &tk, const CUtensorMap &tv,        \
                                        dim3 grid, cudaStream_t stream) {                    \
        constexpr int smem = PfCfg<D_, DV_>::SMEM_BYTES;                                     \
        static int regs = -1;                                                                \
        cudaError_t e = check_launch_regs(prefill_kernel<D_, DV_>, kPfLaunchRegs, &regs);    \
        if (e != cudaSuccess) return e;                                                      \
        e = cudaFuncSetAttribute(prefill_kernel<D_, DV_>,                                    \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);         \
        if (e != cudaSuccess) return e;                                                      \
        return launch_after_plan(prefill_kernel<D_, DV_>, p, tq, tk, tv, grid, kPfThreads, smem, stream); \
    }

// The few-rows kernel carrying R rows (see decode_kernel).
template <int D, int DV, int R>
inline cudaError_t launch_decode_rows(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                                      const CUtensorMap &tv, dim3 grid, cudaStream_t stream) {
    constexpr int smem = DecCfg<D, DV>::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, DV, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_after_plan(decode_kernel<D, DV, R>, p, tq, tk, tv, grid, kDecThreads, smem, stream);
}

// Defines launch_decode<D, DV> (the few-rows kernel, dv a multiple of 128): 4 or 8 carried
// rows when a tile's real rows (query positions in the tile x q-heads per kv-head) fit.
#define FA8_DEFINE_DECODE(D_, DV_)                                                           \
    template <>                                                                              \
    cudaError_t launch_decode<D_, DV_>(const FwdParams &p, const CUtensorMap &tq,            \
                                       const CUtensorMap &tk, const CUtensorMap &tv,         \
                                       dim3 grid, cudaStream_t stream) {                     \
        const int rows = (p.Sq < p.pos_per_tile ? p.Sq : p.pos_per_tile) * p.G;              \
        return rows <= 4   ? launch_decode_rows<D_, DV_, 4>(p, tq, tk, tv, grid, stream)     \
               : rows <= 8 ? launch_decode_rows<D_, DV_, 8>(p, tq, tk, tv, grid, stream)     \
                           : launch_decode_rows<D_, DV_, 16>(p, tq, tk, tv, grid, stream);   \
    }

}  // namespace fa8
