// fa8_launch.h -- internal: typed launchers, one translation unit per head-dim pair so the
// instantiations compile in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa8_decode.cuh"
#include "fa8_kernel.cuh"

namespace fa8 {

template <int D, int DV>
cudaError_t launch_fwd(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                       const CUtensorMap &tv, dim3 grid, cudaStream_t stream);

template <int DV>
cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream);

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
        e = cudaFuncSetAttribute(fwd_kernel<D_, DV_>,                                        \
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                                             smem);                                          \
        if (e != cudaSuccess) return e;                                                      \
        fwd_kernel<D_, DV_><<<grid, kNumThreads, smem, stream>>>(p, tq, tk, tv);             \
        return cudaGetLastError();                                                           \
    }

// Defines launch_decode<D, DV> (the few-rows kernel, dv a multiple of 128).
#define FA8_DEFINE_DECODE(D_, DV_)                                                           \
    template <>                                                                              \
    cudaError_t launch_decode<D_, DV_>(const FwdParams &p, const CUtensorMap &tq,            \
                                       const CUtensorMap &tk, const CUtensorMap &tv,         \
                                       dim3 grid, cudaStream_t stream) {                     \
        constexpr int smem = DecCfg<D_, DV_>::SMEM_BYTES;                                    \
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<D_, DV_>,                         \
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,    \
                                             smem);                                          \
        if (e != cudaSuccess) return e;                                                      \
        decode_kernel<D_, DV_><<<grid, kDecThreads, smem, stream>>>(p, tq, tk, tv);          \
        return cudaGetLastError();                                                           \
    }

}  // namespace fa8
