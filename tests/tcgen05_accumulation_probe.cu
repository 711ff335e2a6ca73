// Accumulation precision of tcgen05.mma kind::f8f6f4 (E4M3 x E4M3 -> fp32 in TMEM), the
// property that decides whether PV needs two-level accumulation on this hardware (the FP8
// Hopper forward adds each tile's PV to an fp32 O because the FP8 tensor-core accumulator
// there keeps too few bits).
// O (128 x 128, TMEM) is preset to L, then O += P V over 128 keys (4 MMAs of K = 32, all
// accumulating), P from TMEM, V from smem (MN-major, 128-byte swizzle via TMA), exactly as the
// forward kernels issue PV.  Exact fp32 accumulation adds sum_j P_j V_j to L.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdio>
#include <cstdlib>
#include <cmath>
#include <vector>
#include "fa8_kernel.cuh"

using namespace fa8;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn enc;

static void make_map(CUtensorMap *m, void *base, int rows, int cols) {
    cuuint64_t gd[4] = {(cuuint64_t)cols, 1, (cuuint64_t)rows, 1};
    cuuint64_t gs[3] = {(cuuint64_t)cols, (cuuint64_t)cols, (cuuint64_t)cols * rows};
    cuuint32_t bd[4] = {128, 1, 128, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, gd, gs, bd, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) { printf("encode failed %d\n", (int)r); exit(1); }
}

__global__ void __launch_bounds__(128, 1) acc_probe(const __grid_constant__ CUtensorMap tv, const uint8_t *pcodes,
                                                    float init, float *o_out, unsigned *status) {
    extern __shared__ uint8_t raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sV = ptx::smem_u32(sm);
    uint8_t *misc = sm + 128 * 128;
    const uint32_t bar = ptx::smem_u32(misc);
    uint32_t *tslot = (uint32_t *)(misc + 64);
    volatile int *ab = (volatile int *)(misc + 68);
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        ptx::mbar_init(bar, 1);
        ptx::mbar_init(bar + 8, 1);
        *ab = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0) { ptx::tmem_alloc(ptx::smem_u32(tslot), 512); ptx::tmem_relinquish(); }
    ptx::tc_fence_before(); __syncthreads(); ptx::tc_fence_after();
    const uint32_t tmem = *tslot;
    const Waiter W{ab, 1000000000ull, status};
    const uint32_t lb = (uint32_t)(warp * 32) << 16;
    // P codes of row tid -> TMEM columns 128..159; O preset to init in columns 256..383
    uint32_t w[32];
    for (int k = 0; k < 32; ++k) {
        const uint8_t *pc = pcodes + tid * 128 + 4 * k;
        w[k] = (uint32_t)pc[0] | ((uint32_t)pc[1] << 8) | ((uint32_t)pc[2] << 16) | ((uint32_t)pc[3] << 24);
    }
    ptx::tmem_st32(tmem + lb + 128, w);
    for (int j = 0; j < 4; ++j) {
        uint32_t v[32];
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(init);
        ptx::tmem_st32(tmem + lb + 256 + 32 * j, v);
    }
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (tid == 0) {
        ptx::mbar_arrive_expect_tx(bar, 128 * 128);
        ptx::tma_load_4d(sV, &tv, bar, 0, 0, 0, 0);
        W.wait(bar, 0);
        ptx::tc_fence_after();
        constexpr uint32_t idp = idesc_e4m3(128, 128, true);
        for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = sdesc(sV + kk * 32 * 128, 128 * 128, 8 * 128, swz_layout(128));
            ptx::mma_f8_ts(tmem + 256, tmem + 128 + kk * 8, bd, idp, 1u);
        }
        ptx::tc_commit(bar + 8);
        W.wait(bar + 8, 0);
    }
    __syncthreads();
    ptx::tc_fence_after();
    for (int j = 0; j < 4; ++j) {
        uint32_t u[32];
        ptx::tmem_ld32(tmem + lb + 256 + 32 * j, u);
        ptx::tmem_wait_ld();
        ptx::reg_fence32(u);
        for (int i = 0; i < 32; ++i) o_out[tid * 128 + 32 * j + i] = __uint_as_float(u[i]);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) { ptx::tc_fence_after(); ptx::tmem_dealloc(tmem, 512); }
}

static double dec(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

// p0/v0: codes of key 0 (P of every row, V of every column); p/v: codes of keys 1..127
static void run(const char *name, float init, uint8_t p0, uint8_t p, uint8_t v0, uint8_t v) {
    std::vector<uint8_t> pc(128 * 128), vv(128 * 128);
    for (int r = 0; r < 128; ++r)
        for (int j = 0; j < 128; ++j) pc[r * 128 + j] = j == 0 ? p0 : p;
    for (int j = 0; j < 128; ++j)
        for (int c = 0; c < 128; ++c) vv[j * 128 + c] = j == 0 ? v0 : v;
    uint8_t *dp, *dv; float *dO; unsigned *dst;
    cudaMalloc(&dp, pc.size()); cudaMalloc(&dv, vv.size()); cudaMalloc(&dO, 128 * 128 * 4); cudaMalloc(&dst, 4);
    cudaMemset(dst, 0, 4);
    cudaMemcpy(dp, pc.data(), pc.size(), cudaMemcpyHostToDevice);
    cudaMemcpy(dv, vv.data(), vv.size(), cudaMemcpyHostToDevice);
    CUtensorMap tv;
    make_map(&tv, dv, 128, 128);
    const int smem = 128 * 128 + 1024 + 1024;
    cudaFuncSetAttribute(acc_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    acc_probe<<<1, 128, smem>>>(tv, dp, init, dO, dst);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) { printf("%s: CUDA error %s\n", name, cudaGetErrorString(e)); exit(2); }
    unsigned st; cudaMemcpy(&st, dst, 4, cudaMemcpyDeviceToHost);
    std::vector<float> O(128 * 128);
    cudaMemcpy(O.data(), dO, O.size() * 4, cudaMemcpyDeviceToHost);
    const double add = dec(p0) * dec(v0) + 127.0 * dec(p) * dec(v);
    const double exact = (double)init + add;
    const float fp32_once = (float)exact;  // the sum rounded once to fp32
    double lo = 1e300, hi = -1e300;
    for (float x : O) { lo = fmin(lo, x); hi = fmax(hi, x); }
    // one line per case: name | L | exact addend | min O | max O | fp32(L + addend) | status
    printf("%s|%.9g|%.12g|%.12g|%.12g|%.12g|%u\n", name, (double)init, add, lo, hi, (double)fp32_once, st);
    cudaFree(dp); cudaFree(dv); cudaFree(dO); cudaFree(dst);
}

int main() {
    void *p = nullptr; cudaDriverEntryPointQueryResult qr;
    cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr);
    enc = (EncodeTiledFn)p;
    const uint8_t ONE = 0x38, TINY = 0x01 /* 2^-9 */, BIG = 0x78 /* 256 */, HALF = 0x30;
    for (float L : {0.f, 16.f, 256.f, 4096.f, 65536.f, 1048576.f})
        run("128 x (1 * 2^-9) onto L", L, ONE, ONE, TINY, TINY);
    for (float L : {0.f, 4096.f, 65536.f})
        run("128 x (1 * 0.5) onto L", L, ONE, ONE, HALF, HALF);
    run("256*1 + 127 x (1 * 2^-9), one MMA set", 0.f, BIG, ONE, ONE, TINY);
    run("256*256 + 127 x (1 * 2^-9)", 0.f, BIG, ONE, BIG, TINY);
    return 0;
}
