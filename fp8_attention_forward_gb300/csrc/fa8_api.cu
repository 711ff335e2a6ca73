// fa8_api.cu -- host side of the C ABI declared in include/fa8.h: argument validation,
// the launch planner (tile packing, grid, split count; from shapes and the SM count
// only), TMA descriptor encoding, and the launches of the forward and combine kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <numeric>
#include <string>

#include "fa8.h"
#include "fa8_launch.h"

// Device status word of the library (timeouts, out-of-range block-table entries),
// one per device that loads the library; read and cleared by fa8_check().
__device__ unsigned int g_fa8_status_word;

// Split-KV partials of fa8_fwd_static_scratch: one array per device that loads the
// library, shared by every call (see the header for the ordering rule).
static __device__ __align__(256) unsigned char g_fa8_static_scratch[FA8_STATIC_SCRATCH_BYTES];

namespace fa8 {

__global__ void split_plan_kernel(const __grid_constant__ FwdParams p) {
    ptx::griddep_launch_dependents();  // the forward kernel's CTAs may launch meanwhile
    const int cap = split_tile_cap(p.B, p.Hkv, p.kv_mode, p.Sk, p.cu_k, p.q_varlen, p.Sq, p.cu_q, p.pos_per_tile,
                                   p.num_splits, p.slots);
    if (threadIdx.x == 0) *p.split_cap = cap;
}

__global__ void wait_probe_kernel(unsigned long long timeout_ns, unsigned int *status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bar), 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const Waiter w{&abort_flag, timeout_ns, status};
        w.wait(ptx::smem_u32(&bar), 0);  // nothing ever arrives on this barrier
    }
}

#define FA8_DEFINE_COMBINE(DV_)                                                             \
    template <>                                                                             \
    cudaError_t launch_combine<DV_>(const CombineParams &p, cudaStream_t s) {               \
        const long long rows = (long long)p.total_q * p.Hq;                                 \
        const long long per_cta = 8 / p.wpr;                                                \
        const unsigned blocks = (unsigned)((rows + per_cta - 1) / per_cta);                 \
        /* programmatic dependent launch: the merge's CTAs start while the forward        \
           kernel drains and wait for it (griddep_wait) before reading anything */        \
        cudaLaunchConfig_t cfg = {};                                                        \
        cfg.gridDim = dim3(blocks, 1, 1);                                                   \
        cfg.blockDim = dim3(256, 1, 1);                                                     \
        cfg.stream = s;                                                                     \
        cudaLaunchAttribute attr[1];                                                        \
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;                    \
        attr[0].val.programmaticStreamSerializationAllowed = 1;                             \
        cfg.attrs = attr;                                                                   \
        cfg.numAttrs = 1;                                                                   \
        return cudaLaunchKernelEx(&cfg, combine_kernel<DV_>, p);                            \
    }
FA8_DEFINE_COMBINE(64)
FA8_DEFINE_COMBINE(96)
FA8_DEFINE_COMBINE(128)
FA8_DEFINE_COMBINE(192)
FA8_DEFINE_COMBINE(256)

}  // namespace fa8

namespace {

thread_local std::string g_last_error;
// Process-wide settings, written by the setters and read once per fa8_fwd call; atomics, so
// that a setter on one host thread and a forward call on another never race.
std::atomic<unsigned long long> g_timeout_ns{2000000000ull};
std::atomic<unsigned long long *> g_trace{nullptr};  // pipeline trace buffer (FA8_TRACE builds)
std::atomic<bool> g_decode_kernel{true};             // few-rows shapes go to decode_kernel

fa8_status fail(fa8_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

fa8_status cuda_fail(cudaError_t e, const char *what) {
    return fail(FA8_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------- per-device state
struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    unsigned int *status = nullptr;
};
std::mutex g_mu;
DeviceState g_dev[64];

fa8_status device_state(DeviceState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(FA8_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_fa8_status_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
        d.status = static_cast<unsigned int *>(ptr);
        d.ready = true;
    }
    *out = &d;
    return FA8_SUCCESS;
}

// Device address of g_fa8_static_scratch on the current device, looked up on the first
// request for each device.
void *g_scratch_ptr[64];

fa8_status static_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(FA8_ERR_CUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_fa8_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        if (!ptr) return fail(FA8_ERR_CUDA, "static scratch has no device address");
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return FA8_SUCCESS;
}

// ---------------------------------------------------------------- TMA descriptor encoding
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode(fa8_status *st) {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!fn) *st = fail(FA8_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(err));
    return fn;
}

CUtensorMapSwizzle swizzle_for(int chunk_bytes) {
    return chunk_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                              : (chunk_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

// 4-D byte tensor {inner, d1, d2, d3} with byte strides {s1, s2, s3}, box {b0, b1, b2, 1}.
fa8_status encode4(CUtensorMap *m, void *base, const uint64_t dims[4], const uint64_t strides[3],
                   const uint32_t box[4], int chunk_bytes, CUtensorMapL2promotion l2) {
    fa8_status st = FA8_SUCCESS;
    EncodeTiledFn fn = get_encode(&st);
    if (!fn) return st;
    cuuint64_t gd[4] = {dims[0], dims[1], dims[2], dims[3]};
    cuuint64_t gs[3] = {strides[0], strides[1], strides[2]};
    cuuint32_t bd[4] = {box[0], box[1], box[2], box[3]};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, gd, gs, bd, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle_for(chunk_bytes), l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(FA8_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) dims {%llu,%llu,%llu,%llu} strides {%llu,%llu,%llu}",
                    (int)r, (unsigned long long)dims[0], (unsigned long long)dims[1], (unsigned long long)dims[2],
                    (unsigned long long)dims[3], (unsigned long long)strides[0], (unsigned long long)strides[1],
                    (unsigned long long)strides[2]);
    return FA8_SUCCESS;
}

int chunk_of(int d) { return (d % 128 == 0) ? 128 : ((d % 64 == 0) ? 64 : 32); }

bool supported_dims(int d, int dv) {
    return (d == 64 && dv == 64) || (d == 96 && dv == 96) || (d == 128 && dv == 128) || (d == 192 && dv == 128) ||
           (d == 192 && dv == 192) || (d == 256 && dv == 256);
}

// ---------------------------------------------------------------- planner
struct Plan {
    int D = 0, DV = 0, B = 0, Hq = 0, Hkv = 0, G = 0, P = 0, rows_per_tile = 0;
    int q_varlen = 0, kv_mode = 0;
    int Sq = 0, Sk = 0, total_q = 0, total_k = 0;
    int num_pages = 0, page_size = 0, max_pages = 0, box_n = 0;
    long long num_slots = 0;
    int mblocks_per_batch = 0;
    int splits = 1;
    long long max_lk = 0;
    size_t ws_bytes = 0;
    int decode = 0;  // launch decode_kernel (at most 16 rows per kv-head, dv % 128 == 0)
    int prefill = 0;  // launch prefill_kernel (persistent, one 128-row Q tile per work unit, dv <= 128)
    long long base_units = 0;  // (tile of query rows, kv-head) pairs, before splitting
    long long units = 0;       // (slot, kv-head, split) work units
    int cap = 0;  // split cap chosen on the host (dense K/V, batched q); 0: as the launch decides
};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The split cap for dense K/V with batched q: every request has the same key and query
// counts, so the host knows all that split_plan_kernel would read.  The same model as
// fa8::split_tile_cap (fixed cost F per unit, tail weight beta, candidates 2, 4, ..., 512 and
// the finest cap the launch allows), plus one candidate the device does not try: the finest
// cap whose units all run in one wave (the powers of two can miss it by up to 2x, leaving SMs
// idle for the whole launch).
int uniform_split_cap(int B, int Hkv, int Sk, int Sq, int P, int n, int slots) {
    const long long t = Sk > 0 ? (Sk + 127) / 128 : 0;
    const long long mb = Sq > 0 ? (Sq + P - 1) / P : 0;
    const int t_fine = (int)std::max<long long>(2, (t + n - 1) / n);
    const float tiles = (float)(B * t * mb);
    auto cost = [&](long long T) {
        const float units = (float)((long long)B * mb * ((t + T - 1) / T)) * (float)Hkv;
        const float tail = fa8::kFixedTiles + (float)std::min<long long>(T, t);
        return units <= (float)slots ? tail
                                     : (fa8::kFixedTiles * units + tiles * (float)Hkv) * (1.f / (float)slots) +
                                           fa8::kTailWeight * tail;
    };
    int best_cap = t_fine;
    float best = 3.0e38f;
    for (int c = 0; c < 10; ++c) {
        const int T = c < 9 ? (2 << c) : t_fine;
        if (T < t_fine) continue;
        const float m = cost(T);
        if (m < best) {
            best = m;
            best_cap = T;
        }
    }
    const long long per_split = (long long)B * mb * Hkv;  // units per split of every request
    if (t > 0 && per_split > 0 && per_split <= slots) {
        const long long k = slots / per_split;  // splits per request that still fit one wave
        const long long T = std::max<long long>(t_fine, (t + k - 1) / k);
        if (cost(T) < best) best_cap = (int)T;
    }
    return best_cap;
}

fa8_status check_int_vec(const fa8_tensor *t, const char *name, long long n) {
    if (t->dtype != FA8_DTYPE_I32) return fail(FA8_ERR_INVALID_ARG, "%s must be int32", name);
    if (t->ndim != 1 || t->shape[0] != n || (n > 1 && t->stride[0] != 1))
        return fail(FA8_ERR_INVALID_ARG, "%s must be a contiguous 1-D tensor of %lld entries", name, n);
    if (!t->data) return fail(FA8_ERR_INVALID_ARG, "%s has a null data pointer", name);
    return FA8_SUCCESS;
}

// Q/K/V payload: last dim contiguous, other strides multiples of 16 bytes, 16-byte base.
fa8_status check_payload(const fa8_tensor *t, const char *name) {
    if (t->ndim < 3 || t->ndim > 4) return fail(FA8_ERR_INVALID_ARG, "%s must have 3 or 4 dims", name);
    if (t->stride[t->ndim - 1] != 1) return fail(FA8_ERR_INVALID_ARG, "%s: last dim must be contiguous", name);
    for (int i = 0; i < t->ndim - 1; ++i) {
        if (t->shape[i] < 0) return fail(FA8_ERR_INVALID_ARG, "%s: negative extent", name);
        if (t->stride[i] <= 0 || t->stride[i] % 16 != 0)
            return fail(FA8_ERR_INVALID_ARG, "%s: stride[%d]=%lld must be a positive multiple of 16 bytes", name, i,
                        (long long)t->stride[i]);
    }
    if (t->shape[t->ndim - 1] < 0) return fail(FA8_ERR_INVALID_ARG, "%s: negative extent", name);
    if (!aligned16(t->data)) return fail(FA8_ERR_INVALID_ARG, "%s: data must be 16-byte aligned", name);
    return FA8_SUCCESS;
}

fa8_status make_plan(const fa8_tensor *q, const fa8_tensor *k, const fa8_tensor *v, const fa8_tensor *cu_q,
                     const fa8_tensor *cu_k, const fa8_tensor *bt, int page_size, int num_splits, int sm_count,
                     bool use_decode, Plan *pl) {
    if (!q || !k || !v) return fail(FA8_ERR_INVALID_ARG, "q, k and v are required");
    for (const fa8_tensor *t : {q, k, v}) {
        if (t->dtype == FA8_DTYPE_E5M2) return fail(FA8_ERR_UNSUPPORTED, "E5M2 inputs are not supported (E4M3 only)");
    }
    if (q->dtype != FA8_DTYPE_E4M3 || k->dtype != FA8_DTYPE_E4M3 || v->dtype != FA8_DTYPE_E4M3) {
        if (q->dtype == k->dtype && k->dtype == v->dtype)
            return fail(FA8_ERR_UNSUPPORTED, "q/k/v must be E4M3");
        return fail(FA8_ERR_UNSUPPORTED, "mixed q/k/v dtypes are not supported (all must be E4M3)");
    }
    fa8_status st;
    if ((st = check_payload(q, "q")) || (st = check_payload(k, "k")) || (st = check_payload(v, "v"))) return st;
    if (num_splits < 0) return fail(FA8_ERR_INVALID_ARG, "num_splits must be >= 0");

    Plan p;
    p.D = (int)q->shape[q->ndim - 1];
    p.Hq = (int)q->shape[q->ndim - 2];
    p.DV = (int)v->shape[v->ndim - 1];
    if (k->shape[k->ndim - 1] != p.D) return fail(FA8_ERR_INVALID_ARG, "k head dim %lld != q head dim %d", (long long)k->shape[k->ndim - 1], p.D);
    if (!supported_dims(p.D, p.DV))
        return fail(FA8_ERR_UNSUPPORTED, "(d, dv) = (%d, %d) is not supported", p.D, p.DV);
    if (k->ndim != v->ndim) return fail(FA8_ERR_INVALID_ARG, "k and v must have the same rank");
    for (int i = 0; i < k->ndim - 1; ++i)
        if (k->shape[i] != v->shape[i]) return fail(FA8_ERR_INVALID_ARG, "k and v leading shapes differ at dim %d", i);
    p.Hkv = (int)k->shape[k->ndim - 2];
    if (p.Hq <= 0 || p.Hkv <= 0 || p.Hq % p.Hkv != 0)
        return fail(FA8_ERR_INVALID_ARG, "q heads (%d) must be a positive multiple of kv heads (%d)", p.Hq, p.Hkv);
    p.G = p.Hq / p.Hkv;
    if (p.G > 128) return fail(FA8_ERR_UNSUPPORTED, "more than 128 q-heads per kv-head (%d)", p.G);
    p.P = 128 / p.G;
    p.rows_per_tile = p.P * p.G;
    // Decode shapes: batched q whose rows per kv-head (Sq x G) fit one 16-row tile.
    // (Its launch puts the kv-heads and then the requests on grid x and the splits on grid
    // y, so that the CTAs of one request, which read neighbouring bytes of the same pages,
    // run together.)
    if (use_decode && q->ndim == 4 && p.DV % 128 == 0 && 16 % p.G == 0 && q->shape[1] * p.G <= 16 &&
        q->shape[1] > 0 && (long long)q->shape[0] * p.Hkv <= 0x7fffffffLL) {
        p.decode = 1;
        p.P = 16 / p.G;
        p.rows_per_tile = 16;
    } else if (p.DV <= 128) {
        // the persistent prefill kernel: one work unit per 128-row Q tile (P positions x G heads)
        p.prefill = 1;
    }

    // ---- Q layout
    if (q->ndim == 4) {
        if (cu_q) return fail(FA8_ERR_INVALID_ARG, "cu_seqlens_q is only valid with a 3-D (varlen) q");
        p.q_varlen = 0;
        p.B = (int)q->shape[0];
        p.Sq = (int)q->shape[1];
        p.total_q = p.B * p.Sq;
    } else {
        if (!cu_q) return fail(FA8_ERR_INVALID_ARG, "a 3-D (varlen) q needs cu_seqlens_q");
        p.q_varlen = 1;
        if (cu_q->ndim != 1 || cu_q->shape[0] < 2) return fail(FA8_ERR_INVALID_ARG, "cu_seqlens_q must have B+1 >= 2 entries");
        p.B = (int)cu_q->shape[0] - 1;
        p.total_q = (int)q->shape[0];
        p.Sq = 0;
    }
    if (cu_q && (st = check_int_vec(cu_q, "cu_seqlens_q", p.B + 1))) return st;
    if (p.B <= 0) return fail(FA8_ERR_INVALID_ARG, "batch must be >= 1");

    // ---- K/V layout
    if (bt) {
        p.kv_mode = 2;
        if (k->ndim != 4) return fail(FA8_ERR_INVALID_ARG, "paged k must be (num_pages, page_size, Hkv, d)");
        if (!cu_k) return fail(FA8_ERR_INVALID_ARG, "paged K/V needs cu_seqlens_k for the per-request key counts");
        if (bt->dtype != FA8_DTYPE_I32 || bt->ndim != 2) return fail(FA8_ERR_INVALID_ARG, "block_table must be a 2-D int32 tensor");
        if (bt->shape[0] != p.B) return fail(FA8_ERR_INVALID_ARG, "block_table rows (%lld) != batch (%d)", (long long)bt->shape[0], p.B);
        if (bt->shape[1] < 1 || (bt->shape[1] > 1 && bt->stride[1] != 1) || bt->stride[0] < 0)
            return fail(FA8_ERR_INVALID_ARG, "block_table rows must be contiguous (stride(1) == 1)");
        if (!bt->data) return fail(FA8_ERR_INVALID_ARG, "block_table has a null data pointer");
        if (page_size != (int)k->shape[1]) return fail(FA8_ERR_INVALID_ARG, "page_size (%d) != k.shape[1] (%lld)", page_size, (long long)k->shape[1]);
        if (page_size <= 0 || page_size % 8 != 0) return fail(FA8_ERR_UNSUPPORTED, "page_size must be a positive multiple of 8");
        p.page_size = page_size;
        p.num_pages = (int)k->shape[0];
        p.max_pages = (int)bt->shape[1];
        p.box_n = std::gcd(page_size, 128);
        p.max_lk = (long long)p.max_pages * page_size;
    } else if (k->ndim == 4) {
        p.kv_mode = 0;
        if (cu_k) return fail(FA8_ERR_INVALID_ARG, "cu_seqlens_k is only valid with varlen (3-D) or paged k");
        if (k->shape[0] != p.B) return fail(FA8_ERR_INVALID_ARG, "k batch (%lld) != q batch (%d)", (long long)k->shape[0], p.B);
        p.Sk = (int)k->shape[1];
        p.max_lk = p.Sk;
    } else {
        p.kv_mode = 1;
        if (!cu_k) return fail(FA8_ERR_INVALID_ARG, "a 3-D (varlen) k needs cu_seqlens_k");
        p.total_k = (int)k->shape[0];
        p.max_lk = p.total_k;
    }
    if (cu_k && (st = check_int_vec(cu_k, "cu_seqlens_k", p.B + 1))) return st;

    // ---- grid and splits (shapes and SM count only: safe under graph capture)
    const long long pos_per_slot = p.P;
    if (p.q_varlen) {
        p.num_slots = ((long long)p.total_q + pos_per_slot - 1) / pos_per_slot + p.B;
    } else {
        p.mblocks_per_batch = (int)((p.Sq + pos_per_slot - 1) / pos_per_slot);
        p.num_slots = (long long)p.B * p.mblocks_per_batch;
    }
    if (p.num_slots > 0x7fffffffLL) return fail(FA8_ERR_UNSUPPORTED, "problem too large for the grid");
    const long long real_mblocks =
        p.q_varlen ? ((long long)p.total_q + pos_per_slot - 1) / pos_per_slot : p.num_slots;
    const long long base_ctas = std::max(1LL, real_mblocks * p.Hkv);
    p.base_units = base_ctas;
    const int max_tiles = (int)std::max(1LL, (p.max_lk + 127) / 128);
    int splits;
    if (num_splits == 0) {
        // enough CTAs to fill the SMs several times over, never fewer than two tiles a split
        // (the decode kernel, cheaper per CTA, may split up to 128 ways)
        const long long target = 8LL * sm_count;
        const long long cap = p.decode ? 128 : 64;
        // few (tile, kv-head) pairs: as many splits as fit in one wave of CTAs.  With every
        // launched split in one wave the finest cap is the model's answer whatever the key
        // counts (split_tile_cap), so the launch passes it and runs no plan kernel.
        const long long one_wave = (long long)(p.decode ? fa8::decode_ctas_per_sm(p.D, p.DV) : 1) * sm_count;
        if (base_ctas >= target || max_tiles < 4) {
            splits = 1;
        } else {
            long long s = 2 * base_ctas <= one_wave ? one_wave / base_ctas : (target + base_ctas - 1) / base_ctas;
            s = std::min<long long>(s, max_tiles / 2);
            s = std::min<long long>(s, cap);
            splits = (int)std::max(1LL, s);
        }
    } else {
        splits = std::min(num_splits, max_tiles);
    }
    // Dense K/V with batched q: every request has the same key and query counts, so the host
    // can choose the split cap itself (uniform_split_cap) instead of a plan kernel, and with
    // the heuristic's split count launch only the splits that run.
    if (splits > 1 && p.kv_mode == 0 && !p.q_varlen && p.Sk > 0) {
        const int per_sm = p.decode ? fa8::decode_ctas_per_sm(p.D, p.DV) : 1;
        const int slots = per_sm * sm_count;
        if (base_ctas * splits > (long long)slots) {
            p.cap = uniform_split_cap(p.B, p.Hkv, p.Sk, p.Sq, p.P, splits, slots);
            if (num_splits == 0) {
                const long long t = (p.Sk + 127) / 128;
                splits = (int)std::max<long long>(1, std::min<long long>(splits, (t + p.cap - 1) / p.cap));
            }
        }
    }
    if ((long long)splits * p.Hkv > 65535) return fail(FA8_ERR_UNSUPPORTED, "kv_heads x splits exceeds the grid limit");
    p.splits = splits;
    p.units = p.num_slots * p.Hkv * splits;
    if (p.prefill && p.units > 0x7fffffffLL) return fail(FA8_ERR_UNSUPPORTED, "problem too large for the unit list");
    if (splits > 1 && p.total_q > 0) {
        // fp32 O and LSE partials, then 256 bytes where the forward kernel records the split
        // cap it chose for the combine kernel
        const size_t rows = (size_t)p.total_q * p.Hq * splits;
        const size_t o_bytes = (rows * p.DV * sizeof(float) + 255) & ~(size_t)255;
        p.ws_bytes = o_bytes + ((rows * sizeof(float) + 255) & ~(size_t)255) + 256;
    }
    *pl = p;
    return FA8_SUCCESS;
}

fa8_status check_descale(const fa8_tensor *t, const char *name, const Plan &p, const float **ptr, long long *sb,
                         long long *sh) {
    *ptr = nullptr;
    *sb = *sh = 0;
    if (!t) return FA8_SUCCESS;
    if (t->dtype != FA8_DTYPE_F32) return fail(FA8_ERR_INVALID_ARG, "%s must be fp32", name);
    if (!t->data) return fail(FA8_ERR_INVALID_ARG, "%s has a null data pointer", name);
    if (t->ndim == 0) {
    } else if (t->ndim == 2 && t->shape[0] == p.B && t->shape[1] == p.Hkv) {
        *sb = t->stride[0];
        *sh = t->stride[1];
    } else {
        return fail(FA8_ERR_INVALID_ARG, "%s must be 0-d or (batch=%d, kv_heads=%d)", name, p.B, p.Hkv);
    }
    *ptr = static_cast<const float *>(t->data);
    return FA8_SUCCESS;
}

}  // namespace

extern "C" {

int fa8_version(void) { return FA8_VERSION; }

const char *fa8_last_error(void) { return g_last_error.c_str(); }

const char *fa8_status_string(fa8_status s) {
    switch (s) {
        case FA8_SUCCESS: return "success";
        case FA8_ERR_INVALID_ARG: return "invalid argument";
        case FA8_ERR_UNSUPPORTED: return "unsupported";
        case FA8_ERR_WORKSPACE: return "workspace missing or too small";
        case FA8_ERR_CUDA: return "CUDA error";
        case FA8_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case FA8_ERR_DEVICE_BOUNDS: return "device index out of range";
    }
    return "unknown status";
}

fa8_status fa8_set_decode_kernel(int enable) {
    g_last_error.clear();
    if (enable != 0 && enable != 1) return fail(FA8_ERR_INVALID_ARG, "enable must be 0 or 1");
    g_decode_kernel.store(enable == 1);
    return FA8_SUCCESS;
}

fa8_status fa8_set_wait_timeout_ns(uint64_t ns) {
    if (ns < 100000ull) return fail(FA8_ERR_INVALID_ARG, "timeout must be >= 1e5 ns");
    g_timeout_ns.store(ns);
    return FA8_SUCCESS;
}

fa8_status fa8_fwd_plan(const fa8_tensor *q, const fa8_tensor *k, const fa8_tensor *v,
                        const fa8_tensor *cu_seqlens_q, const fa8_tensor *cu_seqlens_k,
                        const fa8_tensor *block_table, int page_size, int num_splits, int sm_count,
                        int *splits_out, size_t *bytes_out, int64_t *grid_out) {
    g_last_error.clear();
    if (sm_count <= 0) return fail(FA8_ERR_INVALID_ARG, "sm_count must be positive");
    Plan pl;
    fa8_status st = make_plan(q, k, v, cu_seqlens_q, cu_seqlens_k, block_table, page_size, num_splits, sm_count,
                              g_decode_kernel.load(), &pl);
    if (st) return st;
    if (splits_out) *splits_out = pl.splits;
    if (bytes_out) *bytes_out = pl.ws_bytes;
    if (grid_out) {
        grid_out[0] = pl.num_slots;
        grid_out[1] = (int64_t)pl.Hkv * pl.splits;
    }
    return FA8_SUCCESS;
}

fa8_status fa8_fwd_workspace_size(const fa8_tensor *q, const fa8_tensor *k, const fa8_tensor *v,
                                  const fa8_tensor *cu_seqlens_q, const fa8_tensor *cu_seqlens_k,
                                  const fa8_tensor *block_table, int page_size, int num_splits, int *splits_out,
                                  size_t *bytes_out) {
    g_last_error.clear();
    Plan pl;
    const bool use_decode = g_decode_kernel.load();
    fa8_status st =
        make_plan(q, k, v, cu_seqlens_q, cu_seqlens_k, block_table, page_size, num_splits, 1, use_decode, &pl);
    if (st) return st;
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds))) return st;
    st = make_plan(q, k, v, cu_seqlens_q, cu_seqlens_k, block_table, page_size, num_splits, ds->sm_count, use_decode,
                   &pl);
    if (st) return st;
    if (splits_out) *splits_out = pl.splits;
    if (bytes_out) *bytes_out = pl.ws_bytes;
    return FA8_SUCCESS;
}

fa8_status fa8_check(void *stream) {
    g_last_error.clear();
    DeviceState *ds = nullptr;
    fa8_status st = device_state(&ds);
    if (st) return st;
    // everything on the caller's stream: the read is ordered after the work enqueued there,
    // and no other stream is waited for
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned int word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, ds->status, sizeof(word), cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    if (word) {
        e = cudaMemsetAsync(ds->status, 0, sizeof(unsigned int), s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device status word");
    }
    if (word & fa8::kStatusTimeout) return fail(FA8_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait");
    if (word & fa8::kStatusBounds) return fail(FA8_ERR_DEVICE_BOUNDS, "a kernel saw an out-of-range block-table entry or length");
    return FA8_SUCCESS;
}

fa8_status fa8_debug_set_trace_buffer(void *device_buffer, size_t bytes) {
    g_last_error.clear();
#ifdef FA8_TRACE
    const size_t need = sizeof(unsigned long long) * fa8::kTraceCtas * fa8::kTraceEvents * fa8::kTraceTiles;
    if (device_buffer && bytes < need) return fail(FA8_ERR_INVALID_ARG, "trace buffer needs %zu bytes", need);
    g_trace.store(static_cast<unsigned long long *>(device_buffer));
    return FA8_SUCCESS;
#else
    (void)device_buffer;
    (void)bytes;
    return fail(FA8_ERR_UNSUPPORTED, "library built without FA8_TRACE");
#endif
}

fa8_status fa8_debug_wait_probe(void *stream) {
    g_last_error.clear();
    DeviceState *ds = nullptr;
    fa8_status st = device_state(&ds);
    if (st) return st;
    fa8::wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(g_timeout_ns.load(), ds->status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "wait probe launch");
    return fa8_check(stream);
}

fa8_status fa8_fwd(const fa8_tensor *q, const fa8_tensor *k, const fa8_tensor *v, const fa8_tensor *descale_q,
                   const fa8_tensor *descale_k, const fa8_tensor *descale_v, fa8_tensor *out, fa8_tensor *lse,
                   const fa8_tensor *cu_seqlens_q, const fa8_tensor *cu_seqlens_k, const fa8_tensor *block_table,
                   int page_size, int causal, int window_left, const fa8_tensor *sink, float softmax_scale,
                   int num_splits, void *workspace, size_t workspace_bytes, void *stream) {
    g_last_error.clear();
    Plan pl;
    // the settings are read once, so one call sees one consistent set of them
    const bool use_decode = g_decode_kernel.load();
    const unsigned long long timeout_ns = g_timeout_ns.load();
    unsigned long long *const trace = g_trace.load();
    // shape validation first (host only), then the device-dependent plan
    fa8_status st =
        make_plan(q, k, v, cu_seqlens_q, cu_seqlens_k, block_table, page_size, num_splits, 1, use_decode, &pl);
    if (st) return st;

    // ---- output
    if (!out || !out->data) return fail(FA8_ERR_INVALID_ARG, "out is required");
    if (out->dtype != FA8_DTYPE_BF16 && out->dtype != FA8_DTYPE_F16)
        return fail(FA8_ERR_INVALID_ARG, "out must be bf16 or fp16");
    if (out->ndim != q->ndim) return fail(FA8_ERR_INVALID_ARG, "out must have q's rank");
    for (int i = 0; i < q->ndim - 1; ++i)
        if (out->shape[i] != q->shape[i]) return fail(FA8_ERR_INVALID_ARG, "out shape differs from q at dim %d", i);
    if (out->shape[out->ndim - 1] != pl.DV) return fail(FA8_ERR_INVALID_ARG, "out last dim must be dv=%d", pl.DV);
    if (out->stride[out->ndim - 1] != 1) return fail(FA8_ERR_INVALID_ARG, "out: last dim must be contiguous");
    for (int i = 0; i < out->ndim - 1; ++i)
        if (out->stride[i] % 8 != 0) return fail(FA8_ERR_INVALID_ARG, "out strides must be multiples of 8 elements");
    if (!aligned16(out->data)) return fail(FA8_ERR_INVALID_ARG, "out must be 16-byte aligned");
    long long o_sb = 0, o_ss, o_sh;
    if (pl.q_varlen) {
        o_ss = out->stride[0];
        o_sh = out->stride[1];
    } else {
        o_sb = out->stride[0];
        o_ss = out->stride[1];
        o_sh = out->stride[2];
    }
    // ---- lse
    long long l_sb = 0, l_sh = 0, l_ss = 0;
    if (lse) {
        if (lse->dtype != FA8_DTYPE_F32 || !lse->data) return fail(FA8_ERR_INVALID_ARG, "lse must be fp32");
        if (pl.q_varlen) {
            if (lse->ndim != 2 || lse->shape[0] != pl.Hq || lse->shape[1] != pl.total_q)
                return fail(FA8_ERR_INVALID_ARG, "varlen lse must be (Hq, total_q)");
            l_sh = lse->stride[0];
            l_ss = lse->stride[1];
        } else {
            if (lse->ndim != 3 || lse->shape[0] != pl.B || lse->shape[1] != pl.Hq || lse->shape[2] != pl.Sq)
                return fail(FA8_ERR_INVALID_ARG, "lse must be (B, Hq, Sq)");
            l_sb = lse->stride[0];
            l_sh = lse->stride[1];
            l_ss = lse->stride[2];
        }
    }
    // ---- descales, sink, flags
    fa8::FwdParams p;
    memset(&p, 0, sizeof(p));
    if ((st = check_descale(descale_q, "descale_q", pl, &p.dq, &p.dq_sb, &p.dq_sh)) ||
        (st = check_descale(descale_k, "descale_k", pl, &p.dk, &p.dk_sb, &p.dk_sh)) ||
        (st = check_descale(descale_v, "descale_v", pl, &p.dv, &p.dv_sb, &p.dv_sh)))
        return st;
    if (sink) {
        if (sink->dtype != FA8_DTYPE_F32 || sink->ndim != 1 || sink->shape[0] != pl.Hq ||
            (pl.Hq > 1 && sink->stride[0] != 1) || !sink->data)
            return fail(FA8_ERR_INVALID_ARG, "sink must be a contiguous fp32 (Hq,) tensor");
        p.sink = static_cast<const float *>(sink->data);
    }
    if (causal != 0 && causal != 1) return fail(FA8_ERR_INVALID_ARG, "causal must be 0 or 1");
    if (window_left < -1) return fail(FA8_ERR_INVALID_ARG, "window_left must be -1 or >= 0");
    if (!std::isfinite(softmax_scale)) return fail(FA8_ERR_INVALID_ARG, "softmax_scale must be finite");
    if (softmax_scale <= 0.f) softmax_scale = 1.0f / std::sqrt((float)pl.D);
    // ---- device-dependent plan (split count from the SM count)
    DeviceState *ds = nullptr;
    if ((st = device_state(&ds))) return st;
    st = make_plan(q, k, v, cu_seqlens_q, cu_seqlens_k, block_table, page_size, num_splits, ds->sm_count, use_decode,
                   &pl);
    if (st) return st;
    if (pl.splits > 1) {
        if (!workspace || workspace_bytes < pl.ws_bytes)
            return fail(FA8_ERR_WORKSPACE, "split-KV (%d splits) needs %zu bytes of workspace, got %zu", pl.splits,
                        pl.ws_bytes, workspace ? workspace_bytes : (size_t)0);
        if (!aligned16(workspace)) return fail(FA8_ERR_WORKSPACE, "workspace must be 16-byte aligned");
    }
    if (pl.total_q == 0) return FA8_SUCCESS;

    // ---- TMA descriptors
    CUtensorMap tq, tk, tv;
    memset(&tq, 0, sizeof(tq));
    memset(&tk, 0, sizeof(tk));
    memset(&tv, 0, sizeof(tv));
    const int cw = chunk_of(pl.D), cwv = chunk_of(pl.DV);
    {
        uint64_t dims[4], strides[3];
        dims[0] = pl.D;
        dims[1] = pl.Hq;
        if (pl.q_varlen) {
            dims[2] = pl.total_q;
            dims[3] = 1;
            strides[0] = q->stride[1];
            strides[1] = q->stride[0];
            strides[2] = (uint64_t)q->stride[0] * pl.total_q;
        } else {
            dims[2] = pl.Sq;
            dims[3] = pl.B;
            strides[0] = q->stride[2];
            strides[1] = q->stride[1];
            strides[2] = q->stride[0];
        }
        // one Q tile per TMA load
        const uint32_t box[4] = {(uint32_t)cw, (uint32_t)pl.G, (uint32_t)pl.P, 1};
        if ((st = encode4(&tq, q->data, dims, strides, box, cw, CU_TENSOR_MAP_L2_PROMOTION_L2_128B))) return st;
    }
    const bool kv_empty = (pl.kv_mode == 0 && pl.Sk == 0) || (pl.kv_mode == 1 && pl.total_k == 0) ||
                          (pl.kv_mode == 2 && pl.num_pages == 0);
    if (!kv_empty) {
        for (int which = 0; which < 2; ++which) {
            const fa8_tensor *t = which ? v : k;
            const int d = which ? pl.DV : pl.D;
            const int c = which ? cwv : cw;
            uint64_t dims[4], strides[3];
            dims[0] = d;
            dims[1] = pl.Hkv;
            uint32_t rows = 128;
            if (pl.kv_mode == 1) {
                dims[2] = pl.total_k;
                dims[3] = 1;
                strides[0] = t->stride[1];
                strides[1] = t->stride[0];
                strides[2] = (uint64_t)t->stride[0] * pl.total_k;
            } else {
                dims[2] = t->shape[1];
                dims[3] = t->shape[0];
                strides[0] = t->stride[2];
                strides[1] = t->stride[1];
                strides[2] = t->stride[0];
                if (pl.kv_mode == 2) rows = (uint32_t)pl.box_n;
            }
            const uint32_t box[4] = {(uint32_t)c, 1, rows, 1};
            if ((st = encode4(which ? &tv : &tk, t->data, dims, strides, box, c, CU_TENSOR_MAP_L2_PROMOTION_L2_256B)))
                return st;
        }
    }

    // ---- kernel parameters
    p.B = pl.B;
    p.Hq = pl.Hq;
    p.Hkv = pl.Hkv;
    p.G = pl.G;
    p.rows_per_tile = pl.rows_per_tile;
    p.pos_per_tile = pl.P;
    p.q_varlen = pl.q_varlen;
    p.kv_mode = pl.kv_mode;
    p.Sq = pl.Sq;
    p.Sk = pl.Sk;
    p.total_q = pl.total_q;
    p.total_k = pl.total_k;
    p.mblocks_per_batch = pl.mblocks_per_batch;
    p.cu_q = cu_seqlens_q ? static_cast<const int *>(cu_seqlens_q->data) : nullptr;
    p.cu_k = cu_seqlens_k ? static_cast<const int *>(cu_seqlens_k->data) : nullptr;
    if (block_table) {
        p.block_table = static_cast<const int *>(block_table->data);
        p.bt_stride = block_table->stride[0];
        p.max_pages = pl.max_pages;
        p.page_size = pl.page_size;
        p.box_n = pl.box_n;
        p.boxes_per_tile = 128 / pl.box_n;
        p.num_pages = pl.num_pages;
    }
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.causal = causal;
    p.window_left = window_left;
    p.num_splits = pl.splits;
    p.split_mode = pl.splits > 1;
    p.units = (int)std::min<long long>(pl.units, 0x7fffffffLL);
    p.o = out->data;
    p.o_sb = o_sb;
    p.o_ss = o_ss;
    p.o_sh = o_sh;
    p.out_fp16 = out->dtype == FA8_DTYPE_F16;
    p.lse = lse ? static_cast<float *>(lse->data) : nullptr;
    p.lse_sb = l_sb;
    p.lse_sh = l_sh;
    p.lse_ss = l_ss;
    if (p.split_mode) {
        const size_t rows = (size_t)pl.total_q * pl.Hq * pl.splits;
        p.o_part = static_cast<float *>(workspace);
        p.lse_part = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                               ((rows * pl.DV * sizeof(float) + 255) & ~(size_t)255));
        p.split_cap = reinterpret_cast<int *>(static_cast<char *>(workspace) + pl.ws_bytes - 256);
        // CTAs that run at once: two decode CTAs per SM for (128, 128), one otherwise
        const int per_sm = pl.decode ? fa8::decode_ctas_per_sm(pl.D, pl.DV) : 1;
        p.slots = per_sm * ds->sm_count;
        // when every launched split fits in one wave the finest cap is always the model's
        // choice (split_tile_cap): pass it and skip the plan kernel
        if (pl.cap > 0) p.cap_const = pl.cap;  // chosen with the plan (dense K/V, batched q)
        else if (pl.base_units * pl.splits <= (long long)p.slots) p.cap_const = 2;
    }
    p.timeout_ns = timeout_ns;
    p.status = ds->status;
    p.trace = trace;

    const dim3 grid((unsigned)pl.num_slots, (unsigned)(pl.Hkv * pl.splits), 1);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (p.split_mode && p.cap_const <= 0) {  // the split cap, chosen on the device from the key counts
        fa8::split_plan_kernel<<<1, 32, 0, s>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "split plan kernel launch");
    }
    if (pl.decode) {
        // kv-heads fastest, then request slots, splits slowest: the CTAs of one request run
        // side by side, and splits that a request does not use come last and exit at once
        const dim3 dgrid((unsigned)((long long)pl.Hkv * pl.num_slots), (unsigned)pl.splits, 1);
        switch (pl.D * 1000 + pl.DV) {
            case 128128: e = fa8::launch_decode<128, 128>(p, tq, tk, tv, dgrid, s); break;
            case 192128: e = fa8::launch_decode<192, 128>(p, tq, tk, tv, dgrid, s); break;
            case 256256: e = fa8::launch_decode<256, 256>(p, tq, tk, tv, dgrid, s); break;
            default: return fail(FA8_ERR_UNSUPPORTED, "no decode kernel for (%d, %d)", pl.D, pl.DV);
        }
    } else if (pl.prefill) {
        // persistent: one CTA per SM (or per unit when there are fewer), each walking the unit list
        const dim3 pgrid((unsigned)std::max(1LL, std::min<long long>(pl.units, (long long)ds->sm_count)), 1, 1);
        switch (pl.D * 1000 + pl.DV) {
            case 64064: e = fa8::launch_prefill<64, 64>(p, tq, tk, tv, pgrid, s); break;
            case 96096: e = fa8::launch_prefill<96, 96>(p, tq, tk, tv, pgrid, s); break;
            case 128128: e = fa8::launch_prefill<128, 128>(p, tq, tk, tv, pgrid, s); break;
            case 192128: e = fa8::launch_prefill<192, 128>(p, tq, tk, tv, pgrid, s); break;
            default: return fail(FA8_ERR_UNSUPPORTED, "no prefill kernel for (%d, %d)", pl.D, pl.DV);
        }
    } else switch (pl.D * 1000 + pl.DV) {  // the one-tile kernel: dv > 128
        case 192192: e = fa8::launch_fwd<192, 192>(p, tq, tk, tv, grid, s); break;
        case 256256: e = fa8::launch_fwd<256, 256>(p, tq, tk, tv, grid, s); break;
        default: return fail(FA8_ERR_UNSUPPORTED, "no kernel for (%d, %d)", pl.D, pl.DV);
    }
    if (e != cudaSuccess) return cuda_fail(e, "forward kernel launch");
    if (p.split_mode) {
        fa8::CombineParams cp;
        memset(&cp, 0, sizeof(cp));
        cp.total_q = pl.total_q;
        cp.Hq = pl.Hq;
        cp.num_splits = pl.splits;
        cp.wpr = pl.splits >= 8 ? 8 : (pl.splits >= 4 ? 4 : (pl.splits >= 2 ? 2 : 1));
        cp.q_varlen = pl.q_varlen;
        cp.Sq = pl.Sq;
        cp.B = p.B;
        cp.pos_per_tile = p.pos_per_tile;
        cp.kv_mode = p.kv_mode;
        cp.Sk = p.Sk;
        cp.causal = p.causal;
        cp.window_left = p.window_left;
        cp.cu_q = p.cu_q;
        cp.cu_k = p.cu_k;
        cp.split_cap = p.split_cap;
        cp.cap_const = p.cap_const;
        cp.o_part = p.o_part;
        cp.lse_part = p.lse_part;
        cp.o = p.o;
        cp.o_sb = o_sb;
        cp.o_ss = o_ss;
        cp.o_sh = o_sh;
        cp.out_fp16 = p.out_fp16;
        cp.lse = p.lse;
        cp.lse_sb = l_sb;
        cp.lse_sh = l_sh;
        cp.lse_ss = l_ss;
        switch (pl.DV) {
            case 64: e = fa8::launch_combine<64>(cp, s); break;
            case 96: e = fa8::launch_combine<96>(cp, s); break;
            case 128: e = fa8::launch_combine<128>(cp, s); break;
            case 192: e = fa8::launch_combine<192>(cp, s); break;
            default: e = fa8::launch_combine<256>(cp, s); break;
        }
        if (e != cudaSuccess) return cuda_fail(e, "combine kernel launch");
    }
    return FA8_SUCCESS;
}

fa8_status fa8_fwd_static_scratch(const fa8_tensor *q, const fa8_tensor *k, const fa8_tensor *v,
                                  const fa8_tensor *descale_q, const fa8_tensor *descale_k,
                                  const fa8_tensor *descale_v, fa8_tensor *out, fa8_tensor *lse,
                                  const fa8_tensor *cu_seqlens_q, const fa8_tensor *cu_seqlens_k,
                                  const fa8_tensor *block_table, int page_size, int causal, int window_left,
                                  const fa8_tensor *sink, float softmax_scale, int num_splits, void *stream) {
    g_last_error.clear();
    void *scratch = nullptr;
    fa8_status st = static_scratch(&scratch);
    if (st) return st;
    int splits = 0;
    size_t need = 0;
    st = fa8_fwd_workspace_size(q, k, v, cu_seqlens_q, cu_seqlens_k, block_table, page_size, num_splits, &splits,
                                &need);
    if (st) return st;
    if (need > FA8_STATIC_SCRATCH_BYTES)
        return fail(FA8_ERR_WORKSPACE,
                    "split-KV partials (%d splits) need %zu bytes but the static scratch holds %zu; "
                    "pass a smaller num_splits or call fa8_fwd with a workspace",
                    splits, need, (size_t)FA8_STATIC_SCRATCH_BYTES);
    return fa8_fwd(q, k, v, descale_q, descale_k, descale_v, out, lse, cu_seqlens_q, cu_seqlens_k, block_table,
                   page_size, causal, window_left, sink, softmax_scale, num_splits, scratch,
                   FA8_STATIC_SCRATCH_BYTES, stream);
}

}  // extern "C"
