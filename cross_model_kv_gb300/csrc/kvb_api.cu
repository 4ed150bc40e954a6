// Host side of libkvb: argument validation, contexts, dispatch of the mapper
// apply.  Every entry point returns a status; nothing aborts the process.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "kvb_internal.h"
#include "kvb_host.h"

namespace kvb {

thread_local std::string g_last_error;

kvb_status fail(kvb_status s, const std::string& msg) {
    g_last_error = msg;
    return s;
}

kvb_status cuda_fail(cudaError_t e, const char* what) {
    (void)cudaGetLastError();  // clear a sticky launch error so the next call starts clean
    std::string m = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    return fail(e == cudaErrorMemoryAllocation ? KVB_ERR_OOM : KVB_ERR_CUDA, m);
}

EncodeTiledFn get_encode_tiled() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kvb_status check_device_ptrs(std::initializer_list<const void*> ptrs, const char* what) {
    for (const void* p : ptrs) {
        if (!p) return fail(KVB_ERR_INVALID_ARG, std::string(what) + ": null device pointer");
        if (!aligned16(p)) return fail(KVB_ERR_INVALID_ARG, std::string(what) + ": device pointer not 16-byte aligned");
    }
    return KVB_OK;
}

kvb_status check_selection(const kvb_ctx* c, const int32_t* sel, const char* name, SelTable* tab, int kv,
                           int t_begin, int t_end) {
    if (!sel) return fail(KVB_ERR_INVALID_ARG, std::string(name) + " is NULL");
    if (t_end < 0) t_end = c->L_t;
    for (int t = t_begin; t < t_end; ++t) {
        for (int j = 0; j < c->k; ++j) {
            const int32_t v = sel[t * c->k + j];
            if (v < 0 || v >= c->L_s)
                return fail(KVB_ERR_INVALID_ARG, std::string(name) + ": entry out of range [0, L_src)");
            for (int i = 0; i < j; ++i)
                if (sel[t * c->k + i] == v)
                    return fail(KVB_ERR_INVALID_ARG, std::string(name) + ": repeated source layer in a row");
            if (tab) tab->s[kv][t][j] = static_cast<uint8_t>(v);
        }
    }
    return KVB_OK;
}

// Report (and clear) kernel-recorded errors mirrored to the host by earlier calls.
kvb_status take_device_error(kvb_ctx* c) {
    const int code = c->err_mirror ? *c->err_mirror : 0;
    if (code == 0) return KVB_OK;
    *c->err_mirror = 0;
    cudaMemset(c->err_dev, 0, sizeof(int));
    if (code == DEV_ERR_TIMEOUT)
        return fail(KVB_ERR_TIMEOUT, "a bounded device wait gave up in an earlier kernel on this context");
    if (code == DEV_ERR_BOUNDS)
        return fail(KVB_ERR_CUDA, "an index check of the checked build failed in an earlier kernel on this context");
    return fail(KVB_ERR_INVALID_ARG, "a position outside [0, max_pos) was seen by an earlier kernel on this context");
}

void mirror_device_error(kvb_ctx* c, cudaStream_t s) {
    cudaMemcpyAsync(c->err_mirror, c->err_dev, sizeof(int), cudaMemcpyDeviceToHost, s);
}

DevErr dev_err(const kvb_ctx* c) { return DevErr{c->err_dev, c->timeout_ns}; }

kvb_status ensure_scratch(kvb_ctx* c, size_t bytes) {
    if (bytes <= c->scratch_bytes) return KVB_OK;
    if (c->scratch) {
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "sync before growing scratch");
        cudaFree(c->scratch);
        c->scratch = nullptr;
        c->scratch_bytes = 0;
    }
    cudaError_t e = cudaMalloc(&c->scratch, bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc strip scratch");
    c->scratch_bytes = bytes;
    return KVB_OK;
}

struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) cudaSetDevice(dev);
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

}  // namespace kvb

using namespace kvb;

extern "C" {

const char* kvb_last_error(void) { return g_last_error.c_str(); }

int32_t kvb_version(void) { return (0 << 16) | 1; }

kvb_status kvb_ctx_create(const kvb_model_spec* src, const kvb_model_spec* tgt, int32_t top_k, int32_t max_pos,
                          int32_t device, kvb_ctx** out) {
    g_last_error.clear();
    if (!out) return fail(KVB_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!src || !tgt) return fail(KVB_ERR_INVALID_ARG, "model spec is NULL");
    if (src->rope_interleaved || tgt->rope_interleaved)
        return fail(KVB_ERR_UNSUPPORTED, "interleaved (traditional) RoPE is refused");
    if (src->rope_scaling || tgt->rope_scaling) return fail(KVB_ERR_UNSUPPORTED, "rope_scaling is refused");
    if (src->n_kv_heads != tgt->n_kv_heads || src->head_dim != tgt->head_dim)
        return fail(KVB_ERR_SHAPE_MISMATCH, "source and target KV heads / head_dim differ (matched-KV pairs only)");
    if (src->n_layers < 1 || tgt->n_layers < 1 || src->n_kv_heads < 1 || src->head_dim < 2)
        return fail(KVB_ERR_INVALID_ARG, "layers, heads and head_dim must be positive");
    if (src->head_dim % 2) return fail(KVB_ERR_UNSUPPORTED, "head_dim must be even");
    if (src->head_dim % 8 || src->head_dim > 256)
        return fail(KVB_ERR_UNSUPPORTED, "head_dim must be a multiple of 8 and at most 256");
    if (src->n_layers > MAX_LS) return fail(KVB_ERR_UNSUPPORTED, "more than 255 source layers");
    if (tgt->n_layers > MAX_LT) return fail(KVB_ERR_UNSUPPORTED, "more than 128 target layers");
    if (top_k < 1 || top_k > src->n_layers) return fail(KVB_ERR_INVALID_ARG, "top_k must be in [1, L_src]");
    if (top_k > MAX_K) return fail(KVB_ERR_UNSUPPORTED, "top_k above 16");
    if (!(src->rope_theta > 1.0) || !(tgt->rope_theta > 1.0))
        return fail(KVB_ERR_INVALID_ARG, "rope_theta must be > 1");
    if (max_pos < 1) return fail(KVB_ERR_INVALID_ARG, "max_pos must be >= 1");
    int ndev = 0;
    cudaError_t e = cudaGetDeviceCount(&ndev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceCount");
    if (device < 0 || device >= ndev) return fail(KVB_ERR_INVALID_ARG, "device index out of range");
    DeviceGuard g(device);

    kvb_ctx* c = new (std::nothrow) kvb_ctx();
    if (!c) return fail(KVB_ERR_OOM, "host allocation failed");
    c->src = *src;
    c->tgt = *tgt;
    c->L_s = src->n_layers;
    c->L_t = tgt->n_layers;
    c->H = src->n_kv_heads;
    c->d = src->head_dim;
    c->k = top_k;
    c->max_pos = max_pos;
    c->device = device;
    c->timeout_ns = 2000ull * 1000 * 1000;
    if (const char* s = std::getenv("KVB_WAIT_TIMEOUT_MS")) {
        const long long ms = std::atoll(s);
        if (ms >= 0) c->timeout_ns = static_cast<uint64_t>(ms) * 1000 * 1000;
    }
    cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device);
    const size_t tab_bytes = static_cast<size_t>(max_pos) * (c->d / 2) * sizeof(float2);
    kvb_status st = KVB_OK;
    do {
        if ((e = cudaMalloc(&c->tab_s, tab_bytes)) != cudaSuccess) { st = cuda_fail(e, "cudaMalloc rope table"); break; }
        if ((e = cudaMalloc(&c->tab_t, tab_bytes)) != cudaSuccess) { st = cuda_fail(e, "cudaMalloc rope table"); break; }
        if ((e = cudaMalloc(&c->err_dev, sizeof(int))) != cudaSuccess) { st = cuda_fail(e, "cudaMalloc error word"); break; }
        if ((e = cudaMalloc(&c->strip_ctr, 4 * sizeof(int))) != cudaSuccess) { st = cuda_fail(e, "cudaMalloc counters"); break; }
        if ((e = cudaHostAlloc(&c->err_mirror, sizeof(int), cudaHostAllocDefault)) != cudaSuccess) { st = cuda_fail(e, "cudaHostAlloc"); break; }
        *c->err_mirror = 0;
        if ((e = cudaMemset(c->err_dev, 0, sizeof(int))) != cudaSuccess) { st = cuda_fail(e, "cudaMemset"); break; }
        if ((e = launch_rope_table(c->tab_s, max_pos, c->d, src->rope_theta, 0)) != cudaSuccess) { st = cuda_fail(e, "rope table"); break; }
        if ((e = launch_rope_table(c->tab_t, max_pos, c->d, tgt->rope_theta, 0)) != cudaSuccess) { st = cuda_fail(e, "rope table"); break; }
        if ((e = cudaStreamSynchronize(0)) != cudaSuccess) { st = cuda_fail(e, "rope table build"); break; }
    } while (0);
    if (st != KVB_OK) {
        kvb_ctx_destroy(c);
        return st;
    }
    *out = c;
    return KVB_OK;
}

kvb_status kvb_ctx_destroy(kvb_ctx* c) {
    if (!c) return KVB_OK;
    DeviceGuard g(c->device);
    cudaDeviceSynchronize();
    cudaFree(c->tab_s);
    cudaFree(c->tab_t);
    cudaFree(c->scratch);
    cudaFree(c->err_dev);
    cudaFree(c->strip_ctr);
    if (c->err_mirror) cudaFreeHost(c->err_mirror);
    for (auto& r : c->prof) {
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.end);
    }
    for (auto e : c->event_pool) cudaEventDestroy(e);
    delete c;
    return KVB_OK;
}

kvb_status kvb_ctx_reserve(kvb_ctx* c, int64_t T) {
    g_last_error.clear();
    if (!c) return fail(KVB_ERR_INVALID_ARG, "ctx is NULL");
    if (T < 0) return fail(KVB_ERR_INVALID_ARG, "T < 0");
    DeviceGuard g(c->device);
    return ensure_scratch(c, static_cast<size_t>(c->L_s) * c->H * static_cast<size_t>(T) * c->d * 2);
}

kvb_status kvb_ctx_check(kvb_ctx* c, void* stream) {
    g_last_error.clear();
    if (!c) return fail(KVB_ERR_INVALID_ARG, "ctx is NULL");
    DeviceGuard g(c->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "stream sync");
    int code = 0;
    e = cudaMemcpy(&code, c->err_dev, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read error word");
    *c->err_mirror = code;
    return take_device_error(c);
}

kvb_status kvb_map_apply(kvb_ctx* c, kvb_dtype dtype, const void* src_k, const void* src_v,
                         const int32_t* positions, int64_t T, const int32_t* sel_k, const int32_t* sel_v,
                         const void* W_k, const void* W_v, const float* b_k, const float* b_v, void* out_k,
                         void* out_v, void* stream) {
    g_last_error.clear();
    if (!c) return fail(KVB_ERR_INVALID_ARG, "ctx is NULL");
    if (dtype != KVB_F32 && dtype != KVB_BF16) return fail(KVB_ERR_UNSUPPORTED, "dtype must be KVB_F32 or KVB_BF16");
    if (T < 0) return fail(KVB_ERR_INVALID_ARG, "T < 0");
    if (T > 0x7fffffffLL) return fail(KVB_ERR_UNSUPPORTED, "T above 2^31-1");
    SelTable tab;
    std::memset(&tab, 0, sizeof(tab));
    kvb_status st;
    if ((st = check_selection(c, sel_k, "sel_k", &tab, 0)) != KVB_OK) return st;
    if ((st = check_selection(c, sel_v, "sel_v", &tab, 1)) != KVB_OK) return st;
    if ((st = take_device_error(c)) != KVB_OK) return st;
    if (T == 0) return KVB_OK;
    if ((st = check_device_ptrs({src_k, src_v, positions, W_k, W_v, b_k, b_v, out_k, out_v}, "kvb_map_apply")) != KVB_OK)
        return st;
    DeviceGuard g(c->device);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Shape sh{c->L_s, c->L_t, c->H, c->d, c->k, T, c->max_pos};
    cudaError_t e;
    if (dtype == KVB_BF16 && map_gemm_tc_supported(sh)) {
        const size_t need = static_cast<size_t>(c->L_s) * c->H * static_cast<size_t>(T) * c->d * 2;
        if ((st = ensure_scratch(c, need)) != KVB_OK) return st;
        // The strip runs inside the map kernel (its epilogue warps strip the source
        // keys while the value tiles are computed) unless KVB_MAP_FUSED_STRIP=0.
        const char* fs = std::getenv("KVB_MAP_FUSED_STRIP");
        const bool fused = !(fs && std::strcmp(fs, "0") == 0) && map_gemm_fused_strip_supported(sh);
        e = cudaMemsetAsync(c->strip_ctr, 0, 4 * sizeof(int), s);  // strip and tile counters
        if (e == cudaSuccess && !fused) {
            ProfScope ps(c, s, "rope_strip_bf16");
            e = launch_strip_bf16(static_cast<const __nv_bfloat16*>(src_k), static_cast<__nv_bfloat16*>(c->scratch),
                                  positions, c->tab_s, static_cast<int64_t>(c->L_s) * c->H, T, c->d, c->max_pos,
                                  dev_err(c), c->num_sms, s);
        }
        if (e != cudaSuccess) return cuda_fail(e, "strip launch");
        MapGemmArgs a{};
        a.sh = sh;
        if (fused) {
            a.fuse_strip = true;
            a.k_raw = src_k;
            a.tab_s = c->tab_s;
            a.strip_ctr = c->strip_ctr;
        }
        const char* ps = std::getenv("KVB_MAP_PAIR_STATIC");  // fixed tiles per pair (comparison runs)
        a.tile_ctr = (ps && std::strcmp(ps, "1") == 0) ? nullptr : c->strip_ctr + 2;
        a.a_src[0] = c->scratch;
        a.a_src[1] = src_v;
        a.w[0] = W_k;
        a.w[1] = W_v;
        a.bias[0] = b_k;
        a.bias[1] = b_v;
        a.out[0] = out_k;
        a.out[1] = out_v;
        a.pos = positions;
        a.tab_t = c->tab_t;
        a.sel = tab;
        a.err = dev_err(c);
        a.num_sms = c->num_sms;
        std::string why;
        {
            ProfScope ps(c, s, "map_gemm_tcgen05");
            e = launch_map_gemm_tc(a, s, &why);
        }
        if (e != cudaSuccess) {
            if (!why.empty()) return fail(KVB_ERR_CUDA, "map GEMM launch: " + why);
            return cuda_fail(e, "map GEMM launch");
        }
    } else if (dtype == KVB_F32 && map_gemm_tc_supported(sh)) {
        // fp32 caches on the tensor cores: stripped keys, values and both
        // maps are split into bf16 (hi, lo) pairs in the context's scratch,
        // then one three-pass GEMM accumulates hi*hi + hi*lo + lo*hi in fp32.
        const size_t n_src = static_cast<size_t>(c->L_s) * c->H * static_cast<size_t>(T) * c->d;
        const size_t n_w = static_cast<size_t>(c->L_t) * c->H * c->d * static_cast<size_t>(c->k) * c->H * c->d;
        if ((st = ensure_scratch(c, (4 * n_src + 4 * n_w) * 2)) != KVB_OK) return st;
        __nv_bfloat16* base = static_cast<__nv_bfloat16*>(c->scratch);
        __nv_bfloat16* a_hi[2] = {base, base + 2 * n_src};
        __nv_bfloat16* a_lo[2] = {base + n_src, base + 3 * n_src};
        __nv_bfloat16* w_hi[2] = {base + 4 * n_src, base + 4 * n_src + 2 * n_w};
        __nv_bfloat16* w_lo[2] = {base + 4 * n_src + n_w, base + 4 * n_src + 3 * n_w};
        {
            ProfScope ps(c, s, "split_f32");
            e = launch_strip_split_f32(static_cast<const float*>(src_k), a_hi[0], a_lo[0], positions, c->tab_s,
                                       static_cast<int64_t>(c->L_s) * c->H, T, c->d, c->max_pos, dev_err(c),
                                       c->num_sms, s);
            if (e == cudaSuccess)
                e = launch_split_f32(static_cast<const float*>(src_v), a_hi[1], a_lo[1], static_cast<int64_t>(n_src),
                                     c->num_sms, s);
            if (e == cudaSuccess)
                e = launch_split_f32(static_cast<const float*>(W_k), w_hi[0], w_lo[0], static_cast<int64_t>(n_w),
                                     c->num_sms, s);
            if (e == cudaSuccess)
                e = launch_split_f32(static_cast<const float*>(W_v), w_hi[1], w_lo[1], static_cast<int64_t>(n_w),
                                     c->num_sms, s);
        }
        if (e != cudaSuccess) return cuda_fail(e, "fp32 split launch");
        MapGemmArgs a{};
        a.sh = sh;
        a.split = true;
        for (int kv = 0; kv < 2; ++kv) {
            a.a_src[kv] = a_hi[kv];
            a.a_lo[kv] = a_lo[kv];
            a.w[kv] = w_hi[kv];
            a.w_lo[kv] = w_lo[kv];
        }
        a.bias[0] = b_k;
        a.bias[1] = b_v;
        a.out[0] = out_k;
        a.out[1] = out_v;
        a.pos = positions;
        a.tab_t = c->tab_t;
        a.sel = tab;
        a.err = dev_err(c);
        a.num_sms = c->num_sms;
        const char* ps_env = std::getenv("KVB_MAP_PAIR_STATIC");  // fixed tiles per pair (comparison runs)
        a.tile_ctr = (ps_env && std::strcmp(ps_env, "1") == 0) ? nullptr : c->strip_ctr + 2;
        e = cudaMemsetAsync(c->strip_ctr, 0, 4 * sizeof(int), s);
        if (e != cudaSuccess) return cuda_fail(e, "counter reset");
        std::string why;
        {
            ProfScope ps(c, s, "map_gemm_tcgen05_split3");
            e = launch_map_gemm_tc(a, s, &why);
        }
        if (e != cudaSuccess) {
            if (!why.empty()) return fail(KVB_ERR_CUDA, "map GEMM launch: " + why);
            return cuda_fail(e, "map GEMM launch");
        }
    } else {
        MapSimtArgs a{};
        a.sh = sh;
        a.dtype = dtype;
        a.src[0] = src_k;
        a.src[1] = src_v;
        a.w[0] = W_k;
        a.w[1] = W_v;
        a.bias[0] = b_k;
        a.bias[1] = b_v;
        a.out[0] = out_k;
        a.out[1] = out_v;
        a.pos = positions;
        a.tab_s = c->tab_s;
        a.tab_t = c->tab_t;
        a.sel = tab;
        a.err = dev_err(c);
        {
            ProfScope ps(c, s, "map_simt");
            e = launch_map_simt(a, s);
        }
        if (e != cudaSuccess) return cuda_fail(e, "SIMT map launch");
    }
    mirror_device_error(c, s);
    return KVB_OK;
}

}  // extern "C"

// ------------------------------------------------------------ kernel timing
namespace kvb {

static cudaEvent_t pool_event(kvb_ctx* c) {
    if (!c->event_pool.empty()) {
        cudaEvent_t e = c->event_pool.back();
        c->event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

ProfScope::ProfScope(kvb_ctx* ctx, cudaStream_t stream, const char* name) : c(ctx), s(stream) {
    if (!c->profiling) return;
    kvb_ctx::ProfRec r{name, pool_event(c), pool_event(c)};
    if (!r.start || !r.end) return;
    cudaEventRecord(r.start, s);
    c->prof.push_back(r);
    idx = static_cast<int>(c->prof.size()) - 1;
}

ProfScope::~ProfScope() {
    if (idx >= 0) cudaEventRecord(c->prof[idx].end, s);
}

}  // namespace kvb

extern "C" {

kvb_status kvb_profile_enable(kvb_ctx* c, int32_t on) {
    g_last_error.clear();
    if (!c) return fail(KVB_ERR_INVALID_ARG, "ctx is NULL");
    c->profiling = on != 0;
    return KVB_OK;
}

kvb_status kvb_profile_read(kvb_ctx* c, kvb_kernel_time* out, int32_t cap, int32_t* count) {
    g_last_error.clear();
    if (!c || !count || (cap > 0 && !out)) return fail(KVB_ERR_INVALID_ARG, "NULL argument");
    DeviceGuard g(c->device);
    std::vector<kvb_kernel_time> acc;
    kvb_status st = KVB_OK;
    for (auto& r : c->prof) {
        float ms = 0.f;
        cudaError_t e = cudaEventSynchronize(r.end);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start, r.end);
        if (e != cudaSuccess && st == KVB_OK) st = cuda_fail(e, "reading kernel timing events");
        size_t i = 0;
        while (i < acc.size() && std::strncmp(acc[i].name, r.name, sizeof(acc[i].name)) != 0) ++i;
        if (i == acc.size()) {
            kvb_kernel_time t{};
            std::strncpy(t.name, r.name, sizeof(t.name) - 1);
            acc.push_back(t);
        }
        acc[i].launches += 1;
        acc[i].total_ms += ms;
        c->event_pool.push_back(r.start);
        c->event_pool.push_back(r.end);
    }
    c->prof.clear();
    int32_t n = 0;
    for (; n < cap && n < static_cast<int32_t>(acc.size()); ++n) out[n] = acc[n];
    *count = n;
    return st;
}

}  // extern "C"
