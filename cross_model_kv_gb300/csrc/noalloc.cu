// kvb_map_apply_noalloc: the mapper apply for callers that cannot allocate
// device memory.
//
// Some callers are not allowed to call cudaMalloc at all: code that runs
// inside another framework's caching allocator or memory pool (which owns
// every byte of the device and would be bypassed or fragmented by a raw
// allocation), or a runtime that hands out a fixed device-memory budget up
// front.  Such callers cannot create a kvb_ctx (it allocates RoPE tables and
// the strip scratch).  This entry point runs the same two kernels as the
// tensor-core path of kvb_map_apply, but keeps its scratch -- both RoPE
// tables, the RoPE-stripped source keys and the kernels' error word -- in the
// fixed array below, which lives in the library's own device image.
//
// Cost of that choice: every GPU that loads this library holds the array
// (64 MiB) until the process exits, and all calls share it.
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kvb_host.h"

namespace kvb {
namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB

// Scratch of kvb_map_apply_noalloc.  In host code this name is only a
// host-side stand-in: the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // ID of the context the address belongs to

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// ID of the current context (unique for the life of the process), or false if
// no context is current or the driver lacks the calls.
bool current_context_id(unsigned long long* id) {
    static std::once_flag once;
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext cur = nullptr;
    if (!get_current || !get_id || get_current(&cur) != CUDA_SUCCESS || !cur) return false;
    return get_id(cur, id) == CUDA_SUCCESS;
}

// Device address of the scratch on the current device.  Set-up runs on the
// first call on a device and again whenever that device's context is not the
// one the address was taken in (after cudaDeviceReset, say), so a stale
// address is never handed to a kernel.
kvb_status scratch_on_device(int dev, unsigned char** out) {
    if (dev < 0 || dev >= kMaxDevices) return fail(KVB_ERR_UNSUPPORTED, "device index above 63");
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    unsigned long long id = 0;
    const bool known = current_context_id(&id);
    if (!g_scratch_ptr[dev] || !known || id != g_scratch_ctx[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the static scratch");
        g_scratch_ptr[dev] = p;
        // the lookup above makes the device's context current if none was
        g_scratch_ctx[dev] = current_context_id(&id) ? id : 0;
    }
    *out = static_cast<unsigned char*>(g_scratch_ptr[dev]);
    return KVB_OK;
}

size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

}  // namespace
}  // namespace kvb

using namespace kvb;

extern "C" kvb_status kvb_map_apply_noalloc(const kvb_model_spec* src, const kvb_model_spec* tgt, int32_t top_k,
                                            int32_t max_pos, const void* src_k, const void* src_v,
                                            const int32_t* positions, int64_t T, const int32_t* sel_k,
                                            const int32_t* sel_v, const void* W_k, const void* W_v,
                                            const float* b_k, const float* b_v, void* out_k, void* out_v,
                                            void* stream) {
    g_last_error.clear();
    if (!src || !tgt) return fail(KVB_ERR_INVALID_ARG, "model spec is NULL");
    if (src->rope_interleaved || tgt->rope_interleaved)
        return fail(KVB_ERR_UNSUPPORTED, "interleaved (traditional) RoPE is refused");
    if (src->rope_scaling || tgt->rope_scaling) return fail(KVB_ERR_UNSUPPORTED, "rope_scaling is refused");
    if (src->n_kv_heads != tgt->n_kv_heads || src->head_dim != tgt->head_dim)
        return fail(KVB_ERR_SHAPE_MISMATCH, "source and target KV heads / head_dim differ (matched-KV pairs only)");
    if (src->n_layers < 1 || tgt->n_layers < 1 || src->n_kv_heads < 1)
        return fail(KVB_ERR_INVALID_ARG, "layers and heads must be positive");
    if (src->n_layers > MAX_LS || tgt->n_layers > MAX_LT)
        return fail(KVB_ERR_UNSUPPORTED, "more than 255 source or 128 target layers");
    if (top_k < 1 || top_k > src->n_layers || top_k > MAX_K)
        return fail(KVB_ERR_INVALID_ARG, "top_k must be in [1, min(L_src, 16)]");
    if (!(src->rope_theta > 1.0) || !(tgt->rope_theta > 1.0)) return fail(KVB_ERR_INVALID_ARG, "rope_theta must be > 1");
    if (max_pos < 1) return fail(KVB_ERR_INVALID_ARG, "max_pos must be >= 1");
    if (T < 0 || T > 0x7fffffffLL) return fail(KVB_ERR_INVALID_ARG, "T outside [0, 2^31)");
    Shape sh{src->n_layers, tgt->n_layers, src->n_kv_heads, src->head_dim, top_k, T, max_pos};
    if (!map_gemm_tc_supported(sh))
        return fail(KVB_ERR_UNSUPPORTED, "kvb_map_apply_noalloc needs head_dim 128 and n_kv_heads * 128 a multiple of 256");

    // Scratch layout: [source table | target table | stripped keys | error word, tile counter].
    const size_t tab_bytes = align256(size_t(max_pos) * (sh.d / 2) * sizeof(float2));
    const size_t keys_bytes = align256(size_t(sh.L_s) * sh.H * size_t(T) * sh.d * 2);
    const size_t need = 2 * tab_bytes + keys_bytes + 256;
    if (need > kStaticScratchBytes)
        return fail(KVB_ERR_INVALID_ARG,
                    "kvb_map_apply_noalloc: 8*max_pos*head_dim + 2*L_src*H*T*head_dim bytes exceed its fixed "
                    "64 MiB scratch; use kvb_map_apply or a shorter T / max_pos");

    // Same host-side checks as kvb_map_apply, against a stand-in context.
    kvb_ctx shape_only;
    shape_only.L_s = sh.L_s;
    shape_only.L_t = sh.L_t;
    shape_only.k = top_k;
    SelTable tab;
    std::memset(&tab, 0, sizeof(tab));
    kvb_status st;
    if ((st = check_selection(&shape_only, sel_k, "sel_k", &tab, 0)) != KVB_OK) return st;
    if ((st = check_selection(&shape_only, sel_v, "sel_v", &tab, 1)) != KVB_OK) return st;
    if (T == 0) return KVB_OK;
    if ((st = check_device_ptrs({src_k, src_v, positions, W_k, W_v, b_k, b_v, out_k, out_v}, "kvb_map_apply_noalloc")) !=
        KVB_OK)
        return st;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    unsigned char* base = nullptr;
    if ((st = scratch_on_device(dev, &base)) != KVB_OK) return st;
    float2* tab_s = reinterpret_cast<float2*>(base);
    float2* tab_t = reinterpret_cast<float2*>(base + tab_bytes);
    __nv_bfloat16* keys = reinterpret_cast<__nv_bfloat16*>(base + 2 * tab_bytes);
    int* err_word = reinterpret_cast<int*>(base + 2 * tab_bytes + keys_bytes);

    int num_sms = 0;
    e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    uint64_t timeout_ns = 2000ull * 1000 * 1000;
    if (const char* s = std::getenv("KVB_WAIT_TIMEOUT_MS")) {
        const long long ms = std::atoll(s);
        if (ms >= 0) timeout_ns = static_cast<uint64_t>(ms) * 1000 * 1000;
    }
    const DevErr err{err_word, timeout_ns};
    cudaStream_t cs = static_cast<cudaStream_t>(stream);

    // The error word and the tile counter start at zero; the tables and keys are fully rewritten.
    e = cudaMemsetAsync(err_word, 0, 2 * sizeof(int), cs);
    if (e == cudaSuccess) e = launch_rope_table(tab_s, max_pos, sh.d, src->rope_theta, cs);
    if (e == cudaSuccess) e = launch_rope_table(tab_t, max_pos, sh.d, tgt->rope_theta, cs);
    if (e == cudaSuccess)
        e = launch_strip_bf16(static_cast<const __nv_bfloat16*>(src_k), keys, positions, tab_s,
                              static_cast<int64_t>(sh.L_s) * sh.H, T, sh.d, max_pos, err, num_sms, cs);
    if (e != cudaSuccess) return cuda_fail(e, "kvb_map_apply_noalloc: table / strip launch");
    MapGemmArgs a{};
    a.sh = sh;
    a.a_src[0] = keys;
    a.a_src[1] = src_v;
    a.w[0] = W_k;
    a.w[1] = W_v;
    a.bias[0] = b_k;
    a.bias[1] = b_v;
    a.out[0] = out_k;
    a.out[1] = out_v;
    a.pos = positions;
    a.tab_t = tab_t;
    a.sel = tab;
    a.err = err;
    a.num_sms = num_sms;
    a.tile_ctr = err_word + 1;
    std::string why;
    e = launch_map_gemm_tc(a, cs, &why);
    if (e != cudaSuccess) {
        if (!why.empty()) return fail(KVB_ERR_CUDA, "kvb_map_apply_noalloc: " + why);
        return cuda_fail(e, "kvb_map_apply_noalloc: GEMM launch");
    }
    // Wait for the kernels so their error word can be reported by this call.
    int code = 0;
    e = cudaMemcpyAsync(&code, err_word, sizeof(int), cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return cuda_fail(e, "kvb_map_apply_noalloc");
    if (code == DEV_ERR_TIMEOUT) return fail(KVB_ERR_TIMEOUT, "kvb_map_apply_noalloc: a bounded device wait gave up");
    if (code == DEV_ERR_BOUNDS) return fail(KVB_ERR_CUDA, "kvb_map_apply_noalloc: an index check of the checked build failed");
    if (code != 0)
        return fail(KVB_ERR_INVALID_ARG, "kvb_map_apply_noalloc: a position outside [0, max_pos) (row written as zeros)");
    return KVB_OK;
}
