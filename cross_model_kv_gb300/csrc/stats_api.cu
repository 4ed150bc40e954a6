// Calibration statistics, layer selection and ridge solve: entry points.
//
// One kvb_stats object keeps, for K and for V, the centered statistics of ALL
// source features against ALL target columns ("KVBridge" README, "Loading"),
// so that selection can be decided before any per-target system is formed:
// the statistics of a selection are sub-blocks (centering commutes with
// choosing columns).
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "fit_internal.h"
#include "kvb_host.h"

using namespace kvb;

struct kvb_stats {
    kvb_ctx* ctx = nullptr;
    kvb_dtype dtype = KVB_BF16;
    int64_t max_T = 0, ld = 0;  // ld: columns of the compact batch matrices (multiple of 64)
    int64_t Fs = 0, Ft = 0;     // all source features; target columns of the block
    int t0 = 0, nt = 0;         // target layers [t0, t0 + nt) held by this object
    long long* n_dev = nullptr;
    int* nb_dev = nullptr;
    float* coef_dev = nullptr;  // {f = n_a n_b / n, g = n_b} of the current batch
    int* rows = nullptr;
    float* mean[4] = {};   // running means: source K, source V, target K, target V
    float* bmean[4] = {};  // batch means (generic gather)
    float* delta[4] = {};  // batch mean - running mean before the merge
    float* zbar[4] = {};   // mean of the shifted batch (0 on the generic gather)
    float* zsum[4] = {};   // column sums of the shifted batch (single-pass gather)
    float* shift[4] = {};  // shift of the batch (single-pass gather)
    float* part = nullptr; // [ld/64][max(Fs, Ft)] per-chunk column sums of one matrix
    // four-matrix gather (bf16, head_dim 128): per-chunk column sums of all four
    // matrices [ld/128][2 Fs + 2 Ft] and target sums of squares [ld/128][2 Ft]
    float* part_all = nullptr;
    float* part_sq = nullptr;
    float* gram[2] = {};   // [Fs][Fs], lower triangle kept
    float* cross[2] = {};  // [Fs][Ft]
    float* syy[2] = {};    // [Ft]
    void* XT[2] = {};      // centered batch, [Fs][ld]: float32, or bf16 hi part
    void* YT[2] = {};      // centered batch, [Ft][ld]: float32, or bf16 hi part
    void* XT_lo[2] = {};   // bf16 lo parts (tensor-core path only)
    void* YT_lo[2] = {};
    void* XT_3[2] = {};    // third bf16 parts (tensor-core path, fp32 caches)
    void* YT_3[2] = {};
    StatsGemmPlan* plan = nullptr;
    bool use_tc = false;
    // fit workspace, allocated on first use
    float* wsG = nullptr;
    size_t wsG_bytes = 0;
    float* wsR = nullptr;
    size_t wsR_bytes = 0;
    float* wsD = nullptr;
    size_t wsD_bytes = 0;
    float* wsS = nullptr;
    size_t wsS_bytes = 0;
    float* wsL = nullptr;  // inverses of the 64 x 64 diagonal blocks of the factors
    size_t wsL_bytes = 0;
    float* wsT = nullptr;  // bf16 parts of the tensor-core update operands
    size_t wsT_bytes = 0;
    float* r2 = nullptr;  // [2][L_t][L_s]
    int* sel = nullptr;   // [2][L_t][k]
    int* numeric = nullptr;
    std::vector<void*> allocs;
};

namespace {

// Bytes of solve workspace per batch of systems: half the free device memory,
// between 4 and 48 GiB (more systems per batch keep more SMs busy in the
// panel steps of the factorisations, which work one diagonal block at a time).
// KVB_FIT_WORKSPACE_MB lowers the cap (a caller sharing the device, or a test
// that wants the systems split over several batches); a batch always holds at
// least one system.
size_t ws_budget() {
    size_t free_b = 0, total_b = 0;
    if (cudaMemGetInfo(&free_b, &total_b) != cudaSuccess) {
        cudaGetLastError();
        free_b = 0;
    }
    size_t budget = std::max<size_t>(size_t(4) << 30, std::min<size_t>(size_t(48) << 30, free_b / 2));
    if (const char* cap = std::getenv("KVB_FIT_WORKSPACE_MB")) {
        const long long mb = std::atoll(cap);
        if (mb > 0) budget = std::min<size_t>(budget, static_cast<size_t>(mb) << 20);
    }
    return budget;
}

kvb_status st_alloc(kvb_stats* st, void** p, size_t bytes) {
    cudaError_t e = cudaMalloc(p, bytes ? bytes : 16);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc statistics");
    st->allocs.push_back(*p);
    return KVB_OK;
}

kvb_status ws_grow(kvb_stats* st, float** p, size_t* have, size_t bytes) {
    if (bytes <= *have) return KVB_OK;
    if (*p) {
        cudaFree(*p);
        *p = nullptr;
        *have = 0;
    }
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(p), bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc fit workspace");
    *have = bytes;
    return KVB_OK;
}

kvb_status zero_stats(kvb_stats* st, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    const int64_t len[4] = {st->Fs, st->Fs, st->Ft, st->Ft};
    for (int m = 0; m < 4 && e == cudaSuccess; ++m) e = cudaMemsetAsync(st->mean[m], 0, len[m] * 4, s);
    for (int kv = 0; kv < 2 && e == cudaSuccess; ++kv) {
        e = cudaMemsetAsync(st->gram[kv], 0, st->Fs * st->Fs * 4, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(st->cross[kv], 0, st->Fs * st->Ft * 4, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(st->syy[kv], 0, st->Ft * 4, s);
    }
    if (e == cudaSuccess) e = cudaMemsetAsync(st->n_dev, 0, sizeof(long long), s);
    if (e != cudaSuccess) return cuda_fail(e, "zeroing statistics");
    return KVB_OK;
}

void free_stats(kvb_stats* st) {
    for (void* p : st->allocs) cudaFree(p);
    cudaFree(st->wsG);
    cudaFree(st->wsR);
    cudaFree(st->wsD);
    cudaFree(st->wsS);
    cudaFree(st->wsL);
    cudaFree(st->wsT);
    if (st->plan) stats_gemm_tc_free(st->plan);
    delete st;
}

void stats_jobs(const kvb_stats* st, StatsJob jobs[4]) {
    for (int kv = 0; kv < 2; ++kv) {
        StatsJob& g = jobs[kv];  // Gram: lower triangle only
        g.A = st->XT[kv];
        g.B = st->XT[kv];
        g.A_lo = st->XT_lo[kv];
        g.B_lo = st->XT_lo[kv];
        g.A_3 = st->XT_3[kv];
        g.B_3 = st->XT_3[kv];
        g.out = st->gram[kv];
        g.da = st->delta[kv];
        g.db = st->delta[kv];
        g.za = st->zbar[kv];
        g.zb = st->zbar[kv];
        g.Ma = st->Fs;
        g.Nb = st->Fs;
        g.ldo = st->Fs;
        g.lower = 1;
        StatsJob& x = jobs[2 + kv];  // cross statistics against every target column
        x.A = st->XT[kv];
        x.B = st->YT[kv];
        x.A_lo = st->XT_lo[kv];
        x.B_lo = st->YT_lo[kv];
        x.A_3 = st->XT_3[kv];
        x.B_3 = st->YT_3[kv];
        x.out = st->cross[kv];
        x.da = st->delta[kv];
        x.db = st->delta[2 + kv];
        x.za = st->zbar[kv];
        x.zb = st->zbar[2 + kv];
        x.Ma = st->Fs;
        x.Nb = st->Ft;
        x.ldo = st->Ft;
        x.lower = 0;
    }
}

struct DevGuard {
    int prev = -1;
    explicit DevGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) cudaSetDevice(dev);
    }
    ~DevGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

}  // namespace

extern "C" {

kvb_status kvb_stats_create(kvb_ctx* ctx, kvb_dtype dtype, int64_t max_batch_tokens, kvb_stats** out) {
    g_last_error.clear();
    if (!ctx) {
        if (out) *out = nullptr;
        return fail(KVB_ERR_INVALID_ARG, "NULL argument");
    }
    return kvb_stats_create_block(ctx, dtype, max_batch_tokens, 0, ctx->L_t, out);
}

kvb_status kvb_stats_create_block(kvb_ctx* ctx, kvb_dtype dtype, int64_t max_batch_tokens, int32_t t_begin,
                                  int32_t t_end, kvb_stats** out) {
    g_last_error.clear();
    if (out) *out = nullptr;
    if (!ctx || !out) return fail(KVB_ERR_INVALID_ARG, "NULL argument");
    if (t_begin < 0 || t_end <= t_begin || t_end > ctx->L_t)
        return fail(KVB_ERR_INVALID_ARG, "target block must satisfy 0 <= t_begin < t_end <= L_tgt");
    if (dtype != KVB_F32 && dtype != KVB_BF16) return fail(KVB_ERR_UNSUPPORTED, "dtype must be KVB_F32 or KVB_BF16");
    if (max_batch_tokens < 1 || max_batch_tokens > (int64_t(1) << 30))
        return fail(KVB_ERR_INVALID_ARG, "max_batch_tokens must be in [1, 2^30]");
    DevGuard g(ctx->device);
    kvb_stats* st = new (std::nothrow) kvb_stats();
    if (!st) return fail(KVB_ERR_OOM, "host allocation failed");
    st->ctx = ctx;
    st->dtype = dtype;
    st->max_T = max_batch_tokens;
    st->ld = (max_batch_tokens + 127) & ~int64_t(127);  // whole 128-row gather chunks
    const int64_t q = static_cast<int64_t>(ctx->H) * ctx->d;
    st->Fs = ctx->L_s * q;
    st->t0 = t_begin;
    st->nt = t_end - t_begin;
    st->Ft = st->nt * q;
    kvb_status s = KVB_OK;
    auto A = [&](void** p, size_t bytes) {
        if (s == KVB_OK) s = st_alloc(st, p, bytes);
    };
    A(reinterpret_cast<void**>(&st->n_dev), sizeof(long long));
    A(reinterpret_cast<void**>(&st->nb_dev), sizeof(int));
    A(reinterpret_cast<void**>(&st->coef_dev), 2 * sizeof(float));
    A(reinterpret_cast<void**>(&st->numeric), sizeof(int));
    A(reinterpret_cast<void**>(&st->rows), st->max_T * sizeof(int));
    const int64_t len[4] = {st->Fs, st->Fs, st->Ft, st->Ft};
    for (int m = 0; m < 4; ++m) {
        A(reinterpret_cast<void**>(&st->mean[m]), len[m] * 4);
        A(reinterpret_cast<void**>(&st->bmean[m]), len[m] * 4);
        A(reinterpret_cast<void**>(&st->delta[m]), len[m] * 4);
        A(reinterpret_cast<void**>(&st->zbar[m]), len[m] * 4);
        A(reinterpret_cast<void**>(&st->zsum[m]), len[m] * 4);
        A(reinterpret_cast<void**>(&st->shift[m]), len[m] * 4);
    }
    for (int kv = 0; kv < 2; ++kv) {
        A(reinterpret_cast<void**>(&st->gram[kv]), static_cast<size_t>(st->Fs) * st->Fs * 4);
        A(reinterpret_cast<void**>(&st->cross[kv]), static_cast<size_t>(st->Fs) * st->Ft * 4);
        A(reinterpret_cast<void**>(&st->syy[kv]), st->Ft * 4);
    }
    // Tensor-core statistics when the shapes tile by 128 x 256: bf16 caches as two
    // bf16 parts, fp32 caches as three (unless KVB_STATS_TC_F32=0)
    const char* f32tc = std::getenv("KVB_STATS_TC_F32");
    const bool three = dtype == KVB_F32;
    if (s == KVB_OK && (dtype == KVB_BF16 || !(f32tc && std::strcmp(f32tc, "0") == 0))) {
        StatsJob jobs[4];
        stats_jobs(st, jobs);
        st->use_tc = stats_gemm_tc_supported(jobs, 4);
    }
    for (int kv = 0; kv < 2; ++kv) {
        if (st->use_tc) {
            A(&st->XT[kv], static_cast<size_t>(st->Fs) * st->ld * 2);
            A(&st->XT_lo[kv], static_cast<size_t>(st->Fs) * st->ld * 2);
            A(&st->YT[kv], static_cast<size_t>(st->Ft) * st->ld * 2);
            A(&st->YT_lo[kv], static_cast<size_t>(st->Ft) * st->ld * 2);
            if (three) {
                A(&st->XT_3[kv], static_cast<size_t>(st->Fs) * st->ld * 2);
                A(&st->YT_3[kv], static_cast<size_t>(st->Ft) * st->ld * 2);
            }
        } else {
            A(&st->XT[kv], static_cast<size_t>(st->Fs) * st->ld * 4);
            A(&st->YT[kv], static_cast<size_t>(st->Ft) * st->ld * 4);
        }
    }
    A(reinterpret_cast<void**>(&st->part), static_cast<size_t>(st->ld / 128) * std::max(st->Fs, st->Ft) * 4);
    // one gather launch for all four matrices unless KVB_GATHER_ALL=0 (one launch per matrix)
    const char* gall = std::getenv("KVB_GATHER_ALL");
    if (st->use_tc && gather_all_supported(dtype, ctx->d) && !(gall && std::strcmp(gall, "0") == 0)) {
        A(reinterpret_cast<void**>(&st->part_all), static_cast<size_t>(st->ld / 128) * 2 * (st->Fs + st->Ft) * 4);
        A(reinterpret_cast<void**>(&st->part_sq), static_cast<size_t>(st->ld / 128) * 2 * st->Ft * 4);
    }
    A(reinterpret_cast<void**>(&st->r2), 2ull * ctx->L_t * ctx->L_s * 4);
    A(reinterpret_cast<void**>(&st->sel), 2ull * ctx->L_t * ctx->k * 4);
    if (s == KVB_OK) s = zero_stats(st, 0);
    if (s == KVB_OK && cudaMemset(st->numeric, 0, sizeof(int)) != cudaSuccess)
        s = fail(KVB_ERR_CUDA, "cudaMemset");
    if (s == KVB_OK && st->use_tc) {
        StatsJob jobs[4];
        stats_jobs(st, jobs);
        cudaError_t e = stats_gemm_tc_plan(jobs, 4, &st->plan);
        if (e != cudaSuccess) s = cuda_fail(e, "planning the statistics GEMM");
    }
    if (s == KVB_OK) {
        cudaError_t e = cudaStreamSynchronize(0);
        if (e != cudaSuccess) s = cuda_fail(e, "statistics set-up");
    }
    if (s != KVB_OK) {
        free_stats(st);
        return s;
    }
    *out = st;
    return KVB_OK;
}

kvb_status kvb_stats_destroy(kvb_stats* st) {
    if (!st) return KVB_OK;
    DevGuard g(st->ctx->device);
    cudaDeviceSynchronize();
    free_stats(st);
    return KVB_OK;
}

kvb_status kvb_stats_reset(kvb_stats* st, void* stream) {
    g_last_error.clear();
    if (!st) return fail(KVB_ERR_INVALID_ARG, "stats is NULL");
    DevGuard g(st->ctx->device);
    return zero_stats(st, static_cast<cudaStream_t>(stream));
}

kvb_status kvb_stats_accumulate(kvb_ctx* c, kvb_stats* st, const void* src_k, const void* src_v, const void* tgt_k,
                                const void* tgt_v, const int32_t* positions, int64_t T, int32_t stride,
                                void* stream) {
    g_last_error.clear();
    if (!c || !st) return fail(KVB_ERR_INVALID_ARG, "NULL context or statistics");
    if (st->ctx != c) return fail(KVB_ERR_INVALID_ARG, "statistics belong to another context");
    if (T < 0 || T > st->max_T) return fail(KVB_ERR_INVALID_ARG, "T outside [0, max_batch_tokens]");
    if (stride < 1) return fail(KVB_ERR_INVALID_ARG, "stride must be >= 1");
    kvb_status s;
    if ((s = take_device_error(c)) != KVB_OK) return s;
    if (T == 0) return KVB_OK;
    if ((s = check_device_ptrs({src_k, src_v, tgt_k, tgt_v, positions}, "kvb_stats_accumulate")) != KVB_OK) return s;
    DevGuard g(c->device);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const DevErr err = dev_err(c);
    const kvb_dtype dt = st->dtype;
    const int64_t LsH = static_cast<int64_t>(c->L_s) * c->H, LtH = static_cast<int64_t>(st->nt) * c->H;
    // the block's target layers: [t0, t0 + nt) of the [L_tgt][H][T][d] target caches
    const size_t tgt_off = static_cast<size_t>(st->t0) * c->H * static_cast<size_t>(T) * c->d * (dt == KVB_F32 ? 4 : 2);
    const void* caches[4] = {src_k, src_v, static_cast<const char*>(tgt_k) + tgt_off,
                             static_cast<const char*>(tgt_v) + tgt_off};
    const int64_t slabs[4] = {LsH, LsH, LtH, LtH};
    const float2* tabs[4] = {c->tab_s, nullptr, c->tab_t, nullptr};
    void* outs[4] = {st->XT[0], st->XT[1], st->YT[0], st->YT[1]};
    void* outs_lo[4] = {st->XT_lo[0], st->XT_lo[1], st->YT_lo[0], st->YT_lo[1]};
    void* outs_3[4] = {st->XT_3[0], st->XT_3[1], st->YT_3[0], st->YT_3[1]};
    cudaError_t e;
    {
        ProfScope ps(c, cs, "calib_select_rows");
        e = launch_select_rows(positions, T, stride, c->max_pos, st->rows, st->nb_dev, err, cs);
    }
    if (e != cudaSuccess) return cuda_fail(e, "row selection");
    const bool fused = st->part_all != nullptr;  // one launch for the four matrices, S_yy in the merge
    const bool single = gather_single_pass_ok(dt, c->d);
    if (single) {  // the first batch's own means become the shift (returns at once on later batches)
        ProfScope ps(c, cs, "calib_first_mean");
        FirstMeanArgs fm{};
        for (int m = 0; m < 4; ++m) {
            fm.cache[m] = static_cast<const __nv_bfloat16*>(caches[m]);
            fm.n_slabs[m] = slabs[m];
            fm.tab[m] = tabs[m];
            fm.mean[m] = st->mean[m];
        }
        fm.T = T;
        fm.d = c->d;
        fm.rows = st->rows;
        fm.nb = st->nb_dev;
        fm.n_seen = st->n_dev;
        fm.pos = positions;
        e = launch_first_mean(fm, cs);
        if (e != cudaSuccess) return cuda_fail(e, "first-batch means");
    }
    {
        ProfScope ps(c, cs, "calib_gather_center");
        if (fused) {
            GatherAllArgs ga{};
            int64_t fo = 0, qo = 0;
            for (int m = 0; m < 4; ++m) {
                ga.cache[m] = static_cast<const __nv_bfloat16*>(caches[m]);
                ga.n_slabs[m] = slabs[m];
                ga.foff[m] = fo;
                fo += slabs[m] * c->d;
                ga.qoff[m] = m >= 2 ? qo : -1;
                if (m >= 2) qo += slabs[m] * c->d;
                ga.tab[m] = tabs[m];
                ga.mean_a[m] = st->mean[m];
                ga.shift[m] = st->shift[m];
                ga.out[m] = static_cast<__nv_bfloat16*>(outs[m]);
                ga.out_lo[m] = static_cast<__nv_bfloat16*>(outs_lo[m]);
            }
            ga.T = T;
            ga.ld = st->ld;
            ga.Fall = fo;
            ga.Fsq = qo;
            ga.rows = st->rows;
            ga.nb = st->nb_dev;
            ga.n_seen = st->n_dev;
            ga.pos = positions;
            ga.part = st->part_all;
            ga.part_sq = st->part_sq;
            ga.err = err;
            ga.stride = stride;
            ga.max_pos = c->max_pos;
            e = launch_gather_all(ga, c->num_sms, cs);
        }
        for (int m = 0; m < 4 && e == cudaSuccess && !fused; ++m) {
            GatherArgs g{};
            g.dt = dt;
            g.cache = caches[m];
            g.n_slabs = slabs[m];
            g.T = T;
            g.stride = stride > 1 ? stride : 1;
            g.num_sms = c->num_sms;
            g.d = c->d;
            g.rows = st->rows;
            g.nb = st->nb_dev;
            g.n_seen = st->n_dev;
            g.pos = positions;
            g.tab = tabs[m];
            g.strip = tabs[m] != nullptr;
            g.mean_a = st->mean[m];
            g.shift = st->shift[m];
            g.part = st->part;
            g.zsum = st->zsum[m];
            g.bmean = st->bmean[m];
            g.out = outs[m];
            g.out_lo = outs_lo[m];
            g.out_3 = outs_3[m];
            g.ld = st->ld;
            e = launch_gather(g, cs);
        }
    }
    if (e != cudaSuccess) return cuda_fail(e, "gather/center");
    {
        ProfScope ps(c, cs, "calib_chan_prepare");
        MeanSet ms{};
        if (fused) {
            ms.part = st->part_all;
            ms.part_sq = st->part_sq;
            int64_t fo = 0, qo = 0;
            for (int m = 0; m < 4; ++m) {
                const int64_t w = slabs[m] * c->d;
                ms.foff[m] = fo;
                fo += w;
                ms.qoff[m] = m >= 2 ? qo : -1;
                if (m >= 2) qo += w;
            }
            ms.Fall = fo;
            ms.Fsq = qo;
            ms.syy[0] = st->syy[0];
            ms.syy[1] = st->syy[1];
        }
        for (int m = 0; m < 4; ++m) {
            ms.mean[m] = st->mean[m];
            ms.bmean[m] = st->bmean[m];
            ms.zsum[m] = single ? st->zsum[m] : nullptr;
            ms.shift[m] = single ? st->shift[m] : nullptr;
            ms.delta[m] = st->delta[m];
            ms.zbar[m] = st->zbar[m];
        }
        ms.len[0] = ms.len[1] = st->Fs;
        ms.len[2] = ms.len[3] = st->Ft;
        if (e == cudaSuccess) e = launch_chan_prepare(ms, st->n_dev, st->nb_dev, st->coef_dev, cs);
    }
    if (e != cudaSuccess) return cuda_fail(e, "Chan merge preparation");
    StatsJob jobs[4];
    stats_jobs(st, jobs);
    if (st->use_tc) {
        std::string why;
        ProfScope ps(c, cs, "stats_gemm_tcgen05");
        e = launch_stats_gemm_tc(st->plan, jobs, 4, st->ld, st->coef_dev, st->nb_dev, err, c->num_sms, cs, &why);
        if (e != cudaSuccess && !why.empty()) return fail(KVB_ERR_CUDA, "statistics GEMM: " + why);
    } else {
        ProfScope ps(c, cs, "stats_gemm_simt");
        for (int j = 0; j < 4 && e == cudaSuccess; ++j)
            e = launch_stats_gemm_simt(static_cast<const float*>(jobs[j].A), static_cast<const float*>(jobs[j].B),
                                       st->ld, jobs[j].Ma, jobs[j].Nb, jobs[j].lower != 0, jobs[j].da, jobs[j].db,
                                       jobs[j].za, jobs[j].zb, st->coef_dev, st->nb_dev, jobs[j].out, jobs[j].ldo, cs);
    }
    if (e != cudaSuccess) return cuda_fail(e, "statistics GEMM");
    {
        ProfScope ps(c, cs, "calib_syy_merge");
        for (int kv = 0; kv < 2 && e == cudaSuccess && !fused; ++kv)  // (fused: done in the merge)
            e = launch_syy(st->YT[kv], st->YT_lo[kv], st->YT_3[kv], st->ld, st->Ft, st->nb_dev, st->delta[2 + kv], st->zbar[2 + kv],
                           st->coef_dev, st->syy[kv], cs);
        if (e == cudaSuccess) e = launch_chan_finish(st->n_dev, st->nb_dev, cs);
    }
    if (e != cudaSuccess) return cuda_fail(e, "S_yy / merge");
    mirror_device_error(c, cs);
    return KVB_OK;
}

kvb_status kvb_stats_count(kvb_stats* st, int64_t* n_obs, void* stream) {
    g_last_error.clear();
    if (!st || !n_obs) return fail(KVB_ERR_INVALID_ARG, "NULL argument");
    DevGuard g(st->ctx->device);
    long long n = 0;
    cudaError_t e = cudaMemcpyAsync(&n, st->n_dev, sizeof(n), cudaMemcpyDeviceToHost, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "reading the observation count");
    *n_obs = n;
    return KVB_OK;
}

kvb_status kvb_stats_export(kvb_stats* st, int32_t kv, int64_t* n_obs, float* mean_x, float* mean_y, float* gram,
                            float* cross, float* syy, void* stream) {
    g_last_error.clear();
    if (!st || kv < 0 || kv > 1) return fail(KVB_ERR_INVALID_ARG, "NULL statistics or kv not 0/1");
    DevGuard g(st->ctx->device);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    auto cp = [&](float* dst, const float* src, int64_t n) {
        if (dst && e == cudaSuccess) e = cudaMemcpyAsync(dst, src, n * 4, cudaMemcpyDeviceToDevice, cs);
    };
    cp(mean_x, st->mean[kv], st->Fs);
    cp(mean_y, st->mean[2 + kv], st->Ft);
    cp(cross, st->cross[kv], st->Fs * st->Ft);
    cp(syy, st->syy[kv], st->Ft);
    if (gram && e == cudaSuccess) e = launch_symmetrize(st->gram[kv], gram, st->Fs, cs);
    if (e != cudaSuccess) return cuda_fail(e, "exporting statistics");
    if (n_obs) return kvb_stats_count(st, n_obs, stream);
    return KVB_OK;
}

kvb_status kvb_stats_import(kvb_stats* st, int32_t kv, int64_t n_obs, const float* mean_x, const float* mean_y,
                            const float* gram, const float* cross, const float* syy, void* stream) {
    g_last_error.clear();
    if (!st || kv < 0 || kv > 1) return fail(KVB_ERR_INVALID_ARG, "NULL statistics or kv not 0/1");
    if (n_obs < 0) return fail(KVB_ERR_INVALID_ARG, "n_obs < 0");
    if (!mean_x || !mean_y || !gram || !cross || !syy) return fail(KVB_ERR_INVALID_ARG, "NULL statistics buffer");
    DevGuard g(st->ctx->device);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    auto cp = [&](float* dst, const float* src, int64_t n) {
        if (e == cudaSuccess) e = cudaMemcpyAsync(dst, src, n * 4, cudaMemcpyDeviceToDevice, cs);
    };
    cp(st->mean[kv], mean_x, st->Fs);
    cp(st->mean[2 + kv], mean_y, st->Ft);
    cp(st->gram[kv], gram, st->Fs * st->Fs);
    cp(st->cross[kv], cross, st->Fs * st->Ft);
    cp(st->syy[kv], syy, st->Ft);
    long long n = n_obs;
    if (e == cudaSuccess) e = cudaMemcpyAsync(st->n_dev, &n, sizeof(n), cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return cuda_fail(e, "importing statistics");
    return KVB_OK;
}

kvb_status kvb_layer_select(kvb_ctx* c, kvb_stats* st, double lambda, int32_t* sel_k_host, int32_t* sel_v_host,
                            float* r2_out, void* stream) {
    g_last_error.clear();
    if (!c || !st || !sel_k_host || !sel_v_host) return fail(KVB_ERR_INVALID_ARG, "NULL argument");
    if (st->ctx != c) return fail(KVB_ERR_INVALID_ARG, "statistics belong to another context");
    if (!(lambda >= 0.0)) return fail(KVB_ERR_INVALID_ARG, "lambda must be >= 0");
    if (r2_out && !aligned16(r2_out)) return fail(KVB_ERR_INVALID_ARG, "r2 not 16-byte aligned");
    kvb_status s;
    if ((s = take_device_error(c)) != KVB_OK) return s;
    DevGuard g(c->device);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int q = c->H * c->d;
    const int64_t Ft = st->Ft;
    // The K and V systems of every source layer go through the factorisation and
    // the solves together, as many per batch as the workspace budget holds.
    const int n_sys = 2 * c->L_s;
    const int64_t lq0 = ((q + 63) / 64) * 64 * 64;
    const int64_t per_sys = 4 * (int64_t(q) * Ft + int64_t(q) * q + lq0 + Ft + q) +
                            static_cast<int64_t>(tc_update_ws_bytes(q, Ft, 1));
    const int64_t budget = static_cast<int64_t>(ws_budget());
    int B = static_cast<int>(std::min<int64_t>(n_sys, std::max<int64_t>(1, budget / per_sys)));
    if ((s = ws_grow(st, &st->wsG, &st->wsG_bytes, size_t(B) * q * q * 4)) != KVB_OK) return s;
    if ((s = ws_grow(st, &st->wsR, &st->wsR_bytes, size_t(B) * q * Ft * 4)) != KVB_OK) return s;
    if ((s = ws_grow(st, &st->wsD, &st->wsD_bytes, size_t(B) * q * 4)) != KVB_OK) return s;
    if ((s = ws_grow(st, &st->wsS, &st->wsS_bytes, size_t(B) * Ft * 4)) != KVB_OK) return s;
    const int64_t lq = ((q + 63) / 64) * 64 * 64;  // Linv floats per system
    if ((s = ws_grow(st, &st->wsL, &st->wsL_bytes, size_t(B) * lq * 4)) != KVB_OK) return s;
    if ((s = ws_grow(st, &st->wsT, &st->wsT_bytes, tc_update_ws_bytes(q, Ft, B))) != KVB_OK) return s;
    const TcSolve tc{reinterpret_cast<__nv_bfloat16*>(st->wsT), st->wsT_bytes, dev_err(c), c->num_sms};
    cudaError_t e = cudaMemsetAsync(st->numeric, 0, sizeof(int), cs);
    const float lam = static_cast<float>(lambda);
    {
        ProfScope ps(c, cs, "r2_single_source");
        for (int s0 = 0; s0 < n_sys && e == cudaSuccess; s0 += B) {
            ProfScope pb(c, cs, "r2_solve_batch");
            const int nb = std::min(B, n_sys - s0);
            // the batch's systems of one cache at a time (system i: kv i / L_s, source
            // layer i % L_s), at most MAX_SYS per launch of the per-system kernels
            auto slices = [&](auto&& fn) {
                for (int a = 0; a < nb && e == cudaSuccess;) {
                    const int kv = (s0 + a) / c->L_s;
                    const int end = std::min({nb, (kv + 1) * c->L_s - s0, a + MAX_SYS});
                    SysLayers L;
                    std::memset(&L, 0, sizeof(L));
                    for (int b = a; b < end; ++b) L.layer[b - a][0] = (s0 + b) % c->L_s;
                    e = fn(kv, static_cast<size_t>(a), end - a, L);
                    a = end;
                }
            };
            slices([&](int kv, size_t o, int cnt, const SysLayers& L) {
                cudaError_t r = launch_gather_system(st->gram[kv], st->Fs, L, q, q, lam, st->wsG + o * q * q,
                                                     int64_t(q) * q, st->wsD + o * q, cnt, cs);
                if (r == cudaSuccess)
                    r = launch_gather_rhs(st->cross[kv], Ft, L, q, q, Ft, st->wsD + o * q, st->wsR + o * q * Ft,
                                          int64_t(q) * Ft, cnt, cs);
                return r;
            });
            if (e == cudaSuccess)
                e = chol_factor_batched(st->wsG, q, int64_t(q) * q, q, nb, st->numeric, st->wsL, lq, &tc, cs);
            if (e == cudaSuccess)
                e = chol_solve_batched(st->wsG, q, int64_t(q) * q, q, st->wsL, lq, st->wsR, Ft, int64_t(q) * Ft, Ft, nb,
                                       &tc, cs);
            slices([&](int kv, size_t o, int cnt, const SysLayers& L) {
                cudaError_t r = launch_sse(st->cross[kv], Ft, L, q, q, Ft, st->wsD + o * q, st->wsR + o * q * Ft,
                                           int64_t(q) * Ft, st->syy[kv], lam, st->wsS + o * Ft, cnt, cs);
                if (r == cudaSuccess)
                    r = launch_r2_head(st->wsS + o * Ft, Ft, st->syy[kv], st->nt, c->H, c->d, L,
                                       st->r2 + (size_t(kv) * c->L_t + st->t0) * c->L_s, c->L_s, cnt, cs);
                return r;
            });
        }
        for (int kv = 0; kv < 2 && e == cudaSuccess; ++kv)
            e = launch_topk(st->r2 + (size_t(kv) * c->L_t + st->t0) * c->L_s, st->nt, c->L_s, c->k,
                            st->sel + (size_t(kv) * c->L_t + st->t0) * c->k, cs);
    }
    if (e != cudaSuccess) return cuda_fail(e, "layer selection");
    if (r2_out) {  // the block's rows only
        for (int kv = 0; kv < 2 && e == cudaSuccess; ++kv) {
            const size_t off = (size_t(kv) * c->L_t + st->t0) * c->L_s;
            e = cudaMemcpyAsync(r2_out + off, st->r2 + off, size_t(st->nt) * c->L_s * 4, cudaMemcpyDeviceToDevice, cs);
        }
        if (e != cudaSuccess) return cuda_fail(e, "copying R^2");
    }
    std::vector<int32_t> sel(2ull * c->L_t * c->k);
    int numeric = 0;
    e = cudaMemcpyAsync(sel.data(), st->sel, sel.size() * 4, cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&numeric, st->numeric, sizeof(int), cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return cuda_fail(e, "layer selection");
    const size_t o = size_t(st->t0) * c->k, n_sel = size_t(st->nt) * c->k;
    std::memcpy(sel_k_host + o, sel.data() + o, n_sel * 4);
    std::memcpy(sel_v_host + o, sel.data() + size_t(c->L_t) * c->k + o, n_sel * 4);
    if ((s = take_device_error(c)) != KVB_OK) return s;
    if (numeric) return fail(KVB_ERR_NUMERIC, "a single-source system was not positive definite");
    return KVB_OK;
}

kvb_status kvb_ridge_solve(kvb_ctx* c, kvb_stats* st, const int32_t* sel_k_host, const int32_t* sel_v_host,
                           double lambda, kvb_dtype w_dtype, void* W_k, void* W_v, float* b_k, float* b_v,
                           void* stream) {
    g_last_error.clear();
    if (!c || !st) return fail(KVB_ERR_INVALID_ARG, "NULL context or statistics");
    if (st->ctx != c) return fail(KVB_ERR_INVALID_ARG, "statistics belong to another context");
    if (w_dtype != KVB_F32 && w_dtype != KVB_BF16) return fail(KVB_ERR_UNSUPPORTED, "w_dtype must be KVB_F32 or KVB_BF16");
    if (!(lambda >= 0.0)) return fail(KVB_ERR_INVALID_ARG, "lambda must be >= 0");
    kvb_status s;
    SelTable tab;
    const int t_end = st->t0 + st->nt;  // the statistics' target block
    if ((s = check_selection(c, sel_k_host, "sel_k", &tab, 0, st->t0, t_end)) != KVB_OK) return s;
    if ((s = check_selection(c, sel_v_host, "sel_v", &tab, 1, st->t0, t_end)) != KVB_OK) return s;
    if ((s = check_device_ptrs({W_k, W_v, b_k, b_v}, "kvb_ridge_solve")) != KVB_OK) return s;
    if ((s = take_device_error(c)) != KVB_OK) return s;
    DevGuard g(c->device);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int q = c->H * c->d;
    const int64_t p = static_cast<int64_t>(c->k) * q;
    const size_t wes = w_dtype == KVB_F32 ? 4 : 2;
    // The K and V systems of every target layer go through the factorisation and
    // the solves together, as many per batch as the workspace budget holds.
    const int n_sys = 2 * st->nt;
    const int64_t lp0 = ((p + 63) / 64) * 64 * 64;
    const int64_t per_sys = 4 * (p * p + p * q + lp0 + p) + static_cast<int64_t>(tc_update_ws_bytes(p, q, 1));
    const int64_t budget = static_cast<int64_t>(ws_budget());
    int B = static_cast<int>(std::min<int64_t>(n_sys, std::max<int64_t>(1, budget / per_sys)));
    if ((s = ws_grow(st, &st->wsG, &st->wsG_bytes, size_t(B) * p * p * 4)) != KVB_OK) return s;
    if ((s = ws_grow(st, &st->wsR, &st->wsR_bytes, size_t(B) * p * q * 4)) != KVB_OK) return s;
    if ((s = ws_grow(st, &st->wsD, &st->wsD_bytes, size_t(B) * p * 4)) != KVB_OK) return s;
    const int64_t lp = ((p + 63) / 64) * 64 * 64;  // Linv floats per system
    if ((s = ws_grow(st, &st->wsL, &st->wsL_bytes, size_t(B) * lp * 4)) != KVB_OK) return s;
    if ((s = ws_grow(st, &st->wsT, &st->wsT_bytes, tc_update_ws_bytes(p, q, B))) != KVB_OK) return s;
    const TcSolve tc{reinterpret_cast<__nv_bfloat16*>(st->wsT), st->wsT_bytes, dev_err(c), c->num_sms};
    cudaError_t e = cudaMemsetAsync(st->numeric, 0, sizeof(int), cs);
    const float lam = static_cast<float>(lambda);
    void* Wout[2] = {W_k, W_v};
    float* bout[2] = {b_k, b_v};
    const int32_t* selh[2] = {sel_k_host, sel_v_host};
    {
        ProfScope ps(c, cs, "ridge_solve");
        for (int s0 = 0; s0 < n_sys && e == cudaSuccess; s0 += B) {
            ProfScope pb(c, cs, "ridge_solve_batch");
            const int nb = std::min(B, n_sys - s0);
            // the batch's systems of one cache at a time (system i: kv i / nt, target
            // layer t0 + i % nt), at most MAX_SYS per launch of the per-system kernels
            auto slices = [&](auto&& fn) {
                for (int a = 0; a < nb && e == cudaSuccess;) {
                    const int kv = (s0 + a) / st->nt;
                    const int end = std::min({nb, (kv + 1) * st->nt - s0, a + MAX_SYS});
                    SysLayers L;
                    SysOut O;
                    std::memset(&L, 0, sizeof(L));
                    std::memset(&O, 0, sizeof(O));
                    for (int b = a; b < end; ++b) {
                        const int t = st->t0 + (s0 + b) % st->nt;
                        for (int j = 0; j < c->k; ++j) L.layer[b - a][j] = selh[kv][t * c->k + j];
                        L.col0[b - a] = int64_t(t - st->t0) * q;  // column of the block's statistics
                        O.W[b - a] = static_cast<char*>(Wout[kv]) + size_t(t) * q * p * wes;
                        O.bias[b - a] = bout[kv] + size_t(t) * q;
                    }
                    e = fn(kv, static_cast<size_t>(a), end - a, L, O);
                    a = end;
                }
            };
            slices([&](int kv, size_t o, int cnt, const SysLayers& L, const SysOut&) {
                cudaError_t r = launch_gather_system(st->gram[kv], st->Fs, L, q, p, lam, st->wsG + o * p * p, p * p,
                                                     st->wsD + o * p, cnt, cs);
                if (r == cudaSuccess)
                    r = launch_gather_rhs(st->cross[kv], st->Ft, L, q, p, q, st->wsD + o * p, st->wsR + o * p * q,
                                          p * q, cnt, cs);
                return r;
            });
            if (e == cudaSuccess) e = chol_factor_batched(st->wsG, p, p * p, p, nb, st->numeric, st->wsL, lp, &tc, cs);
            if (e == cudaSuccess)
                e = chol_solve_batched(st->wsG, p, p * p, p, st->wsL, lp, st->wsR, q, p * q, q, nb, &tc, cs);
            slices([&](int kv, size_t o, int cnt, const SysLayers& L, const SysOut& O) {
                cudaError_t r =
                    launch_write_w(w_dtype, st->wsR + o * p * q, p * q, st->wsD + o * p, p, q, O, cnt, cs);
                if (r == cudaSuccess)
                    r = launch_bias(st->wsR + o * p * q, p * q, st->wsD + o * p, p, q, L, q, st->mean[kv],
                                    st->mean[2 + kv], O, cnt, cs);
                return r;
            });
        }
    }
    if (e != cudaSuccess) return cuda_fail(e, "ridge solve");
    int numeric = 0;
    e = cudaMemcpyAsync(&numeric, st->numeric, sizeof(int), cudaMemcpyDeviceToHost, cs);
    if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return cuda_fail(e, "ridge solve");
    if (numeric) return fail(KVB_ERR_NUMERIC, "a ridge system was not positive definite");
    return take_device_error(c);
}

}  // extern "C"
