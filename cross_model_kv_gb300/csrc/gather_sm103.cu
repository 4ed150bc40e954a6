// Calibration gather of one batch, all four matrices in one launch (bf16
// caches, head_dim 128): source keys, source values, target keys, target
// values.  For every kept row (a token whose position is a multiple of the
// stride) and every (layer, head) slab, keys are RoPE-stripped with their own
// model's theta, every value is shifted by a per-feature shift known before
// the pass (the running mean; on the first batch the batch's own column
// means, from a pre-pass), and the centered values are written feature-major as a bf16 pair
// (hi, lo) for the tensor-core statistics ("KVBridge" README, "Loading":
// stride-sampled, centered statistics merged batch by batch).  The same pass
// produces the column sums of the centered values (for the Chan merge) and,
// for the targets, their sums of squares (S_yy), as per-chunk partial sums
// that the merge kernel adds up in a fixed order.
//
// Work items (matrix, 128-row chunk, slab) are ordered matrix-major, then
// chunk, then slab, and split into one contiguous range per CTA (one CTA per
// SM).  Warp 0 copies: per item the chunk's kept rows of the slab and the
// slab's 128 shifts (the running means) into one of four stages, and per
// (key matrix, chunk) the chunk's RoPE table rows; all of it completes on
// mbarriers.  When a chunk's kept rows are evenly spaced by the stride (every
// chunk inside one sequence), its rows come in two or four TMA tensor copies
// that step the token coordinate by the stride (element strides of the tensor
// map), and so do its table rows when its positions are evenly spaced too;
// other chunks (sequence boundaries, packed short sequences) take one bulk
// copy per row, which costs the copy engine far more per byte.  Warps 1-16
// each strip, center and store 16 rows x 32 RoPE pairs of an item and leave
// their per-feature sums in the stage; warp 0 adds the eight row groups up (in
// order) when it refills the stage.  The consumer warps never wait on each
// other.
#include <cstring>

#include "stats_internal.h"

namespace kvb {
namespace {

constexpr int GD = 128;                 // head_dim
constexpr int GHALF = GD / 2;           // RoPE pairs
constexpr int GROWS = 128;              // kept rows per chunk
constexpr int GSTAGES = 4;
constexpr int GGROUPS = 8;              // row groups of 16 rows
constexpr int GCONS = 2 * GGROUPS;      // consumer warps: (row group, half of the RoPE pairs)
constexpr int GTHREADS = 32 * (1 + GCONS);
constexpr int GRPW = GROWS / GGROUPS;   // rows per consumer warp
static_assert(GRPW == 16, "one 32-byte output run per feature and warp");

constexpr size_t G_RAW = static_cast<size_t>(GROWS) * GD * 2;         // 32 KB per stage
constexpr size_t G_TAB = static_cast<size_t>(GROWS) * GHALF * 8;      // 64 KB
constexpr size_t G_SHIFT = GD * 4;                                    // 512 B per stage
constexpr size_t G_SUMS = static_cast<size_t>(GGROUPS) * GD * 4;      // 4 KB per stage (and as much for squares)
constexpr size_t G_OFF_TAB = GSTAGES * G_RAW;
constexpr size_t G_OFF_SHIFT = G_OFF_TAB + G_TAB;
constexpr size_t G_OFF_SUMS = G_OFF_SHIFT + GSTAGES * G_SHIFT;
constexpr size_t G_OFF_SQS = G_OFF_SUMS + GSTAGES * G_SUMS;
constexpr size_t G_OFF_BAR = G_OFF_SQS + GSTAGES * G_SUMS;
constexpr size_t G_OFF_RING = G_OFF_BAR + 2 * GSTAGES * 8 + 16 + 16;  // barriers, abort flag (padded)
constexpr size_t G_SMEM = G_OFF_RING + GSTAGES * 16;                  // where each stage's sums go
static_assert(G_SMEM <= 227 * 1024, "shared memory of one CTA");

// Item geometry of one batch, from the kept-row count on the device.
struct Geo {
    int n;              // kept rows
    int nchunks;
    int64_t base[5];    // first item of each matrix; base[4] = all items
};

// (matrix, chunk, slab) of an item, stepped one item at a time; ns caches the
// current matrix's slab count (parameter arrays indexed at run time are read
// through generic loads, so they are read only when the matrix changes).
struct Cursor {
    int m, chunk;
    int64_t slab, ns;
    __device__ void init(const GatherAllArgs& a, const Geo& g, int64_t it) {
        m = 0;
        while (m < 3 && it >= g.base[m + 1]) ++m;
        ns = a.n_slabs[m];
        const int64_t local = it - g.base[m];
        chunk = static_cast<int>(local / ns);
        slab = local % ns;
    }
    __device__ void next(const GatherAllArgs& a, const Geo& g) {
        if (++slab < ns) return;
        slab = 0;
        if (++chunk < g.nchunks) return;
        chunk = 0;
        if (++m < 4) ns = a.n_slabs[m];
    }
};

// Where the partial sums of a stage's item go: part + sum_off and part_sq + sq_off (-1: none).
struct __align__(16) SumDest {
    int64_t sum_off, sq_off;
};

// Tensor maps of the four caches ([slabs][T][128] bf16, box 128 x rows*stride x 1,
// element strides 1 x stride x 1) and of the two RoPE tables ([max_pos][128]
// fp32, box 128 x rows*stride, element strides 1 x stride).  rows = 0: none.
struct GatherMaps {
    CUtensorMap cache[4];
    CUtensorMap tab[4];  // [0] source keys, [2] target keys
    int rows;            // kept rows per tensor copy: 64 (stride <= 4), 32 (stride <= 8), 0 (no tensor copies)
};

__device__ __forceinline__ void tma_load_2d_f(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y) {
    tma_load_2d(dst, m, bar, x, y);
}

__global__ void __launch_bounds__(GTHREADS, 1) gather_all_kernel(const __grid_constant__ GatherAllArgs A,
                                                                 const __grid_constant__ GatherMaps M) {
    extern __shared__ __align__(128) uint8_t sm[];
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + G_OFF_BAR);
    uint64_t* empty = full + GSTAGES;
    uint64_t* tab_full = empty + GSTAGES;
    uint64_t* tab_empty = tab_full + 1;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tab_empty + 1);
    float2* stab = reinterpret_cast<float2*>(sm + G_OFF_TAB);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    Geo G;
    G.n = *A.nb;
    G.nchunks = (G.n + GROWS - 1) / GROWS;
    G.base[0] = 0;
#pragma unroll
    for (int m = 0; m < 4; ++m) G.base[m + 1] = G.base[m] + static_cast<int64_t>(G.nchunks) * A.n_slabs[m];
    const int64_t total = G.base[4];
    const int64_t per = (total + gridDim.x - 1) / gridDim.x;
    const int64_t it0 = blockIdx.x * per;
    const int64_t it1 = it0 + per < total ? it0 + per : total;
    const int mine = it0 < it1 ? static_cast<int>(it1 - it0) : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < GSTAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, GCONS);
        }
        mbar_init(tab_full, 1);
        mbar_init(tab_empty, GCONS);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (mine == 0) return;
    const DevErr& err = A.err;

    if (warp == 0) {
        // ------------------------------------------------------------ copy warp
        Cursor cur;
        cur.init(A, G, it0);
        SumDest* ring = reinterpret_cast<SumDest*>(sm + G_OFF_RING);  // where each stage's sums go
        int loaded = -1;       // table run in shared memory
        int reg_chunk = -1;    // chunk whose spacing was checked
        bool reg_rows = false, reg_pos = false;
        int tok0 = 0, p0 = 0;
        uint32_t te_par = 0;   // next phase of tab_empty to wait for
        int issued = 0;
        bool ok = true;
        // the current matrix's parameters
        int pm = -1;
        const __nv_bfloat16* p_cache = nullptr;
        const float* p_mean = nullptr;
        const float2* p_tab = nullptr;
        const CUtensorMap* p_map = nullptr;
        const CUtensorMap* p_tmap = nullptr;
        int64_t p_foff = 0, p_qoff = -1;
        auto reduce = [&](int s) {  // the eight row groups' sums of the stage's item, in order
            const SumDest dst = ring[s];
            const float4* sums = reinterpret_cast<const float4*>(sm + G_OFF_SUMS + s * G_SUMS);
            float4 a = sums[lane];
#pragma unroll
            for (int w = 1; w < GGROUPS; ++w) {
                const float4 b = sums[w * (GD / 4) + lane];
                a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
            }
            *reinterpret_cast<float4*>(A.part + dst.sum_off + 4 * lane) = a;
            if (dst.sq_off >= 0) {
                const float4* sq = reinterpret_cast<const float4*>(sm + G_OFF_SQS + s * G_SUMS);
                float4 q = sq[lane];
#pragma unroll
                for (int w = 1; w < GGROUPS; ++w) {
                    const float4 b = sq[w * (GD / 4) + lane];
                    q.x += b.x; q.y += b.y; q.z += b.z; q.w += b.w;
                }
                *reinterpret_cast<float4*>(A.part_sq + dst.sq_off + 4 * lane) = q;
            }
        };
        for (int j = 0; j < mine; ++j, cur.next(A, G)) {
            const int s = j % GSTAGES, use = j / GSTAGES;
            if (use > 0 && !mbar_wait(empty + s, (use - 1) & 1, err, abort_flag)) {
                ok = false;
                break;
            }
            const int m = cur.m;
            if (m != pm) {
                pm = m;
                p_cache = A.cache[m];
                p_mean = A.mean_a[m];
                p_tab = A.tab[m];
                p_map = &M.cache[m];
                p_tmap = &M.tab[m];
                p_foff = A.foff[m];
                p_qoff = A.qoff[m];
            }
            const int r0 = cur.chunk * GROWS;
            const int nvalid = G.n - r0 < GROWS ? G.n - r0 : GROWS;
            uint8_t* raw = sm + s * G_RAW;
            float* shift = reinterpret_cast<float*>(sm + G_OFF_SHIFT + s * G_SHIFT);
            const __nv_bfloat16* slab_base = p_cache + cur.slab * A.T * GD;
            if (cur.chunk != reg_chunk) {  // are this chunk's rows (and positions) evenly spaced?
                reg_chunk = cur.chunk;
                tok0 = __ldg(A.rows + r0);
                p0 = __ldg(A.pos + tok0);
                bool okr = M.rows > 0, okp = M.rows > 0;
                for (int t = lane; t < nvalid; t += 32) {
                    const int row = __ldg(A.rows + r0 + t);
                    okr = okr && row == tok0 + t * A.stride;
                    okp = okp && __ldg(A.pos + row) == p0 + t * A.stride;
                }
                reg_rows = __all_sync(0xffffffffu, okr);
                reg_pos = __all_sync(0xffffffffu, okp);
            }
            if (reg_rows) {  // GROWS / M.rows tensor copies, every box full (rows past T read as zeros)
                if (lane == 0) {
                    mbar_expect_tx(full + s, GROWS * GD * 2 + G_SHIFT);
                    for (int b = 0; b < GROWS / M.rows; ++b)
                        tma_load_3d(raw + b * M.rows * GD * 2, p_map, full + s, 0,
                                    tok0 + b * M.rows * A.stride, static_cast<int>(cur.slab));
                }
            } else {
                if (lane == 0) mbar_expect_tx(full + s, nvalid * GD * 2 + G_SHIFT);
                __syncwarp();
                for (int t = lane; t < nvalid; t += 32) {
                    const int row = __ldg(A.rows + r0 + t);
                    bulk_g2s(raw + t * GD * 2, slab_base + static_cast<int64_t>(row) * GD, GD * 2, full + s);
                }
            }
            if (lane == 0) bulk_g2s(shift, p_mean + cur.slab * GD, G_SHIFT, full + s);
            if (use > 0) reduce(s);  // the stage's previous item (its sums are not copied over)
            __syncwarp();  // every lane has read the stage's previous item
            if (lane == 0) {
                const int64_t col = cur.slab * GD;
                ring[s] = SumDest{static_cast<int64_t>(cur.chunk) * A.Fall + p_foff + col,
                                  p_qoff >= 0 ? static_cast<int64_t>(cur.chunk) * A.Fsq + p_qoff + col : -1};
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(full + s);
            ++issued;
            const int key = p_tab ? m * 65536 + cur.chunk : -1;  // table run: (key matrix, chunk)
            if (key >= 0 && key != loaded) {  // this item starts a new table run
                if (loaded >= 0) {
                    if (!mbar_wait(tab_empty, te_par, err, abort_flag)) {
                        ok = false;
                        break;
                    }
                    te_par ^= 1;
                }
                if (reg_pos) {  // positions p0, p0 + stride, ...: tensor copies of the table rows
                    if (lane == 0) {
                        mbar_expect_tx(tab_full, GROWS * GHALF * 8);
                        for (int b = 0; b < GROWS / M.rows; ++b)
                            tma_load_2d_f(stab + b * M.rows * GHALF, p_tmap, tab_full, 0,
                                          p0 + b * M.rows * A.stride);
                    }
                } else {
                    if (lane == 0) mbar_expect_tx(tab_full, nvalid * GHALF * 8);
                    __syncwarp();
                    for (int t = lane; t < nvalid; t += 32) {
                        const int p = __ldg(A.pos + __ldg(A.rows + r0 + t));
                        bulk_g2s(stab + t * GHALF, p_tab + static_cast<int64_t>(p) * GHALF, GHALF * 8, tab_full);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(tab_full);
                loaded = key;
            }
        }
        if (ok) {  // sums of the last items
            for (int j = mine - GSTAGES > 0 ? mine - GSTAGES : 0; j < mine; ++j) {
                const int s = j % GSTAGES;
                if (!mbar_wait(empty + s, (j / GSTAGES) & 1, err, abort_flag)) {
                    ok = false;
                    break;
                }
                reduce(s);
            }
        }
        if (!ok) {  // a wait gave up: let this CTA's copies land before it exits
            const uint64_t limit = err.timeout_ns + 1000000000ull;
            for (int j = issued - GSTAGES > 0 ? issued - GSTAGES : 0; j < issued; ++j)
                mbar_wait_drain(full + j % GSTAGES, (j / GSTAGES) & 1, limit);
        }
        return;
    }

    // ---------------------------------------------------------------- consumer warps
    const int q = (warp - 1) >> 1;                // rows q*16 .. q*16 + 15 of each chunk
    const int i = ((warp - 1) & 1) * 32 + lane;   // RoPE pair (i, i + 64): features i and 64 + i
    Cursor cur;
    cur.init(A, G, it0);
    int cons_key = -1;
    uint32_t tf_par = 0;
    // the current matrix's parameters
    int pm = -1;
    bool p_strip = false, p_target = false;
    __nv_bfloat16* p_out = nullptr;
    __nv_bfloat16* p_lo = nullptr;
    float* p_shift = nullptr;
    for (int j = 0; j < mine; ++j) {
        const int s = j % GSTAGES;
        if (!mbar_wait(full + s, (j / GSTAGES) & 1, err, abort_flag)) return;
        const int m = cur.m;
        if (m != pm) {
            pm = m;
            p_strip = A.tab[m] != nullptr;
            p_target = A.qoff[m] >= 0;
            p_out = A.out[m];
            p_lo = A.out_lo[m];
            p_shift = A.shift[m];
        }
        const int key = p_strip ? m * 65536 + cur.chunk : -1;  // table run: (key matrix, chunk)
        if (key >= 0 && key != cons_key) {
            if (!mbar_wait(tab_full, tf_par, err, abort_flag)) return;
            tf_par ^= 1;
            cons_key = key;
        }
        const bool strip = key >= 0;
        const int r0 = cur.chunk * GROWS;
        const int nvalid = G.n - r0 < GROWS ? G.n - r0 : GROWS;
        const __nv_bfloat16* raw = reinterpret_cast<const __nv_bfloat16*>(sm + s * G_RAW);
        const float* shift = reinterpret_cast<const float*>(sm + G_OFF_SHIFT + s * G_SHIFT);
        const float shl = shift[i], shh = shift[GHALF + i];
        const int64_t f0 = cur.slab * GD;
        const int64_t F_m = A.n_slabs[m] * GD;  // features of this matrix
        if (cur.chunk == 0 && q == 0 && KVB_IN_BOUNDS(err, f0 + i, GHALF + 1, F_m)) {
            p_shift[f0 + i] = shl;
            p_shift[f0 + GHALF + i] = shh;
        }
        // centered values z = (stripped) value - shift; rows past the batch's kept rows are 0
        float z[2][GRPW];
#pragma unroll
        for (int u = 0; u < GRPW; ++u) {
            const int t = q * GRPW + u;
            const float x = __bfloat162float(raw[t * GD + i]);
            const float y = __bfloat162float(raw[t * GD + GHALF + i]);
            if (strip) {  // a = x c + y s, b = y c - x s, shift folded into the FMAs
                const float2 cs = stab[t * GHALF + i];
                z[0][u] = fmaf(x, cs.x, fmaf(y, cs.y, -shl));
                z[1][u] = fmaf(y, cs.x, fmaf(-x, cs.y, -shh));
            } else {
                z[0][u] = x - shl;
                z[1][u] = y - shh;
            }
        }
        if (q * GRPW + GRPW > nvalid) {  // the batch's last, partial chunk
#pragma unroll
            for (int u = 0; u < GRPW; ++u) {
                if (q * GRPW + u >= nvalid) z[0][u] = z[1][u] = 0.f;
            }
        }
        float sum[2] = {0.f, 0.f};
        float sq[2] = {0.f, 0.f};
        const bool target = p_target;
#pragma unroll
        for (int f = 0; f < 2; ++f) {
#pragma unroll
            for (int u = 0; u < GRPW; ++u) sum[f] += z[f][u];
            if (target) {  // S_yy terms
#pragma unroll
                for (int u = 0; u < GRPW; ++u) sq[f] = fmaf(z[f][u], z[f][u], sq[f]);
            }
        }
#pragma unroll
        for (int f = 0; f < 2; ++f) {
            const int64_t o = (f0 + f * GHALF + i) * A.ld + r0 + q * GRPW;
            if (!KVB_IN_BOUNDS(err, o, GRPW, F_m * A.ld)) continue;
            uint32_t hw[8], lw[8];
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(z[f][2 * w], z[f][2 * w + 1]);
                const float2 hv = __bfloat1622float2(h);
                hw[w] = *reinterpret_cast<const uint32_t*>(&h);
                lw[w] = pack_bf16x2(z[f][2 * w] - hv.x, z[f][2 * w + 1] - hv.y);
            }
            st_global_v8(p_out + o, hw);
            st_global_v8(p_lo + o, lw);
        }
        float* ssum = reinterpret_cast<float*>(sm + G_OFF_SUMS + s * G_SUMS) + q * GD;
        ssum[i] = sum[0];
        ssum[GHALF + i] = sum[1];
        if (target) {
            float* ssq = reinterpret_cast<float*>(sm + G_OFF_SQS + s * G_SUMS) + q * GD;
            ssq[i] = sq[0];
            ssq[GHALF + i] = sq[1];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + s);
        const int chunk = cur.chunk;
        cur.next(A, G);
        if (strip && (j + 1 == mine || cur.m != m || cur.chunk != chunk)) {  // last item of this table run
            if (lane == 0) mbar_arrive(tab_empty);
        }
    }
}

}  // namespace

bool gather_all_supported(kvb_dtype dt, int d) { return dt == KVB_BF16 && d == GD; }

namespace {

bool encode_strided(CUtensorMap* m, CUtensorMapDataType dt, uint32_t rank, const void* base, const cuuint64_t* dims,
                    const cuuint64_t* strides, const cuuint32_t* box, const cuuint32_t* estr) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) return false;
    return enc(m, dt, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gather_all(const GatherAllArgs& a, int num_sms, cudaStream_t s) {
    GatherMaps M;
    std::memset(&M, 0, sizeof(M));
    // a tensor copy traverses at most 256 tokens: 64 kept rows at stride <= 4, 32 at stride <= 8
    M.rows = a.stride <= 4 ? 64 : (a.stride <= 8 ? 32 : 0);
    const cuuint32_t span = static_cast<cuuint32_t>(M.rows * a.stride);
    for (int m = 0; m < 4 && M.rows > 0; ++m) {
        const cuuint64_t dims[3] = {GD, static_cast<cuuint64_t>(a.T), static_cast<cuuint64_t>(a.n_slabs[m])};
        const cuuint64_t strides[2] = {GD * 2, static_cast<cuuint64_t>(a.T) * GD * 2};
        const cuuint32_t box[3] = {GD, span, 1};
        const cuuint32_t estr[3] = {1, static_cast<cuuint32_t>(a.stride), 1};
        bool ok = encode_strided(&M.cache[m], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.cache[m], dims, strides, box, estr);
        if (ok && a.tab[m]) {
            const cuuint64_t tdims[2] = {GD, static_cast<cuuint64_t>(a.max_pos)};  // (c, s) of 64 pairs per row
            const cuuint64_t tstrides[1] = {GD * 4};
            const cuuint32_t tbox[2] = {GD, span};
            const cuuint32_t testr[2] = {1, static_cast<cuuint32_t>(a.stride)};
            ok = encode_strided(&M.tab[m], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.tab[m], tdims, tstrides, tbox, testr);
        }
        if (!ok) M.rows = 0;  // every chunk takes the per-row copies
    }
    cudaError_t e = cudaFuncSetAttribute(gather_all_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(G_SMEM));
    if (e != cudaSuccess) return e;
    gather_all_kernel<<<static_cast<unsigned>(num_sms), GTHREADS, G_SMEM, s>>>(a, M);
    return cudaGetLastError();
}

}  // namespace kvb
