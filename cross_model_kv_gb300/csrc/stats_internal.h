// Internal declarations of the statistics, selection and ridge-solve kernels.
#pragma once

#include <string>

#include "kvb_internal.h"

namespace kvb {

// Four running-mean vectors: source keys, source values, target keys, target values.
// zsum/shift are set (single-pass path) or NULL (generic path, bmean used).
// With part set (the four-matrix gather), the column sums are the per-chunk
// partial sums part[chunk][foff[m] + c] added in chunk order, and the targets'
// S_yy is updated here from part_sq[chunk][qoff[m] + c] (no separate pass).
struct MeanSet {
    float* mean[4];
    const float* bmean[4];
    const float* zsum[4];
    const float* shift[4];
    float* delta[4];
    float* zbar[4];
    int64_t len[4];
    const float* part;
    const float* part_sq;
    int64_t foff[4], qoff[4], Fall, Fsq;
    float* syy[2];
};

// One batch of all four matrices (bf16 caches, head_dim 128) in one launch:
// kept rows stripped (keys), shifted, written feature-major as bf16 (hi, lo);
// per-chunk column sums into part, per-chunk target sums of squares into part_sq.
struct GatherAllArgs {
    const __nv_bfloat16* cache[4];  // [n_slabs][T][128]
    int64_t n_slabs[4];
    int64_t foff[4];                // columns of matrix m in a row of part
    int64_t qoff[4];                // columns of matrix m in a row of part_sq, -1 for sources
    const float2* tab[4];           // RoPE table (keys) or NULL (values)
    const float* mean_a[4];         // running means before the batch
    float* shift[4];                // shift used, written
    __nv_bfloat16* out[4];          // [n_slabs*128][ld]
    __nv_bfloat16* out_lo[4];
    int64_t T, ld, Fall, Fsq;
    const int* rows;                // kept rows, [nb]
    const int* nb;
    const long long* n_seen;
    const int* pos;
    float* part;                    // [chunks][Fall]
    float* part_sq;                 // [chunks][Fsq]
    DevErr err;
    int stride;                     // kept positions are multiples of it
    int max_pos;                    // rows of the RoPE tables
};
bool gather_all_supported(kvb_dtype dt, int d);
// tab_src / tab_tgt: the two RoPE tables (keys of matrices 0 and 2).
cudaError_t launch_gather_all(const GatherAllArgs& a, int num_sms, cudaStream_t s);

// One matrix of one batch: kept rows of `cache` [n_slabs][T][d] -> centered,
// transposed operand out ([n_slabs*d][ld]; float32, or bf16 hi/lo if out_lo).
struct GatherArgs {
    kvb_dtype dt;
    const void* cache;
    int64_t n_slabs, T;
    int stride;               // positions kept: multiples of stride (sizes the single-pass grid)
    int num_sms;
    int d;
    const int* rows;
    const int* nb;
    const long long* n_seen;  // observations merged before this batch
    const int* pos;
    const float2* tab;        // RoPE table (keys), or NULL
    bool strip;
    const float* mean_a;      // running mean before the batch (single-pass shift)
    float* shift;             // [n_slabs*d] shift used (single-pass path)
    float* part;              // [T/64][n_slabs*d] per-chunk column sums (single-pass path)
    float* zsum;              // [n_slabs*d] column sums of z (single-pass path)
    float* bmean;             // [n_slabs*d] batch mean (generic path)
    void* out;
    void* out_lo;
    void* out_3;              // third bf16 part (fp32 caches on the tensor-core path), or NULL
    int64_t ld;
};
bool gather_single_pass_ok(kvb_dtype dt, int d);

// First batch only (device count *n_seen == 0): mean[m] = the column means of
// the batch's first 128 kept rows (keys stripped), the shift of the
// single-pass gathers.
struct FirstMeanArgs {
    const __nv_bfloat16* cache[4];
    int64_t n_slabs[4];
    const float2* tab[4];
    float* mean[4];
    int64_t T;
    int d;
    const int* rows;
    const int* nb;
    const long long* n_seen;
    const int* pos;
};
cudaError_t launch_first_mean(const FirstMeanArgs& a, cudaStream_t s);
cudaError_t launch_gather(const GatherArgs& g, cudaStream_t s);

cudaError_t launch_select_rows(const int* pos, int64_t T, int stride, int max_pos, int* rows, int* nb, DevErr err,
                               cudaStream_t s);
// coef = {f = n_a n_b / n, g = n_b}
cudaError_t launch_chan_prepare(const MeanSet& ms, const long long* n_dev, const int* nb, float* coef,
                                cudaStream_t s);
cudaError_t launch_symmetrize(const float* src, float* dst, int64_t n, cudaStream_t s);
cudaError_t launch_chan_finish(long long* n_dev, const int* nb, cudaStream_t s);
cudaError_t launch_syy(const void* Y, const void* Ylo, const void* Y3, int64_t ld, int64_t rows_n, const int* nb, const float* dy,
                       const float* zy, const float* coef, float* syy, cudaStream_t s);
cudaError_t launch_stats_gemm_simt(const float* A, const float* B, int64_t ld, int64_t Ma, int64_t Nb, bool lower,
                                   const float* da, const float* db, const float* za, const float* zb,
                                   const float* coef, const int* nb, float* out, int64_t ldo, cudaStream_t s);

// Statistics GEMM jobs, K = observations:
//   out[i][j] += sum_r A[i][r] B[j][r] - g za[i] zb[j] + f da[i] db[j].
// CUDA-core path: A, B float32 [rows][ld].  Tensor-core path, bf16 caches: A =
// A + A_lo and B = B + B_lo as bf16 pairs; the product is taken as A.B + A.B_lo
// + A_lo.B (three bf16 passes into one fp32 accumulator; A_lo.B_lo is below fp32
// noise).  Tensor-core path, fp32 caches: three parts A + A_lo + A_3 (24
// significant bits) and the six products down to 2^-16 of the leading one.
struct StatsJob {
    const void* A;   // [Ma][ld]
    const void* B;   // [Nb][ld]
    const void* A_lo;
    const void* B_lo;
    const void* A_3;  // third parts, or NULL (two-part operands)
    const void* B_3;
    float* out;      // [Ma][ldo]
    const float* da;
    const float* db;
    const float* za;
    const float* zb;
    int64_t Ma, Nb, ldo;
    int lower;       // only tiles touching the lower triangle (j <= i)
};
struct StatsGemmPlan;  // device tile list, built once per statistics object
bool stats_gemm_tc_supported(const StatsJob* jobs, int n_jobs);
cudaError_t stats_gemm_tc_plan(const StatsJob* jobs, int n_jobs, StatsGemmPlan** plan);
void stats_gemm_tc_free(StatsGemmPlan* plan);
cudaError_t launch_stats_gemm_tc(StatsGemmPlan* plan, const StatsJob* jobs, int n_jobs, int64_t ld,
                                 const float* coef, const int* nb, DevErr err, int num_sms, cudaStream_t s,
                                 std::string* why);

// ---------------------------------------------------------------- dense solves (fp32, batched)
// C[b] = alpha * op(A[b]) op(B[b]) + beta * C[b];  A(m,k) = A[m*sam + k*sak],
// B(k,n) = B[k*sbk + n*sbn], C(m,n) = C[m*ldc + n].  lower: skip tiles above the diagonal.
struct GemmArgs {
    const float* A;
    const float* B;
    float* C;
    int64_t sam, sak, sbk, sbn, ldc;
    int64_t strideA, strideB, strideC;  // per batch item
    int64_t M, N, K;
    float alpha, beta;
    int batch;
    int lower;
};
cudaError_t launch_gemm_f32(const GemmArgs& g, cudaStream_t s);

// In-place blocked Cholesky of batch SPD matrices (lower triangle used; 256-wide
// super-panels of four 64-wide steps), then in-place solve of G X = C for m
// right-hand sides.  The factor also leaves the inverse of every 64 x 64 diagonal block in Linv
// ([batch][n/64 * 64][64], strideL floats per system), so both triangular
// solves run as GEMMs.  A non-positive pivot sets *numeric_flag.
// Rank <= 256 updates on the tensor cores with fp32 operands carried as three
// bf16 parts (solve_tc_sm103.cu).  An operand is rows x K (K <= 256) fp32 with
// element (r, k) of batch item b at src[b * s_batch + r * s_row + k * s_k].
struct TcOperand {
    const float* src;
    int64_t rows, s_row, s_k, s_batch;
};
struct TcSolve {
    __nv_bfloat16* ws;  // split operands, tc_update_ws_bytes()
    size_t ws_bytes;
    DevErr err;
    int num_sms;
};
size_t tc_update_ws_bytes(int64_t rows_a, int64_t rows_b, int batch);
bool tc_update_supported(const TcSolve* tc, int64_t M, int64_t N, int K, const float* C, int64_t ldc);
// An operand already split into its three bf16 parts: part i of row r of batch item
// b at base[i * part + (b * rows + r) * ld + k], k < K (16-byte aligned base, ld a
// multiple of 8).
struct TcPreSplit {
    __nv_bfloat16* base;
    int64_t part, ld;
};
// Split K columns of an operand into `dst` (K <= 64 columns, zero-padded to 64).
cudaError_t tc_split_into(const TcOperand& o, int K, int batch, const TcPreSplit& dst, cudaStream_t s);
// C[b] = alpha * A[b] B[b]^T + beta * C[b] (B == NULL: B = A); lower skips tiles above the diagonal.
// With pre_b, B's parts are read from there (B->rows still gives its row count).
cudaError_t launch_tc_update(const TcSolve& tc, const TcOperand& A, const TcOperand* B, int K, float* C, int64_t ldc,
                             int64_t strideC, float alpha, float beta, bool lower, int batch, cudaStream_t s,
                             std::string* why, const TcPreSplit* pre_b = nullptr);

// tc (may be NULL): run the large updates on the tensor cores.
cudaError_t chol_factor_batched(float* G, int64_t ldg, int64_t strideG, int64_t n, int batch, int* numeric_flag,
                                float* Linv, int64_t strideL, const TcSolve* tc, cudaStream_t s);
cudaError_t chol_solve_batched(const float* L, int64_t ldg, int64_t strideG, int64_t n, const float* Linv,
                               int64_t strideL, float* C, int64_t ldc, int64_t strideC, int64_t m, int batch,
                               const TcSolve* tc, cudaStream_t s);

}  // namespace kvb
