// Internal declarations shared by the host side of libkvb and its kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <cstdint>
#include <string>

#include "../../include/kvb.h"
#include "sm103_ptx.cuh"

namespace kvb {

constexpr int MAX_LT = 128;  // target layers a context can describe
constexpr int MAX_LS = 255;  // source layers (selection entries are bytes)
constexpr int MAX_K = 16;    // top_k

// Selection table passed by value to kernels: [kv][target layer][j].
struct SelTable {
    uint8_t s[2][MAX_LT][MAX_K];
};

struct Shape {
    int L_s, L_t, H, d, k;
    int64_t T;
    int max_pos;
};

// ------------------------------------------------------------ launchers
// RoPE cos/sin table: tab[p][i] = (cos(p w_i), sin(p w_i)), w_i = theta^(-2i/d).
cudaError_t launch_rope_table(float2* tab, int max_pos, int d, double theta, cudaStream_t s);

// Strip source RoPE from bf16 keys [LH][T][d] into `out` (same layout).
cudaError_t launch_strip_bf16(const __nv_bfloat16* in, __nv_bfloat16* out, const int* pos,
                              const float2* tab, int64_t LH, int64_t T, int d, int max_pos,
                              DevErr err, int num_sms, cudaStream_t s);

// fp32 operands as bf16 (hi, lo) pairs for the tensor-core map: strip fp32
// keys [LH][T][d] and split them; split n fp32 values (n % 8 == 0).
cudaError_t launch_strip_split_f32(const float* in, __nv_bfloat16* hi, __nv_bfloat16* lo, const int* pos,
                                   const float2* tab, int64_t LH, int64_t T, int d, int max_pos, DevErr err,
                                   int num_sms, cudaStream_t s);
cudaError_t launch_split_f32(const float* in, __nv_bfloat16* hi, __nv_bfloat16* lo, int64_t n, int num_sms,
                             cudaStream_t s);

// tcgen05 mapper GEMM with fused bias + target RoPE epilogue (d == 128).  With
// split set, operands are fp32 values carried as bf16 (hi, lo) pairs: the
// accumulation runs hi*hi + hi*lo + lo*hi and the output is fp32; otherwise
// bf16 operands and bf16 output.
struct MapGemmArgs {
    Shape sh;
    const void* a_src[2];   // [L_s*H][T][d] bf16: stripped keys, raw values (hi parts when split)
    const void* w[2];       // [L_t][q][p] bf16 (hi parts when split)
    const void* a_lo[2];    // lo parts when split
    const void* w_lo[2];
    bool split;
    // strip fused into the kernel: a_src[0] is then written by the kernel from k_raw
    bool fuse_strip;
    const void* k_raw;      // [L_s*H][T][d] bf16 source keys as stored
    const float2* tab_s;    // source RoPE table
    int* strip_ctr;         // [2] zeroed before the launch
    int* tile_ctr;          // CTA-pair kernel: tile claim counter zeroed before the launch, or null (fixed tiles)
    const float* bias[2];   // [L_t][q]
    void* out[2];           // [L_t][H][T][d] bf16 (fp32 when split)
    const int* pos;
    const float2* tab_t;    // target RoPE table
    SelTable sel;
    DevErr err;
    int num_sms;
};
bool map_gemm_tc_supported(const Shape& sh);
bool map_gemm_fused_strip_supported(const Shape& sh);
cudaError_t launch_map_gemm_tc(const MapGemmArgs& a, cudaStream_t s, std::string* why);

// SIMT mapper (any even d with d % 8 == 0): strip fused into the operand load,
// bias + target RoPE in the epilogue.  dtype selects fp32 or bf16 storage.
struct MapSimtArgs {
    Shape sh;
    kvb_dtype dtype;
    const void* src[2];
    const void* w[2];
    const float* bias[2];
    void* out[2];
    const int* pos;
    const float2* tab_s;
    const float2* tab_t;
    SelTable sel;
    DevErr err;
};
cudaError_t launch_map_simt(const MapSimtArgs& a, cudaStream_t s);

// Attention-output cosine on the tensor cores (bf16 caches, head_dim 128, 1 <= T < 2^31,
// fewer than 2^31 query rows L * Hq * Tq).
bool attn_tc_supported(kvb_dtype dtype, int d, int64_t T, int64_t q_rows);
cudaError_t launch_attn_cosine_tc(const void* q, const int* q_pos, const void* k_a, const void* v_a, const void* k_b,
                                  const void* v_b, const int* kv_pos, float* cos_out, int L, int H, int Hq, int Tq,
                                  int64_t T, DevErr err, cudaStream_t s, std::string* why);

// Tensor-map encoder fetched from the driver at run time.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_tiled();

}  // namespace kvb
