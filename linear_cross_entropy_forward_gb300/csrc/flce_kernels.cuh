// Small kernels of the path (argument structs and declarations): the combine of the
// forward's partial statistics, the reductions over rows, the backward's per-row
// constants, the gradient-in-forward dlogits, and helpers.  Defined in
// flce_kernels.cu, launched by flce_api.cu.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace flce {

// One block of 8 warps handles 32 rows; warp w merges parts w, w+8, ...
// Label smoothing / class weights of the combine (Smoothing.eps == 0 and cw == NULL:
// plain cross-entropy).  psw holds the partial sums_v w_v z_v, wsum = sum_v w_v.
struct Smoothing {
  float eps;
  const float* cw;
  const float* psw;
  const float* wsum;  // device scalar (NULL: V, all weights 1)
};

// Partial statistics to merge per row: part p of row n holds (m, d, s) at
// offset p * part_stride + n of pm / pd / ps.  The label logit comes from
// zlabel[n], or, when pzy is set (vocabulary shards), is the sum over the parts of
// pzy[p * part_stride + n] (the one shard that holds the label contributes it).
struct Parts {
  const float* pm;
  const float* pd;
  const float* ps;
  const float* pzy;
  int64_t n_parts;
  int64_t part_stride;
};

// dlogits_from_z_kernel: threads per block, columns per block
constexpr int kDlzThreads = 256;
constexpr int kDlzCols = 2 * 8 * kDlzThreads;  // columns per block

__global__ void __launch_bounds__(256) fwd_combine_kernel(
    Parts pt, int64_t N, const float* __restrict__ zlabel, const int64_t* __restrict__ labels,
    int64_t V, int64_t ignore_index, float zcoef, Smoothing sm, float* __restrict__ lse_out,
    float* __restrict__ ez_out, float* __restrict__ loss_row, float* __restrict__ ent_row,
    uint32_t* err);

__global__ void __launch_bounds__(1024) reduce_rows_kernel(
    const float* __restrict__ loss_row, const float* __restrict__ ent_row,
    const int64_t* __restrict__ labels, int64_t N, int64_t ignore_index, int mean,
    const float* __restrict__ cw, const float* __restrict__ lse, float zcoef,
    float* __restrict__ loss_out, float* __restrict__ ent_out);

__global__ void __launch_bounds__(1024) class_weight_sum_kernel(const float* __restrict__ cw,
                                                                int64_t V, float* wsum);

__global__ void __launch_bounds__(256) shard_stats_kernel(
    const float* __restrict__ pm, const float* __restrict__ pd, const float* __restrict__ ps,
    int64_t n_parts, int64_t N, const float* __restrict__ zlabel,
    const int64_t* __restrict__ labels, int64_t v_offset, int64_t v_shard,
    float* __restrict__ stats);

__global__ void __launch_bounds__(1024) bwd_prep_kernel(
    const int64_t* __restrict__ labels, const int64_t* __restrict__ den_labels, int64_t den_n,
    const float* __restrict__ lse, const float* __restrict__ ez,
    const float* __restrict__ g_loss, const float* __restrict__ g_ent, int64_t N, int64_t V,
    int64_t ignore_index, int per_token, int mean, float zcoef, float eps,
    const float* __restrict__ cw, float4* __restrict__ rowc, float* __restrict__ rowd);

// dlogits [rows, ldz] bf16 from the kept fp32 logits z [rows, ldz] (rows of two per
// block; the soft-cap and smoothing variants chosen here).
cudaError_t launch_dlogits_from_z(const float* z, int64_t rows, int64_t ldz,
                                  const float4* rowc, const float* rowd, const int64_t* labels,
                                  int64_t V, float softcap, bool smooth, const float* cw,
                                  __nv_bfloat16* dl, cudaStream_t st);

__global__ void __launch_bounds__(256) scale_bf16_kernel(__nv_bfloat16* __restrict__ x,
                                                         int64_t n, const float* __restrict__ g);

__global__ void wait_timeout_selftest_kernel(uint32_t* err, uint64_t limit_ns);

}  // namespace flce
