// Small kernels of the path: everything that is not a tcgen05 GEMM (declared in
// flce_kernels.cuh).  The per-element dlogits arithmetic is the GEMM epilogue's own
// (dlogit_of in flce_gemm.cuh), so the two paths that form dlogits agree bit for bit.
#include "flce_gemm.cuh"
#include "flce_kernels.cuh"

namespace flce {

__device__ __forceinline__ void merge_stats(float& M, float& D, float& S, float m, float d,
                                            float s) {
  const float Mn = fmaxf(M, m);
  const float a1 = exp2f(M - Mn);
  const float a2 = exp2f(m - Mn);
  S = a1 * fmaf(M - Mn, D, S) + a2 * fmaf(m - Mn, d, s);
  D = a1 * D + a2 * d;
  M = Mn;
}


// Merges the parts of 32 rows per block (8 warps over the parts) and finalises:
// lse, E_p[z], CE (+ smoothing / class weights), z-loss, entropy, ignore mask.
// V is the whole vocabulary (labels outside [0, V) that are not ignored are errors).
__global__ void __launch_bounds__(256) fwd_combine_kernel(
    Parts pt, int64_t N, const float* __restrict__ zlabel, const int64_t* __restrict__ labels,
    int64_t V, int64_t ignore_index, float zcoef, Smoothing sm, float* __restrict__ lse_out,
    float* __restrict__ ez_out, float* __restrict__ loss_row, float* __restrict__ ent_row,
    uint32_t* err) {
  __shared__ float sM[8][32], sD[8][32], sS[8][32], sW[8][32], sZ[8][32];
  const int w = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t n = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  const bool smooth = sm.eps != 0.0f;
  float M = -1e30f, D = 0.0f, S = 0.0f, SW = 0.0f, ZY = 0.0f;
  if (n < N) {
    for (int64_t p = w; p < pt.n_parts; p += 8) {
      const int64_t o = p * pt.part_stride + n;
      merge_stats(M, D, S, pt.pm[o], pt.pd[o], pt.ps[o]);
      if (smooth) SW += sm.psw[o];
      if (pt.pzy) ZY += pt.pzy[o];
    }
  }
  sM[w][lane] = M;
  sD[w][lane] = D;
  sS[w][lane] = S;
  sW[w][lane] = SW;
  sZ[w][lane] = ZY;
  __syncthreads();
  if (w != 0 || n >= N) return;
  M = sM[0][lane];
  D = sD[0][lane];
  S = sS[0][lane];
  SW = sW[0][lane];
  ZY = sZ[0][lane];
  for (int k = 1; k < 8; ++k) {
    merge_stats(M, D, S, sM[k][lane], sD[k][lane], sS[k][lane]);
    SW += sW[k][lane];
    ZY += sZ[k][lane];
  }
  // M, S in log2 units: lse = ln2 (M + log2 D); entropy = ln d - s_c/d = ln2 (log2 D - S/D)
  const float l2d = log2f(D);
  const float lse = kLn2 * (M + l2d);
  const float ent = kLn2 * (l2d - S / D);
  lse_out[n] = lse;
  ez_out[n] = lse - ent;
  const int64_t y = labels[n];
  float lt = 0.0f, et = 0.0f;
  if (y != ignore_index) {
    if (y < 0 || y >= V) {
      atomicOr(err, FLCE_DEVERR_LABEL);
      lt = et = __int_as_float(0x7fc00000);
    } else {
      float ce = lse - (pt.pzy ? ZY : zlabel[n]);
      if (smooth || sm.cw) {
        // (1 - eps) w_y (lse - z_y) + eps/V (W lse - sum_v w_v z_v)
        const float wy = sm.cw ? sm.cw[y] : 1.0f;
        const float W = sm.wsum ? *sm.wsum : static_cast<float>(V);
        ce = (1.0f - sm.eps) * wy * ce;
        if (smooth) ce += sm.eps / static_cast<float>(V) * (W * lse - SW);
      }
      lt = ce + zcoef * lse * lse;
      et = ent;
    }
  }
  loss_row[n] = lt;
  ent_row[n] = et;
}

// Deterministic fixed-order reduction over rows (one block): mean or sum.
// With class weights cw the mean divides the cross-entropy part of the rows
// (loss_row - zcoef lse^2) by the summed w_y and the z-loss part by the row count.
__global__ void __launch_bounds__(1024) reduce_rows_kernel(
    const float* __restrict__ loss_row, const float* __restrict__ ent_row,
    const int64_t* __restrict__ labels, int64_t N, int64_t ignore_index, int mean,
    const float* __restrict__ cw, const float* __restrict__ lse, float zcoef,
    float* __restrict__ loss_out, float* __restrict__ ent_out) {
  __shared__ double sl[1024], se[1024], sz[1024], sw[1024];
  __shared__ long long sc[1024];
  double l = 0.0, e = 0.0, zl = 0.0, wsum = 0.0;
  long long c = 0;
  for (int64_t n = threadIdx.x; n < N; n += blockDim.x) {
    l += loss_row[n];
    e += ent_row[n];
    const int64_t y = labels[n];
    if (y != ignore_index) {
      ++c;
      if (cw) {
        const double ln = lse[n];
        zl += static_cast<double>(zcoef) * ln * ln;
        wsum += cw[y];
      }
    }
  }
  sl[threadIdx.x] = l;
  se[threadIdx.x] = e;
  sz[threadIdx.x] = zl;
  sw[threadIdx.x] = wsum;
  sc[threadIdx.x] = c;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) {
      sl[threadIdx.x] += sl[threadIdx.x + s];
      se[threadIdx.x] += se[threadIdx.x + s];
      sz[threadIdx.x] += sz[threadIdx.x + s];
      sw[threadIdx.x] += sw[threadIdx.x + s];
      sc[threadIdx.x] += sc[threadIdx.x + s];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    double L = sl[0], E = se[0];
    if (mean) {
      const long long nv = sc[0];
      const double rn = nv > 0 ? 1.0 / static_cast<double>(nv) : 0.0;
      if (cw) {
        const double ce = L - sz[0];
        L = (sw[0] != 0.0 ? ce / sw[0] : 0.0) + sz[0] * rn;
      } else {
        L = L * rn;
      }
      E = E * rn;
    }
    loss_out[0] = static_cast<float>(L);
    ent_out[0] = static_cast<float>(E);
  }
}

// wsum[0] = sum_v cw[v] (one block, fixed order).
__global__ void __launch_bounds__(1024) class_weight_sum_kernel(const float* __restrict__ cw,
                                                                int64_t V, float* wsum) {
  __shared__ double sw[1024];
  double a = 0.0;
  for (int64_t v = threadIdx.x; v < V; v += blockDim.x) a += cw[v];
  sw[threadIdx.x] = a;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) sw[threadIdx.x] += sw[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) wsum[0] = static_cast<float>(sw[0]);
}

// One vocabulary shard's statistics per row, [4, N]: the merge of its column
// parts (m, d, s in log2 units) and the label logit if the label is in the shard.
__global__ void __launch_bounds__(256) shard_stats_kernel(
    const float* __restrict__ pm, const float* __restrict__ pd, const float* __restrict__ ps,
    int64_t n_parts, int64_t N, const float* __restrict__ zlabel,
    const int64_t* __restrict__ labels, int64_t v_offset, int64_t v_shard,
    float* __restrict__ stats) {
  __shared__ float sM[8][32], sD[8][32], sS[8][32];
  const int w = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t n = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  float M = -1e30f, D = 0.0f, S = 0.0f;
  if (n < N)
    for (int64_t p = w; p < n_parts; p += 8) merge_stats(M, D, S, pm[p * N + n], pd[p * N + n],
                                                         ps[p * N + n]);
  sM[w][lane] = M;
  sD[w][lane] = D;
  sS[w][lane] = S;
  __syncthreads();
  if (w != 0 || n >= N) return;
  M = sM[0][lane];
  D = sD[0][lane];
  S = sS[0][lane];
  for (int k = 1; k < 8; ++k) merge_stats(M, D, S, sM[k][lane], sD[k][lane], sS[k][lane]);
  const int64_t y = labels[n] - v_offset;
  stats[n] = M;
  stats[N + n] = D;
  stats[2 * N + n] = S;
  stats[3 * N + n] = (y >= 0 && y < v_shard) ? zlabel[n] : 0.0f;
}

// Per-row constants of the dlogits epilogue, with a_ce / a_z / b the upstream
// gradients of the cross-entropy part, the z-loss and the entropy after the
// reduction (mean: a_ce / sum w_y, a_z and b / n_valid) and zero on ignored rows:
//   rowc = (lse log2e, A1, b, C_y),  rowd = D,  where
//   A1 = a_ce ((1 - eps) w_y + eps W / V) + 2 coef lse a_z + b Ez,
//   C_y = a_ce (1 - eps) w_y,  D = a_ce eps / V,
// so that dlogits = p (A1 - b z) - C_y [v == y] - D w_v.
// The mean's denominators count the rows of den_labels [den_n] (all rows of the
// call), the constants are written for the N rows of labels (a chunk of them).
__global__ void __launch_bounds__(1024) bwd_prep_kernel(
    const int64_t* __restrict__ labels, const int64_t* __restrict__ den_labels, int64_t den_n,
    const float* __restrict__ lse, const float* __restrict__ ez,
    const float* __restrict__ g_loss, const float* __restrict__ g_ent, int64_t N, int64_t V,
    int64_t ignore_index, int per_token, int mean, float zcoef, float eps,
    const float* __restrict__ cw, float4* __restrict__ rowc, float* __restrict__ rowd) {
  __shared__ long long sc[1024];
  __shared__ double sw[1024], sww[1024];
  long long c = 0;
  double wy_sum = 0.0, w_all = 0.0;
  for (int64_t n = threadIdx.x; n < den_n; n += blockDim.x) {
    const int64_t y = den_labels[n];
    if (y != ignore_index) {
      ++c;
      if (cw) wy_sum += cw[y];
    }
  }
  if (cw && eps != 0.0f)
    for (int64_t v = threadIdx.x; v < V; v += blockDim.x) w_all += cw[v];
  sc[threadIdx.x] = c;
  sw[threadIdx.x] = wy_sum;
  sww[threadIdx.x] = w_all;
  __syncthreads();
  for (int s = blockDim.x / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) {
      sc[threadIdx.x] += sc[threadIdx.x + s];
      sw[threadIdx.x] += sw[threadIdx.x + s];
      sww[threadIdx.x] += sww[threadIdx.x + s];
    }
    __syncthreads();
  }
  const long long nv = sc[0];
  const float scale = mean ? (nv > 0 ? 1.0f / static_cast<float>(nv) : 0.0f) : 1.0f;
  const bool plain = eps == 0.0f && cw == nullptr;
  const float scale_ce =
      (mean && cw) ? (sw[0] != 0.0 ? static_cast<float>(1.0 / sw[0]) : 0.0f) : scale;
  const float W = cw ? static_cast<float>(sww[0]) : static_cast<float>(V);
  for (int64_t n = threadIdx.x; n < N; n += blockDim.x) {
    const int64_t y = labels[n];
    const bool valid = y != ignore_index;
    const int64_t gi = per_token ? n : 0;
    const float gl = g_loss ? g_loss[gi] : 0.0f;
    const float ge = g_ent ? g_ent[gi] : 0.0f;
    const float a = valid ? gl * scale : 0.0f;
    const float b = valid ? ge * scale : 0.0f;
    const float l = lse[n];
    if (plain) {
      rowc[n] = make_float4(l * kLog2e, fmaf(a, fmaf(2.0f * zcoef, l, 1.0f), b * ez[n]), b, a);
      continue;
    }
    const float a_ce = valid ? gl * scale_ce : 0.0f;
    const float wy = (cw && valid && y >= 0 && y < V) ? cw[y] : 1.0f;
    const float cy = a_ce * (1.0f - eps) * wy;
    const float a1 = fmaf(a_ce, eps * W / static_cast<float>(V), cy) +
                     fmaf(2.0f * zcoef * l, a, b * ez[n]);
    rowc[n] = make_float4(l * kLog2e, a1, b, cy);
    if (eps != 0.0f) rowd[n] = a_ce * eps / static_cast<float>(V);
  }
}

// dlogits [rows, ldz] (bf16) from the raw fp32 logits z [rows, ldz] the forward
// GEMM kept, with the per-row constants of bwd_prep_kernel; the same per-element
// arithmetic as the recompute epilogue (dlogit_of), zero beyond column V.  Each
// thread converts two groups of 8 columns a block-width apart in each of two rows and
// issues all four groups' loads first: 128 bytes in flight per thread (the logits are
// read once: evict-first).  The soft-cap and smoothing terms are template choices, so
// the plain case carries none of their registers: 71 registers, 3 blocks per SM.
// Measured in the gradient-in-forward step on the Llama-3 head shape (8192 x 128256):
// 0.955 ms (6.6 TB/s); one row per block, 1.068 ms; two rows with the terms chosen at
// run time (121 registers, 2 blocks per SM), 1.50 ms.

template <bool CAP, bool SMOOTH>
__device__ __forceinline__ uint4 dlogits8(const float (&x)[8], int64_t c0, const float4& rc,
                                          float dcoef, int64_t y, int64_t V, float softcap,
                                          float k, const float* __restrict__ cw) {
  uint32_t pk[4];
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    float g2[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t v = c0 + j + h;
      const bool in = v < V;
      const float dw = (SMOOTH && in) ? __fmul_rn(dcoef, cw ? __ldg(cw + v) : 1.0f) : 0.0f;
      const float g = dlogit_of(x[j + h], rc, v == y, SMOOTH, dw, CAP, softcap, k);
      g2[h] = in ? g : 0.0f;
    }
    pk[j / 2] = pack_bf16x2(g2[0], g2[1]);
  }
  return make_uint4(pk[0], pk[1], pk[2], pk[3]);
}

__device__ __forceinline__ void load8_cs(const float* p, float (&x)[8]) {
  const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
  const float4 b = __ldcs(reinterpret_cast<const float4*>(p + 4));
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

template <bool CAP, bool SMOOTH>
__global__ void __launch_bounds__(kDlzThreads) dlogits_from_z_kernel(
    const float* __restrict__ z, int64_t rows, int64_t ldz, const float4* __restrict__ rowc,
    const float* __restrict__ rowd, const int64_t* __restrict__ labels, int64_t V,
    float softcap, const float* __restrict__ cw, __nv_bfloat16* __restrict__ dl) {
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kDlzCols + threadIdx.x * 8;
  const int64_t c1 = c0 + kDlzThreads * 8;
  if (c0 >= ldz) return;
  const bool has1 = c1 < ldz;
  const float k = CAP ? 2.0f * kLog2e / softcap : 0.0f;
  for (int64_t r = 2 * static_cast<int64_t>(blockIdx.y); r < rows;
       r += 2 * static_cast<int64_t>(gridDim.y)) {
    const bool two = r + 1 < rows;
    float x[4][8];
    load8_cs(z + r * ldz + c0, x[0]);
    if (has1) load8_cs(z + r * ldz + c1, x[1]);
    if (two) {
      load8_cs(z + (r + 1) * ldz + c0, x[2]);
      if (has1) load8_cs(z + (r + 1) * ldz + c1, x[3]);
    }
    {
      const float4 rc = rowc[r];
      const float dcoef = SMOOTH ? rowd[r] : 0.0f;
      const int64_t yl = labels[r];
      const int64_t y = (yl >= 0 && yl < V) ? yl : -1;
      *reinterpret_cast<uint4*>(dl + r * ldz + c0) =
          dlogits8<CAP, SMOOTH>(x[0], c0, rc, dcoef, y, V, softcap, k, cw);
      if (has1)
        *reinterpret_cast<uint4*>(dl + r * ldz + c1) =
            dlogits8<CAP, SMOOTH>(x[1], c1, rc, dcoef, y, V, softcap, k, cw);
    }
    if (two) {
      const float4 rc = rowc[r + 1];
      const float dcoef = SMOOTH ? rowd[r + 1] : 0.0f;
      const int64_t yl = labels[r + 1];
      const int64_t y = (yl >= 0 && yl < V) ? yl : -1;
      *reinterpret_cast<uint4*>(dl + (r + 1) * ldz + c0) =
          dlogits8<CAP, SMOOTH>(x[2], c0, rc, dcoef, y, V, softcap, k, cw);
      if (has1)
        *reinterpret_cast<uint4*>(dl + (r + 1) * ldz + c1) =
            dlogits8<CAP, SMOOTH>(x[3], c1, rc, dcoef, y, V, softcap, k, cw);
    }
  }
}

cudaError_t launch_dlogits_from_z(const float* z, int64_t rows, int64_t ldz,
                                  const float4* rowc, const float* rowd, const int64_t* labels,
                                  int64_t V, float softcap, bool smooth, const float* cw,
                                  __nv_bfloat16* dl, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const int64_t row_pairs = (rows + 1) / 2;
  const dim3 grid(static_cast<unsigned>((ldz + kDlzCols - 1) / kDlzCols),
                  static_cast<unsigned>(row_pairs < 65535 ? row_pairs : 65535));
  const bool cap = softcap != 0.0f;
  if (cap && smooth)
    dlogits_from_z_kernel<true, true><<<grid, kDlzThreads, 0, st>>>(z, rows, ldz, rowc, rowd,
                                                                     labels, V, softcap, cw, dl);
  else if (cap)
    dlogits_from_z_kernel<true, false><<<grid, kDlzThreads, 0, st>>>(z, rows, ldz, rowc, rowd,
                                                                      labels, V, softcap, cw, dl);
  else if (smooth)
    dlogits_from_z_kernel<false, true><<<grid, kDlzThreads, 0, st>>>(z, rows, ldz, rowc, rowd,
                                                                      labels, V, softcap, cw, dl);
  else
    dlogits_from_z_kernel<false, false><<<grid, kDlzThreads, 0, st>>>(z, rows, ldz, rowc, rowd,
                                                                       labels, V, softcap, cw,
                                                                       dl);
  return cudaGetLastError();
}

// x *= g[0] over n bf16 values, 8 per thread (grid-stride), zero products as +0;
// nothing when g[0] == 1.
__global__ void __launch_bounds__(256) scale_bf16_kernel(__nv_bfloat16* __restrict__ x,
                                                         int64_t n, const float* __restrict__ g) {
  const float s = *g;
  if (s == 1.0f) return;
  const int64_t n8 = n / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += stride) {
    uint4 v = reinterpret_cast<uint4*>(x)[i];
    uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float lo = __uint_as_float(w[k] << 16);
      const float hi = __uint_as_float(w[k] & 0xffff0000u);
      // + 0: a zero stays +0 under a negative scale (ignored rows stay bitwise zero)
      w[k] = pack_bf16x2(__fmaf_rn(lo, s, 0.0f), __fmaf_rn(hi, s, 0.0f));
    }
    reinterpret_cast<uint4*>(x)[i] = v;
  }
  if (blockIdx.x == 0 && threadIdx.x < n - n8 * 8) {
    const int64_t i = n8 * 8 + threadIdx.x;
    x[i] = __float2bfloat16_rn(__fmaf_rn(__bfloat162float(x[i]), s, 0.0f));
  }
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing will
// ever arrive on, with the pipeline kernels' own wait, until `limit_ns` of global
// time has passed; the wait then records FLCE_DEVERR_TIMEOUT in the error word and
// the kernel returns, leaving the context usable.
__global__ void wait_timeout_selftest_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(&bar, 1);
  fence_mbar_init();
  mbar_wait(&bar, 0, &abort_flag, err, limit_ns);
}

}  // namespace flce
