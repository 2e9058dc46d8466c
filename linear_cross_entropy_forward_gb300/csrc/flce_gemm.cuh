// Persistent, warp-specialised tcgen05 GEMM with fused epilogues for the fused
// linear cross-entropy + entropy path (verl PR #462, "Equivalent compute logic":
// logits = hidden @ weight are never stored; every use of them is fused here).
//
// A CTA pair (a cluster of two CTAs, ranks 0 and 1) owns 256 x TN output tiles:
//   warp 0      TMA producer (both CTAs): this CTA's 128 rows of A and TN/2
//               columns of B into a ring of 128B-swizzled shared-memory stages;
//               completion is counted on the pair leader's (rank 0) full barrier.
//   warp 1      UMMA issuer (leader only): 256 x TN x 16 tcgen05.mma.cta_group::2
//               into one of 512/TN fp32 TMEM accumulators; each commit arrives on
//               the same barrier of both CTAs of the pair.
//   warps 2..   epilogue (both CTAs, 4 or 8 warps, see epi_warps): tcgen05.ld one
//               row per thread (warp w reads TMEM lanes 32*(w%4)..+31 and, with 8
//               warps, column half (w-2)/4 of the tile), then one of:
//     EPI_FWD_STATS  online-softmax partials per row and warp column block:
//                    running max m, sum-exp d and centred s = sum e^{u-m}(u-m)
//                    in log2 units, plus the label logit (Liger-Kernel PR #551:
//                    m and d of the online softmax feed the entropy); optionally
//                    also the raw fp32 logits (gradient in forward).
//     EPI_DLOGITS    recomputed logits -> dlogits (bf16) of the CE, z-loss and
//                    entropy terms, with the soft-cap chain rule (Liger-Kernel
//                    issue #127: tanh capping after the matmul).
//     EPI_STORE_BF16 plain bf16 store (dweight tiles).
//     EPI_ACCUM      fp32 accumulation across vocabulary chunks (dhidden) or token
//                    chunks (dweight); the last chunk writes bf16.
//   Arrays in the workspace (kept logits, dlogits, fp32 accumulators: 256-byte
//   aligned, pitches multiples of 32 bytes) are accessed 256 bits per thread; the
//   caller's dweight / dhidden (16-byte alignment promised) 128 bits.
//
// A cluster is exactly one pair, and every TMA load lands in the shared memory of
// the CTA that issues it: no tile is delivered to more than one CTA.
//
// Tiles are handed out dynamically: each pair takes its first tile by its cluster
// index and every later one from a global counter in the workspace header, so the
// tiles in flight stay a window of consecutive tiles of the raster order however
// unevenly the pairs progress (a static round-robin let them drift apart by many
// tiles over a long schedule, and the operand panels they shared fell out of L2).
// The peer CTA's warp 1 (idle otherwise: the leader issues the pair's UMMAs) is the
// pair's scheduler: it draws the tiles and publishes them through a two-slot ring in
// shared memory to every role of both CTAs, so no role on the pipeline's critical
// path waits for a global atomic.  The last pair to finish resets the counter for the
// next launch.
//
// Operands arrive as 64-row pieces of 8 KB ({64 K, 64 rows} boxes for K-major,
// {64 MN, 64 K} boxes of the transposed view for MN-major); operand majorness is a
// template choice, so no transposed copy of any tensor is made.  Every barrier
// wait is bounded (flce_device.cuh).
#pragma once

#include <atomic>

#include "flce_check.cuh"
#include "flce_device.cuh"

namespace flce {

constexpr int BK = 64;  // one 128-byte swizzle row of bf16
constexpr int UK = 16;  // K of one kind::f16 UMMA
constexpr int PAIR_BM = 256;  // rows of a pair tile (128 per CTA)
enum EpiKind { EPI_FWD_STATS = 0, EPI_DLOGITS = 1, EPI_STORE_BF16 = 2, EPI_ACCUM = 3 };

// Epilogue warps per CTA: 4 (one per TMEM lane quadrant, all of a tile's columns)
// or 8 (two per quadrant, half the columns each).  Epilogue arithmetic costs the
// UMMA issuer issue slots, so fewer warps are better where the epilogue of a tile
// stays well inside the next tile's mainloop; the dlogits epilogue (with the
// soft-cap, on tiles of only H/64 k-steps) needs 8 to stay hidden.
#ifndef FLCE_EPI_WARPS
#define FLCE_EPI_WARPS 0  // 0: per epilogue kind as below; 4 or 8: every kind
#endif
template <int EPI>
__host__ __device__ constexpr int epi_warps() {
  return FLCE_EPI_WARPS ? FLCE_EPI_WARPS : (EPI == EPI_DLOGITS ? 8 : 4);
}
template <int EPI>
__host__ __device__ constexpr int pair_threads() {
  return 64 + 32 * epi_warps<EPI>();
}
constexpr int TMEM_COLS = 512;
// Depth of the ring that publishes each pair's tiles: the scheduler runs at most this
// many tiles (plus the one it has drawn) ahead of the slowest role of the pair, which
// keeps the tiles in flight across the GPU close together in the raster order.
constexpr int TILE_RING = 2;
constexpr uint32_t MN_ATOM_BYTES = 64 * BK * 2;  // one {64 MN x 64 K} box
constexpr int SMEM_LIMIT = 232448;               // 227 KB per CTA

#ifndef FLCE_MAX_STAGES
#define FLCE_MAX_STAGES 9
#endif

// Per-tile-width (and epilogue-warp-count) configuration of the pair kernel.
template <int TN, int EW>
struct PairCfg {
  static_assert(TN == 128 || TN == 256, "tile width");
  static constexpr int B_ROWS = TN / 2;                // this CTA's share of B's columns
  static constexpr int A_BYTES = 128 * BK * 2;         // 16 KB
  static constexpr int B_BYTES = B_ROWS * BK * 2;      // 8 or 16 KB
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int NACC = TMEM_COLS / TN;          // TMEM accumulators
  static_assert(EW == 4 || EW == 8, "epilogue warps");
  static constexpr int EPI_COLS = TN * 4 / EW;          // columns per epilogue warp
  static constexpr int EPI_CHUNKS = EPI_COLS / 32;     // tcgen05.ld x32 per warp per tile
  static constexpr int PARTS = TN / EPI_COLS;           // statistics parts per tile
  static constexpr int BAR_BYTES = 512;
  static constexpr int STAGES_FIT = (SMEM_LIMIT - 1024 - BAR_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > FLCE_MAX_STAGES ? FLCE_MAX_STAGES : STAGES_FIT;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory");
  static_assert((2 * STAGES + 2 * NACC + 2 * TILE_RING) * 8 + 8 + 4 * TILE_RING <= BAR_BYTES,
                "barrier area");
};

// Tile width (UMMA N) of each kernel of the path.
#ifndef FLCE_TN_FWD
#define FLCE_TN_FWD 256
#endif
#ifndef FLCE_TN_DLOGITS
#define FLCE_TN_DLOGITS 256
#endif
#ifndef FLCE_TN_DWEIGHT
#define FLCE_TN_DWEIGHT 256
#endif
#ifndef FLCE_TN_DHIDDEN
#define FLCE_TN_DHIDDEN 256
#endif
constexpr int TN_FWD = FLCE_TN_FWD;
constexpr int TN_DLOGITS = FLCE_TN_DLOGITS;
constexpr int TN_DWEIGHT = FLCE_TN_DWEIGHT;
constexpr int TN_DHIDDEN = FLCE_TN_DHIDDEN;

enum AccMode { ACC_FIRST = 0, ACC_MID = 1, ACC_LAST = 2, ACC_ONLY = 3 };

struct GemmShape {
  int m_tiles, n_tiles, k_blocks;
  int raster;                 // 0: m fastest, 1: n fastest (within a group)
  int group;                  // tiles of the fast dimension per group (see tile_coords)
  int a_mn_off, a_k_off;      // added to A's (mn, k) tile coordinates
  int b_mn_off, b_k_off;      // added to B's (mn, k) tile coordinates
  uint32_t mn_lbo, mn_sbo;    // descriptor strides of MN-major operands (bytes)
  int a_hint, b_hint;         // L2 eviction priority of A / B tile loads (L2Hint)
  // dynamic schedule: sched[0] counts the tiles drawn after each pair's first,
  // sched[1] the pairs that finished; both zero at launch, and zero again when the
  // kernel ends (the last pair to finish resets them)
  unsigned int* sched;
  // extents (inner, outer) of the arrays behind the A and B tensor maps: the
  // FLCE_DEBUG build checks every TMA box against them
  int64_t a_inner, a_outer, b_inner, b_outer;
};

struct EpiArgs {
  int rows;            // valid output rows (M extent)
  int cols;            // valid output columns, relative to the problem's column 0
  int col_base;        // global column (vocab index) of problem column 0
  int64_t V;           // vocabulary size (masking of the softmax)
  float softcap;       // 0 = off
  const int64_t* labels;
  int64_t label_offset;  // vocabulary index of problem column 0's shard (0 unsharded)
  int64_t ignore_index;
  // EPI_FWD_STATS
  float* pm;
  float* pd;
  float* ps;
  int64_t part_stride;  // elements between consecutive column parts
  float* zlabel;
  // label smoothing (FWD_STATS and DLOGITS): eps != 0 turns it on; cw are the
  // per-class weights (NULL: all 1)
  float smooth;
  const float* cw;
  float* psw;           // FWD_STATS: per part sum_v w_v z_v (same layout as pm)
  float* zout;          // FWD_STATS: if set, the raw fp32 accumulators, [rows, ld_z]
  int64_t ld_z;
  // EPI_DLOGITS
  const float4* rowc;   // per row: (lse*log2e, A1, b, C_y), see bwd_prep_kernel
  const float* rowd;    // per row: D, the coefficient of -w_v (label smoothing)
  __nv_bfloat16* dl;
  int64_t ld_dl;
  // EPI_STORE_BF16
  __nv_bfloat16* out;
  int64_t ld_out;
  // EPI_ACCUM
  float* acc;
  __nv_bfloat16* acc_out;
  int64_t ld_acc;
  int acc_mode;
  uint32_t* err;
  int64_t n_parts;      // EPI_FWD_STATS: column parts of pm / pd / ps (bounds checks)
};

// A bounds check of the FLCE_DEBUG build: true in the regular build; in the debug
// build a failing check records FLCE_DEVERR_BOUNDS and the caller skips the access.
#if FLCE_DEBUG
__device__ __forceinline__ bool debug_ok(bool ok, uint32_t* err) {
  if (!ok && err) atomicOr(err, FLCE_DEVERR_BOUNDS);
  return ok;
}
#define FLCE_CHECK(cond, err) ::flce::debug_ok((cond), (err))
#else
#define FLCE_CHECK(cond, err) true
#endif

// Tile order of the persistent schedule.  raster 0: groups of `group` consecutive
// m-tiles, m fastest within a group, every n-tile of the group before the next
// group (group >= the m-tile count: plain m-fastest order).  raster 1: the same
// with the roles of m and n swapped.  Grouping bounds how much of the operand
// revisited by every tile must stay in L2.  (Host callable too, so the order can
// be checked without a GPU.)
__host__ __device__ __forceinline__ void tile_coords(int t, const GemmShape& sh, int& mt,
                                                     int& nt) {
  const int cm = sh.m_tiles, cn = sh.n_tiles;
  const bool m_major = sh.raster == 0;
  const int fast_tiles = m_major ? cm : cn;
  const int slow_tiles = m_major ? cn : cm;
  const int g = sh.group < fast_tiles ? sh.group : fast_tiles;
  const int per_group = g * slow_tiles;
  const int grp = t / per_group;
  const int r = t - grp * per_group;
  const int rem = fast_tiles - grp * g;
  const int gsize = rem < g ? rem : g;
  const int f = grp * g + r % gsize;
  const int sl = r / gsize;
  mt = m_major ? f : sl;
  nt = m_major ? sl : f;
}

constexpr uint32_t PIECE_BYTES = 64 * BK * 2;  // 64 rows (MN) x 64 (K), either majorness

// One stage of an operand: ROWS (MN) x 64 (K) as ROWS/64 pieces of 64 rows, 8 KB
// apart (K-major: {64, 64} boxes; MN-major: {64, 64} boxes of the transposed view),
// all loaded into this CTA's own shared memory.  The FLCE_DEBUG build checks each box
// against the array's extents (inner, outer) first and returns false, loading
// nothing more, at the first one out of range.
template <bool MN, int ROWS>
__device__ __forceinline__ bool load_operand(uint8_t* dst, const CUtensorMap* map, uint32_t fb,
                                             int mn0, int k0, uint64_t pol, int64_t inner,
                                             int64_t outer) {
  static_assert(ROWS % 64 == 0, "operand rows");
#pragma unroll
  for (int j = 0; j < ROWS / 64; ++j) {
    const int x = MN ? mn0 + 64 * j : k0;
    const int y = MN ? k0 : mn0 + 64 * j;
#if FLCE_DEBUG
    if (!tma_box_ok(x, y, inner, outer)) return false;
#endif
    tma_load_2d_pair_hint(dst + j * PIECE_BYTES, map, fb, x, y, pol);
  }
  return true;
}

template <bool MN>
__host__ __device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kk,
                                                          const GemmShape& sh) {
  if constexpr (!MN) {
    // K-major: the k-th 16-element slice starts 32 bytes further into each
    // 128-byte swizzled row; 8-row groups are 1024 bytes apart.
    return sdesc_sw128(base + kk * (UK * 2), 16, 1024);
  } else {
    // MN-major: 16 K-rows of 128 bytes per slice; 64-wide MN atoms 8 KB apart.
    return sdesc_sw128(base + kk * (UK * 128), sh.mn_lbo, sh.mn_sbo);
  }
}

// ------------------------------------------------------------------ epilogues
// Each epilogue thread owns one row `row` and CH * 32 consecutive columns
// starting at problem column `col0`; `tbase` addresses them in TMEM.
template <int EPI>
struct Epilogue;

// Online-softmax partial statistics of one row over its CH*32 columns, in log2
// units: u = log2e * z for the (capped) logit z, m = max u, d = sum 2^{u - m},
// s = sum 2^{u - m} (u - m).  Each 32-column chunk takes its maximum before any
// exponential: without the cap over the raw accumulators x (u = log2e x is monotone
// in x, so max u = log2e max x exactly); with it over r = 1 / (1 + 2^{k x}), since the
// capped logit u = c log2e - 2 c log2e r falls as r grows (max u is that of min r).
// Then t = u - m is one FMA per logit, and d, s follow.
template <>
struct Epilogue<EPI_FWD_STATS> {
  template <int CH>
  static __device__ __forceinline__ void run(const EpiArgs& ea, uint32_t tbase, int row,
                                             int col0) {
    const bool row_ok = row < ea.rows;
    int y = -1;
    if (row_ok) {
      const int64_t yl = ea.labels[row] - ea.label_offset;
      if (yl >= 0 && yl < ea.V) y = static_cast<int>(yl);
    }
    const bool cap = ea.softcap != 0.0f;
    const float c = ea.softcap;
    const float k = cap ? 2.0f * kLog2e / c : 0.0f;
    const float c_l2 = c * kLog2e, m2c_l2 = -2.0f * c * kLog2e;
    // u = A * v + B0 for the chunk value v (v = x without the cap, v = r with it)
    const float A = cap ? m2c_l2 : kLog2e;
    const float B0 = cap ? c_l2 : 0.0f;
    const int vcol0 = ea.col_base + col0;
    const bool smooth = ea.smooth != 0.0f;
    float mx = -1e30f, d = 0.0f, s = 0.0f, zy = 0.0f, sw = 0.0f;
    bool hit = false;
    float* zrow = (ea.zout && row_ok) ? ea.zout + static_cast<int64_t>(row) * ea.ld_z + col0
                                      : nullptr;
#pragma unroll 1
    for (int ch = 0; ch < CH; ++ch) {
      float x[32];
      tmem_ld32(tbase + ch * 32, x);
      const int vb = vcol0 + ch * 32;
      const int nvalid = static_cast<int>(ea.V - vb);
      if (zrow && FLCE_CHECK(row_run_ok(col0 + ch * 32, 32, ea.ld_z), ea.err)) {
        // 32-byte aligned: 256-aligned workspace, pitch a multiple of 256 floats
#pragma unroll
        for (int q = 0; q < 4; ++q) st_global_cs_v8f(zrow + ch * 32 + q * 8, x + q * 8);
      }
      // the label's logit (natural units), from the one chunk that holds it
      if (static_cast<unsigned>(y - vb) < 32u) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j == y - vb) zy = cap ? fmaf(-2.0f * c, softcap_r(x[j], k), c) : x[j];
        hit = true;
      }
      float cm;  // the chunk's maximum of u
      if (cap) {
        // x -> r = 1 / (1 + 2^{k x}), the lanes of softcap_r two at a time
        const uint64_t k2 = f2_pack(k, k), one2 = f2_pack(1.0f, 1.0f);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          float e0, e1, r0, r1;
          f2_unpack(f2_mul(f2_pack(x[j], x[j + 1]), k2), e0, e1);
          f2_unpack(f2_add(one2, f2_pack(fast_ex2(e0), fast_ex2(e1))), r0, r1);
          x[j] = fast_rcp(r0);
          x[j + 1] = fast_rcp(r1);
        }
        if (smooth) {  // sum of w_v z_v, natural units
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nvalid)
              sw = fmaf(ea.cw ? __ldg(ea.cw + vb + j) : 1.0f, fmaf(-2.0f * c, x[j], c), sw);
        }
        if (nvalid < 32) {  // r lies in [0, 1]: 2 is never the minimum
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j >= nvalid) x[j] = 2.0f;
        }
        cm = fmaf(m2c_l2, min32(x), c_l2);
      } else {
        if (smooth) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nvalid) sw = fmaf(ea.cw ? __ldg(ea.cw + vb + j) : 1.0f, x[j], sw);
        }
        if (nvalid < 32) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j >= nvalid) x[j] = -1e30f;
        }
        cm = kLog2e * max32(x);
      }
      if (cm > mx) {
        const float a = fast_ex2(mx - cm);
        s = a * fmaf(mx - cm, d, s);
        d *= a;
        mx = cm;
      }
      const float B = B0 - mx;  // t = A v + B = u - m
      if (nvalid >= 32) {
        // two lanes of (d, s) per chunk, added into the running sums at its end
        const uint64_t A2 = f2_pack(A, A), B2 = f2_pack(B, B);
        uint64_t dd = f2_pack(0.0f, 0.0f), ss = dd;
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const uint64_t t = f2_fma(A2, f2_pack(x[j], x[j + 1]), B2);
          float t0, t1;
          f2_unpack(t, t0, t1);
          const uint64_t e = f2_pack(fast_ex2(t0), fast_ex2(t1));
          dd = f2_add(dd, e);
          ss = f2_fma(e, t, ss);
        }
        float d0, d1, s0, s1;
        f2_unpack(dd, d0, d1);
        f2_unpack(ss, s0, s1);
        d += d0 + d1;
        s += s0 + s1;
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float t = fmaf(A, x[j], B);
          const float e = (j < nvalid) ? fast_ex2(t) : 0.0f;
          d += e;
          s = fmaf(e, t, s);
        }
      }
    }
    if (row_ok && FLCE_CHECK(index_ok(vcol0 / (CH * 32), ea.n_parts) &&
                                 index_ok(row, ea.part_stride),
                             ea.err)) {
      const int64_t part = vcol0 / (CH * 32);
      const int64_t o = part * ea.part_stride + row;
      ea.pm[o] = mx;
      ea.pd[o] = d;
      ea.ps[o] = s;
      if (smooth) ea.psw[o] = sw;
      if (hit) ea.zlabel[row] = zy;
    }
  }
};

// dlogit of one logit from its raw fp32 accumulator x, with the row's constants
// rc = (lse log2e, A1, b, C_y) and dw = D w_v (label smoothing, else 0):
//   z = c tanh(x / c) (soft-cap, c != 0),  p = 2^{z log2e - lse log2e},
//   g = p (A1 - b z) - C_y [v == y] - D w_v,  times 1 - tanh^2 under the cap.
// Products that feed a sum are rounded explicitly, so every caller (the GEMM
// epilogue, the gradient-in-forward kernel) gets the same bits.  k = 2 log2e / c.
__device__ __forceinline__ float dlogit_of(float x, const float4& rc, bool is_label, bool smooth,
                                           float dw, bool cap, float softcap, float k) {
  float z = x;
  float th = 0.0f;
  if (cap) {
    th = fmaf(-2.0f, softcap_r(x, k), 1.0f);
    z = __fmul_rn(softcap, th);
  }
  const float p = fast_ex2(fmaf(z, kLog2e, -rc.x));
  float g = __fmul_rn(p, fmaf(-rc.z, z, rc.y));
  if (is_label) g = __fsub_rn(g, rc.w);
  if (smooth) g = __fsub_rn(g, dw);
  if (cap) g = __fmul_rn(g, fmaf(-th, th, 1.0f));
  return g;
}

// dlogit_of for two logits that are neither the label nor under label smoothing,
// with the packed f32x2 arithmetic: lane by lane the same operations, so the same
// bits as two calls of dlogit_of.
__device__ __forceinline__ void dlogit_of2(float x0, float x1, const float4& rc, bool cap,
                                           float softcap, float k, float& g0, float& g1) {
  const uint64_t one2 = f2_pack(1.0f, 1.0f);
  uint64_t z = f2_pack(x0, x1), th = 0;
  if (cap) {
    float e0, e1, r0, r1;
    f2_unpack(f2_mul(z, f2_pack(k, k)), e0, e1);
    f2_unpack(f2_add(one2, f2_pack(fast_ex2(e0), fast_ex2(e1))), r0, r1);
    th = f2_fma(f2_pack(-2.0f, -2.0f), f2_pack(fast_rcp(r0), fast_rcp(r1)), one2);
    z = f2_mul(f2_pack(softcap, softcap), th);
  }
  float q0, q1;
  f2_unpack(f2_fma(z, f2_pack(kLog2e, kLog2e), f2_pack(-rc.x, -rc.x)), q0, q1);
  const uint64_t p = f2_pack(fast_ex2(q0), fast_ex2(q1));
  uint64_t g = f2_mul(p, f2_fma(f2_pack(-rc.z, -rc.z), z, f2_pack(rc.y, rc.y)));
  if (cap) g = f2_mul(g, f2_fma(th ^ 0x8000000080000000ull, th, one2));
  f2_unpack(g, g0, g1);
}

// dlogits of one row over its columns of the current vocabulary chunk.
template <>
struct Epilogue<EPI_DLOGITS> {
  template <int CH>
  static __device__ __forceinline__ void run(const EpiArgs& ea, uint32_t tbase, int row,
                                             int col0) {
    const bool row_ok = row < ea.rows;
    const bool smooth = ea.smooth != 0.0f;
    float4 rc = make_float4(0.f, 0.f, 0.f, 0.f);
    float dcoef = 0.0f;
    int y = -1;
    if (row_ok) {
      rc = ea.rowc[row];
      if (smooth) dcoef = ea.rowd[row];
      const int64_t yl = ea.labels[row] - ea.label_offset;
      if (yl >= 0 && yl < ea.V) y = static_cast<int>(yl);
    }
    const bool cap = ea.softcap != 0.0f;
    const float k = cap ? 2.0f * kLog2e / ea.softcap : 0.0f;
    const int vcol0 = ea.col_base + col0;
    __nv_bfloat16* dst = ea.dl + static_cast<int64_t>(row) * ea.ld_dl + col0;
#pragma unroll 1
    for (int ch = 0; ch < CH; ++ch) {
      float x[32];
      tmem_ld32(tbase + ch * 32, x);
      const int vb = vcol0 + ch * 32;
      const int nvalid = static_cast<int>(ea.V - vb);
      const int jy = static_cast<unsigned>(y - vb) < 32u ? y - vb : -1;  // label column, if here
      float g[32];
      if (!smooth && nvalid >= 32) {
#pragma unroll
        for (int j = 0; j < 32; j += 2)
          dlogit_of2(x[j], x[j + 1], rc, cap, ea.softcap, k, g[j], g[j + 1]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const bool in = j < nvalid;
          const float dw =
              (smooth && in) ? __fmul_rn(dcoef, ea.cw ? __ldg(ea.cw + vb + j) : 1.0f) : 0.0f;
          const float gj = dlogit_of(x[j], rc, false, smooth, dw, cap, ea.softcap, k);
          g[j] = in ? gj : 0.0f;
        }
      }
      if (jy >= 0) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (j == jy) {
            const float dw = smooth ? __fmul_rn(dcoef, ea.cw ? __ldg(ea.cw + vb + j) : 1.0f) : 0.0f;
            g[j] = dlogit_of(x[j], rc, true, smooth, dw, cap, ea.softcap, k);
          }
        }
      }
      if (row_ok && FLCE_CHECK(row_run_ok(col0 + ch * 32, 32, ea.ld_dl), ea.err)) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(g[2 * j], g[2 * j + 1]);
        // 32-byte aligned: 256-aligned workspace, chunk pitch a multiple of 256 columns
        st_global_v8(dst + ch * 32, *reinterpret_cast<const uint32_t(*)[8]>(pk));
        st_global_v8(dst + ch * 32 + 16, *reinterpret_cast<const uint32_t(*)[8]>(pk + 8));
      }
    }
  }
};

// bf16 store of a row segment (dweight).
template <>
struct Epilogue<EPI_STORE_BF16> {
  template <int CH>
  static __device__ __forceinline__ void run(const EpiArgs& ea, uint32_t tbase, int row,
                                             int col0) {
    const bool row_ok = row < ea.rows;
    __nv_bfloat16* dst = ea.out + static_cast<int64_t>(row) * ea.ld_out + ea.col_base + col0;
#pragma unroll 1
    for (int c = 0; c < CH; ++c) {
      float x[32];
      tmem_ld32(tbase + c * 32, x);
      if (!row_ok) continue;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int col = col0 + c * 32 + q * 8;
        if (col < ea.cols && FLCE_CHECK(row_run_ok(ea.col_base + col, 8, ea.ld_out), ea.err)) {
          uint4 v = make_uint4(pack_bf16x2(x[q * 8 + 0], x[q * 8 + 1]),
                               pack_bf16x2(x[q * 8 + 2], x[q * 8 + 3]),
                               pack_bf16x2(x[q * 8 + 4], x[q * 8 + 5]),
                               pack_bf16x2(x[q * 8 + 6], x[q * 8 + 7]));
          *reinterpret_cast<uint4*>(dst + c * 32 + q * 8) = v;
        }
      }
    }
  }
};

// fp32 accumulation across vocabulary chunks (dhidden).
template <>
struct Epilogue<EPI_ACCUM> {
  template <int CH>
  static __device__ __forceinline__ void run(const EpiArgs& ea, uint32_t tbase, int row,
                                             int col0) {
    const bool row_ok = row < ea.rows;
    const int64_t base = static_cast<int64_t>(row) * ea.ld_acc + col0;
#pragma unroll 1
    for (int c = 0; c < CH; ++c) {
      float x[32];
      tmem_ld32(tbase + c * 32, x);
      if (!row_ok) continue;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int col = col0 + c * 32 + q * 8;
        if (col >= ea.cols || !FLCE_CHECK(row_run_ok(col, 8, ea.ld_acc), ea.err)) continue;
        // the fp32 accumulator lives in the workspace (256-aligned, pitch a multiple
        // of 8 floats): 32-byte aligned
        float* a = ea.acc + base + c * 32 + q * 8;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = x[q * 8 + i];
        if (ea.acc_mode == ACC_MID || ea.acc_mode == ACC_LAST) {
          float o[8];
          ld_global_v8f(a, o);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] += o[i];
        }
        if (ea.acc_mode == ACC_FIRST || ea.acc_mode == ACC_MID) {
          st_global_v8f(a, v);
        } else {
          uint4 o = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                               pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
          *reinterpret_cast<uint4*>(ea.acc_out + base + c * 32 + q * 8) = o;
        }
      }
    }
  }
};

// ------------------------------------------------------------------ pair kernel
// Both producers of a pair load their halves; completion is counted on the pair
// leader's full barrier, which expects the bytes landing in both CTAs.  The leader's
// UMMA warp commits to the empty and tmem-full barriers of both CTAs.  Each CTA's
// epilogue reads its own 128 TMEM lanes (rows) and arrives on the leader's
// tmem-empty barrier.
template <int EPI, bool A_MN, bool B_MN, int TN>
__global__ void __launch_bounds__(pair_threads<EPI>(), 1)
    flce_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB, const GemmShape sh,
                          const EpiArgs ea) {
  using C = PairCfg<TN, epi_warps<EPI>()>;
  constexpr int EW = epi_warps<EPI>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + C::STAGES * C::A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + C::STAGES * C::B_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* tfull = bars + 2 * C::STAGES;
  uint64_t* tempty = bars + 2 * C::STAGES + C::NACC;
  uint64_t* rfull = bars + 2 * C::STAGES + 2 * C::NACC;  // tile ring: slot written
  uint64_t* rempty = rfull + TILE_RING;                  // tile ring: slot read by all
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(rempty + TILE_RING);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  volatile int* ring = reinterpret_cast<volatile int*>(tmem_holder + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t prank = cluster_ctarank();  // 0: pair leader, 1: its peer
  constexpr uint32_t kLead = 0;
  constexpr uint16_t kPairMask = 0x3;  // both CTAs of the pair
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(cluster_count_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);  // the leader's commit
    }
    for (int a = 0; a < C::NACC; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * EW);
    }
    for (int r = 0; r < TILE_RING; ++r) {
      mbar_init(&rfull[r], 1);  // the scheduler publishes
      // (peer's copy) read by: both producers, the leader's UMMA warp, every epilogue
      // warp of both CTAs
      mbar_init(&rempty[r], 3 + 2 * EW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc_pair(tmem_holder, TMEM_COLS);
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const int total = sh.m_tiles * sh.n_tiles;
  constexpr uint32_t kSched = 1;  // the CTA whose warp 1 schedules the pair's tiles
  const uint32_t rempty_sched = mapa_shared(smem_u32(&rempty[0]), kSched);

  // The i-th tile of this pair, read from ring slot i % TILE_RING once published (a
  // value >= total ends the schedule); the read is then acknowledged to the scheduler.
  // The acknowledgement is a relaxed arrive: the acquire load orders it after the
  // read, so the scheduler cannot overwrite the slot before it was read, and no role
  // (the UMMA issuer in particular) waits for its own earlier memory operations.
  auto take_tile = [&](int i, bool ack) -> int {
    const int slot = i % TILE_RING;
    if (!mbar_wait<true>(&rfull[slot], (i / TILE_RING) & 1, abort_flag, ea.err)) return total;
    const int t = ld_acquire_shared(ring + slot);
    if (ack) mbar_arrive_cluster_relaxed(rempty_sched + slot * 8);
    return t;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs)
      const uint64_t pol_a = l2_policy(sh.a_hint);
      const uint64_t pol_b = l2_policy(sh.b_hint);
      const uint32_t abort_peer =
          mapa_shared(smem_u32(const_cast<int*>(abort_flag)), prank ^ 1u);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int t = take_tile(i, true);
        if (t >= total) break;
        int mt, nt;
        tile_coords(t, sh, mt, nt);
        const int am0 = mt * PAIR_BM + static_cast<int>(prank) * 128 + sh.a_mn_off;
        const int bn0 = nt * TN + static_cast<int>(prank) * C::B_ROWS + sh.b_mn_off;
        for (int kb = 0; kb < sh.k_blocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, ea.err)) {
            ok = false;
            break;
          }
          const uint32_t fb = mapa_shared(smem_u32(&full[stage]), kLead);
          if (prank == 0) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
          const int k0 = kb * BK;
          const bool in_a = load_operand<A_MN, 128>(sA + stage * C::A_BYTES, &tmA, fb, am0,
                                                    k0 + sh.a_k_off, pol_a, sh.a_inner,
                                                    sh.a_outer);
          const bool in_b = in_a && load_operand<B_MN, C::B_ROWS>(
                                        sB + stage * C::B_BYTES, &tmB, fb, bn0,
                                        k0 + sh.b_k_off, pol_b, sh.b_inner, sh.b_outer);
          if (!in_b) {
            // (FLCE_DEBUG build only) a box out of range was not loaded: its stage can
            // never fill, so stop both CTAs of the pair instead of letting them wait
            atomicOr(ea.err, FLCE_DEVERR_BOUNDS);
            *abort_flag = 1;
            st_shared_cluster_u32(abort_peer, 1u);
            ok = false;
            break;
          }
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // drain: every stage this CTA filled has been released by the leader's UMMAs
      // (its commits target this CTA's barriers, so they must land before exit)
      for (int i = 0; i < C::STAGES && ok; ++i) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, ea.err)) break;
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1 && prank == kSched) {
    if (lane == 0) {
      // ---------------- tile scheduler (the peer CTA's warp 1)
      const uint32_t ring_lead = mapa_shared(smem_u32(const_cast<int*>(ring)), kLead);
      const uint32_t rfull_lead = mapa_shared(smem_u32(&rfull[0]), kLead);
      int t = cid;  // the pair's first tile; later ones come from the counter
      for (int i = 0;; ++i) {
        const int slot = i % TILE_RING;
        if (!mbar_wait<true>(&rempty[slot], ((i / TILE_RING) & 1) ^ 1u, abort_flag, ea.err))
          break;
        ring[slot] = t;
        st_shared_cluster_u32(ring_lead + slot * 4, static_cast<uint32_t>(t));
        mbar_arrive_local(&rfull[slot]);
        mbar_arrive_cluster(rfull_lead + slot * 8);
        if (t >= total) break;
        t = ncl + static_cast<int>(atomicAdd(sh.sched, 1u));
      }
      // this pair draws no more tiles; the last pair to get here resets the counters
      // (every other pair's draws happened before its increment)
      __threadfence();
      if (atomicAdd(sh.sched + 1, 1u) == static_cast<unsigned int>(ncl - 1)) {
        __threadfence();
        atomicExch(sh.sched, 0u);
        atomicExch(sh.sched + 1, 0u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && prank == 0) {
      // ---------------- UMMA issuer (pair leaders only)
      constexpr uint32_t IDESC = idesc_bf16_f32(PAIR_BM, TN, A_MN, B_MN);
      // Shared-memory descriptors of stage 0, k-slice 0, computed once: the start-address
      // field (bits 0-13, address >> 4; every address here is below 2^18) then advances by a
      // stage's bytes >> 4 and a k-slice's offset >> 4.  Rebuilding all eight descriptors
      // every k-block kept the UMMA thread busy enough that, with the epilogue's arithmetic
      // beside it on the SM, the tensor pipe starved: the soft-capped Gemma-2 forward lost
      // twice the cycles.
      const uint64_t a_desc0 = operand_desc<A_MN>(smem_u32(sA), 0, sh);
      const uint64_t b_desc0 = operand_desc<B_MN>(smem_u32(sB), 0, sh);
      constexpr uint64_t kKA = (A_MN ? UK * 128 : UK * 2) >> 4;
      constexpr uint64_t kKB = (B_MN ? UK * 128 : UK * 2) >> 4;
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        if (take_tile(it, true) >= total) break;
        const int acc = it % C::NACC;
        const uint32_t aph = (it / C::NACC) & 1;
        // the epilogues of both CTAs arrive here (cluster-scope acquire)
        if (!mbar_wait<true>(&tempty[acc], aph ^ 1u, abort_flag, ea.err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * TN;
        for (int kb = 0; kb < sh.k_blocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, ea.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t a_st = a_desc0 + stage * (C::A_BYTES >> 4);
          const uint64_t b_st = b_desc0 + stage * (C::B_BYTES >> 4);
          uint64_t ad[BK / UK], bd[BK / UK];
#pragma unroll
          for (int kk = 0; kk < BK / UK; ++kk) {
            ad[kk] = a_st + kk * kKA;
            bd[kk] = b_st + kk * kKB;
          }
          umma_bf16_pair_x4(d_tmem, ad, bd, IDESC, kb != 0 ? 1u : 0u);
          umma_commit_pair(&empty[stage], kPairMask);
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit_pair(&tfull[acc], kPairMask);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps (both CTAs)
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    const uint32_t tempty_leader = mapa_shared(smem_u32(&tempty[0]), kLead);
    for (int it = 0;; ++it) {
      const int t = take_tile(it, false);
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(rempty_sched + (it % TILE_RING) * 8);
      if (t >= total) break;
      int mt, nt;
      tile_coords(t, sh, mt, nt);
      const int acc = it % C::NACC;
      const uint32_t aph = (it / C::NACC) & 1;
      if (!mbar_wait(&tfull[acc], aph, abort_flag, ea.err)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * TN +
                             half * C::EPI_COLS;
      if (FLCE_CHECK(tmem_ok(acc * TN + half * C::EPI_COLS, C::EPI_CHUNKS * 32, q, warp),
                     ea.err))
        Epilogue<EPI>::template run<C::EPI_CHUNKS>(
            ea, tbase, mt * PAIR_BM + static_cast<int>(prank) * 128 + r,
            nt * TN + half * C::EPI_COLS);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader + acc * 8);
    }
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// Host-side launcher of the pair kernel: clusters of 2 CTAs, as many as can be
// resident at once (persistent), never more than there are tiles.
template <int EPI, bool A_MN, bool B_MN, int TN>
cudaError_t launch_gemm_pair(const CUtensorMap& tmA, const CUtensorMap& tmB,
                             const GemmShape& sh, const EpiArgs& ea, int max_clusters,
                             cudaStream_t stream) {
  using C = PairCfg<TN, epi_warps<EPI>()>;
  auto kern = flce_gemm_pair_kernel<EPI, A_MN, B_MN, TN>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if (sh.m_tiles <= 0 || sh.n_tiles <= 0) return cudaSuccess;
  if (!sh.sched) return cudaErrorInvalidValue;  // the dynamic schedule's counters
  constexpr int csize = 2;
  const int total = sh.m_tiles * sh.n_tiles;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(pair_threads<EPI>(), 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int clusters = total < max_clusters ? total : max_clusters;
  cfg.gridDim = dim3(csize * clusters, 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, sh, ea);
}

// Largest number of co-resident CTA pairs of this kernel on the current device.
template <int EPI, bool A_MN, bool B_MN, int TN>
cudaError_t pair_max_clusters(int* out) {
  using C = PairCfg<TN, epi_warps<EPI>()>;
  auto kern = flce_gemm_pair_kernel<EPI, A_MN, B_MN, TN>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(pair_threads<EPI>(), 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(out, kern, &cfg);
}

// Launch with the co-resident pair count of this instantiation, queried once per
// device (the query needs the kernel's attributes set, so it is cached here).
template <int EPI, bool A_MN, bool B_MN, int TN>
cudaError_t launch_pair_cached(const CUtensorMap& tmA, const CUtensorMap& tmB,
                               const GemmShape& sh, const EpiArgs& ea, cudaStream_t stream) {
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int mc = max_clusters[dev].load();
  if (mc <= 0) {
    e = pair_max_clusters<EPI, A_MN, B_MN, TN>(&mc);
    if (e != cudaSuccess) return e;
    if (mc <= 0) return cudaErrorInvalidConfiguration;
    max_clusters[dev].store(mc);
  }
  return launch_gemm_pair<EPI, A_MN, B_MN, TN>(tmA, tmB, sh, ea, mc, stream);
}

// CTA pairs that fit on the current device at once; every pair kernel takes a
// whole SM's shared memory, so one query serves them all.  0 if the query fails.
int pair_capacity();

// Launchers of the instantiations the path uses (one translation unit each).
#define FLCE_DECLARE_LAUNCHER(name)                                                  \
  cudaError_t name(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmShape& sh, \
                   const EpiArgs& ea, cudaStream_t stream)
#define FLCE_DEFINE_LAUNCHER(name, EPI, A_MN, B_MN, TN)                                  \
  FLCE_DECLARE_LAUNCHER(name) {                                                          \
    return launch_pair_cached<EPI, A_MN, B_MN, TN>(tmA, tmB, sh, ea, stream);           \
  }

// weight stored [H, V]
FLCE_DECLARE_LAUNCHER(launch_fwd_stats);     // hidden (K) x weight (MN)
FLCE_DECLARE_LAUNCHER(launch_bwd_dlogits);   // hidden (K) x weight (MN)
FLCE_DECLARE_LAUNCHER(launch_bwd_dweight);   // hidden^T (MN) x dlogits (MN); also dlogits^T (MN) x hidden (MN)
FLCE_DECLARE_LAUNCHER(launch_bwd_dweight_acc);  // the same, fp32-accumulated over token chunks
FLCE_DECLARE_LAUNCHER(launch_bwd_dhidden);   // dlogits (K) x weight (K)
// weight stored [V, H] (the nn.Linear layout)
FLCE_DECLARE_LAUNCHER(launch_fwd_stats_vh);    // hidden (K) x weight (K)
FLCE_DECLARE_LAUNCHER(launch_bwd_dlogits_vh);  // hidden (K) x weight (K)
FLCE_DECLARE_LAUNCHER(launch_bwd_dhidden_vh);  // dlogits (K) x weight (MN)

}  // namespace flce
