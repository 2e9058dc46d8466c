// C ABI of libflce.so: argument checks, workspace layout, TMA descriptors and
// the launch sequence of the forward and backward passes (declared in flce.h).
//
// Forward  (verl PR #462, "Equivalent compute logic", without the [N,V] logits):
//   1. fwd_stats GEMM: hidden @ weight tile by tile, each row's 256 columns of a
//      tile reduced to online-softmax partials (m, d, s) plus the label logit.
//   2. fwd_combine: merge the partials of a row -> lse, E_p[z], CE, entropy,
//      z-loss, ignore mask (Liger-Kernel PR #551 / PR #435 semantics).
//   3. reduce (mean/sum only): fixed-order fp64 sum over rows.
// Backward, per vocabulary chunk of width Vc (after a per-row prep kernel):
//   4. bwd_dlogits GEMM: recompute logits, write dlogits[N, Vc] (bf16).
//   5. bwd_dhidden GEMM: dhidden (fp32 accumulator) += dlogits @ weight[:, chunk]^T;
//      the last chunk writes bf16.
//   6. bwd_dweight GEMM, beside dhidden on a side stream: dweight[:, chunk] =
//      hidden^T @ dlogits.
// Forward + backward in one call (gradient in forward), per chunk of tokens:
//   1. fwd_stats GEMM that also keeps the raw fp32 logits of the chunk,
//   2. combine, prep, then dlogits from the kept logits (no recompute),
//   3. dhidden rows of the chunk = dlogits @ weight^T (all of V in one GEMM), and
//      beside it on the side stream dweight = hidden^T @ dlogits, written once (one
//      chunk) or accumulated.
// Every GEMM hands its tiles out dynamically from counters in the workspace header.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/flce.h"
#include "flce_gemm.cuh"
#include "flce_kernels.cuh"

namespace flce {

namespace {

constexpr int kVersion = 300;  // 0.3.0: flce_params.dhidden_fp32, flce_check_params, FLCE_ERR_BOUNDS, flce_plan_tiles without operand sharing
constexpr size_t kHeaderBytes = 256;
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;
// dlogits chunk target of the backward: fewer, wider chunks mean fewer fp32 passes
// over the dhidden accumulator, fewer partly idle last rounds of tiles and longer
// k-loops (1 GiB measured 3-4 % faster than 256 MB on the Llama-3, Qwen2.5 and Gemma-2
// head shapes; 2 GiB 0.3-0.5 % faster than 1 GiB on Llama-3 and Qwen2.5, the same on
// Gemma-2; 4 GiB no faster than 2)
constexpr int64_t kDefaultChunkBytes = int64_t(2) << 30;

// Descriptor strides of the MN-major operand tiles: 64-wide MN atoms 8 KB apart
// (leading byte offset), 8-row K groups 1 KB apart (stride byte offset).
constexpr uint32_t kMnLbo = MN_ATOM_BYTES;
constexpr uint32_t kMnSbo = 1024;

// ------------------------------------------------------------ host helpers
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline size_t align4k(size_t x) { return (x + 4095) & ~size_t(4095); }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct FwdLayout {
  size_t pm, pd, ps, psw, zlabel, loss_row, ent_row, total;
  int64_t n_parts;
};

constexpr size_t kWsumOffset = 64;  // float in the workspace header: sum of class weights
// Pairs of uint32 counters of the GEMMs' dynamic tile schedule in the workspace header
// (zeroed with the header at the start of every call, and by each GEMM at its end):
// slot 0 for the GEMMs on the caller's stream, slot 1 for dweight, which runs beside
// dhidden on the side stream.
constexpr size_t kSchedOffset = 128;

inline unsigned int* sched_counters(uint32_t* header, int slot = 0) {
  return reinterpret_cast<unsigned int*>(reinterpret_cast<uint8_t*>(header) + kSchedOffset +
                                         8 * slot);
}

FwdLayout fwd_layout(const flce_params* p) {
  FwdLayout L{};
  L.n_parts = PairCfg<TN_FWD, epi_warps<EPI_FWD_STATS>()>::PARTS * cdiv(p->V, TN_FWD);  // parts per tile x tiles
  const size_t part_bytes = align256(static_cast<size_t>(L.n_parts * p->N) * 4);
  const size_t row_bytes = align256(static_cast<size_t>(p->N) * 4);
  size_t off = kHeaderBytes;
  L.pm = off; off += part_bytes;
  L.pd = off; off += part_bytes;
  L.ps = off; off += part_bytes;
  L.psw = off;
  if (p->label_smoothing != 0.0f) off += part_bytes;
  L.zlabel = off; off += row_bytes;
  L.loss_row = off; off += row_bytes;
  L.ent_row = off; off += row_bytes;
  L.total = off;
  return L;
}

struct BwdLayout {
  size_t rowc, rowd, dl, acc, total;
  int64_t Vc, chunks;
};

int64_t chunk_width(const flce_params* p) {
  constexpr int64_t kAlign = 256;  // chunk widths are whole tiles of every kernel
  const int64_t vfull = cdiv(p->V, kAlign) * kAlign;
  int64_t vc = p->chunk_v;
  if (vc <= 0) {
    const int64_t n = p->N > 0 ? p->N : 1;
    vc = (kDefaultChunkBytes / (2 * n)) / kAlign * kAlign;
  }
  if (vc < kAlign) vc = kAlign;
  if (vc > vfull) vc = vfull;
  return vc;
}

BwdLayout bwd_layout(const flce_params* p) {
  BwdLayout L{};
  L.Vc = chunk_width(p);
  L.chunks = cdiv(p->V, L.Vc);
  size_t off = kHeaderBytes;
  L.rowc = off; off += align256(static_cast<size_t>(p->N) * 16);
  L.rowd = off;
  if (p->label_smoothing != 0.0f) off += align256(static_cast<size_t>(p->N) * 4);
  L.dl = off; off += align256(static_cast<size_t>(p->N) * L.Vc * 2);
  L.acc = off;
  // several chunks accumulate dhidden in fp32: here, unless the caller's fp32 dhidden
  // is the accumulator itself
  if (L.chunks > 1 && !p->dhidden_fp32) off += align256(static_cast<size_t>(p->N) * p->H * 4);
  L.total = off;
  return L;
}

// Token chunk of flce_forward_backward: the rows whose fp32 logits and bf16
// dlogits fit FLCE_FUSED_BUDGET, a multiple of 512 rows (two pair tiles), capped
// at N rounded up to a whole 256-row tile.
#ifndef FLCE_FUSED_BUDGET
#define FLCE_FUSED_BUDGET (int64_t(8) << 30)
#endif

struct FusedLayout {
  size_t pm, pd, ps, psw, zlabel, loss_row, ent_row, rowc, rowd, z, dl, dwacc, total;
  int64_t Nc, chunks, ldz, n_parts;
};

FusedLayout fused_layout(const flce_params* p) {
  FusedLayout L{};
  L.ldz = cdiv(p->V, 256) * 256;
  int64_t nc = p->chunk_n;
  if (nc <= 0) nc = FLCE_FUSED_BUDGET / (L.ldz * 6) / 512 * 512;
  if (nc < 512) nc = 512;
  const int64_t ncap = cdiv(p->N > 0 ? p->N : 1, 256) * 256;
  L.Nc = nc < ncap ? nc : ncap;
  L.chunks = cdiv(p->N, L.Nc);
  L.n_parts = PairCfg<TN_FWD, epi_warps<EPI_FWD_STATS>()>::PARTS * cdiv(p->V, TN_FWD);
  const size_t part_bytes = align256(static_cast<size_t>(L.n_parts * L.Nc) * 4);
  const size_t chunk_row_bytes = align256(static_cast<size_t>(L.Nc) * 4);
  const size_t row_bytes = align256(static_cast<size_t>(p->N) * 4);
  size_t off = kHeaderBytes;
  L.pm = off; off += part_bytes;
  L.pd = off; off += part_bytes;
  L.ps = off; off += part_bytes;
  L.psw = off;
  if (p->label_smoothing != 0.0f) off += part_bytes;
  L.zlabel = off; off += chunk_row_bytes;
  L.loss_row = off; off += row_bytes;
  L.ent_row = off; off += row_bytes;
  L.rowc = off; off += align256(static_cast<size_t>(L.Nc) * 16);
  L.rowd = off;
  if (p->label_smoothing != 0.0f) off += chunk_row_bytes;
  // the kept logits and the dlogits start on 4 KB boundaries: dlogits_from_z, which
  // streams them, measured up to 4 % slower with rows starting 256 bytes past one
  off = align4k(off);
  L.z = off; off = align4k(off + static_cast<size_t>(L.Nc * L.ldz) * 4);
  L.dl = off; off += align256(static_cast<size_t>(L.Nc * L.ldz) * 2);
  L.dwacc = off;
  if (L.chunks > 1) off += align256(static_cast<size_t>(p->H * p->V) * 4);
  L.total = off;
  return L;
}

int check_params(const flce_params* p) {
  if (!p) return FLCE_ERR_BAD_ARG;
  if (p->reduction < FLCE_RED_NONE || p->reduction > FLCE_RED_SUM) return FLCE_ERR_BAD_ARG;
  if (!(p->zloss_coef >= 0.0f) || !(p->softcap >= 0.0f)) return FLCE_ERR_BAD_ARG;
  if (p->N < 0 || p->H < 8 || p->V < 1) return FLCE_ERR_BAD_SHAPE;
  if (p->N > kMaxDim || p->H > kMaxDim || p->V > kMaxDim) return FLCE_ERR_BAD_SHAPE;
  // row strides of the TMA engine are multiples of 16 bytes: H always (hidden, a [V,H]
  // weight), V only where it is a row length (a [H,V] weight and its dweight)
  if (p->H % 8 != 0) return FLCE_ERR_ALIGN;
  if (p->weight_layout == FLCE_WEIGHT_HV && p->V % 8 != 0) return FLCE_ERR_ALIGN;
  if (p->chunk_v < 0 || (p->chunk_v > 0 && p->chunk_v % 256 != 0)) return FLCE_ERR_BAD_ARG;
  if (p->chunk_n < 0 || p->chunk_n % 512 != 0) return FLCE_ERR_BAD_ARG;
  if (p->dhidden_fp32 != 0 && p->dhidden_fp32 != 1) return FLCE_ERR_BAD_ARG;
  if (p->weight_layout != FLCE_WEIGHT_HV && p->weight_layout != FLCE_WEIGHT_VH)
    return FLCE_ERR_BAD_ARG;
  if (!(p->label_smoothing >= 0.0f && p->label_smoothing <= 1.0f)) return FLCE_ERR_BAD_ARG;
  if (p->v_total < 0 || p->v_offset < 0) return FLCE_ERR_BAD_ARG;
  if (p->v_total == 0 && p->v_offset != 0) return FLCE_ERR_BAD_ARG;
  if (p->v_total > 0) {
    if (p->v_offset + p->V > p->v_total || p->v_total > kMaxDim) return FLCE_ERR_BAD_SHAPE;
    if (p->label_smoothing != 0.0f || p->class_weight) return FLCE_ERR_BAD_ARG;
  }
  if (reinterpret_cast<uintptr_t>(p->class_weight) & 3) return FLCE_ERR_ALIGN;
  // chunk-relative and vocabulary column indices are 32-bit inside the kernels
  if (cdiv(p->V, 256) * 256 > kMaxDim) return FLCE_ERR_BAD_SHAPE;
  return FLCE_OK;
}

inline bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; }
// dhidden: bf16 needs 16-byte alignment; fp32 is the accumulator of the 256-bit
// accesses of the dhidden epilogue and needs 32
inline bool dhidden_aligned(const flce_params* p, const void* ptr) {
  return (reinterpret_cast<uintptr_t>(ptr) & (p->dhidden_fp32 ? 31 : 15)) == 0;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the library
// links no libcuda at build time.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// L2 sector promotion of operand loads (CUtensorMapL2promotion: 0 none, 1 64 B,
// 2 128 B, 3 256 B).
#ifndef FLCE_L2_PROMOTION
#define FLCE_L2_PROMOTION 3
#endif

// A 2-D bf16 tensor map and the extents of the array it covers (the FLCE_DEBUG
// build checks every TMA box of a GEMM against them).
struct Map {
  CUtensorMap m;
  int64_t inner = 0, outer = 0;
};

// Tensor map over a row-major [outer, inner] bf16 array with a {box_inner, box_outer}
// box, 128-byte swizzle, zero fill out of bounds.
bool make_map(Map* map, const void* base, int64_t inner, int64_t outer, int64_t row_elems,
              int box_inner, int box_outer) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  map->inner = inner;
  map->outer = outer;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_elems * 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
  cuuint32_t estr[2] = {1, 1};
  return enc(&map->m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             static_cast<CUtensorMapL2promotion>(FLCE_L2_PROMOTION),
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The GEMM's A and B operand extents, from their maps.
void set_extents(GemmShape* sh, const Map& a, const Map& b) {
  sh->a_inner = a.inner;
  sh->a_outer = a.outer;
  sh->b_inner = b.inner;
  sh->b_outer = b.outer;
}

struct DevInfo {
  int sms = 0;
  bool ok = false;
};

int device_info(DevInfo* out) {
  static std::mutex mu;
  static DevInfo cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FLCE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(mu);
  if (!cache[dev].ok) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FLCE_ERR_CUDA;
    if (major != 10 || minor != 3) return FLCE_ERR_DEVICE;
    cache[dev].sms = sms;
    cache[dev].ok = true;
  }
  *out = cache[dev];
  return FLCE_OK;
}

// The error word is copied on `st` itself, after the call's work, so that reading it
// waits for nothing but that stream (a plain cudaMemcpy would also wait for the legacy
// default stream).
int read_status(const void* workspace, cudaStream_t st) {
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return FLCE_ERR_CUDA;
  if (word & FLCE_DEVERR_BOUNDS) return FLCE_ERR_BOUNDS;
  if (word & FLCE_DEVERR_TIMEOUT) return FLCE_ERR_TIMEOUT;
  if (word & FLCE_DEVERR_LABEL) return FLCE_ERR_LABEL;
  return FLCE_OK;
}

inline int cuda_rc(cudaError_t e) { return e == cudaSuccess ? FLCE_OK : FLCE_ERR_CUDA; }

// dweight and dhidden read the same dlogits and write different outputs, so they run
// concurrently: dhidden on the caller's stream, dweight on a side stream forked from it
// after the dlogits and joined back before anything reads or rewrites them.  dhidden is
// launched first and takes every SM; as its pairs run out of tiles (its last round of
// tiles is only partly full), dweight's pairs start on the SMs they free, and the
// dynamic tile schedule balances the work between them.  The side stream and its two
// events are created once per host thread and device: events are never shared between
// threads, and a stream wait binds to the record before it, so reusing them across one
// thread's calls is safe.  They are destroyed when the thread exits (destroying a stream
// or an event with work still pending is allowed: the work completes first).
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

struct SideStreams {
  SideStream per_device[64];
  ~SideStreams() {
    for (SideStream& ss : per_device) {
      if (!ss.stream) continue;
      // at process exit the runtime may already be unloaded: the calls then fail
      // harmlessly
      cudaEventDestroy(ss.fork);
      cudaEventDestroy(ss.join);
      cudaStreamDestroy(ss.stream);
    }
  }
};

int side_stream(SideStream** out) {
  thread_local SideStreams cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FLCE_ERR_CUDA;
  SideStream& ss = cache.per_device[dev];
  if (!ss.stream) {
    SideStream n;
    if (cudaStreamCreateWithFlags(&n.stream, cudaStreamNonBlocking) != cudaSuccess)
      return FLCE_ERR_CUDA;
    if (cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming) != cudaSuccess) {
      if (n.fork) cudaEventDestroy(n.fork);
      cudaStreamDestroy(n.stream);
      return FLCE_ERR_CUDA;
    }
    ss = n;
  }
  *out = &ss;
  return FLCE_OK;
}

// Fork: `side` waits for the work enqueued on `st` so far.  Join: `st` waits for `side`.
int fork_side(const SideStream& ss, cudaStream_t st) {
  int rc = cuda_rc(cudaEventRecord(ss.fork, st));
  return rc ? rc : cuda_rc(cudaStreamWaitEvent(ss.stream, ss.fork, 0));
}
int join_side(const SideStream& ss, cudaStream_t st) {
  int rc = cuda_rc(cudaEventRecord(ss.join, ss.stream));
  return rc ? rc : cuda_rc(cudaStreamWaitEvent(st, ss.join, 0));
}

// a_hint / b_hint: the operand whose panels every tile of a group revisits keeps
// its L2 lines (evict_last).  The streamed operand keeps the normal policy: with
// evict_first its tiles left L2 before all the tiles sharing them had read them.
#ifndef FLCE_L2_PANEL_BUDGET
#define FLCE_L2_PANEL_BUDGET (int64_t(40) << 20)
#endif

// Tiles of the fast raster dimension per group so that the panels of the operand
// every tile revisits (each `panel_bytes` long) stay within an L2 budget; the
// other operand is then streamed once per group.
int raster_group(int64_t panel_bytes, int fast_tiles) {
  if (FLCE_L2_PANEL_BUDGET <= 0 || panel_bytes <= 0) return fast_tiles;
  int64_t g = FLCE_L2_PANEL_BUDGET / panel_bytes;
  if (g < 1) g = 1;
  return g < fast_tiles ? static_cast<int>(g) : fast_tiles;
}

// The raster group and L2 policies of one GEMM, from its tile counts and the
// number of CTA pairs (c2) the GPU holds at once: host arithmetic only.
// `panel_bytes` is the revisited operand's size per tile of the fast raster
// dimension.
void plan_tiles_for(GemmShape* sh, int64_t panel_bytes, int64_t c2) {
  const bool m_fast = sh->raster == 0;
  const int fast = m_fast ? sh->m_tiles : sh->n_tiles;
  // When few panels fit the L2 budget, a square-ish set of resident tiles reads
  // fewer distinct rows and columns: the k-steps of all resident tiles advance
  // together (persistent schedule), so only the k-slices in flight need to be in L2.
  int g = 1;
  while (int64_t(g + 1) * (g + 1) <= c2) ++g;
  const int budget_group = raster_group(panel_bytes, fast);
  if (budget_group < g && budget_group < fast) {
    sh->group = g < fast ? g : fast;
    // No panel stays in L2 for long here: an evict_last policy would only pin
    // hundreds of MB of lines that later loads (and later kernels) then miss around.
    sh->a_hint = L2_NORMAL;
    sh->b_hint = L2_NORMAL;
  } else {
    sh->group = budget_group;
  }
}

void plan_tiles(GemmShape* sh, int64_t panel_bytes) {
  plan_tiles_for(sh, panel_bytes, pair_capacity());
}

GemmShape base_shape(int a_hint, int b_hint) {
  GemmShape sh{};
  sh.group = 1 << 30;
  sh.mn_lbo = kMnLbo;
  sh.mn_sbo = kMnSbo;
  sh.a_hint = a_hint;
  sh.b_hint = b_hint;
  return sh;
}

}  // namespace
}  // namespace flce

using namespace flce;

extern "C" {

int flce_version(void) { return kVersion; }

const char* flce_strerror(int code) {
  switch (code) {
    case FLCE_OK: return "ok";
    case FLCE_ERR_BAD_ARG: return "invalid argument";
    case FLCE_ERR_BAD_SHAPE: return "unsupported shape (need N >= 0, H >= 8, V >= 1)";
    case FLCE_ERR_ALIGN:
      return "H (and V of a [H,V] weight) must be multiples of 8 and pointers 16-byte aligned "
             "(fp32 dhidden: 32)";
    case FLCE_ERR_WS_TOO_SMALL: return "workspace smaller than flce_workspace_size()";
    case FLCE_ERR_LABEL: return "label outside [0, V) that is not ignore_index";
    case FLCE_ERR_TIMEOUT: return "device pipeline wait timed out";
    case FLCE_ERR_CUDA: return "CUDA call failed";
    case FLCE_ERR_DEVICE: return "current device is not an sm_103 GPU";
    case FLCE_ERR_BOUNDS:
      return "a device-side bounds check of the FLCE_DEBUG build failed (access skipped)";
    case FLCE_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than flce_forward_noalloc's static 64 MiB array";
    default: return "unknown status";
  }
}

int flce_check_params(const flce_params* p) { return check_params(p); }

size_t flce_workspace_size(const flce_params* p, int phase) {
  if (check_params(p) != FLCE_OK) return 0;
  if (phase == 0) return fwd_layout(p).total;
  if (phase == 1) return bwd_layout(p).total;
  if (phase == 2) return kHeaderBytes + 2 * align256(static_cast<size_t>(p->N) * 4);
  if (phase == 3) return fused_layout(p).total;
  return 0;
}

int flce_kernel_launches(const flce_params* p, int phase) {
  if (check_params(p) != FLCE_OK || p->N == 0) return check_params(p) != FLCE_OK ? -1 : 0;
  const int reduce = p->reduction == FLCE_RED_NONE ? 0 : 1;
  switch (phase) {
    case 0:  // flce_forward: GEMM, [class-weight sum], combine, [reduce]
      return 2 + reduce + (p->label_smoothing != 0.0f && p->class_weight ? 1 : 0);
    case 1:  // flce_backward: prep + 3 GEMMs (dlogits, dhidden, dweight) per vocabulary chunk
      return 1 + 3 * static_cast<int>(bwd_layout(p).chunks);
    case 2:  // flce_combine_shards: combine, [reduce]
      return 1 + reduce;
    case 3:  // flce_shard_stats: GEMM, shard merge
      return 2;
    case 4:  // flce_forward_backward: [class-weight sum], 6 per token chunk, [reduce]
      return 6 * static_cast<int>(fused_layout(p).chunks) + reduce +
             (p->label_smoothing != 0.0f && p->class_weight ? 1 : 0);
    default:
      return -1;
  }
}

int flce_status(const void* workspace, void* stream) {
  if (!workspace) return FLCE_ERR_BAD_ARG;
  return read_status(workspace, static_cast<cudaStream_t>(stream));
}

int flce_plan_tiles(int32_t m_tiles, int32_t n_tiles, int32_t raster, int64_t panel_bytes,
                    int32_t a_hint, int32_t b_hint, int32_t pairs, int32_t* out) {
  if (!out || m_tiles < 1 || n_tiles < 1 || (raster != 0 && raster != 1) || panel_bytes < 0 ||
      a_hint < 0 || a_hint > 2 || b_hint < 0 || b_hint > 2 || pairs < 1)
    return FLCE_ERR_BAD_ARG;
  GemmShape sh = base_shape(a_hint, b_hint);
  sh.m_tiles = m_tiles;
  sh.n_tiles = n_tiles;
  sh.raster = raster;
  plan_tiles_for(&sh, panel_bytes, pairs);
  out[0] = sh.group;
  out[1] = sh.a_hint;
  out[2] = sh.b_hint;
  return FLCE_OK;
}

}  // extern "C"

namespace flce {
namespace {

// Where the forward GEMM's epilogue writes: per-row, per-column-block partials
// (part p of row n at p * part_stride + n), the label logits, and optionally the
// raw fp32 logits [rows, ld_z].
struct StatsOut {
  float *pm, *pd, *ps, *psw, *zlabel, *zout;
  int64_t part_stride, ld_z, n_parts;
};

// Logits tiles of hidden rows [n0, n0 + rows) @ weight reduced to online-softmax
// partials; `labels` points at row n0's label.
int launch_stats(const flce_params* p, const void* hidden, const void* weight,
                 const int64_t* labels, int64_t n0, int64_t rows, const StatsOut& o,
                 uint32_t* err, cudaStream_t st) {
  const int64_t N = p->N, H = p->H, V = p->V;
  const bool vh = p->weight_layout == FLCE_WEIGHT_VH;
  Map tmA, tmB;
  if (!make_map(&tmA, hidden, H, N, H, BK, 64)) return FLCE_ERR_CUDA;
  // weight as B: [H,V] is MN-major, [V,H] K-major ({64,64} boxes either way)
  if (!(vh ? make_map(&tmB, weight, H, V, H, BK, 64)
           : make_map(&tmB, weight, V, H, V, 64, BK)))
    return FLCE_ERR_CUDA;
  // hidden is revisited by every vocabulary tile of its group; the weight streams
  GemmShape sh = base_shape(L2_EVICT_LAST, L2_NORMAL);
  sh.m_tiles = static_cast<int>(cdiv(rows, PAIR_BM));
  sh.n_tiles = static_cast<int>(cdiv(V, TN_FWD));
  sh.k_blocks = static_cast<int>(cdiv(H, BK));
  sh.a_mn_off = static_cast<int>(n0);
  sh.raster = 0;
  sh.sched = sched_counters(err);
  plan_tiles(&sh, int64_t(PAIR_BM) * H * 2);
  EpiArgs ea{};
  ea.rows = static_cast<int>(rows);
  ea.cols = static_cast<int>(V);
  ea.col_base = 0;
  ea.V = V;
  ea.softcap = p->softcap;
  ea.labels = labels;
  ea.label_offset = p->v_offset;
  ea.ignore_index = p->ignore_index;
  ea.pm = o.pm;
  ea.pd = o.pd;
  ea.ps = o.ps;
  ea.part_stride = o.part_stride;
  ea.zlabel = o.zlabel;
  ea.smooth = p->label_smoothing;
  ea.cw = p->class_weight;
  ea.psw = o.psw;
  ea.zout = o.zout;
  ea.ld_z = o.ld_z;
  ea.err = err;
  ea.n_parts = o.n_parts;
  set_extents(&sh, tmA, tmB);
  return cuda_rc((vh ? launch_fwd_stats_vh : launch_fwd_stats)(tmA.m, tmB.m, sh, ea, st));
}

// Stage 1 of the forward over all rows, into the forward workspace layout.
int run_fwd_stats(const flce_params* p, const void* hidden, const void* weight,
                  const int64_t* labels, uint8_t* ws, const FwdLayout& L, uint32_t* err,
                  cudaStream_t st, StatsOut* out) {
  StatsOut o{};
  o.pm = reinterpret_cast<float*>(ws + L.pm);
  o.pd = reinterpret_cast<float*>(ws + L.pd);
  o.ps = reinterpret_cast<float*>(ws + L.ps);
  o.psw = reinterpret_cast<float*>(ws + L.psw);
  o.zlabel = reinterpret_cast<float*>(ws + L.zlabel);
  o.part_stride = p->N;
  o.n_parts = L.n_parts;
  *out = o;
  return launch_stats(p, hidden, weight, labels, 0, p->N, o, err, st);
}

// Stage 2: per-row outputs from the merged parts, then the reduction over rows.
int run_fwd_finish(const flce_params* p, const Parts& pt, const float* zlabel,
                   const int64_t* labels, const Smoothing& sm, float* loss, float* entropy,
                   float* lse, float* ez, uint8_t* ws, size_t loss_row_off, size_t ent_row_off,
                   uint32_t* err, cudaStream_t st) {
  const int64_t N = p->N;
  const int64_t V_all = p->v_total > 0 ? p->v_total : p->V;
  const bool per_token = p->reduction == FLCE_RED_NONE;
  float* loss_row = per_token ? loss : reinterpret_cast<float*>(ws + loss_row_off);
  float* ent_row = per_token ? entropy : reinterpret_cast<float*>(ws + ent_row_off);
  fwd_combine_kernel<<<static_cast<unsigned>(cdiv(N, 32)), 256, 0, st>>>(
      pt, N, zlabel, labels, V_all, p->ignore_index, p->zloss_coef, sm, lse, ez, loss_row,
      ent_row, err);
  int rc = cuda_rc(cudaGetLastError());
  if (rc || per_token) return rc;
  reduce_rows_kernel<<<1, 1024, 0, st>>>(loss_row, ent_row, labels, N, p->ignore_index,
                                         p->reduction == FLCE_RED_MEAN, p->class_weight, lse,
                                         p->zloss_coef, loss, entropy);
  return cuda_rc(cudaGetLastError());
}

// Common entry checks and workspace header reset; returns the status and, on
// success, the stream and the error word.
int begin_call(const void* workspace, size_t ws_bytes, size_t need, void* stream,
               cudaStream_t* st, uint32_t** err) {
  if (ws_bytes < need) return FLCE_ERR_WS_TOO_SMALL;
  DevInfo di;
  int rc = device_info(&di);
  if (rc) return rc;
  *st = static_cast<cudaStream_t>(stream);
  *err = static_cast<uint32_t*>(const_cast<void*>(workspace));
  return cuda_rc(cudaMemsetAsync(const_cast<void*>(workspace), 0, kHeaderBytes, *st));
}

int zero_reduced(const flce_params* p, float* loss, float* entropy, cudaStream_t st) {
  if (p->reduction == FLCE_RED_NONE) return FLCE_OK;
  int rc = cuda_rc(cudaMemsetAsync(loss, 0, 4, st));
  return rc ? rc : cuda_rc(cudaMemsetAsync(entropy, 0, 4, st));
}

}  // namespace
}  // namespace flce

extern "C" {

int flce_forward(const flce_params* p, const void* hidden, const void* weight,
                 const int64_t* labels, float* loss, float* entropy, float* lse, float* ez,
                 void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_params(p);
  if (rc) return rc;
  // a shard's softmax is not the whole vocabulary's: shards use flce_shard_stats
  if (p->v_total > 0 && !(p->v_offset == 0 && p->v_total == p->V)) return FLCE_ERR_BAD_ARG;
  if (!loss || !entropy || !workspace || !weight) return FLCE_ERR_BAD_ARG;
  if (p->N > 0 && (!hidden || !labels || !lse || !ez)) return FLCE_ERR_BAD_ARG;
  if (!aligned16(hidden) || !aligned16(weight) || !aligned16(labels) || !aligned16(loss) ||
      !aligned16(entropy) || !aligned16(lse) || !aligned16(ez) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255))
    return FLCE_ERR_ALIGN;
  const FwdLayout L = fwd_layout(p);
  cudaStream_t st;
  uint32_t* err;
  if ((rc = begin_call(workspace, ws_bytes, L.total, stream, &st, &err))) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (p->N == 0) {
    if ((rc = zero_reduced(p, loss, entropy, st))) return rc;
    return p->validate ? read_status(ws, st) : FLCE_OK;
  }
  StatsOut ea;
  if ((rc = run_fwd_stats(p, hidden, weight, labels, ws, L, err, st, &ea))) return rc;
  Smoothing sm{p->label_smoothing, p->class_weight, ea.psw, nullptr};
  if (p->label_smoothing != 0.0f && p->class_weight) {
    float* wsum = reinterpret_cast<float*>(ws + kWsumOffset);
    class_weight_sum_kernel<<<1, 1024, 0, st>>>(p->class_weight, p->V, wsum);
    if ((rc = cuda_rc(cudaGetLastError()))) return rc;
    sm.wsum = wsum;
  }
  const Parts pt{ea.pm, ea.pd, ea.ps, nullptr, L.n_parts, p->N};
  if ((rc = run_fwd_finish(p, pt, ea.zlabel, labels, sm, loss, entropy, lse, ez, ws,
                           L.loss_row, L.ent_row, err, st)))
    return rc;
  return p->validate ? read_status(ws, st) : FLCE_OK;
}

int flce_shard_stats(const flce_params* p, const void* hidden, const void* weight,
                     const int64_t* labels, float* stats, void* workspace, size_t ws_bytes,
                     void* stream) {
  int rc = check_params(p);
  if (rc) return rc;
  if (!stats || !workspace || !weight) return FLCE_ERR_BAD_ARG;
  if (p->N > 0 && (!hidden || !labels)) return FLCE_ERR_BAD_ARG;
  if (!aligned16(hidden) || !aligned16(weight) || !aligned16(labels) || !aligned16(stats) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255))
    return FLCE_ERR_ALIGN;
  const FwdLayout L = fwd_layout(p);
  cudaStream_t st;
  uint32_t* err;
  if ((rc = begin_call(workspace, ws_bytes, L.total, stream, &st, &err))) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (p->N > 0) {
    StatsOut ea;
    if ((rc = run_fwd_stats(p, hidden, weight, labels, ws, L, err, st, &ea))) return rc;
    shard_stats_kernel<<<static_cast<unsigned>(cdiv(p->N, 32)), 256, 0, st>>>(
        ea.pm, ea.pd, ea.ps, L.n_parts, p->N, ea.zlabel, labels, p->v_offset, p->V, stats);
    if ((rc = cuda_rc(cudaGetLastError()))) return rc;
  }
  return p->validate ? read_status(ws, st) : FLCE_OK;
}

int flce_combine_shards(const flce_params* p, const float* stats, int32_t n_shards,
                        const int64_t* labels, float* loss, float* entropy, float* lse,
                        float* ez, void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_params(p);
  if (rc) return rc;
  if (n_shards < 1 || !loss || !entropy || !workspace) return FLCE_ERR_BAD_ARG;
  if (p->N > 0 && (!stats || !labels || !lse || !ez)) return FLCE_ERR_BAD_ARG;
  if (!aligned16(stats) || !aligned16(labels) || !aligned16(loss) || !aligned16(entropy) ||
      !aligned16(lse) || !aligned16(ez) || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return FLCE_ERR_ALIGN;
  const size_t row_bytes = align256(static_cast<size_t>(p->N) * 4);
  cudaStream_t st;
  uint32_t* err;
  if ((rc = begin_call(workspace, ws_bytes, kHeaderBytes + 2 * row_bytes, stream, &st, &err)))
    return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (p->N == 0) {
    if ((rc = zero_reduced(p, loss, entropy, st))) return rc;
    return p->validate ? read_status(ws, st) : FLCE_OK;
  }
  const int64_t N = p->N;
  const Parts pt{stats, stats + N, stats + 2 * N, stats + 3 * N, n_shards, 4 * N};
  const Smoothing sm{0.0f, nullptr, nullptr, nullptr};
  if ((rc = run_fwd_finish(p, pt, nullptr, labels, sm, loss, entropy, lse, ez, ws, kHeaderBytes,
                           kHeaderBytes + row_bytes, err, st)))
    return rc;
  return p->validate ? read_status(ws, st) : FLCE_OK;
}

int flce_backward(const flce_params* p, const void* hidden, const void* weight,
                  const int64_t* labels, const float* lse, const float* ez,
                  const float* g_loss, const float* g_entropy, void* dhidden, void* dweight,
                  void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_params(p);
  if (rc) return rc;
  if (!weight || !dweight || !workspace) return FLCE_ERR_BAD_ARG;
  if (p->N > 0 && (!hidden || !labels || !lse || !ez || !dhidden)) return FLCE_ERR_BAD_ARG;
  if (!aligned16(hidden) || !aligned16(weight) || !aligned16(labels) || !aligned16(lse) ||
      !aligned16(ez) || !dhidden_aligned(p, dhidden) || !aligned16(dweight) ||
      (reinterpret_cast<uintptr_t>(g_loss) & 3) || (reinterpret_cast<uintptr_t>(g_entropy) & 3) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255))
    return FLCE_ERR_ALIGN;
  const BwdLayout L = bwd_layout(p);
  if (ws_bytes < L.total) return FLCE_ERR_WS_TOO_SMALL;
  DevInfo di;
  if ((rc = device_info(&di))) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* err = reinterpret_cast<uint32_t*>(ws);
  if ((rc = cuda_rc(cudaMemsetAsync(ws, 0, kHeaderBytes, st)))) return rc;
  const int64_t N = p->N, H = p->H, V = p->V;

  if (N == 0) {
    // no rows: dweight = 0 (dhidden has no elements)
    if ((rc = cuda_rc(cudaMemsetAsync(dweight, 0, static_cast<size_t>(H * V) * 2, st))))
      return rc;
    return p->validate ? read_status(ws, st) : FLCE_OK;
  }

  SideStream* ss = nullptr;
  if ((rc = side_stream(&ss))) return rc;
  float4* rowc = reinterpret_cast<float4*>(ws + L.rowc);
  __nv_bfloat16* dl = reinterpret_cast<__nv_bfloat16*>(ws + L.dl);
  float* acc = reinterpret_cast<float*>(ws + L.acc);
  float* rowd = reinterpret_cast<float*>(ws + L.rowd);
  bwd_prep_kernel<<<1, 1024, 0, st>>>(labels, labels, N, lse, ez, g_loss, g_entropy, N, V,
                                      p->ignore_index,
                                      p->reduction == FLCE_RED_NONE,
                                      p->reduction == FLCE_RED_MEAN, p->zloss_coef,
                                      p->label_smoothing, p->class_weight, rowc, rowd);
  if ((rc = cuda_rc(cudaGetLastError()))) return rc;

  // Operand tensor maps.  hidden: K-major (recompute) and MN-major (dweight);
  // dlogits chunk: MN-major (dweight) and K-major (dhidden); weight: as the
  // recompute's B and as dhidden's B, each K- or MN-major depending on its layout.
  const bool vh = p->weight_layout == FLCE_WEIGHT_VH;
  Map mHidK, mHidMn, mDlMn, mDlK, mWRec, mWDh;
  bool ok = make_map(&mHidK, hidden, H, N, H, BK, 64) &&
            make_map(&mHidMn, hidden, H, N, H, 64, BK) &&
            make_map(&mDlMn, dl, L.Vc, N, L.Vc, 64, BK) &&
            make_map(&mDlK, dl, L.Vc, N, L.Vc, BK, 64);
  if (vh)
    ok = ok && make_map(&mWRec, weight, H, V, H, BK, 64) &&
         make_map(&mWDh, weight, H, V, H, 64, BK);
  else
    ok = ok && make_map(&mWRec, weight, V, H, V, 64, BK) &&
         make_map(&mWDh, weight, V, H, V, BK, 64);
  if (!ok) return FLCE_ERR_CUDA;

  for (int64_t c = 0; c < L.chunks; ++c) {
    const int64_t v0 = c * L.Vc;
    const int64_t w = (V - v0) < L.Vc ? (V - v0) : L.Vc;

    // dlogits[N, w] = f(hidden @ weight[:, v0:v0+w])
    GemmShape s3 = base_shape(L2_EVICT_LAST, L2_NORMAL);
    s3.m_tiles = static_cast<int>(cdiv(N, PAIR_BM));
    s3.n_tiles = static_cast<int>(cdiv(w, TN_DLOGITS));
    s3.k_blocks = static_cast<int>(cdiv(H, BK));
    s3.raster = 0;
    s3.sched = sched_counters(err);
    plan_tiles(&s3, int64_t(PAIR_BM) * H * 2);
    s3.b_mn_off = static_cast<int>(v0);
    EpiArgs e3{};
    e3.rows = static_cast<int>(N);
    e3.cols = static_cast<int>(w);
    e3.col_base = static_cast<int>(v0);
    e3.V = V;
    e3.softcap = p->softcap;
    e3.labels = labels;
    e3.label_offset = p->v_offset;
    e3.ignore_index = p->ignore_index;
    e3.rowc = rowc;
    e3.rowd = rowd;
    e3.smooth = p->label_smoothing;
    e3.cw = p->class_weight;
    e3.dl = dl;
    e3.ld_dl = L.Vc;
    e3.err = err;
    set_extents(&s3, mHidK, mWRec);
    if ((rc = cuda_rc((vh ? launch_bwd_dlogits_vh : launch_bwd_dlogits)(mHidK.m, mWRec.m, s3, e3,
                                                                        st))))
      return rc;

    // dweight for the chunk, written once: [H,V] -> dweight[:, v0:v0+w] = hidden^T @ dlogits
    // (rows h, hidden^T revisited); [V,H] -> dweight[v0:v0+w, :] = dlogits^T @ hidden
    // (rows v, hidden revisited as B).  Both operands are MN-major views.
    GemmShape s4 = vh ? base_shape(L2_NORMAL, L2_EVICT_LAST) : base_shape(L2_EVICT_LAST, L2_NORMAL);
    s4.k_blocks = static_cast<int>(cdiv(N, BK));
    s4.sched = sched_counters(err, 1);
    EpiArgs e4{};
    e4.V = V;
    e4.err = err;
    e4.col_base = 0;
    if (vh) {
      s4.m_tiles = static_cast<int>(cdiv(w, PAIR_BM));
      s4.n_tiles = static_cast<int>(cdiv(H, TN_DWEIGHT));
      s4.raster = 1;
      plan_tiles(&s4, int64_t(TN_DWEIGHT) * N * 2);
      e4.rows = static_cast<int>(w);
      e4.cols = static_cast<int>(H);
      e4.out = static_cast<__nv_bfloat16*>(dweight) + v0 * H;
      e4.ld_out = H;
    } else {
      s4.m_tiles = static_cast<int>(cdiv(H, PAIR_BM));
      s4.n_tiles = static_cast<int>(cdiv(w, TN_DWEIGHT));
      s4.raster = 0;
      plan_tiles(&s4, int64_t(PAIR_BM) * N * 2);
      e4.rows = static_cast<int>(H);
      e4.cols = static_cast<int>(w);
      e4.col_base = static_cast<int>(v0);
      e4.out = static_cast<__nv_bfloat16*>(dweight);
      e4.ld_out = V;
    }
    set_extents(&s4, vh ? mDlMn : mHidMn, vh ? mHidMn : mDlMn);

    // dhidden (+)= dlogits @ weight[:, v0:v0+w]^T
    // the weight chunk is revisited by every row tile; dlogits rows streamed
    GemmShape s5 = base_shape(L2_NORMAL, L2_EVICT_LAST);
    s5.m_tiles = static_cast<int>(cdiv(N, PAIR_BM));
    s5.n_tiles = static_cast<int>(cdiv(H, TN_DHIDDEN));
    s5.k_blocks = static_cast<int>(cdiv(w, BK));
    s5.raster = 1;
    s5.sched = sched_counters(err);
    plan_tiles(&s5, int64_t(TN_DHIDDEN) * w * 2);
    s5.b_k_off = static_cast<int>(v0);
    EpiArgs e5{};
    e5.rows = static_cast<int>(N);
    e5.cols = static_cast<int>(H);
    e5.V = V;
    e5.ld_acc = H;
    if (p->dhidden_fp32) {
      // the caller's fp32 dhidden is the accumulator: stored by the first chunk,
      // added to by the others, never rounded
      e5.acc = static_cast<float*>(dhidden);
      e5.acc_mode = c == 0 ? ACC_FIRST : ACC_MID;
    } else {
      e5.acc = acc;
      e5.acc_out = static_cast<__nv_bfloat16*>(dhidden);
      e5.acc_mode = L.chunks == 1 ? ACC_ONLY
                    : c == 0      ? ACC_FIRST
                    : c == L.chunks - 1 ? ACC_LAST
                                        : ACC_MID;
    }
    e5.err = err;
    set_extents(&s5, mDlK, mWDh);

    // dhidden on the caller's stream, dweight beside it on the side stream (SideStream)
    if ((rc = fork_side(*ss, st))) return rc;
    if ((rc = cuda_rc((vh ? launch_bwd_dhidden_vh : launch_bwd_dhidden)(mDlK.m, mWDh.m, s5, e5,
                                                                        st))))
      return rc;
    if ((rc = cuda_rc(vh ? launch_bwd_dweight(mDlMn.m, mHidMn.m, s4, e4, ss->stream)
                         : launch_bwd_dweight(mHidMn.m, mDlMn.m, s4, e4, ss->stream))))
      return rc;
    if ((rc = join_side(*ss, st))) return rc;
  }
  return p->validate ? read_status(ws, st) : FLCE_OK;
}

int flce_forward_backward(const flce_params* p, const void* hidden, const void* weight,
                          const int64_t* labels, const float* g_loss, const float* g_entropy,
                          float* loss, float* entropy, float* lse, float* ez, void* dhidden,
                          void* dweight, void* workspace, size_t ws_bytes, void* stream) {
  using namespace flce;
  int rc = check_params(p);
  if (rc) return rc;
  // the dlogits of a shard need the whole vocabulary's logsumexp first
  if (p->v_total > 0 && !(p->v_offset == 0 && p->v_total == p->V)) return FLCE_ERR_BAD_ARG;
  if (!loss || !entropy || !workspace || !weight || !dweight) return FLCE_ERR_BAD_ARG;
  if (p->N > 0 && (!hidden || !labels || !lse || !ez || !dhidden)) return FLCE_ERR_BAD_ARG;
  if (!aligned16(hidden) || !aligned16(weight) || !aligned16(labels) || !aligned16(loss) ||
      !aligned16(entropy) || !aligned16(lse) || !aligned16(ez) || !dhidden_aligned(p, dhidden) ||
      !aligned16(dweight) || (reinterpret_cast<uintptr_t>(g_loss) & 3) ||
      (reinterpret_cast<uintptr_t>(g_entropy) & 3) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255))
    return FLCE_ERR_ALIGN;
  const FusedLayout L = fused_layout(p);
  cudaStream_t st;
  uint32_t* err;
  if ((rc = begin_call(workspace, ws_bytes, L.total, stream, &st, &err))) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int64_t N = p->N, H = p->H, V = p->V;
  if (N == 0) {
    if ((rc = zero_reduced(p, loss, entropy, st))) return rc;
    if ((rc = cuda_rc(cudaMemsetAsync(dweight, 0, static_cast<size_t>(H * V) * 2, st))))
      return rc;
    return p->validate ? read_status(ws, st) : FLCE_OK;
  }
  const bool vh = p->weight_layout == FLCE_WEIGHT_VH;
  const bool per_token = p->reduction == FLCE_RED_NONE;
  const bool smooth = p->label_smoothing != 0.0f;
  SideStream* ss = nullptr;
  if ((rc = side_stream(&ss))) return rc;
  Smoothing sm{p->label_smoothing, p->class_weight, reinterpret_cast<float*>(ws + L.psw),
               nullptr};
  if (smooth && p->class_weight) {
    float* wsum = reinterpret_cast<float*>(ws + kWsumOffset);
    class_weight_sum_kernel<<<1, 1024, 0, st>>>(p->class_weight, V, wsum);
    if ((rc = cuda_rc(cudaGetLastError()))) return rc;
    sm.wsum = wsum;
  }
  StatsOut so{};
  so.pm = reinterpret_cast<float*>(ws + L.pm);
  so.pd = reinterpret_cast<float*>(ws + L.pd);
  so.ps = reinterpret_cast<float*>(ws + L.ps);
  so.psw = reinterpret_cast<float*>(ws + L.psw);
  so.zlabel = reinterpret_cast<float*>(ws + L.zlabel);
  so.zout = reinterpret_cast<float*>(ws + L.z);
  so.part_stride = L.Nc;
  so.ld_z = L.ldz;
  so.n_parts = L.n_parts;
  float* loss_row = per_token ? loss : reinterpret_cast<float*>(ws + L.loss_row);
  float* ent_row = per_token ? entropy : reinterpret_cast<float*>(ws + L.ent_row);
  float4* rowc = reinterpret_cast<float4*>(ws + L.rowc);
  float* rowd = reinterpret_cast<float*>(ws + L.rowd);
  __nv_bfloat16* dl = reinterpret_cast<__nv_bfloat16*>(ws + L.dl);
  float* dwacc = reinterpret_cast<float*>(ws + L.dwacc);

  // hidden as dweight's operand (MN-major, tokens along K); weight as dhidden's B
  Map mHidMn, mWDh;
  bool ok = make_map(&mHidMn, hidden, H, N, H, 64, BK);
  ok = ok && (vh ? make_map(&mWDh, weight, H, V, H, 64, BK)
                 : make_map(&mWDh, weight, V, H, V, BK, 64));
  if (!ok) return FLCE_ERR_CUDA;

  for (int64_t c = 0; c < L.chunks; ++c) {
    const int64_t n0 = c * L.Nc;
    const int64_t rows = (N - n0) < L.Nc ? (N - n0) : L.Nc;
    const int64_t* lab = labels + n0;

    // logits of the chunk: online-softmax partials and the raw fp32 values
    if ((rc = launch_stats(p, hidden, weight, lab, n0, rows, so, err, st))) return rc;
    const Parts pt{so.pm, so.pd, so.ps, nullptr, L.n_parts, L.Nc};
    fwd_combine_kernel<<<static_cast<unsigned>(cdiv(rows, 32)), 256, 0, st>>>(
        pt, rows, so.zlabel, lab, V, p->ignore_index, p->zloss_coef, sm, lse + n0, ez + n0,
        loss_row + n0, ent_row + n0, err);
    if ((rc = cuda_rc(cudaGetLastError()))) return rc;
    bwd_prep_kernel<<<1, 1024, 0, st>>>(
        lab, labels, N, lse + n0, ez + n0, g_loss && per_token ? g_loss + n0 : g_loss,
        g_entropy && per_token ? g_entropy + n0 : g_entropy, rows, V, p->ignore_index,
        per_token, p->reduction == FLCE_RED_MEAN, p->zloss_coef, p->label_smoothing,
        p->class_weight, rowc, rowd);
    if ((rc = cuda_rc(cudaGetLastError()))) return rc;
    if ((rc = cuda_rc(launch_dlogits_from_z(so.zout, rows, L.ldz, rowc, rowd, lab, V,
                                            p->softcap, smooth, p->class_weight, dl, st))))
      return rc;

    // the chunk's dlogits [rows, V]: rows past `rows` read as zeros
    Map mDlK, mDlMn;
    ok = make_map(&mDlK, dl, V, rows, L.ldz, BK, 64) &&
         make_map(&mDlMn, dl, V, rows, L.ldz, 64, BK);
    if (!ok) return FLCE_ERR_CUDA;

    // dhidden[n0 : n0 + rows] = dlogits @ weight^T, all of V in one contraction;
    // the k-steps of every tile advance together, so a square-ish group of tiles
    // keeps the k-slices in flight small in L2
    GemmShape s5 = base_shape(L2_NORMAL, L2_NORMAL);
    s5.m_tiles = static_cast<int>(cdiv(rows, PAIR_BM));
    s5.n_tiles = static_cast<int>(cdiv(H, TN_DHIDDEN));
    s5.k_blocks = static_cast<int>(cdiv(V, BK));
    s5.raster = 0;
    s5.sched = sched_counters(err);
    plan_tiles(&s5, int64_t(PAIR_BM) * V * 2);
    EpiArgs e5{};
    e5.rows = static_cast<int>(rows);
    e5.cols = static_cast<int>(H);
    e5.V = V;
    e5.ld_acc = H;
    if (p->dhidden_fp32) {
      e5.acc = static_cast<float*>(dhidden) + n0 * H;  // 32-byte aligned: H % 8 == 0
      e5.acc_mode = ACC_FIRST;
    } else {
      e5.acc_out = static_cast<__nv_bfloat16*>(dhidden) + n0 * H;
      e5.acc_mode = ACC_ONLY;
    }
    e5.err = err;
    set_extents(&s5, mDlK, mWDh);
    // dhidden on the caller's stream, dweight beside it on the side stream (SideStream)
    if ((rc = fork_side(*ss, st))) return rc;
    if ((rc = cuda_rc((vh ? launch_bwd_dhidden_vh : launch_bwd_dhidden)(mDlK.m, mWDh.m, s5, e5,
                                                                        st))))
      return rc;

    // dweight (+)= hidden[n0 : n0 + rows]^T @ dlogits ([H,V]) or its transpose ([V,H])
    GemmShape s4 = vh ? base_shape(L2_NORMAL, L2_EVICT_LAST) : base_shape(L2_EVICT_LAST, L2_NORMAL);
    s4.k_blocks = static_cast<int>(cdiv(rows, BK));
    s4.sched = sched_counters(err, 1);
    EpiArgs e4{};
    e4.V = V;
    e4.err = err;
    e4.col_base = 0;
    if (vh) {
      s4.m_tiles = static_cast<int>(cdiv(V, PAIR_BM));
      s4.n_tiles = static_cast<int>(cdiv(H, TN_DWEIGHT));
      s4.b_k_off = static_cast<int>(n0);
      s4.raster = 1;
      plan_tiles(&s4, int64_t(TN_DWEIGHT) * rows * 2);
      e4.rows = static_cast<int>(V);
      e4.cols = static_cast<int>(H);
    } else {
      s4.m_tiles = static_cast<int>(cdiv(H, PAIR_BM));
      s4.n_tiles = static_cast<int>(cdiv(V, TN_DWEIGHT));
      s4.a_k_off = static_cast<int>(n0);
      s4.raster = 0;
      plan_tiles(&s4, int64_t(PAIR_BM) * rows * 2);
      e4.rows = static_cast<int>(H);
      e4.cols = static_cast<int>(V);
    }
    const int64_t ld_dw = vh ? H : V;
    const Map& a4 = vh ? mDlMn : mHidMn;
    const Map& b4 = vh ? mHidMn : mDlMn;
    set_extents(&s4, a4, b4);
    if (L.chunks == 1) {
      e4.out = static_cast<__nv_bfloat16*>(dweight);
      e4.ld_out = ld_dw;
      rc = cuda_rc(launch_bwd_dweight(a4.m, b4.m, s4, e4, ss->stream));
    } else {
      e4.acc = dwacc;
      e4.acc_out = static_cast<__nv_bfloat16*>(dweight);
      e4.ld_acc = ld_dw;
      e4.acc_mode = c == 0 ? ACC_FIRST : c == L.chunks - 1 ? ACC_LAST : ACC_MID;
      rc = cuda_rc(launch_bwd_dweight_acc(a4.m, b4.m, s4, e4, ss->stream));
    }
    if (rc) return rc;
    if ((rc = join_side(*ss, st))) return rc;
  }
  if (!per_token) {
    reduce_rows_kernel<<<1, 1024, 0, st>>>(loss_row, ent_row, labels, N, p->ignore_index,
                                           p->reduction == FLCE_RED_MEAN, p->class_weight, lse,
                                           p->zloss_coef, loss, entropy);
    if ((rc = cuda_rc(cudaGetLastError()))) return rc;
  }
  return p->validate ? read_status(ws, st) : FLCE_OK;
}

int flce_scale_bf16(void* x, int64_t n, const float* g, void* stream) {
  using namespace flce;
  if (n < 0 || !g || (n > 0 && !x)) return FLCE_ERR_BAD_ARG;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(g) & 3)) return FLCE_ERR_ALIGN;
  if (n == 0) return FLCE_OK;
  DevInfo di;
  int rc = device_info(&di);
  if (rc) return rc;
  const int64_t blocks = cdiv(cdiv(n, 8), 256);
  const int64_t cap = int64_t(di.sms) * 8;
  scale_bf16_kernel<<<static_cast<unsigned>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap), 256,
                      0, static_cast<cudaStream_t>(stream)>>>(static_cast<__nv_bfloat16*>(x), n,
                                                              g);
  return cuda_rc(cudaGetLastError());
}

int flce_selftest_wait_timeout(void* workspace, size_t ws_bytes, uint64_t limit_ns,
                                void* stream) {
  using namespace flce;
  if (!workspace) return FLCE_ERR_BAD_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return FLCE_ERR_ALIGN;
  if (limit_ns == 0 || limit_ns > FLCE_WAIT_LIMIT_NS) return FLCE_ERR_BAD_ARG;
  cudaStream_t st;
  uint32_t* err;
  int rc = begin_call(workspace, ws_bytes, kHeaderBytes, stream, &st, &err);
  if (rc) return rc;
  wait_timeout_selftest_kernel<<<1, 32, 0, st>>>(err, limit_ns);
  return cuda_rc(cudaGetLastError());
}

}  // extern "C"
