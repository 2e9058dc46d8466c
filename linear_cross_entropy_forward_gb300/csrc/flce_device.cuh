// Device-side primitives for sm_103a: mbarriers, TMA tile loads, tcgen05 (TMEM
// allocation, UMMA issue/commit, TMEM loads) and the shared-memory / instruction
// descriptors the UMMA consumes.  All of it is hand-written inline PTX.
//
// Every wait on an mbarrier is bounded: after FLCE_WAIT_LIMIT_NS of global time
// the wait gives up, records FLCE_DEVERR_TIMEOUT in the device error word and
// returns false, so a broken pipeline ends the kernel instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#ifndef FLCE_WAIT_LIMIT_NS
#define FLCE_WAIT_LIMIT_NS 2000000000ull  // 2 s
#endif

// Upper bound (ns) on how long one mbarrier.try_wait may keep its thread suspended
// before it re-checks.  Without it the suspended thread resumed well after the
// phase completed: the producer / UMMA handshake then starved the tensor pipe
// (~73 % busy on the forward GEMM instead of ~85 %).  Any value of 10-100 ns gives
// the same cycles; a tight test_wait spin is slower (it takes issue slots).
#ifndef FLCE_WAIT_HINT_NS
#define FLCE_WAIT_HINT_NS 20
#endif

namespace flce {

// Device error word bits (OR-ed into the workspace header).
enum : uint32_t {
  FLCE_DEVERR_TIMEOUT = 1u,
  FLCE_DEVERR_LABEL = 2u,
  FLCE_DEVERR_BOUNDS = 4u,  // an in-kernel bounds check of the FLCE_DEBUG build failed
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "n"(FLCE_WAIT_HINT_NS)
      : "memory");
  return ok != 0;
}

// Cluster-scope acquire: for barriers that other CTAs of the cluster arrive on.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "n"(FLCE_WAIT_HINT_NS)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// (and flags a timeout) if it does not complete within the limit, or if another
// role of the CTA has already aborted (*abort != 0).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint32_t* err, uint64_t limit_ns = FLCE_WAIT_LIMIT_NS) {
  auto try_once = [&]() {
    return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (try_once()) return true;
  uint64_t t0 = global_timer_ns();
  uint32_t spins = 0;
  while (true) {
    if (try_once()) return true;
    if (((++spins) & 63u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort = 1;
        if (err) atomicOr(err, FLCE_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- clusters (CTA pairs)
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// shared::cluster address of the same shared variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t cta_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(cta_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Arrive without release semantics on a barrier of any CTA of the cluster: it orders
// none of this thread's earlier memory operations.  A release arrive on the thread
// that issues the UMMAs waited for its tensor operations in flight and drained the
// pipe (measured), so that thread acknowledges with this one, after an acquire load.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// 32-bit shared-memory load with acquire semantics: no later memory operation of this
// thread (a relaxed arrive that hands the slot back, say) is performed before it.
__device__ __forceinline__ int ld_acquire_shared(const volatile int* p) {
  int v;
  asm volatile("ld.acquire.cluster.shared::cta.b32 %0, [%1];"
               : "=r"(v)
               : "r"(smem_u32(const_cast<const int*>(p)))
               : "memory");
  return v;
}
// Arrive on a barrier of this CTA (release at CTA scope).
__device__ __forceinline__ void mbar_arrive_local(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// 32-bit store to a shared::cluster address (another CTA's shared memory).
__device__ __forceinline__ void st_shared_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// Tile load into this CTA's shared memory whose completion is signalled on an
// mbarrier that may live in the peer CTA of the pair (shared::cluster address),
// with an L2 eviction-priority policy (createpolicy) for the loaded lines.
__device__ __forceinline__ void tma_load_2d_pair_hint(void* dst, const CUtensorMap* map,
                                                      uint32_t mbar_cluster_addr, int32_t x,
                                                      int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(mbar_cluster_addr), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// L2 policies: lines loaded with evict_last outlive evict_normal / evict_first lines.
enum L2Hint : int { L2_NORMAL = 0, L2_EVICT_FIRST = 1, L2_EVICT_LAST = 2 };

__device__ __forceinline__ uint64_t l2_policy(int hint) {
  uint64_t p = 0;
  if (hint == L2_EVICT_FIRST) {
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  } else if (hint == L2_EVICT_LAST) {
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  } else {
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  }
  return p;
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Pair versions: issued by one warp of each CTA of the pair, together.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// CTA-pair UMMA (M = 256 across the pair): each CTA supplies its 128 rows of A and
// its half of B's N columns at the same shared-memory offsets; issued by the
// leader CTA only, and each CTA's TMEM receives its own 128 rows of D.  The four
// K=16 slices of one 64-deep k-block go out back to back from one asm statement;
// the first accumulates into D only if `accumulate` is set.
__device__ __forceinline__ void umma_bf16_pair_x4(uint32_t d_tmem, const uint64_t (&ad)[4],
                                                  const uint64_t (&bd)[4], uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %10, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %9, p;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %3, %4, %9, 1;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %5, %6, %9, 1;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %7, %8, %9, 1;\n\t}" ::"r"(d_tmem),
      "l"(ad[0]), "l"(bd[0]), "l"(ad[1]), "l"(bd[1]), "l"(ad[2]), "l"(bd[2]), "l"(ad[3]),
      "l"(bd[3]), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at the same offset in every CTA of `mask` when the
// pair UMMAs issued so far by this thread have completed.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one row per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile
// (Blackwell format: start>>4 in [0,14), LBO>>4 in [16,30), SBO>>4 in [32,46),
// version 1 at bit 46, swizzle mode 2 = 128B at bits [61,64)).
__host__ __device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 D.
// a_mn / b_mn select an MN-major (transposed) operand in shared memory.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                                  // D format: f32
         | (1u << 7)                                // A format: bf16
         | (1u << 10)                               // B format: bf16
         | (static_cast<uint32_t>(a_mn) << 15)      // A major
         | (static_cast<uint32_t>(b_mn) << 16)      // B major
         | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// ---------------------------------------------------------------- math helpers
__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Soft-cap by one exponential and one reciprocal: tanh(a) = 1 - 2 / (1 + e^{2a}), so
// with k = 2 log2e / c and r = 1 / (1 + 2^{k x}),  tanh(x / c) = 1 - 2r  and
// c tanh(x / c) = c - 2c r.  2^{k x} overflowing to +inf gives r = 0 (z = c), and
// underflowing gives r = 1 (z = -c); near x = 0 the absolute error stays near one
// fp32 ulp of 1 times c.  The epilogues run this per logit; every instruction they
// save is issue time the UMMA issuer on the same SM gets back.
__device__ __forceinline__ float softcap_r(float x, float k) {
  return fast_rcp(1.0f + fast_ex2(__fmul_rn(x, k)));
}

// Two fp32 lanes in one 64-bit register pair, for the packed f32x2 arithmetic of
// sm_100-class SMs: one instruction per two lanes, each lane rounded exactly like the
// scalar instruction (rn), so packed and scalar code give the same bits.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Three-input maximum / minimum (sm_100-class SMs): one instruction for two steps
// of a reduction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Maximum / minimum of 32 values in 16 instructions, as a tree (5 levels deep).
__device__ __forceinline__ float max32(const float (&x)[32]) {
  float a[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) a[i] = fmax3(x[3 * i], x[3 * i + 1], x[3 * i + 2]);
  a[10] = fmaxf(x[30], x[31]);
  const float b0 = fmax3(a[0], a[1], a[2]), b1 = fmax3(a[3], a[4], a[5]);
  const float b2 = fmax3(a[6], a[7], a[8]), b3 = fmaxf(a[9], a[10]);
  return fmaxf(fmax3(b0, b1, b2), b3);
}
__device__ __forceinline__ float min32(const float (&x)[32]) {
  float a[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) a[i] = fmin3(x[3 * i], x[3 * i + 1], x[3 * i + 2]);
  a[10] = fminf(x[30], x[31]);
  const float b0 = fmin3(a[0], a[1], a[2]), b1 = fmin3(a[3], a[4], a[5]);
  const float b2 = fmin3(a[6], a[7], a[8]), b3 = fminf(a[9], a[10]);
  return fminf(fmin3(b0, b1, b2), b3);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 256-bit global accesses (one full 32-byte sector per thread; sm_100 and later).
// The address must be 32-byte aligned: callers use them only on workspace arrays
// whose base is 256-byte aligned and whose row pitch and offsets are multiples of
// 32 bytes.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               :: "l"(p), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
                  "r"(v[6]), "r"(v[7])
               : "memory");
}

// Evict-first variant, for data that the next kernel streams once.
__device__ __forceinline__ void st_global_cs_v8f(float* p, const float* v) {
  asm volatile("st.global.cs.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               :: "l"(p), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]),
                  "f"(v[6]), "f"(v[7])
               : "memory");
}

__device__ __forceinline__ void st_global_v8f(float* p, const float* v) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               :: "l"(p), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]),
                  "f"(v[6]), "f"(v[7])
               : "memory");
}

__device__ __forceinline__ void ld_global_v8f(const float* p, float* v) {
  asm volatile("ld.global.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
                 "=f"(v[6]), "=f"(v[7])
               : "l"(p)
               : "memory");
}

}  // namespace flce
