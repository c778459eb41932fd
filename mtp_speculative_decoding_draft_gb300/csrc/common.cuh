// Device helpers shared by the mtpspec kernels: TMA bulk copies driven by
// mbarriers, bounded waits, programmatic dependent launch, thread-block-cluster
// barriers and distributed shared memory, warp reductions.  Inline PTX for
// sm_103a.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace mtp {

// Status bits (mirror MTP_STATUS_* of the public header).
constexpr int kStatusTimeout = 1;
constexpr int kStatusBadToken = 2;
constexpr int kStatusBadCtx = 4;
constexpr int kStatusNonFinite = 8;
constexpr int kStatusBounds = 16;  // bounds-checked build: an index outside its buffer, access skipped

// A wait that has not finished after this long gives up and flags the status.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void set_status(int *status, int bits) {
  if (status) atomicOr(status, bits);
}

// Bounds-checked build (compiled with -DMTP_BOUNDS): an index outside its
// buffer sets kStatusBounds in the status word and the access is skipped --
// no trap, the context stays usable.  The default build checks nothing.
#ifdef MTP_BOUNDS
__device__ __forceinline__ bool in_bounds(bool ok, int *status) {
  if (!ok) set_status(status, kStatusBounds);
  return ok;
}
#else
__device__ __forceinline__ constexpr bool in_bounds(bool, int *) { return true; }
#endif

// Global-memory flags between CTAs of one grid (GPU scope).
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(unsigned *p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Atomic add with acquire and release semantics at GPU scope: the caller's
// earlier writes are visible to whoever observes the new value, and what the
// earlier adders wrote is visible to the caller afterwards.
__device__ __forceinline__ unsigned atomic_add_acq_rel(unsigned *p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy and the cluster.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// kWaitLimitNs, flags MTP_STATUS_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *status) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u && global_timer_ns() - t0 > kWaitLimitNs) {
      set_status(status, kStatusTimeout);
      return false;
    }
  }
}

// The same bounded wait, parking the warp between tries (suspend-time hint):
// the hardware wakes it when the phase completes, and a warp that waits for
// data does not take issue slots from the warps computing.
__device__ __forceinline__ bool mbar_sleep_wait(uint64_t *bar, uint32_t parity, int *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
        : "memory");
    if (done) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      set_status(status, kStatusTimeout);
      return false;
    }
  }
}

// Cross-CTA flavour: acquire at cluster scope, so stores other CTAs of the
// cluster made before their (release) arrivals are visible afterwards.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, int *status) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 255u) == 255u && global_timer_ns() - t0 > kWaitLimitNs) {
      set_status(status, kStatusTimeout);
      return false;
    }
  }
}

// Arrive (release, cluster scope) on the mbarrier at the same shared-memory
// location in CTA `rank` of this cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint64_t *local_bar, uint32_t rank) {
  uint32_t raddr;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(smem_u32(local_bar)), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(raddr) : "memory");
}

// ---------------------------------------------------------------- TMA bulk copy

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 eviction-priority hint (for data streamed exactly once).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal_all() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Read-only global loads that skip L1 and carry an L2 eviction-priority policy.
__device__ __forceinline__ float4 ld_stream_f4(const float4 *p, uint64_t pol) {
  float4 v;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
      : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
      : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ float ld_stream_f32(const float *p, uint64_t pol) {
  float v;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// ---------------------------------------------------------------- launch trace
//
// Built with -DMTP_TRACE: thread 0 of every CTA folds the global timer into
// its launch's record (slot = grid id mod kTraceSlots) at the kernel's start,
// after its wait for the previous kernel and at its end.  Each source file
// has its own record array (internal linkage) and its own collector,
// trace_collect_<file>(), defined by MTP_TRACE_COLLECTOR at the file's end.
// Start and dependency times are stored complemented so that one atomicMax
// keeps the earliest.  Without MTP_TRACE the marks compile to nothing.
// (TraceRec, kTraceSlots and the record kinds are in internal.h)

#ifdef MTP_TRACE
static __device__ TraceRec g_trace[kTraceSlots];

__device__ __forceinline__ TraceRec &trace_rec(int kind) {
  unsigned long long g;
  asm volatile("mov.u64 %0, %%gridid;" : "=l"(g));
  TraceRec &r = g_trace[g % kTraceSlots];
  r.grid = g;
  r.kind = kind;
  return r;
}
__device__ __forceinline__ void trace_start(int kind) {
  if (threadIdx.x == 0) atomicMax(&trace_rec(kind).nstart, ~global_timer_ns());
}
__device__ __forceinline__ void trace_dep(int kind) {
  if (threadIdx.x == 0) atomicMax(&trace_rec(kind).ndep, ~global_timer_ns());
}
__device__ __forceinline__ void trace_end(int kind) {
  if (threadIdx.x == 0) atomicMax(&trace_rec(kind).end, global_timer_ns());
}
__device__ __forceinline__ void trace_mark(int kind, int i) {
  if (threadIdx.x == 0) atomicMax(&trace_rec(kind).mark[i & 3], global_timer_ns());
}
#define MTP_TRACE_COLLECTOR(name)                                                                   \
  int trace_collect_##name(TraceRec *out, int max) {                                               \
    static TraceRec host[kTraceSlots];                                                             \
    if (cudaMemcpyFromSymbol(host, g_trace, sizeof(host)) != cudaSuccess) return -1;               \
    void *dev = nullptr;                                                                           \
    if (cudaGetSymbolAddress(&dev, g_trace) != cudaSuccess) return -1;                             \
    if (cudaMemset(dev, 0, sizeof(host)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) \
      return -1;                                                                                   \
    int n = 0;                                                                                     \
    for (int i = 0; i < kTraceSlots && n < max; ++i)                                               \
      if (host[i].grid != 0ull) out[n++] = host[i];                                                \
    return n;                                                                                      \
  }
#else
__device__ __forceinline__ void trace_start(int) {}
__device__ __forceinline__ void trace_dep(int) {}
__device__ __forceinline__ void trace_end(int) {}
__device__ __forceinline__ void trace_mark(int, int) {}
#define MTP_TRACE_COLLECTOR(name) \
  int trace_collect_##name(TraceRec *, int) { return 0; }
#endif

// ---------------------------------------------------------------- PDL

// Wait until the grids this one depends on have completed and flushed memory.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next kernel in the stream to start launching.
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
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

// Full cluster barrier with release/acquire semantics for shared memory.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void *local, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(local)), "r"(rank));
  return out;
}

// Generic pointer to the same shared variable in CTA `rank` of this cluster.
// Loads through it are ordinary memory operations: the compiler may batch
// independent ones, and the cluster barrier's memory clobber orders them.
template <class T>
__device__ __forceinline__ const T *dsmem_ptr(const T *local, uint32_t rank) {
  uint64_t out;
  asm("mapa.u64 %0, %1, %2;" : "=l"(out) : "l"(reinterpret_cast<uint64_t>(local)), "r"(rank));
  return reinterpret_cast<const T *>(out);
}

template <class T>
__device__ __forceinline__ T *dsmem_ptr_mut(T *local, uint32_t rank) {
  uint64_t out;
  asm("mapa.u64 %0, %1, %2;" : "=l"(out) : "l"(reinterpret_cast<uint64_t>(local)), "r"(rank));
  return reinterpret_cast<T *>(out);
}

// Named barrier over the first `nthreads` threads of the CTA (warp-aligned).
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ double dsmem_ld_f64(uint32_t addr) {
  double v;
  asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ int dsmem_ld_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// ---------------------------------------------------------------- numerics

constexpr float kLog2e = 1.4426950408889634f;

// 2^x, hardware approximation (relative error about 2^-22; -inf gives +0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf16_to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// 8 bf16 (one 16-byte vector) dotted with 8 floats, accumulated into acc.
__device__ __forceinline__ float dot8(uint4 w, const float *a, float acc) {
  acc = fmaf(bf16_lo(w.x), a[0], acc);
  acc = fmaf(bf16_hi(w.x), a[1], acc);
  acc = fmaf(bf16_lo(w.y), a[2], acc);
  acc = fmaf(bf16_hi(w.y), a[3], acc);
  acc = fmaf(bf16_lo(w.z), a[4], acc);
  acc = fmaf(bf16_hi(w.z), a[5], acc);
  acc = fmaf(bf16_lo(w.w), a[6], acc);
  acc = fmaf(bf16_hi(w.w), a[7], acc);
  return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// (value, index) maximum with the lowest index winning ties.
__device__ __forceinline__ void argmax_merge(float &v, int &i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__device__ __forceinline__ void warp_argmax(float &v, int &i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    argmax_merge(v, i, v2, i2);
  }
}

// Online softmax state over scaled logits: m = running max of x (raw logits),
// s = sum exp2((x - m) * c).  Merging two states keeps the larger max.
__device__ __forceinline__ void lse_merge(float &m, float &s, float m2, float s2, float c) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  if (m2 > m) {
    s = s * exp2f((m - m2) * c) + s2;
    m = m2;
  } else {
    s = s + s2 * exp2f((m2 - m) * c);
  }
}

__device__ __forceinline__ void warp_lse(float &m, float &s, float c) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_merge(m, s, m2, s2, c);
  }
}

}  // namespace mtp
