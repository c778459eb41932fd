// Verification of k drafted tokens per sequence ("The Tiny Draft Model Hidden
// Inside Qwen", section "How the draft becomes real output"; "Speculative
// Decoding and MTP: Why Guessing Is Free", sections "Speculative decoding:
// draft, then verify" and "It's exact, not approximate").
//
// Work items, one per position of one sequence, in position-major order:
//  greedy      row t_j, j = 0..k            -> its (max, lowest argmax);
//  stochastic  the pair (t_j, q_j), j < k, then the bonus row t_k.
//              A pair yields the ratio test at j and, when the test rejects,
//              the inverse-CDF draw from max(0, p_j - q_j); the bonus row
//              yields the draw from p_k.
// Every item is taken by one thread-block cluster of C CTAs; CTA r owns the
// r-th of C contiguous runs of 512-element sub-chunks of every row.  The
// items are independent: position j does not wait for the outcome of the
// positions before it.  A rejecting pair makes its draw unless an earlier
// position is already known to reject (a per-sequence word that rejecting
// items raise); the item of the position claimed last gathers the
// positions' records, picks the first rejection and writes the outputs.
//
// Inside a CTA: a producer warp streams the CTA's sub-chunks through a ring
// of 8 KB shared-memory stages with 1-D bulk copies (up to eight stages at a
// time, one per lane; a row piece is 4 sub-chunks of one row in one copy);
// five worker warps take the stages round-robin and reduce them (per
// sub-chunk max and sum of exp2, or argmax) and, for a rejecting pair,
// re-read the pair -- a few microseconds after the first read, partly from
// L2 -- for the per-sub-chunk sampling weights; three decider warps, item n
// going to decider n mod 3, combine the sub-chunks, exchange the CTA partials
// with the other CTAs of the cluster through distributed shared memory (a
// remote store and a remote mbarrier arrive per peer), take the decision and,
// for a draw, locate the crossing CTA, sub-chunk and element (the last 512
// elements rescanned in float64).  A claimer warp of the cluster's first CTA
// takes items from one global counter, a few ahead of its producer, and hands
// them to every CTA of the cluster.
//
// No result depends on which cluster ran which item.  Every wait is bounded
// and gives up (flagging the status word) once any thread has timed out.
// Each call leaves the state in the workspace zero for the next one.
#include <stdlib.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace mtp {

namespace {

constexpr int kSub = 512;        // sub-chunk: elements of one stage part
#ifndef MTP_VERIFY_WORKERS
#define MTP_VERIFY_WORKERS 5
#endif
constexpr int kWorkers = MTP_VERIFY_WORKERS;  // streaming warps
#ifndef MTP_VERIFY_DECIDERS
#define MTP_VERIFY_DECIDERS 3
#endif
constexpr int kDeciders = MTP_VERIFY_DECIDERS;  // decision warps
constexpr int kProducerWarp = kWorkers;
constexpr int kClaimerWarp = kWorkers + 1;
constexpr int kFirstDecider = kWorkers + 2;
constexpr int kVerifyThreads = 32 * (kWorkers + 2 + kDeciders);
#ifndef MTP_VERIFY_QD
#define MTP_VERIFY_QD 9
#endif
constexpr int kQD = MTP_VERIFY_QD;  // item slots per CTA
static_assert(kQD % kDeciders == 0, "a slot always goes to the same decider");
#ifndef MTP_VERIFY_STAGES
#define MTP_VERIFY_STAGES 11
#endif
constexpr int kStages = MTP_VERIFY_STAGES;  // ring stages
constexpr int kStageF = 4 * kSub;           // floats per stage (8 KB)
constexpr int kRowSubs = 4;                 // sub-chunks of one row per stage
constexpr int kPairSubs = 2;                // sub-chunks of each of two rows per stage
#ifndef MTP_VERIFY_MAXP
#define MTP_VERIFY_MAXP 64
#endif
constexpr int kMaxP = MTP_VERIFY_MAXP;  // sub-chunks per CTA slice, at most
constexpr int kMaxC = 16;        // CTAs per cluster, at most
constexpr unsigned kFull = 0xffffffffu;

enum : int { kItemStop = 0, kItemGreedy = 1, kItemPair = 2, kItemBonus = 3 };
enum : int { kPieceStop = 0, kPieceRow = 1, kPieceRowDraft = 2, kPieceWeights = 3 };
// bits of a position's record word
constexpr int kRecAccept = 1, kRecBadToken = 2, kRecNonFinite = 4, kRecWritten = 8;

struct ItemInfo {
  int kind, b, j, kb;  // kb: drafts sequence b keeps (k unless the draft length is dynamic)
};

// A CTA's partial of one item, sent to every CTA of the cluster (32 bytes).
struct Xchg {
  double z0, z1;  // partition sums of rows 0 / 1, or residual / target weight sums
  float m0, m1;   // row maxima
  int i0, i1;     // argmax, rejection hint, or last sub-chunk with positive weight
};

// What one ring stage holds: local sub-chunks p .. p+np-1 (up to 4) of the
// item's target or draft row (a row piece), or of both rows (a weight piece,
// up to 2 of each, the draft span in the stage's second half).  Each
// span's 16-byte aligned body arrives by one bulk copy; an unaligned head or
// tail is read from global memory by the worker.
struct Tag {
  int slot, kind, p, np;  // item slot, piece kind, first local sub-chunk, sub-chunks
  unsigned seq;           // piece number + 1: which use of the stage this is
  int pad[3];
};

struct SlotState {
  ItemInfo info;           // written by the cluster's first CTA
  float Mt, Ml, iZt, iZl;  // normalisers of the sampling weights
  // per sub-chunk: (max, sum | argmax) of rows 0 and 1; once a pair's
  // statistics are combined, .xy takes its residual and target weight sums
  float4 stats[kMaxP];
  Xchg x1[kMaxC], x2[kMaxC];
};

struct Shared {
  uint64_t full[kStages], empty[kStages];
  uint64_t item_full[kQD], item_empty[kQD], adone[kQD], bdone[kQD], x1bar[kQD], x2bar[kQD];
  Tag tag[kStages];
  SlotState slot[kQD];
  int bq[kQD];             // weight passes requested by the deciders, in order
  unsigned bq_seq[kQD];
  unsigned bq_tail;
  unsigned prod_item;      // items the producer has started
  unsigned dec_done;       // deciders finished
};

constexpr size_t kHdr = (sizeof(Shared) + 127) / 128 * 128;
constexpr size_t kSmemBytes = kHdr + (size_t)kStages * kStageF * 4;
static_assert(kSmemBytes <= 112 * 1024, "two CTAs per SM");

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ unsigned ld_vol(const unsigned *p) { return *reinterpret_cast<const volatile unsigned *>(p); }
__device__ __forceinline__ int ld_vol_i(const int *p) { return *reinterpret_cast<const volatile int *>(p); }

__device__ __forceinline__ ItemInfo read_info(const ItemInfo *p) {
  const volatile int *q = reinterpret_cast<const volatile int *>(p);
  return ItemInfo{q[0], q[1], q[2], q[3]};
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// One try on a phase of a barrier whose arrivals come from this CTA: parks
// the warp up to `ns` nanoseconds (the completing arrival wakes it).
__device__ __forceinline__ bool try_phase_local(uint64_t *bar, uint32_t parity, uint32_t ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return done != 0;
}

// Non-blocking test of a phase of a barrier that other CTAs of the cluster
// arrive on (acquire at cluster scope).
__device__ __forceinline__ bool test_phase_cluster(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait for a phase.  Gives up after kWaitLimitNs (flagging a
// timeout), or as soon as another thread of the launch has flagged one.
template <bool kCluster>
__device__ bool wait_phase(uint64_t *bar, uint32_t parity, int *status) {
  if (kCluster ? test_phase_cluster(bar, parity) : try_phase_local(bar, parity, 0u)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (kCluster) {
      if (test_phase_cluster(bar, parity)) return true;
      __nanosleep(32);
    } else if (try_phase_local(bar, parity, 20000u)) {
      return true;
    }
    if ((it & (kCluster ? 63u : 15u)) == 0u) {
      if (ld_vol_i(status) & kStatusTimeout) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        set_status(status, kStatusTimeout);
        return false;
      }
    }
  }
}


// Sampling weight of one element: residual max(0, p - q) (kind 0), target p
// (kind 1), unnormalised target weight exp2((t - Mt) c) (kind 2).
__device__ __forceinline__ float weight(int kind, float t, float l, float Mt, float Ml, float iZt, float iZl,
                                        float c) {
  const float e = ex2_approx((t - Mt) * c);
  if (kind == 2) return e;
  // both products rounded on their own (no fused multiply-add): where p and q
  // are equal the residual must be exactly zero, so that the draw falls back to p
  const float p = __fmul_rn(e, iZt);
  if (kind == 1) return p;
  return fmaxf(0.f, p - __fmul_rn(ex2_approx((l - Ml) * c), iZl));
}

__device__ __forceinline__ double warp_incl_scan_d(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// Elements [e0, e0+n) of a row, the body [h, h+L) 16-byte aligned.
__device__ __forceinline__ void part_geom(const float *row, int e0, int n, int &h, int &L) {
  const unsigned mis = (unsigned)(reinterpret_cast<uintptr_t>(row + e0) & 15u);
  int hh = (int)(((16u - mis) & 15u) >> 2);
  if (hh > n) hh = n;
  h = hh;
  L = (n - hh) & ~3;
}

// Span q of a stage: its row and elements [e0, e0+n), body [h, h+L).
struct Span {
  const float *row;
  int e0, n, h, L;
};

__device__ __forceinline__ Span stage_span(const VerifyArgs &a, const ItemInfo &it, int kind, int s0, int p, int np,
                                           int q) {
  Span sp{nullptr, 0, 0, 0, 0};
  const float *trow = a.target + ((size_t)it.b * (a.k + 1) + it.j) * a.V;
  if (kind == kPieceWeights)
    sp.row = q == 0 ? trow : a.draft + ((size_t)it.b * a.k + it.j) * a.V;
  else if (kind == kPieceRow && q == 0)
    sp.row = trow;
  else if (kind == kPieceRowDraft && q == 0)
    sp.row = a.draft + ((size_t)it.b * a.k + it.j) * a.V;
  if (sp.row) {
    sp.e0 = (s0 + p) * kSub;
    sp.n = min(np * kSub, a.V - sp.e0);
    part_geom(sp.row, sp.e0, sp.n, sp.h, sp.L);
  }
  return sp;
}

// This lane's 16 elements of sub-chunk i of a span held at buf -- element
// 512 i + 4*(lane + 32 m) + c at x[4 m + c] -- with `fill` past the span's end.
__device__ __forceinline__ void load_sub(const float *buf, const Span &sp, int i, float fill, float (&x)[16]) {
  const int lane = threadIdx.x & 31;
  const int base = i * kSub, n = sp.n - base, h = sp.h, L = sp.L;
  if (h == 0 && L == sp.n) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int f = lane + 32 * m;
      const float4 v =
          4 * f < n ? reinterpret_cast<const float4 *>(buf + base)[f] : make_float4(fill, fill, fill, fill);
      x[4 * m] = v.x;
      x[4 * m + 1] = v.y;
      x[4 * m + 2] = v.z;
      x[4 * m + 3] = v.w;
    }
  } else {
    const float *row = sp.row + sp.e0;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const int e = base + 4 * (lane + 32 * (m >> 2)) + (m & 3);
      x[m] = e >= sp.n ? fill : (e < h || e >= h + L) ? __ldcg(row + e) : buf[e - h];
    }
  }
}

__device__ __forceinline__ void mbar_arrive_n(uint64_t *bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}

// Warp maximum of a float in one instruction (-inf for an empty warp maximum).
__device__ __forceinline__ float redux_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Two warp sums with their shuffle rounds interleaved.
__device__ __forceinline__ void warp_sum2(float &a, float &b) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ta = __shfl_xor_sync(kFull, a, o), tb = __shfl_xor_sync(kFull, b, o);
    a += ta;
    b += tb;
  }
}

__device__ __forceinline__ float lane_max16(const float (&x)[16]) {
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = fmaxf(x[i], x[i + 8]);
#pragma unroll
  for (int i = 0; i < 4; ++i) m[i] = fmaxf(m[i], m[i + 4]);
  return fmaxf(fmaxf(m[0], m[2]), fmaxf(m[1], m[3]));
}

// sum exp2((x - M) c) over this lane's 16 elements (0 when M is -inf).
__device__ __forceinline__ float lane_sumexp16(const float (&x)[16], float M, float c) {
  if (M == -INFINITY) return 0.f;
  const float mc = M * c;
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    s0 += ex2_approx(fmaf(x[i], c, -mc));
    s1 += ex2_approx(fmaf(x[i + 1], c, -mc));
  }
  return s0 + s1;
}

// Four warp sums with their shuffle rounds interleaved.
__device__ __forceinline__ void warp_sum4(float (&v)[4]) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float t[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) t[q] = __shfl_xor_sync(kFull, v[q], o);
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] += t[q];
  }
}

// (max, lowest index) of a part over the warp; e0 is the part's first element.
__device__ __forceinline__ float2 part_argmax(const float (&x)[16], int e0) {
  const int lane = threadIdx.x & 31;
  const float M = redux_max(lane_max16(x));
  int cand = 0x7fffffff;
#pragma unroll
  for (int i = 15; i >= 0; --i)  // the last assignment is this lane's lowest index
    if (x[i] == M) cand = e0 + 4 * (lane + 32 * (i >> 2)) + (i & 3);
  return make_float2(M, __int_as_float(__reduce_min_sync(kFull, cand)));
}

// Target and draft rows of an item.
__device__ __forceinline__ const float *target_row(const VerifyArgs &a, int b, int j) {
  return a.target + ((size_t)b * (a.k + 1) + j) * a.V;
}
__device__ __forceinline__ const float *draft_row(const VerifyArgs &a, int b, int j) {
  return a.draft + ((size_t)b * a.k + j) * a.V;
}

// Item idx in position-major order: position j = idx / B of sequence idx % B;
// in stochastic mode positions 0..kb-1 are pairs and position kb the bonus
// row.  With a dynamic draft length (kb < k) the positions past kb carry no
// draft: their items take the plain one-row form (read, recorded, ignored by
// the gather), so every item still runs the same barrier protocol.
__device__ __forceinline__ ItemInfo decode(const VerifyArgs &a, unsigned idx) {
  ItemInfo it{kItemStop, 0, 0, 0};
  if (idx >= a.p.total) return it;
  const unsigned B = (unsigned)a.B;
  it.j = (int)(idx / B);
  it.b = (int)(idx % B);
  if (!in_bounds(it.j <= a.k && it.b < a.B, a.status)) return it;  // a stop item
  it.kb = a.k;
  if (a.k_eff) it.kb = min(max(__ldcg(&a.k_eff[it.b]), 0), a.k);
  if (a.mode == 0 || it.j > it.kb) it.kind = kItemGreedy;
  else it.kind = it.j < it.kb ? kItemPair : kItemBonus;
  return it;
}

// ---------------------------------------------------------------- producer

// The whole warp issues: a batch of up to kBatch consecutive stages, lane i
// filling stage g+i as soon as a worker has released it.
constexpr int kBatch = 8;

__device__ void producer(const VerifyArgs &a, Shared &sh, float *ring, int s0, int P) {
  const int lane = threadIdx.x & 31;
  const uint64_t pol_first = l2_policy_evict_first(), pol_norm = l2_policy_evict_normal();
  uint32_t g = 0, n = 0, bq_head = 0;
  bool ok = true, have = false, stopped = false, dep = false;
  ItemInfo it{};
  int pn = 0, half = 0;  // next sub-chunk of the current row; 1 on a pair's draft row
  uint64_t t_idle = 0;

  // m pieces of one kind: piece i covers local sub-chunks pbase + i * pstep
  // onwards, pstep of them (fewer at the slice's end)
  auto issue_batch = [&](int m, int kind, int slot, const ItemInfo &inf, int pbase, int pstep,
                         uint64_t pol) -> bool {
    bool lok = true;
    if (lane < m) {
      const uint32_t gi = g + (uint32_t)lane;
      const int st = (int)(gi % kStages);
      if (gi >= (uint32_t)kStages) lok = wait_phase<false>(&sh.empty[st], ((gi / kStages) - 1u) & 1u, a.status);
      if (lok) {
        const int p = pbase + lane * pstep;
        const int np = kind == kPieceStop ? 0 : min(pstep, P - p);
        Tag &tg = sh.tag[st];
        *reinterpret_cast<int4 *>(&tg) = make_int4(slot, kind, p, np);
        *reinterpret_cast<volatile unsigned *>(&tg.seq) = gi + 1u;
        const Span p0 = stage_span(a, inf, kind, s0, p, np, 0), p1 = stage_span(a, inf, kind, s0, p, np, 1);
        mbar_arrive_expect_tx(&sh.full[st], (uint32_t)(p0.L + p1.L) * 4u);
        float *dst = ring + (size_t)st * kStageF;
        if (p0.L > 0) bulk_g2s_hint(dst, p0.row + p0.e0 + p0.h, (uint32_t)p0.L * 4u, &sh.full[st], pol);
        if (p1.L > 0)
          bulk_g2s_hint(dst + kPairSubs * kSub, p1.row + p1.e0 + p1.h, (uint32_t)p1.L * 4u, &sh.full[st], pol);
      }
    }
    g += (uint32_t)m;
    return __all_sync(kFull, lok);
  };

  while (ok) {
    // weight passes of rejecting pairs go first: their rows are still in L2
    unsigned seq = lane == 0 ? ld_vol(&sh.bq_seq[bq_head % kQD]) : 0u;
    seq = __shfl_sync(kFull, seq, 0);
    if (seq == bq_head + 1u) {
      __threadfence_block();
      int slot = lane == 0 ? ld_vol_i(&sh.bq[bq_head % kQD]) : 0;
      slot = __shfl_sync(kFull, slot, 0);
      const ItemInfo bt = read_info(&sh.slot[slot].info);
      const int pieces = (P + kPairSubs - 1) / kPairSubs;
      for (int q = 0; q < pieces && ok; q += kBatch)
        ok = issue_batch(min(kBatch, pieces - q), kPieceWeights, slot, bt, q * kPairSubs, kPairSubs, pol_first);
      ++bq_head;
      t_idle = 0;
      continue;
    }
    if (!have) {
      if (stopped) {
        unsigned dd = lane == 0 ? ld_vol(&sh.dec_done) : 0u;
        if (__shfl_sync(kFull, dd, 0) == (unsigned)kDeciders) break;
      } else {
        bool full = lane == 0 && test_phase_cluster(&sh.item_full[n % kQD], (n / kQD) & 1u);
        full = __shfl_sync(kFull, full, 0);
        if (full) {
          it = read_info(&sh.slot[n % kQD].info);
          t_idle = 0;
          if (it.kind == kItemStop) {
            stopped = true;
            continue;
          }
          have = true;
          pn = 0;
          half = 0;
          if (it.kind == kItemPair && !dep) {
            grid_dep_wait();  // the draft rows come from the drafter
            dep = true;
          }
          if (lane == 0) *reinterpret_cast<volatile unsigned *>(&sh.prod_item) = n + 1u;
        }
      }
      if (!have) {
        // nothing to issue yet: poll again shortly, for a bounded time
        if (t_idle == 0) {
          t_idle = global_timer_ns();
        } else if (global_timer_ns() - t_idle > kWaitLimitNs) {
          if (lane == 0) set_status(a.status, kStatusTimeout);
          ok = false;
        } else if (ld_vol_i(a.status) & kStatusTimeout) {
          ok = false;
        }
        ok = __all_sync(kFull, ok);
        __nanosleep(64);
        continue;
      }
    }
    // a pair streams its target row, then its draft row
    const int slot = (int)(n % kQD);
    const bool pair = it.kind == kItemPair;
    const int m = min(kBatch, (P - pn + kRowSubs - 1) / kRowSubs);
    ok = issue_batch(m, half ? kPieceRowDraft : kPieceRow, slot, it, pn, kRowSubs, pair ? pol_norm : pol_first);
    pn += m * kRowSubs;
    if (pn >= P) {
      if (pair && half == 0) {
        half = 1;
        pn = 0;
      } else {
        have = false;
        ++n;
      }
    }
  }
  if (ok) ok = issue_batch(kWorkers, kPieceStop, 0, it, 0, 0, 0);
  if (!ok && lane == 0) {
    // let copies still in flight land before the CTA exits
    for (uint32_t q = g > (uint32_t)kStages ? g - kStages : 0u; q < g; ++q)
      if (!mbar_wait(&sh.full[q % kStages], (q / kStages) & 1u, a.status)) break;
  }
}

// ---------------------------------------------------------------- workers

__device__ void worker(const VerifyArgs &a, Shared &sh, const float *ring, int w, int s0) {
  const int lane = threadIdx.x & 31;
  const float c = kLog2e / a.T;
  const bool greedy = a.mode == 0;
  for (uint32_t g = (uint32_t)w;; g += kWorkers) {
    const int st = (int)(g % kStages);
    // Stages are shared round-robin, so this warp can reach a stage whose
    // previous piece (another warp's) has not landed yet -- the barrier's
    // parity would then read as complete.  The stage's piece number tells.
    bool ok = true;
    {
      const uint64_t t0 = global_timer_ns();
      for (uint32_t it = 0;; ++it) {
        if (ld_vol(&sh.tag[st].seq) == g + 1u) {
          if (try_phase_local(&sh.full[st], (g / kStages) & 1u, 20000u)) break;
        } else {
          __nanosleep(32);
        }
        if ((it & 63u) == 63u) {
          if (ld_vol_i(a.status) & kStatusTimeout) {
            ok = false;
            break;
          }
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            set_status(a.status, kStatusTimeout);
            ok = false;
            break;
          }
        }
      }
    }
    ok = __all_sync(kFull, ok);
    if (!ok) break;
    const Tag t = sh.tag[st];
    if (t.kind == kPieceStop) break;
    const float *buf = ring + (size_t)st * kStageF;
    SlotState &ss = sh.slot[t.slot];
    const ItemInfo inf = ss.info;
    const Span s0p = stage_span(a, inf, t.kind, s0, t.p, t.np, 0);
    if (t.kind == kPieceRow || t.kind == kPieceRowDraft) {
      // a row's sub-chunks two at a time, their reductions interleaved; the
      // first-pass barrier counts two arrivals per sub-chunk: one per row of a
      // pair, two for a lone row
      const int half = t.kind == kPieceRowDraft ? 1 : 0;
      const uint32_t cnt = inf.kind == kItemPair ? 1u : 2u;
      // all four sub-chunks at once (past the piece's end: -inf), so that
      // their reductions overlap
      float x[4][16];
#pragma unroll
      for (int i = 0; i < kRowSubs; ++i) load_sub(buf, s0p, i, -INFINITY, x[i]);
      float2 r[4];
      if (greedy) {
#pragma unroll
        for (int i = 0; i < kRowSubs; ++i) r[i] = part_argmax(x[i], s0p.e0 + i * kSub);
      } else {
        float m[4], sm[4];
#pragma unroll
        for (int i = 0; i < kRowSubs; ++i) m[i] = redux_max(lane_max16(x[i]));
#pragma unroll
        for (int i = 0; i < kRowSubs; ++i) sm[i] = lane_sumexp16(x[i], m[i], c);
        warp_sum4(sm);
#pragma unroll
        for (int i = 0; i < kRowSubs; ++i) r[i] = make_float2(m[i], sm[i]);
      }
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < kRowSubs; ++i)
          if (i < t.np) {
            reinterpret_cast<float2 *>(&ss.stats[t.p + i])[half] = r[i];
            mbar_arrive_n(&sh.adone[t.slot], cnt);
          }
      }
    } else {
      const Span s1p = stage_span(a, inf, t.kind, s0, t.p, t.np, 1);
      const float *buf1 = buf + kPairSubs * kSub;
      const float Mt = ss.Mt, Ml = ss.Ml, iZt = ss.iZt, iZl = ss.iZl;
      for (int i = 0; i < t.np; ++i) {
        float x[16], y[16];
        load_sub(buf, s0p, i, -INFINITY, x);
        load_sub(buf1, s1p, i, -INFINITY, y);
        float sr = 0.f, sp = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          sr += weight(0, x[m], y[m], Mt, Ml, iZt, iZl, c);
          sp += weight(1, x[m], y[m], Mt, Ml, iZt, iZl, c);
        }
        warp_sum2(sr, sp);
        if (lane == 0) {
          reinterpret_cast<float2 *>(&ss.stats[t.p + i])[0] = make_float2(sr, sp);
          mbar_arrive(&sh.bdone[t.slot]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.empty[st]);
  }
}

// ---------------------------------------------------------------- claimer

// The cluster's first CTA: takes items from the global counter, at most
// a.p.lookahead items ahead of its producer, and hands each to every CTA of the
// cluster (a remote store and a remote arrive per CTA).
__device__ void claimer(const VerifyArgs &a, Shared &sh, int C) {
  const int lane = threadIdx.x & 31;
  int stops = 0;
  bool ok = true;
  if (a.k_eff) grid_dep_wait();  // the drafts kept come from the drafter
  for (uint32_t n = 0; stops < kDeciders && ok; ++n) {
    const int s = (int)(n % kQD);
    if (stops == 0) {
      // stay close behind the producer, so the last items spread over the clusters
      const uint64_t t0 = global_timer_ns();
      while (ld_vol(&sh.prod_item) + (unsigned)a.p.lookahead < n) {
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          if (lane == 0) set_status(a.status, kStatusTimeout);
          ok = false;
          break;
        }
        if (ld_vol_i(a.status) & kStatusTimeout) {
          ok = false;
          break;
        }
        __nanosleep(64);
      }
      ok = __all_sync(kFull, ok);
      if (!ok) break;
    }
    if (n >= (uint32_t)kQD) {
      ok = wait_phase<true>(&sh.item_empty[s], ((n / kQD) - 1u) & 1u, a.status);
      ok = __all_sync(kFull, ok);
      if (!ok) break;
    }
    // items come only from the counter: a cluster that is not yet resident
    // owns nothing another one could be waiting for
    unsigned idx = 0xffffffffu;
    if (stops == 0 && lane == 0) idx = atomicAdd(&a.ctl[0], 1u);
    idx = __shfl_sync(kFull, idx, 0);
    const ItemInfo it = stops == 0 ? decode(a, idx) : ItemInfo{kItemStop, 0, 0, 0};
    if (it.kind == kItemStop) ++stops;
    if (lane < C) {
      int4 *dst = dsmem_ptr_mut(reinterpret_cast<int4 *>(&sh.slot[s].info), (uint32_t)lane);
      *dst = make_int4(it.kind, it.b, it.j, it.kb);
      mbar_arrive_remote(&sh.item_full[s], (uint32_t)lane);
    }
  }
}

// ---------------------------------------------------------------- deciders

// Send this CTA's partial to slot s of every CTA of the cluster, then wait
// for all C partials to arrive here.
__device__ bool exchange(Xchg *slot_x, uint64_t *bar, uint32_t parity, const Xchg &mine, int rank, int C,
                         int *status) {
  const int lane = threadIdx.x & 31;
  if (lane < C) {
    Xchg *dst = dsmem_ptr_mut(slot_x + rank, (uint32_t)lane);
    *dst = mine;
    mbar_arrive_remote(bar, (uint32_t)lane);
  }
  const bool ok = wait_phase<true>(bar, parity, status);
  return __all_sync(kFull, ok);
}

// The inverse-CDF draw of an item, made by the CTA whose slice holds the
// crossing (or, if rounding leaves none, the last positive weight).  mass(p)
// is local sub-chunk p's weight, summed the way every reader sums it: lane l
// holds sub-chunks 2l and 2l+1, then an inclusive scan over the lanes.
template <typename MassFn>
__device__ int draw_in_slice(const VerifyArgs &a, MassFn mass, int P, int s0, bool crossing_here, double before,
                             double tgt, int slast, int wk, const float *rt, const float *rl, float Mt, float Ml,
                             float iZt, float iZl, float c) {
  const int lane = threadIdx.x & 31, V = a.V;
  const int p0 = 2 * lane, p1 = 2 * lane + 1;
  const double m0 = p0 < P ? mass(p0) : 0.0, m1 = p1 < P ? mass(p1) : 0.0;
  const double incl = warp_incl_scan_d(m0 + m1);
  int sb = -1;
  double bef = 0.0;
  if (crossing_here) {
    const unsigned cross = __ballot_sync(kFull, p0 < P && before + incl > tgt);
    if (cross) {
      const int cl = __ffs(cross) - 1;
      if (lane == cl) {
        const double ex = before + (incl - (m0 + m1));
        if (ex + m0 > tgt || !(p1 < P)) {
          sb = s0 + p0;
          bef = ex;
        } else {
          sb = s0 + p1;
          bef = ex + m0;
        }
      }
      sb = __shfl_sync(kFull, sb, cl);
      bef = __shfl_sync(kFull, bef, cl);
    } else {
      // rounding: this slice's own last positive sub-chunk
      slast = warp_max_i(m1 > 0.0 ? s0 + p1 : (m0 > 0.0 ? s0 + p0 : -1));
      crossing_here = false;
    }
  }
  if (!crossing_here) sb = slast;
  if (sb < 0) return -1;
  // rescan sub-chunk sb: each lane a contiguous run of 16 elements, float64
  constexpr int RUN = kSub / 32;
  const int e0 = sb * kSub, e1 = min(V, e0 + kSub);
  const int q0 = min(e1, e0 + lane * RUN), q1 = min(e1, q0 + RUN);
  float wv[RUN];
#pragma unroll
  for (int i = 0; i < RUN; ++i)
    wv[i] = q0 + i < q1 ? weight(wk, __ldcg(rt + q0 + i), wk == 2 ? 0.f : __ldcg(rl + q0 + i), Mt, Ml, iZt, iZl, c)
                        : 0.f;
  double ls = 0.0;
  int lastpos = -1;
#pragma unroll
  for (int i = 0; i < RUN; ++i) {
    ls += (double)wv[i];
    if (wv[i] > 0.f) lastpos = q0 + i;
  }
  const double inc = warp_incl_scan_d(ls);
  int found = 0x7fffffff;
  if (crossing_here && bef + inc > tgt) {
    double run = bef + (inc - ls);
#pragma unroll
    for (int i = 0; i < RUN; ++i) {
      run += (double)wv[i];
      if (found == 0x7fffffff && run > tgt && q0 + i < q1) found = q0 + i;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    found = min(found, __shfl_xor_sync(kFull, found, o));
    lastpos = max(lastpos, __shfl_xor_sync(kFull, lastpos, o));
  }
  return found != 0x7fffffff ? found : lastpos;
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// The position of a sequence claimed last: k (the bonus row in stochastic mode).
__device__ __forceinline__ int last_position(const VerifyArgs &a) { return a.k; }

// Record position j's outcome (flags, token) as one 64-bit word.  The item of
// the position claimed last also gathers the other positions' words (lane l
// holds position l's word in `pre`, loaded when the item started; missing ones
// are polled, bounded), picks the first rejection, writes the outputs and
// resets the sequence's state (warp-collective).
__device__ void record(const VerifyArgs &a, int b, int j, int kb, int word, int tok, unsigned long long pre) {
  const int lane = threadIdx.x & 31, k = a.k, V = a.V;
  unsigned long long *rb = a.rec + (size_t)b * (k + 1);
  const unsigned long long mine = ((unsigned long long)(unsigned)tok << 32) | (unsigned)(word | kRecWritten);
  if (!in_bounds(b < a.B && j <= k, a.status)) return;
  if (j != last_position(a)) {
    if (lane == 0) st_relaxed_u64(rb + j, mine);
    return;
  }
  unsigned long long r = lane == j ? mine : pre;
  if (lane <= k && !(r & (unsigned long long)kRecWritten)) {
    const uint64_t t0 = global_timer_ns();
    for (;;) {
      r = ld_relaxed_u64(rb + lane);
      if (r & (unsigned long long)kRecWritten) break;
      if (ld_vol_i(a.status) & kStatusTimeout) break;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        set_status(a.status, kStatusTimeout);
        break;
      }
      __nanosleep(256);
    }
  }
  const int rw = (int)(unsigned)r, rt = (int)(unsigned)(r >> 32);
  int d = 0;
  if (lane < kb) d = __ldcg(&a.draft_tok[(size_t)b * k + lane]);
  const bool bad = lane < kb && (d < 0 || d >= V);
  bool acc;
  if (a.mode == 0) acc = lane < kb && !bad && rt == d;
  else acc = lane < kb && !bad && (rw & kRecAccept) != 0;
  const unsigned rejm = __ballot_sync(kFull, lane < kb && !acc);
  const int n_acc = rejm ? __ffs(rejm) - 1 : kb;
  const int tok_out = __shfl_sync(kFull, rt, n_acc);
  // flags of the positions the chain reached
  int flags = lane <= n_acc ? (rw & (kRecBadToken | kRecNonFinite)) : 0;
  if (lane <= n_acc && bad) flags |= kRecBadToken;
  flags = (int)__reduce_or_sync(kFull, (unsigned)flags);
  int *o = a.out_tok + (size_t)b * (k + 1);
  if (lane <= k) {
    o[lane] = lane < n_acc ? d : (lane == n_acc ? tok_out : -1);
    rb[lane] = 0ull;
  }
  if (lane == 0) {
    a.accept_len[b] = n_acc + 1;
    a.num_accepted[b] = n_acc;
    a.hint[b] = 0u;
    if (flags & kRecBadToken) set_status(a.status, kStatusBadToken);
    if (flags & kRecNonFinite) set_status(a.status, kStatusNonFinite);
  }
}

__device__ void decider(const VerifyArgs &a, Shared &sh, int d, int rank, int C, int s0, int P) {
  const int lane = threadIdx.x & 31, k = a.k, V = a.V;
  const float c = kLog2e / a.T;
  const Xchg none{0.0, 0.0, -INFINITY, -INFINITY, 0x7fffffff, 0};
  const Xchg none2{0.0, 0.0, 0.f, 0.f, -1, -1};
  uint32_t bpar = 0, x2par = 0;  // phase bits of the weight pass / second exchange, per slot
  grid_dep_wait();  // draft tokens and logits come from the drafter
  for (uint32_t n = (uint32_t)d;; n += kDeciders) {
    const int s = (int)(n % kQD);
    const uint32_t par = (n / kQD) & 1u;
    bool ok = wait_phase<true>(&sh.item_full[s], par, a.status);
    if (!__all_sync(kFull, ok)) break;
    SlotState &ss = sh.slot[s];
    const ItemInfo it = read_info(&ss.info);
    if (it.kind == kItemStop) break;
    const int b = it.b, j = it.j;
    const bool pair = it.kind == kItemPair, bonus = it.kind == kItemBonus;
    // inputs of the decision, fetched while the rows stream
    int dtok = -1;
    float v = 0.f;
    unsigned hv = 0;
    if (pair) dtok = __ldcg(&a.draft_tok[(size_t)b * k + j]);
    const bool valid = dtok >= 0 && dtok < V;
    if (pair && valid && lane == 0) v = __ldg(target_row(a, b, j) + dtok);
    if (pair && valid && lane == 1) v = __ldcg(draft_row(a, b, j) + dtok);
    if (pair && lane == 2) v = __ldg(&a.u_accept[(size_t)b * k + j]);
    if ((pair || bonus) && lane == 3) v = __ldg(&a.u_final[b]);
    if ((pair || bonus) && rank == 0 && lane == 4) hv = ld_vol(&a.hint[b]);
    unsigned long long pre = 0ull;
    if (j == last_position(a) && lane <= k) pre = ld_relaxed_u64(a.rec + (size_t)b * (k + 1) + lane);

    ok = wait_phase<false>(&sh.adone[s], par, a.status);
    if (!__all_sync(kFull, ok)) break;

    // this CTA's partial: lane l combines sub-chunks l and l+32
    Xchg mine = none;
    if (!pair && !bonus) {
      float m = -INFINITY;
      int idx = 0x7fffffff;
      for (int p = lane; p < P; p += 32) argmax_merge(m, idx, ss.stats[p].x, __float_as_int(ss.stats[p].y));
      warp_argmax(m, idx);
      mine.m0 = m;
      mine.i0 = idx;
    } else {
      float m0 = -INFINITY, m1 = -INFINITY;
      for (int p = lane; p < P; p += 32) {
        m0 = fmaxf(m0, ss.stats[p].x);
        if (pair) m1 = fmaxf(m1, ss.stats[p].z);
      }
      m0 = warp_max(m0);
      m1 = warp_max(m1);
      double z0 = 0.0, z1 = 0.0;
      for (int p = lane; p < P; p += 32) {
        const float4 q = ss.stats[p];
        if (q.x != -INFINITY) z0 += (double)q.y * (double)ex2_approx((q.x - m0) * c);
        if (pair && q.z != -INFINITY) z1 += (double)q.w * (double)ex2_approx((q.z - m1) * c);
      }
      mine.z0 = warp_sum_d(z0);
      mine.z1 = warp_sum_d(z1);
      mine.m0 = m0;
      mine.m1 = m1;
      mine.i0 = (int)__shfl_sync(kFull, hv, 4);
    }
    if (!exchange(ss.x1, &sh.x1bar[s], par, mine, rank, C, a.status)) break;

    // combine the C partials (every CTA computes the same)
    const Xchg xr = lane < C ? ss.x1[lane] : none;
    if (!pair && !bonus) {
      float m = xr.m0;
      int idx = xr.i0;
      warp_argmax(m, idx);
      if (lane == 0) mbar_arrive_remote(&sh.item_empty[s], 0u);
      if (rank == 0) record(a, b, j, it.kb, m > -INFINITY ? 0 : kRecNonFinite, idx == 0x7fffffff ? 0 : idx, pre);
      continue;
    }
    const float M0 = warp_max(xr.m0), M1 = warp_max(xr.m1);
    const double Z0 = warp_sum_d(lane < C && xr.m0 != -INFINITY ? xr.z0 * (double)ex2_approx((xr.m0 - M0) * c) : 0.0);
    const double Z1 = warp_sum_d(lane < C && xr.m1 != -INFINITY ? xr.z1 * (double)ex2_approx((xr.m1 - M1) * c) : 0.0);
    const unsigned hint0 = (unsigned)__shfl_sync(kFull, xr.i0, 0);
    const float td = __shfl_sync(kFull, v, 0), ldv = __shfl_sync(kFull, v, 1);
    const float ua = __shfl_sync(kFull, v, 2), uf = __shfl_sync(kFull, v, 3);
    int word = 0;
    bool draw;
    if (pair) {
      bool accept = false;
      if (!valid) {
        word |= kRecBadToken;
      } else {
        if (M0 == -INFINITY || M1 == -INFINITY) word |= kRecNonFinite;
        const double p = exp2(((double)td - (double)M0) * (double)c) / Z0;
        const double q = exp2(((double)ldv - (double)M1) * (double)c) / Z1;
        accept = (double)ua * q < p;
      }
      if (accept) word |= kRecAccept;
      if (!accept && rank == 0 && lane == 0) atomicMax(&a.hint[b], (unsigned)(k + 1 - j));
      // the draw is needed only if no earlier position is known to reject
      draw = !accept && !(hint0 > (unsigned)(k + 1 - j));
    } else {
      draw = hint0 == 0u;  // the bonus token is needed only if nothing rejected
    }
    if (!draw) {
      if (lane == 0) mbar_arrive_remote(&sh.item_empty[s], 0u);
      if (rank == 0) record(a, b, j, it.kb, word, 0, pre);
      continue;
    }
    const float Mt = M0, Ml = M1;
    const float iZt = (float)(1.0 / Z0), iZl = pair ? (float)(1.0 / Z1) : 0.f;
    auto bonus_mass = [&](int p) -> double {
      const float4 q = ss.stats[p];
      return q.x == -INFINITY ? 0.0 : (double)q.y * (double)ex2_approx((q.x - Mt) * c);
    };
    Xchg mine2 = none2;
    const int p0 = 2 * lane, p1 = 2 * lane + 1;
    if (pair) {
      // the weight pass: the pair again (from L2) through the ring
      if (lane == 0) {
        ss.Mt = Mt;
        ss.Ml = Ml;
        ss.iZt = iZt;
        ss.iZl = iZl;
        const unsigned pos = atomicAdd(&sh.bq_tail, 1u);
        sh.bq[pos % kQD] = s;
        __threadfence_block();
        *reinterpret_cast<volatile unsigned *>(&sh.bq_seq[pos % kQD]) = pos + 1u;
      }
      ok = wait_phase<false>(&sh.bdone[s], (bpar >> s) & 1u, a.status);
      bpar ^= 1u << s;
      if (!__all_sync(kFull, ok)) break;
      const double r0 = p0 < P ? (double)ss.stats[p0].x : 0.0, r1 = p1 < P ? (double)ss.stats[p1].x : 0.0;
      const double q0 = p0 < P ? (double)ss.stats[p0].y : 0.0, q1 = p1 < P ? (double)ss.stats[p1].y : 0.0;
      mine2.z0 = __shfl_sync(kFull, warp_incl_scan_d(r0 + r1), 31);
      mine2.z1 = __shfl_sync(kFull, warp_incl_scan_d(q0 + q1), 31);
      mine2.i0 = warp_max_i(r1 > 0.0 ? s0 + p1 : (r0 > 0.0 ? s0 + p0 : -1));
      mine2.i1 = warp_max_i(q1 > 0.0 ? s0 + p1 : (q0 > 0.0 ? s0 + p0 : -1));
    } else {
      // bonus: the sub-chunk weights follow from the first pass
      const double q0 = p0 < P ? bonus_mass(p0) : 0.0, q1 = p1 < P ? bonus_mass(p1) : 0.0;
      mine2.z1 = __shfl_sync(kFull, warp_incl_scan_d(q0 + q1), 31);
      mine2.i1 = warp_max_i(q1 > 0.0 ? s0 + p1 : (q0 > 0.0 ? s0 + p0 : -1));
    }
    if (!exchange(ss.x2, &sh.x2bar[s], (x2par >> s) & 1u, mine2, rank, C, a.status)) break;
    x2par ^= 1u << s;
    const Xchg yr = lane < C ? ss.x2[lane] : none2;
    const double SR = warp_sum_d(yr.z0);
    const bool use_p = bonus || !(SR > 0.0);
    const double own = use_p ? yr.z1 : yr.z0;
    const double tgt = (double)uf * warp_sum_d(own);
    const double incl = warp_incl_scan_d(own);
    const unsigned cross = __ballot_sync(kFull, lane < C && incl > tgt);
    int chooser, slast = -1;
    double before = 0.0;
    if (cross) {
      chooser = __ffs(cross) - 1;
      before = __shfl_sync(kFull, incl - own, chooser);
    } else {
      const int mylast = use_p ? yr.i1 : yr.i0;
      slast = warp_max_i(mylast);
      const unsigned holder = __ballot_sync(kFull, lane < C && slast >= 0 && mylast == slast);
      chooser = holder ? __ffs(holder) - 1 : 0;
    }
    if (rank == chooser) {
      const int wk = bonus ? 2 : (use_p ? 1 : 0);
      const float *rt = target_row(a, b, j);
      const float *rl = pair ? draft_row(a, b, j) : rt;
      int chosen;
      if (bonus) {
        chosen = draw_in_slice(a, bonus_mass, P, s0, cross != 0u, before, tgt, slast, wk, rt, rl, Mt, Ml, iZt, iZl,
                               c);
      } else if (use_p) {
        auto pm = [&](int p) -> double { return (double)ss.stats[p].y; };
        chosen = draw_in_slice(a, pm, P, s0, cross != 0u, before, tgt, slast, wk, rt, rl, Mt, Ml, iZt, iZl, c);
      } else {
        auto rm = [&](int p) -> double { return (double)ss.stats[p].x; };
        chosen = draw_in_slice(a, rm, P, s0, cross != 0u, before, tgt, slast, wk, rt, rl, Mt, Ml, iZt, iZl, c);
      }
      if (chosen < 0) {
        word |= kRecNonFinite;
        chosen = 0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(&sh.item_empty[s], 0u);
      record(a, b, j, it.kb, word, chosen, pre);
    } else if (lane == 0) {
      mbar_arrive_remote(&sh.item_empty[s], 0u);
    }
  }
  __syncwarp();
  if (lane == 0) atomicAdd(&sh.dec_done, 1u);
}

}  // namespace

__global__ void __launch_bounds__(kVerifyThreads, 2) verify_kernel(VerifyArgs a) {
  trace_start(kTkVerify);
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Shared &sh = *reinterpret_cast<Shared *>(smem_raw);
  float *ring = reinterpret_cast<float *>(smem_raw + kHdr);
  const int warp = threadIdx.x >> 5;
  const int C = (int)cluster_size(), rank = (int)cluster_rank();
  const int NS = a.p.NS;
  const int s0 = (int)(((long long)rank * NS) / C), s1 = (int)(((long long)(rank + 1) * NS) / C);
  const int P = s1 - s0;  // >= 1: a cluster is never wider than a row has sub-chunks
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sh.full[i], 1);
      mbar_init(&sh.empty[i], 1);
      sh.tag[i].seq = 0u;
    }
    for (int i = 0; i < kQD; ++i) {
      mbar_init(&sh.item_full[i], 1);
      mbar_init(&sh.item_empty[i], C);
      mbar_init(&sh.adone[i], 2 * P);
      mbar_init(&sh.bdone[i], P);
      mbar_init(&sh.x1bar[i], C);
      mbar_init(&sh.x2bar[i], C);
      sh.bq[i] = 0;
      sh.bq_seq[i] = 0u;
    }
    sh.bq_tail = 0u;
    sh.prod_item = 0u;
    sh.dec_done = 0u;
    fence_barrier_init();
  }
  __syncthreads();
  cluster_sync();  // every CTA's barriers exist before the first remote arrive
  grid_dep_launch();
  if (warp < kWorkers) {
    worker(a, sh, ring, warp, s0);
  } else if (warp == kProducerWarp) {
    producer(a, sh, ring, s0, P);
  } else if (warp == kClaimerWarp) {
    if (rank == 0) claimer(a, sh, C);
  } else {
    decider(a, sh, warp - kFirstDecider, rank, C, s0, P);
  }
  __syncwarp();
  cluster_sync();  // no CTA leaves while a peer may still write to its shared memory
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&a.ctl[1], 1u) == gridDim.x - 1u) {  // the last CTA resets the counters
      a.ctl[0] = 0u;
      a.ctl[1] = 0u;
    }
  }
  grid_dep_wait();
  trace_end(kTkVerify);
}

// ---------------------------------------------------------------- host side

namespace {
size_t up256(size_t x) { return (x + 255) / 256 * 256; }
int sub_chunks(int V) { return (V + kSub - 1) / kSub; }
long long env_int(const char *name, long long dflt) {
  const char *v = getenv(name);
  return v && *v ? atoll(v) : dflt;
}
int g_max_clusters[kMaxC + 1];  // resident clusters per cluster size (0: not asked yet)

int max_clusters(int C) {
  if (g_max_clusters[C] > 0) return g_max_clusters[C];
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)C * 64u);
  cfg.blockDim = dim3(kVerifyThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, verify_kernel, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = 1;
  }
  g_max_clusters[C] = n;
  return n;
}
}  // namespace

size_t verify_state_bytes(int B, int k, int V) {
  size_t n = 256;                       // claim / exit counters
  n += up256((size_t)B * 4);            // rejection hints
  n += up256((size_t)B * (k + 1) * 8);  // per-position records
  n += split_state_bytes(B, k, V);      // the ticketed stochastic kernel's
  return n;
}

void verify_bind_state(VerifyArgs &a, void *state) {
  char *p = static_cast<char *>(state);
  a.ctl = reinterpret_cast<unsigned *>(p);
  p += 256;
  a.hint = reinterpret_cast<unsigned *>(p);
  p += up256((size_t)a.B * 4);
  a.rec = reinterpret_cast<unsigned long long *>(p);
  p += up256((size_t)a.B * (a.k + 1) * 8);
  // residual items start about this many 128 KB items after their sequence's statistics
  split_bind_state(a, p, (int)std::max(1ll, std::min(1ll << 20, env_int("MTP_SPLIT_LAG", 512))));
  a.shint = (int)std::max(0ll, std::min(12ll, env_int("MTP_SPLIT_HINT", 4)));
}

bool plan_verify(int B, int k, int V, VerifyPlan *p) {
  VerifyPlan q{};
  q.NS = sub_chunks(V);
  int C = (int)env_int("MTP_VERIFY_C", 6);
  C = std::max(1, std::min(kMaxC, C));
  while (C < kMaxC && (q.NS + C - 1) / C > kMaxP) ++C;
  C = std::min(C, q.NS);
  if ((q.NS + C - 1) / C > kMaxP) return false;
  q.C = C;
  q.lookahead = (int)std::max(1ll, std::min(6ll, env_int("MTP_VERIFY_LA", 2)));
  const long long total = (long long)B * (k + 1);
  if (total >= (1ll << 31)) return false;
  q.total = (unsigned)total;
  const int g = (int)env_int("MTP_VERIFY_G", 0);
  q.G = (int)std::max<long long>(1, std::min<long long>(g > 0 ? g : max_clusters(C), total));
  *p = q;
  return true;
}

cudaError_t verify_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(verify_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t s, bool pdl) {
  if (a.split) return launch_verify_split(a, s, pdl);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(a.p.G * a.p.C));
  cfg.blockDim = dim3(kVerifyThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)a.p.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  note_launch();
  return cudaLaunchKernelEx(&cfg, verify_kernel, a);
}

MTP_TRACE_COLLECTOR(verify)

}  // namespace mtp
