// Verification of k drafted tokens per sequence ("The Tiny Draft Model Hidden
// Inside Qwen", section "How the draft becomes real output"; "Speculative
// Decoding and MTP: Why Guessing Is Free", sections "Speculative decoding:
// draft, then verify" and "It's exact, not approximate").
//
// Every logit row is cut into chunks of 8 slices, a slice being m sub-chunks
// of 512 elements.  Each CTA has 8 worker warps and a coordinator warp; work
// items are chunks:
//  pass-1 item (b, row, chunk)  reduced to (max, lowest argmax) -- greedy -- or
//                               to the max and sum exp2((x - max) * log2e / T);
//  pass-2 item (b, chunk)       stochastic only: the sampling weights -- max(0,
//                               p - q) and p at the first rejection, or p at the
//                               bonus position -- summed per sub-chunk.
// Coordinators claim the pass-1 items in index order (sequence by sequence)
// from one atomic counter and queue them in shared memory; worker w streams
// slice w of every queued chunk through its own ring of 4 KB shared-memory
// stages (1-D TMA bulk copies issued up to three stages ahead, across items)
// and hands its partial back through shared memory.  The coordinator merges
// the slices and publishes the chunk's partial; a third role, the decider
// warp, takes the tickets (up to 32 per round trip) so that the coordinator
// never waits on one.  The decider that takes a sequence's last ticket
// combines the partials in chunk order, takes the accept / reject decisions
// and publishes them.  Pass-2 item (b, u) is
// owned by CTA (b U + u) mod G, which queues it ahead of new claims as soon as
// b is decided -- so the re-read rows are still in L2 and the work is spread
// evenly -- and the decider that takes its last pass-2 ticket locates the
// sub-chunk holding the inverse-CDF crossing and rescans it in float64.  No
// result depends on which CTA ran which pass-1 item.
//
// Partials and masses are published with relaxed stores of words that are
// never zero and read by polling until non-zero; decisions with a release /
// acquire flag.  Readers zero what they consumed, as they do the tickets and
// flags, so each call leaves the state in the workspace zero for the next
// one.  A coordinator never blocks: it waits for nothing but published data
// whose producers were all claimed by running CTAs.  Every wait is bounded and
// flags the status word when it gives up.
#include <stdlib.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace mtp {

namespace {

constexpr int kWorkers = 8;      // worker warps; then the coordinator and the decider warp
constexpr int kDQ = 64;          // published items waiting for their tickets
constexpr int kScr = 1024;       // decider scratch: published words gathered at once
constexpr int kStages = 3;       // ring stages per worker
#ifndef MTP_VERIFY_STAGE
#define MTP_VERIFY_STAGE 1024
#endif
constexpr int kStage = MTP_VERIFY_STAGE;  // floats per stage
constexpr int kSub = 512;        // sampling sub-chunk (elements)
#ifndef MTP_VERIFY_Q
#define MTP_VERIFY_Q 3
#endif
constexpr int kQ = MTP_VERIFY_Q;  // queued items per CTA
constexpr int kMaxM = 16;        // sub-chunks per slice, at most
constexpr unsigned kFull = 0xffffffffu;

// One queued item.
struct Slot {
  int pass, b, r, u;        // pass 0: stop
  const float *p0, *p1;     // row bases: the row (pass 1); target, draft (pass 2)
  int draft, keep, kind, pad;
  float Mt, Ml, iZt, iZl;   // pass 2: the sequence's decision
  float2 part[kWorkers];    // pass 1: per-slice partials
  float2 mass[kWorkers][kMaxM];  // pass 2: per-sub-chunk (residual, target) masses
};

struct Shared {
  Slot slot[kQ];
  uint64_t ready[kQ];  // coordinator -> workers
  uint64_t done[kQ];   // workers -> coordinator
  uint64_t ring_bar[kWorkers][kStages];
  // coordinator -> decider: published items (b, pass) awaiting their tickets
  int dq_b[kDQ], dq_pass[kDQ];
  unsigned dq_tail, dq_head;
  int coord_done;
  unsigned long long scr[kScr];  // decider: a sequence's partials or masses
};

constexpr size_t kHdr = (sizeof(Shared) + 127) / 128 * 128;
constexpr size_t kSmemBytes = kHdr + (size_t)kWorkers * kStages * kStage * 4;

// ---------------------------------------------------------------- gpu-scope memory

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(unsigned *p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed64(const void *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed64(void *p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// A published word: poll until it is non-zero (bounded).
__device__ unsigned long long poll64(const void *p, int *status) {
  unsigned long long v = ld_relaxed64(p);
  if (v) return v;
  const uint64_t t0 = global_timer_ns();
  while ((v = ld_relaxed64(p)) == 0ull) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      set_status(status, kStatusTimeout);
      return 0ull;
    }
    __nanosleep(32);
  }
  return v;
}

// Up to kBatch published words per lane (lane + 32 i < n): all loads issued
// first, then the few that had not landed are polled.
constexpr int kBatch = 4;
__device__ __forceinline__ void load_batch(const unsigned long long *base, int n, int lane, unsigned long long *w,
                                           int *status) {
#pragma unroll
  for (int i = 0; i < kBatch; ++i) w[i] = lane + 32 * i < n ? ld_relaxed64(base + lane + 32 * i) : 1ull;
#pragma unroll
  for (int i = 0; i < kBatch; ++i)
    if (w[i] == 0ull) w[i] = poll64(base + lane + 32 * i, status);
}

__device__ __forceinline__ unsigned long long pack(float lo, float hi) {
  return (unsigned long long)__float_as_uint(lo) | ((unsigned long long)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float lo_f(unsigned long long w) { return __uint_as_float((unsigned)w); }
__device__ __forceinline__ float hi_f(unsigned long long w) { return __uint_as_float((unsigned)(w >> 32)); }

// Non-zero encodings of a published partial.  Stochastic (max, sum): a finite
// max has sum >= 1 and -inf is not zero.  Greedy (max, argmax + 1).
__device__ __forceinline__ unsigned long long enc_greedy(float v, int i) {
  return (unsigned long long)__float_as_uint(v) | ((unsigned long long)((unsigned)i + 1u) << 32);
}
__device__ __forceinline__ int dec_greedy_idx(unsigned long long w) { return (int)((unsigned)(w >> 32) - 1u); }
// Masses (>= 0) carry the sign bit.
__device__ __forceinline__ unsigned long long enc_mass(float r, float p) {
  return pack(__uint_as_float(__float_as_uint(r) | 0x80000000u), __uint_as_float(__float_as_uint(p) | 0x80000000u));
}

__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// 2^x, hardware approximation (relative error about 2^-22; -inf gives +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Sampling weight of one element: residual max(0, p - q) (kind 0), target p
// (kind 1), unnormalised target weight exp2((t - Mt) c) (kind 2).
__device__ __forceinline__ float weight(int kind, float t, float l, float Mt, float Ml, float iZt, float iZl,
                                        float c) {
  const float e = ex2((t - Mt) * c);
  if (kind == 2) return e;
  const float p = e * iZt;
  if (kind == 1) return p;
  return fmaxf(0.f, p - ex2((l - Ml) * c) * iZl);
}

// ---------------------------------------------------------------- items

struct Item {
  int pass;  // 1, 2; 0: none
  int b, r, u;
};

__device__ __forceinline__ Item decode(const VerifyArgs &a, unsigned idx) {
  const VerifyPlan &p = a.p;
  Item it{0, 0, 0, 0};
  if (idx >= p.total) return it;
  const unsigned n1 = (unsigned)p.n1, U = (unsigned)p.U;
  const unsigned rem = idx % n1;
  it.pass = 1;
  it.b = (int)(idx / n1);
  it.r = (int)(rem / U);
  it.u = (int)(rem % U);
  return it;
}

// Stream row r of a sequence -- greedy: target k .. 0; stochastic: target
// k .. 1, draft k-1 .. 1, target 0, draft 0 -- as an index into the target
// [B, k+1] or draft [B, k] row arrays.
__device__ __forceinline__ size_t stream_row(const VerifyArgs &a, int b, int r, bool &draft) {
  const int k = a.k;
  int pos;
  draft = false;
  if (a.mode == 0 || r < k) {
    pos = k - r;
  } else if (r < 2 * k - 1) {
    pos = 2 * k - 1 - r;
    draft = true;
  } else {
    pos = 0;
    draft = r == 2 * k;
  }
  return draft ? (size_t)b * k + pos : (size_t)b * (k + 1) + pos;
}

// Stream rows of target position j and of draft position j.
__device__ __forceinline__ int trow(int mode, int k, int j) { return mode == 0 ? k - j : (j == 0 ? 2 * k - 1 : k - j); }
__device__ __forceinline__ int drow(int k, int j) { return j == 0 ? 2 * k : 2 * k - 1 - j; }

// Sub-chunks [s0, s1) of slice w of chunk u.
__device__ __forceinline__ void slice_subs(const VerifyPlan &p, int u, int w, int &s0, int &s1) {
  s0 = min(p.NS, (u * kWorkers + w) * p.m);
  s1 = min(p.NS, s0 + p.m);
}

// What a worker's ring streams for one item: nq pieces of `per` elements from
// p0 (and, for the residual, the same from p1 into the second half of the stage).
struct Src {
  const float *p0, *p1;
  int len, per, nq;
  uint64_t pol;
  bool draft;  // reads draft logits: the drafter must have finished
  bool valid;
};

// ---------------------------------------------------------------- decisions

__device__ __forceinline__ const unsigned long long *part1_row(const VerifyArgs &a, int b, int r) {
  return reinterpret_cast<const unsigned long long *>(a.part1) + ((size_t)b * a.p.nrows + r) * a.p.U;
}

// Combined (max, sum) of stream row r of sequence b over its U chunks, in
// chunk order; every lane gets the result.
__device__ void row_lse(const VerifyArgs &a, int b, int r, float c, float &M, double &Z) {
  const int U = a.p.U, lane = threadIdx.x & 31;
  const unsigned long long *row = part1_row(a, b, r);
  float m = -INFINITY;
  double z = 0.0;
  for (int u0 = 0; u0 < U; u0 += 32 * kBatch) {  // one round of loads per 128 chunks
    unsigned long long w[kBatch];
    load_batch(row + u0, U - u0, lane, w, a.status);
    float mm = -INFINITY;
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (lane + 32 * i < U - u0) mm = fmaxf(mm, lo_f(w[i]));
    mm = warp_max(mm);
    const float mn = fmaxf(m, mm);
    if (mn != -INFINITY) {
      double zz = 0.0;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const float pm = lo_f(w[i]);
        if (lane + 32 * i < U - u0 && pm != -INFINITY) zz += (double)hi_f(w[i]) * (double)ex2((pm - mn) * c);
      }
      z = (m == -INFINITY ? 0.0 : z * (double)ex2((m - mn) * c)) + zz;
      m = mn;
    }
  }
  M = m;
  Z = warp_sum_d(z);
}

// (max, lowest argmax) of stream row r of sequence b; every lane gets it.
__device__ void row_argmax(const VerifyArgs &a, int b, int r, float &M, int &I) {
  const int U = a.p.U, lane = threadIdx.x & 31;
  const unsigned long long *row = part1_row(a, b, r);
  M = -INFINITY;
  I = 0x7fffffff;
  for (int u0 = 0; u0 < U; u0 += 32 * kBatch) {
    unsigned long long w[kBatch];
    load_batch(row + u0, U - u0, lane, w, a.status);
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (lane + 32 * i < U - u0) argmax_merge(M, I, lo_f(w[i]), dec_greedy_idx(w[i]));
  }
  warp_argmax(M, I);
}

// Zero the sequence's published partials for the next call (each is read,
// i.e. has landed, before it is overwritten).
__device__ void clear_part1(const VerifyArgs &a, int b) {
  const int lane = threadIdx.x & 31, n = a.p.nrows * a.p.U;
  unsigned long long *base = reinterpret_cast<unsigned long long *>(a.part1) + (size_t)b * n;
  for (int i0 = 0; i0 < n; i0 += 32 * kBatch) {
    unsigned long long w[kBatch];
    load_batch(base + i0, n - i0, lane, w, a.status);
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (lane + 32 * i < n - i0) st_relaxed64(base + i0 + lane + 32 * i, 0ull);
  }
}

// Gather n <= kScr published words into scratch: all loads of a round (16
// per lane) are issued before any is looked at, then late ones are polled.
__device__ void gather(const unsigned long long *src, int n, unsigned long long *scr, int *status) {
  const int lane = threadIdx.x & 31;
  for (int i0 = 0; i0 < n; i0 += 512) {
    unsigned long long w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int e = i0 + lane + 32 * i;
      w[i] = e < n ? ld_relaxed64(src + e) : 1ull;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int e = i0 + lane + 32 * i;
      if (e < n) scr[e] = w[i] ? w[i] : poll64(src + e, status);
    }
  }
  __syncwarp();
}

// Row statistics from gathered partials (entries r*U .. r*U+U-1).
__device__ void scr_row_lse(const unsigned long long *scr, int U, int r, float c, float &M, double &Z) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  for (int u = lane; u < U; u += 32) m = fmaxf(m, lo_f(scr[r * U + u]));
  M = warp_max(m);
  double z = 0.0;
  if (M != -INFINITY)
    for (int u = lane; u < U; u += 32) {
      const unsigned long long w = scr[r * U + u];
      if (lo_f(w) != -INFINITY) z += (double)hi_f(w) * (double)ex2((lo_f(w) - M) * c);
    }
  Z = warp_sum_d(z);
}

__device__ void scr_row_argmax(const unsigned long long *scr, int U, int r, float &M, int &I) {
  const int lane = threadIdx.x & 31;
  M = -INFINITY;
  I = 0x7fffffff;
  for (int u = lane; u < U; u += 32) argmax_merge(M, I, lo_f(scr[r * U + u]), dec_greedy_idx(scr[r * U + u]));
  warp_argmax(M, I);
}

// Zero n gathered (so landed) published words for the next call.
__device__ void zero_words(unsigned long long *dst, int n) {
  for (int i = threadIdx.x & 31; i < n; i += 32) st_relaxed64(dst + i, 0ull);
}

// Greedy decision of sequence b (warp-collective): accept drafts while they
// equal the target argmax, then emit the argmax of the first disagreeing row.
__device__ void decide_greedy(const VerifyArgs &a, int b, unsigned long long *scr) {
  const int k = a.k, V = a.V, lane = threadIdx.x & 31, U = a.p.U, n = a.p.nrows * U;
  grid_dep_wait();  // the drafts come from the drafter
  const int my = lane < k ? __ldcg(&a.draft_tok[(size_t)b * k + lane]) : 0;
  unsigned long long *src = reinterpret_cast<unsigned long long *>(a.part1) + (size_t)b * n;
  const bool gathered = n <= kScr;
  if (gathered) gather(src, n, scr, a.status);
  int acc_n = 0;
  float M;
  int I;
  for (;;) {
    if (gathered) scr_row_argmax(scr, U, trow(0, k, acc_n), M, I);
    else row_argmax(a, b, trow(0, k, acc_n), M, I);
    if (acc_n == k) break;
    const int d = __shfl_sync(kFull, my, acc_n);
    if (d < 0 || d >= V) {
      if (lane == 0) set_status(a.status, kStatusBadToken);
      break;
    }
    if (!(M > -INFINITY) && lane == 0) set_status(a.status, kStatusNonFinite);
    if (I != d) break;
    ++acc_n;
  }
  int *o = a.out_tok + (size_t)b * (k + 1);
  if (lane <= k) o[lane] = lane < acc_n ? my : (lane == acc_n ? (I == 0x7fffffff ? 0 : I) : -1);
  if (lane == 0) {
    a.accept_len[b] = acc_n + 1;
    a.num_accepted[b] = acc_n;
    a.cnt1[b] = 0u;
  }
  if (gathered) zero_words(src, n);
  else clear_part1(a, b);
}

// Stochastic decision of sequence b (warp-collective): the ratio tests in
// position order; publishes the sampling task for the pass-2 items.
__device__ void decide_stochastic(const VerifyArgs &a, int b, float c, unsigned long long *scr) {
  const int k = a.k, V = a.V, lane = threadIdx.x & 31, U = a.p.U, n = a.p.nrows * U;
  grid_dep_wait();
  // lanes 0-7: target logit at drafted token j; 8-15: draft logit at it;
  // 16-23: u_accept; lane 24: u_final
  const int j = lane & 7, g = lane >> 3;
  const int dj = j < k ? __ldcg(&a.draft_tok[(size_t)b * k + j]) : -1;
  const bool valid = dj >= 0 && dj < V;
  float val = 0.f;
  if (g == 0 && j < k && valid) val = __ldg(&a.target[((size_t)b * (k + 1) + j) * V + dj]);
  if (g == 1 && j < k && valid) val = __ldcg(&a.draft[((size_t)b * k + j) * V + dj]);
  if (g == 2 && j < k) val = __ldg(&a.u_accept[(size_t)b * k + j]);
  if (lane == 24) val = __ldg(&a.u_final[b]);
  unsigned long long *src = reinterpret_cast<unsigned long long *>(a.part1) + (size_t)b * n;
  const bool gathered = n <= kScr;
  if (gathered) gather(src, n, scr, a.status);
  auto stats = [&](int r, float &M, double &Z) {
    if (gathered) scr_row_lse(scr, U, r, c, M, Z);
    else row_lse(a, b, r, c, M, Z);
  };
  int acc_n = 0, rej = k;
  float Mt = 0.f, Ml = 0.f;
  double Zt = 1.0, Zl = 1.0;
  for (int q = 0; q < k; ++q) {
    const int d = __shfl_sync(kFull, dj, q);
    const float td = __shfl_sync(kFull, val, q), ld = __shfl_sync(kFull, val, 8 + q);
    const float ua = __shfl_sync(kFull, val, 16 + q);
    bool accept = false;
    stats(trow(1, k, q), Mt, Zt);
    stats(drow(k, q), Ml, Zl);
    if (d < 0 || d >= V) {
      if (lane == 0) set_status(a.status, kStatusBadToken);
    } else {
      if ((Mt == -INFINITY || Ml == -INFINITY) && lane == 0) set_status(a.status, kStatusNonFinite);
      const double p = exp2(((double)td - (double)Mt) * (double)c) / Zt;
      const double qq = exp2(((double)ld - (double)Ml) * (double)c) / Zl;
      accept = (double)ua * qq < p;
    }
    if (!accept) {
      rej = q;
      break;
    }
    ++acc_n;
  }
  if (rej == k) stats(trow(1, k, k), Mt, Zt);  // bonus token from target row k
  const float uf = __shfl_sync(kFull, val, 24);
  if (gathered) zero_words(src, n);
  else clear_part1(a, b);
  if (lane == 0) {
    VerifyDecision &dd = a.dec[b];
    dd.acc_n = acc_n;
    dd.rej = rej;
    dd.kind = rej == k ? 2 : 0;
    dd.uf = uf;
    dd.Mt = Mt;
    dd.iZt = (float)(1.0 / Zt);
    dd.Ml = rej < k ? Ml : 0.f;
    dd.iZl = rej < k ? (float)(1.0 / Zl) : 0.f;
    a.cnt1[b] = 0u;
    st_release(&a.flag[b], 1u);
  }
}

// Final sampling of sequence b (warp-collective): locate the sub-chunk holding
// the inverse-CDF crossing from the per-sub-chunk masses, rescan it in
// float64, write the outputs.
__device__ void sample_final(const VerifyArgs &a, int b, const VerifyDecision &dd, float c,
                             unsigned long long *scr) {
  const int k = a.k, V = a.V, lane = threadIdx.x & 31;
  grid_dep_wait();
  const int my = lane < dd.acc_n ? __ldcg(&a.draft_tok[(size_t)b * k + lane]) : 0;
  const int NS = a.p.NS;
  unsigned long long *msg = reinterpret_cast<unsigned long long *>(a.mass2) + (size_t)b * NS;
  const bool gathered = NS <= kScr;
  if (gathered) gather(msg, NS, scr, a.status);
  const unsigned long long *ms = gathered ? scr : msg;
  const int per = (NS + 31) / 32;
  const int s0 = min(NS, lane * per), s1 = min(NS, s0 + per);
  double lr = 0.0, lp = 0.0;
  int lastR = -1, lastP = -1;
  for (int s = s0; s < s1; ++s) {
    const unsigned long long w = gathered ? ms[s] : poll64(msg + s, a.status);
    const float mr = fabsf(lo_f(w)), mp = fabsf(hi_f(w));
    lr += (double)mr;
    lp += (double)mp;
    if (mr > 0.f) lastR = s;
    if (mp > 0.f) lastP = s;
  }
  const double SR = warp_sum_d(lr);
  const double SP = warp_sum_d(lp);
  // weights: the residual; the target itself if the residual is identically
  // zero; the unnormalised target row k for the bonus token
  const bool use_p = dd.kind == 2 || !(SR > 0.0);
  const double own = use_p ? lp : lr;
  const double tgt = (double)dd.uf * (use_p ? SP : SR);
  double incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  const unsigned cross = __ballot_sync(kFull, s1 > s0 && incl > tgt);
  int sstar = -1;
  double before = 0.0;
  if (cross) {
    const int cl = __ffs(cross) - 1;
    if (lane == cl) {
      double cum = incl - own;
      for (int s = s0; s < s1; ++s) {
        const unsigned long long w = gathered ? ms[s] : ld_relaxed64(msg + s);
        const double m = use_p ? (double)fabsf(hi_f(w)) : (double)fabsf(lo_f(w));
        if (cum + m > tgt) {
          sstar = s;
          before = cum;
          break;
        }
        cum += m;
      }
    }
    sstar = __shfl_sync(kFull, sstar, cl);
    before = __shfl_sync(kFull, before, cl);
  }
  int slast = use_p ? lastP : lastR;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) slast = max(slast, __shfl_xor_sync(kFull, slast, o));
  const int sb = sstar >= 0 ? sstar : slast;

  const int pos = dd.kind == 2 ? k : dd.rej;
  const float *rt = a.target + ((size_t)b * (k + 1) + pos) * V;
  const float *rl = dd.kind == 2 ? rt : a.draft + ((size_t)b * k + pos) * V;
  const int wk = dd.kind == 2 ? 2 : (use_p ? 1 : 0);
  int chosen = -1;
  if (sb >= 0) {
    // each lane a contiguous run of 16 elements, float64 prefix sums
    constexpr int RUN = kSub / 32;
    const int e0 = sb * kSub, e1 = min(V, e0 + kSub);
    const int a0 = min(e1, e0 + lane * RUN), a1 = min(e1, a0 + RUN);
    float wv[RUN];
#pragma unroll
    for (int i = 0; i < RUN; ++i)
      wv[i] = a0 + i < a1 ? weight(wk, __ldcg(rt + a0 + i), wk == 2 ? 0.f : __ldcg(rl + a0 + i), dd.Mt, dd.Ml,
                                   dd.iZt, dd.iZl, c)
                          : 0.f;
    double ls = 0.0;
    int lastpos = -1;
#pragma unroll
    for (int i = 0; i < RUN; ++i) {
      ls += (double)wv[i];
      if (wv[i] > 0.f) lastpos = a0 + i;
    }
    double inc = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double t = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += t;
    }
    int found = 0x7fffffff;
    if (sstar >= 0 && before + inc > tgt) {
      double run = before + (inc - ls);
#pragma unroll
      for (int i = 0; i < RUN; ++i) {
        run += (double)wv[i];
        if (found == 0x7fffffff && run > tgt && a0 + i < a1) found = a0 + i;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      found = min(found, __shfl_xor_sync(kFull, found, o));
      lastpos = max(lastpos, __shfl_xor_sync(kFull, lastpos, o));
    }
    chosen = found != 0x7fffffff ? found : lastpos;
  }
  if (chosen < 0) {
    if (lane == 0) set_status(a.status, kStatusNonFinite);
    chosen = 0;
  }
  int *o = a.out_tok + (size_t)b * (k + 1);
  if (lane <= k) o[lane] = lane < dd.acc_n ? my : (lane == dd.acc_n ? chosen : -1);
  // every mass was read above, so it has landed: zero them for the next call
  zero_words(msg, NS);
  if (lane == 0) {
    a.accept_len[b] = dd.acc_n + 1;
    a.num_accepted[b] = dd.acc_n;
    a.cnt2[b] = 0u;
    a.flag[b] = 0u;
  }
}

// ---------------------------------------------------------------- worker warp

__device__ void worker(const VerifyArgs &a, Shared &sh, float *ring, uint64_t *bar, int w) {
  const int lane = threadIdx.x & 31;
  const int V = a.V;
  const bool stoch = a.mode == 1;
  const float c = kLog2e / a.T;
  const uint64_t pol_first = l2_policy_evict_first();
  const uint64_t pol_keep = a.p.pol == 1 ? l2_policy_evict_normal() : l2_policy_evict_last();

  uint32_t n_iss = 0, n_cons = 0, n_done = 0;  // ring pieces: issued (lane 0), consumed, confirmed
  bool ok = true, dep_waited = false;
  // issue cursor (lane 0): source `is` of queue position n_is, piece qi
  Src is{};
  uint32_t n_is = 0xffffffffu;
  int qi = 0;

  auto src_for = [&](const Slot &sl) {
    Src s{};
    int s0, s1;
    slice_subs(a.p, sl.u, w, s0, s1);
    const int e0 = s0 * kSub, e1 = min(V, s1 * kSub);
    s.valid = true;
    s.draft = sl.draft != 0;
    if (sl.pass == 1) {
      const int mis = (int)((reinterpret_cast<uintptr_t>(sl.p0 + e0) >> 2) & 3u);
      const int h1 = min(e1, e0 + ((4 - mis) & 3));
      const int b1 = h1 + max(0, e1 - h1) / 4 * 4;
      s.p0 = sl.p0 + h1;
      s.p1 = nullptr;
      s.len = b1 - h1;
      s.per = kStage;
      s.nq = s.len > 0 ? (s.len + kStage - 1) / kStage : 0;
      s.pol = sl.keep ? pol_keep : pol_first;
    } else if ((V & 3) == 0) {
      s.p0 = sl.p0 + e0;
      s.p1 = sl.p1 ? sl.p1 + e0 : nullptr;
      s.len = e1 - e0;
      s.per = kSub;
      s.nq = max(0, s1 - s0);
      s.pol = pol_first;
    } else {
      s.nq = 0;  // unaligned rows: plain loads
    }
    return s;
  };
  // lane 0: keep up to kStages pieces in flight, moving on to the next queued
  // item once it is ready
  auto top_up = [&](uint32_t n) {
    while (ok && n_iss - n_cons < (uint32_t)kStages) {
      if (qi >= is.nq) {
        if (n_is != n) break;  // already one item ahead
        const uint32_t nn = n + 1;
        if (!mbar_test(&sh.ready[nn % kQ], (nn / kQ) & 1u)) break;
        const Slot &sl = sh.slot[nn % kQ];
        if (sl.pass == 0) break;
        is = src_for(sl);
        n_is = nn;
        qi = 0;
        continue;
      }
      if (is.draft && !dep_waited) {
        grid_dep_wait();
        dep_waited = true;
      }
      const int st = (int)(n_iss % kStages);
      const int cnt = min(is.per, is.len - qi * is.per);
      const uint32_t bytes = (uint32_t)cnt * 4u;
      float *dst = ring + (size_t)st * kStage;
      mbar_arrive_expect_tx(&bar[st], is.p1 ? 2u * bytes : bytes);
      bulk_g2s_hint(dst, is.p0 + (size_t)qi * is.per, bytes, &bar[st], is.pol);
      if (is.p1) bulk_g2s_hint(dst + kStage / 2, is.p1 + (size_t)qi * is.per, bytes, &bar[st], is.pol);
      ++qi;
      ++n_iss;
    }
  };
  auto wait_piece = [&]() -> const float * {
    const int st = (int)(n_cons % kStages);
    if (ok) ok = mbar_sleep_wait(&bar[st], (n_cons / kStages) & 1u, a.status);
    ok = __all_sync(kFull, ok);
    if (ok) n_done = n_cons + 1;
    return ring + (size_t)st * kStage;
  };

  for (uint32_t n = 0;; ++n) {
    const int q = (int)(n % kQ);
    if (ok) ok = mbar_sleep_wait(&sh.ready[q], (n / kQ) & 1u, a.status);
    ok = __all_sync(kFull, ok);
    if (!ok) break;
    const Slot &sl = sh.slot[q];
    if (sl.pass == 0) break;
    if (lane == 0) {
      if (n_is != n) {  // the cursor had not reached this item yet
        is = src_for(sl);
        n_is = n;
        qi = 0;
      }
      top_up(n);
    }
    int s0, s1;
    slice_subs(a.p, sl.u, w, s0, s1);
    const int e0 = s0 * kSub, e1 = min(V, s1 * kSub);

    if (sl.pass == 1) {
      // ------------------------------------------------------------ pass 1
      const float *rowp = sl.p0;
      const bool draft = sl.draft != 0;
      const int mis = (int)((reinterpret_cast<uintptr_t>(rowp + e0) >> 2) & 3u);
      const int h1 = min(e1, e0 + ((4 - mis) & 3));
      const int b1 = h1 + max(0, e1 - h1) / 4 * 4;
      const int len = b1 - h1, nq = len > 0 ? (len + kStage - 1) / kStage : 0;
      float bv = -INFINITY, m = -INFINITY, s = 0.f;
      int bi = 0x7fffffff;
      for (int p = 0; p < nq; ++p) {
        const float4 *b4 = reinterpret_cast<const float4 *>(wait_piece());
        const int nf4 = min(kStage, len - p * kStage) / 4;
        const int vbase = h1 + p * kStage;
        if (!stoch) {
          // this lane's maximum over the piece (a balanced tree), then -- only
          // when it beats the running maximum -- its lowest index
          float4 x[kStage / 128];
          float mi[kStage / 128];
#pragma unroll
          for (int i = 0; i < kStage / 128; ++i) {
            const int f = lane + 32 * i;
            x[i] = f < nf4 ? b4[f] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            mi[i] = fmaxf(fmaxf(x[i].x, x[i].y), fmaxf(x[i].z, x[i].w));
          }
#pragma unroll
          for (int h = kStage / 256; h > 0; h >>= 1)
#pragma unroll
            for (int i = 0; i < h; ++i) mi[i] = fmaxf(mi[i], mi[i + h]);
          const float pm = mi[0];
          if (pm > bv) {
            int idx = 0x7fffffff;
#pragma unroll
            for (int i = kStage / 128 - 1; i >= 0; --i) {  // the last assignment is the lowest index
              const int v = vbase + 4 * (lane + 32 * i);
              if (x[i].w == pm) idx = v + 3;
              if (x[i].z == pm) idx = v + 2;
              if (x[i].y == pm) idx = v + 1;
              if (x[i].x == pm) idx = v;
            }
            bv = pm;
            bi = idx;
          }
        } else {
          float4 x[kStage / 128];
          float pm = -INFINITY;
#pragma unroll
          for (int i = 0; i < kStage / 128; ++i) {
            const int f = lane + 32 * i;
            x[i] = f < nf4 ? b4[f] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            pm = fmaxf(pm, fmaxf(fmaxf(x[i].x, x[i].y), fmaxf(x[i].z, x[i].w)));
          }
          if (pm > m) {
            s = m == -INFINITY ? 0.f : s * ex2((m - pm) * c);
            m = pm;
          }
          if (m != -INFINITY) {
            const float mc = m * c;
#pragma unroll
            for (int i = 0; i < kStage / 128; ++i) {
              s += ex2(fmaf(x[i].x, c, -mc)) + ex2(fmaf(x[i].y, c, -mc));
              s += ex2(fmaf(x[i].z, c, -mc)) + ex2(fmaf(x[i].w, c, -mc));
            }
          }
        }
        __syncwarp();
        ++n_cons;
        if (lane == 0) {
          fence_proxy_async_smem();
          top_up(n);
        }
      }
      if (lane < 4) {  // unaligned head / tail elements of the slice
        for (int h = 0; h < 2; ++h) {
          const int v = h == 0 ? e0 + lane : b1 + lane;
          if (h == 0 ? v < h1 : v < e1) {
            if (draft) grid_dep_wait();
            const float x = __ldcg(rowp + v);
            if (!stoch) {
              argmax_merge(bv, bi, x, v);
            } else if (x != -INFINITY) {
              if (x > m) {
                s = (m == -INFINITY ? 0.f : s * ex2((m - x) * c)) + 1.f;
                m = x;
              } else {
                s += ex2((x - m) * c);
              }
            }
          }
        }
      }
      if (!stoch) warp_argmax(bv, bi);
      else warp_lse(m, s, c);
      if (lane == 0) sh.slot[q].part[w] = stoch ? make_float2(m, s) : make_float2(bv, __int_as_float(bi));
    } else {
      // ------------------------------------------------------------ pass 2
      const int kind = sl.kind;
      const float Mt = sl.Mt, Ml = sl.Ml, iZt = sl.iZt, iZl = sl.iZl;
      if (sl.draft) grid_dep_wait();
      if ((V & 3) == 0) {
        // ring pieces of 512 target (and draft) elements, one sub-chunk each
        for (int p = 0; p < s1 - s0; ++p) {
          const float *buf = wait_piece();
          const int nf4 = min(kSub, e1 - e0 - p * kSub) / 4;
          float sr = 0.f, sp = 0.f;
#pragma unroll
          for (int i = 0; i < kSub / 128; ++i) {
            const int f = lane + 32 * i;
            if (f < nf4) {
              const float4 t = reinterpret_cast<const float4 *>(buf)[f];
              if (kind == 2) {
                sp += weight(2, t.x, 0.f, Mt, Ml, iZt, iZl, c) + weight(2, t.y, 0.f, Mt, Ml, iZt, iZl, c);
                sp += weight(2, t.z, 0.f, Mt, Ml, iZt, iZl, c) + weight(2, t.w, 0.f, Mt, Ml, iZt, iZl, c);
              } else {
                const float4 l = reinterpret_cast<const float4 *>(buf + kStage / 2)[f];
                sr += weight(0, t.x, l.x, Mt, Ml, iZt, iZl, c) + weight(0, t.y, l.y, Mt, Ml, iZt, iZl, c);
                sr += weight(0, t.z, l.z, Mt, Ml, iZt, iZl, c) + weight(0, t.w, l.w, Mt, Ml, iZt, iZl, c);
                sp += weight(1, t.x, l.x, Mt, Ml, iZt, iZl, c) + weight(1, t.y, l.y, Mt, Ml, iZt, iZl, c);
                sp += weight(1, t.z, l.z, Mt, Ml, iZt, iZl, c) + weight(1, t.w, l.w, Mt, Ml, iZt, iZl, c);
              }
            }
          }
          __syncwarp();
          ++n_cons;
          if (lane == 0) {
            fence_proxy_async_smem();
            top_up(n);
          }
          sr = warp_sum(sr);
          sp = warp_sum(sp);
          if (lane == 0) sh.slot[q].mass[w][p] = make_float2(sr, sp);
        }
      } else {
        // unaligned rows: plain loads, one sub-chunk at a time
        for (int p = 0; p < s1 - s0; ++p) {
          const int v0 = e0 + p * kSub, v1 = min(e1, v0 + kSub);
          float sr = 0.f, sp = 0.f;
          for (int v = v0 + lane; v < v1; v += 32) {
            const float t = __ldcg(sl.p0 + v);
            if (kind == 2) {
              sp += weight(2, t, 0.f, Mt, Ml, iZt, iZl, c);
            } else {
              const float l = __ldcg(sl.p1 + v);
              sr += weight(0, t, l, Mt, Ml, iZt, iZl, c);
              sp += weight(1, t, l, Mt, Ml, iZt, iZl, c);
            }
          }
          sr = warp_sum(sr);
          sp = warp_sum(sp);
          if (lane == 0) sh.slot[q].mass[w][p] = make_float2(sr, sp);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sh.done[q]);
  }

  if (lane == 0) {
    // after a timeout, let copies still in flight land before the CTA exits
    for (uint32_t n = n_done; n < n_iss; ++n)
      if (!mbar_wait(&bar[n % kStages], (n / kStages) & 1u, a.status)) break;
  }
}

// ---------------------------------------------------------------- coordinator warp

__device__ void coordinator(const VerifyArgs &a, Shared &sh) {
  const int lane = threadIdx.x & 31;
  const int k = a.k, V = a.V, U = a.p.U;
  const bool stoch = a.mode == 1;
  const float c = kLog2e / a.T;

  // pass-1 claims run one ahead: the next index is requested when one is consumed
  unsigned pre = 0;
  bool have_pre = false, claims_done = false;
  auto claim = [&]() -> unsigned {
    unsigned i = 0;
    if (lane == 0) i = have_pre ? pre : atomicAdd(&a.ctl[0], 1u);
    i = __shfl_sync(kFull, i, 0);
    have_pre = i < a.p.total;
    if (lane == 0 && have_pre) pre = atomicAdd(&a.ctl[0], 1u);
    return i;
  };

  // pass-2 items owned by this CTA: g = blockIdx.x + t * gridDim.x < B * U.
  // Their readiness is probed without waiting: the flag is loaded, looked at
  // on a later iteration, then the decision is loaded and looked at later still.
  const unsigned n2 = stoch ? (unsigned)a.B * (unsigned)U : 0u;
  const unsigned own = blockIdx.x < n2 ? (n2 - blockIdx.x + gridDim.x - 1) / gridDim.x : 0u;
  unsigned t2 = 0;
  int p2 = 0;  // 0: to probe, 1: flag load in flight, 2: decision load in flight
  unsigned fl = 0;
  long long p2_at = 0;  // when the in-flight load may be looked at / the next probe may go
  int d_kind = 0, d_rej = 0;
  float d_Mt = 0.f, d_Ml = 0.f, d_iZt = 0.f, d_iZl = 0.f;
  auto owned_b = [&]() { return (int)((blockIdx.x + t2 * gridDim.x) / (unsigned)U); };
  auto owned_u = [&]() { return (int)((blockIdx.x + t2 * gridDim.x) % (unsigned)U); };
  // Loads are only looked at a round trip after they were issued, so a probe
  // never stalls the coordinator.
  constexpr long long kRoundTrip = 3000, kReprobe = 6000;  // SM clocks
  auto probe = [&]() {  // advance the readiness pipeline of the next owned item
    if (t2 >= own) return;
    const long long now = clock64();
    if (now < p2_at || p2 == 2) return;
    if (p2 == 0) {
      if (lane == 0) fl = ld_acquire(&a.flag[owned_b()]);
      p2 = 1;
      p2_at = now + kRoundTrip;
    } else if (__shfl_sync(kFull, fl, 0) != 0u) {
      if (lane == 0) {
        const VerifyDecision *g = &a.dec[owned_b()];
        d_kind = __ldcg(&g->kind);
        d_rej = __ldcg(&g->rej);
        d_Mt = __ldcg(&g->Mt);
        d_Ml = __ldcg(&g->Ml);
        d_iZt = __ldcg(&g->iZt);
        d_iZl = __ldcg(&g->iZl);
      }
      p2 = 2;
      p2_at = now + kRoundTrip;
    } else {
      p2 = 0;
      p2_at = now + kReprobe;
    }
  };

  // hand a published item to the decider warp (lane 0; waits for ring space)
  auto push = [&](int b, int pass) {
    if (lane == 0) {
      volatile unsigned *vh = &sh.dq_head;
      if (sh.dq_tail - *vh >= (unsigned)kDQ) {
        const uint64_t t0 = global_timer_ns();
        while (sh.dq_tail - *vh >= (unsigned)kDQ) {
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            set_status(a.status, kStatusTimeout);
            break;
          }
          __nanosleep(64);
        }
      }
      const unsigned t = sh.dq_tail;
      sh.dq_b[t % kDQ] = b;
      sh.dq_pass[t % kDQ] = pass;
      __threadfence_block();
      *(volatile unsigned *)&sh.dq_tail = t + 1;
    }
  };

  auto enqueue = [&](uint32_t n, const Item &it) {
    if (lane == 0) {
      Slot &sl = sh.slot[n % kQ];
      sl.pass = it.pass;
      sl.b = it.b;
      sl.r = it.r;
      sl.u = it.u;
      if (it.pass == 1) {
        bool draft;
        const size_t row = stream_row(a, it.b, it.r, draft);
        sl.p0 = (draft ? a.draft : a.target) + row * (size_t)V;
        sl.p1 = nullptr;
        sl.draft = draft;
        sl.keep = stoch && (a.p.pol != 0 || it.r >= 2 * k - 1);  // rows a rejection may read again
      } else if (it.pass == 2) {
        const int pos = d_kind == 2 ? k : d_rej;
        sl.p0 = a.target + ((size_t)it.b * (k + 1) + pos) * V;
        sl.p1 = d_kind == 2 ? nullptr : a.draft + ((size_t)it.b * k + pos) * V;
        sl.draft = d_kind != 2;
        sl.keep = 0;
        sl.kind = d_kind;
        sl.Mt = d_Mt;
        sl.Ml = d_Ml;
        sl.iZt = d_iZt;
        sl.iZl = d_iZl;
      }
      mbar_arrive(&sh.ready[n % kQ]);
    }
    __syncwarp();
  };

  // a finished item: publish its partial or masses, pass it to the decider
  auto complete = [&](uint32_t n) {
    const Slot &sl = sh.slot[n % kQ];
    const int b = sl.b;
    if (sl.pass == 1) {
      float m = -INFINITY, s = 0.f;
      int i = 0x7fffffff;
      if (lane < kWorkers) {
        const float2 p = sl.part[lane];
        m = p.x;
        if (stoch) s = p.y;
        else i = __float_as_int(p.y);
      }
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) {  // the 8 slices, a fixed merge tree
        const float m2 = __shfl_xor_sync(kFull, m, o), s2 = __shfl_xor_sync(kFull, s, o);
        const int i2 = __shfl_xor_sync(kFull, i, o);
        if (stoch) lse_merge(m, s, m2, s2, c);
        else argmax_merge(m, i, m2, i2);
      }
      if (lane == 0) {
        void *dst = a.part1 + ((size_t)b * a.p.nrows + sl.r) * U + sl.u;
        st_relaxed64(dst, stoch ? pack(m, s) : enc_greedy(m, i));
      }
      push(b, 1);
    } else {
      unsigned long long *ms = reinterpret_cast<unsigned long long *>(a.mass2) + (size_t)b * a.p.NS;
      const int base = sl.u * kWorkers * a.p.m;
      for (int e = lane; e < kWorkers * a.p.m; e += 32) {
        const int s = base + e;
        if (s < a.p.NS) {
          const float2 v = sl.mass[e / a.p.m][e % a.p.m];
          st_relaxed64(ms + s, enc_mass(v.x, v.y));
        }
      }
      __syncwarp();
      push(b, 2);
    }
    __syncwarp();
  };

  // Pass-2 items normally wait until the pass-1 claims run out: they then fill
  // the time the last sequences' decisions take instead of leaving it idle.
  // MTP_VERIFY_P2_FIRST=1 queues them as soon as their sequence is decided.
  const bool p2_first = a.p.p2_first != 0;
  uint32_t fill = 0, drain = 0;
  uint64_t idle_since = 0;
  for (;;) {
    bool did = false;
    if (drain < fill) {
      bool fin = false;
      if (lane == 0) {
        if (fill - drain == (uint32_t)kQ)  // nothing else to do: park until it is done
          fin = mbar_sleep_wait(&sh.done[drain % kQ], (drain / kQ) & 1u, a.status);
        else
          fin = mbar_test(&sh.done[drain % kQ], (drain / kQ) & 1u);
      }
      if (__shfl_sync(kFull, fin, 0)) {
        complete(drain);
        ++drain;
        did = true;
      }
    }
    probe();
    if (fill - drain < (uint32_t)kQ) {
      if (p2 == 2 && clock64() >= p2_at && (claims_done || p2_first)) {  // a decided owned pass-2 item
        enqueue(fill, Item{2, owned_b(), 0, owned_u()});
        ++fill;
        ++t2;
        p2 = 0;
        p2_at = 0;
        did = true;
      } else if (!claims_done) {
        const Item it = decode(a, claim());
        if (it.pass) {
          enqueue(fill, it);
          ++fill;
        } else {
          claims_done = true;
        }
        did = true;
      }
    }
    if (claims_done && t2 >= own && drain == fill) {
      enqueue(fill, Item{0, 0, 0, 0});  // stop: the workers leave
      break;
    }
    if (did) {
      idle_since = 0;
    } else {
      const uint64_t now = global_timer_ns();
      if (idle_since == 0) idle_since = now;
      if (now - idle_since > kWaitLimitNs) {  // nothing moved for too long
        if (lane == 0) set_status(a.status, kStatusTimeout);
        if (drain == fill) enqueue(fill, Item{0, 0, 0, 0});
        break;
      }
      __nanosleep(64);
    }
  }
  if (lane == 0) *(volatile int *)&sh.coord_done = 1;
}

// ---------------------------------------------------------------- decider warp

// Takes the tickets of the items the coordinator published -- one atomic per
// lane, up to 32 in flight together -- and, for a sequence's last pass-1
// ticket, decides it; for its last pass-2 ticket, samples it.
__device__ void decider(const VerifyArgs &a, Shared &sh) {
  const int lane = threadIdx.x & 31;
  const bool stoch = a.mode == 1;
  const float c = kLog2e / a.T;
  unsigned head = 0;
  for (;;) {
    unsigned tail = 0;
    int cdone = 0;
    if (lane == 0) {
      cdone = *(volatile int *)&sh.coord_done;
      __threadfence_block();
      tail = *(volatile unsigned *)&sh.dq_tail;
    }
    tail = __shfl_sync(kFull, tail, 0);
    cdone = __shfl_sync(kFull, cdone, 0);
    if (tail == head) {
      if (cdone) break;
      __nanosleep(128);
      continue;
    }
    const unsigned n = min(tail - head, 32u);
    int b = 0, pass = 0;
    unsigned old = 0;
    if ((unsigned)lane < n) {
      b = *(volatile int *)&sh.dq_b[(head + lane) % kDQ];
      pass = *(volatile int *)&sh.dq_pass[(head + lane) % kDQ];
      old = atomicAdd(pass == 1 ? &a.cnt1[b] : &a.cnt2[b], 1u);
    }
    head += n;
    __syncwarp();
    if (lane == 0) *(volatile unsigned *)&sh.dq_head = head;
    const bool last = (unsigned)lane < n && old == (pass == 1 ? (unsigned)a.p.n1 - 1u : (unsigned)a.p.U - 1u);
    unsigned mask = __ballot_sync(kFull, last);
    while (mask) {
      const int j = __ffs(mask) - 1;
      mask &= mask - 1;
      const int bj = __shfl_sync(kFull, b, j), pj = __shfl_sync(kFull, pass, j);
      if (pj == 1) {
        if (stoch) decide_stochastic(a, bj, c, sh.scr);
        else decide_greedy(a, bj, sh.scr);
      } else {
        VerifyDecision dd;
        const VerifyDecision *g = &a.dec[bj];
        dd.acc_n = __ldcg(&g->acc_n);
        dd.rej = __ldcg(&g->rej);
        dd.kind = __ldcg(&g->kind);
        dd.uf = __ldcg(&g->uf);
        dd.Mt = __ldcg(&g->Mt);
        dd.Ml = __ldcg(&g->Ml);
        dd.iZt = __ldcg(&g->iZt);
        dd.iZl = __ldcg(&g->iZl);
        sample_final(a, bj, dd, c, sh.scr);
      }
    }
  }
  // the last CTA out resets the claim counter for the next call
  if (lane == 0 && atomicAdd(&a.ctl[1], 1u) == gridDim.x - 1u) {
    a.ctl[0] = 0u;
    a.ctl[1] = 0u;
  }
}

}  // namespace

constexpr int kMinBlocks = kStage > 1024 ? 1 : 2;  // CTAs per SM the rings allow

__global__ void __launch_bounds__(kVerifyThreads, kMinBlocks) verify_kernel(VerifyArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Shared &sh = *reinterpret_cast<Shared *>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    sh.dq_tail = 0u;
    sh.dq_head = 0u;
    sh.coord_done = 0;
    for (int q = 0; q < kQ; ++q) {
      mbar_init(&sh.ready[q], 1);
      mbar_init(&sh.done[q], kWorkers);
    }
    for (int w = 0; w < kWorkers; ++w)
      for (int s = 0; s < kStages; ++s) mbar_init(&sh.ring_bar[w][s], 1);
    fence_barrier_init();
  }
  __syncthreads();
  grid_dep_launch();
  (void)lane;
  if (warp < kWorkers) {
    float *ring = reinterpret_cast<float *>(smem_raw + kHdr) + (size_t)warp * kStages * kStage;
    worker(a, sh, ring, sh.ring_bar[warp], warp);
  } else if (warp == kWorkers) {
    coordinator(a, sh);
  } else {
    decider(a, sh);
  }
  grid_dep_wait();
}

// ---------------------------------------------------------------- host side

namespace {
size_t up256(size_t x) { return (x + 255) / 256 * 256; }
int sub_chunks(int V) { return (V + kSub - 1) / kSub; }
int max_chunks(int V) { return (sub_chunks(V) + kWorkers - 1) / kWorkers; }  // slices of one sub-chunk
long long env_int(const char *name, long long dflt) {
  const char *v = getenv(name);
  return v && *v ? atoll(v) : dflt;
}
}  // namespace

size_t verify_state_bytes(int B, int k, int V) {
  size_t n = 256;                                           // claim / exit counters
  n += 3 * up256((size_t)B * 4);                            // tickets and flags
  n += up256((size_t)B * sizeof(VerifyDecision));           // decisions
  n += up256((size_t)B * (2 * k + 1) * max_chunks(V) * 8);  // published partials
  n += up256((size_t)B * sub_chunks(V) * 8);                // published masses
  return n;
}

void verify_bind_state(VerifyArgs &a, void *state) {
  char *p = static_cast<char *>(state);
  const int B = a.B, k = a.k, V = a.V;
  a.ctl = reinterpret_cast<unsigned *>(p);
  p += 256;
  a.cnt1 = reinterpret_cast<unsigned *>(p);
  p += up256((size_t)B * 4);
  a.cnt2 = reinterpret_cast<unsigned *>(p);
  p += up256((size_t)B * 4);
  a.flag = reinterpret_cast<unsigned *>(p);
  p += up256((size_t)B * 4);
  a.dec = reinterpret_cast<VerifyDecision *>(p);
  p += up256((size_t)B * sizeof(VerifyDecision));
  a.part1 = reinterpret_cast<float2 *>(p);
  p += up256((size_t)B * (2 * k + 1) * max_chunks(V) * 8);
  a.mass2 = reinterpret_cast<float2 *>(p);
}

bool plan_verify(int B, int k, int V, int mode, int num_sms, int blocks_per_sm, VerifyPlan *p) {
  VerifyPlan q{};
  const bool stoch = mode == 1;
  q.nrows = stoch ? 2 * k + 1 : k + 1;
  q.NS = sub_chunks(V);
  const long long ctas = (long long)num_sms * blocks_per_sm;
  // the widest slice (8 sub-chunks, down to 1) that
  // still gives every CTA about four items
  int m = (int)env_int(stoch ? "MTP_VERIFY_SM" : "MTP_VERIFY_GM", 8);
  m = std::max(1, std::min(kMaxM, m));
  for (;;) {
    q.U = (q.NS + kWorkers * m - 1) / (kWorkers * m);
    if (m <= 1 || (long long)B * q.nrows * q.U >= 4 * ctas) break;
    m /= 2;
  }
  q.m = m;
  q.n1 = q.nrows * q.U;
  q.pol = (int)env_int("MTP_VERIFY_POL", 0);
  q.p2_first = (int)env_int("MTP_VERIFY_P2_FIRST", 0);
  const long long total = (long long)B * q.n1;
  if (total >= (1ll << 31)) return false;
  q.total = (unsigned)total;
  q.grid = (int)std::max<long long>(1, std::min<long long>(ctas, total));
  *p = q;
  return true;
}

cudaError_t verify_set_attributes() {
  return cudaFuncSetAttribute(verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
}

int verify_blocks_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, verify_kernel, kVerifyThreads, kSmemBytes) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  return n < 1 ? 1 : n;
}

cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.p.grid);
  cfg.blockDim = dim3(kVerifyThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  note_launch();
  return cudaLaunchKernelEx(&cfg, verify_kernel, a);
}

}  // namespace mtp
