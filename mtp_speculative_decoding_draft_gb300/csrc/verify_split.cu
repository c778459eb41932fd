// Stochastic verification as one streaming kernel of small CTAs ("The Tiny
// Draft Model Hidden Inside Qwen", section "How the draft becomes real
// output"; "Speculative Decoding and MTP: Why Guessing Is Free", sections
// "Speculative decoding: draft, then verify" and "It's exact, not
// approximate"): the same rule, the same uniforms and the same draw order as
// the cluster kernel of verify.cu.
//
// Every CTA takes one work item by ticket (an atomic counter), so the order
// in which items start is the ticket order whatever the hardware's dispatch
// order.  Per sequence b there are two groups of items:
//   statistics items, one per (row, 32768-element chunk) of its 2k+1 logit
//     rows (target rows t_0..t_k, draft rows q_0..q_{k-1}): the chunk's
//     (max, sum of exp2((x - max) log2e / T)), read in four passes of 8192.
//     The item that completes the sequence (the last to arrive: a fence,
//     then an acquire-release increment) combines the chunks into per-row
//     (max, partition sum), takes u q(d) < p(d) at every kept position at
//     once (the first rejection as taking them in order finds it) and
//     publishes the decision (a release store).  If every draft is accepted
//     it then makes the bonus draw from p of the bonus row -- the chunk
//     masses follow from the statistics, so only the crossing chunk is read
//     again -- and writes the outputs.
//   residual items, one per chunk, placed about `lag` items later in ticket
//     order: each waits for the decision (acquire, bounded; by then it has
//     mostly been made), and after a rejection at position j computes the
//     masses of max(0, p_j - q_j) over its chunk's 512-element sub-chunks.
//     The pairs j <= 1, where the first rejection mostly falls, were read
//     with an evict-last L2 policy and everything else evict-first, so these
//     re-reads mostly hit L2.  The last to arrive finds the crossing chunk,
//     then sub-chunk, then element (float64 running sums, in index order),
//     and writes the outputs.
// A residual item waits only on statistics items with smaller tickets, which
// were taken by CTAs already running, so every wait ends.
#include "common.cuh"
#include "verify_rule.cuh"
#include "internal.h"

namespace mtp {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPer = 32;                   // elements a thread per pass of a statistics item
constexpr int kPiece = kThreads * kPer;    // 8192 elements a pass
constexpr int kPasses = 4;
constexpr int kChunk = kPiece * kPasses;   // 32768 elements an item
constexpr int kSub = 512;                  // draw sub-chunk
constexpr int kSubs = kChunk / kSub;       // 64 sub-chunks a chunk
constexpr int kMaxRows = 17;               // 2 k + 1 rows a sequence, k <= 8
constexpr unsigned kDecidedReject = 1u, kDecidedDone = 2u;

struct Shared {
  float red[kWarps], red2[kWarps];
  float M[kMaxRows];
  double Z[kMaxRows];
  float sub[kSubs];
  SplitRec rec;
  unsigned ticket, dec;
  int last, rej, flags, chosen, ch;
  double tgt, before;
};

struct Item {
  int residual;  // 0: statistics item, 1: residual item
  int b, local;
};

// Ticket t -> item: the statistics groups of sequences 0..lag-1, then per
// sequence s >= lag the statistics group of s followed by the residual group
// of s - lag, then the residual groups of the last lag sequences.
__device__ __forceinline__ Item decode_ticket(const VerifyArgs &a, unsigned long long t) {
  const unsigned long long NA = a.sNA, NB = a.sNB, D = a.sD, B = a.B, P = NA + NB;
  if (t < D * NA) return Item{0, (int)(t / NA), (int)(t % NA)};
  t -= D * NA;
  if (t < (B - D) * P) {
    const unsigned long long p = t / P, r = t % P;
    return r < NA ? Item{0, (int)(D + p), (int)r} : Item{1, (int)p, (int)(r - NA)};
  }
  t -= (B - D) * P;
  return Item{1, (int)(B - D + t / NB), (int)(t % NB)};
}

__device__ __forceinline__ double incl_scan_d(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

__device__ __forceinline__ int warp_min_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ int warp_max_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sampling weight of one element: the residual max(0, p - q) (kind 0), the
// unnormalised target weight exp2((t - Mt) c) (kind 2).
struct Wt {
  int kind;
  float Mt, iZt, Ml, iZl, c;
};

__device__ __forceinline__ float wval(const Wt &w, float t, float l) {
  const float e = ex2_approx((t - w.Mt) * w.c);
  if (w.kind == 2) return e;
  // both products rounded on their own (no fused multiply-add): where p and q
  // are equal the residual must be exactly zero, so that the draw falls back to p
  return fmaxf(0.f, __fmul_rn(e, w.iZt) - __fmul_rn(ex2_approx((l - w.Ml) * w.c), w.iZl));
}

__device__ __forceinline__ float wsum4(const Wt &w, float4 t, float4 l) {
  return (wval(w, t.x, l.x) + wval(w, t.y, l.y)) + (wval(w, t.z, l.z) + wval(w, t.w, l.w));
}

// One warp: the total of mass(0..n-1), summed in index order.
template <typename F>
__device__ double warp_total(F mass, int n) {
  const int lane = threadIdx.x & 31;
  double tot = 0.0;
  for (int b = 0; b < n; b += 32) tot += __shfl_sync(0xffffffffu, incl_scan_d(b + lane < n ? mass(b + lane) : 0.0), 31);
  return tot;
}

// One warp: the smallest index whose running sum (in index order) passes
// tgt, with the mass before it; else the last index of positive mass with
// before = -1; else -1.
template <typename F>
__device__ int warp_crossing(F mass, int n, double tgt, double &before_out) {
  const int lane = threadIdx.x & 31;
  int cross = -1, lastpos = -1;
  double before = 0.0, run = 0.0;
  for (int b = 0; b < n && cross < 0; b += 32) {
    const double x = b + lane < n ? mass(b + lane) : 0.0;
    const double incl = incl_scan_d(x);
    const unsigned hit = __ballot_sync(0xffffffffu, b + lane < n && run + incl > tgt);
    if (hit) {
      const int l = __ffs(hit) - 1;
      cross = b + l;
      before = run + __shfl_sync(0xffffffffu, incl - x, l);
    }
    const unsigned pos = __ballot_sync(0xffffffffu, b + lane < n && x > 0.0);
    if (pos) lastpos = b + 31 - __clz(pos);
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  before_out = cross >= 0 ? before : -1.0;
  return cross >= 0 ? cross : lastpos;
}

// The masses of the 64 sub-chunks of chunk ch into sh.sub: warp w takes
// sub-chunks w, w + 8, ...; a residual pass (two rows) one sub-chunk at a
// time, a target-only pass two at a time, all loads of a step issued first.
// Block-collective, ends with a barrier.
__device__ void chunk_sub_masses(Shared &sh, const Wt &w, const float *trow, const float *lrow, int V, int ch,
                                 uint64_t pol) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool vec = ((reinterpret_cast<uintptr_t>(trow) | reinterpret_cast<uintptr_t>(lrow)) & 15u) == 0;
  const bool pair = w.kind == 0;
  const int step = pair ? 1 : 2;
#pragma unroll 1
  for (int s = warp; s < kSubs; s += step * kWarps) {
    float acc[2] = {0.f, 0.f};
    const int e0 = ch * kChunk + s * kSub, e1 = e0 + kWarps * kSub;  // the step's sub-chunks
    if (vec && (step == 1 ? e0 + kSub : e1 + kSub) <= V) {
      const float4 *t0 = reinterpret_cast<const float4 *>(trow + e0) + lane;
      const float4 *t1 = reinterpret_cast<const float4 *>(trow + e1) + lane;
      const float4 *l0 = reinterpret_cast<const float4 *>(lrow + e0) + lane;
      float4 u[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) u[q] = ld_stream_f4(t0 + 32 * q, pol);
#pragma unroll
      for (int q = 0; q < 4; ++q) u[4 + q] = ld_stream_f4((pair ? l0 : t1) + 32 * q, pol);
      if (pair) {
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[0] += wsum4(w, u[q], u[4 + q]);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[0] += wsum4(w, u[q], u[q]);
          acc[1] += wsum4(w, u[4 + q], u[4 + q]);
        }
      }
    } else {
      for (int h = 0; h < step; ++h) {
        const int f0 = h ? e1 : e0;
        for (int i = f0 + lane; i < min(V, f0 + kSub); i += 32)
          acc[h] += wval(w, ld_stream_f32(trow + i, pol), pair ? ld_stream_f32(lrow + i, pol) : 0.f);
      }
    }
    for (int h = 0; h < step; ++h) {
      const float t = warp_sum(acc[h]);
      if (lane == 0) sh.sub[s + h * kWarps] = t;
    }
  }
  __syncthreads();
}

// One warp: the element of sub-chunk s (global sub-chunk index) at which the
// running sum (`before` ahead of the sub-chunk) passes tgt; before < 0, or
// nothing passing: the last element of positive weight.  -1 if none.
__device__ int warp_rescan(const Wt &w, const float *trow, const float *lrow, int V, int s, double before,
                           double tgt) {
  const int lane = threadIdx.x & 31;
  constexpr int PER = kSub / 32;
  const bool pair = w.kind == 0;
  const int e0 = s * kSub + lane * PER;
  // the lane's weights eight at a time, the eight loads issued together
  constexpr int G = 8;
  double ls = 0.0;
  int lp = -1;
#pragma unroll 1
  for (int q0 = 0; q0 < PER; q0 += G) {
    float x[G];
#pragma unroll
    for (int q = 0; q < G; ++q) {
      const int i = e0 + q0 + q;
      x[q] = i < V ? wval(w, __ldcg(trow + i), pair ? __ldcg(lrow + i) : 0.f) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < G; ++q) {
      ls += (double)x[q];
      if (x[q] > 0.f) lp = e0 + q0 + q;
    }
  }
  const double inc = incl_scan_d(ls);
  int f = 0x7fffffff;
  if (before >= 0.0 && before + inc > tgt) {
    double r = before + (inc - ls);
#pragma unroll 1
    for (int q0 = 0; q0 < PER && f == 0x7fffffff; q0 += G) {
      float x[G];
#pragma unroll
      for (int q = 0; q < G; ++q) {
        const int i = e0 + q0 + q;
        x[q] = i < V ? wval(w, __ldcg(trow + i), pair ? __ldcg(lrow + i) : 0.f) : 0.f;
      }
#pragma unroll
      for (int q = 0; q < G; ++q) {
        r += (double)x[q];
        if (f == 0x7fffffff && x[q] > 0.f && r > tgt) f = e0 + q0 + q;
      }
    }
  }
  f = warp_min_int(f);
  lp = warp_max_int(lp);
  return f != 0x7fffffff ? f : lp;
}

// Within chunk ch whose sub-chunk masses are in sh.sub, with `base` the mass
// before the chunk (< 0: the chunk was taken as the last of positive mass):
// the crossing sub-chunk, then the element.  Warp 0 only.
__device__ int warp_draw_in_chunk(Shared &sh, const Wt &w, const float *trow, const float *lrow, int V, int ch,
                                  double base, double tgt) {
  double b2;
  const int s = warp_crossing([&](int i) { return (double)sh.sub[i]; }, kSubs, base >= 0.0 ? tgt - base : 1e300, b2);
  if (s < 0) return -1;
  const double bef = base >= 0.0 && b2 >= 0.0 ? base + b2 : -1.0;
  return warp_rescan(w, trow, lrow, V, ch * kSubs + s, bef, tgt);
}

// A draw from p of a target row whose chunk statistics are known: the
// crossing chunk from their masses, then its sub-chunks, then its elements.
// Block-collective.
__device__ int draw_from_stats(Shared &sh, const Wt &w, const float2 *pp, int nch, const float *trow, int V,
                               double u) {
  if (threadIdx.x < 32) {
    auto mass = [&](int i) {
      const float2 p = __ldcg(&pp[i]);
      return p.x == -INFINITY ? 0.0 : (double)(p.y * ex2_approx((p.x - w.Mt) * w.c));
    };
    const double tgt = u * warp_total(mass, nch);
    double before;
    const int ch = warp_crossing(mass, nch, tgt, before);
    if (threadIdx.x == 0) {
      sh.ch = ch;
      sh.tgt = tgt;
      sh.before = before;
    }
  }
  __syncthreads();
  const int ch = sh.ch;
  if (ch < 0) return -1;
  chunk_sub_masses(sh, w, trow, trow, V, ch, l2_policy_evict_first());
  if (threadIdx.x < 32) {
    const int f = warp_draw_in_chunk(sh, w, trow, trow, V, ch, sh.before, sh.tgt);
    if (threadIdx.x == 0) sh.chosen = f;
  }
  __syncthreads();
  return sh.chosen;
}

// Rows of sequence b: target j at slot j (j <= k), draft j at slot k + 1 + j.
__device__ __forceinline__ const float *seq_row(const VerifyArgs &a, int b, int i) {
  return i <= a.k ? a.target + ((size_t)b * (a.k + 1) + i) * a.V
                  : a.draft + ((size_t)b * a.k + (i - a.k - 1)) * a.V;
}

__device__ __forceinline__ int drafts_kept(const VerifyArgs &a, int b) {
  return a.k_eff ? min(max(__ldg(&a.k_eff[b]), 0), a.k) : a.k;
}

__device__ void write_outputs(const VerifyArgs &a, int b, int n_acc, int chosen, int flags) {
  const int k = a.k;
  if (chosen < 0) {
    flags |= kStatusNonFinite;
    chosen = 0;
  }
  if (threadIdx.x <= k) {
    const int t = threadIdx.x;
    a.out_tok[(size_t)b * (k + 1) + t] = t < n_acc ? __ldg(&a.draft_tok[(size_t)b * k + t]) : (t == n_acc ? chosen : -1);
  }
  if (threadIdx.x == 0) {
    a.accept_len[b] = n_acc + 1;
    a.num_accepted[b] = n_acc;
    if (flags) set_status(a.status, flags);
  }
}

// The item that completed sequence b's statistics: per-row (max, partition
// sum), the accept decisions, and either the bonus draw (all accepted) or the
// rejection record for the residual items.
__device__ void decide(Shared &sh, const VerifyArgs &a, int b, int kb) {
  const int k = a.k, V = a.V, R = 2 * k + 1, nch = a.snch;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float c = kLog2e / a.T;
  for (int i = warp; i < R; i += kWarps) {
    if (i <= k ? i > kb : i - (k + 1) >= kb) continue;
    const float2 *pp = a.spart + ((size_t)b * R + i) * nch;
    float m = -INFINITY;
    for (int ch = lane; ch < nch; ch += 32) m = fmaxf(m, __ldcg(&pp[ch]).x);
    m = warp_max(m);
    double z = 0.0;
    if (m != -INFINITY)
      for (int ch = lane; ch < nch; ch += 32) {
        const float2 p = __ldcg(&pp[ch]);
        if (p.x != -INFINITY) z += (double)p.y * (double)ex2_approx((p.x - m) * c);
      }
    z = warp_sum_d(z);
    if (lane == 0) {
      sh.M[i] = m;
      sh.Z[i] = z;
    }
  }
  __syncthreads();
  // u q(d) < p(d) at every kept position at once, lane j of warp 0 position
  // j (its token, the logits there and its uniform loaded together); the
  // first rejection and the flags are those of taking them in order
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int dl = -1;
    float tdl = 0.f, ldl = 0.f;
    double ua = 0.0;
    if (lane < kb) {
      dl = __ldg(&a.draft_tok[(size_t)b * k + lane]);
      ua = (double)__ldg(&a.u_accept[(size_t)b * k + lane]);
      if (dl >= 0 && dl < V) {
        tdl = __ldg(seq_row(a, b, lane) + dl);
        ldl = __ldg(seq_row(a, b, k + 1 + lane) + dl);
      }
    }
    const bool valid = dl >= 0 && dl < V;
    bool finite = true, accept = true;
    if (lane < kb && valid) {
      finite = sh.M[lane] > -INFINITY && sh.M[k + 1 + lane] > -INFINITY;
      const double p = exp2(((double)tdl - (double)sh.M[lane]) * (double)c) / sh.Z[lane];
      const double q = exp2(((double)ldl - (double)sh.M[k + 1 + lane]) * (double)c) / sh.Z[k + 1 + lane];
      accept = ua * q < p;
    }
    int fl;
    const int rj = first_rejection(kb, valid, finite, accept, fl);
    if (lane == 0) {
      sh.rej = rj;
      sh.flags = fl;
      if (rj >= 0) {
        SplitRec r;
        r.Mt = sh.M[rj];
        r.iZt = (float)(1.0 / sh.Z[rj]);
        r.Ml = sh.M[k + 1 + rj];
        r.iZl = (float)(1.0 / sh.Z[k + 1 + rj]);
        r.j = rj;
        r.flags = fl;
        a.srec[b] = r;
        __threadfence();
      }
      // published at once: the residual items of the sequence wait for it (a
      // bonus draw's outputs need nothing of theirs)
      st_release_u32(&a.sseq[4 * b + 2], rj >= 0 ? kDecidedReject : kDecidedDone);
    }
  }
  __syncthreads();
  const int rj = sh.rej;
  if (rj < 0) {
    const Wt w{2, sh.M[kb], 0.f, 0.f, 0.f, c};
    const int chosen =
        draw_from_stats(sh, w, a.spart + ((size_t)b * R + kb) * nch, nch, seq_row(a, b, kb), V, (double)__ldg(&a.u_final[b]));
    write_outputs(a, b, kb, chosen, sh.flags);
  }
}

__device__ void statistics_item(Shared &sh, const VerifyArgs &a, int b, int local) {
  const int k = a.k, V = a.V, nch = a.snch;
  const int i = local / nch, ch = local % nch;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb = drafts_kept(a, b);
  const bool used = i <= k ? i <= kb : i - (k + 1) < kb;
  // per thread: a running (max, sum of exp2) over its elements of the passes
  const float c = kLog2e / a.T;
  float mt = -INFINITY, st = 0.f;
  if (used) {
    const float *src = seq_row(a, b, i);
    const bool vec = (reinterpret_cast<uintptr_t>(src) & 15u) == 0;
    // pair rows (t_j, q_j, j < kb) may be read again by the residual pass
    // (hint 3 + n: only the pairs j <= n are kept, the first rejection's usual positions)
    const bool pair_row = (i <= k ? i < kb : true) && (a.shint < 3 || (i <= k ? i : i - (k + 1)) <= a.shint - 3);
    const uint64_t pol = a.shint == 0 ? l2_policy_evict_normal_all()
                         : !pair_row  ? l2_policy_evict_first()
                         : a.shint != 2 ? l2_policy_evict_last() : l2_policy_evict_normal_all();
#pragma unroll 1
    for (int p = 0; p < kPasses; ++p) {
      const int e0 = ch * kChunk + p * kPiece, n = min(kPiece, V - e0);
      if (n <= 0) break;
      float x[kPer];
      if (n == kPiece && vec) {
        const float4 *s4 = reinterpret_cast<const float4 *>(src + e0) + threadIdx.x;
#pragma unroll
        for (int m = 0; m < kPer / 4; ++m) {
          const float4 v = ld_stream_f4(s4 + kThreads * m, pol);
          x[4 * m] = v.x;
          x[4 * m + 1] = v.y;
          x[4 * m + 2] = v.z;
          x[4 * m + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int m = 0; m < kPer; ++m) {
          const int e = threadIdx.x + kThreads * m;
          x[m] = e < n ? ld_stream_f32(src + e0 + e, pol) : -INFINITY;
        }
      }
      float m = x[0];
#pragma unroll
      for (int q = 1; q < kPer; ++q) m = fmaxf(m, x[q]);
      if (m > mt) {
        st = mt == -INFINITY ? 0.f : st * ex2_approx((mt - m) * c);
        mt = m;
      }
      if (mt != -INFINITY) {
        const float mc = mt * c;
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int q = 0; q < kPer; q += 2) {
          s0 += ex2_approx(fmaf(x[q], c, -mc));
          s1 += ex2_approx(fmaf(x[q + 1], c, -mc));
        }
        st += s0 + s1;
      }
    }
  }
  // merge the threads' (max, sum) pairs: a warp, then the CTA
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, mt, o), s2 = __shfl_xor_sync(0xffffffffu, st, o);
    const float mm = fmaxf(mt, m2);
    st = (mt == -INFINITY ? 0.f : st * ex2_approx((mt - mm) * c)) + (m2 == -INFINITY ? 0.f : s2 * ex2_approx((m2 - mm) * c));
    mt = mm;
  }
  if (lane == 0) {
    sh.red[warp] = mt;
    sh.red2[warp] = st;
  }
  __syncthreads();
  float M = -INFINITY, S = 0.f;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sh.red[w]);
    if (M != -INFINITY)
#pragma unroll
      for (int w = 0; w < kWarps; ++w)
        if (sh.red[w] != -INFINITY) S += sh.red2[w] * ex2_approx((sh.red[w] - M) * c);
  }
  if (threadIdx.x == 0) {
    const int R = 2 * k + 1;
    a.spart[((size_t)b * R + i) * nch + ch] = make_float2(M, S);
    sh.last = atomic_add_acq_rel(&a.sseq[4 * b], 1u) + 1u == (unsigned)a.sNA;
    if (sh.last) a.sseq[4 * b] = 0u;  // left zero for the next call
  }
  __syncthreads();
  if (sh.last) decide(sh, a, b, kb);
}

__device__ void residual_item(Shared &sh, const VerifyArgs &a, int b, int ch) {
  const int nch = a.snch, V = a.V;
  if (threadIdx.x == 0) {
    unsigned d = ld_acquire_u32(&a.sseq[4 * b + 2]);
    if (d == 0u) {
      const uint64_t t0 = global_timer_ns();
      while ((d = ld_acquire_u32(&a.sseq[4 * b + 2])) == 0u) {
        __nanosleep(256);
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          set_status(a.status, kStatusTimeout);
          break;
        }
      }
    }
    sh.dec = d;
    if (d == kDecidedReject) {
      const float4 *r4 = reinterpret_cast<const float4 *>(&a.srec[b]);
      const float4 x = __ldcg(r4);
      const int4 y = __ldcg(reinterpret_cast<const int4 *>(r4 + 1));
      sh.rec = SplitRec{x.x, x.y, x.z, x.w, y.x, y.y, 0, 0};
    }
  }
  __syncthreads();
  const unsigned dec = sh.dec;
  const float c = kLog2e / a.T;
  if (dec == kDecidedReject) {
    const SplitRec r = sh.rec;
    const Wt w{0, r.Mt, r.iZt, r.Ml, r.iZl, c};
    chunk_sub_masses(sh, w, seq_row(a, b, r.j), seq_row(a, b, a.k + 1 + r.j), V, ch,
                     a.shint ? l2_policy_evict_first() : l2_policy_evict_normal_all());
    if (threadIdx.x < kSubs) a.smass[((size_t)b * nch + ch) * kSubs + threadIdx.x] = sh.sub[threadIdx.x];
    if (threadIdx.x == 0) {
      double cm = 0.0;
      for (int s = 0; s < kSubs; ++s) cm += (double)sh.sub[s];
      a.cmass[(size_t)b * nch + ch] = cm;
    }
    __threadfence();
    __syncthreads();
  }
  if (threadIdx.x == 0) sh.last = atomic_add_acq_rel(&a.sseq[4 * b + 1], 1u) + 1u == (unsigned)a.sNB;
  __syncthreads();
  if (!sh.last) return;
  if (dec == kDecidedReject) {
    // the crossing chunk over the residual chunk masses, then its sub-chunks
    const SplitRec r = sh.rec;
    const Wt w{0, r.Mt, r.iZt, r.Ml, r.iZl, c};
    const float *trow = seq_row(a, b, r.j), *lrow = seq_row(a, b, a.k + 1 + r.j);
    const double u = (double)__ldg(&a.u_final[b]);
    if (threadIdx.x < 32) {
      const double *cmb = a.cmass + (size_t)b * nch;
      auto mass = [&](int i) { return __ldcg(&cmb[i]); };
      const double tgt = u * warp_total(mass, nch);
      double before;
      const int cx = warp_crossing(mass, nch, tgt, before);
      int f = -1;
      if (cx >= 0) {
        const float *sm = a.smass + ((size_t)b * nch + cx) * kSubs;
        for (int q = threadIdx.x; q < kSubs; q += 32) sh.sub[q] = __ldcg(&sm[q]);
        __syncwarp();
        f = warp_draw_in_chunk(sh, w, trow, lrow, V, cx, before, tgt);
      }
      if (threadIdx.x == 0) sh.chosen = f;
    }
    __syncthreads();
    int chosen = sh.chosen;
    __syncthreads();
    if (chosen < 0) {  // the residual is zero everywhere (p = q): draw from p itself
      const Wt wp{2, r.Mt, 0.f, 0.f, 0.f, c};
      chosen = draw_from_stats(sh, wp, a.spart + ((size_t)b * (2 * a.k + 1) + r.j) * nch, nch, trow, V, u);
    }
    write_outputs(a, b, r.j, chosen, r.flags);
  }
  if (threadIdx.x == 0) {
    a.sseq[4 * b + 1] = 0u;  // left zero for the next call
    a.sseq[4 * b + 2] = 0u;
    // the last sequence to finish: every ticket has been taken
    if (atomic_add_acq_rel(&a.ctl[1], 1u) + 1u == (unsigned)a.B) {
      a.ctl[0] = 0u;
      a.ctl[1] = 0u;
    }
  }
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 4) verify_split_kernel(const VerifyArgs a) {
  trace_start(kTkVerifySplit);
  __shared__ Shared sh;
  grid_dep_wait();  // the draft rows may come from the drafter
  grid_dep_launch();
  trace_dep(kTkVerifySplit);
  if (threadIdx.x == 0) sh.ticket = atomicAdd(&a.ctl[0], 1u);
  __syncthreads();
  const Item it = decode_ticket(a, sh.ticket);
  if (in_bounds(it.b >= 0 && it.b < a.B && it.local >= 0 && it.local < (it.residual ? a.sNB : a.sNA), a.status)) {
    if (it.residual)
      residual_item(sh, a, it.b, it.local);
    else
      statistics_item(sh, a, it.b, it.local);
  }
  trace_end(kTkVerifySplit);
}

// ---------------------------------------------------------------- host side

int split_chunks(int V) { return (V + kChunk - 1) / kChunk; }

bool split_shape_ok(int B, int k, int V) {
  const long long nch = split_chunks(V);
  return 2 * k + 1 <= kMaxRows && (long long)B * (2 * k + 2) * nch < (1ll << 31);
}

static size_t up256(size_t n) { return (n + 255) / 256 * 256; }

size_t split_state_bytes(int B, int k, int V) {
  const size_t nch = split_chunks(V);
  return up256((size_t)B * 16)                        // per-sequence counters and decision
         + up256((size_t)B * sizeof(SplitRec))        // rejection records
         + up256((size_t)B * (2 * k + 1) * nch * 8)   // chunk statistics
         + up256((size_t)B * nch * 8)                 // residual chunk masses
         + up256((size_t)B * nch * kSubs * 4);        // residual sub-chunk masses
}

void split_bind_state(VerifyArgs &a, void *state, int lag_items) {
  char *p = static_cast<char *>(state);
  const size_t nch = split_chunks(a.V);
  a.sseq = reinterpret_cast<unsigned *>(p);
  p += up256((size_t)a.B * 16);
  a.srec = reinterpret_cast<SplitRec *>(p);
  p += up256((size_t)a.B * sizeof(SplitRec));
  a.spart = reinterpret_cast<float2 *>(p);
  p += up256((size_t)a.B * (2 * a.k + 1) * nch * 8);
  a.cmass = reinterpret_cast<double *>(p);
  p += up256((size_t)a.B * nch * 8);
  a.smass = reinterpret_cast<float *>(p);
  a.snch = (int)nch;
  a.sNA = (2 * a.k + 1) * a.snch;
  a.sNB = a.snch;
  const int D = (lag_items + a.sNA - 1) / a.sNA;  // the residual group's lag, in sequences
  a.sD = D < 1 ? 1 : (D > a.B ? a.B : D);
}

cudaError_t launch_verify_split(const VerifyArgs &a, cudaStream_t s, bool pdl) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)((long long)a.B * (a.sNA + a.sNB)));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  note_launch();
  return cudaLaunchKernelEx(&cfg, verify_split_kernel, a);
}

MTP_TRACE_COLLECTOR(verify_split)

}  // namespace mtp
