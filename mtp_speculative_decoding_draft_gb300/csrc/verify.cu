// Verification of k drafted tokens per sequence ("The Tiny Draft Model Hidden
// Inside Qwen", section "How the draft becomes real output"; "Speculative
// Decoding and MTP: Why Guessing Is Free", sections "Speculative decoding:
// draft, then verify" and "It's exact, not approximate").
//
// One thread-block cluster of C CTAs handles one sequence at a time; CTA r owns
// the vocabulary slice [r*S, (r+1)*S) of every logit row of the sequence.  At
// most 64 sequences are in flight (persistent clusters loop over the rest).
//
// Warp roles in every CTA:
//  producer (1 warp)   streams the rows of its slices -- target k, then target /
//                      draft k-1 .. 1, then target / draft 0 -- through a ring
//                      of 16 KB shared-memory pieces with 1-D TMA bulk copies,
//                      paced by per-piece full / empty mbarriers;
//  consumers (8 warps) reduce every slice to (max, lowest argmax) -- greedy --
//                      or to the max and sum exp2((x - max) * log2e / T)
//                      (per piece: its max, then one exp pass), send the
//                      per-row partials to CTA 0 of the cluster (remote stores
//                      and a remote mbarrier arrive), and, at the first
//                      rejection r or for the bonus token, sum the sampling
//                      weights max(0, p - q) (or p) of their slices of the rows
//                      at r per 512-element sub-chunk;
//  agent (1 warp, CTA 0 only) combines the partials in rank order, takes the
//                      accept / reject decisions, picks the CTA that holds the
//                      inverse-CDF crossing and broadcasts both through remote
//                      stores and arrives.  That CTA rescans one sub-chunk in
//                      float64 and writes the outputs.
//
// No cluster barrier runs inside the loop, so the producer keeps streaming
// while a sequence is decided.  The rows of position 0 are read last with an
// L2 evict-last hint: with at most 64 sequences in flight they are still in L2
// when a rejection at position 0 re-reads them.  Every wait is a bounded
// mbarrier wait that gives up after a time limit and flags the status word.
#include "common.cuh"
#include "internal.h"

namespace mtp {

namespace {

constexpr int kSub = 512;      // sampling sub-chunk (elements)
constexpr int kPiece = 4096;   // floats per ring piece (16 KB)
constexpr int kCons = 256;     // consumer threads (warps 0..7)
constexpr int kConsWarps = kCons / 32;
constexpr int kProducerWarp = 8, kAgentWarp = 9;
constexpr int kMaxRows = 17;   // 2k+1 rows for k <= 8
constexpr int kMaxRing = 8;
constexpr int kMaxC = 16;

struct RowSlice {  // one row's slice: the 16-byte aligned body [h1, b1) of [v0, v1)
  const float *row;
  int h1, b1;
};

struct Smem {
  // CTA 0 (leader) side: the cluster's partials, per sequence parity
  float part[2][kMaxC][kMaxRows][2];  // max, sum | argmax bits
  double tot[2][kMaxC][2];            // residual mass, target mass
  uint64_t stats_bar, samp_bar;       // C arrivals per sequence
  // every CTA: the leader's broadcasts
  uint64_t dec_bar, sdec_bar;         // 1 arrival per sequence
  uint64_t full[kMaxRing], empty[kMaxRing];
  int acc_n, rej, kind;
  float Mt, Ml, iZt, iZl;
  int owner, use_p;
  double target;
  float red[2 * kConsWarps];
  float subR[2], subP[2];  // placeholders; the sub-chunk arrays follow the ring
};

__host__ __device__ constexpr size_t smem_hdr() { return (sizeof(Smem) + 127) / 128 * 128; }

__host__ __device__ inline int slice_len(int V, int C) { return ((V + C - 1) / C + 3) / 4 * 4; }

__device__ __forceinline__ void slice_bounds(size_t row_index, int V, int v0, int v1, int &h1, int &b1) {
  const size_t e0 = row_index * (size_t)V + v0;
  h1 = min(v1, v0 + (int)((4 - (e0 & 3)) & 3));
  b1 = h1 + (v1 - h1) / 4 * 4;
}

// Sampling weight of one element: residual max(0, p - q) (kind 0), target p
// (kind 1), unnormalised target weight exp2((t - Mt) c) (kind 2).
__device__ __forceinline__ float weight(int kind, float t, float l, float Mt, float Ml, float iZt, float iZl,
                                        float c) {
  const float e = exp2f((t - Mt) * c);
  if (kind == 2) return e;
  const float p = e * iZt;
  if (kind == 1) return p;
  return fmaxf(0.f, p - exp2f((l - Ml) * c) * iZl);
}

struct Layout {
  int ring;  // ring pieces
  size_t bytes;
};

__host__ __device__ inline Layout layout(int V, int C) {
  Layout L{};
  const int chunk = slice_len(V, C);
  const int nsub = (chunk + kSub - 1) / kSub + 2;
  const size_t fixed = smem_hdr() + (size_t)2 * nsub * 4 + 64;
  const size_t budget = 108 * 1024;  // two CTAs per SM
  L.ring = (int)((budget - fixed) / ((size_t)kPiece * 4));
  if (L.ring > kMaxRing) L.ring = kMaxRing;
  if (L.ring < 2) L.ring = 2;
  L.bytes = fixed + (size_t)L.ring * kPiece * 4;
  return L;
}

}  // namespace

size_t verify_smem_bytes(int B, int k, int V, int cluster) {
  (void)B;
  (void)k;
  return layout(V, cluster).bytes;
}

__global__ void __launch_bounds__(kVerifyThreads, 2) verify_kernel(VerifyArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = (int)cluster_size();
  const int rank = (int)cluster_rank();
  const int V = a.V, k = a.k;
  const bool stoch = a.mode == 1;
  const float c = kLog2e / a.T;
  const int chunk = slice_len(V, C);
  const int v0 = min(V, rank * chunk), v1 = min(V, v0 + chunk);
  const Layout L = layout(V, C);
  const int R = L.ring;
  float *ring = reinterpret_cast<float *>(smem_raw + smem_hdr());
  const int nsub = (chunk + kSub - 1) / kSub + 2;  // head, body sub-chunks, tail
  float *subR = ring + (size_t)R * kPiece;
  float *subP = subR + nsub;

  const int b_first = (int)cluster_id_x(), b_step = (int)cluster_count_x();
  const int nseq = b_first < a.B ? (a.B - 1 - b_first) / b_step + 1 : 0;
  const int nrows = stoch ? 2 * k + 1 : k + 1;

  if (tid == 0) {
    for (int s = 0; s < R; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], kConsWarps);
    }
    mbar_init(&sm.stats_bar, C);
    mbar_init(&sm.samp_bar, C);
    mbar_init(&sm.dec_bar, 1);
    mbar_init(&sm.sdec_bar, 1);
    fence_barrier_init();
  }
  // every CTA's barriers are initialised before any remote arrival
  cluster_sync();

  // Row r of the stream order: target k, (target j, draft j) for j = k-1..1,
  // then target 0 and draft 0 (greedy: target k .. target 0).
  auto row_desc = [&](int b, int r, RowSlice &rs, int &isd) {
    int pos;
    if (!stoch) {
      pos = k - r;
      isd = 0;
    } else if (r == 0) {
      pos = k;
      isd = 0;
    } else if (r < 2 * k - 1) {
      pos = k - (r + 1) / 2;
      isd = (r & 1) == 0;
    } else {
      pos = 0;
      isd = r == 2 * k;
    }
    const size_t idx = isd ? (size_t)b * k + pos : (size_t)b * (k + 1) + pos;
    rs.row = (isd ? a.draft : a.target) + idx * (size_t)V;
    slice_bounds(idx, V, v0, v1, rs.h1, rs.b1);
  };

  bool ok = true;
  if (warp == kProducerWarp) {
    // ================================================================ producer
    if (lane == 0) {
      const uint64_t pol_stream = l2_policy_evict_first();  // rows read once
      const uint64_t pol_keep = l2_policy_evict_last();     // position 0: likely re-read
      bool waited = false;
      uint32_t n = 0;
      for (int it = 0; it < nseq && ok; ++it) {
        const int b = b_first + it * b_step;
        for (int r = 0; r < nrows && ok; ++r) {
          RowSlice rs;
          int isd;
          row_desc(b, r, rs, isd);
          if (isd && !waited) {  // draft rows come from the drafter launched just before
            grid_dep_wait();
            waited = true;
          }
          const uint64_t pol = (stoch && r >= nrows - 2) ? pol_keep : pol_stream;
          for (int off = 0; off < rs.b1 - rs.h1 && ok; off += kPiece, ++n) {
            const int slot = (int)(n % R);
            ok = mbar_wait(&sm.empty[slot], ((n / R) & 1u) ^ 1u, a.status);
            if (!ok) break;
            const int cnt = min(kPiece, rs.b1 - rs.h1 - off);
            mbar_arrive_expect_tx(&sm.full[slot], (uint32_t)cnt * 4u);
            bulk_g2s_hint(ring + (size_t)slot * kPiece, rs.row + rs.h1 + off, (uint32_t)cnt * 4u, &sm.full[slot],
                          pol);
          }
        }
      }
      if (!waited) grid_dep_wait();
    }
    grid_dep_launch();
  } else if (warp == kAgentWarp) {
    // ================================================================ agent (CTA 0)
    if (rank == 0 && lane == 0) {
      grid_dep_wait();  // the decisions read the drafts
      auto trow = [&](int j) { return !stoch ? k - j : (j == k ? 0 : (j == 0 ? 2 * k - 1 : 2 * (k - j) - 1)); };
      auto drow = [&](int j) { return j == 0 ? 2 * k : 2 * (k - j); };
      for (int it = 0; it < nseq; ++it) {
        const int b = b_first + it * b_step;
        const int par = it & 1;
        // the sequence's drafts, uniforms and logits at the drafts, fetched
        // while its rows stream in
        int dtok[8];
        float td[8], ld[8], ua[8], uf = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < k) dtok[j] = __ldcg(&a.draft_tok[(size_t)b * k + j]);
        if (stoch) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (j < k) {
              const int d = dtok[j];
              const bool valid = d >= 0 && d < V;
              td[j] = valid ? __ldg(&a.target[((size_t)b * (k + 1) + j) * V + d]) : 0.f;
              ld[j] = valid ? __ldcg(&a.draft[((size_t)b * k + j) * V + d]) : 0.f;
              ua[j] = __ldg(&a.u_accept[(size_t)b * k + j]);
            }
          uf = __ldg(&a.u_final[b]);
        }
        if (ok) ok = mbar_wait_cluster(&sm.stats_bar, (uint32_t)par, a.status);
        // combine every row's partials in rank order
        float M[kMaxRows];
        double Z[kMaxRows];
        int I[kMaxRows];
        for (int r = 0; r < nrows; ++r) {
          M[r] = -INFINITY;
          Z[r] = 0.0;
          I[r] = 0x7fffffff;
          for (int q = 0; q < C; ++q) {
            if (stoch) M[r] = fmaxf(M[r], sm.part[par][q][r][0]);
            else argmax_merge(M[r], I[r], sm.part[par][q][r][0], __float_as_int(sm.part[par][q][r][1]));
          }
          if (stoch && M[r] != -INFINITY)
            for (int q = 0; q < C; ++q) {
              const float pm = sm.part[par][q][r][0];
              if (pm != -INFINITY) Z[r] += (double)sm.part[par][q][r][1] * (double)exp2f((pm - M[r]) * c);
            }
        }
        int acc_n = 0, rej = k;
        for (int j = 0; j < k; ++j) {
          const int d = dtok[j];
          bool accept = false;
          if (d < 0 || d >= V) {
            set_status(a.status, kStatusBadToken);
          } else if (!stoch) {
            if (!(M[trow(j)] > -INFINITY)) set_status(a.status, kStatusNonFinite);
            accept = I[trow(j)] == d;
          } else {
            const int tr = trow(j), dr = drow(j);
            if (M[tr] == -INFINITY || M[dr] == -INFINITY) set_status(a.status, kStatusNonFinite);
            const double p = exp2(((double)td[j] - (double)M[tr]) * (double)c) / Z[tr];
            const double q = exp2(((double)ld[j] - (double)M[dr]) * (double)c) / Z[dr];
            accept = (double)ua[j] * q < p;
          }
          if (!accept) {
            rej = j;
            break;
          }
          ++acc_n;
        }
        if (!stoch) {
          // greedy: the emitted token is the argmax of the first disagreeing row
          int *o = a.out_tok + (size_t)b * (k + 1);
          for (int q = 0; q < acc_n; ++q) o[q] = dtok[q];
          const int e = I[trow(acc_n)];
          o[acc_n] = e == 0x7fffffff ? 0 : e;
          for (int q = acc_n + 1; q <= k; ++q) o[q] = -1;
          a.accept_len[b] = acc_n + 1;
          a.num_accepted[b] = acc_n;
          for (int q = 0; q < C; ++q) mbar_arrive_remote(&sm.dec_bar, q);
          continue;
        }
        // stochastic: broadcast the sampling task
        const int tr = trow(rej);
        const int kind = rej == k ? 2 : 0;
        const float Mt = M[tr], iZt = (float)(1.0 / Z[tr]);
        const float Ml = rej < k ? M[drow(rej)] : 0.f;
        const float iZl = rej < k ? (float)(1.0 / Z[drow(rej)]) : 0.f;
        for (int q = 0; q < C; ++q) {
          Smem *rm = dsmem_ptr_mut(&sm, q);
          rm->acc_n = acc_n;
          rm->rej = rej;
          rm->kind = kind;
          rm->Mt = Mt;
          rm->Ml = Ml;
          rm->iZt = iZt;
          rm->iZl = iZl;
        }
        for (int q = 0; q < C; ++q) mbar_arrive_remote(&sm.dec_bar, q);
        // gather the per-CTA sampling masses, find the CTA holding the crossing
        if (ok) ok = mbar_wait_cluster(&sm.samp_bar, (uint32_t)par, a.status);
        double SR = 0.0, SP = 0.0;
        for (int q = 0; q < C; ++q) {
          SR += sm.tot[par][q][0];
          SP += sm.tot[par][q][1];
        }
        // weights: the residual; the target itself if the residual is
        // identically zero; the unnormalised target row k for the bonus token
        const bool use_p = kind == 2 || !(SR > 0.0);
        const double target = (double)uf * (use_p ? SP : SR);
        int owner = -1, last = -1;
        double before = 0.0, cum = 0.0;
        for (int q = 0; q < C; ++q) {
          const double m = use_p ? sm.tot[par][q][1] : sm.tot[par][q][0];
          if (m > 0.0) last = q;
          if (owner < 0 && cum + m > target) {
            owner = q;
            before = cum;
          }
          cum += m;
        }
        const int own = owner >= 0 ? owner : (last >= 0 ? last : 0);
        const double tg = owner >= 0 ? target - before : -1.0;  // -1: no crossing, the last positive
        for (int q = 0; q < C; ++q) {
          Smem *rm = dsmem_ptr_mut(&sm, q);
          rm->owner = own;
          rm->use_p = use_p;
          rm->target = tg;
        }
        for (int q = 0; q < C; ++q) mbar_arrive_remote(&sm.sdec_bar, q);
      }
    }
    grid_dep_launch();
  } else {
    // ================================================================ consumers
    uint32_t n = 0;
    const int ctid = tid;  // 0..255
    if (stoch) grid_dep_wait();  // the sampling pass reads draft rows directly
    for (int it = 0; it < nseq; ++it) {
      const int b = b_first + it * b_step;
      const int par = it & 1;
      Smem *leader = dsmem_ptr_mut(&sm, 0);
      for (int r = 0; r < nrows; ++r) {
        RowSlice rs;
        int isd;
        row_desc(b, r, rs, isd);
        float m = -INFINITY, s = 0.f;  // stochastic: running (max, sum)
        float bv = -INFINITY;          // greedy: (max, lowest argmax)
        int bi = 0x7fffffff;
        for (int off = 0; off < rs.b1 - rs.h1; off += kPiece, ++n) {
          const int slot = (int)(n % R);
          if (ok) ok = mbar_wait(&sm.full[slot], (n / R) & 1u, a.status);
          const float4 *b4 = reinterpret_cast<const float4 *>(ring + (size_t)slot * kPiece);
          const int nf = min(kPiece, rs.b1 - rs.h1 - off) / 4;
          const int vbase = rs.h1 + off;
          float pm = -INFINITY;
          for (int f = ctid; f < nf; f += kCons) {
            const float4 x = b4[f];
            const float m4 = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
            if (!stoch && m4 > bv) {
              const int v = vbase + 4 * f;
              bi = x.x == m4 ? v : (x.y == m4 ? v + 1 : (x.z == m4 ? v + 2 : v + 3));
              bv = m4;
            }
            pm = fmaxf(pm, m4);
          }
          if (stoch && pm != -INFINITY) {
            const float mn = fmaxf(m, pm);
            float acc = m == -INFINITY ? 0.f : s * exp2f((m - mn) * c);
            for (int f = ctid; f < nf; f += kCons) {
              const float4 x = b4[f];
              acc += exp2f((x.x - mn) * c) + exp2f((x.y - mn) * c);
              acc += exp2f((x.z - mn) * c) + exp2f((x.w - mn) * c);
            }
            m = mn;
            s = acc;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&sm.empty[slot]);  // this warp is done with the piece
        }
        if (ctid < 4) {  // unaligned head / tail elements of the slice
          for (int q = 0; q < 2; ++q) {
            const int v = q == 0 ? v0 + ctid : rs.b1 + ctid;
            if (q == 0 ? v < rs.h1 : v < v1) {
              if (isd) grid_dep_wait();
              const float x = __ldcg(rs.row + v);
              if (!stoch) {
                argmax_merge(bv, bi, x, v);
              } else if (x != -INFINITY) {
                if (x > m) {
                  s = (m == -INFINITY ? 0.f : s * exp2f((m - x) * c)) + 1.f;
                  m = x;
                } else {
                  s += exp2f((x - m) * c);
                }
              }
            }
          }
        }
        // reduction of this row's slice over the consumer warps
        if (!stoch) {
          warp_argmax(bv, bi);
          if (lane == 0) {
            sm.red[warp] = bv;
            sm.red[kConsWarps + warp] = __int_as_float(bi);
          }
        } else {
          warp_lse(m, s, c);
          if (lane == 0) {
            sm.red[warp] = m;
            sm.red[kConsWarps + warp] = s;
          }
        }
        named_sync(1, kCons);
        if (ctid == 0) {
          float M = -INFINITY, Sx = 0.f;
          int I = 0x7fffffff;
          for (int w = 0; w < kConsWarps; ++w) {
            if (stoch) lse_merge(M, Sx, sm.red[w], sm.red[kConsWarps + w], c);
            else argmax_merge(M, I, sm.red[w], __float_as_int(sm.red[kConsWarps + w]));
          }
          leader->part[par][rank][r][0] = M;
          leader->part[par][rank][r][1] = stoch ? Sx : __int_as_float(I);
        }
        named_sync(1, kCons);
      }
      if (ctid == 0) mbar_arrive_remote(&sm.stats_bar, 0);
      // the leader's decision (greedy: it only paces the partial buffers); the
      // bounded wait starts once the drafter has finished
      if (it == 0 && !stoch) grid_dep_wait();
      if (ok) ok = mbar_wait_cluster(&sm.dec_bar, (uint32_t)par, a.status);
      if (!stoch) continue;

      // ---------------- sampling at the rejected position / the bonus row
      const int kind = sm.kind, pos = sm.rej, acc_n = sm.acc_n;
      const float Mt = sm.Mt, Ml = sm.Ml, iZt = sm.iZt, iZl = sm.iZl;
      RowSlice rt, rl;
      {
        const size_t ti = (size_t)b * (k + 1) + pos;
        rt.row = a.target + ti * (size_t)V;
        slice_bounds(ti, V, v0, v1, rt.h1, rt.b1);
        if (kind == 0) {
          const size_t li = (size_t)b * k + pos;
          rl.row = a.draft + li * (size_t)V;
          slice_bounds(li, V, v0, v1, rl.h1, rl.b1);
        } else {
          rl = rt;
        }
      }
      auto sub_range = [&](int sb, int &e0, int &e1) {  // 0: head, nsub-1: tail, else body
        if (sb == 0) {
          e0 = v0;
          e1 = rt.h1;
        } else if (sb == nsub - 1) {
          e0 = rt.b1;
          e1 = v1;
        } else {
          e0 = min(rt.b1, rt.h1 + (sb - 1) * kSub);
          e1 = min(rt.b1, e0 + kSub);
        }
      };
      const bool vec = kind == 2 || rt.h1 == rl.h1;
      for (int sb = warp; sb < nsub; sb += kConsWarps) {
        int e0, e1;
        sub_range(sb, e0, e1);
        float sr = 0.f, sp = 0.f;
        if (sb > 0 && sb < nsub - 1 && vec && e1 - e0 == kSub) {
          float4 tv[kSub / 128], lv[kSub / 128];
#pragma unroll
          for (int i = 0; i < kSub / 128; ++i) {
            tv[i] = __ldcg(reinterpret_cast<const float4 *>(rt.row + e0) + lane + 32 * i);
            if (kind == 0) lv[i] = __ldcg(reinterpret_cast<const float4 *>(rl.row + e0) + lane + 32 * i);
          }
#pragma unroll
          for (int i = 0; i < kSub / 128; ++i) {
            const float t4[4] = {tv[i].x, tv[i].y, tv[i].z, tv[i].w};
            if (kind == 2) {
#pragma unroll
              for (int q = 0; q < 4; ++q) sp += weight(2, t4[q], 0.f, Mt, Ml, iZt, iZl, c);
            } else {
              const float l4[4] = {lv[i].x, lv[i].y, lv[i].z, lv[i].w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                sr += weight(0, t4[q], l4[q], Mt, Ml, iZt, iZl, c);
                sp += weight(1, t4[q], l4[q], Mt, Ml, iZt, iZl, c);
              }
            }
          }
        } else {
          for (int v = e0 + lane; v < e1; v += 32) {
            const float t = __ldcg(rt.row + v);
            if (kind == 2) {
              sp += weight(2, t, 0.f, Mt, Ml, iZt, iZl, c);
            } else {
              const float l = __ldcg(rl.row + v);
              sr += weight(0, t, l, Mt, Ml, iZt, iZl, c);
              sp += weight(1, t, l, Mt, Ml, iZt, iZl, c);
            }
          }
        }
        sr = warp_sum(sr);
        sp = warp_sum(sp);
        if (lane == 0) {
          subR[sb] = sr;
          subP[sb] = sp;
        }
      }
      named_sync(1, kCons);
      if (ctid == 0) {
        double tR = 0.0, tP = 0.0;
        for (int sb = 0; sb < nsub; ++sb) {
          tR += (double)subR[sb];
          tP += (double)subP[sb];
        }
        leader->tot[par][rank][0] = tR;
        leader->tot[par][rank][1] = tP;
        mbar_arrive_remote(&sm.samp_bar, 0);
      }
      if (ok) ok = mbar_wait_cluster(&sm.sdec_bar, (uint32_t)par, a.status);
      if (rank == sm.owner && warp == 0) {
        const bool use_p = sm.use_p;
        const double tgt = sm.target;
        const float *wsub = use_p ? subP : subR;
        const int wk = kind == 2 ? 2 : (use_p ? 1 : 0);
        auto elem = [&](int v) -> float {
          return weight(wk, __ldcg(rt.row + v), wk == 2 ? 0.f : __ldcg(rl.row + v), Mt, Ml, iZt, iZl, c);
        };
        int sstar = -1, slast = -1;
        double before = 0.0;
        if (lane == 0) {
          double cum = 0.0;
          for (int sb = 0; sb < nsub; ++sb) {
            const double m = (double)wsub[sb];
            if (m > 0.0) slast = sb;
            if (tgt >= 0.0 && sstar < 0 && cum + m > tgt) {
              sstar = sb;
              before = cum;
            }
            cum += m;
          }
        }
        sstar = __shfl_sync(0xffffffffu, sstar, 0);
        slast = __shfl_sync(0xffffffffu, slast, 0);
        before = __shfl_sync(0xffffffffu, before, 0);
        const int sb = sstar >= 0 ? sstar : slast;
        int chosen = -1;
        if (sb >= 0) {
          int e0, e1;
          sub_range(sb, e0, e1);
          // each lane a contiguous run of 16 elements (loaded first), float64 prefix sums
          constexpr int RUN = kSub / 32;
          const int a0 = min(e1, e0 + lane * RUN), a1 = min(e1, a0 + RUN);
          float wv[RUN];
#pragma unroll
          for (int i = 0; i < RUN; ++i) wv[i] = a0 + i < a1 ? elem(a0 + i) : 0.f;
          double ls = 0.0;
          int lastpos = -1;
#pragma unroll
          for (int i = 0; i < RUN; ++i) {
            ls += (double)wv[i];
            if (wv[i] > 0.f) lastpos = a0 + i;
          }
          double incl = ls;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const double t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
          }
          int found = 0x7fffffff;
          if (sstar >= 0 && before + incl > tgt) {
            double run = before + (incl - ls);
#pragma unroll
            for (int i = 0; i < RUN; ++i) {
              run += (double)wv[i];
              if (found == 0x7fffffff && run > tgt && a0 + i < a1) found = a0 + i;
            }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            found = min(found, __shfl_xor_sync(0xffffffffu, found, o));
            lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, o));
          }
          chosen = found != 0x7fffffff ? found : lastpos;
        }
        if (lane == 0) {
          if (chosen < 0) {
            set_status(a.status, kStatusNonFinite);
            chosen = 0;
          }
          int *o = a.out_tok + (size_t)b * (k + 1);
          for (int q = 0; q < acc_n; ++q) o[q] = __ldcg(&a.draft_tok[(size_t)b * k + q]);
          o[acc_n] = chosen;
          for (int q = acc_n + 1; q <= k; ++q) o[q] = -1;
          a.accept_len[b] = acc_n + 1;
          a.num_accepted[b] = acc_n;
        }
      }
      named_sync(1, kCons);  // the sub-chunk masses may be overwritten by the next sequence
    }
    grid_dep_wait();
    grid_dep_launch();
  }
  // no CTA may leave while another can still read or arrive on its shared memory
  cluster_sync();
}

// Clusters: at most 64 sequences in flight (their position-0 rows then fit in
// L2), about 256 CTAs in all, at least 4 CTAs per sequence.
static int verify_clusters(int B) { return B < 64 ? B : 64; }

int verify_cluster_size(int B, int num_sms, int max_cluster) {
  (void)num_sms;
  const int n = verify_clusters(B);
  int C = 4;
  while (C < max_cluster && C * 2 * n <= 256) C *= 2;
  return C;
}

cudaError_t verify_set_attributes(int max_cluster) {
  cudaError_t e = cudaFuncSetAttribute(verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 112 * 1024);
  if (e != cudaSuccess) return e;
  if (max_cluster > 8) {
    e = cudaFuncSetAttribute(verify_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int verify_max_active_clusters(int cluster) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(cluster);
  cfg.blockDim = dim3(kVerifyThreads);
  cfg.dynamicSmemBytes = verify_smem_bytes(1, 8, 151936, cluster);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, verify_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_verify(const VerifyArgs &a, int cluster, cudaStream_t s, bool pdl) {
  const int nclusters = verify_clusters(a.B);  // persistent: each loops over B / 64 sequences
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(nclusters * cluster);
  cfg.blockDim = dim3(kVerifyThreads);
  cfg.dynamicSmemBytes = layout(a.V, cluster).bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  note_launch();
  return cudaLaunchKernelEx(&cfg, verify_kernel, a);
}

}  // namespace mtp
