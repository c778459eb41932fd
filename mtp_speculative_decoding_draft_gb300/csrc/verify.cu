// Verification of k drafted tokens per sequence ("The Tiny Draft Model Hidden
// Inside Qwen", section "How the draft becomes real output"; "Speculative
// Decoding and MTP: Why Guessing Is Free", sections "Speculative decoding:
// draft, then verify" and "It's exact, not approximate").
//
// One thread-block cluster of C CTAs handles one sequence at a time; CTA r of
// the cluster owns the vocabulary slice [r*V/C, (r+1)*V/C) of every logit row of
// that sequence.
//
//  pass 1  every row of the sequence (k+1 target rows, plus k draft rows when
//          stochastic) streams through a ring of 16 KB shared-memory stages
//          filled by 1-D TMA bulk copies; each CTA reduces its slice of each row
//          to (max, sum of exp2((x-max)*log2e/T)) or to (max, lowest argmax).
//          Rows are read in descending position order so the rows a rejection
//          most likely needs again (position 0) are the most recently read and
//          still in L2.
//  combine the per-slice partials are exchanged through distributed shared
//          memory after a cluster barrier; every CTA combines them in rank order
//          and takes the same accept / reject decisions.
//  pass 2  (stochastic only) the rows of the rejected position (or the bonus
//          row) are read again, from L2, in 512-element sub-chunks whose masses
//          are kept; after a second exchange the CTA holding the inverse-CDF
//          crossing rescans one sub-chunk in float64 and writes the outputs.
//
// The cluster barriers are hardware barriers; the only software wait is on the
// TMA mbarriers, which gives up after a time limit and flags the status word.
#include "common.cuh"
#include "internal.h"

namespace mtp {

namespace {

constexpr int kMaxRows = 17;     // 2*8 + 1 rows for k <= 8
constexpr int kSub = 512;        // pass-2 sub-chunk (elements)
constexpr int kWarps = kVerifyThreads / 32;

struct RowDesc {
  const float *ptr;  // row start
  int h1, b1;        // TMA body [h1, b1) inside the slice [v0, v1); head/tail by plain loads
  int p0, np;        // first piece (phase-local) and piece count
  int is_draft;
};

struct Smem {
  RowDesc rows[kMaxRows];
  float rowpart[2][kMaxRows][4];  // per-slice (max, sum | argmax) of each row, double-buffered
  float rowM[kMaxRows];
  double rowZ[kMaxRows];
  int rowI[kMaxRows];
  double tot[2][2];               // this slice's pass-2 masses (residual, target), double-buffered
  float red[3 * kWarps];
  int nrows, npieces;
  int a, rej, owner_rank, use_p;
  double target;
  int out_final;
};

__host__ __device__ constexpr size_t smem_ring_offset() { return (sizeof(Smem) + 127) / 128 * 128; }

// Pass-2 weight of one element: residual max(0, p - q), target p, or the
// unnormalised bonus weight.
__device__ __forceinline__ float p2_weight(int kind, float t, float l, float Mt, float Ml, float iZt, float iZl,
                                           float c) {
  const float p = exp2f((t - Mt) * c) * iZt;
  if (kind == 1) return p;
  return fmaxf(0.f, p - exp2f((l - Ml) * c) * iZl);
}

}  // namespace

size_t verify_smem_bytes(int B, int k, int V, int cluster) {
  (void)B;
  (void)k;
  const int slice = ((V + cluster - 1) / cluster + 3) / 4 * 4;
  const int nsub = (slice + kSub - 1) / kSub;
  return smem_ring_offset() + (size_t)kVerifyStages * (kVerifyPiece * 4 + 8) + (size_t)2 * 2 * nsub * 4 + 64;
}

__global__ void __launch_bounds__(kVerifyThreads) verify_kernel(VerifyArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
  float *ring = reinterpret_cast<float *>(smem_raw + smem_ring_offset());
  uint64_t *bars = reinterpret_cast<uint64_t *>(ring + (size_t)kVerifyStages * kVerifyPiece);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = (int)cluster_size();
  const int rank = (int)cluster_rank();
  const int V = a.V, k = a.k;
  const int chunk = ((V + C - 1) / C + 3) / 4 * 4;
  const int v0 = min(V, rank * chunk), v1 = min(V, v0 + chunk);
  const int nsub = (chunk + kSub - 1) / kSub;
  float *subs = reinterpret_cast<float *>(bars + kVerifyStages);  // [2 buf][2 kinds][nsub]
  const bool stoch = a.mode == 1;
  const float c = kLog2e / a.T;

  if (tid == 0) {
    for (int s = 0; s < kVerifyStages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  const uint64_t pol = l2_policy_evict_first();
  bool waited_dep = false;     // thread 0: has passed griddepcontrol.wait
  bool ok = true;
  uint32_t gpiece = 0;          // pieces consumed over the kernel's life (ring phase)
  int it = 0;

  for (int b = (int)cluster_id_x(); b < a.B; b += (int)cluster_count_x(), ++it) {
    const int buf = it & 1;
    // ---------------- schedule of pass 1 for sequence b
    if (tid == 0) {
      int nr = 0, np = 0;
      auto add = [&](const float *base, size_t row_index, int is_draft) {
        RowDesc &r = sm.rows[nr++];
        r.ptr = base + row_index * (size_t)V;
        const size_t e0 = row_index * (size_t)V + v0;
        int h1 = v0 + (int)((4 - (e0 & 3)) & 3);
        h1 = min(h1, v1);
        const int b1 = h1 + (v1 - h1) / 4 * 4;
        r.h1 = h1;
        r.b1 = b1;
        r.p0 = np;
        r.np = (b1 - h1 + kVerifyPiece - 1) / kVerifyPiece;
        r.is_draft = is_draft;
        np += r.np;
      };
      for (int j = k; j >= 1; --j) add(a.target, (size_t)b * (k + 1) + j, 0);
      if (stoch)
        for (int j = k - 1; j >= 1; --j) add(a.draft, (size_t)b * k + j, 1);
      add(a.target, (size_t)b * (k + 1), 0);
      if (stoch) add(a.draft, (size_t)b * k, 1);
      sm.nrows = nr;
      sm.npieces = np;
    }
    __syncthreads();
    const int nrows = sm.nrows, npieces = sm.npieces;

    // piece n of this sequence -> (row, element range)
    auto locate = [&](int n, int &row, int &e0, int &cnt) {
      row = 0;
      while (row + 1 < nrows && sm.rows[row + 1].p0 <= n) ++row;
      const RowDesc &r = sm.rows[row];
      e0 = r.h1 + (n - r.p0) * kVerifyPiece;
      cnt = min(kVerifyPiece, r.b1 - e0);
    };
    auto issue = [&](int n) {  // thread 0
      int row, e0, cnt;
      locate(n, row, e0, cnt);
      if (sm.rows[row].is_draft && !waited_dep) {
        grid_dep_wait();
        waited_dep = true;
      }
      const int stage = (int)((gpiece + n) % kVerifyStages);
      mbar_arrive_expect_tx(&bars[stage], (uint32_t)cnt * 4u);
      bulk_g2s_hint(ring + (size_t)stage * kVerifyPiece, sm.rows[row].ptr + e0, (uint32_t)cnt * 4u, &bars[stage], pol);
    };
    if (tid == 0 && ok)
      for (int n = 0; n < min(kVerifyStages, npieces); ++n) issue(n);

    // ---------------- pass 1
    int n = 0;
    for (int row = 0; row < nrows; ++row) {
      const RowDesc &rd = sm.rows[row];
      float m = -INFINITY, s = 0.f;  // stochastic: online (max, sum)
      float bv = -INFINITY;          // greedy: (max, lowest index)
      int bi = 0x7fffffff;
      auto consume = [&](float x, int v) {
        if (stoch) {
          if (x > m) {
            s = (m == -INFINITY ? 0.f : s * exp2f((m - x) * c)) + 1.f;
            m = x;
          } else if (x != -INFINITY) {
            s += exp2f((x - m) * c);
          }
        } else {
          argmax_merge(bv, bi, x, v);
        }
      };
      // draft rows come from the drafter launched just before this kernel
      if (rd.is_draft) grid_dep_wait();
      // unaligned head / tail of the slice
      if (tid < 4) {
        const int v = v0 + tid;
        if (v < rd.h1) consume(__ldcg(rd.ptr + v), v);
        const int vt = rd.b1 + tid;
        if (vt < v1) consume(__ldcg(rd.ptr + vt), vt);
      }
      for (int pc = 0; pc < rd.np; ++pc, ++n) {
        const int stage = (int)((gpiece + n) % kVerifyStages);
        const uint32_t parity = (uint32_t)((gpiece + n) / kVerifyStages) & 1u;
        if (ok) ok = mbar_wait(&bars[stage], parity, a.status);
        const int e0 = rd.h1 + pc * kVerifyPiece;
        const int cnt = min(kVerifyPiece, rd.b1 - e0);
        const float4 *buf = reinterpret_cast<const float4 *>(ring + (size_t)stage * kVerifyPiece);
        if (stoch) {
          float4 x[kVerifyPiece / 4 / kVerifyThreads];
          float lm = -INFINITY;
#pragma unroll
          for (int i = 0; i < kVerifyPiece / 4 / kVerifyThreads; ++i) {
            const int f = tid + i * kVerifyThreads;
            x[i] = f * 4 < cnt ? buf[f] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            lm = fmaxf(lm, fmaxf(fmaxf(x[i].x, x[i].y), fmaxf(x[i].z, x[i].w)));
          }
          if (lm != -INFINITY) {
            const float mn = fmaxf(m, lm);
            float acc = m == -INFINITY ? 0.f : s * exp2f((m - mn) * c);
#pragma unroll
            for (int i = 0; i < kVerifyPiece / 4 / kVerifyThreads; ++i) {
              acc += exp2f((x[i].x - mn) * c) + exp2f((x[i].y - mn) * c);
              acc += exp2f((x[i].z - mn) * c) + exp2f((x[i].w - mn) * c);
            }
            m = mn;
            s = acc;
          }
        } else {
#pragma unroll
          for (int i = 0; i < kVerifyPiece / 4 / kVerifyThreads; ++i) {
            const int f = tid + i * kVerifyThreads;
            if (f * 4 < cnt) {
              const float4 x = buf[f];
              const int v = e0 + f * 4;
              argmax_merge(bv, bi, x.x, v);
              argmax_merge(bv, bi, x.y, v + 1);
              argmax_merge(bv, bi, x.z, v + 2);
              argmax_merge(bv, bi, x.w, v + 3);
            }
          }
        }
        ok = __syncthreads_and(ok);  // every thread is done with this stage
        if (tid == 0 && ok && n + kVerifyStages < npieces) {
          fence_proxy_async_smem();
          issue(n + kVerifyStages);
        }
      }
      // row reduction over the CTA
      if (stoch) {
        warp_lse(m, s, c);
        if (lane == 0) {
          sm.red[warp] = m;
          sm.red[kWarps + warp] = s;
        }
      } else {
        warp_argmax(bv, bi);
        if (lane == 0) {
          sm.red[warp] = bv;
          sm.red[kWarps + warp] = __int_as_float(bi);
        }
      }
      __syncthreads();
      if (tid == 0) {
        float M = -INFINITY, Sx = 0.f;
        int I = 0x7fffffff;
        for (int w = 0; w < kWarps; ++w) {
          if (stoch) lse_merge(M, Sx, sm.red[w], sm.red[kWarps + w], c);
          else argmax_merge(M, I, sm.red[w], __float_as_int(sm.red[kWarps + w]));
        }
        sm.rowpart[buf][row][0] = M;
        sm.rowpart[buf][row][1] = Sx;
        sm.rowpart[buf][row][2] = __int_as_float(I);
      }
      __syncthreads();
    }
    gpiece += (uint32_t)npieces;

    // the decision needs the drafts: from here on, wait for the drafter
    grid_dep_wait();
    grid_dep_launch();

    // ---------------- combine across the cluster (rank order)
    cluster_sync();
    if (tid < nrows) {
      float pm[16], ps[16];
      int pi[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        if (r < C) {
          const float *src = dsmem_ptr(&sm.rowpart[buf][tid][0], r);
          pm[r] = src[0];
          ps[r] = src[1];
          pi[r] = __float_as_int(src[2]);
        }
      }
      float M = -INFINITY;
      int I = 0x7fffffff;
      double Z = 0.0;
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        if (r < C) {
          if (stoch) M = fmaxf(M, pm[r]);
          else argmax_merge(M, I, pm[r], pi[r]);
        }
      }
      if (stoch && M != -INFINITY) {
#pragma unroll
        for (int r = 0; r < 16; ++r)
          if (r < C && pm[r] != -INFINITY) Z += (double)ps[r] * (double)exp2f((pm[r] - M) * c);
      }
      sm.rowM[tid] = M;
      sm.rowZ[tid] = Z;
      sm.rowI[tid] = I;
    }
    __syncthreads();

    // ---------------- decisions (identical in every CTA of the cluster)
    // Row indices in the pass-1 order: target j >= 1 at k - j; draft j >= 1 at
    // k + (k - 1 - j) (stochastic); target 0 and draft 0 last.
    auto trow = [&](int j) { return j >= 1 ? k - j : (stoch ? 2 * k - 1 : k); };
    auto drow = [&](int j) { return j >= 1 ? k + (k - 1 - j) : 2 * k; };
    if (tid == 0) {
      int acc_n = 0, rej = k;
      for (int j = 0; j < k; ++j) {
        const int d = __ldcg(&a.draft_tok[(size_t)b * k + j]);
        bool accept;
        if (d < 0 || d >= V) {
          set_status(a.status, kStatusBadToken);
          accept = false;
        } else if (!stoch) {
          const int tr = trow(j);
          if (sm.rowM[tr] != sm.rowM[tr] || sm.rowM[tr] == -INFINITY) set_status(a.status, kStatusNonFinite);
          accept = sm.rowI[tr] == d;
        } else {
          const int tr = trow(j), dr = drow(j);
          const float td = __ldg(&a.target[((size_t)b * (k + 1) + j) * V + d]);
          const float ld = __ldcg(&a.draft[((size_t)b * k + j) * V + d]);
          if (sm.rowM[tr] == -INFINITY || sm.rowM[dr] == -INFINITY) set_status(a.status, kStatusNonFinite);
          const double p = exp2(((double)td - (double)sm.rowM[tr]) * (double)c) / sm.rowZ[tr];
          const double q = exp2(((double)ld - (double)sm.rowM[dr]) * (double)c) / sm.rowZ[dr];
          accept = (double)__ldg(&a.u_accept[(size_t)b * k + j]) * q < p;
        }
        if (!accept) {
          rej = j;
          break;
        }
        ++acc_n;
      }
      sm.a = acc_n;
      sm.rej = rej;
      if (!stoch) sm.out_final = sm.rowI[trow(acc_n)];
    }
    __syncthreads();
    const int acc_n = sm.a, rej = sm.rej;

    if (!stoch) {
      if (rank == 0 && tid == 0) {
        int *o = a.out_tok + (size_t)b * (k + 1);
        for (int j = 0; j < acc_n; ++j) o[j] = __ldcg(&a.draft_tok[(size_t)b * k + j]);
        o[acc_n] = sm.out_final;
        for (int j = acc_n + 1; j <= k; ++j) o[j] = -1;
        a.accept_len[b] = acc_n + 1;
        a.num_accepted[b] = acc_n;
      }
      continue;
    }

    // ---------------- pass 2: masses of the sampling distribution per sub-chunk
    const bool bonus = rej == k;
    const int pos = bonus ? k : rej;
    const float Mt = sm.rowM[trow(pos)];
    const float iZt = (float)(1.0 / sm.rowZ[trow(pos)]);
    const float Ml = bonus ? 0.f : sm.rowM[drow(pos)];
    const float iZl = bonus ? 0.f : (float)(1.0 / sm.rowZ[drow(pos)]);
    const float *tr_ptr = a.target + ((size_t)b * (k + 1) + pos) * V;
    const float *dr_ptr = bonus ? nullptr : a.draft + ((size_t)b * k + pos) * V;
    float *subR = subs + (size_t)buf * 2 * nsub;
    float *subP = subR + nsub;
    // rows whose every element is 16-byte aligned in this slice take float4
    // loads, 4 per lane and row in flight; others take scalar loads
    const bool vec = ((((size_t)b * (k + 1) + pos) * (size_t)V) & 3) == 0 &&
                     (bonus || ((((size_t)b * k + pos) * (size_t)V) & 3) == 0);
    for (int sb = warp; sb < nsub; sb += kWarps) {
      const int e0 = v0 + sb * kSub, e1 = min(v1, e0 + kSub);
      float sr = 0.f, sp = 0.f;
      if (vec && e1 - e0 == kSub) {
        float4 tv[kSub / 128], lv[kSub / 128];
#pragma unroll
        for (int i = 0; i < kSub / 128; ++i) {
          tv[i] = __ldg(reinterpret_cast<const float4 *>(tr_ptr + e0) + lane + 32 * i);
          if (!bonus) lv[i] = __ldcg(reinterpret_cast<const float4 *>(dr_ptr + e0) + lane + 32 * i);
        }
#pragma unroll
        for (int i = 0; i < kSub / 128; ++i) {
          const float t4[4] = {tv[i].x, tv[i].y, tv[i].z, tv[i].w};
          if (bonus) {
#pragma unroll
            for (int q = 0; q < 4; ++q) sp += exp2f((t4[q] - Mt) * c);
          } else {
            const float l4[4] = {lv[i].x, lv[i].y, lv[i].z, lv[i].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              sr += p2_weight(0, t4[q], l4[q], Mt, Ml, iZt, iZl, c);
              sp += p2_weight(1, t4[q], l4[q], Mt, Ml, iZt, iZl, c);
            }
          }
        }
      } else {
        for (int v = e0 + lane; v < e1; v += 32) {
          const float t = __ldg(tr_ptr + v);
          if (bonus) {
            sp += exp2f((t - Mt) * c);
          } else {
            const float l = __ldcg(dr_ptr + v);
            sr += p2_weight(0, t, l, Mt, Ml, iZt, iZl, c);
            sp += p2_weight(1, t, l, Mt, Ml, iZt, iZl, c);
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
    __syncthreads();
    if (tid == 0) {
      double tR = 0.0, tP = 0.0;
      for (int sb = 0; sb < nsub; ++sb) {
        tR += (double)subR[sb];
        tP += (double)subP[sb];
      }
      sm.tot[buf][0] = tR;
      sm.tot[buf][1] = tP;
    }
    cluster_sync();
    if (tid == 0) {
      double tr[16], tp[16];
      double SR = 0.0, SP = 0.0;
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        if (r < C) {
          const double *src = dsmem_ptr(&sm.tot[buf][0], r);
          tr[r] = src[0];
          tp[r] = src[1];
        }
      }
      for (int r = 0; r < C; ++r) {
        SR += tr[r];
        SP += tp[r];
      }
      // weights: the residual; the target itself if the residual is identically
      // zero; the unnormalised target row k for the bonus token
      const bool use_p = bonus || !(SR > 0.0);
      const double S = use_p ? SP : SR;
      const double target = (double)__ldg(&a.u_final[b]) * S;
      int owner = -1, last = -1;
      double before = 0.0, cum = 0.0;
      for (int r = 0; r < C; ++r) {
        const double m = use_p ? tp[r] : tr[r];
        if (m > 0.0) last = r;
        if (owner < 0 && cum + m > target) {
          owner = r;
          before = cum;
        }
        cum += m;
      }
      sm.use_p = use_p;
      if (owner >= 0) {
        sm.owner_rank = owner;
        sm.target = target - before;  // offset inside the owner's slice
      } else {
        sm.owner_rank = last >= 0 ? last : 0;
        sm.target = -1.0;             // no crossing: the last positive element
      }
    }
    __syncthreads();
    if (rank == sm.owner_rank && warp == 0) {
      const bool use_p = sm.use_p;
      const double tgt = sm.target;
      const float *wsub = use_p ? subP : subR;
      const int kind = bonus ? 2 : (use_p ? 1 : 0);
      auto weight = [&](int v) -> float {
        const float t = __ldg(tr_ptr + v);
        if (kind == 2) return exp2f((t - Mt) * c);
        return p2_weight(kind, t, __ldcg(dr_ptr + v), Mt, Ml, iZt, iZl, c);
      };
      // sub-chunk holding the crossing (lane 0 walks the masses in order)
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
        // rescan one sub-chunk: each lane a contiguous run of 16 elements,
        // float64 running sums in index order
        const int e0 = v0 + sb * kSub, e1 = min(v1, e0 + kSub);
        const int a0 = e0 + lane * (kSub / 32), a1 = min(e1, a0 + kSub / 32);
        double ls = 0.0;
        int lastpos = -1;
        for (int v = a0; v < a1; ++v) {
          const float w = weight(v);
          ls += (double)w;
          if (w > 0.f) lastpos = v;
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
          for (int v = a0; v < a1; ++v) {
            run += (double)weight(v);
            if (run > tgt) {
              found = v;
              break;
            }
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
        for (int j = 0; j < acc_n; ++j) o[j] = __ldcg(&a.draft_tok[(size_t)b * k + j]);
        o[acc_n] = chosen;
        for (int j = acc_n + 1; j <= k; ++j) o[j] = -1;
        a.accept_len[b] = acc_n + 1;
        a.num_accepted[b] = acc_n;
      }
    }
    __syncthreads();
  }
  // no CTA may leave while another can still read its shared memory
  cluster_sync();
  grid_dep_launch();
}

int verify_cluster_size(int B, int num_sms, int max_cluster) {
  int target = 2 * num_sms;
  int C = 1;
  while (C * 2 <= max_cluster && (long long)B * C * 2 <= target) C *= 2;
  return C;
}

static int g_max_cluster_attr = 0;

cudaError_t verify_set_attributes(int max_cluster) {
  cudaError_t e = cudaFuncSetAttribute(verify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 120 * 1024);
  if (e != cudaSuccess) return e;
  if (max_cluster > 8) {
    e = cudaFuncSetAttribute(verify_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  g_max_cluster_attr = max_cluster;
  return cudaSuccess;
}

int verify_max_active_clusters(int cluster) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(cluster);
  cfg.blockDim = dim3(kVerifyThreads);
  cfg.dynamicSmemBytes = verify_smem_bytes(1, 8, 256000, cluster);
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
  cudaLaunchConfig_t cfg{};
  const int nclusters = a.B;  // one cluster per sequence
  cfg.gridDim = dim3(nclusters * cluster);
  cfg.blockDim = dim3(kVerifyThreads);
  cfg.dynamicSmemBytes = verify_smem_bytes(a.B, a.k, a.V, cluster);
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
