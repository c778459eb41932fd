// Verification from the target's hidden states ("The Tiny Draft Model Hidden
// Inside Qwen", section "How the draft becomes real output": the target runs
// once over all candidate positions and its own vocabulary head gives its
// distribution at every one of them).  Instead of target logits [B, k+1, V]
// the call receives what the target's head consumes at each position, its
// final hidden state h (bf16, [B (k+1), d]), and the head E [V, d]:
//
//   t[r, v] = sum_i E[v, i] h[r, i]      (bf16 operands, fp32 accumulation)
//
// fv_gemm_kernel: tcgen05 GEMM with the hidden rows on the MMA's M side (128
//   rows a tile, up to two tiles a unit) and 256-row tiles of E on its N side,
//   the accumulators in TMEM.  Each epilogue thread owns one hidden row and
//   reduces its 256 logits of the unit on its own -- greedy: (max, lowest
//   argmax); stochastic: (max, sum of exp2((t - max) log2e / T)) -- into one
//   partial per (row, vocabulary tile).
//   Greedy writes no logits at all.  Stochastic also stores the rows' fp32
//   logits: the residual draw needs every element of the first rejecting row
//   once the target's normaliser is known, and reading that row back is far
//   cheaper than streaming E a second time to recompute it.
// fv_draft_stats_kernel (stochastic, beside the GEMM): the draft rows'
//   per-tile (max, sum of exp2) in the same tiling, every draft logit read
//   once; its warps claim tiles from a counter, so that however many of its
//   CTAs find room beside the GEMM's, those take all the tiles.
// fv_finish_kernel: one CTA per sequence combines the partials of its rows in
//   vocabulary-tile order and takes the decisions of spec_verify (the same
//   rule): greedy longest prefix and the argmax; stochastic u q(d) < p(d) at
//   every position at once, the first rejection as the position-by-position
//   rule finds it.
// fv_residual_kernel (stochastic): the inverse-CDF draw at u_final -- over
//   max(0, p - q) of the first rejecting pair (over p if that is identically
//   zero), one CTA per 16384 logits of the pair, or over p of row k when every
//   draft is accepted, whose tile masses follow from the partials so that only
//   the crossing tile is read again.
#include <cuda.h>
#include <stdlib.h>

#include "common.cuh"
#include "verify_rule.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace mtp {

namespace {

constexpr int kFvThreads = 192;   // warp 0 TMA, warp 1 MMA and TMEM, warps 2-5 read TMEM back
constexpr int kMRows = 128;       // hidden rows per MMA tile (M)
constexpr int kVt = 256;          // vocabulary rows per unit (MMA N)
constexpr int kBK = 64;           // K per stage: one 128-byte swizzle row of bf16
constexpr uint32_t kATile = kMRows * kBK * 2;  // 16 KB
constexpr uint32_t kBTile = kVt * kBK * 2;     // 32 KB
constexpr int kMaxMt = 2;         // hidden-row tiles per unit: 2 x 256 TMEM columns
constexpr int kSmemBudget = 227 * 1024 - 1024 - 256;
constexpr int kFinThreads = 512;
constexpr int kFinWarps = kFinThreads / 32;
constexpr int kResChunk = 16384;  // logits of both rows of a rejecting pair per residual CTA
constexpr int kResThreads = 256;
constexpr int kResSub = 512;      // residual sub-chunk
constexpr int kResSubs = kResChunk / kResSub;  // 32 (one warp's lanes take them)
static_assert(kResSubs <= 32 && kResSubs % 8 == 0, "sub-chunks of a residual CTA");

__host__ __device__ inline uint32_t fv_stage_bytes(int mt) { return (uint32_t)mt * kATile + kBTile; }

}  // namespace

struct FvMaps {
  CUtensorMap hid;   // [Na, d] bf16, boxes of 128 rows x 64 columns
  CUtensorMap head;  // [V, d] bf16, boxes of 256 rows x 64 columns
};

// A sequence's first rejection, for the residual kernel (j < 0: none).
struct alignas(16) FvRes {
  float Mt, iZt, Ml, iZl;  // target / draft row max and inverse partition sum
  int j, row, pad0, pad1;  // the rejecting position; its target row b (k+1) + j
};

struct FvArgs {
  int Na, V, d, k, mode;  // Na = B (k + 1) hidden rows, row b (k + 1) + j
  float c;                // log2(e) / T (1 / T = 1 when greedy)
  int n_mt, groups;       // 128-row tiles per unit; row groups of n_mt tiles
  int n_vt, kbs;          // 256-row vocabulary tiles; 64-wide k-blocks
  int stages, nunits;     // ring depth; (group, vocabulary tile) units
  const int *draft_tok;   // [B, k]
  const float *draft;     // [B, k, V] (stochastic)
  const float *u_accept;  // [B, k]
  const float *u_final;   // [B]
  float4 *part;           // [Na, n_vt] (max, sum of exp2 | argmax) per row and tile
  float4 *dpart;          // [B k, n_vt] (max, sum of exp2) of the draft rows (stochastic)
  float *tgt;             // [Na, V] stored logits (stochastic), else null
  int *status;
  unsigned *dctr;         // draft tiles claimed (in the status slot; zeroed by the finish kernel)
  // stochastic: the residual draw, spread over one CTA per kResChunk logits
  int nrc;                // residual chunks per row
  FvRes *rrec;            // [B] the first rejection of each sequence
  unsigned *rcnt;         // [B] residual CTAs arrived (zeroed by the finish kernel)
  float *rsub;            // [B, nrc, kResSubs] residual sub-chunk masses
  double *rcm;            // [B, nrc] residual chunk masses
};

struct FvOut {
  int *out_tok, *accept_len, *num_accepted;
};

namespace {


}  // namespace

// ---------------------------------------------------------------- GEMM kernel

// Unit u: vocabulary tile u % n_vt of hidden-row group u / n_vt.  Persistent
// CTAs take units blockIdx.x, blockIdx.x + gridDim.x, ...; the stage ring runs
// on across units; with one row tile the accumulator is double-buffered.
template <int MODE>
__global__ void __launch_bounds__(kFvThreads, 1) fv_gemm_kernel(const __grid_constant__ FvMaps maps,
                                                                  const FvArgs g) {
  trace_start(kTkFusedGemm);
  extern __shared__ unsigned char smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char *sm = smem_raw + pad;
  const int S = g.stages, MT = g.n_mt;
  const uint32_t sb = fv_stage_bytes(MT);
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + (size_t)S * sb);
  uint64_t *empty = full + S;
  uint64_t *done = empty + S;  // [2] accumulator ready for the epilogue
  uint64_t *tfree = done + 2;  // [2] accumulator read back
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tfree + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ncols = MT * kVt;
  const int nbuf = 2 * ncols <= 512 ? 2 : 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&done[q], 1);
      mbar_init(&tfree[q], 4);
    }
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, (uint32_t)(nbuf * ncols));
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_launch();

  if (warp == 0) {
    if (lane == 0) {
      // the head streams once (per row group); the hidden rows stay in L2
      const uint64_t pol_w = l2_policy_evict_first(), pol_a = l2_policy_evict_last();
      grid_dep_wait();
      bool ok = true;
      uint32_t i = 0;  // k-blocks issued by this CTA
      for (int u = blockIdx.x; u < g.nunits && ok; u += gridDim.x) {
        const int grp = u / g.n_vt, vt = u % g.n_vt;
        for (int kb = 0; kb < g.kbs && ok; ++kb, ++i) {
          const int s = (int)(i % S);
          if (i >= (uint32_t)S) ok = mbar_wait(&empty[s], ((i / S) - 1u) & 1u, g.status);
          if (!ok) break;
          unsigned char *st = sm + (size_t)s * sb;
          mbar_arrive_expect_tx(&full[s], sb);
          const int x = kb * kBK;
          tma_load_2d(st, &maps.head, x, vt * kVt, &full[s], pol_w);
          for (int m = 0; m < MT; ++m)
            tma_load_2d(st + kBTile + m * kATile, &maps.hid, x, (grp * MT + m) * kMRows, &full[s], pol_a);
        }
      }
      if (!ok)  // let copies still in flight land before the CTA exits
        for (uint32_t q = i > (uint32_t)S ? i - S : 0u; q < i; ++q)
          if (!mbar_wait(&full[q % S], (q / S) & 1u, g.status)) break;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kMRows, kVt);
      bool ok = true;
      uint32_t i = 0;
      for (int u = blockIdx.x, n = 0; u < g.nunits && ok; u += gridDim.x, ++n) {
        const int buf = n % nbuf;
        if (n >= nbuf) ok = mbar_wait(&tfree[buf], (uint32_t)((n / nbuf) - 1) & 1u, g.status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(buf * ncols);
        for (int kb = 0; kb < g.kbs && ok; ++kb, ++i) {
          const int s = (int)(i % S);
          ok = mbar_wait(&full[s], (i / S) & 1u, g.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t st = smem_u32(sm + (size_t)s * sb);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {  // 16 bf16 = 32 bytes: +2 in the >>4 address field
            const uint64_t bd = sw128_kmajor_desc(st) + 2 * kk;
            for (int m = 0; m < MT; ++m)  // row tile m accumulates in columns [m 256, (m + 1) 256)
              mma_bf16(acc + (uint32_t)(m * kVt), sw128_kmajor_desc(st + kBTile + m * kATile) + 2 * kk, bd, idesc,
                       (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&empty[s]);  // the stage is free once these MMAs have read it
        }
        mma_commit(&done[buf]);
      }
    }
  } else {
    // warp w reads TMEM lanes 32 (w % 4) .. + 31: one hidden row per thread
    const int q = warp & 3;
    const float c = g.c;
    bool ok = true;
    for (int u = blockIdx.x, n = 0; u < g.nunits && ok; u += gridDim.x, ++n) {
      const int grp = u / g.n_vt, vt = u % g.n_vt;
      const int buf = n % nbuf;
      ok = mbar_wait(&done[buf], (uint32_t)(n / nbuf) & 1u, g.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)(buf * ncols);
      const int v0 = vt * kVt;
      for (int m = 0; m < MT; ++m) {
        const int row = (grp * MT + m) * kMRows + q * 32 + lane;
        const bool valid = row < g.Na;
        float M = -INFINITY, Ssum = 0.f;
        int I = 0x7fffffff;
        float *trow = (MODE == 1 && valid) ? g.tgt + (size_t)row * g.V : nullptr;
        for (int c0 = 0; c0 < kVt; c0 += 32) {
          float v[32];
          tmem_ld32(acc + ((uint32_t)(q * 32) << 16) + (uint32_t)(m * kVt + c0), v);
          const int e0 = v0 + c0;
          const int nv = min(32, g.V - e0);  // columns past the vocabulary hold zeros
          if (MODE == 0) {
#pragma unroll
            for (int t = 0; t < 32; ++t)
              if (t < nv && v[t] > M) {  // ascending order: the first maximum stays
                M = v[t];
                I = e0 + t;
              }
          } else {
            float cm = -INFINITY;
#pragma unroll
            for (int t = 0; t < 32; ++t)
              if (t < nv) cm = fmaxf(cm, v[t]);
            if (cm > M) {
              if (M != -INFINITY) Ssum *= ex2_approx((M - cm) * c);
              M = cm;
            }
            if (M != -INFINITY) {
              const float mc = M * c;
              float s0 = 0.f, s1 = 0.f;
#pragma unroll
              for (int t = 0; t < 32; t += 2) {
                if (t < nv) s0 += ex2_approx(fmaf(v[t], c, -mc));
                if (t + 1 < nv) s1 += ex2_approx(fmaf(v[t + 1], c, -mc));
              }
              Ssum += s0 + s1;
            }
            if (trow && nv > 0) {
              float *dst = trow + e0;
              if (nv == 32 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
#pragma unroll
                for (int t = 0; t < 32; t += 4)
                  *reinterpret_cast<float4 *>(dst + t) = make_float4(v[t], v[t + 1], v[t + 2], v[t + 3]);
              } else {
#pragma unroll
                for (int t = 0; t < 32; ++t)
                  if (t < nv) dst[t] = v[t];
              }
            }
          }
        }
        if (valid && in_bounds(vt < g.n_vt, g.status))
          g.part[(size_t)row * g.n_vt + vt] = make_float4(M, MODE == 0 ? __int_as_float(I) : Ssum, 0.f, 0.f);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tfree[buf]);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)(nbuf * ncols));
  }
  trace_end(kTkFusedGemm);
}

// ---------------------------------------------------------------- draft-row statistics (stochastic)

// Per (draft row, 256-token tile): (max, sum of exp2((x - max) log2e / T)) of
// the draft logits, in the target partials' tiling.  A few CTAs per SM take
// the (row, tile) items grid-stride, a warp four tiles at a time (each lane
// 8 elements of each, loads issued together): every draft logit is read once.
// It reads only the caller's draft logits, so it runs beside the GEMM (which
// leaves room for it on every SM); it waits for the GEMM once its work is
// done, so that the finish kernel's wait on this kernel covers both.
__global__ void __launch_bounds__(256) fv_draft_stats_kernel(const FvArgs g) {
  trace_start(kTkFusedAux);
  const int lane = threadIdx.x & 31;
  grid_dep_launch();
  const long long total = (long long)g.Na / (g.k + 1) * g.k * g.n_vt;  // B k rows x n_vt tiles
  // each warp claims four tiles at a time: however many of the CTAs find room
  // beside the GEMM's, those that run take all the tiles
  for (;;) {
    long long i0 = 0;
    if (lane == 0) i0 = (long long)atomicAdd(g.dctr, 4u);
    i0 = __shfl_sync(0xffffffffu, i0, 0);
    if (i0 >= total) break;
    float x[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long i = i0 + u;
      const int r = (int)(i / g.n_vt), t = (int)(i - (long long)r * g.n_vt);
      const float *row = g.draft + (size_t)r * g.V;
      const int e0 = t * kVt, n = i < total ? min(kVt, g.V - e0) : 0;
      if (n == kVt && (reinterpret_cast<uintptr_t>(row + e0) & 15u) == 0) {
        const float4 a = __ldcg(reinterpret_cast<const float4 *>(row + e0) + lane);
        const float4 b = __ldcg(reinterpret_cast<const float4 *>(row + e0) + 32 + lane);
        x[u][0] = a.x; x[u][1] = a.y; x[u][2] = a.z; x[u][3] = a.w;
        x[u][4] = b.x; x[u][5] = b.y; x[u][6] = b.z; x[u][7] = b.w;
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int e = (q < 4 ? 4 * lane + q : 128 + 4 * lane + q - 4);
          x[u][q] = e < n ? __ldcg(row + e0 + e) : -INFINITY;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const long long i = i0 + u;
      float m = x[u][0];
#pragma unroll
      for (int q = 1; q < 8; ++q) m = fmaxf(m, x[u][q]);
      m = warp_max(m);
      float sum = 0.f;
      if (m != -INFINITY) {
        const float mc = m * g.c;
#pragma unroll
        for (int q = 0; q < 8; ++q) sum += ex2_approx(fmaf(x[u][q], g.c, -mc));
      }
      sum = warp_sum(sum);
      if (lane == 0 && i < total) {
        const int r = (int)(i / g.n_vt), t = (int)(i - (long long)r * g.n_vt);
        g.dpart[(size_t)r * g.n_vt + t] = make_float4(m, sum, 0.f, 0.f);
      }
    }
  }
  __syncthreads();
  trace_mark(kTkFusedAux, 0);  // this CTA found no tile left
  grid_dep_wait();
  trace_dep(kTkFusedAux);
  trace_end(kTkFusedAux);
}

// ---------------------------------------------------------------- finish kernel

namespace {

__device__ __forceinline__ double fv_warp_incl_scan(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

struct FinShared {
  float M[9], Ml[8];
  double Z[9], Zl[8];
  int I[9];
};

// Sampling weight of an element: the residual max(0, p - q) (kind 0), the
// target probability p (kind 1), the unnormalised target weight (kind 2).
struct Wt {
  int kind;
  float Mt, iZt, Ml, iZl, c;
};

__device__ __forceinline__ float wval(const Wt &w, float t, float l) {
  const float e = ex2_approx((t - w.Mt) * w.c);
  if (w.kind == 2) return e;
  // both products rounded on their own (no fused multiply-add): where p and q
  // are equal the residual must be exactly zero, so that the draw falls back to p
  const float p = __fmul_rn(e, w.iZt);
  if (w.kind == 1) return p;
  return fmaxf(0.f, p - __fmul_rn(ex2_approx((l - w.Ml) * w.c), w.iZl));
}

// Row j's (max, partition sum relative to it) from its per-tile partials, in
// tile order per lane, lanes combined in a fixed tree (warp-collective).  The
// lane's (max, sum) pairs are loaded 24 at a time (all of them, up to 768
// tiles a row), so that their loads overlap.
__device__ __forceinline__ void combine_lse(const float4 *pp, int n_vt, float c, float &M, double &Z) {
  constexpr int NB = 24;
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  double z = 0.0;
  for (int t0 = lane; t0 < n_vt; t0 += NB * 32) {  // online over batches of NB tiles
    float2 p[NB];
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int t = t0 + 32 * i;
      p[i] = t < n_vt ? __ldcg(reinterpret_cast<const float2 *>(pp + t)) : make_float2(-INFINITY, 0.f);
    }
    float bm = p[0].x;
#pragma unroll
    for (int i = 1; i < NB; ++i) bm = fmaxf(bm, p[i].x);
    if (bm > m) {
      if (m != -INFINITY) z *= (double)ex2_approx((m - bm) * c);
      m = bm;
    }
    if (m != -INFINITY)
#pragma unroll
      for (int i = 0; i < NB; ++i)
        if (p[i].x != -INFINITY) z += (double)p[i].y * (double)ex2_approx((p[i].x - m) * c);
  }
  // lanes: rescale to the warp maximum, then sum in a fixed tree
  const float wm = warp_max(m);
  z = (m == -INFINITY) ? 0.0 : z * (double)ex2_approx((m - wm) * c);
  M = wm;
  Z = warp_sum_d(z);
}

}  // namespace

// One CTA per sequence: the decisions of spec_verify from the GEMM's
// partials (and, stochastic, the draft rows' partials), then the draw.
template <int MODE>
__global__ void __launch_bounds__(kFinThreads, 1) fv_finish_kernel(const FvArgs g, FvOut o) {
  trace_start(kTkFusedAux);
  extern __shared__ __align__(16) unsigned char fin_smem[];
  FinShared &sh = *reinterpret_cast<FinShared *>(fin_smem);
  const int b = blockIdx.x, k = g.k, V = g.V;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float c = g.c;
  grid_dep_wait();
  grid_dep_launch();
  trace_dep(kTkFusedAux);
  if (MODE == 1 && b == 0 && threadIdx.x == 0) *g.dctr = 0u;  // the draft statistics have ended: left zero
  // each row's statistics from its partials, in vocabulary-tile order
  for (int j = warp; j <= k; j += kFinWarps) {
    const float4 *pp = g.part + (size_t)(b * (k + 1) + j) * g.n_vt;
    if (MODE == 0) {
      float m = -INFINITY;
      int idx = 0x7fffffff;
      for (int t0 = lane; t0 < g.n_vt; t0 += 8 * 32) {  // eight partials in flight per lane
        float4 p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int t = t0 + 32 * i;
          p[i] = t < g.n_vt ? __ldcg(&pp[t]) : make_float4(-INFINITY, __int_as_float(0x7fffffff), 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) argmax_merge(m, idx, p[i].x, __float_as_int(p[i].y));
      }
      warp_argmax(m, idx);
      if (lane == 0) {
        sh.M[j] = m;
        sh.I[j] = idx;
      }
    } else {
      float m;
      double z;
      combine_lse(pp, g.n_vt, c, m, z);
      if (lane == 0) {
        sh.M[j] = m;
        sh.Z[j] = z;
      }
    }
  }
  if (MODE == 1)  // the draft rows on the warps after the target rows'
    for (int j = (warp + kFinWarps - (k + 1) % kFinWarps) % kFinWarps; j < k; j += kFinWarps) {
      float m;
      double z;
      combine_lse(g.dpart + (size_t)(b * k + j) * g.n_vt, g.n_vt, c, m, z);
      if (lane == 0) {
        sh.Ml[j] = m;
        sh.Zl[j] = z;
      }
    }
  __syncthreads();
  trace_mark(kTkFusedAux, 0);  // rows' statistics combined
  const int *dt = g.draft_tok + (size_t)b * k;
  int n_acc = 0, tok = 0, flags = 0;
  if (MODE == 0) {
    while (n_acc < k) {
      const int d = __ldg(&dt[n_acc]);
      if (d < 0 || d >= V) {
        flags |= kStatusBadToken;
        break;
      }
      if (!(sh.M[n_acc] > -INFINITY) || sh.I[n_acc] != d) break;
      ++n_acc;
    }
    tok = sh.I[n_acc];
    if (!(sh.M[n_acc] > -INFINITY) || tok == 0x7fffffff) {
      flags |= kStatusNonFinite;
      tok = 0;
    }
  } else {
    // u q(d) < p(d) at every position at once, lane j of warp 0 position j
    // (its token, the logits there and its uniform loaded together); the
    // first rejection and the flags are those of taking them in order
    if (warp == 0) {
      float tdl = 0.f, ldl = 0.f;
      int dl = -1;
      double ua = 0.0;
      if (lane < k) {
        dl = __ldg(&dt[lane]);
        ua = (double)__ldg(&g.u_accept[(size_t)b * k + lane]);
        if (dl >= 0 && dl < V) {
          tdl = __ldcg(g.tgt + (size_t)(b * (k + 1) + lane) * V + dl);
          ldl = __ldcg(g.draft + ((size_t)b * k + lane) * V + dl);
        }
      }
      const bool valid = dl >= 0 && dl < V;
      bool finite = true, accept = true;
      if (lane < k && valid) {
        finite = sh.M[lane] > -INFINITY && sh.Ml[lane] > -INFINITY;
        const double p = exp2(((double)tdl - (double)sh.M[lane]) * (double)c) / sh.Z[lane];
        const double q = exp2(((double)ldl - (double)sh.Ml[lane]) * (double)c) / sh.Zl[lane];
        accept = ua * q < p;
      }
      int fl;
      const int rj = first_rejection(k, valid, finite, accept, fl);
      if (lane == 0) {
        sh.I[0] = rj;
        sh.I[1] = fl;
      }
    }
    __syncthreads();
    trace_mark(kTkFusedAux, 1);  // decisions taken
    const int rej = sh.I[0];
    flags |= sh.I[1];
    // the draw is the residual kernel's: over max(0, p - q) of the rejected
    // pair, or over p of row k when every draft is accepted
    const int r = rej >= 0 ? rej : k;
    n_acc = r;
    if (threadIdx.x == 0) {
      float4 *r4 = reinterpret_cast<float4 *>(&g.rrec[b]);
      r4[0] = make_float4(sh.M[r], (float)(1.0 / sh.Z[r]), rej >= 0 ? sh.Ml[rej] : 0.f,
                          rej >= 0 ? (float)(1.0 / sh.Zl[rej]) : 0.f);
      reinterpret_cast<int4 *>(r4)[1] = make_int4(r, b * (k + 1) + r, 0, 0);
      g.rcnt[b] = 0u;
    }
    tok = -2;  // written by the residual kernel
  }
  if (threadIdx.x <= k) {
    const int t = threadIdx.x;
    if (!(t == n_acc && tok == -2))
      o.out_tok[(size_t)b * (k + 1) + t] = t < n_acc ? __ldg(&dt[t]) : (t == n_acc ? tok : -1);
  }
  if (threadIdx.x == 0) {
    o.accept_len[b] = n_acc + 1;
    o.num_accepted[b] = n_acc;
    if (flags) set_status(g.status, flags);
  }
  trace_end(kTkFusedAux);
}

// ---------------------------------------------------------------- residual kernel

namespace {

// One warp: the crossing of u x (total of mass(0..n-1), summed in index
// order): the smallest index whose running sum passes it, with the mass
// before it; else the last index of positive mass (before = -1); else -1.
template <typename F>
__device__ int fv_warp_cross(F mass, int n, double u, double &tgt, double &before_out) {
  const int lane = threadIdx.x & 31;
  double tot = 0.0;
  for (int b = 0; b < n; b += 32)
    tot += __shfl_sync(0xffffffffu, fv_warp_incl_scan(b + lane < n ? mass(b + lane) : 0.0), 31);
  tgt = u * tot;
  int cross = -1, lastpos = -1;
  double before = 0.0, run = 0.0;
  for (int b = 0; b < n && cross < 0; b += 32) {
    const double x = b + lane < n ? mass(b + lane) : 0.0;
    const double incl = fv_warp_incl_scan(x);
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

// One warp: in the LEN elements from e0 (lane l a contiguous run of LEN / 32,
// its weights taken eight at a time with the eight loads issued together),
// the element whose running sum (`before` ahead of e0) passes tgt; before < 0,
// or nothing passing: the last element of positive weight; -1 if none.
template <int LEN>
__device__ int fv_warp_rescan(const Wt &w, const float *trow, const float *lrow, int V, int e0, double before,
                              double tgt) {
  constexpr int PER = LEN / 32, G = 8;
  static_assert(PER % G == 0, "whole batches");
  const int lane = threadIdx.x & 31;
  const int a0 = e0 + lane * PER;
  const bool pair = w.kind == 0;
  double ls = 0.0;
  int lp = -1;
#pragma unroll 1
  for (int q0 = 0; q0 < PER; q0 += G) {
    float x[G];
#pragma unroll
    for (int q = 0; q < G; ++q) {
      const int i = a0 + q0 + q;
      x[q] = i < V ? wval(w, __ldcg(trow + i), pair ? __ldcg(lrow + i) : 0.f) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < G; ++q) {
      ls += (double)x[q];
      if (x[q] > 0.f) lp = a0 + q0 + q;
    }
  }
  const double inc = fv_warp_incl_scan(ls);
  int f = 0x7fffffff;
  if (before >= 0.0 && before + inc > tgt) {
    double r = before + (inc - ls);
#pragma unroll 1
    for (int q0 = 0; q0 < PER && f == 0x7fffffff; q0 += G) {
      float x[G];
#pragma unroll
      for (int q = 0; q < G; ++q) {
        const int i = a0 + q0 + q;
        x[q] = i < V ? wval(w, __ldcg(trow + i), pair ? __ldcg(lrow + i) : 0.f) : 0.f;
      }
#pragma unroll
      for (int q = 0; q < G; ++q) {
        r += (double)x[q];
        if (f == 0x7fffffff && x[q] > 0.f && r > tgt) f = a0 + q0 + q;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    f = min(f, __shfl_xor_sync(0xffffffffu, f, o));
    lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
  }
  return f != 0x7fffffff ? f : lp;
}

struct ResShared {
  float sub[kResSubs];
  double wtot[kResThreads / 32];
  int wlast[kResThreads / 32];
  int last, tok;
};

// Block-collective: a draw from p of target row `row` at u, the tile masses
// from the GEMM's partials (a tile's sum of exp2((t - m) c) rescaled to the
// row's maximum Mt).  Each warp sums a contiguous run of tiles; warp 0 finds
// the run holding the crossing from the runs' totals, then the tile within it
// (all running sums in index order), then rescans that tile's logits.
// Returns the token, -1 if every weight is zero.
__device__ int draw_p_tiles(ResShared &rs, const FvArgs &g, int row, float Mt, double u) {
  constexpr int W = kResThreads / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = g.n_vt, wrun = (n + W - 1) / W;
  const float4 *pp = g.part + (size_t)row * n;
  auto mass = [&](int i) {
    const float2 p = __ldcg(reinterpret_cast<const float2 *>(pp + i));
    return p.x == -INFINITY ? 0.0 : (double)p.y * (double)ex2_approx((p.x - Mt) * g.c);
  };
  {
    const int c0 = warp * wrun, c1 = min(n, c0 + wrun);
    double tot = 0.0;
    int lastpos = -1;
    for (int b = c0; b < c1; b += 32) {
      const double x = b + lane < c1 ? mass(b + lane) : 0.0;
      tot += __shfl_sync(0xffffffffu, fv_warp_incl_scan(x), 31);
      const unsigned pos = __ballot_sync(0xffffffffu, b + lane < c1 && x > 0.0);
      if (pos) lastpos = b + 31 - __clz(pos);
    }
    if (lane == 0) {
      rs.wtot[warp] = tot;
      rs.wlast[warp] = lastpos;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const double x = lane < W ? rs.wtot[lane] : 0.0;
    const double incl = fv_warp_incl_scan(x);
    const double tgt = u * __shfl_sync(0xffffffffu, incl, 31);
    const unsigned hit = __ballot_sync(0xffffffffu, lane < W && incl > tgt);
    int cross = -1;
    double before = -1.0;
    if (hit) {
      // the run's tiles (and, should rounding carry the crossing past it, the next)
      const int cw = __ffs(hit) - 1;
      double run = __shfl_sync(0xffffffffu, incl - x, cw);
      for (int b = cw * wrun; b < n && cross < 0; b += 32) {
        const double y = b + lane < n ? mass(b + lane) : 0.0;
        const double in2 = fv_warp_incl_scan(y);
        const unsigned h2 = __ballot_sync(0xffffffffu, b + lane < n && run + in2 > tgt);
        if (h2) {
          const int l = __ffs(h2) - 1;
          cross = b + l;
          before = run + __shfl_sync(0xffffffffu, in2 - y, l);
        }
        run += __shfl_sync(0xffffffffu, in2, 31);
      }
    }
    if (cross < 0) {  // nothing passes: the last tile of positive mass
      const unsigned pw = __ballot_sync(0xffffffffu, lane < W && rs.wlast[lane] >= 0);
      if (pw) cross = rs.wlast[31 - __clz(pw)];
      before = -1.0;
    }
    int tok = -1;
    if (cross >= 0) {
      const Wt wp{2, Mt, 0.f, 0.f, 0.f, g.c};
      const float *trow = g.tgt + (size_t)row * g.V;
      tok = fv_warp_rescan<kVt>(wp, trow, trow, g.V, cross * kVt, before, tgt);
    }
    if (lane == 0) rs.tok = tok;
  }
  __syncthreads();
  return rs.tok;
}

}  // namespace

// The draws of the stochastic call, after the finish kernel.  After a
// rejection at j, CTA (c, b) sums max(0, p - q) over the 32 sub-chunks of
// chunk c of sequence b's rejected pair (the stored target row and the draft
// row); the CTA that completes the sequence finds the crossing chunk, then
// sub-chunk, then element (float64 running sums in index order), and writes
// the replacement token.  With every draft accepted, CTA (0, b) makes the
// bonus draw from p of row k over the GEMM's tile partials.
__global__ void __launch_bounds__(kResThreads, 4) fv_residual_kernel(const FvArgs g, FvOut o) {
  trace_start(kTkFusedAux);
  __shared__ ResShared rs;
  const int ch = blockIdx.x, b = blockIdx.y, V = g.V, k = g.k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_wait();  // the finish kernel's records
  grid_dep_launch();
  trace_dep(kTkFusedAux);
  const float4 *r4 = reinterpret_cast<const float4 *>(&g.rrec[b]);
  const float4 rx = __ldcg(r4);
  const int4 ry = __ldcg(reinterpret_cast<const int4 *>(r4 + 1));
  const int j = ry.x, row = ry.y;
  if (!in_bounds(j >= 0 && j <= k && row == b * (k + 1) + j, g.status) || (j == k && ch != 0)) {
    trace_end(kTkFusedAux);
    return;
  }
  const double u = (double)__ldg(&g.u_final[b]);
  int tok = -1;
  if (j < k) {
    const Wt w{0, rx.x, rx.y, rx.z, rx.w, g.c};
    const float *trow = g.tgt + (size_t)row * V, *lrow = g.draft + ((size_t)b * k + j) * V;
    const bool vec = ((reinterpret_cast<uintptr_t>(trow) | reinterpret_cast<uintptr_t>(lrow)) & 15u) == 0;
    // sub-chunks warp + 8 h, a lane 4 float4 of each row of a sub-chunk
#pragma unroll
    for (int h = 0; h < kResSubs / 8; ++h) {
      const int s = warp + 8 * h;
      const int e0 = ch * kResChunk + s * kResSub;
      float acc = 0.f;
      if (vec && e0 + kResSub <= V) {
        float4 tv[4], lv[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          tv[q] = __ldcg(reinterpret_cast<const float4 *>(trow + e0) + lane + 32 * q);
          lv[q] = __ldcg(reinterpret_cast<const float4 *>(lrow + e0) + lane + 32 * q);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          acc += (wval(w, tv[q].x, lv[q].x) + wval(w, tv[q].y, lv[q].y)) +
                 (wval(w, tv[q].z, lv[q].z) + wval(w, tv[q].w, lv[q].w));
      } else {
        for (int i = e0 + lane; i < min(V, e0 + kResSub); i += 32) acc += wval(w, __ldcg(trow + i), __ldcg(lrow + i));
      }
      acc = warp_sum(acc);
      if (lane == 0) rs.sub[s] = acc;
    }
    __syncthreads();
    if (threadIdx.x < kResSubs) g.rsub[((size_t)b * g.nrc + ch) * kResSubs + threadIdx.x] = rs.sub[threadIdx.x];
    if (threadIdx.x == 0) {
      double cm = 0.0;
      for (int s = 0; s < kResSubs; ++s) cm += (double)rs.sub[s];
      g.rcm[(size_t)b * g.nrc + ch] = cm;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned arrived = atomic_add_acq_rel(&g.rcnt[b], 1u) + 1u;
      rs.last = arrived == (unsigned)g.nrc;
      if (rs.last) g.rcnt[b] = 0u;  // left zero
    }
    __syncthreads();
    if (!rs.last) {
      trace_end(kTkFusedAux);
      return;
    }
    if (warp == 0) {
      const double *cm = g.rcm + (size_t)b * g.nrc;
      double tgt, base;
      const int cx = fv_warp_cross([&](int i) { return __ldcg(&cm[i]); }, g.nrc, u, tgt, base);
      int t = -1;
      if (cx >= 0) {
        const float *sm = g.rsub + ((size_t)b * g.nrc + cx) * kResSubs;
        // within the chunk: its sub-chunk masses against tgt - base
        const double rel = base >= 0.0 ? tgt - base : 1e300;
        const double x = lane < kResSubs ? (double)__ldcg(&sm[lane]) : 0.0;
        const double incl = fv_warp_incl_scan(x);
        const unsigned hit = __ballot_sync(0xffffffffu, lane < kResSubs && incl > rel);
        const unsigned pos = __ballot_sync(0xffffffffu, lane < kResSubs && x > 0.0);
        int s = -1;
        double bef = -1.0;
        if (hit) {
          s = __ffs(hit) - 1;
          bef = base + __shfl_sync(0xffffffffu, incl - x, s);
        } else if (pos) {
          s = 31 - __clz(pos);
        }
        if (s >= 0) t = fv_warp_rescan<kResSub>(w, trow, lrow, V, cx * kResChunk + s * kResSub, bef, tgt);
      }
      if (lane == 0) rs.tok = t;
    }
    __syncthreads();
    tok = rs.tok;
  }
  // every draft accepted (the bonus draw), or a residual that is zero
  // everywhere (p = q, so the draw falls back to p itself): p of the row
  if (tok < 0) tok = draw_p_tiles(rs, g, row, rx.x, u);
  if (threadIdx.x == 0) {
    if (tok < 0) {
      set_status(g.status, kStatusNonFinite);
      tok = 0;
    }
    o.out_tok[(size_t)b * (k + 1) + j] = tok;
  }
  trace_end(kTkFusedAux);
}

// ---------------------------------------------------------------- host side

namespace {

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

int fv_sms() {
  static int sms = 0;
  int dev = 0;
  if (sms <= 0 && (cudaGetDevice(&dev) != cudaSuccess ||
                   cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess))
    sms = 0;
  return sms > 0 ? sms : 152;
}

}  // namespace

bool fused_shape_ok(int B, int k, int V, int d) {
  if (B < 1 || k < 1 || k > 8 || V < 1 || d < 8 || d % 8) return false;
  if ((long long)B * (k + 1) >= (1ll << 30) || V > (1 << 30)) return false;
  return true;
}

size_t fused_workspace_bytes(int B, int k, int V, int d, int mode) {
  (void)d;
  const size_t Na = (size_t)B * (k + 1);
  const size_t n_vt = ((size_t)V + kVt - 1) / kVt;
  size_t n = 256;                   // status word
  n += up256(Na * n_vt * 16);       // partials
  if (mode == 1) {
    n += up256((size_t)B * k * n_vt * 16);  // the draft rows' partials
    n += up256(Na * (size_t)V * 4);         // stored logits (the residual draw reads one row)
    const size_t nrc = ((size_t)V + kResChunk - 1) / kResChunk;
    n += up256((size_t)B * sizeof(FvRes));  // residual records
    n += up256((size_t)B * 4);              // residual arrival counters
    n += up256((size_t)B * nrc * kResSubs * 4);
    n += up256((size_t)B * nrc * 8);
  }
  return n;
}

cudaError_t fused_set_attributes() {
  const int g_bytes = kSmemBudget + 1024 + 256;
  cudaError_t e = cudaFuncSetAttribute(fv_gemm_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, g_bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fv_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, g_bytes);
  const int f_bytes = (int)sizeof(FinShared);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fv_finish_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, f_bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fv_finish_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, f_bytes);
  return e;
}

cudaError_t launch_fused_verify(const FusedCall &fc, cudaStream_t s, bool pdl) {
  FvArgs g{};
  g.Na = fc.B * (fc.k + 1);
  g.V = fc.V;
  g.d = fc.d;
  g.k = fc.k;
  g.mode = fc.mode;
  g.c = kLog2e / (fc.mode == 1 ? fc.T : 1.f);
  // one or two 128-row tiles per unit; more rows run in groups (the head is
  // streamed once per group)
  g.n_mt = g.Na > kMRows ? kMaxMt : 1;
  g.groups = (g.Na + g.n_mt * kMRows - 1) / (g.n_mt * kMRows);
  g.n_vt = (fc.V + kVt - 1) / kVt;
  g.kbs = (fc.d + kBK - 1) / kBK;
  g.nunits = g.groups * g.n_vt;
  g.stages = (int)(kSmemBudget / fv_stage_bytes(g.n_mt));
  if (g.stages > 6) g.stages = 6;
  g.draft_tok = fc.draft_tok;
  g.draft = fc.draft;
  g.u_accept = fc.u_accept;
  g.u_final = fc.u_final;
  char *p = static_cast<char *>(fc.ws);
  g.status = reinterpret_cast<int *>(p);
  g.dctr = reinterpret_cast<unsigned *>(p + 128);
  p += 256;
  g.part = reinterpret_cast<float4 *>(p);
  p += up256((size_t)g.Na * g.n_vt * 16);
  if (fc.mode == 1) {
    g.dpart = reinterpret_cast<float4 *>(p);
    p += up256((size_t)fc.B * fc.k * g.n_vt * 16);
    g.tgt = reinterpret_cast<float *>(p);
    p += up256((size_t)g.Na * fc.V * 4);
    g.nrc = (fc.V + kResChunk - 1) / kResChunk;
    g.rrec = reinterpret_cast<FvRes *>(p);
    p += up256((size_t)fc.B * sizeof(FvRes));
    g.rcnt = reinterpret_cast<unsigned *>(p);
    p += up256((size_t)fc.B * 4);
    g.rsub = reinterpret_cast<float *>(p);
    p += up256((size_t)fc.B * g.nrc * kResSubs * 4);
    g.rcm = reinterpret_cast<double *>(p);
  }

  FvMaps maps{};
  if (!make_bf16_map(&maps.hid, fc.hidden, (uint64_t)fc.d, (uint64_t)g.Na, (uint64_t)fc.d, kMRows))
    return cudaErrorInvalidValue;
  if (!make_bf16_map(&maps.head, fc.head, (uint64_t)fc.d, (uint64_t)fc.V, (uint64_t)fc.d, kVt))
    return cudaErrorInvalidValue;

  cudaError_t e = cudaSuccess;
  const size_t smem = (size_t)g.stages * fv_stage_bytes(g.n_mt) + (size_t)(2 * g.stages + 4) * 8 + 16 + 1024;
  const int sms = fv_sms();
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(g.nunits < sms ? g.nunits : sms));
  cfg.blockDim = dim3(kFvThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.numAttrs = 0;
  note_launch();
  e = fc.mode == 1 ? cudaLaunchKernelEx(&cfg, fv_gemm_kernel<1>, maps, g)
                   : cudaLaunchKernelEx(&cfg, fv_gemm_kernel<0>, maps, g);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute pattr[1];
  pattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pattr[0].val.programmaticStreamSerializationAllowed = 1;
  if (fc.mode == 1) {  // the draft rows' statistics, beside the GEMM (it needs no smem)
    cudaLaunchConfig_t dcfg{};
    dcfg.gridDim = dim3((unsigned)(2 * sms));  // grid-stride: two CTAs an SM, beside the GEMM's
    dcfg.blockDim = dim3(256);
    dcfg.stream = s;
    dcfg.attrs = pattr;
    dcfg.numAttrs = pdl ? 1 : 0;
    note_launch();
    e = cudaLaunchKernelEx(&dcfg, fv_draft_stats_kernel, g);
    if (e != cudaSuccess) return e;
  }

  FvOut o{fc.out_tok, fc.accept_len, fc.num_accepted};
  cudaLaunchConfig_t fcfg{};
  fcfg.gridDim = dim3((unsigned)fc.B);
  fcfg.blockDim = dim3(kFinThreads);
  fcfg.dynamicSmemBytes = sizeof(FinShared);
  fcfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  fcfg.attrs = attr;
  fcfg.numAttrs = pdl ? 1 : 0;
  note_launch();
  if (fc.mode == 0) return cudaLaunchKernelEx(&fcfg, fv_finish_kernel<0>, g, o);
  e = cudaLaunchKernelEx(&fcfg, fv_finish_kernel<1>, g, o);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t rcfg{};
  rcfg.gridDim = dim3((unsigned)g.nrc, (unsigned)fc.B);
  rcfg.blockDim = dim3(kResThreads);
  rcfg.stream = s;
  rcfg.attrs = attr;
  rcfg.numAttrs = pdl ? 1 : 0;
  note_launch();
  return cudaLaunchKernelEx(&rcfg, fv_residual_kernel, g, o);
}

MTP_TRACE_COLLECTOR(fused)

}  // namespace mtp
