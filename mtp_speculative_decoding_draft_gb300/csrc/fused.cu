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
// fv_finish_kernel: one CTA per sequence combines the partials of its k+1
//   rows in vocabulary-tile order and takes the decisions of spec_verify (the
//   same rule): greedy longest prefix; stochastic u q(d) < p(d) position by
//   position with the draft row's normaliser from one pass over it, then the
//   inverse-CDF draw at u_final over max(0, p - q) of the first rejecting row
//   (over p if that is identically zero), or over p of row k when every draft
//   is accepted.  Only the rows the decisions reach are read.
#include <cuda.h>
#include <stdlib.h>

#include "common.cuh"
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
constexpr int kFinThreads = 256;
constexpr int kFinWarps = kFinThreads / 32;
constexpr int kMaxChunks = 4096;  // inverse-CDF chunk sums per row, at most

__host__ __device__ inline uint32_t fv_stage_bytes(int mt) { return (uint32_t)mt * kATile + kBTile; }

}  // namespace

struct FvMaps {
  CUtensorMap hid;   // [Na, d] bf16, boxes of 128 rows x 64 columns
  CUtensorMap head;  // [V, d] bf16, boxes of 256 rows x 64 columns
};

struct FvArgs {
  int Na, V, d, k, mode;  // Na = B (k + 1) hidden rows, row b (k + 1) + j
  float c;                // log2(e) / T (1 / T = 1 when greedy)
  int n_mt, groups;       // 128-row tiles per unit; row groups of n_mt tiles
  int n_vt, kbs;          // 256-row vocabulary tiles; 64-wide k-blocks
  int stages, nunits;     // ring depth; (group, vocabulary tile) units
  int chunk;              // elements per chunk of the finish kernel's draws
  const int *draft_tok;   // [B, k]
  const float *draft;     // [B, k, V] (stochastic)
  const float *u_accept;  // [B, k]
  const float *u_final;   // [B]
  float4 *part;           // [Na, n_vt] (max, sum of exp2 | argmax) per row and tile
  float *tgt;             // [Na, V] stored logits (stochastic), else null
  int *status;
};

struct FvOut {
  int *out_tok, *accept_len, *num_accepted;
};

namespace {

// 2^x, hardware approximation (relative error about 2^-22; -inf gives +0).
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace

// ---------------------------------------------------------------- GEMM kernel

// Unit u: vocabulary tile u % n_vt of hidden-row group u / n_vt.  Persistent
// CTAs take units blockIdx.x, blockIdx.x + gridDim.x, ...; the stage ring runs
// on across units; with one row tile the accumulator is double-buffered.
template <int MODE>
__global__ void __launch_bounds__(kFvThreads, 1) fv_gemm_kernel(const __grid_constant__ FvMaps maps,
                                                                  const FvArgs g) {
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
              if (M != -INFINITY) Ssum *= ex2f((M - cm) * c);
              M = cm;
            }
            if (M != -INFINITY) {
              const float mc = M * c;
              float s0 = 0.f, s1 = 0.f;
#pragma unroll
              for (int t = 0; t < 32; t += 2) {
                if (t < nv) s0 += ex2f(fmaf(v[t], c, -mc));
                if (t + 1 < nv) s1 += ex2f(fmaf(v[t + 1], c, -mc));
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
        if (valid) g.part[(size_t)row * g.n_vt + vt] = make_float4(M, MODE == 0 ? __int_as_float(I) : Ssum, 0.f, 0.f);
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
  float M[9];
  double Z[9];
  int I[9];
  float red_f[kFinWarps];
  double red_d[kFinWarps];
  int red_i[kFinWarps];
  int chosen;
  double csum[kMaxChunks];
};

// Block-wide (max over the block of m, then sum over threads of s 2^((m - M) c))
// -- this thread holds (m, s) over its own elements.  Every thread gets both.
__device__ void block_lse(FinShared &sh, float m, float s, float c, float &Mout, double &Zout) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float wm = warp_max(m);
  if (lane == 0) sh.red_f[warp] = wm;
  __syncthreads();
  float M = -INFINITY;
  for (int w = 0; w < kFinWarps; ++w) M = fmaxf(M, sh.red_f[w]);
  double z = (m == -INFINITY || M == -INFINITY) ? 0.0 : (double)s * (double)ex2f((m - M) * c);
  z = warp_sum_d(z);
  if (lane == 0) sh.red_d[warp] = z;
  __syncthreads();
  double Z = 0.0;
  for (int w = 0; w < kFinWarps; ++w) Z += sh.red_d[w];
  __syncthreads();
  Mout = M;
  Zout = Z;
}

// Inverse-CDF draw over weights wfn(i), i in [0, V): the smallest i with C_i >
// u S (C the running sum in index order, S the total), else the last index of
// positive weight; -1 if every weight is zero.  Chunk sums in float64 by the
// whole block (each lane adds its elements in float, the lanes in float64),
// then warp 0 scans the chunks and rescans the crossing chunk in float64.
template <class WFn>
__device__ int block_inverse_cdf(FinShared &sh, WFn wfn, int V, int chunk, double u) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nch = (V + chunk - 1) / chunk;
  for (int ch = warp; ch < nch; ch += kFinWarps) {
    const int e0 = ch * chunk, e1 = min(V, e0 + chunk);
    float s = 0.f;
    for (int i = e0 + lane; i < e1; i += 32) s += wfn(i);
    const double t = warp_sum_d((double)s);
    if (lane == 0) sh.csum[ch] = t;
  }
  __syncthreads();
  if (warp == 0) {
    // total, then the first chunk whose running sum passes u S
    double tot = 0.0;
    for (int b = 0; b < nch; b += 32) {
      const double x = b + lane < nch ? sh.csum[b + lane] : 0.0;
      tot += __shfl_sync(0xffffffffu, fv_warp_incl_scan(x), 31);
    }
    const double tgt = u * tot;
    int cross = -1, lastpos = -1;
    double before = 0.0, run = 0.0;
    for (int b = 0; b < nch && cross < 0; b += 32) {
      const double x = b + lane < nch ? sh.csum[b + lane] : 0.0;
      const double incl = fv_warp_incl_scan(x);
      const unsigned hit = __ballot_sync(0xffffffffu, b + lane < nch && run + incl > tgt);
      if (hit) {
        const int l = __ffs(hit) - 1;
        cross = b + l;
        before = run + __shfl_sync(0xffffffffu, incl - x, l);
      }
      const unsigned pos = __ballot_sync(0xffffffffu, b + lane < nch && x > 0.0);
      if (pos) lastpos = b + 31 - __clz(pos);
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    int found = -1;
    const int ch = cross >= 0 ? cross : lastpos;
    if (ch >= 0) {
      // rescan chunk ch: lane l a contiguous run of chunk / 32 elements
      const int per = chunk / 32;
      const int e0 = ch * chunk + lane * per, e1 = min(V, e0 + per);
      double ls = 0.0;
      int lp = -1;
      for (int i = e0; i < e1; ++i) {
        const float w = wfn(i);
        ls += (double)w;
        if (w > 0.f) lp = i;
      }
      const double inc = fv_warp_incl_scan(ls);
      int f = 0x7fffffff;
      if (cross >= 0 && before + inc > tgt) {
        double r = before + (inc - ls);
        for (int i = e0; i < e1; ++i) {
          r += (double)wfn(i);
          if (r > tgt) {
            f = i;
            break;
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        f = min(f, __shfl_xor_sync(0xffffffffu, f, o));
        lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
      }
      found = f != 0x7fffffff ? f : lp;
    }
    if (lane == 0) sh.chosen = found;
  }
  __syncthreads();
  const int r = sh.chosen;
  __syncthreads();
  return r;
}

}  // namespace

// One CTA per sequence: the decisions of spec_verify from the GEMM's partials.
template <int MODE>
__global__ void __launch_bounds__(kFinThreads) fv_finish_kernel(const FvArgs g, FvOut o) {
  extern __shared__ __align__(16) unsigned char fin_smem[];
  FinShared &sh = *reinterpret_cast<FinShared *>(fin_smem);
  const int b = blockIdx.x, k = g.k, V = g.V;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float c = g.c;
  grid_dep_wait();
  grid_dep_launch();
  // combine each row's partials in vocabulary-tile order (fixed lane order)
  for (int j = warp; j <= k; j += kFinWarps) {
    const float4 *pp = g.part + (size_t)(b * (k + 1) + j) * g.n_vt;
    float m = -INFINITY;
    int idx = 0x7fffffff;
    for (int t = lane; t < g.n_vt; t += 32) {
      const float4 p = __ldcg(&pp[t]);
      if (MODE == 0) argmax_merge(m, idx, p.x, __float_as_int(p.y));
      else m = fmaxf(m, p.x);
    }
    if (MODE == 0) {
      warp_argmax(m, idx);
    } else {
      m = warp_max(m);
    }
    double z = 0.0;
    if (MODE == 1 && m != -INFINITY)
      for (int t = lane; t < g.n_vt; t += 32) {
        const float4 p = __ldcg(&pp[t]);
        if (p.x != -INFINITY) z += (double)p.y * (double)ex2f((p.x - m) * c);
      }
    z = warp_sum_d(z);
    if (lane == 0) {
      sh.M[j] = m;
      sh.Z[j] = z;
      sh.I[j] = idx;
    }
  }
  __syncthreads();
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
    // position by position: the draft row's normaliser, then u q(d) < p(d)
    int rej = -1;
    float Ml = -INFINITY;
    double Zl = 0.0;
    const float *drow = nullptr;
    for (int j = 0; j < k; ++j) {
      const int d = __ldg(&dt[j]);
      drow = g.draft + ((size_t)b * k + j) * V;
      float m = -INFINITY, s = 0.f;
      for (int i = threadIdx.x; i < V; i += kFinThreads) {  // online (max, sum) of this thread's elements
        const float x = __ldcg(drow + i);
        if (x > m) {
          if (m != -INFINITY) s *= ex2f((m - x) * c);
          m = x;
        }
        if (m != -INFINITY) s += ex2f((x - m) * c);
      }
      block_lse(sh, m, s, c, Ml, Zl);
      if (d < 0 || d >= V) {
        flags |= kStatusBadToken;
        rej = j;
        break;
      }
      if (!(sh.M[j] > -INFINITY) || !(Ml > -INFINITY)) flags |= kStatusNonFinite;
      const double td = (double)__ldcg(g.tgt + (size_t)(b * (k + 1) + j) * V + d);
      const double ld = (double)__ldcg(drow + d);
      const double p = exp2((td - (double)sh.M[j]) * (double)c) / sh.Z[j];
      const double q = exp2((ld - (double)Ml) * (double)c) / Zl;
      const double ua = (double)__ldg(&g.u_accept[(size_t)b * k + j]);
      if (!(ua * q < p)) {
        rej = j;
        break;
      }
    }
    const double uf = (double)__ldg(&g.u_final[b]);
    int chosen;
    if (rej >= 0) {
      n_acc = rej;
      const float *trow = g.tgt + (size_t)(b * (k + 1) + rej) * V;
      const float Mt = sh.M[rej], iZt = (float)(1.0 / sh.Z[rej]), iZl = (float)(1.0 / Zl);
      auto resid = [&](int i) -> float {
        const float p = ex2f((__ldcg(trow + i) - Mt) * c) * iZt;
        return fmaxf(0.f, p - ex2f((__ldcg(drow + i) - Ml) * c) * iZl);
      };
      chosen = block_inverse_cdf(sh, resid, V, g.chunk, uf);
      if (chosen < 0) {  // p = q everywhere: draw from p itself
        auto pw = [&](int i) -> float { return ex2f((__ldcg(trow + i) - Mt) * c) * iZt; };
        chosen = block_inverse_cdf(sh, pw, V, g.chunk, uf);
      }
    } else {
      n_acc = k;
      const float *trow = g.tgt + (size_t)(b * (k + 1) + k) * V;
      const float Mt = sh.M[k];
      auto pw = [&](int i) -> float { return ex2f((__ldcg(trow + i) - Mt) * c); };
      chosen = block_inverse_cdf(sh, pw, V, g.chunk, uf);
    }
    if (chosen < 0) {
      flags |= kStatusNonFinite;
      chosen = 0;
    }
    tok = chosen;
  }
  if (threadIdx.x <= k) {
    const int t = threadIdx.x;
    o.out_tok[(size_t)b * (k + 1) + t] = t < n_acc ? __ldg(&dt[t]) : (t == n_acc ? tok : -1);
  }
  if (threadIdx.x == 0) {
    o.accept_len[b] = n_acc + 1;
    o.num_accepted[b] = n_acc;
    if (flags) set_status(g.status, flags);
  }
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
  if (mode == 1) n += up256(Na * (size_t)V * 4);  // stored logits (the draws read them)
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
  p += 256;
  g.part = reinterpret_cast<float4 *>(p);
  p += up256((size_t)g.Na * g.n_vt * 16);
  g.tgt = fc.mode == 1 ? reinterpret_cast<float *>(p) : nullptr;
  int chunk = (fc.V + kMaxChunks - 1) / kMaxChunks;
  chunk = chunk < 512 ? 512 : (chunk + 31) / 32 * 32;
  g.chunk = chunk;

  FvMaps maps{};
  if (!make_bf16_map(&maps.hid, fc.hidden, (uint64_t)fc.d, (uint64_t)g.Na, (uint64_t)fc.d, kMRows))
    return cudaErrorInvalidValue;
  if (!make_bf16_map(&maps.head, fc.head, (uint64_t)fc.d, (uint64_t)fc.V, (uint64_t)fc.d, kVt))
    return cudaErrorInvalidValue;

  const size_t smem = (size_t)g.stages * fv_stage_bytes(g.n_mt) + (size_t)(2 * g.stages + 4) * 8 + 16 + 1024;
  const int sms = fv_sms();
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(g.nunits < sms ? g.nunits : sms));
  cfg.blockDim = dim3(kFvThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.numAttrs = 0;
  note_launch();
  cudaError_t e = fc.mode == 1 ? cudaLaunchKernelEx(&cfg, fv_gemm_kernel<1>, maps, g)
                               : cudaLaunchKernelEx(&cfg, fv_gemm_kernel<0>, maps, g);
  if (e != cudaSuccess) return e;

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
  return fc.mode == 1 ? cudaLaunchKernelEx(&fcfg, fv_finish_kernel<1>, g, o)
                      : cudaLaunchKernelEx(&fcfg, fv_finish_kernel<0>, g, o);
}

}  // namespace mtp
