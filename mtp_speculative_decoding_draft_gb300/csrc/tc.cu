// The draft chain for batches of several sequences on the fifth-generation
// tensor cores.  A weight-streaming GEMV reads every weight matrix once per
// couple of sequences; here each depth reads it once for the whole batch:
//
//   out[b, n] = sum_k W[n, k] a[b, k]         (fp32 accumulation in TMEM)
//
// with the fp32 activation a split into three bf16 terms a = hi + mid + lo
// (hi = bf16(a), mid = bf16(a - hi), lo = bf16(a - hi - mid)): the three
// terms' products keep the activation's 24 significant bits (for batches of
// up to 64 one tcgen05.mma of N = 3 nb per k-step, the terms side by side in
// N; beyond, three of N = nb), so the products match an fp32 GEMV ("The Tiny
// Draft Model Hidden Inside Qwen", opening section: the module is one
// full-attention block; the same module is applied k times, "One step deeper
// than the main model").
//
// Per depth: prep(FC input) -> GEMM FC -> mid(x0, QKV input) -> GEMM QKV ->
// mid(q, K/V append) -> attention -> prep(WO input) -> GEMM WO -> mid(x1,
// gate/up input) -> GEMM gate/up -> mid(SwiGLU, down input) -> GEMM down ->
// mid(x2, LM-head input) -> GEMM LM head -> draft-token selection.  The GEMM
// is split over K where the output has few 128-row tiles; the mid kernels (one
// CTA per sequence) sum the split-K partials and apply the same epilogues as
// the GEMV path (residual adds, SwiGLU, bf16 K/V append) before writing the
// next GEMM's bf16 terms.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdlib.h>

#include <mutex>

#include "common.cuh"
#include "draft_ops.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace mtp {

namespace {

constexpr int kTcThreads = 192;  // warp 0 TMA, warp 1 MMA and TMEM, warps 2-5 read TMEM back
constexpr int kTileM = 128;      // output rows per tile (MMA M)
constexpr int kBK = 64;          // K per stage: one 128-byte swizzle row of bf16
constexpr uint32_t kWTileBytes = kTileM * kBK * 2;
// stage ring budget: the 227 KB a CTA may hold, less the 1024-byte alignment
// pad and the barriers
constexpr int kSmemBudget = 227 * 1024 - 1024 - 256;
constexpr int kMaxSplits = 32;
constexpr int kPrepThreads = 256;

struct TcMaps {
  CUtensorMap w[3];  // weight row blocks (QKV: wq, wk, wv; gate/up: wgate, wup)
  CUtensorMap a[3];  // activation terms hi, mid, lo
};

struct TcGemmArgs {
  int nmaps, mt;                   // weight maps; 128-row tiles per CTA (sharing each activation stage)
  int rows[3], groups[3], base[3];  // rows and mt-tile groups of each map; its first output row
  int ks, kb_per, kbs;             // K splits, 64-wide k-blocks per split and in all
  int nb, stages;                  // padded batch rows, pipeline depth
  int B, arow0;                    // batch rows, first batch row of this group
  int nunits;                      // (row group, K split) units, taken by the CTAs in turn
  float *out;                      // element (split s, batch b, row n) at out + s*sstride + b*bstride + n
  size_t sstride, bstride;
  int *status;
};

__host__ __device__ inline uint32_t a_tile_bytes(int nb) { return (uint32_t)nb * kBK * 2; }
constexpr int kTerms = 3;
__host__ __device__ inline uint32_t stage_bytes(int nb, int mt) {
  return (uint32_t)mt * kWTileBytes + kTerms * a_tile_bytes(nb);
}
// TMEM columns of one accumulator buffer: mt tiles of N columns each
__host__ __device__ inline int tmem_cols(int n_mma, int mt) {
  int n = 32;
  while (n < n_mma * mt) n *= 2;
  return n;
}

}  // namespace

// ---------------------------------------------------------------- GEMM kernel

// A unit of work: one group of MT row tiles of map m and one K split.
struct TcUnit {
  int m, row0, split, kb0, nkb;
};

__device__ __forceinline__ TcUnit tc_unit(const TcGemmArgs &g, int u) {
  TcUnit w;
  w.split = u % g.ks;
  int grp = u / g.ks, m = 0;
  while (m < g.nmaps - 1 && grp >= g.groups[m]) {
    grp -= g.groups[m];
    ++m;
  }
  w.m = m;
  w.row0 = grp * g.mt * kTileM;  // within map m
  w.kb0 = w.split * g.kb_per;
  w.nkb = max(0, min(g.kb_per, g.kbs - w.kb0));
  return w;
}

// Persistent: CTA c takes units c, c + gridDim.x, ...  The stage ring runs on
// across units; the accumulator is double-buffered in TMEM (when two fit), so
// that the epilogue of one unit overlaps the MMAs of the next.
// FUSE: the three activation terms lie back to back in a stage, one K-major
// operand of 3 nb rows, so one MMA of N = 3 nb per k-step and tile reads the
// weight tile once (three MMAs of N = nb would read it three times); each
// term accumulates in its own block of nb columns and the epilogue adds them.
template <bool FUSE>
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(const __grid_constant__ TcMaps maps,
                                                                  const TcGemmArgs g) {
  trace_start(kTkTcGemm);
  extern __shared__ unsigned char smem_raw[];
  // SW128 tiles need 1024-byte alignment
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  unsigned char *sm = smem_raw + pad;
  const int S = g.stages;
  const int MT = g.mt;
  const uint32_t ab = a_tile_bytes(g.nb), sb = stage_bytes(g.nb, MT), wb = (uint32_t)MT * kWTileBytes;
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + (size_t)S * sb);
  uint64_t *empty = full + S;
  uint64_t *done = empty + S;   // [2] accumulator buffer ready for the epilogue
  uint64_t *tfree = done + 2;   // [2] accumulator buffer read back
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tfree + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nmma = FUSE ? kTerms * g.nb : g.nb;  // accumulator columns of one tile
  const int ncols = tmem_cols(nmma, MT);
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
      // Weights do not depend on the previous kernel: the first unit's first
      // stages are requested before waiting for it; activations only after.
      const uint64_t pol_w = l2_policy_evict_first(), pol_a = l2_policy_evict_last();
      const TcUnit u0 = tc_unit(g, blockIdx.x);
      const int pre = (int)blockIdx.x < g.nunits ? min(S, u0.nkb) : 0;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], sb);
        for (int t = 0; t < MT; ++t)
          tma_load_2d(sm + (size_t)i * sb + t * kWTileBytes, &maps.w[u0.m], (u0.kb0 + i) * kBK,
                      u0.row0 + t * kTileM, &full[i], pol_w);
      }
      grid_dep_wait();
      bool ok = true;
      uint32_t i = 0;  // k-blocks issued by this CTA
      for (int u = blockIdx.x, n = 0; u < g.nunits && ok; u += gridDim.x, ++n) {
        const TcUnit w = tc_unit(g, u);
        for (int kb = 0; kb < w.nkb && ok; ++kb, ++i) {
          const int s = (int)(i % S);
          unsigned char *st = sm + (size_t)s * sb;
          const int x = (w.kb0 + kb) * kBK;
          if (!(n == 0 && kb < pre)) {
            if (i >= (uint32_t)S) ok = mbar_wait(&empty[s], ((i / S) - 1u) & 1u, g.status);
            if (!ok) break;
            mbar_arrive_expect_tx(&full[s], sb);
            for (int t = 0; t < MT; ++t)
              tma_load_2d(st + t * kWTileBytes, &maps.w[w.m], x, w.row0 + t * kTileM, &full[s], pol_w);
          }
#pragma unroll
          for (int tt = 0; tt < kTerms; ++tt)
            tma_load_2d(st + wb + tt * ab, &maps.a[tt], x, g.arow0, &full[s], pol_a);
        }
      }
      if (!ok)  // let copies still in flight land before the CTA exits
        for (uint32_t q = i > (uint32_t)S ? i - S : 0u; q < i; ++q)
          if (!mbar_wait(&full[q % S], (q / S) & 1u, g.status)) break;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTileM, nmma);
      bool ok = true;
      uint32_t i = 0;  // k-blocks consumed
      for (int u = blockIdx.x, n = 0; u < g.nunits && ok; u += gridDim.x, ++n) {
        const TcUnit w = tc_unit(g, u);
        const int buf = n % nbuf;
        if (n >= nbuf) ok = mbar_wait(&tfree[buf], (uint32_t)((n / nbuf) - 1) & 1u, g.status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)(buf * ncols);
        for (int kb = 0; kb < w.nkb && ok; ++kb, ++i) {
          const int s = (int)(i % S);
          ok = mbar_wait(&full[s], (i / S) & 1u, g.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t st = smem_u32(sm + (size_t)s * sb);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)  // 16 bf16 = 32 bytes: +2 in the >>4 address field
            for (int t = 0; t < MT; ++t) {  // tile t accumulates in columns [t nmma, (t + 1) nmma)
              const uint64_t dw = sw128_kmajor_desc(st + t * kWTileBytes) + 2 * kk;
              if (FUSE) {
                mma_bf16(acc + (uint32_t)(t * nmma), dw, sw128_kmajor_desc(st + wb) + 2 * kk, idesc,
                         (kb | kk) != 0 ? 1u : 0u);
              } else {
#pragma unroll
                for (int tt = 0; tt < kTerms; ++tt)
                  mma_bf16(acc + (uint32_t)(t * nmma), dw, sw128_kmajor_desc(st + wb + tt * ab) + 2 * kk, idesc,
                           (kb | kk | tt) != 0 ? 1u : 0u);
              }
            }
          mma_commit(&empty[s]);  // the stage is free once these MMAs have read it
        }
        mma_commit(&done[buf]);
      }
    }
  } else {
    // read the accumulators back: warp w reads TMEM lanes 32 (w % 4) .. + 31
    const int q = warp & 3;
    bool ok = true;
    for (int u = blockIdx.x, n = 0; u < g.nunits && ok; u += gridDim.x, ++n) {
      const TcUnit w = tc_unit(g, u);
      const int buf = n % nbuf;
      ok = mbar_wait(&done[buf], (uint32_t)(n / nbuf) & 1u, g.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t acc = tmem + (uint32_t)(buf * ncols);
      for (int t = 0; t < MT; ++t) {
        const int row = w.row0 + t * kTileM + q * 32 + lane;
        const bool valid = w.nkb > 0 && row < g.rows[w.m];
        float *o = g.out + (size_t)w.split * g.sstride + (size_t)g.base[w.m] + row;
        for (int c0 = 0; c0 < g.nb; c0 += 32) {
          float v[32];
          const uint32_t ta = acc + ((uint32_t)(q * 32) << 16) + (uint32_t)(t * nmma + c0);
          tmem_ld32(ta, v);
          if (FUSE) {  // hi + mid + lo products
            float v1[32];
            tmem_ld32(ta + (uint32_t)g.nb, v1);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] += v1[i];
            tmem_ld32(ta + (uint32_t)(2 * g.nb), v1);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] += v1[i];
          }
          if (valid) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int b = g.arow0 + c0 + i;
              if (b < g.B) o[(size_t)b * g.bstride] = v[i];
            }
          }
        }
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
  trace_end(kTkTcGemm);
}

// ---------------------------------------------------------------- per-sequence kernels

namespace {

// Eight values into the three bf16 terms of activation row b at column col.
__device__ __forceinline__ void store_split8(const TcBufs &t, int b, int col, const float *v) {
  uint32_t w[kTerms][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float r0 = v[2 * i], r1 = v[2 * i + 1];
#pragma unroll
    for (int tt = 0; tt < kTerms; ++tt) {
      const __nv_bfloat16 h0 = __float2bfloat16_rn(r0), h1 = __float2bfloat16_rn(r1);
      w[tt][i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
      r0 -= __bfloat162float(h0);
      r1 -= __bfloat162float(h1);
    }
  }
  const size_t off = (size_t)b * t.kmax + col;
#pragma unroll
  for (int tt = 0; tt < kTerms; ++tt)
    *reinterpret_cast<uint4 *>(t.a[tt] + off) = make_uint4(w[tt][0], w[tt][1], w[tt][2], w[tt][3]);
}

// Sum over the K splits of eight consecutive outputs (row n) of sequence b.
// The split-K partials of eight outputs summed in split order; the splits'
// loads four at a time, issued together (one after another they would cost
// an L2 round trip per split).
__device__ __forceinline__ void sum8(const float *part, int ks, size_t sstride, size_t boff, float *y) {
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = 0.f;
  for (int s0 = 0; s0 < ks; s0 += 4) {
    float v[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (s0 + u < ks) load8_f32(part + (size_t)(s0 + u) * sstride + boff, v[u]);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (s0 + u < ks)
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] += v[u][i];
  }
}

__device__ __forceinline__ float sumsq8(const float *v, float acc) {
#pragma unroll
  for (int i = 0; i < 8; ++i) acc = fmaf(v[i], v[i], acc);
  return acc;
}

}  // namespace

// Input of the input projection: [rms(E[tok]) g_emb ; rms(x) g_hid], x = h at
// depth 0, else the previous depth's x2.
__global__ void __launch_bounds__(kPrepThreads) tc_prep_fc_kernel(DraftCtx c, TcBufs t) {
  trace_start(kTkTcAux);
  __shared__ float red[2 * kGemvWarps];
  const int b = blockIdx.x, d = c.d;
  grid_dep_wait();
  grid_dep_launch();
  if (c.k_eff && c.j == 0 && threadIdx.x == 0) {  // dynamic draft length: every sequence drafting
    c.k_eff[b] = c.k;
    if (b == 0) *c.n_active = (unsigned)c.B;
  }
  if (c.seq_order && c.j == 0) {
    // this sequence's place in the longest-context-first order (ties by index)
    const int L = __ldg(&c.ctx_len[b]);
    int before = 0;
    for (int o = threadIdx.x; o < c.B; o += kPrepThreads) {
      const int Lo = __ldg(&c.ctx_len[o]);
      before += (Lo > L || (Lo == L && o < b)) ? 1 : 0;
    }
    before = (int)block_sum_256((float)before, red);
    if (threadIdx.x == 0) c.seq_order[before] = b;
    __syncthreads();
  }
  const int tok = depth_token(c, b);
  const uint16_t *e = c.E + (size_t)tok * d;
  float s0 = 0.f, s1 = 0.f;
  for (int i = threadIdx.x * 8; i < d; i += kPrepThreads * 8) {
    float v[8], x[8];
    load8_bf16(e + i, v);
    if (c.j == 0) load8_bf16(c.h + (size_t)b * d + i, x);
    else load8_f32(c.x2 + (size_t)b * d + i, x);
    s0 = sumsq8(v, s0);
    s1 = sumsq8(x, s1);
  }
  s0 = block_sum_256(s0, red);
  s1 = block_sum_256(s1, red + kGemvWarps);
  const float r0 = rsqrtf(s0 / (float)d + c.eps), r1 = rsqrtf(s1 / (float)d + c.eps);
  for (int i = threadIdx.x * 8; i < d; i += kPrepThreads * 8) {
    float v[8], x[8], g[8];
    load8_bf16(e + i, v);
    load8_bf16(c.g_emb + i, g);
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = v[q] * r0 * g[q];
    store_split8(t, b, i, v);
    if (c.j == 0) load8_bf16(c.h + (size_t)b * d + i, x);
    else load8_f32(c.x2 + (size_t)b * d + i, x);
    load8_bf16(c.g_hid + i, g);
#pragma unroll
    for (int q = 0; q < 8; ++q) x[q] = x[q] * r1 * g[q];
    store_split8(t, b, d + i, x);
  }
  trace_end(kTkTcAux);
}

// Input of the output projection: the attention output as is.
__global__ void __launch_bounds__(kPrepThreads) tc_prep_wo_kernel(DraftCtx c, TcBufs t) {
  trace_start(kTkTcAux);
  const int b = blockIdx.x, n = c.Hq * c.Dh;
  grid_dep_wait();
  grid_dep_launch();
  for (int i = threadIdx.x * 8; i < n; i += kPrepThreads * 8) {
    float v[8];
    load8_f32(c.o + (size_t)b * n + i, v);
    store_split8(t, b, i, v);
  }
  trace_end(kTkTcAux);
}

// Sum the split-K partials of OP for sequence b (CTA r of the sequence's
// cluster takes the r-th share of the columns), apply OP's epilogue and write
// the next GEMM's input terms.
template <int OP>
__global__ void __launch_bounds__(kPrepThreads) tc_mid_kernel(DraftCtx c, TcBufs t, int ks, int N) {
  trace_start(kTkTcAux);
  __shared__ float red[kGemvWarps];
  __shared__ float css;  // this CTA's sum of squares, read by the cluster's other CTAs
  const int b = blockIdx.y, d = c.d, NC = (int)gridDim.x, r = (int)blockIdx.x;
  const size_t sstride = (size_t)c.B * N, boff = (size_t)b * N;
  // this CTA's share of the op's columns, in whole groups of eight
  const int ncol = OP == OP_QKV ? N : (OP == OP_GATEUP ? c.F : d);
  const int g8 = ncol / 8, c0 = 8 * (int)(((long long)r * g8) / NC), c1 = 8 * (int)(((long long)(r + 1) * g8) / NC);
  grid_dep_wait();
  grid_dep_launch();
  if (OP == OP_QKV) {
    const int nq = c.Hq * c.Dh, nkv = c.Hkv * c.Dh;
    int L = __ldg(&c.ctx_len[b]);
    if (L < 0 || L + c.k > c.Lmax) {
      if (threadIdx.x == 0 && r == 0) set_status(c.status, kStatusBadCtx);
      L = min(max(L, 0), c.Lmax - c.k);
    }
    for (int i = c0 + threadIdx.x * 8; i < c1; i += kPrepThreads * 8) {
      float y[8];
      sum8(t.part, ks, sstride, boff + i, y);
      if (i < nq) {
        *reinterpret_cast<float4 *>(c.q + (size_t)b * nq + i) = make_float4(y[0], y[1], y[2], y[3]);
        *reinterpret_cast<float4 *>(c.q + (size_t)b * nq + i + 4) = make_float4(y[4], y[5], y[6], y[7]);
      } else {
        int rr = i - nq;
        uint16_t *cache = rr < nkv ? c.kc : c.vc;
        if (rr >= nkv) rr -= nkv;
        const int kvh = rr / c.Dh, dd = rr % c.Dh;  // 8 | Dh: the eight stay in one head
        uint16_t *dst = cache + (((size_t)b * c.Hkv + kvh) * c.Lmax + L + c.jc) * c.Dh + dd;
        if (in_bounds(L + c.jc < c.Lmax && kvh < c.Hkv && dd + 8 <= c.Dh, c.status))
#pragma unroll
          for (int q = 0; q < 8; ++q) dst[q] = __bfloat16_as_ushort(__float2bfloat16_rn(y[q]));
      }
    }
    trace_end(kTkTcAux);
    return;
  }
  if (OP == OP_GATEUP) {  // SwiGLU: gate rows [0, F), up rows [F, 2F)
    const int F = c.F;
    for (int i = c0 + threadIdx.x * 8; i < c1; i += kPrepThreads * 8) {
      float gt[8], up[8];
      sum8(t.part, ks, sstride, boff + i, gt);
      sum8(t.part, ks, sstride, boff + F + i, up);
#pragma unroll
      for (int q = 0; q < 8; ++q) gt[q] = silu_f(gt[q]) * up[q];
      store_split8(t, b, i, gt);
    }
    trace_end(kTkTcAux);
    return;
  }
  // FC -> x0, WO -> x1 = x0 + y, DOWN -> x2 = x1 + y; then the next input
  // rms(x) g, the sum of squares added over the cluster's CTAs in rank order
  float *xo = OP == OP_FC ? c.x0 : (OP == OP_WO ? c.x1 : c.x2);
  const float *xr = OP == OP_WO ? c.x0 : c.x1;
  const uint16_t *gain = OP == OP_FC ? c.g_attn : (OP == OP_WO ? c.g_mlp : c.g_final);
  float ss = 0.f;
  for (int i = c0 + threadIdx.x * 8; i < c1; i += kPrepThreads * 8) {
    float y[8];
    sum8(t.part, ks, sstride, boff + i, y);
    if (OP != OP_FC) {
      float rv[8];
      load8_f32(xr + (size_t)b * d + i, rv);
#pragma unroll
      for (int q = 0; q < 8; ++q) y[q] += rv[q];
    }
    *reinterpret_cast<float4 *>(xo + (size_t)b * d + i) = make_float4(y[0], y[1], y[2], y[3]);
    *reinterpret_cast<float4 *>(xo + (size_t)b * d + i + 4) = make_float4(y[4], y[5], y[6], y[7]);
    ss = sumsq8(y, ss);
  }
  ss = block_sum_256(ss, red);
  if (threadIdx.x == 0) css = ss;
  cluster_sync();  // every CTA's sum is in place; this CTA's x writes are visible to it
  float tot = 0.f;
  for (int q = 0; q < NC; ++q) tot += *dsmem_ptr(&css, (uint32_t)q);
  const float rs = rsqrtf(tot / (float)d + c.eps);
  for (int i = c0 + threadIdx.x * 8; i < c1; i += kPrepThreads * 8) {
    float y[8], g[8];
    load8_f32(xo + (size_t)b * d + i, y);
    load8_bf16(gain + i, g);
#pragma unroll
    for (int q = 0; q < 8; ++q) y[q] = y[q] * rs * g[q];
    store_split8(t, b, i, y);
  }
  cluster_sync();  // no CTA leaves before its peers have read its sum
  trace_end(kTkTcAux);
}

// Draft-token selection over the batch's logits rows, in two launches.
// tc_select_part_kernel: one CTA per 4096 elements of a row, a warp per
// 1024-element sub-segment: its (max, lowest argmax) and, in stochastic mode,
// sum exp2((x - max) c).  tc_select_fin_kernel: one warp per sequence
// combines the sub-segments in order -- the argmax, or the inverse CDF of
// softmax(x / T) at u_draft: float64 sub-segment masses, the crossing
// sub-segment rescanned in float64 (each lane a contiguous run of 32).
constexpr int kSelSub = 1024;
constexpr int kSelWarps = 4;
constexpr int kSelThreads = 32 * kSelWarps;

__host__ __device__ inline int sel_subs(int V) { return (V + kSelSub - 1) / kSelSub; }

__global__ void __launch_bounds__(kSelThreads) tc_select_part_kernel(DraftCtx c, const float *logits, size_t bstride,
                                                                     float4 *part) {
  trace_start(kTkTcAux);
  const int b = blockIdx.y, V = c.Vd, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int q = blockIdx.x * kSelWarps + warp, nq = sel_subs(V);
  grid_dep_wait();
  grid_dep_launch();
  if (q >= nq) return;
  const float *row = logits + (size_t)b * bstride;
  const int e0 = q * kSelSub, n = min(kSelSub, V - e0);
  float x[32];
  if ((reinterpret_cast<uintptr_t>(row + e0) & 15u) == 0 && n == kSelSub) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(row + e0) + lane + 32 * i);
      x[4 * i] = v.x;
      x[4 * i + 1] = v.y;
      x[4 * i + 2] = v.z;
      x[4 * i + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = 4 * (lane + 32 * i) + u;
        x[4 * i + u] = e < n ? __ldcg(row + e0 + e) : -INFINITY;
      }
  }
  // element 4 (lane + 32 i) + u of the sub-segment is x[4 i + u]
  float M = -INFINITY;
  int I = 0x7fffffff;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (x[i] > M) {  // ascending element order per lane: the first maximum stays
      M = x[i];
      I = e0 + 4 * (lane + 32 * (i >> 2)) + (i & 3);
    }
  warp_argmax(M, I);
  float sum = 0.f;
  if ((c.mode == 1 || c.k_eff) && M != -INFINITY) {
    const float cT = kLog2e / c.T, mc = M * cT;
#pragma unroll
    for (int i = 0; i < 32; ++i) sum += exp2f(fmaf(x[i], cT, -mc));
    sum = warp_sum(sum);
  }
  if (lane == 0 && in_bounds(b < c.B && q < nq, c.status)) part[(size_t)b * nq + q] = make_float4(M, __int_as_float(I), sum, 0.f);
  trace_end(kTkTcAux);
}

__global__ void __launch_bounds__(32) tc_select_fin_kernel(DraftCtx c, const float *logits, size_t bstride,
                                                           const float4 *part) {
  trace_start(kTkTcAux);
  const int b = blockIdx.x, V = c.Vd, lane = threadIdx.x, nq = sel_subs(V);
  grid_dep_wait();
  grid_dep_launch();
  const float4 *pp = part + (size_t)b * nq;
  // lane l owns sub-segments [l per, (l+1) per) in order
  const int per = (nq + 31) / 32, q0 = min(nq, lane * per), q1 = min(nq, q0 + per);
  float M = -INFINITY;
  int I = 0x7fffffff;
  for (int q = q0; q < q1; ++q) argmax_merge(M, I, pp[q].x, __float_as_int(pp[q].y));
  warp_argmax(M, I);
  int tok = I;
  const bool finite = !(M == -INFINITY || !(M == M));
  const float cT = kLog2e / c.T;
  // float64 masses of this lane's sub-segments, their inclusive scan and the
  // partition sum relative to the largest term
  double own = 0.0, incl = 0.0, Z = 0.0;
  int lastq = -1;
  if (finite && (c.mode == 1 || c.k_eff)) {
    for (int q = q0; q < q1; ++q) {
      const float4 v = pp[q];
      const double m = v.x == -INFINITY ? 0.0 : (double)v.z * (double)exp2f((v.x - M) * cT);
      own += m;
      if (m > 0.0) lastq = q;
    }
    incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    Z = __shfl_sync(0xffffffffu, incl, 31);
  }
  if (!finite) {
    if (lane == 0) set_status(c.status, kStatusNonFinite);
    tok = 0;
  } else if (c.mode == 1) {
    const double target = (double)__ldg(&c.u_draft[b * c.k + c.j]) * Z;
    int qs = -1;
    double before = 0.0;
    const unsigned cross = __ballot_sync(0xffffffffu, q1 > q0 && incl > target);
    if (cross) {
      const int cl = __ffs(cross) - 1;
      if (lane == cl) {
        double cum = incl - own;
        for (int q = q0; q < q1; ++q) {
          const float4 v = pp[q];
          const double m = v.x == -INFINITY ? 0.0 : (double)v.z * (double)exp2f((v.x - M) * cT);
          if (cum + m > target) {
            qs = q;
            before = cum;
            break;
          }
          cum += m;
        }
      }
      qs = __shfl_sync(0xffffffffu, qs, cl);
      before = __shfl_sync(0xffffffffu, before, cl);
    }
    int ql = lastq;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ql = max(ql, __shfl_xor_sync(0xffffffffu, ql, o));
    const bool crossing = qs >= 0;
    const int qr = crossing ? qs : ql;
    int found = 0x7fffffff, lastpos = -1;
    if (qr >= 0) {
      // rescan sub-segment qr: lane l takes elements [32 l, 32 l + 32), float64
      const float *row = logits + (size_t)b * bstride;
      const int e0 = qr * kSelSub, n = min(kSelSub, V - e0);
      float w[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int e = 32 * lane + i;
        w[i] = e < n ? exp2f((__ldcg(row + e0 + e) - M) * cT) : 0.f;
      }
      double ls = 0.0;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        ls += (double)w[i];
        if (w[i] > 0.f) lastpos = e0 + 32 * lane + i;
      }
      double inc = ls;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
      }
      if (crossing && before + inc > target) {
        double run = before + (inc - ls);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          run += (double)w[i];
          if (found == 0x7fffffff && run > target && 32 * lane + i < n) found = e0 + 32 * lane + i;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        found = min(found, __shfl_xor_sync(0xffffffffu, found, o));
        lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, o));
      }
    }
    tok = found != 0x7fffffff ? found : (lastpos >= 0 ? lastpos : I);
  }
  if (finite) tok = vocab_id(c, tok);  // head row -> vocabulary id
  if (lane == 0 && in_bounds(b < c.B && c.j < c.k, c.status)) c.draft_tok[b * c.k + c.j] = tok;
  if (lane == 0 && c.k_eff && finite) stop_check(c, b, 1.0 / Z);
  trace_end(kTkTcAux);
}

// A reduced draft vocabulary: head row i's logit to its vocabulary id in the
// caller's full-vocabulary logits (the other ids hold -inf from the start of
// the call).
__global__ void __launch_bounds__(256) tc_scatter_logits_kernel(DraftCtx c, const float *lg) {
  trace_start(kTkTcAux);
  const int b = blockIdx.y;
  grid_dep_wait();
  grid_dep_launch();
  for (int i = blockIdx.x * 256 + threadIdx.x; i < c.Vd; i += gridDim.x * 256) {
    const int v = vocab_id(c, i);
    if (v >= 0) c.logits[((size_t)b * c.k + c.j) * c.V + v] = __ldcg(&lg[(size_t)b * c.Vd + i]);
  }
  trace_end(kTkTcAux);
}

// ---------------------------------------------------------------- host side

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn();

}  // namespace

bool make_bf16_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t ld, uint32_t box_rows);

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t ld, uint32_t box_rows) {
  return make_bf16_map(m, base, cols, rows, ld, box_rows);
}

}  // namespace

// 2-D bf16 map over a row-major [rows, cols] matrix with row stride ld
// (elements), boxes of box_rows x 64 columns, 128-byte swizzle.
bool make_bf16_map(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t ld, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {ld * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

struct OpShape {
  int nmaps;
  const uint16_t *w[3];
  int rows[3];
  int K;
};

OpShape op_shape(const DraftCtx &c, int op) {
  OpShape s{};
  s.nmaps = 1;
  switch (op) {
    case OP_FC: s.w[0] = c.fc; s.rows[0] = c.d; s.K = 2 * c.d; break;
    case OP_QKV:
      s.nmaps = 3;
      s.w[0] = c.wq; s.rows[0] = c.Hq * c.Dh;
      s.w[1] = c.wk; s.rows[1] = c.Hkv * c.Dh;
      s.w[2] = c.wv; s.rows[2] = c.Hkv * c.Dh;
      s.K = c.d;
      break;
    case OP_WO: s.w[0] = c.wo; s.rows[0] = c.d; s.K = c.Hq * c.Dh; break;
    case OP_GATEUP:
      s.nmaps = 2;
      s.w[0] = c.wgate; s.rows[0] = c.F;
      s.w[1] = c.wup; s.rows[1] = c.F;
      s.K = c.d;
      break;
    case OP_DOWN: s.w[0] = c.wdown; s.rows[0] = c.d; s.K = c.F; break;
    default: s.w[0] = c.head; s.rows[0] = c.Vd; s.K = c.d; break;
  }
  return s;
}

int op_rows(const OpShape &s) {
  int n = 0;
  for (int i = 0; i < s.nmaps; ++i) n += s.rows[i];
  return n;
}

int op_groups(const OpShape &s, int mt) {
  int n = 0;
  for (int i = 0; i < s.nmaps; ++i) n += ((s.rows[i] + kTileM - 1) / kTileM + mt - 1) / mt;
  return n;
}

int num_sms() {
  static int sms = 0;
  if (sms <= 0 && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess) sms = 0;
  return sms > 0 ? sms : 152;
}

// K splits of an op with `groups` row groups, whole k-blocks per split.  The
// persistent CTAs take the (group, split) units in turn, so the busiest CTA
// runs ceil(units / SMs) units of kb_per k-blocks each, plus a little per
// unit (the accumulator read-back and the turn to the next unit; half a
// k-block here).  The split count minimises that; a larger count must gain
// 5% over a smaller one, since it leaves more partials to sum.  (A unit count
// just above the SM count would run a second wave of a few units.)
// MTP_TC_SPLITS fixes the count.
void op_splits(int groups, int K, int sms, int *ks, int *kb_per) {
  const int kbs = K / kBK;
  const char *v = getenv("MTP_TC_SPLITS");
  if (v && *v) {
    int s = atoi(v);
    s = s < 1 ? 1 : (s > kMaxSplits ? kMaxSplits : (s > kbs ? kbs : s));
    *kb_per = (kbs + s - 1) / s;
    *ks = (kbs + *kb_per - 1) / *kb_per;
    return;
  }
  long best = -1;
  *ks = 1;
  *kb_per = kbs;
  for (int s = 1; s <= kMaxSplits && s <= kbs; ++s) {
    const int kb = (kbs + s - 1) / s;
    if ((kbs + kb - 1) / kb != s) continue;  // the same split as a smaller count
    const long waves = ((long)groups * s + sms - 1) / sms;
    const long cost = waves * (2L * kb + 1);
    if (best < 0 || 20 * cost < 19 * best) {
      best = cost;
      *ks = s;
      *kb_per = kb;
    }
  }
}

int batch_nb(int B) { return B <= 32 ? 32 : (B <= 64 ? 64 : 128); }

// Shared memory for the stage ring; MTP_TC_SMEM_KB lowers it.
int smem_budget() {
  const char *v = getenv("MTP_TC_SMEM_KB");
  const int kb = v && *v ? atoi(v) : 0;
  return kb > 0 && kb * 1024 < kSmemBudget ? kb * 1024 : kSmemBudget;
}

// One MMA of N = 3 nb per k-step and tile instead of three of N = nb: the
// weight tile is then read from shared memory once per k-step, not three
// times.  N is at most 256, so batches of up to 64 rows.  MTP_TC_FUSE=0 turns
// it off.
bool use_fuse(int nb) {
  const char *v = getenv("MTP_TC_FUSE");
  return kTerms * nb <= 256 && !(v && *v == '0');
}

// 128-row weight tiles per unit: each activation stage in shared memory serves
// mt tiles, so the activations are re-read from L2 once per mt tiles.  With
// three MMAs per tile the LM head takes 3 for batches of up to 32, 4 up to 64
// and 2 for 128-row batches (measured best on the deep-chain and batch-of-64
// workloads); the block's GEMMs take 2: smaller stages keep more of their few
// k-blocks in flight (measured: 2 beats 1 and 4 over the same workloads).
// With the fused MMA a tile's accumulator takes 3 nb TMEM columns: the LM head
// takes 3 tiles for batches of up to 32 (288 columns; three 60 KB stages fit)
// and 2 for 64 (384 columns), the block's GEMMs 2 (measured on the same
// workloads: 4 tiles at a batch of 32 leave room for two stages only, 1 tile
// re-reads the activations too often).  Two pipeline stages at least must fit.
// MTP_TC_MT and MTP_TC_MT_BLOCK override.
int op_mt(int nb, int op, bool fuse) {
  const char *v = getenv(op == OP_LMHEAD ? "MTP_TC_MT" : "MTP_TC_MT_BLOCK");
  int mt = 2;
  if (v && *v) mt = atoi(v);
  else if (op == OP_LMHEAD) mt = nb <= 32 ? 3 : (nb <= 64 && !fuse ? 4 : 2);
  if (mt < 1) mt = 1;
  const int nmma = fuse ? kTerms * nb : nb;
  while (mt > 1 && (2 * stage_bytes(nb, mt) > (uint32_t)kSmemBudget || nmma * mt > 512)) --mt;
  return mt;
}

template <class K, class... Args>
cudaError_t launch(K kern, dim3 grid, int threads, size_t smem, cudaStream_t s, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  note_launch();
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The mid kernels: one cluster of nc CTAs per sequence, each CTA a share of
// the columns (about 1024 of them, at most 8 CTAs).
template <int OP>
cudaError_t launch_mid(const DraftCtx &c, const TcBufs &t, int ks, int N, cudaStream_t s, bool pdl) {
  const int ncol = OP == OP_QKV ? N : (OP == OP_GATEUP ? c.F : c.d);
  int nc = ncol / 1024;
  nc = nc < 1 ? 1 : (nc > 8 ? 8 : nc);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(nc, c.B);
  cfg.blockDim = dim3(kPrepThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)nc;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  note_launch();
  return cudaLaunchKernelEx(&cfg, tc_mid_kernel<OP>, c, t, ks, N);
}

}  // namespace

// The tensor-core path needs K % 64 == 0 for every GEMM and weight blocks of
// at least one tile; it pays off from a handful of sequences up (the GEMV
// re-reads the weights once per couple of sequences).  MTP_TC_MIN_B overrides
// the threshold (0 turns the path off).
bool tc_shape_ok(const MtpShape &s) {
  if (s.d % kBK || (s.Hq * s.Dh) % kBK || s.F % kBK) return false;
  if (s.d < kTileM || s.F < kTileM || s.Hkv * s.Dh < kTileM || s.V < kTileM) return false;
  const char *v = getenv("MTP_TC_MIN_B");
  const int min_b = v && *v ? atoi(v) : 5;
  return min_b > 0 && s.B >= min_b;
}

bool tc_available() { return encode_fn() != nullptr; }

TcSizes tc_sizes(const MtpShape &s) {
  TcSizes z{};
  const int nb = batch_nb(s.B);
  z.rows = (s.B + nb - 1) / nb * nb;
  z.kmax = 2 * s.d;
  if (s.Hq * s.Dh > z.kmax) z.kmax = s.Hq * s.Dh;
  if (s.F > z.kmax) z.kmax = s.F;
  DraftCtx c{};
  c.d = s.d; c.Hq = s.Hq; c.Hkv = s.Hkv; c.Dh = s.Dh; c.F = s.F; c.V = s.V;
  // LM-head logits when the caller keeps none, then the selection's partials
  size_t part = ((size_t)s.B * s.V + 3) / 4 * 4 + (size_t)s.B * sel_subs(s.V) * 4;
  for (int op = OP_FC; op <= OP_DOWN; ++op) {
    const OpShape sh = op_shape(c, op);
    int ks, kb_per;
    const int nb = batch_nb(s.B);
    op_splits(op_groups(sh, op_mt(nb, op, use_fuse(nb))), sh.K, num_sms(), &ks, &kb_per);
    const size_t n = (size_t)ks * s.B * op_rows(sh);
    if (n > part) part = n;
  }
  z.part_floats = part;
  return z;
}

// The GEMM's shared-memory ceiling: what the largest stage ring needs (the
// ring budget with its alignment pad and barriers), or the ring budget that
// MTP_TC_SMEM_KB sets.
cudaError_t tc_set_attributes() {
  const int bytes = smem_budget() + 1024 + 256;
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(tc_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

namespace {

// One GEMM: out[s][b][n] = W[n, K-range s] . a[b, K-range s] for every
// 128-row tile of the op's weight blocks and every K split.
cudaError_t run_gemm(const DraftCtx &c, const TcBufs &t, int op, float *out, size_t bstride, cudaStream_t s,
                     bool pdl, int *ks_out) {
  const OpShape sh = op_shape(c, op);
  TcMaps maps{};
  TcGemmArgs g{};
  g.nmaps = sh.nmaps;
  const int nb = batch_nb(c.B);
  const bool fuse = use_fuse(nb);
  g.mt = op_mt(nb, op, fuse);
  int base = 0, groups = 0;
  for (int i = 0; i < sh.nmaps; ++i) {
    if (!make_map(&maps.w[i], sh.w[i], (uint64_t)sh.K, (uint64_t)sh.rows[i], (uint64_t)sh.K, kTileM))
      return cudaErrorInvalidValue;
    g.rows[i] = sh.rows[i];
    g.groups[i] = ((sh.rows[i] + kTileM - 1) / kTileM + g.mt - 1) / g.mt;
    g.base[i] = base;
    base += sh.rows[i];
    groups += g.groups[i];
  }
  for (int tt = 0; tt < kTerms; ++tt)
    if (!make_map(&maps.a[tt], t.a[tt], (uint64_t)sh.K, (uint64_t)t.rows, (uint64_t)t.kmax, (uint32_t)nb))
      return cudaErrorInvalidValue;
  int ks = 1, kb_per = sh.K / kBK;
  if (op != OP_LMHEAD) {
    op_splits(groups, sh.K, num_sms(), &ks, &kb_per);
    while (ks > 1 && (size_t)ks * c.B * base > t.part_floats) {  // what the workspace holds
      kb_per = (sh.K / kBK + ks - 2) / (ks - 1);
      ks = (sh.K / kBK + kb_per - 1) / kb_per;
    }
  }
  g.ks = ks;
  g.kb_per = kb_per;
  g.kbs = sh.K / kBK;
  g.nb = nb;
  g.stages = (int)(smem_budget() / stage_bytes(nb, g.mt));
  if (g.stages < 2) g.stages = 2;
  if (g.stages > 8) g.stages = 8;
  g.B = c.B;
  g.out = out;
  g.sstride = (size_t)c.B * base;
  g.bstride = bstride;
  g.status = c.status;
  const size_t smem = (size_t)g.stages * stage_bytes(nb, g.mt) + (size_t)(2 * g.stages + 4) * 8 + 16 + 1024;
  g.nunits = groups * ks;
  const int sms = num_sms();
  const int grid = g.nunits < sms ? g.nunits : sms;
  *ks_out = ks;
  cudaError_t e = cudaSuccess;
  for (int r0 = 0; r0 < c.B && e == cudaSuccess; r0 += nb) {  // batch groups of nb rows
    g.arow0 = r0;
    e = fuse ? launch(tc_gemm_kernel<true>, dim3(grid), kTcThreads, smem, s, pdl, maps, g)
             : launch(tc_gemm_kernel<false>, dim3(grid), kTcThreads, smem, s, pdl, maps, g);
  }
  return e;
}

}  // namespace

// One depth in three phases (the caller times them separately): the block up
// to the attention inputs, the block after the attention, the LM head with
// the draft-token selection.
cudaError_t run_block_pre_tc(const DraftCtx &c, const TcBufs &t, cudaStream_t s, bool pdl) {
  const dim3 gb(c.B);
  cudaError_t e;
  int ks = 1;
  const int nqkv = (c.Hq + 2 * c.Hkv) * c.Dh;
  if ((e = launch(tc_prep_fc_kernel, gb, kPrepThreads, 0, s, pdl, c, t))) return e;
  if ((e = run_gemm(c, t, OP_FC, t.part, (size_t)c.d, s, pdl, &ks))) return e;
  if ((e = launch_mid<OP_FC>(c, t, ks, c.d, s, pdl))) return e;
  if ((e = run_gemm(c, t, OP_QKV, t.part, (size_t)nqkv, s, pdl, &ks))) return e;
  return launch_mid<OP_QKV>(c, t, ks, nqkv, s, pdl);
}

cudaError_t run_block_post_tc(const DraftCtx &c, const TcBufs &t, cudaStream_t s, bool pdl) {
  const dim3 gb(c.B);
  cudaError_t e;
  int ks = 1;
  if ((e = launch(tc_prep_wo_kernel, gb, kPrepThreads, 0, s, pdl, c, t))) return e;
  if ((e = run_gemm(c, t, OP_WO, t.part, (size_t)c.d, s, pdl, &ks))) return e;
  if ((e = launch_mid<OP_WO>(c, t, ks, c.d, s, pdl))) return e;
  if ((e = run_gemm(c, t, OP_GATEUP, t.part, (size_t)(2 * c.F), s, pdl, &ks))) return e;
  if ((e = launch_mid<OP_GATEUP>(c, t, ks, 2 * c.F, s, pdl))) return e;
  if ((e = run_gemm(c, t, OP_DOWN, t.part, (size_t)c.d, s, pdl, &ks))) return e;
  return launch_mid<OP_DOWN>(c, t, ks, c.d, s, pdl);
}

cudaError_t run_lmhead_tc(const DraftCtx &c, const TcBufs &t, cudaStream_t s, bool pdl) {
  // straight into the caller's logits when it keeps them (and the head is
  // the full vocabulary); a reduced head's Vd logits go to the workspace and
  // are scattered to their vocabulary ids after the selection
  const bool direct = c.logits && !c.vmap;
  float *lg = direct ? c.logits + (size_t)c.j * c.V : t.part;
  const size_t lstride = direct ? (size_t)c.k * c.V : (size_t)c.Vd;
  int ks = 1;
  cudaError_t e = run_gemm(c, t, OP_LMHEAD, lg, lstride, s, pdl, &ks);
  if (e) return e;
  // past the logits, on a 16-byte boundary
  float4 *sel = reinterpret_cast<float4 *>(t.part + ((size_t)c.B * c.V + 3) / 4 * 4);
  e = launch(tc_select_part_kernel, dim3((sel_subs(c.Vd) + kSelWarps - 1) / kSelWarps, c.B), kSelThreads, 0, s,
             pdl, c, (const float *)lg, lstride, sel);
  if (e) return e;
  e = launch(tc_select_fin_kernel, dim3(c.B), 32, 0, s, pdl, c, (const float *)lg, lstride, (const float4 *)sel);
  if (e || direct || !c.logits) return e;
  return launch(tc_scatter_logits_kernel, dim3((c.Vd + 255) / 256 < 64 ? (c.Vd + 255) / 256 : 64, c.B), 256, 0, s,
                pdl, c, (const float *)lg);
}

MTP_TRACE_COLLECTOR(tc)

}  // namespace mtp
