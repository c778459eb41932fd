// Kernels of one depth of the MTP draft chain.
//
// The module ("The Tiny Draft Model Hidden Inside Qwen", sections "One step
// deeper than the main model" and "What vLLM and SGLang do with the weights")
// is a handful of matrix-vector products around one attention step.  At small
// batch every product is bound by streaming its bf16 weight matrix from HBM
// once ("Speculative Decoding and MTP: Why Guessing Is Free", section "The part
// that got me": decoding is bound by moving weights, not by arithmetic), so the
// GEMV kernel below is built to keep HBM busy:
//
//  * one weight row is cut into P column pieces (P divides the 8 warps of a
//    CTA); warp w always owns piece w % P, so its slice of the activation vector
//    sits in registers for the whole launch;
//  * each warp streams its pieces through its own ring of shared-memory stages
//    filled by 1-D TMA bulk copies (cp.async.bulk) that complete on mbarriers;
//  * the first ring fill is issued before griddepcontrol.wait, so the weight
//    stream of launch n+1 overlaps the tail of launch n (programmatic dependent
//    launch);
//  * normalisation (RMSNorm of the input), residual adds, SiLU-gating, the K/V
//    append into the cache and the LM head's logit statistics are fused into
//    the prologue / epilogue, and the draft token is selected by the last CTA
//    of the LM-head launch (a ticket counter; no spin-waits).
//
// Decode attention is split over chunks of 64 cache positions per (sequence,
// kv head); the GQA group's query heads share each K/V chunk, which is staged by
// TMA.  The last chunk CTA of a (sequence, kv head) combines the partial
// (max, sum, output) triples.
#include <stdlib.h>

#include "common.cuh"
#include "draft_ops.cuh"
#include "internal.h"

namespace mtp {

// ---------------------------------------------------------------- GEMV kernel

// Shared memory: [ring: W*S*PC*2 B][mbarriers: W*S*8 B][part: rpc*P*BG f32]
//                [ys: rpc*BG f32 (LM head)][scales: 2*B f32][red: 64 f32]
//                [sq: W*BG*2 f32 (per-warp sums of squares)]
template <int OP, int NV, int BG>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(DraftCtx c, GemvPlan g) {
  trace_start(kTkGemv + OP);
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = g.stages, P = g.P, R = kGemvWarps / P;
  const int PCB = g.PC * 2;
  unsigned char *ring = smem + (size_t)warp * S * PCB;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)kGemvWarps * S * PCB) + warp * S;
  float *part = reinterpret_cast<float *>(smem + (size_t)kGemvWarps * S * (PCB + 8));
  float *ys = part + (size_t)g.rows_per_cta * P * BG;
  float *scales = ys + (OP == OP_LMHEAD ? (size_t)g.rows_per_cta * BG : 0);
  float *red = scales + 2 * c.B;
  float *sq = red + 64;

  const int p = warp % P, rs = warp / P;
  const int row0 = blockIdx.x * g.rows_per_cta;
  const int nrows = max(0, min(g.rows_per_cta, g.N - row0));
  const int col0 = p * g.PC;
  const int ncols = max(0, min(g.PC, g.K - col0));
  const uint32_t piece_bytes = (uint32_t)ncols * 2u;
  const int units_per_group = nrows > rs ? (nrows - rs + R - 1) / R : 0;
  const int total_units = ncols > 0 ? units_per_group * g.ngroups : 0;

  // Ring set-up and the first fill: weights only, so it may run before the
  // previous kernel of the chain has finished.
  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();
  const uint64_t pol = l2_policy_evict_first();
  auto issue = [&](int n) {
    const int rl = rs + (n % units_per_group) * R;
    const int stage = n % S;
    mbar_arrive_expect_tx(&bars[stage], piece_bytes);
    bulk_g2s_hint(ring + (size_t)stage * PCB, weight_row<OP>(c, row0 + rl, g.K) + col0, piece_bytes, &bars[stage],
                  pol);
  };
  const int pre = min(g.pre, S);
  if (lane == 0)
    for (int n = 0; n < min(pre, total_units); ++n) issue(n);

  grid_dep_wait();
  grid_dep_launch();
  trace_dep(kTkGemv + OP);

  // Dynamic draft length: once every sequence has stopped drafting, the later
  // depths have nothing to do -- let the weight copies already issued land and
  // leave (the flag is written only by earlier launches, so every CTA reads the
  // same value).
  if (c.n_active && c.j > 0 && *reinterpret_cast<volatile unsigned *>(c.n_active) == 0u) {
    if (lane == 0)
      for (int n = 0; n < min(pre, total_units); ++n)
        if (!mbar_sleep_wait(&bars[n], 0u, c.status)) break;
    trace_end(kTkGemv + OP);
    return;
  }
  if (OP == OP_FC && c.zero_counters && blockIdx.x == 0) {
    if (threadIdx.x == 0) *c.lm_cnt = 0u;
    if (c.k_eff) {
      for (int b = threadIdx.x; b < c.B; b += kGemvThreads) c.k_eff[b] = c.k;
      if (threadIdx.x == 0) *c.n_active = (unsigned)c.B;
    }
  }
  const bool fac = g.factor != 0;
  if (!fac) compute_scales<OP>(c, scales, red);

  int n = 0;
  bool ok = true;
  for (int grp = 0; grp < g.ngroups; ++grp) {
    // this warp's activation slice for the group's batch rows
    float a[BG][NV][8];
    float s0[BG], s1[BG];
#pragma unroll
    for (int bb = 0; bb < BG; ++bb) {
      const int b = grp * BG + bb;
      s0[bb] = 0.f;
      s1[bb] = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int v = lane + 32 * i;
        if (b < c.B && v * 8 < ncols) {
          if (fac) act8_unscaled<OP>(c, b, col0 + v * 8, a[bb][i], s0[bb], s1[bb]);
          else act8<OP>(c, b, col0 + v * 8, scales, a[bb][i]);
        } else {
#pragma unroll
          for (int t = 0; t < 8; ++t) a[bb][i][t] = 0.f;
        }
      }
    }
    if (fac) {
      // the warps of the first row set cover the input once: their sums of
      // squares, combined in warp order in the epilogue, give the norm's scale
#pragma unroll
      for (int bb = 0; bb < BG; ++bb) {
        s0[bb] = warp_sum(s0[bb]);
        if (OP == OP_FC) s1[bb] = warp_sum(s1[bb]);
        if (lane == 0 && rs == 0) {
          sq[(warp * BG + bb) * 2] = s0[bb];
          sq[(warp * BG + bb) * 2 + 1] = s1[bb];
        }
      }
    }
    if (grp == 0) {
      trace_mark(kTkGemv + OP, 0);  // activations loaded
      // the rest of the first ring fill, after the activation loads
      if (lane == 0)
        for (int q = pre; q < min(S, total_units); ++q) issue(q);
    }
    for (int u = 0; u < units_per_group && ncols > 0; ++u, ++n) {
      const int stage = n % S;
      if (ok) ok = mbar_sleep_wait(&bars[stage], (uint32_t)(n / S) & 1u, c.status);
      ok = __all_sync(0xffffffffu, ok);
      float acc[BG];
#pragma unroll
      for (int bb = 0; bb < BG; ++bb) acc[bb] = 0.f;
      const unsigned char *buf = ring + (size_t)stage * PCB;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int v = lane + 32 * i;
        if (v * 8 < ncols) {
          const uint4 w = *reinterpret_cast<const uint4 *>(buf + v * 16);
#pragma unroll
          for (int bb = 0; bb < BG; ++bb) acc[bb] = dot8(w, a[bb][i], acc[bb]);
        }
      }
#pragma unroll
      for (int bb = 0; bb < BG; ++bb) acc[bb] = warp_sum(acc[bb]);
      const int rl = rs + u * R;
      if (lane == 0) {
#pragma unroll
        for (int bb = 0; bb < BG; ++bb) part[((size_t)rl * P + p) * BG + bb] = acc[bb];
      }
      __syncwarp();
      if (lane == 0 && ok && n + S < total_units) {
        fence_proxy_async_smem();
        issue(n + S);
      }
    }
    __syncthreads();
    trace_mark(kTkGemv + OP, 1);  // the group's last weight piece used

    // epilogue for this batch group (the norm's scales, the op's outputs and,
    // for the LM head, this CTA's partials)
    gemv_epilogue<OP, BG>(c, P, g.PC, row0, nrows, grp, fac, part, sq, ys, red, (int)blockIdx.x);
    __syncthreads();
    trace_mark(kTkGemv + OP, 2);  // epilogue done
  }

  trace_end(kTkGemv + OP);
  if (OP != OP_LMHEAD) return;

  // ---- draft-token selection by the last CTA to finish
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(c.lm_cnt, 1u) == gridDim.x - 1;
  __syncthreads();
  trace_end(kTkGemv + OP);
  if (!s_last) return;
  __threadfence();
  if (warp == 0) {
    lm_select_warp(c, c.lm_grid, c.lm_rpc);
    if (lane == 0) *c.lm_cnt = 0u;
  }
  trace_end(kTkGemv + OP);
}

// ---------------------------------------------------------------- planning / launch

// Tuning knobs (environment, read per call): MTP_GEMV_CTAS_PER_SM (default 2),
// MTP_GEMV_STAGES (ring depth per warp, default 6), MTP_GEMV_PIECE (maximum
// columns per TMA piece, default 1024), MTP_GEMV_SMEM_KB (shared-memory cap per
// CTA, default 110).  Two CTAs of 8 warps per SM with 6 stages of 2 KB each keep
// about 190 KB of weight copies in flight per SM.
static int env_int(const char *name, int dflt) {
  const char *v = getenv(name);
  return v && *v ? atoi(v) : dflt;
}

GemvPlan plan_gemv(int op, int N, int K, int B, int num_sms) {
  GemvPlan g{};
  g.op = op;
  g.N = N;
  g.K = K;
  const int piece_max = env_int("MTP_GEMV_PIECE", 1024);
  int P = 1;
  while (P < kGemvWarps && (K + P - 1) / P > piece_max) P *= 2;
  g.P = P;
  g.PC = (((K + P - 1) / P) + 7) / 8 * 8;
  int nv = (g.PC + 255) / 256;
  nv = nv <= 1 ? 1 : nv <= 2 ? 2 : nv <= 4 ? 4 : nv <= 6 ? 6 : 9;
  g.nv = nv;
  g.bg = (B > 1 && nv <= 4) ? 2 : 1;
  g.ngroups = (B + g.bg - 1) / g.bg;
  int grid = num_sms * env_int("MTP_GEMV_CTAS_PER_SM", 2);
  int rpc = (N + grid - 1) / grid;
  if (op == OP_GATEUP && (rpc & 1)) ++rpc;
  g.rows_per_cta = rpc;
  g.grid = (N + rpc - 1) / rpc;
  g.stages = env_int("MTP_GEMV_STAGES", 6);
  // four of the six stages before the wait: the rest after the activation
  // loads, which the full fill would queue behind (measured 1085 -> 1091
  // steps/s at the single-sequence workload)
  g.pre = env_int("MTP_GEMV_PRE", 4);
  // the norm's scale after the dot products: the ops with an input norm, when
  // no piece of the input projection straddles its two halves (and
  // MTP_GEMV_FACTOR is not 0)
  g.factor = (op == OP_FC || op == OP_QKV || op == OP_GATEUP || op == OP_LMHEAD) &&
             (op != OP_FC || (K / 2) % g.PC == 0) && env_int("MTP_GEMV_FACTOR", 1) != 0;
  auto smem_for = [&](int stages) {
    size_t s = (size_t)kGemvWarps * stages * (g.PC * 2 + 8);
    s += (size_t)g.rows_per_cta * g.P * g.bg * 4;
    if (op == OP_LMHEAD) s += (size_t)g.rows_per_cta * g.bg * 4;
    s += (size_t)2 * B * 4 + 64 * 4 + (size_t)kGemvWarps * 2 * 2 * 4;
    return s;
  };
  const int smem_cap = env_int("MTP_GEMV_SMEM_KB", 110) * 1024;
  while (g.stages > 2 && smem_for(g.stages) > (size_t)smem_cap) --g.stages;
  g.smem = smem_for(g.stages);
  return g;
}

template <int OP, int NV, int BG>
static cudaError_t launch_one(const DraftCtx &c, const GemvPlan &g, cudaStream_t s, bool pdl) {
  auto kern = gemv_kernel<OP, NV, BG>;
  static unsigned long long attr_ctx = 0;  // the context the attribute was set in
  const unsigned long long cid = context_id();
  if (cid == 0 || cid != attr_ctx) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    attr_ctx = cid;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(g.grid);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  note_launch();
  return cudaLaunchKernelEx(&cfg, kern, c, g);
}

template <int OP>
static cudaError_t launch_op(const DraftCtx &c, const GemvPlan &g, cudaStream_t s, bool pdl) {
  if (g.bg == 2) {
    switch (g.nv) {
      case 1: return launch_one<OP, 1, 2>(c, g, s, pdl);
      case 2: return launch_one<OP, 2, 2>(c, g, s, pdl);
      default: return launch_one<OP, 4, 2>(c, g, s, pdl);
    }
  }
  switch (g.nv) {
    case 1: return launch_one<OP, 1, 1>(c, g, s, pdl);
    case 2: return launch_one<OP, 2, 1>(c, g, s, pdl);
    case 4: return launch_one<OP, 4, 1>(c, g, s, pdl);
    case 6: return launch_one<OP, 6, 1>(c, g, s, pdl);
    default: return launch_one<OP, 9, 1>(c, g, s, pdl);
  }
}

cudaError_t launch_gemv(const DraftCtx &c, const GemvPlan &g, cudaStream_t s, bool pdl) {
  switch (g.op) {
    case OP_FC: return launch_op<OP_FC>(c, g, s, pdl);
    case OP_QKV: return launch_op<OP_QKV>(c, g, s, pdl);
    case OP_WO: return launch_op<OP_WO>(c, g, s, pdl);
    case OP_GATEUP: return launch_op<OP_GATEUP>(c, g, s, pdl);
    case OP_DOWN: return launch_op<OP_DOWN>(c, g, s, pdl);
    default: return launch_op<OP_LMHEAD>(c, g, s, pdl);
  }
}

// ---------------------------------------------------------------- decode attention
//
// One thread-block cluster per (sequence b, kv head g); CTA r of the cluster
// owns the contiguous cache positions [r*T, (r+1)*T) of the ntok = L_b + j + 1
// visible ones, and each of its 8 warps a contiguous eighth of those.  A warp
// works on two cache rows at a time, one per half-warp (DH/16 dims per lane),
// and keeps a private online softmax (running max, sum, rescaled output) for
// every query head of the GQA group, with the K/V rows of the next batch loaded
// into registers while the current batch is computed -- no barriers inside the
// loop.  Warps are merged through shared memory, CTAs through distributed
// shared memory (each CTA finalises a slice of the output).

constexpr int kAttnWarps = 8;    // compute warps; warp kAttnWarps streams K/V
constexpr int kAttnTile = 64;    // rows per ring stage, at most
constexpr int kAttnStages = 3;
// row pairs per warp and tile: 4, or 1 for groups of more than four heads
// (their per-head state takes the registers)
__host__ __device__ constexpr int attn_unroll(int gm) { return gm > 4 ? 1 : 4; }

// Shared memory: [K/V ring: S x (K tile, V tile)][per-warp (max, sum, output)]
// [q, then the CTA's output][CTA (max, sum)][mbarriers]
size_t attention_smem_bytes(int Dh) {
  return (size_t)kAttnStages * 2 * kAttnTile * Dh * 2            // K/V ring
         + (size_t)kAttnWarps * kMaxGroup * (Dh + 2) * 4          // per-warp (max, sum, output)
         + (size_t)kMaxGroup * Dh * 4                             // q, then the CTA's output
         + (size_t)kMaxGroup * 2 * 4                              // CTA (max, sum)
         + (size_t)2 * kAttnStages * (kAttnTile / 16) * 8 + 16;   // mbarriers (up to 12 stages)
}

template <int DPL>
struct RowVec;
template <>
struct RowVec<2> { uint32_t x; };
template <>
struct RowVec<4> { uint2 x; };
template <>
struct RowVec<8> { uint4 x; };

template <int DPL>
__device__ __forceinline__ RowVec<DPL> load_row_smem(const uint16_t *p) {
  RowVec<DPL> r;
  if constexpr (DPL == 2) r.x = *reinterpret_cast<const unsigned int *>(p);
  else if constexpr (DPL == 4) r.x = *reinterpret_cast<const uint2 *>(p);
  else r.x = *reinterpret_cast<const uint4 *>(p);
  return r;
}

template <int DPL>
__device__ __forceinline__ void unpack_row(const RowVec<DPL> &r, float *out) {
  const uint32_t *w = reinterpret_cast<const uint32_t *>(&r.x);
#pragma unroll
  for (int i = 0; i < DPL / 2; ++i) {
    out[2 * i] = bf16_lo(w[i]);
    out[2 * i + 1] = bf16_hi(w[i]);
  }
}

// Decode attention of one (sequence, kv head) over its cache rows 0 .. L+j,
// split over a cluster of C CTAs (CTA r takes a contiguous range of rows).
// Warp kAttnWarps streams the CTA's K and V rows in tiles of 64 through a ring
// of shared-memory stages with 1-D TMA bulk copies (a sequence's rows are
// contiguous); tiles of context rows only -- written by the caller -- are
// requested before the previous kernel of the chain has finished.  Each
// compute warp takes 2U rows of every tile, a half-warp per row: scores for all
// heads of the GQA group, then one online-softmax update per head for the
// warp's rows.  Warps merge through shared memory, the cluster's CTAs through
// distributed shared memory.
template <int DH, int GM>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_kernel(DraftCtx c) {
  trace_start(kTkAttn);
  constexpr int DPL = DH / 16, NW = kAttnWarps, U = attn_unroll(GM);
  constexpr int TT = 2 * U * NW;        // rows per tile
  constexpr int TILE = TT * DH;         // elements of one K (or V) tile
  constexpr int NS = kAttnStages * kAttnTile / TT;  // stages: the ring holds 3 x 64 rows
  extern __shared__ __align__(128) unsigned char smem[];
  uint16_t *ring = reinterpret_cast<uint16_t *>(smem);                  // [S][K tile, V tile]
  float *wst = reinterpret_cast<float *>(ring + (size_t)NS * 2 * TILE);  // [NW][GM][DH+2]
  float *qo = wst + NW * kMaxGroup * (DH + 2);            // [GM][DH]
  float *mrun = qo + kMaxGroup * DH;                      // [GM]
  float *lrun = mrun + kMaxGroup;                         // [GM]
  uint64_t *full = reinterpret_cast<uint64_t *>(lrun + kMaxGroup);
  uint64_t *empty = full + NS;

  const int g = blockIdx.y, b = blockIdx.z;
  const int C = (int)cluster_size(), rank = (int)cluster_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int half = lane >> 4, hl = lane & 15;
  const int group = c.Hq / c.Hkv;
  int L = __ldg(&c.ctx_len[b]);
  L = min(max(L, 0), c.Lmax - c.k);
  const int ntok = L + c.jc + 1;
  const int T = (ntok + C - 1) / C;
  const int r0 = min(ntok, rank * T), r1 = min(ntok, r0 + T);
  const int ntiles = (r1 - r0 + TT - 1) / TT;
  const size_t base = ((size_t)b * c.Hkv + g) * c.Lmax * DH;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    fence_barrier_init();
  }
  __syncthreads();

  bool ok = true;
  if (warp == NW) {
    // ------------------------------------------------ K/V producer
    if (lane == 0) {
      bool waited = false;
      for (int i = 0; i < ntiles && ok; ++i) {
        const int s = i % NS;
        if (i >= NS) ok = mbar_wait(&empty[s], (uint32_t)((i / NS) - 1) & 1u, c.status);
        if (!ok) break;
        const int t0 = r0 + i * TT, n = min(TT, r1 - t0);
        if (!waited && t0 + n > L) {  // rows L.. are appended by this chain
          grid_dep_wait();
          waited = true;
        }
        const uint32_t bytes = (uint32_t)n * DH * 2;
        mbar_arrive_expect_tx(&full[s], 2 * bytes);
        bulk_g2s(ring + (size_t)s * 2 * TILE, c.kc + base + (size_t)t0 * DH, bytes, &full[s]);
        bulk_g2s(ring + (size_t)s * 2 * TILE + TILE, c.vc + base + (size_t)t0 * DH, bytes, &full[s]);
      }
      if (!waited) grid_dep_wait();
    }
    grid_dep_launch();
  } else {
    // ------------------------------------------------ compute warps
    grid_dep_wait();  // q comes from this depth's projection
    grid_dep_launch();
    const int nq = c.Hq * DH;
    float q[GM][DPL];
#pragma unroll
    for (int h = 0; h < GM; ++h)
#pragma unroll
      for (int e = 0; e < DPL; ++e)
        q[h][e] = h < group ? __ldcg(&c.q[(size_t)b * nq + ((size_t)g * group + h) * DH + hl * DPL + e]) : 0.f;
    float m[GM], l[GM], acc[GM][DPL];
#pragma unroll
    for (int h = 0; h < GM; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[h][e] = 0.f;
    }
    const float scale = rsqrtf((float)DH) * kLog2e;

    for (int i = 0; i < ntiles; ++i) {
      const int s = i % NS;
      if (ok) ok = mbar_wait(&full[s], (uint32_t)(i / NS) & 1u, c.status);
      ok = __all_sync(0xffffffffu, ok);
      const int t0 = r0 + i * TT;
      const uint16_t *kt = ring + (size_t)s * 2 * TILE;
      const uint16_t *vt = kt + TILE;
      // this warp's rows of the tile: 2 U w + 2 u + half
      float sc[U][GM];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int rl = 2 * U * warp + 2 * u + half;
        const bool live = t0 + rl < r1;
        float kv[DPL];
        unpack_row<DPL>(load_row_smem<DPL>(kt + (size_t)rl * DH + hl * DPL), kv);
#pragma unroll
        for (int h = 0; h < GM; ++h) {
          float sdot = 0.f;
#pragma unroll
          for (int e = 0; e < DPL; ++e) sdot = fmaf(q[h][e], kv[e], sdot);
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) sdot += __shfl_xor_sync(0xffffffffu, sdot, o);
          sc[u][h] = live ? sdot * scale : -INFINITY;
        }
      }
      float vv[U][DPL];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int rl = 2 * U * warp + 2 * u + half;
        if (t0 + rl < r1) unpack_row<DPL>(load_row_smem<DPL>(vt + (size_t)rl * DH + hl * DPL), vv[u]);
        else {
#pragma unroll
          for (int e = 0; e < DPL; ++e) vv[u][e] = 0.f;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage
      // one online-softmax update per head for the warp's rows
#pragma unroll
      for (int h = 0; h < GM; ++h) {
        if (h < group) {
          float bm = sc[0][h];
#pragma unroll
          for (int u = 1; u < U; ++u) bm = fmaxf(bm, sc[u][h]);
          const float mn = fmaxf(m[h], bm);
          if (mn != -INFINITY) {
            const float f = exp2f(m[h] - mn);   // 0 while m is -inf
            float pw[U], ps = 0.f;
#pragma unroll
            for (int u = 0; u < U; ++u) {
              pw[u] = exp2f(sc[u][h] - mn);
              ps += pw[u];
            }
            l[h] = l[h] * f + ps;
#pragma unroll
            for (int e = 0; e < DPL; ++e) {
              float a = acc[h][e] * f;
#pragma unroll
              for (int u = 0; u < U; ++u) a = fmaf(pw[u], vv[u][e], a);
              acc[h][e] = a;
            }
            m[h] = mn;
          }
        }
      }
    }

    // merge the two half-warps into the warp's slot
#pragma unroll
    for (int h = 0; h < GM; ++h) {
      if (h < group) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m[h], 16);
        const float l2 = __shfl_xor_sync(0xffffffffu, l[h], 16);
        const float M = fmaxf(m[h], m2);
        const float f1 = m[h] == -INFINITY ? 0.f : exp2f(m[h] - M);
        const float f2 = m2 == -INFINITY ? 0.f : exp2f(m2 - M);
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
          const float a2 = __shfl_xor_sync(0xffffffffu, acc[h][e], 16);
          acc[h][e] = acc[h][e] * f1 + a2 * f2;
        }
        l[h] = l[h] * f1 + l2 * f2;
        m[h] = M;
        if (half == 0) {
          float *ws = wst + ((size_t)warp * kMaxGroup + h) * (DH + 2);
          if (hl == 0) {
            ws[0] = m[h];
            ws[1] = l[h];
          }
#pragma unroll
          for (int e = 0; e < DPL; ++e) ws[2 + hl * DPL + e] = acc[h][e];
        }
      }
    }
  }
  __syncthreads();
  // merge the warps of the CTA
  for (int idx = tid; idx < group * DH; idx += kAttnThreads) {
    const int h = idx / DH, e = idx % DH;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, wst[((size_t)w * kMaxGroup + h) * (DH + 2)]);
    float Ls = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float *ws = wst + ((size_t)w * kMaxGroup + h) * (DH + 2);
      if (ws[0] == -INFINITY) continue;
      const float f = exp2f(ws[0] - M);
      Ls = fmaf(ws[1], f, Ls);
      O = fmaf(ws[2 + e], f, O);
    }
    qo[h * DH + e] = O;
    if (e == 0) {
      mrun[h] = M;
      lrun[h] = Ls;
    }
  }
  // combine across the cluster: CTA r finalises pairs (h, e) r, r + C, ...
  const int nq = c.Hq * DH;
  cluster_sync();
  for (int idx = rank + C * tid; idx < group * DH; idx += C * kAttnThreads) {
    const int h = idx / DH, e = idx % DH;
    float mr[16], lr[16], orr[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      if (r < C) {
        mr[r] = *dsmem_ptr(&mrun[h], r);
        lr[r] = *dsmem_ptr(&lrun[h], r);
        orr[r] = *dsmem_ptr(&qo[h * DH + e], r);
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < 16; ++r)
      if (r < C) M = fmaxf(M, mr[r]);
    float Ls = 0.f, O = 0.f;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      if (r < C && mr[r] != -INFINITY) {
        const float wgt = exp2f(mr[r] - M);
        Ls = fmaf(lr[r], wgt, Ls);
        O = fmaf(orr[r], wgt, O);
      }
    }
    c.o[(size_t)b * nq + ((size_t)g * group + h) * DH + e] = O / Ls;
  }
  cluster_sync();  // keep this CTA's shared memory alive until every peer has read it
  trace_end(kTkAttn);
}

__global__ void __launch_bounds__(256) fill_kernel(float *p, size_t n, float v) {
  grid_dep_wait();  // the previous call may still read these
  grid_dep_launch();
  for (size_t i = (size_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (size_t)gridDim.x * 256) p[i] = v;
}

cudaError_t launch_fill(float *p, size_t n, float v, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg{};
  const size_t blocks = (n + 255) / 256;
  cfg.gridDim = dim3((unsigned)(blocks < 4096 ? (blocks > 0 ? blocks : 1) : 4096));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  note_launch();
  return cudaLaunchKernelEx(&cfg, fill_kernel, p, n, v);
}

int attention_cluster_size(int ctx_max, int pairs, int num_sms, int max_cluster, bool tc) {
  const int forced = env_int("MTP_ATTN_CLUSTER", 0);
  if (forced > 0) return forced < max_cluster ? forced : max_cluster;
  // CTAs per (sequence, kv head), and no more than about four CTAs per SM in
  // all.  The CUDA-core kernel (one CTA per SM): one per 512 context rows, at
  // most 8 (a 16-CTA cluster of it does not fit every GPC at once).  The
  // tensor-core kernel (two CTAs per SM): one per 256 rows, at most 16 -- at a
  // single sequence, 8 kv heads and 4096 rows, 16 runs the step 1.3% faster
  // than 8 (measured).
  int C = (ctx_max + (tc ? 255 : 511)) / (tc ? 256 : 512);
  const int by_sms = (4 * num_sms + pairs - 1) / (pairs > 0 ? pairs : 1);
  if (C > by_sms) C = by_sms;
  const int lim = tc ? 16 : 8;
  const int cap = max_cluster < lim ? max_cluster : lim;
  return C < 1 ? 1 : (C > cap ? cap : C);
}

template <int DH, int GM>
static cudaError_t launch_attn(const DraftCtx &c, int cluster, cudaStream_t s, bool pdl) {
  auto kern = attn_kernel<DH, GM>;
  static unsigned long long attr_ctx = 0;  // the context the attributes were set in
  const size_t smem = attention_smem_bytes(DH);
  const unsigned long long cid = context_id();
  if (cid == 0 || cid != attr_ctx) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr_ctx = cid;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(cluster, c.Hkv, c.B);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
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
  return cudaLaunchKernelEx(&cfg, kern, c);
}

template <int DH>
static cudaError_t launch_attn_g(const DraftCtx &c, int cluster, cudaStream_t s, bool pdl) {
  const int group = c.Hq / c.Hkv;
  if (group <= 1) return launch_attn<DH, 1>(c, cluster, s, pdl);
  if (group <= 2) return launch_attn<DH, 2>(c, cluster, s, pdl);
  if (group <= 4) return launch_attn<DH, 4>(c, cluster, s, pdl);
  return launch_attn<DH, 8>(c, cluster, s, pdl);
}

cudaError_t launch_attention(const DraftCtx &c, int cluster, cudaStream_t s, bool pdl) {
  if (attention_tc_shape_ok(c)) return launch_attention_tc(c, cluster, s, pdl);
  switch (c.Dh) {
    case 32: return launch_attn_g<32>(c, cluster, s, pdl);
    case 64: return launch_attn_g<64>(c, cluster, s, pdl);
    default: return launch_attn_g<128>(c, cluster, s, pdl);
  }
}

MTP_TRACE_COLLECTOR(draft)

}  // namespace mtp
