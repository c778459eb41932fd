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
#include "common.cuh"
#include "internal.h"

namespace mtp {

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ void load8_bf16(const uint16_t *p, float *out) {
  uint4 w = __ldg(reinterpret_cast<const uint4 *>(p));
  out[0] = bf16_lo(w.x); out[1] = bf16_hi(w.x);
  out[2] = bf16_lo(w.y); out[3] = bf16_hi(w.y);
  out[4] = bf16_lo(w.z); out[5] = bf16_hi(w.z);
  out[6] = bf16_lo(w.w); out[7] = bf16_hi(w.w);
}

// fp32 data produced by an earlier kernel of the chain: read through L2.
__device__ __forceinline__ void load8_f32(const float *p, float *out) {
  float4 a = __ldcg(reinterpret_cast<const float4 *>(p));
  float4 b = __ldcg(reinterpret_cast<const float4 *>(p) + 1);
  out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
  out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
}

__device__ __forceinline__ float block_sum_256(float v, float *red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < kGemvWarps; ++i) t += red[i];
  return t;
}

// Token feeding depth j of sequence b (validated).
__device__ __forceinline__ int depth_token(const DraftCtx &c, int b) {
  int t = c.j == 0 ? __ldg(&c.last_tok[b]) : __ldcg(&c.draft_tok[b * c.k + c.j - 1]);
  if (t < 0 || t >= c.V) {
    set_status(c.status, kStatusBadToken);
    t = 0;
  }
  return t;
}

__device__ __forceinline__ int clamped_ctx(const DraftCtx &c, int b) {
  int L = __ldg(&c.ctx_len[b]);
  return min(max(L, 0), c.Lmax - c.k);
}

// RMSNorm scale factors 1/sqrt(mean(v^2)+eps) of the vectors this op
// normalises, for every batch row.  scales[2*b] is the first vector's (for the
// input projection: the token embedding), scales[2*b+1] the second's (the
// hidden state).
template <int OP>
__device__ void compute_scales(const DraftCtx &c, float *scales, float *red) {
  if (OP == OP_WO || OP == OP_DOWN) return;
  const int d = c.d;
  for (int b = 0; b < c.B; ++b) {
    float s0 = 0.f, s1 = 0.f;
    if (OP == OP_FC) {
      const uint16_t *e = c.E + (size_t)depth_token(c, b) * d;
      for (int i = threadIdx.x * 8; i < d; i += kGemvThreads * 8) {
        float v[8];
        load8_bf16(e + i, v);
#pragma unroll
        for (int t = 0; t < 8; ++t) s0 = fmaf(v[t], v[t], s0);
      }
      for (int i = threadIdx.x * 8; i < d; i += kGemvThreads * 8) {
        float v[8];
        if (c.j == 0) load8_bf16(c.h + (size_t)b * d + i, v);
        else load8_f32(c.x2 + (size_t)b * d + i, v);
#pragma unroll
        for (int t = 0; t < 8; ++t) s1 = fmaf(v[t], v[t], s1);
      }
    } else {
      const float *x = OP == OP_QKV ? c.x0 : (OP == OP_GATEUP ? c.x1 : c.x2);
      for (int i = threadIdx.x * 8; i < d; i += kGemvThreads * 8) {
        float v[8];
        load8_f32(x + (size_t)b * d + i, v);
#pragma unroll
        for (int t = 0; t < 8; ++t) s0 = fmaf(v[t], v[t], s0);
      }
    }
    s0 = block_sum_256(s0, red);
    if (OP == OP_FC) s1 = block_sum_256(s1, red);
    if (threadIdx.x == 0) {
      scales[2 * b] = rsqrtf(s0 / (float)d + c.eps);
      scales[2 * b + 1] = rsqrtf(s1 / (float)d + c.eps);
    }
  }
  __syncthreads();
}

// Eight consecutive activation values (columns col .. col+7) of batch row b.
template <int OP>
__device__ __forceinline__ void act8(const DraftCtx &c, int b, int col, const float *scales, float *out) {
  const int d = c.d;
  if (OP == OP_FC) {
    float g[8];
    if (col < d) {
      load8_bf16(c.E + (size_t)depth_token(c, b) * d + col, out);
      load8_bf16(c.g_emb + col, g);
      const float s = scales[2 * b];
#pragma unroll
      for (int t = 0; t < 8; ++t) out[t] = out[t] * s * g[t];
    } else {
      const int cc = col - d;
      if (c.j == 0) load8_bf16(c.h + (size_t)b * d + cc, out);
      else load8_f32(c.x2 + (size_t)b * d + cc, out);
      load8_bf16(c.g_hid + cc, g);
      const float s = scales[2 * b + 1];
#pragma unroll
      for (int t = 0; t < 8; ++t) out[t] = out[t] * s * g[t];
    }
  } else if (OP == OP_WO) {
    load8_f32(c.o + (size_t)b * c.Hq * c.Dh + col, out);
  } else if (OP == OP_DOWN) {
    load8_f32(c.act + (size_t)b * c.F + col, out);
  } else {
    const float *x = OP == OP_QKV ? c.x0 : (OP == OP_GATEUP ? c.x1 : c.x2);
    const uint16_t *gp = OP == OP_QKV ? c.g_attn : (OP == OP_GATEUP ? c.g_mlp : c.g_final);
    float g[8];
    load8_f32(x + (size_t)b * d + col, out);
    load8_bf16(gp + col, g);
    const float s = scales[2 * b];
#pragma unroll
    for (int t = 0; t < 8; ++t) out[t] = out[t] * s * g[t];
  }
}

template <int OP>
__device__ __forceinline__ const uint16_t *weight_row(const DraftCtx &c, int row, int K) {
  if (OP == OP_FC) return c.fc + (size_t)row * K;
  if (OP == OP_QKV) {
    const int nq = c.Hq * c.Dh, nkv = c.Hkv * c.Dh;
    if (row < nq) return c.wq + (size_t)row * K;
    row -= nq;
    if (row < nkv) return c.wk + (size_t)row * K;
    return c.wv + (size_t)(row - nkv) * K;
  }
  if (OP == OP_WO) return c.wo + (size_t)row * K;
  if (OP == OP_GATEUP) return ((row & 1) ? c.wup : c.wgate) + (size_t)(row >> 1) * K;
  if (OP == OP_DOWN) return c.wdown + (size_t)row * K;
  return c.E + (size_t)row * K;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.f + __expf(-z)); }

// ---------------------------------------------------------------- GEMV kernel

// Shared memory: [ring: W*S*PC*2 B][mbarriers: W*S*8 B][part: rpc*P*BG f32]
//                [ys: rpc*BG f32 (LM head)][scales: 2*B f32][red: 64 f32]
template <int OP, int NV, int BG>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(DraftCtx c, GemvPlan g) {
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
  if (lane == 0)
    for (int n = 0; n < min(S, total_units); ++n) issue(n);

  grid_dep_wait();
  grid_dep_launch();

  if (OP == OP_FC && c.zero_counters && blockIdx.x == 0) {
    for (int i = threadIdx.x; i < c.B * c.Hkv; i += kGemvThreads) c.attn_cnt[i] = 0u;
    if (threadIdx.x == 0) *c.lm_cnt = 0u;
  }
  compute_scales<OP>(c, scales, red);

  int n = 0;
  bool ok = true;
  for (int grp = 0; grp < g.ngroups; ++grp) {
    // this warp's activation slice for the group's batch rows
    float a[BG][NV][8];
#pragma unroll
    for (int bb = 0; bb < BG; ++bb) {
      const int b = grp * BG + bb;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int v = lane + 32 * i;
        if (b < c.B && v * 8 < ncols) act8<OP>(c, b, col0 + v * 8, scales, a[bb][i]);
        else {
#pragma unroll
          for (int t = 0; t < 8; ++t) a[bb][i][t] = 0.f;
        }
      }
    }
    for (int u = 0; u < units_per_group && ncols > 0; ++u, ++n) {
      const int stage = n % S;
      if (ok) ok = mbar_wait(&bars[stage], (uint32_t)(n / S) & 1u, c.status);
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

    // epilogue for this batch group
    for (int rl = threadIdx.x; rl < nrows; rl += kGemvThreads) {
      const int row = row0 + rl;
      if (OP == OP_GATEUP && (rl & 1)) continue;
#pragma unroll
      for (int bb = 0; bb < BG; ++bb) {
        const int b = grp * BG + bb;
        if (b >= c.B) break;
        float y = 0.f;
        for (int pp = 0; pp < P; ++pp) y += part[((size_t)rl * P + pp) * BG + bb];
        if (OP == OP_FC) {
          c.x0[(size_t)b * c.d + row] = y;
        } else if (OP == OP_QKV) {
          const int nq = c.Hq * c.Dh, nkv = c.Hkv * c.Dh;
          if (row < nq) {
            c.q[(size_t)b * nq + row] = y;
          } else {
            int r = row - nq;
            uint16_t *cache = r < nkv ? c.kc : c.vc;
            if (r >= nkv) r -= nkv;
            const int kvh = r / c.Dh, dd = r % c.Dh;
            int L = __ldg(&c.ctx_len[b]);
            if (L < 0 || L + c.k > c.Lmax) set_status(c.status, kStatusBadCtx);
            L = min(max(L, 0), c.Lmax - c.k);
            const size_t idx = (((size_t)b * c.Hkv + kvh) * c.Lmax + L + c.j) * c.Dh + dd;
            cache[idx] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
          }
        } else if (OP == OP_WO) {
          c.x1[(size_t)b * c.d + row] = __ldcg(&c.x0[(size_t)b * c.d + row]) + y;
        } else if (OP == OP_GATEUP) {
          float up = 0.f;
          for (int pp = 0; pp < P; ++pp) up += part[((size_t)(rl + 1) * P + pp) * BG + bb];
          c.act[(size_t)b * c.F + (row >> 1)] = silu_f(y) * up;
        } else if (OP == OP_DOWN) {
          c.x2[(size_t)b * c.d + row] = __ldcg(&c.x1[(size_t)b * c.d + row]) + y;
        } else {  // LM head
          if (c.logits) c.logits[((size_t)b * c.k + c.j) * c.V + row] = y;
          ys[(size_t)rl * BG + bb] = y;
        }
      }
    }

    if (OP == OP_LMHEAD) {
      __syncthreads();
      const float cT = kLog2e / c.T;
      for (int bb = 0; bb < BG; ++bb) {
        const int b = grp * BG + bb;
        if (b >= c.B) break;
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int rl = threadIdx.x; rl < nrows; rl += kGemvThreads) argmax_merge(bv, bi, ys[(size_t)rl * BG + bb], row0 + rl);
        warp_argmax(bv, bi);
        __syncthreads();
        if (lane == 0) {
          red[warp] = bv;
          red[kGemvWarps + warp] = __int_as_float(bi);
        }
        __syncthreads();
        float m = -INFINITY;
        int mi = 0x7fffffff;
        for (int w = 0; w < kGemvWarps; ++w) argmax_merge(m, mi, red[w], __float_as_int(red[kGemvWarps + w]));
        float s = 0.f;
        if (c.mode == 1 && m != -INFINITY)
          for (int rl = threadIdx.x; rl < nrows; rl += kGemvThreads) s += exp2f((ys[(size_t)rl * BG + bb] - m) * cT);
        s = block_sum_256(s, red + 2 * kGemvWarps);
        if (threadIdx.x == 0) {
          float *pp = c.lm_part + ((size_t)b * c.lm_grid + blockIdx.x) * 4;
          pp[0] = m;
          pp[1] = s;
          pp[2] = __int_as_float(mi);
          pp[3] = 0.f;
        }
      }
    }
    __syncthreads();
  }

  if (OP != OP_LMHEAD) return;

  // ---- draft-token selection by the last CTA to finish
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(c.lm_cnt, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float cT = kLog2e / c.T;
  const int G = c.lm_grid;
  if (warp != 0) return;
  for (int b = 0; b < c.B; ++b) {
    const float *pb = c.lm_part + (size_t)b * G * 4;
    float M = -INFINITY;
    int Mi = 0x7fffffff;
    for (int cta = lane; cta < G; cta += 32) argmax_merge(M, Mi, __ldcg(&pb[cta * 4]), __float_as_int(__ldcg(&pb[cta * 4 + 2])));
    warp_argmax(M, Mi);
    int tok = Mi;
    if (M == -INFINITY || !(M == M)) {
      if (lane == 0) set_status(c.status, kStatusNonFinite);
      tok = 0;
    } else if (c.mode == 1) {
      // Inverse CDF of softmax(logits / T) at u: walk the per-CTA masses in
      // vocabulary order, then rescan the CTA that holds the crossing.
      const double u = (double)__ldg(&c.u_draft[b * c.k + c.j]);
      double Z = 0.0;
      if (lane == 0)
        for (int cta = 0; cta < G; ++cta) {
          const float mc = __ldcg(&pb[cta * 4]);
          if (mc != -INFINITY) Z += (double)__ldcg(&pb[cta * 4 + 1]) * (double)exp2f((mc - M) * cT);
        }
      Z = __shfl_sync(0xffffffffu, Z, 0);
      const double target = u * Z;
      int cstar = -1, clast = -1;
      double before = 0.0;
      if (lane == 0) {
        double cum = 0.0;
        for (int cta = 0; cta < G; ++cta) {
          const float mc = __ldcg(&pb[cta * 4]);
          if (mc == -INFINITY) continue;
          const double mass = (double)__ldcg(&pb[cta * 4 + 1]) * (double)exp2f((mc - M) * cT);
          if (mass > 0.0) clast = cta;
          if (cstar < 0 && cum + mass > target) {
            cstar = cta;
            before = cum;
          }
          cum += mass;
        }
        if (cstar < 0) {
          cstar = clast;
          before = -1.0;  // no crossing: take the last positive index
        }
      }
      cstar = __shfl_sync(0xffffffffu, cstar, 0);
      before = __shfl_sync(0xffffffffu, before, 0);
      // rows of CTA cstar (same split as the launch)
      const int lo = cstar * c.lm_rpc, hi = min(c.V, lo + c.lm_rpc);
      const float *lg = c.logits + ((size_t)b * c.k + c.j) * c.V;
      const int per = (hi - lo + 31) / 32;
      const int a0 = lo + lane * per, a1 = min(hi, a0 + per);
      double ls = 0.0;
      int lastpos = -1;
      for (int i = a0; i < a1; ++i) {
        const float w = exp2f((__ldcg(&lg[i]) - M) * cT);
        ls += (double)w;
        if (w > 0.f) lastpos = i;
      }
      // exclusive prefix of lane sums
      double incl = ls;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const double excl = incl - ls;
      int found = 0x7fffffff;
      if (before >= 0.0 && before + incl > target) {
        double cum = before + excl;
        for (int i = a0; i < a1; ++i) {
          cum += (double)exp2f((__ldcg(&lg[i]) - M) * cT);
          if (cum > target) {
            found = i;
            break;
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) found = min(found, __shfl_xor_sync(0xffffffffu, found, o));
      int lp = lastpos;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(0xffffffffu, lp, o));
      tok = found != 0x7fffffff ? found : (lp >= 0 ? lp : Mi);
    }
    if (lane == 0) c.draft_tok[b * c.k + c.j] = tok;
  }
  if (lane == 0) *c.lm_cnt = 0u;
}

// ---------------------------------------------------------------- planning / launch

GemvPlan plan_gemv(int op, int N, int K, int B, int num_sms) {
  GemvPlan g{};
  g.op = op;
  g.N = N;
  g.K = K;
  int P = 1;
  while (P < kGemvWarps && (K + P - 1) / P > 1024) P *= 2;
  g.P = P;
  g.PC = (((K + P - 1) / P) + 7) / 8 * 8;
  int nv = (g.PC + 255) / 256;
  nv = nv <= 1 ? 1 : nv <= 2 ? 2 : nv <= 4 ? 4 : nv <= 6 ? 6 : 9;
  g.nv = nv;
  g.bg = (B > 1 && nv <= 4) ? 2 : 1;
  g.ngroups = (B + g.bg - 1) / g.bg;
  int grid = num_sms;
  int rpc = (N + grid - 1) / grid;
  if (op == OP_GATEUP && (rpc & 1)) ++rpc;
  g.rows_per_cta = rpc;
  g.grid = (N + rpc - 1) / rpc;
  g.stages = 4;
  auto smem_for = [&](int stages) {
    size_t s = (size_t)kGemvWarps * stages * (g.PC * 2 + 8);
    s += (size_t)g.rows_per_cta * g.P * g.bg * 4;
    if (op == OP_LMHEAD) s += (size_t)g.rows_per_cta * g.bg * 4;
    s += (size_t)2 * B * 4 + 64 * 4;
    return s;
  };
  while (g.stages > 2 && smem_for(g.stages) > 110 * 1024) --g.stages;
  g.smem = smem_for(g.stages);
  return g;
}

template <int OP, int NV, int BG>
static cudaError_t launch_one(const DraftCtx &c, const GemvPlan &g, cudaStream_t s, bool pdl) {
  auto kern = gemv_kernel<OP, NV, BG>;
  static bool attr_done = false;  // per process; all devices share the limit
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    attr_done = true;
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

size_t attention_smem_bytes(int Dh) {
  return (size_t)2 * kAttnChunk * Dh * 2        // K, V chunk (bf16)
         + (size_t)kMaxGroup * Dh * 4           // q
         + (size_t)kMaxGroup * kAttnChunk * 4   // scores / probabilities
         + (size_t)4 * kMaxGroup * Dh * 4       // per-warp partial outputs
         + (size_t)kMaxGroup * 2 * 4 + 16;      // (max, sum) per head + mbarrier
}

template <int DH>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(DraftCtx c) {
  constexpr int CH = kAttnChunk, G8 = kMaxGroup, VPL = DH / 32, NW = kAttnThreads / 32;
  extern __shared__ __align__(128) unsigned char smem[];
  uint16_t *Ks = reinterpret_cast<uint16_t *>(smem);
  uint16_t *Vs = Ks + CH * DH;
  float *qs = reinterpret_cast<float *>(Vs + CH * DH);
  float *sc = qs + G8 * DH;
  float *red = sc + G8 * CH;
  float *ml = red + NW * G8 * DH;
  uint64_t *bar = reinterpret_cast<uint64_t *>(ml + G8 * 2);

  const int ch = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int group = c.Hq / c.Hkv;
  int L = __ldg(&c.ctx_len[b]);
  L = min(max(L, 0), c.Lmax - c.k);
  const int ntok = L + c.j + 1;
  const int t0 = ch * CH;
  if (t0 >= ntok) return;
  const int t1 = min(t0 + CH, ntok);
  const int n = t1 - t0;
  const int nctx = max(0, min(t1, L) - t0);
  const size_t base = (((size_t)b * c.Hkv + g) * c.Lmax + t0) * DH;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // context rows were written by the caller: stage them before waiting
  if (tid == 0 && nctx > 0) {
    const uint32_t bytes = (uint32_t)nctx * DH * 2;
    mbar_arrive_expect_tx(bar, 2 * bytes);
    bulk_g2s(Ks, c.kc + base, bytes, bar);
    bulk_g2s(Vs, c.vc + base, bytes, bar);
  }
  grid_dep_wait();
  grid_dep_launch();

  // rows appended by this call's draft depths, and the queries
  const int napp = n - nctx;
  for (int idx = tid; idx < napp * (DH / 8); idx += kAttnThreads) {
    const int r = nctx + idx / (DH / 8), e = (idx % (DH / 8)) * 8;
    *reinterpret_cast<uint4 *>(Ks + r * DH + e) = __ldcg(reinterpret_cast<const uint4 *>(c.kc + base + (size_t)r * DH + e));
    *reinterpret_cast<uint4 *>(Vs + r * DH + e) = __ldcg(reinterpret_cast<const uint4 *>(c.vc + base + (size_t)r * DH + e));
  }
  const int nq = c.Hq * DH;
  for (int idx = tid; idx < group * DH; idx += kAttnThreads) qs[idx] = __ldcg(&c.q[(size_t)b * nq + (size_t)g * group * DH + idx]);
  bool ok = true;
  if (nctx > 0) ok = mbar_wait(bar, 0, c.status);
  __syncthreads();

  float qr[G8][VPL];
#pragma unroll
  for (int h = 0; h < G8; ++h)
#pragma unroll
    for (int e = 0; e < VPL; ++e) qr[h][e] = h < group ? qs[h * DH + lane * VPL + e] : 0.f;

  const float scale = rsqrtf((float)DH) * kLog2e;
  for (int t = warp; t < n; t += NW) {
    float kv[VPL];
#pragma unroll
    for (int e = 0; e < VPL; ++e) kv[e] = __uint_as_float((uint32_t)Ks[t * DH + lane * VPL + e] << 16);
#pragma unroll
    for (int h = 0; h < G8; ++h) {
      if (h < group) {
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < VPL; ++e) s = fmaf(qr[h][e], kv[e], s);
        s = warp_sum(s);
        if (lane == 0) sc[h * CH + t] = s * scale;
      }
    }
  }
  __syncthreads();
  for (int h = warp; h < group; h += NW) {
    float m = -INFINITY;
    for (int t = lane; t < n; t += 32) m = fmaxf(m, sc[h * CH + t]);
    m = warp_max(m);
    float s = 0.f;
    for (int t = lane; t < n; t += 32) {
      const float pexp = exp2f(sc[h * CH + t] - m);
      sc[h * CH + t] = pexp;
      s += pexp;
    }
    s = warp_sum(s);
    if (lane == 0) {
      ml[2 * h] = m;
      ml[2 * h + 1] = s;
    }
  }
  __syncthreads();
  float acc[G8][VPL];
#pragma unroll
  for (int h = 0; h < G8; ++h)
#pragma unroll
    for (int e = 0; e < VPL; ++e) acc[h][e] = 0.f;
  for (int t = warp; t < n; t += NW) {
    float vv[VPL];
#pragma unroll
    for (int e = 0; e < VPL; ++e) vv[e] = __uint_as_float((uint32_t)Vs[t * DH + lane * VPL + e] << 16);
#pragma unroll
    for (int h = 0; h < G8; ++h) {
      if (h < group) {
        const float pw = sc[h * CH + t];
#pragma unroll
        for (int e = 0; e < VPL; ++e) acc[h][e] = fmaf(pw, vv[e], acc[h][e]);
      }
    }
  }
#pragma unroll
  for (int h = 0; h < G8; ++h)
    if (h < group)
#pragma unroll
      for (int e = 0; e < VPL; ++e) red[(warp * G8 + h) * DH + lane * VPL + e] = acc[h][e];
  __syncthreads();

  float *part = c.attn_part + (((size_t)b * c.Hkv + g) * c.attn_chunks + ch) * group * (DH + 2);
  for (int idx = tid; idx < group * DH; idx += kAttnThreads) {
    const int h = idx / DH, e = idx % DH;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) o += red[(w * G8 + h) * DH + e];
    part[h * (DH + 2) + 2 + e] = o;
  }
  if (tid < group) {
    part[tid * (DH + 2)] = ml[2 * tid];
    part[tid * (DH + 2) + 1] = ml[2 * tid + 1];
  }
  (void)ok;

  // the last chunk of this (sequence, kv head) to finish combines the partials
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  const int nchunks = (ntok + CH - 1) / CH;
  if (tid == 0) s_last = atomicAdd(&c.attn_cnt[b * c.Hkv + g], 1u) == (unsigned)(nchunks - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float *p0 = c.attn_part + ((size_t)b * c.Hkv + g) * c.attn_chunks * group * (DH + 2);
  for (int idx = tid; idx < group * DH; idx += kAttnThreads) {
    const int h = idx / DH, e = idx % DH;
    float M = -INFINITY;
    for (int cc = 0; cc < nchunks; ++cc) M = fmaxf(M, __ldcg(&p0[((size_t)cc * group + h) * (DH + 2)]));
    float Ls = 0.f, O = 0.f;
    for (int cc = 0; cc < nchunks; ++cc) {
      const float *pc = p0 + ((size_t)cc * group + h) * (DH + 2);
      const float wgt = exp2f(__ldcg(&pc[0]) - M);
      Ls = fmaf(__ldcg(&pc[1]), wgt, Ls);
      O = fmaf(__ldcg(&pc[2 + e]), wgt, O);
    }
    c.o[(size_t)b * nq + ((size_t)g * group + h) * DH + e] = O / Ls;
  }
  if (tid == 0) c.attn_cnt[b * c.Hkv + g] = 0u;
}

template <int DH>
static cudaError_t launch_attn_dh(const DraftCtx &c, cudaStream_t s, bool pdl) {
  auto kern = attn_kernel<DH>;
  static bool attr_done = false;
  const size_t smem = attention_smem_bytes(DH);
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(c.attn_chunks, c.Hkv, c.B);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  note_launch();
  return cudaLaunchKernelEx(&cfg, kern, c);
}

cudaError_t launch_attention(const DraftCtx &c, cudaStream_t s, bool pdl) {
  switch (c.Dh) {
    case 32: return launch_attn_dh<32>(c, s, pdl);
    case 64: return launch_attn_dh<64>(c, s, pdl);
    default: return launch_attn_dh<128>(c, s, pdl);
  }
}

}  // namespace mtp
