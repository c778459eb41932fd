// Device helpers shared by the draft-chain kernels (the weight-streaming GEMV
// path and the tensor-core path): RMSNorm scale factors, activation loads, the
// weight-row map of each operation and the draft-token selection over the
// vocabulary.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace mtp {


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

// Full-vocabulary id of draft-head row i (a reduced draft vocabulary maps its
// rows; an id outside [0, V) flags a bad token and reads as -1).
__device__ __forceinline__ int vocab_id(const DraftCtx &c, int i) {
  if (!c.vmap) return i;
  const int v = __ldg(&c.vmap[i]);
  if (v < 0 || v >= c.V) {
    set_status(c.status, kStatusBadToken);
    return -1;
  }
  return v;
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

// The same eight values with the norm's gain but not its scale -- the launch
// applies the scale to the finished dot products, W (s g x) = s (W (g x)), so
// no CTA has to reduce the whole vector before it starts streaming -- and the
// raw values' sum of squares added to sq0 (the first normalised vector) or sq1
// (the input projection's second one, the hidden state).
template <int OP>
__device__ __forceinline__ void act8_unscaled(const DraftCtx &c, int b, int col, float *out, float &sq0,
                                              float &sq1) {
  const int d = c.d;
  float g[8];
  if (OP == OP_FC) {
    if (col < d) {
      load8_bf16(c.E + (size_t)depth_token(c, b) * d + col, out);
      load8_bf16(c.g_emb + col, g);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        sq0 = fmaf(out[t], out[t], sq0);
        out[t] *= g[t];
      }
    } else {
      const int cc = col - d;
      if (c.j == 0) load8_bf16(c.h + (size_t)b * d + cc, out);
      else load8_f32(c.x2 + (size_t)b * d + cc, out);
      load8_bf16(c.g_hid + cc, g);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        sq1 = fmaf(out[t], out[t], sq1);
        out[t] *= g[t];
      }
    }
  } else {
    const float *x = OP == OP_QKV ? c.x0 : (OP == OP_GATEUP ? c.x1 : c.x2);
    const uint16_t *gp = OP == OP_QKV ? c.g_attn : (OP == OP_GATEUP ? c.g_mlp : c.g_final);
    load8_f32(x + (size_t)b * d + col, out);
    load8_bf16(gp + col, g);
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      sq0 = fmaf(out[t], out[t], sq0);
      out[t] *= g[t];
    }
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
  return c.head + (size_t)row * K;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.f + __expf(-z)); }


// The epilogue of one weight-streaming GEMV pass over batch group grp, run by
// the whole CTA: every row's P piece sums (part, in shared memory), the input
// norm's scale(s) from the warps' sums of squares (sq), the op's output -- x0;
// q and the bf16 K/V append; x1 = x0 + y; the SwiGLU product; x2 = x1 + y; the
// logits -- and, for the LM head, this CTA's (max, sum of exp2, argmax)
// partial per sequence in lm_part[b][cta].  ys and red are shared scratch.
template <int OP, int BG>
__device__ void gemv_epilogue(const DraftCtx &c, int P, int PC, int row0, int nrows, int grp, bool fac,
                              const float *part, const float *sq, float *ys, float *red, int cta) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  (void)PC;
  // epilogue for this batch group; the norm's scale(s) from the warps' sums
  float sc0[BG], sc1[BG];
#pragma unroll
  for (int bb = 0; bb < BG; ++bb) {
    sc0[bb] = 1.f;
    sc1[bb] = 1.f;
    if (fac) {
      float t0 = 0.f, t1 = 0.f;
      for (int w = 0; w < P; ++w) {
        t0 += sq[(w * BG + bb) * 2];
        t1 += sq[(w * BG + bb) * 2 + 1];
      }
      sc0[bb] = rsqrtf(t0 / (float)c.d + c.eps);
      sc1[bb] = rsqrtf(t1 / (float)c.d + c.eps);
    }
  }
  for (int rl = threadIdx.x; rl < nrows; rl += kGemvThreads) {
    const int row = row0 + rl;
    if (OP == OP_GATEUP && (rl & 1)) continue;
#pragma unroll
    for (int bb = 0; bb < BG; ++bb) {
      const int b = grp * BG + bb;
      if (b >= c.B) break;
      float y = 0.f;
      if (fac && OP == OP_FC) {  // pieces of the embedding half, then of the hidden half
        float ye = 0.f, yx = 0.f;
        for (int pp = 0; pp < P; ++pp) {
          const float v = part[((size_t)rl * P + pp) * BG + bb];
          if (pp * PC < c.d) ye += v;
          else yx += v;
        }
        y = sc0[bb] * ye + sc1[bb] * yx;
      } else {
        for (int pp = 0; pp < P; ++pp) y += part[((size_t)rl * P + pp) * BG + bb];
        if (fac) y *= sc0[bb];
      }
      if (OP == OP_FC) {
        if (in_bounds(row < c.d, c.status)) c.x0[(size_t)b * c.d + row] = y;
      } else if (OP == OP_QKV) {
        const int nq = c.Hq * c.Dh, nkv = c.Hkv * c.Dh;
        if (row < nq) {
          c.q[(size_t)b * nq + row] = y;
        } else if (in_bounds(row < nq + 2 * nkv, c.status)) {
          int r = row - nq;
          uint16_t *cache = r < nkv ? c.kc : c.vc;
          if (r >= nkv) r -= nkv;
          const int kvh = r / c.Dh, dd = r % c.Dh;
          int L = __ldg(&c.ctx_len[b]);
          if (L < 0 || L + c.k > c.Lmax) set_status(c.status, kStatusBadCtx);
          L = min(max(L, 0), c.Lmax - c.k);
          const size_t idx = (((size_t)b * c.Hkv + kvh) * c.Lmax + L + c.jc) * c.Dh + dd;
          if (in_bounds(L + c.jc < c.Lmax && kvh < c.Hkv, c.status))
            cache[idx] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
        }
      } else if (OP == OP_WO) {
        if (in_bounds(row < c.d, c.status)) c.x1[(size_t)b * c.d + row] = __ldcg(&c.x0[(size_t)b * c.d + row]) + y;
      } else if (OP == OP_GATEUP) {
        float up = 0.f;
        for (int pp = 0; pp < P; ++pp) up += part[((size_t)(rl + 1) * P + pp) * BG + bb];
        if (fac) up *= sc0[bb];
        if (in_bounds((row >> 1) < c.F, c.status)) c.act[(size_t)b * c.F + (row >> 1)] = silu_f(y) * up;
      } else if (OP == OP_DOWN) {
        if (in_bounds(row < c.d, c.status)) c.x2[(size_t)b * c.d + row] = __ldcg(&c.x1[(size_t)b * c.d + row]) + y;
      } else {  // LM head
        if (c.logits) {
          const int v = vocab_id(c, row);
          if (v >= 0 && in_bounds(v < c.V && c.j < c.k, c.status)) c.logits[((size_t)b * c.k + c.j) * c.V + v] = y;
        }
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
      if ((c.mode == 1 || c.k_eff) && m != -INFINITY)
        for (int rl = threadIdx.x; rl < nrows; rl += kGemvThreads) s += exp2f((ys[(size_t)rl * BG + bb] - m) * cT);
      s = block_sum_256(s, red + 2 * kGemvWarps);
      // a launch wider than the LM head's plan (several ops in one launch) has
      // CTAs without vocabulary rows: they own no partial slot
      if (threadIdx.x == 0 && cta < c.lm_grid && in_bounds(c.lm_grid <= kMaxLmGrid, c.status)) {
        float *pp = c.lm_part + ((size_t)b * c.lm_grid + cta) * 4;
        pp[0] = m;
        pp[1] = s;
        pp[2] = __int_as_float(mi);
        pp[3] = 0.f;
      }
    }
  }
}

// Dynamic draft length: a sequence still drafting stops at this depth when the
// draft's largest probability (1 / the partition sum relative to the largest
// term) is below stop_p; it keeps the c.j drafts before this one.
__device__ __forceinline__ void stop_check(const DraftCtx &c, int b, double conf) {
  if (conf < (double)c.stop_p && c.k_eff[b] == c.k) {
    c.k_eff[b] = c.j;
    atomicSub(c.n_active, 1u);
  }
}

// Draft-token selection over the vocabulary, run by one warp after every
// LM-head CTA has written its per-sequence partials lm_part[b][cta] =
// (max, sum of exp2((logit - max) * log2e / T), argmax).  CTA cta owns the
// vocabulary rows [cta * rpc, (cta + 1) * rpc).
// Greedy: the argmax, lowest index on ties.  Stochastic: the inverse CDF of
// softmax(logits / T) at u_draft[b, j] -- walk the per-CTA masses in vocabulary
// order, then rescan the CTA that holds the crossing in float64.
__device__ inline void lm_select_warp(const DraftCtx &c, int G, int rpc) {
  const int lane = threadIdx.x & 31;
  const float cT = kLog2e / c.T;
  for (int b = 0; b < c.B; ++b) {
    const float *pb = c.lm_part + (size_t)b * G * 4;
    float M = -INFINITY;
    int Mi = 0x7fffffff;
    for (int cta = lane; cta < G; cta += 32) argmax_merge(M, Mi, __ldcg(&pb[cta * 4]), __float_as_int(__ldcg(&pb[cta * 4 + 2])));
    warp_argmax(M, Mi);
    int tok = Mi;
    const bool finite = !(M == -INFINITY || !(M == M));
    // the partition sum of softmax(logits / T) relative to its largest term
    double Z = 0.0;
    if (finite && c.mode == 1) {  // in vocabulary order, as the walk below adds them up
      if (lane == 0)
        for (int cta = 0; cta < G; ++cta) {
          const float mc = __ldcg(&pb[cta * 4]);
          if (mc != -INFINITY) Z += (double)__ldcg(&pb[cta * 4 + 1]) * (double)exp2f((mc - M) * cT);
        }
      Z = __shfl_sync(0xffffffffu, Z, 0);
    } else if (finite && c.k_eff) {  // greedy: only the total, over the lanes
      for (int cta = lane; cta < G; cta += 32) {
        const float mc = __ldcg(&pb[cta * 4]);
        if (mc != -INFINITY) Z += (double)__ldcg(&pb[cta * 4 + 1]) * (double)exp2f((mc - M) * cT);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);
    }
    if (!finite) {
      if (lane == 0) set_status(c.status, kStatusNonFinite);
      tok = 0;
    } else if (c.mode == 1) {
      // Inverse CDF of softmax(logits / T) at u: walk the per-CTA masses in
      // vocabulary order, then rescan the CTA that holds the crossing.
      const double u = (double)__ldg(&c.u_draft[b * c.k + c.j]);
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
      const int lo = cstar * rpc, hi = min(c.Vd, lo + rpc);
      const float *lg = c.logits + ((size_t)b * c.k + c.j) * c.V;  // head row i at vocab_id(i)
      const int per = (hi - lo + 31) / 32;
      const int a0 = lo + lane * per, a1 = min(hi, a0 + per);
      auto logit = [&](int i) {
        const int v = vocab_id(c, i);
        return v < 0 ? -INFINITY : __ldcg(&lg[v]);
      };
      double ls = 0.0;
      int lastpos = -1;
      for (int i = a0; i < a1; ++i) {
        const float w = exp2f((logit(i) - M) * cT);
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
          cum += (double)exp2f((logit(i) - M) * cT);
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
    if (finite) tok = vocab_id(c, tok);  // head row -> vocabulary id
    if (lane == 0 && in_bounds(c.j < c.k, c.status)) c.draft_tok[b * c.k + c.j] = tok;
    if (lane == 0 && c.k_eff && finite) stop_check(c, b, 1.0 / Z);
  }
  if (lane == 0) *c.lm_cnt = 0u;
}

}  // namespace mtp
