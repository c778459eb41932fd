// Decode attention on tensor cores ("The Tiny Draft Model Hidden Inside Qwen",
// opening section: the draft block is one full-attention transformer block
// over the KV cache; GQA shapes of the pages' models).
//
// One (sequence, kv head) per cluster of C CTAs, CTA r taking a contiguous
// range of the ntok = L_b + j + 1 visible cache rows (as the CUDA-core
// kernel).  The K/V rows arrive in tiles of 64 by 2-D TMA with the 128-byte
// swizzle, so that ldmatrix reads them without bank conflicts.  Each of four
// compute warps takes 16 rows of every tile and keeps a flash-decoding state
// for the GQA group's query heads, padded to 16 rows:
//   S = Q K^T   mma.m16n8k16 (bf16 in, fp32 accumulate): Q is split into three
//               bf16 terms (hi + mid + lo carry all 24 bits of its fp32
//               mantissa); K is bf16 in the cache, so S is exact to fp32
//               rounding of the products' sum;
//   online softmax on the accumulator fragments (row max and sum over the
//               four lanes holding a head's row);
//   O += P V    P in three bf16 terms again, V bf16 from the cache.
// Warps merge through shared memory, CTAs through distributed shared memory.
#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

#include <stdlib.h>

#include <mutex>

namespace mtp {

namespace {

constexpr int kTcRows = 64;      // cache rows per tile
constexpr int kTcWarps = 4;      // compute warps (16 rows of every tile each)
constexpr int kTcStages = 3;     // ring stages
constexpr int kTcThreads = 32 * (kTcWarps + 1);
constexpr int kBox = 64 * kTcRows * 2;  // one 64-dim x 64-row box: 8 KB
constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kMaxCluster = 16;  // CTAs per (sequence, kv head) at most

struct AttnTcArgs {
  CUtensorMap mk, mv;  // [B*Hkv*Lmax, Dh] bf16 views of the caches
  DraftCtx c;
};

template <int DH>
struct TcLayout {
  static constexpr int NB = DH / 64;                   // boxes per K (or V) tile
  static constexpr int STAGE = 2 * NB * kBox;          // K boxes, then V boxes
  static constexpr int QLD = DH + 8;                   // padded bf16 row of a q term
  static constexpr int RING = kTcStages * STAGE;
  static constexpr int QS = 3 * 16 * QLD * 2;
  static constexpr size_t SMEM = (size_t)RING + QS + 2 * 16 * 4 + 2 * kTcStages * 8 + 1024;
  // after the loop the ring holds the warps' states and the CTA's output
  static constexpr int WST = kTcWarps * 16 * (DH + 2) * 4;
  static_assert(WST + 16 * DH * 4 <= RING, "merge buffers fit the ring");
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A B for one m16n8k16 tile (bf16 operands, fp32 accumulator).
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// Split two fp32 values into three packed bf16 terms that sum to them.
__device__ __forceinline__ void split3(float x, float y, uint32_t &h, uint32_t &m, uint32_t &l) {
  h = pack_bf16(x, y);
  const float rx = x - bf16_lo(h), ry = y - bf16_hi(h);
  m = pack_bf16(rx, ry);
  l = pack_bf16(rx - bf16_lo(m), ry - bf16_hi(m));
}

// Byte offset of (row r, 16-byte chunk c) in a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

}  // namespace

template <int DH>
__global__ void __launch_bounds__(kTcThreads, 2) attn_tc_kernel(const __grid_constant__ AttnTcArgs p) {
  trace_start(kTkAttnTc);
  using Ly = TcLayout<DH>;
  constexpr int NB = Ly::NB, KS = DH / 16, ND = DH / 8;
  extern __shared__ unsigned char smem_raw[];
  // swizzled boxes need 1024-byte alignment
  unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char *ring = smem;
  uint16_t *qs = reinterpret_cast<uint16_t *>(smem + Ly::RING);          // [3][16][QLD]
  float *mrun = reinterpret_cast<float *>(smem + Ly::RING + Ly::QS);    // [16]
  float *lrun = mrun + 16;                                              // [16]
  uint64_t *full = reinterpret_cast<uint64_t *>(lrun + 16);
  uint64_t *empty = full + kTcStages;
  float *wst = reinterpret_cast<float *>(ring);                         // [warps][16][DH+2], after the loop
  float *qo = wst + kTcWarps * 16 * (DH + 2);                           // [16][DH], after the loop

  const DraftCtx &c = p.c;
  // longest contexts first, so that the last clusters to be scheduled are short
  const int g = blockIdx.y, b = c.seq_order ? __ldg(&c.seq_order[blockIdx.z]) : (int)blockIdx.z;
  const int C = (int)cluster_size(), rank = (int)cluster_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int group = c.Hq / c.Hkv;
  int L = __ldg(&c.ctx_len[b]);
  L = min(max(L, 0), c.Lmax - c.k);
  const int ntok = L + c.jc + 1;
  const int T = (ntok + C - 1) / C;
  const int r0 = min(ntok, rank * T), r1 = min(ntok, r0 + T);
  const int ntiles = (r1 - r0 + kTcRows - 1) / kTcRows;
  const int rowbase = (b * c.Hkv + g) * c.Lmax;

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kTcWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  bool ok = true;
  if (warp == kTcWarps) {
    // ------------------------------------------------ K/V producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      bool waited = false;
      int issued = 0;
      for (int i = 0; i < ntiles && ok; ++i) {
        const int s = i % kTcStages;
        if (i >= kTcStages) ok = mbar_wait(&empty[s], (uint32_t)((i / kTcStages) - 1) & 1u, c.status);
        if (!ok) break;
        const int t0 = r0 + i * kTcRows;
        if (!waited && t0 + kTcRows > L) {  // rows L.. are appended by this chain
          grid_dep_wait();
          waited = true;
        }
        mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * NB * kBox));
        unsigned char *st = ring + (size_t)s * Ly::STAGE;
        for (int bx = 0; bx < NB; ++bx) {
          tma_load_2d(st + bx * kBox, &p.mk, 64 * bx, rowbase + t0, &full[s], pol);
          tma_load_2d(st + (NB + bx) * kBox, &p.mv, 64 * bx, rowbase + t0, &full[s], pol);
        }
        issued = i + 1;
      }
      if (!waited) grid_dep_wait();
      if (!ok)  // let copies still in flight land before the CTA exits
        for (int i = max(0, issued - kTcStages); i < issued; ++i)
          if (!mbar_wait(&full[i % kTcStages], (uint32_t)(i / kTcStages) & 1u, c.status)) break;
    }
    grid_dep_launch();
  } else {
    // ------------------------------------------------ compute warps
    grid_dep_wait();  // q comes from this depth's projection
    grid_dep_launch();
    trace_dep(kTkAttnTc);
    // the group's query heads, rows 0..15 (zero past the group), in three bf16 terms
    const int nq = c.Hq * DH;
    {
      // every load first (one round trip), then the splits and stores
      constexpr int PER = 16 * DH / 2 / (32 * kTcWarps);
      float2 qv[PER];
#pragma unroll
      for (int t = 0; t < PER; ++t) {
        const int idx = tid + t * 32 * kTcWarps;
        const int h = idx / (DH / 2), e = 2 * (idx % (DH / 2));
        qv[t] = h < group ? __ldcg(reinterpret_cast<const float2 *>(c.q + (size_t)b * nq +
                                                                     ((size_t)g * group + h) * DH + e))
                          : make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int t = 0; t < PER; ++t) {
        const int idx = tid + t * 32 * kTcWarps;
        const int h = idx / (DH / 2), e = 2 * (idx % (DH / 2));
        uint32_t th, tm, tl;
        split3(qv[t].x, qv[t].y, th, tm, tl);
        *reinterpret_cast<uint32_t *>(qs + (0 * 16 + h) * Ly::QLD + e) = th;
        *reinterpret_cast<uint32_t *>(qs + (1 * 16 + h) * Ly::QLD + e) = tm;
        *reinterpret_cast<uint32_t *>(qs + (2 * 16 + h) * Ly::QLD + e) = tl;
      }
    }
    named_sync(1, 32 * kTcWarps);
    trace_mark(kTkAttnTc, 0);  // query staged

    const int gq = lane >> 2, tq = lane & 3;  // fragment row / column-pair of this lane
    const float scale = rsqrtf((float)DH) * kLog2e;
    // q fragment addresses: lane -> (head row, dim column) of its 8x8 matrix
    const int qrow = (lane & 7) + 8 * ((lane >> 3) & 1), qcol = 8 * (lane >> 4);
    const uint32_t qbase = smem_u32(qs) + (uint32_t)((qrow * Ly::QLD + qcol) * 2);
    float o[ND][4];
#pragma unroll
    for (int n = 0; n < ND; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows gq and gq + 8

    for (int i = 0; i < ntiles; ++i) {
      const int s = i % kTcStages;
      if (ok) ok = mbar_wait(&full[s], (uint32_t)(i / kTcStages) & 1u, c.status);
      ok = __all_sync(kFullMask, ok);
      const int t0 = r0 + i * kTcRows;
      const int R0 = 16 * warp;  // this warp's rows of the tile
      const int nvalid = min(16, max(0, r1 - (t0 + R0)));
      const uint32_t kb = smem_u32(ring + (size_t)s * Ly::STAGE), vb = kb + NB * kBox;
      if (ok && nvalid > 0) {
        // ---- S = Q K^T over this warp's 16 rows (two n-tiles of 8 rows)
        float sacc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ks += 2) {
          uint32_t kf[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int r = R0 + 8 * nt + (lane & 7);
            const int kk = ks + (lane >> 4);            // k-step of this lane's matrix
            const int chunk = 2 * (kk & 3) + ((lane >> 3) & 1);
            ldsm_x4(kb + (uint32_t)((kk >> 2) * kBox) + swz(r, chunk), kf[nt][0], kf[nt][1], kf[nt][2], kf[nt][3]);
          }
#pragma unroll
          for (int kx = 0; kx < 2; ++kx) {
#pragma unroll
            for (int tm = 0; tm < 3; ++tm) {
              uint32_t a0, a1, a2, a3;
              ldsm_x4(qbase + (uint32_t)((tm * 16 * Ly::QLD + (ks + kx) * 16) * 2), a0, a1, a2, a3);
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) mma16816(sacc[nt], a0, a1, a2, a3, kf[nt][2 * kx], kf[nt][2 * kx + 1]);
            }
          }
        }
        // ---- online softmax: rows gq (values 0, 1) and gq + 8 (values 2, 3)
        float sv[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int rr = 8 * nt + 2 * tq + (e & 1);  // row of the warp's 16
            sv[nt][e] = rr < nvalid ? sacc[nt][e] * scale : -INFINITY;
          }
        float x0 = fmaxf(fmaxf(sv[0][0], sv[0][1]), fmaxf(sv[1][0], sv[1][1]));
        float x1 = fmaxf(fmaxf(sv[0][2], sv[0][3]), fmaxf(sv[1][2], sv[1][3]));
        x0 = fmaxf(x0, __shfl_xor_sync(kFullMask, x0, 1));
        x1 = fmaxf(x1, __shfl_xor_sync(kFullMask, x1, 1));
        x0 = fmaxf(x0, __shfl_xor_sync(kFullMask, x0, 2));
        x1 = fmaxf(x1, __shfl_xor_sync(kFullMask, x1, 2));
        const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
        const float f0 = n0 == -INFINITY ? 1.f : exp2f(m0 - n0), f1 = n1 == -INFINITY ? 1.f : exp2f(m1 - n1);
        float pv[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          pv[nt][0] = n0 == -INFINITY ? 0.f : exp2f(sv[nt][0] - n0);
          pv[nt][1] = n0 == -INFINITY ? 0.f : exp2f(sv[nt][1] - n0);
          pv[nt][2] = n1 == -INFINITY ? 0.f : exp2f(sv[nt][2] - n1);
          pv[nt][3] = n1 == -INFINITY ? 0.f : exp2f(sv[nt][3] - n1);
        }
        float s0 = pv[0][0] + pv[0][1] + pv[1][0] + pv[1][1];
        float s1 = pv[0][2] + pv[0][3] + pv[1][2] + pv[1][3];
        s0 += __shfl_xor_sync(kFullMask, s0, 1);
        s1 += __shfl_xor_sync(kFullMask, s1, 1);
        s0 += __shfl_xor_sync(kFullMask, s0, 2);
        s1 += __shfl_xor_sync(kFullMask, s1, 2);
        l0 = l0 * f0 + s0;
        l1 = l1 * f1 + s1;
        m0 = n0;
        m1 = n1;
#pragma unroll
        for (int n = 0; n < ND; ++n) {
          o[n][0] *= f0;
          o[n][1] *= f0;
          o[n][2] *= f1;
          o[n][3] *= f1;
        }
        // ---- O += P V: P as the A operand (its accumulator layout is the
        // A fragment layout), in three bf16 terms
        uint32_t pa[3][4];
        split3(pv[0][0], pv[0][1], pa[0][0], pa[1][0], pa[2][0]);
        split3(pv[0][2], pv[0][3], pa[0][1], pa[1][1], pa[2][1]);
        split3(pv[1][0], pv[1][1], pa[0][2], pa[1][2], pa[2][2]);
        split3(pv[1][2], pv[1][3], pa[0][3], pa[1][3], pa[2][3]);
        const int vr = R0 + (lane & 7) + 8 * ((lane >> 3) & 1);  // V row of this lane's matrix
#pragma unroll
        for (int n = 0; n < ND; n += 2) {
          const int chunk = n + (lane >> 4);  // 8-dim chunk of this lane's matrix
          uint32_t v0, v1, v2, v3;
          ldsm_x4_t(vb + (uint32_t)((chunk >> 3) * kBox) + swz(vr, chunk & 7), v0, v1, v2, v3);
#pragma unroll
          for (int tm = 0; tm < 3; ++tm) {
            mma16816(o[n], pa[tm][0], pa[tm][1], pa[tm][2], pa[tm][3], v0, v1);
            mma16816(o[n + 1], pa[tm][0], pa[tm][1], pa[tm][2], pa[tm][3], v2, v3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage
    }
    // the warp's state for heads gq < group: (m, l) and O[gq][8n + 2tq, +1]
    named_sync(1, 32 * kTcWarps);  // every warp is past the ring: it now holds the states
    trace_mark(kTkAttnTc, 1);      // last tile done
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = gq + 8 * hh;
      if (h < group) {
        float *ws = wst + ((size_t)warp * 16 + h) * (DH + 2);
        if (tq == 0) {
          ws[0] = hh ? m1 : m0;
          ws[1] = hh ? l1 : l0;
        }
#pragma unroll
        for (int n = 0; n < ND; ++n) {
          ws[2 + 8 * n + 2 * tq] = o[n][2 * hh];
          ws[2 + 8 * n + 2 * tq + 1] = o[n][2 * hh + 1];
        }
      }
    }
  }
  __syncthreads();
  // merge the warps of the CTA
  for (int idx = tid; idx < group * DH; idx += kTcThreads) {
    const int h = idx / DH, e = idx % DH;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kTcWarps; ++w) M = fmaxf(M, wst[((size_t)w * 16 + h) * (DH + 2)]);
    float Ls = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kTcWarps; ++w) {
      const float *ws = wst + ((size_t)w * 16 + h) * (DH + 2);
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
  trace_mark(kTkAttnTc, 2);  // CTA merged
  cluster_sync();
  for (int idx = rank + C * tid; idx < group * DH; idx += C * kTcThreads) {
    const int h = idx / DH, e = idx % DH;
    // every peer's (m, l, o) first: the remote loads are independent, so they
    // are all in flight at once
    float mr[kMaxCluster], lr[kMaxCluster], orr[kMaxCluster];
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) {
      if (r < C) {
        mr[r] = *dsmem_ptr(&mrun[h], r);
        lr[r] = *dsmem_ptr(&lrun[h], r);
        orr[r] = *dsmem_ptr(&qo[h * DH + e], r);
      }
    }
    float M = -INFINITY, Ls = 0.f, O = 0.f;
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r)
      if (r < C) M = fmaxf(M, mr[r]);
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) {
      if (r < C && mr[r] != -INFINITY) {
        const float wgt = exp2f(mr[r] - M);
        Ls = fmaf(lr[r], wgt, Ls);
        O = fmaf(orr[r], wgt, O);
      }
    }
    c.o[(size_t)b * nq + ((size_t)g * group + h) * DH + e] = O / Ls;
  }
  trace_mark(kTkAttnTc, 3);  // cluster combined
  cluster_sync();  // keep this CTA's shared memory alive until every peer has read it
  trace_end(kTkAttnTc);
}

// ---------------------------------------------------------------- host side

namespace {

struct MapCache {
  const void *kc = nullptr, *vc = nullptr;
  int B = 0, Hkv = 0, Lmax = 0, Dh = 0;
  CUtensorMap mk{}, mv{};
  bool ok = false;
};
std::mutex g_map_mu;
MapCache g_maps;

template <int DH>
cudaError_t launch_tc(const DraftCtx &c, int cluster, cudaStream_t s, bool pdl) {
  using Ly = TcLayout<DH>;
  static unsigned long long attr_ctx = 0;  // the context the attributes were set in
  auto kern = attn_tc_kernel<DH>;
  const unsigned long long cid = context_id();
  if (cid == 0 || cid != attr_ctx) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Ly::SMEM);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr_ctx = cid;
  }
  AttnTcArgs a;
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    MapCache &m = g_maps;
    if (!m.ok || m.kc != c.kc || m.vc != c.vc || m.B != c.B || m.Hkv != c.Hkv || m.Lmax != c.Lmax || m.Dh != DH) {
      const uint64_t rows = (uint64_t)c.B * c.Hkv * c.Lmax;
      m.ok = make_bf16_map(&m.mk, c.kc, DH, rows, DH, kTcRows) && make_bf16_map(&m.mv, c.vc, DH, rows, DH, kTcRows);
      m.kc = c.kc;
      m.vc = c.vc;
      m.B = c.B;
      m.Hkv = c.Hkv;
      m.Lmax = c.Lmax;
      m.Dh = DH;
      if (!m.ok) return cudaErrorNotSupported;
    }
    a.mk = m.mk;
    a.mv = m.mv;
  }
  a.c = c;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(cluster, c.Hkv, c.B);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = Ly::SMEM;
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
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

bool attention_tc_shape_ok(const DraftCtx &c) {
  const int group = c.Hkv > 0 ? c.Hq / c.Hkv : 0;
  const char *off = getenv("MTP_ATTN_TC");
  if (off && off[0] == '0') return false;
  return (c.Dh == 64 || c.Dh == 128) && group >= 2 && group <= 16 && tc_available() &&
         (uint64_t)c.B * c.Hkv * c.Lmax < (1ull << 31);
}

cudaError_t launch_attention_tc(const DraftCtx &c, int cluster, cudaStream_t s, bool pdl) {
  return c.Dh == 64 ? launch_tc<64>(c, cluster, s, pdl) : launch_tc<128>(c, cluster, s, pdl);
}

MTP_TRACE_COLLECTOR(attn_tc)

}  // namespace mtp
