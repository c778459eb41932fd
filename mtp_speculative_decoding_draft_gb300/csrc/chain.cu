// Several weight-streaming GEMV operations of the draft chain in one
// persistent launch, for the small batches of the GEMV path.
//
// One depth of the module is a run of matrix-vector products ("The Tiny Draft
// Model Hidden Inside Qwen", sections "One step deeper than the main model"
// and "What vLLM and SGLang do with the weights"), and at a batch of one each
// is bound by streaming its weight matrix ("Speculative Decoding and MTP: Why
// Guessing Is Free", section "The part that got me").  Launched one by one,
// every product drains its weight stream at its end and the next one fills its
// own: for the matrices of 30 to 200 MB that costs a fifth of their time.
// Here the products run back to back in one cooperative launch, separated by
// grid barriers, and each warp's weight stream does not stop at a barrier:
//
//  * the whole launch is one stream of weight pieces per warp (op after op:
//    the pieces of op o+1 follow those of op o), fed through a byte ring of
//    shared memory by 1-D TMA bulk copies; a piece is the warp's column slice
//    of one weight row, so pieces of different ops differ in size, and a piece
//    that does not fit at the ring's end starts at its beginning;
//  * weights do not depend on activations, so while a warp finishes op o and
//    waits at the barrier, its ring already fills with op o+1's pieces;
//  * after each op the CTA runs the same epilogue as the one-launch kernel
//    (residual adds, SwiGLU, the bf16 K/V append, the LM head's partials); the
//    barrier after the LM head selects the draft token -- the last CTA to
//    arrive does it before releasing the others -- so the next depth's input
//    projection can start in the same launch.
//
// A launch covers either [input projection, QKV] of depth 0, or [output
// projection, gate/up, down, LM head + selection] of depth j followed by
// [input projection, QKV] of depth j + 1 (the attention of each depth runs as
// its own launch in between).  Every wait is bounded; a timeout flags the
// status word and every CTA leaves at its next barrier.
#include "common.cuh"
#include "draft_ops.cuh"
#include "internal.h"

namespace mtp {

namespace {

constexpr int kRingSlots = 8;  // pieces in flight per warp, at most

// Runtime form of weight_row<OP>.
__device__ __forceinline__ const uint16_t *op_weight_row(const DraftCtx &c, int op, int row, int K) {
  switch (op) {
    case OP_FC: return weight_row<OP_FC>(c, row, K);
    case OP_QKV: return weight_row<OP_QKV>(c, row, K);
    case OP_WO: return weight_row<OP_WO>(c, row, K);
    case OP_GATEUP: return weight_row<OP_GATEUP>(c, row, K);
    case OP_DOWN: return weight_row<OP_DOWN>(c, row, K);
    default: return weight_row<OP_LMHEAD>(c, row, K);
  }
}

// This warp's share of one op: its column piece of the CTA's rows.
struct WarpGeom {
  int P, R, p, rs, row0, nrows, col0, ncols, upg, total;
};

__device__ __forceinline__ WarpGeom warp_geom(const GemvPlan &g, int warp) {
  WarpGeom w;
  w.P = g.P;
  w.R = kGemvWarps / g.P;
  w.p = warp % g.P;
  w.rs = warp / g.P;
  w.row0 = blockIdx.x * g.rows_per_cta;
  w.nrows = max(0, min(g.rows_per_cta, g.N - w.row0));
  w.col0 = w.p * g.PC;
  w.ncols = max(0, min(g.PC, g.K - w.col0));
  w.upg = w.nrows > w.rs ? (w.nrows - w.rs + w.R - 1) / w.R : 0;
  w.total = w.ncols > 0 ? w.upg * g.ngroups : 0;
  return w;
}

// The warp's stream of weight pieces across the launch's ops, through its byte
// ring.  Every field is warp-uniform; lane 0 issues the copies.  Positions in
// the ring and the producer's op geometry advance incrementally: the
// bookkeeping of a piece costs a handful of instructions, not divisions.
struct Ring {
  unsigned char *buf;
  uint64_t *bars;
  uint32_t bytes;               // ring size
  uint32_t prod_off, cons_off;  // byte offsets (monotonic), padding included
  uint32_t prod_pos, cons_pos;  // the same offsets within the ring
  uint32_t n_iss, n_con;        // pieces issued / consumed
  int io;                       // the op whose pieces are being issued
  int left, pu;                 // its pieces still to issue; unit within the batch group
  int rowb, R, upg, col0;       // its geometry for this warp: first row, row step, units, first column
  uint32_t sz;                  // its piece bytes
  int nops;
};

__device__ void ring_issue(Ring &r, const ChainArgs &a, int warp, uint64_t pol) {
  const int lane = threadIdx.x & 31;
  while (r.n_iss - r.n_con < (uint32_t)kRingSlots) {
    if (r.left == 0) {  // on to the next op that gives this warp pieces
      if (r.io + 1 >= r.nops) break;
      ++r.io;
      const WarpGeom w = warp_geom(a.ops[r.io].g, warp);
      r.left = w.total;
      r.pu = 0;
      r.rowb = w.row0 + w.rs;
      r.R = w.R;
      r.upg = w.upg;
      r.col0 = w.col0;
      r.sz = (uint32_t)w.ncols * 2u;
      continue;
    }
    const uint32_t sz = r.sz;
    const uint32_t pad = r.prod_pos + sz > r.bytes ? r.bytes - r.prod_pos : 0u;
    const uint32_t off = r.prod_off + pad;
    if (off + sz > r.cons_off + r.bytes) break;  // no room until the oldest piece is consumed
    const uint32_t pos = pad ? 0u : r.prod_pos;
    const int slot = (int)(r.n_iss & (kRingSlots - 1));
    if (lane == 0) {
      const ChainOp &op = a.ops[r.io];
      const int row = r.rowb + r.pu * r.R;
      mbar_arrive_expect_tx(&r.bars[slot], sz);
      bulk_g2s_hint(r.buf + pos, op_weight_row(a.c[op.ctx], op.op, row, op.g.K) + r.col0, sz, &r.bars[slot], pol);
    }
    r.prod_off = off + sz;
    r.prod_pos = pos + sz;
    ++r.n_iss;
    --r.left;
    if (++r.pu == r.upg) r.pu = 0;
  }
}

// Wait for the next piece (of sz bytes) to land; returns its data.
__device__ __forceinline__ const unsigned char *ring_wait(Ring &r, uint32_t sz, int *status, bool &ok) {
  const int slot = (int)(r.n_con & (kRingSlots - 1));
  if (ok) ok = mbar_sleep_wait(&r.bars[slot], (r.n_con / kRingSlots) & 1u, status);
  ok = __all_sync(0xffffffffu, ok);
  const uint32_t pos = r.cons_pos + sz > r.bytes ? 0u : r.cons_pos;
  return r.buf + pos;
}

// The piece is consumed: its bytes (and any padding before it) are free.
__device__ __forceinline__ void ring_release(Ring &r, uint32_t sz) {
  const uint32_t pad = r.cons_pos + sz > r.bytes ? r.bytes - r.cons_pos : 0u;
  r.cons_off += pad + sz;
  r.cons_pos = (pad ? 0u : r.cons_pos) + sz;
  ++r.n_con;
}

// Grid barrier of the cooperative launch.  With `select`, the last CTA to
// arrive picks the draft token of context cs (one warp; the LM head's
// partials of every CTA are in place by then) before releasing the others.
// Returns false when a wait ran out or another thread has flagged a timeout.
__device__ bool grid_barrier(const ChainArgs &a, bool select, const DraftCtx &cs) {
  __shared__ unsigned s_gen;
  __shared__ int s_last, s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    s_gen = ld_acquire_u32(&a.bar[1]);
    __threadfence();
    s_last = atomicAdd(&a.bar[0], 1u) == gridDim.x - 1u;
    __threadfence();
    s_ok = 1;
  }
  __syncthreads();
  if (s_last) {
    if (select && threadIdx.x < 32) lm_select_warp(cs, cs.lm_grid, cs.lm_rpc);
    __syncthreads();
    if (threadIdx.x == 0) {
      a.bar[0] = 0u;
      __threadfence();
      st_release_u32(&a.bar[1], s_gen + 1u);
    }
  } else if (threadIdx.x == 0) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0; ld_acquire_u32(&a.bar[1]) == s_gen; ++it) {
      if ((it & 63u) == 63u) {
        if (*reinterpret_cast<volatile int *>(a.status) & kStatusTimeout) {
          s_ok = 0;
          break;
        }
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          set_status(a.status, kStatusTimeout);
          s_ok = 0;
          break;
        }
      }
      __nanosleep(64);
    }
    __threadfence();
  }
  __syncthreads();
  return s_ok != 0 && !(*reinterpret_cast<volatile int *>(a.status) & kStatusTimeout);
}

// One op: activations, the warp's pieces, then the CTA's epilogue.
template <int OP, int NVM, int BG>
__device__ bool run_op(const ChainArgs &a, const ChainOp &co, Ring &ring, int warp, float *part, float *sq, float *ys,
                       float *red, uint64_t pol) {
  const DraftCtx &c = a.c[co.ctx];
  const GemvPlan &g = co.g;
  const int lane = threadIdx.x & 31;
  const WarpGeom w = warp_geom(g, warp);
  const bool fac = g.factor != 0;
  const uint32_t sz = (uint32_t)w.ncols * 2u;
  if (OP == OP_FC && c.zero_counters && blockIdx.x == 0 && c.k_eff) {
    for (int b = threadIdx.x; b < c.B; b += kGemvThreads) c.k_eff[b] = c.k;
    if (threadIdx.x == 0) *c.n_active = (unsigned)c.B;
  }
  bool ok = true;
  for (int grp = 0; grp < g.ngroups; ++grp) {
    float act[BG][NVM][8];
    float s0[BG], s1[BG];
#pragma unroll
    for (int bb = 0; bb < BG; ++bb) {
      const int b = grp * BG + bb;
      s0[bb] = 0.f;
      s1[bb] = 0.f;
#pragma unroll
      for (int i = 0; i < NVM; ++i) {
        const int v = lane + 32 * i;
        if (b < c.B && v * 8 < w.ncols) {
          // ops with an input norm apply its scale to the finished dot products
          // (the launch only chains plans that do); the output and down
          // projections read their input as it is
          if (fac) act8_unscaled<OP>(c, b, w.col0 + v * 8, act[bb][i], s0[bb], s1[bb]);
          else act8<OP>(c, b, w.col0 + v * 8, nullptr, act[bb][i]);
        } else {
#pragma unroll
          for (int t = 0; t < 8; ++t) act[bb][i][t] = 0.f;
        }
      }
    }
    if (fac) {
#pragma unroll
      for (int bb = 0; bb < BG; ++bb) {
        s0[bb] = warp_sum(s0[bb]);
        if (OP == OP_FC) s1[bb] = warp_sum(s1[bb]);
        if (lane == 0 && w.rs == 0) {
          sq[(warp * BG + bb) * 2] = s0[bb];
          sq[(warp * BG + bb) * 2 + 1] = s1[bb];
        }
      }
    }
    for (int u = 0; u < w.upg && w.ncols > 0; ++u) {
      const unsigned char *buf = ring_wait(ring, sz, a.status, ok);
      float acc[BG];
#pragma unroll
      for (int bb = 0; bb < BG; ++bb) acc[bb] = 0.f;
#pragma unroll
      for (int i = 0; i < NVM; ++i) {
        const int v = lane + 32 * i;
        if (v * 8 < w.ncols) {
          const uint4 wv = *reinterpret_cast<const uint4 *>(buf + v * 16);
#pragma unroll
          for (int bb = 0; bb < BG; ++bb) acc[bb] = dot8(wv, act[bb][i], acc[bb]);
        }
      }
#pragma unroll
      for (int bb = 0; bb < BG; ++bb) acc[bb] = warp_sum(acc[bb]);
      const int rl = w.rs + u * w.R;
      if (lane == 0) {
#pragma unroll
        for (int bb = 0; bb < BG; ++bb) part[((size_t)rl * w.P + w.p) * BG + bb] = acc[bb];
      }
      __syncwarp();
      ring_release(ring, sz);
      if (ok) {
        if (lane == 0) fence_proxy_async_smem();  // these reads come before the ring's next copies
        ring_issue(ring, a, warp, pol);
      }
    }
    __syncthreads();
    gemv_epilogue<OP, BG>(c, w.P, g.PC, w.row0, w.nrows, grp, fac, part, sq, ys, red, (int)blockIdx.x);
    __syncthreads();
  }
  return ok;
}

template <int NVM, int BG>
__device__ bool run_op_any(const ChainArgs &a, const ChainOp &co, Ring &ring, int warp, float *part, float *sq,
                           float *ys, float *red, uint64_t pol) {
  switch (co.op) {
    case OP_FC: return run_op<OP_FC, NVM, BG>(a, co, ring, warp, part, sq, ys, red, pol);
    case OP_QKV: return run_op<OP_QKV, NVM, BG>(a, co, ring, warp, part, sq, ys, red, pol);
    case OP_WO: return run_op<OP_WO, NVM, BG>(a, co, ring, warp, part, sq, ys, red, pol);
    case OP_GATEUP: return run_op<OP_GATEUP, NVM, BG>(a, co, ring, warp, part, sq, ys, red, pol);
    case OP_DOWN: return run_op<OP_DOWN, NVM, BG>(a, co, ring, warp, part, sq, ys, red, pol);
    default: return run_op<OP_LMHEAD, NVM, BG>(a, co, ring, warp, part, sq, ys, red, pol);
  }
}

}  // namespace

// Shared memory: [rings: 8 x ring_bytes][ring barriers: 8 x kRingSlots]
//                [part: max rows x P x BG][ys: LM-head rows x BG][red: 64][sq: 8 x BG x 2]
template <int NVM, int BG>
__global__ void __launch_bounds__(kGemvThreads, 2) chain_kernel(const __grid_constant__ ChainArgs a) {
  trace_start(kTkChain);
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Ring ring;
  ring.bytes = (uint32_t)a.ring_bytes;
  ring.buf = smem + (size_t)warp * a.ring_bytes;
  ring.bars = reinterpret_cast<uint64_t *>(smem + (size_t)kGemvWarps * a.ring_bytes) + warp * kRingSlots;
  float *part = reinterpret_cast<float *>(smem + (size_t)kGemvWarps * a.ring_bytes +
                                          (size_t)kGemvWarps * kRingSlots * 8);
  float *ys = part + a.part_floats;
  float *red = ys + a.ys_floats;
  float *sq = red + 64;
  ring.prod_off = ring.cons_off = 0u;
  ring.prod_pos = ring.cons_pos = 0u;
  ring.n_iss = ring.n_con = 0u;
  ring.io = -1;
  ring.left = 0;
  ring.pu = 0;
  ring.nops = a.nops;
  if (lane == 0) {
    for (int s = 0; s < kRingSlots; ++s) mbar_init(&ring.bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();
  const uint64_t pol = l2_policy_evict_first();
  // A later depth of a dynamic-length chain whose every sequence has stopped
  // has nothing to do (only earlier launches write the count).
  const DraftCtx &c0 = a.c[a.ops[0].ctx];
  const bool skip_all = c0.n_active && c0.j > 0 && *reinterpret_cast<volatile unsigned *>(c0.n_active) == 0u;
  if (!skip_all) ring_issue(ring, a, warp, pol);  // weights only: the first fill needs nothing of the chain
  bool ok = !skip_all;
  for (int o = 0; o < a.nops && ok; ++o) {
    ok = run_op_any<NVM, BG>(a, a.ops[o], ring, warp, part, sq, ys, red, pol);
    if (o + 1 < a.nops) {
      const bool sel = o == a.select_after;
      const DraftCtx &cs = a.c[a.ops[o].ctx];
      ok = grid_barrier(a, sel, cs) && ok;
      // every sequence stopped drafting at this selection: the rest is moot
      if (ok && sel && cs.n_active && *reinterpret_cast<volatile unsigned *>(cs.n_active) == 0u) break;
    } else if (o == a.select_after) {
      ok = grid_barrier(a, true, a.c[a.ops[o].ctx]) && ok;
    }
  }
  grid_dep_launch();  // the attention launch that follows may start its prologue
  // let the copies still in flight land before the CTA exits
  if (lane == 0)
    for (uint32_t q = ring.n_con; q < ring.n_iss; ++q)
      if (!mbar_sleep_wait(&ring.bars[q & (kRingSlots - 1)], (q / kRingSlots) & 1u, a.status)) break;
  __syncwarp();
  trace_end(kTkChain);
}

// ---------------------------------------------------------------- host side

namespace {

template <int NVM, int BG>
cudaError_t set_chain_attr(size_t smem) {
  return cudaFuncSetAttribute(chain_kernel<NVM, BG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

template <int NVM, int BG>
cudaError_t launch_chain_t(const ChainArgs &a, int grid, size_t smem, cudaStream_t s) {
  static unsigned long long attr_ctx = 0;  // the context the attribute was set in
  const unsigned long long cid = context_id();
  if (cid == 0 || cid != attr_ctx) {
    cudaError_t e = set_chain_attr<NVM, BG>(kChainSmemCap);
    if (e != cudaSuccess) return e;
    attr_ctx = cid;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kGemvThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the grid barriers need it
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  note_launch();
  return cudaLaunchKernelEx(&cfg, chain_kernel<NVM, BG>, a);
}

int nvm_for(int nv) { return nv <= 2 ? 2 : (nv <= 4 ? 4 : (nv <= 6 ? 6 : 9)); }

}  // namespace

bool chain_op_ok(const GemvPlan &g) {
  // ops with an input norm must take its scale after the dot products
  const bool norm = g.op == OP_FC || g.op == OP_QKV || g.op == OP_GATEUP || g.op == OP_LMHEAD;
  return g.nv <= 9 && (!norm || g.factor);
}

cudaError_t launch_chain(ChainArgs a, cudaStream_t s) {
  int nv = 1, grid = 1;
  for (int o = 0; o < a.nops; ++o) {
    nv = nv > a.ops[o].g.nv ? nv : a.ops[o].g.nv;
    grid = grid > a.ops[o].g.grid ? grid : a.ops[o].g.grid;
  }
  const int nvm = nvm_for(nv);
  const int B = a.c[0].B;
  const int bg = (B > 1 && nvm <= 4) ? 2 : 1;  // two batch rows' activations only when they fit in registers
  int part = 0, ys = 0;
  for (int o = 0; o < a.nops; ++o) {
    GemvPlan &g = a.ops[o].g;
    g.bg = bg;
    g.ngroups = (B + bg - 1) / bg;
    const int pf = g.rows_per_cta * g.P * bg;
    part = part > pf ? part : pf;
    if (g.op == OP_LMHEAD) ys = ys > g.rows_per_cta * bg ? ys : g.rows_per_cta * bg;
  }
  a.part_floats = (part + 3) / 4 * 4;
  a.ys_floats = (ys + 3) / 4 * 4;
  const size_t fixed = (size_t)kGemvWarps * 8 * 8 + (size_t)(a.part_floats + a.ys_floats + 64 + kGemvWarps * bg * 2) * 4;
  if (fixed + (size_t)kGemvWarps * 4608 > kChainSmemCap) return cudaErrorInvalidValue;
  a.ring_bytes = (int)(((kChainSmemCap - fixed) / kGemvWarps) / 16 * 16);
  const size_t smem = (size_t)kGemvWarps * a.ring_bytes + fixed;
  switch (nvm * 10 + bg) {
    case 21: return launch_chain_t<2, 1>(a, grid, smem, s);
    case 22: return launch_chain_t<2, 2>(a, grid, smem, s);
    case 41: return launch_chain_t<4, 1>(a, grid, smem, s);
    case 42: return launch_chain_t<4, 2>(a, grid, smem, s);
    case 61: return launch_chain_t<6, 1>(a, grid, smem, s);
    default: return launch_chain_t<9, 1>(a, grid, smem, s);
  }
}

MTP_TRACE_COLLECTOR(chain)

}  // namespace mtp
