// C-ABI entry points of libmtpspec: argument validation, workspace layout and
// the launch sequence of the draft chain and the verifier on one stream.
#include <math.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <nvtx3/nvToolsExt.h>

#include "internal.h"
#include "mtpspec.h"

namespace mtp {

static std::atomic<long long> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// The unique id of the calling thread's current CUDA context (0 when there is
// none, or the driver cannot say).  Per-device state that belongs to a context
// -- a device address inside this module, the kernels' attributes -- is keyed
// on it, so that a context created anew after cudaDeviceReset is set up again
// instead of being handed addresses of the old one.
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

unsigned long long context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

namespace {

constexpr size_t kAlign = 256;

size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct DevInfo {
  bool init = false;
  unsigned long long ctx = 0;  // context the attributes were set in
  int sms = 0;
  int max_cluster = 8;
};
std::mutex g_mu;
DevInfo g_dev[64];

int device_info(DevInfo *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MTP_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo &di = g_dev[dev];
  const unsigned long long cid = context_id();
  if (!di.init || cid == 0 || cid != di.ctx) {
    if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MTP_ERR_CUDA;
    di.max_cluster = 16;  // the non-portable size; the automatic choice stays at 8 or less
    if (verify_set_attributes() != cudaSuccess) return MTP_ERR_CUDA;
    if (tc_set_attributes() != cudaSuccess) return MTP_ERR_CUDA;
    if (fused_set_attributes() != cudaSuccess) return MTP_ERR_CUDA;
    di.ctx = context_id();  // set up (made current) by the calls above
    di.init = true;
  }
  *out = di;
  return MTP_OK;
}

bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dims(const MtpDims *d, int k) {
  if (!d) return MTP_ERR_INVALID_ARG;
  if (k < 1 || k > 8) return MTP_ERR_INVALID_ARG;
  if (d->B < 1 || d->d < 8 || d->Hq < 1 || d->Hkv < 1 || d->F < 8 || d->V < 1) return MTP_ERR_INVALID_ARG;
  if (!(d->rms_eps >= 0.f)) return MTP_ERR_INVALID_ARG;
  if (d->Lmax < k + 1) return MTP_ERR_INVALID_ARG;
  if (d->d % 8 || d->F % 8) return MTP_ERR_UNSUPPORTED_SHAPE;
  if (d->Hq % d->Hkv || d->Hq / d->Hkv > kMaxGroup) return MTP_ERR_UNSUPPORTED_SHAPE;
  if (d->Dh != 32 && d->Dh != 64 && d->Dh != 128) return MTP_ERR_UNSUPPORTED_SHAPE;
  if ((long long)d->B * d->V * 8 >= (1ll << 62)) return MTP_ERR_UNSUPPORTED_SHAPE;
  if (d->V > (1 << 30) || d->B > (1 << 20)) return MTP_ERR_UNSUPPORTED_SHAPE;
  return MTP_OK;
}

struct WsLayout {
  size_t status, lm_cnt, x0, x1, x2, q, o, act, lm_part, logits, vstate, tc_a[3], tc_part, order, total;
  bool tc;
  TcSizes tz;
};

MtpShape shape_of(const MtpDims &d) { return MtpShape{d.B, d.d, d.Hq, d.Hkv, d.Dh, d.F, d.V}; }

// draft_only: the layout of a draft-only call that keeps no logits in its
// workspace and runs no verification (mtp_draft_noalloc's scratch): the logits
// and verifier-state regions are left out.
WsLayout draft_layout(const MtpDims &d, int k, bool draft_only = false) {
  WsLayout L{};
  size_t off = 0;
  L.status = off;
  off += kAlign;
  L.lm_cnt = off;
  off += kAlign;
  L.x0 = off;
  off += up((size_t)d.B * d.d * 4);
  L.x1 = off;
  off += up((size_t)d.B * d.d * 4);
  L.x2 = off;
  off += up((size_t)d.B * d.d * 4);
  L.q = off;
  off += up((size_t)d.B * d.Hq * d.Dh * 4);
  L.o = off;
  off += up((size_t)d.B * d.Hq * d.Dh * 4);
  L.act = off;
  off += up((size_t)d.B * d.F * 4);
  L.lm_part = off;
  off += up((size_t)d.B * kMaxLmGrid * 4 * 4);
  L.logits = off;
  if (!draft_only) off += up((size_t)d.B * k * d.V * 4);
  L.vstate = off;
  if (!draft_only) off += up(verify_state_bytes(d.B, k, d.V));
  L.tc = tc_shape_ok(shape_of(d));
  if (L.tc) {
    L.tz = tc_sizes(shape_of(d));
    for (int t = 0; t < 3; ++t) {
      L.tc_a[t] = off;
      off += up((size_t)L.tz.rows * L.tz.kmax * 2);
    }
    L.tc_part = off;
    off += up(L.tz.part_floats * 4);
    L.order = off;
    off += up((size_t)d.B * 4);
  }
  L.total = off;
  return L;
}

// profiler state
struct Prof {
  bool on = false;
  std::vector<cudaEvent_t> ev[MTP_KC_COUNT];  // start/stop pairs
  size_t used[MTP_KC_COUNT] = {0, 0, 0, 0};
};
Prof g_prof;
std::mutex g_prof_mu;

template <class F>
cudaError_t timed(int kc, cudaStream_t s, F &&launch) {
  if (!g_prof.on) return launch();
  std::lock_guard<std::mutex> lk(g_prof_mu);
  auto &v = g_prof.ev[kc];
  size_t i = g_prof.used[kc];
  if (2 * i + 2 > v.size()) {
    for (int t = 0; t < 256; ++t) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return cudaErrorMemoryAllocation;
      v.push_back(e);
    }
  }
  cudaEventRecord(v[2 * i], s);
  cudaError_t e = launch();
  cudaEventRecord(v[2 * i + 1], s);
  g_prof.used[kc] = i + 1;
  return e;
}

constexpr int kMaxModules = 8;  // one per depth at most

struct Draft {
  DraftCtx c;
  GemvPlan fc, qkv, wo, gateup, down, lm;
  int attn_cluster;
  bool tc;   // tensor-core path
  TcBufs t;
  MtpModule mods[kMaxModules];
  int nmod;
};

// Point the context at module m's weights and K/V cache.
void use_module(DraftCtx &c, const MtpModule &m) {
  auto bf = [](const void *p) { return static_cast<const uint16_t *>(p); };
  const MtpWeights *w = &m.w;
  c.E = bf(w->E); c.fc = bf(w->fc); c.wq = bf(w->wq); c.wk = bf(w->wk); c.wv = bf(w->wv); c.wo = bf(w->wo);
  c.wgate = bf(w->wgate); c.wup = bf(w->wup); c.wdown = bf(w->wdown);
  c.g_emb = bf(w->g_emb); c.g_hid = bf(w->g_hid); c.g_attn = bf(w->g_attn); c.g_mlp = bf(w->g_mlp);
  c.g_final = bf(w->g_final);
  c.kc = static_cast<uint16_t *>(m.k_cache); c.vc = static_cast<uint16_t *>(m.v_cache);
  if (!c.vmap) c.head = c.E;  // a reduced head stays as set
}

// Options beyond the plain chain: the dynamic draft length (k_eff non-null)
// and a reduced draft vocabulary (vmap non-null).
struct DraftOpts {
  float stop_p = 0.f;
  int32_t *k_eff = nullptr;
  const void *head = nullptr;     // [Vd, d] bf16
  const int32_t *vmap = nullptr;  // [Vd]
  int Vd = 0;
};

int prepare_draft(const MtpDims *dims, const MtpModule *mods, int nmod, const void *h, const int32_t *last_tok,
                  const int32_t *ctx_len, int k, float T, int mode, const float *u_draft, int32_t *draft_tok,
                  float *draft_logits, void *ws, size_t ws_bytes, bool logits_in_ws, const DraftOpts &o,
                  Draft *out, bool draft_only = false) {
  int rc = check_dims(dims, k);
  if (rc) return rc;
  if (o.k_eff && (!aligned16(o.k_eff) || !(o.stop_p >= 0.f && o.stop_p < 1e30f))) return MTP_ERR_INVALID_ARG;
  if (o.vmap && (!aligned16(o.vmap) || !aligned16(o.head) || o.Vd < 128 || o.Vd > dims->V))
    return MTP_ERR_INVALID_ARG;
  if (!mods || nmod < 1 || nmod > k) return MTP_ERR_INVALID_ARG;
  if (mode != MTP_GREEDY && mode != MTP_STOCHASTIC) return MTP_ERR_INVALID_ARG;
  if (mode == MTP_STOCHASTIC && !(T > 0.f && T < 1e30f)) return MTP_ERR_INVALID_ARG;
  for (int m = 0; m < nmod; ++m) {
    const MtpWeights *w = &mods[m].w;
    const void *wp[] = {w->E, w->fc, w->wq, w->wk, w->wv, w->wo, w->wgate, w->wup, w->wdown, w->g_emb,
                        w->g_hid, w->g_attn, w->g_mlp, w->g_final, mods[m].k_cache, mods[m].v_cache};
    for (const void *p : wp)
      if (!aligned16(p)) return MTP_ERR_INVALID_ARG;
  }
  const void *ptrs[] = {h, last_tok, ctx_len, draft_tok, ws};
  for (const void *p : ptrs)
    if (!aligned16(p)) return MTP_ERR_INVALID_ARG;
  if (mode == MTP_STOCHASTIC && !aligned16(u_draft)) return MTP_ERR_INVALID_ARG;
  if (mode == MTP_STOCHASTIC && !logits_in_ws && !aligned16(draft_logits)) return MTP_ERR_INVALID_ARG;
  if (draft_logits && !aligned16(draft_logits)) return MTP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MTP_ERR_INVALID_ARG;
  if (draft_only && logits_in_ws) return MTP_ERR_INVALID_ARG;
  const WsLayout L = draft_layout(*dims, k, draft_only);
  if (ws_bytes < L.total) return MTP_ERR_WORKSPACE;
  DevInfo di;
  if ((rc = device_info(&di))) return rc;

  const MtpDims &d = *dims;
  DraftCtx &c = out->c;
  c = DraftCtx{};
  c.B = d.B; c.d = d.d; c.Hq = d.Hq; c.Hkv = d.Hkv; c.Dh = d.Dh; c.F = d.F; c.V = d.V; c.Lmax = d.Lmax;
  c.k = k; c.j = 0; c.jc = 0; c.mode = mode; c.eps = d.rms_eps; c.T = mode == MTP_STOCHASTIC ? T : 1.f;
  c.vmap = o.vmap;
  c.head = static_cast<const uint16_t *>(o.head);
  use_module(c, mods[0]);
  for (int m = 0; m < nmod; ++m) out->mods[m] = mods[m];
  out->nmod = nmod;
  c.h = static_cast<const uint16_t *>(h); c.last_tok = last_tok; c.ctx_len = ctx_len; c.u_draft = u_draft;
  c.draft_tok = draft_tok;
  c.k_eff = o.k_eff;
  c.stop_p = o.stop_p;
  c.Vd = o.vmap ? o.Vd : d.V;
  char *base = static_cast<char *>(ws);
  c.logits = draft_logits ? draft_logits : (logits_in_ws ? reinterpret_cast<float *>(base + L.logits) : nullptr);
  c.status = reinterpret_cast<int *>(base + L.status);
  c.lm_cnt = reinterpret_cast<unsigned *>(base + L.lm_cnt);
  c.n_active = o.k_eff ? c.lm_cnt + 1 : nullptr;  // same 256-byte slot as the ticket counter
  c.x0 = reinterpret_cast<float *>(base + L.x0);
  c.x1 = reinterpret_cast<float *>(base + L.x1);
  c.x2 = reinterpret_cast<float *>(base + L.x2);
  c.q = reinterpret_cast<float *>(base + L.q);
  c.o = reinterpret_cast<float *>(base + L.o);
  c.act = reinterpret_cast<float *>(base + L.act);
  c.lm_part = reinterpret_cast<float *>(base + L.lm_part);
  out->attn_cluster =
      attention_cluster_size(d.Lmax, d.B * d.Hkv, di.sms, di.max_cluster, attention_tc_shape_ok(c));

  out->fc = plan_gemv(OP_FC, d.d, 2 * d.d, d.B, di.sms);
  out->qkv = plan_gemv(OP_QKV, (d.Hq + 2 * d.Hkv) * d.Dh, d.d, d.B, di.sms);
  out->wo = plan_gemv(OP_WO, d.d, d.Hq * d.Dh, d.B, di.sms);
  out->gateup = plan_gemv(OP_GATEUP, 2 * d.F, d.d, d.B, di.sms);
  out->down = plan_gemv(OP_DOWN, d.d, d.F, d.B, di.sms);
  out->lm = plan_gemv(OP_LMHEAD, c.Vd, d.d, d.B, di.sms);
  if (out->lm.grid > kMaxLmGrid) return MTP_ERR_UNSUPPORTED_SHAPE;
  c.lm_grid = out->lm.grid;
  c.lm_rpc = out->lm.rows_per_cta;
  out->tc = L.tc && tc_available();
  if (out->tc) {
    for (int t = 0; t < 3; ++t) out->t.a[t] = reinterpret_cast<uint16_t *>(base + L.tc_a[t]);
    out->t.rows = L.tz.rows;
    out->t.kmax = L.tz.kmax;
    out->t.part = reinterpret_cast<float *>(base + L.tc_part);
    c.seq_order = reinterpret_cast<int *>(base + L.order);
    out->t.part_floats = L.tz.part_floats;
  }
  return MTP_OK;
}

// Programmatic dependent launch between the chained kernels (MTP_PDL=0 turns it
// off, for measurement).
bool use_pdl() {
  const char *v = getenv("MTP_PDL");
  return !(v && v[0] == '0');
}

// Stochastic verification by the streaming kernel of verify_split.cu (the
// default; MTP_VERIFY_SPLIT=0 takes the cluster kernel of verify.cu, which
// greedy verification always takes).
bool use_verify_split() {
  const char *v = getenv("MTP_VERIFY_SPLIT");
  return !(v && v[0] == '0');
}

// The GEMV path's ops in cooperative chain launches, when MTP_CHAIN=1:
// [input projection, QKV] of depth 0, then per depth its attention and [output
// projection, gate/up, down, LM head + draft selection] followed by the next
// depth's [input projection, QKV].  Off by default: at the single-sequence
// workload one launch per op, chained by programmatic dependent launch,
// measured faster (1077 against 911 steps/s).
bool use_chain(const Draft &D) {
  const char *v = getenv("MTP_CHAIN");
  if (!(v && v[0] == '1') || D.tc) return false;
  const GemvPlan *ps[] = {&D.fc, &D.qkv, &D.wo, &D.gateup, &D.down, &D.lm};
  for (const GemvPlan *p : ps)
    if (!chain_op_ok(*p)) return false;
  return true;
}

DraftCtx depth_ctx(const Draft &D, int j) {
  DraftCtx c = D.c;
  const int m = j < D.nmod ? j : D.nmod - 1;  // depth j runs module min(j, nmod - 1)
  use_module(c, D.mods[m]);
  c.j = j;
  c.jc = j - m;
  c.zero_counters = j == 0;
  return c;
}

cudaError_t run_draft_chain(Draft &D, cudaStream_t s, bool pdl) {
  cudaError_t e = cudaSuccess;
  if (D.c.vmap && D.c.logits) {  // a reduced head writes only its ids: the rest of each row is -inf
    e = launch_fill(D.c.logits, (size_t)D.c.B * D.c.k * D.c.V, -INFINITY, s, pdl);
    if (e) return e;
  }
  ChainArgs a{};
  a.bar = D.c.lm_cnt + 8;  // two words of the counters' slot
  a.status = D.c.status;
  a.c[0] = depth_ctx(D, 0);
  a.c[1] = a.c[0];
  a.ops[0] = ChainOp{OP_FC, 0, D.fc};
  a.ops[1] = ChainOp{OP_QKV, 0, D.qkv};
  a.nops = 2;
  a.select_after = -1;
  if ((e = timed(MTP_KC_GEMV, s, [&] { return launch_chain(a, s); }))) return e;
  for (int j = 0; j < D.c.k; ++j) {
    const DraftCtx cj = depth_ctx(D, j);
    if ((e = timed(MTP_KC_ATTN, s, [&] { return launch_attention(cj, D.attn_cluster, s, pdl); }))) return e;
    a.c[0] = cj;
    a.ops[0] = ChainOp{OP_WO, 0, D.wo};
    a.ops[1] = ChainOp{OP_GATEUP, 0, D.gateup};
    a.ops[2] = ChainOp{OP_DOWN, 0, D.down};
    a.ops[3] = ChainOp{OP_LMHEAD, 0, D.lm};
    a.nops = 4;
    a.select_after = 3;
    if (j + 1 < D.c.k) {
      a.c[1] = depth_ctx(D, j + 1);
      a.ops[4] = ChainOp{OP_FC, 1, D.fc};
      a.ops[5] = ChainOp{OP_QKV, 1, D.qkv};
      a.nops = 6;
    }
    if ((e = timed(MTP_KC_LMHEAD, s, [&] { return launch_chain(a, s); }))) return e;
  }
  return e;
}

// NVTX ranges around each call and each depth's launches (MTP_NVTX=1; the
// header-only NVTX API costs nothing unless a profiling tool is attached).
bool use_nvtx() {
  static const bool on = [] {
    const char *v = getenv("MTP_NVTX");
    return v && v[0] == '1';
  }();
  return on;
}

struct NvtxRange {
  bool on;
  explicit NvtxRange(const char *name) : on(use_nvtx()) {
    if (on) nvtxRangePushA(name);
  }
  ~NvtxRange() {
    if (on) nvtxRangePop();
  }
};

const char *depth_name(int j) {
  static const char *names[8] = {"mtp depth 0", "mtp depth 1", "mtp depth 2", "mtp depth 3",
                                 "mtp depth 4", "mtp depth 5", "mtp depth 6", "mtp depth 7"};
  return names[j & 7];
}

cudaError_t run_draft(Draft &D, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  const bool pdl = use_pdl();
  NvtxRange call_range("mtp_draft chain");
  if (use_chain(D)) return run_draft_chain(D, s, pdl);
  if (D.c.vmap && D.c.logits) {  // a reduced head writes only its ids: the rest of each row is -inf
    e = launch_fill(D.c.logits, (size_t)D.c.B * D.c.k * D.c.V, -INFINITY, s, pdl);
    if (e) return e;
  }
  for (int j = 0; j < D.c.k && e == cudaSuccess; ++j) {
    NvtxRange depth_range(depth_name(j));
    DraftCtx c = D.c;
    // depth j runs module min(j, nmod - 1), at the next row of that module's cache
    const int m = j < D.nmod ? j : D.nmod - 1;
    use_module(c, D.mods[m]);
    c.j = j;
    c.jc = j - m;
    c.zero_counters = j == 0;
    if (D.tc) {  // tensor-core path
      if ((e = timed(MTP_KC_GEMV, s, [&] { return run_block_pre_tc(c, D.t, s, pdl); }))) break;
      if ((e = timed(MTP_KC_ATTN, s, [&] { return launch_attention(c, D.attn_cluster, s, pdl); }))) break;
      if ((e = timed(MTP_KC_GEMV, s, [&] { return run_block_post_tc(c, D.t, s, pdl); }))) break;
      if ((e = timed(MTP_KC_LMHEAD, s, [&] { return run_lmhead_tc(c, D.t, s, pdl); }))) break;
      continue;
    }
    if ((e = timed(MTP_KC_GEMV, s, [&] { return launch_gemv(c, D.fc, s, pdl); }))) break;
    if ((e = timed(MTP_KC_GEMV, s, [&] { return launch_gemv(c, D.qkv, s, pdl); }))) break;
    if ((e = timed(MTP_KC_ATTN, s, [&] { return launch_attention(c, D.attn_cluster, s, pdl); }))) break;
    if ((e = timed(MTP_KC_GEMV, s, [&] { return launch_gemv(c, D.wo, s, pdl); }))) break;
    if ((e = timed(MTP_KC_GEMV, s, [&] { return launch_gemv(c, D.gateup, s, pdl); }))) break;
    if ((e = timed(MTP_KC_GEMV, s, [&] { return launch_gemv(c, D.down, s, pdl); }))) break;
    if ((e = timed(MTP_KC_LMHEAD, s, [&] { return launch_gemv(c, D.lm, s, pdl); }))) break;
  }
  return e;
}

int prepare_verify(int B, int k, int V, float T, int mode, const float *target, const float *draft,
                   const int32_t *draft_tok, const float *u_accept, const float *u_final, int32_t *out_tok,
                   int32_t *accept_len, int32_t *num_accepted, void *state, size_t state_bytes, bool draft_check,
                   const int32_t *k_eff, VerifyArgs *a) {
  if (k_eff && !aligned16(k_eff)) return MTP_ERR_INVALID_ARG;
  if (B < 1 || k < 1 || k > 8 || V < 1 || V > (1 << 30) || B > (1 << 20)) return MTP_ERR_INVALID_ARG;
  if (mode != MTP_GREEDY && mode != MTP_STOCHASTIC) return MTP_ERR_INVALID_ARG;
  if (mode == MTP_STOCHASTIC && !(T > 0.f && T < 1e30f)) return MTP_ERR_INVALID_ARG;
  const void *ptrs[] = {target, draft_tok, out_tok, accept_len, num_accepted, state};
  for (const void *p : ptrs)
    if (!aligned16(p)) return MTP_ERR_INVALID_ARG;
  if (mode == MTP_STOCHASTIC) {
    if (draft_check && !aligned16(draft)) return MTP_ERR_INVALID_ARG;
    if (!aligned16(u_accept) || !aligned16(u_final)) return MTP_ERR_INVALID_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(state) & (kAlign - 1)) != 0) return MTP_ERR_INVALID_ARG;
  if (state_bytes < verify_state_bytes(B, k, V)) return MTP_ERR_WORKSPACE;
  DevInfo di;
  int rc = device_info(&di);
  if (rc) return rc;
  a->B = B; a->k = k; a->V = V; a->mode = mode; a->T = mode == MTP_STOCHASTIC ? T : 1.f;
  a->target = target; a->draft = draft; a->draft_tok = draft_tok; a->u_accept = u_accept; a->u_final = u_final;
  a->out_tok = out_tok; a->accept_len = accept_len; a->num_accepted = num_accepted;
  a->k_eff = k_eff;
  if (!plan_verify(B, k, V, &a->p)) return MTP_ERR_UNSUPPORTED_SHAPE;
  verify_bind_state(*a, state);
  a->split = mode == MTP_STOCHASTIC && use_verify_split() && split_shape_ok(B, k, V);
  return MTP_OK;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MTP_OK : MTP_ERR_CUDA; }

// Scratch of mtp_draft_noalloc: one array per device, part of this module's
// device image, so no call allocates.  Static device memory starts zeroed.
__device__ __align__(256) unsigned char g_static_scratch[MTP_STATIC_SCRATCH_BYTES];

struct ScratchSlot {
  bool init = false;
  unsigned long long ctx = 0;  // context the address belongs to
  void *ptr = nullptr;
};
ScratchSlot g_scratch_slot[64];

// The device address of g_static_scratch on the current device, looked up
// once per device and context (with that device current): after
// cudaDeviceReset the next call runs in a new context, where the module may
// sit at another address, so the lookup is made again.
int static_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MTP_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  ScratchSlot &sl = g_scratch_slot[dev];
  const unsigned long long cid = context_id();
  if (!sl.init || cid == 0 || cid != sl.ctx) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      sl.init = false;
      return MTP_ERR_CUDA;
    }
    sl.ptr = p;
    sl.ctx = context_id();  // made current by the lookup if there was none
    sl.init = true;
  }
  *out = sl.ptr;
  return MTP_OK;
}

}  // namespace
static_assert(kTkGemv == MTP_TK_GEMV && kTkAttn == MTP_TK_ATTN && kTkAttnTc == MTP_TK_ATTN_TC &&
                  kTkVerify == MTP_TK_VERIFY && kTkVerifySplit == MTP_TK_VERIFY_SPLIT && kTkTcGemm == MTP_TK_TC_GEMM &&
                  kTkTcAux == MTP_TK_TC_AUX && kTkFusedGemm == MTP_TK_FUSED_GEMM &&
                  kTkFusedAux == MTP_TK_FUSED_AUX && kTkChain == MTP_TK_CHAIN,
              "trace kinds match the header");

// the launch-trace collectors of the kernel files (MTP_TRACE_COLLECTOR)
int trace_collect_draft(TraceRec *, int);
int trace_collect_attn_tc(TraceRec *, int);
int trace_collect_verify(TraceRec *, int);
int trace_collect_verify_split(TraceRec *, int);
int trace_collect_tc(TraceRec *, int);
int trace_collect_fused(TraceRec *, int);
int trace_collect_chain(TraceRec *, int);
int trace_collect_diag(TraceRec *, int);

}  // namespace mtp

using namespace mtp;

extern "C" {

size_t mtp_workspace_size(const MtpDims *dims, int k) {
  if (check_dims(dims, k) != MTP_OK) return 0;
  return draft_layout(*dims, k).total;
}

int mtp_draft_modules(const MtpDims *dims, const MtpModule *modules, int n_modules, const void *h,
                      const int32_t *last_tok, const int32_t *ctx_len, int k, float T, int mode,
                      const float *u_draft, int32_t *draft_tok, float *draft_logits, void *ws, size_t ws_bytes,
                      mtp_stream_t stream) {
  Draft D;
  int rc = prepare_draft(dims, modules, n_modules, h, last_tok, ctx_len, k, T, mode, u_draft, draft_tok,
                         draft_logits, ws, ws_bytes, false, DraftOpts{}, &D);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = run_draft(D, s);
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_rc(e);
}

int mtp_draft(const MtpDims *dims, const MtpWeights *w, const void *h, const int32_t *last_tok, void *k_cache,
              void *v_cache, const int32_t *ctx_len, int k, float T, int mode, const float *u_draft,
              int32_t *draft_tok, float *draft_logits, void *ws, size_t ws_bytes, mtp_stream_t stream) {
  if (!w) return MTP_ERR_INVALID_ARG;
  const MtpModule one{*w, k_cache, v_cache};
  return mtp_draft_modules(dims, &one, 1, h, last_tok, ctx_len, k, T, mode, u_draft, draft_tok, draft_logits, ws,
                           ws_bytes, stream);
}

int mtp_draft_reduced(const MtpDims *dims, const MtpWeights *w, const void *head_rows, const int32_t *vocab_map,
                      int n_draft_vocab, const void *h, const int32_t *last_tok, void *k_cache, void *v_cache,
                      const int32_t *ctx_len, int k, float T, int mode, const float *u_draft, int32_t *draft_tok,
                      float *draft_logits, void *ws, size_t ws_bytes, mtp_stream_t stream) {
  if (!w || !vocab_map) return MTP_ERR_INVALID_ARG;
  const MtpModule one{*w, k_cache, v_cache};
  DraftOpts o;
  o.head = head_rows;
  o.vmap = vocab_map;
  o.Vd = n_draft_vocab;
  Draft D;
  int rc = prepare_draft(dims, &one, 1, h, last_tok, ctx_len, k, T, mode, u_draft, draft_tok, draft_logits, ws,
                         ws_bytes, false, o, &D);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = run_draft(D, s);
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_rc(e);
}

int mtp_draft_dynamic(const MtpDims *dims, const MtpWeights *w, const void *h, const int32_t *last_tok,
                      void *k_cache, void *v_cache, const int32_t *ctx_len, int k, float T, int mode, float stop_p,
                      const float *u_draft, int32_t *draft_tok, float *draft_logits, int32_t *k_eff, void *ws,
                      size_t ws_bytes, mtp_stream_t stream) {
  if (!w || !k_eff) return MTP_ERR_INVALID_ARG;
  const MtpModule one{*w, k_cache, v_cache};
  Draft D;
  DraftOpts o;
  o.stop_p = stop_p;
  o.k_eff = k_eff;
  int rc = prepare_draft(dims, &one, 1, h, last_tok, ctx_len, k, T, mode, u_draft, draft_tok, draft_logits, ws,
                         ws_bytes, false, o, &D);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = run_draft(D, s);
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_rc(e);
}

int mtp_draft_noalloc(const MtpDims *dims, const MtpWeights *w, const void *h, const int32_t *last_tok,
                      void *k_cache, void *v_cache, const int32_t *ctx_len, int k, float T, int mode,
                      const float *u_draft, int32_t *draft_tok, float *draft_logits, int32_t *status,
                      mtp_stream_t stream) {
  int rc = check_dims(dims, k);
  if (rc) return rc;
  if (draft_layout(*dims, k, true).total > MTP_STATIC_SCRATCH_BYTES) return MTP_ERR_SCRATCH_LIMIT;
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u) != 0) return MTP_ERR_INVALID_ARG;
  if (!w) return MTP_ERR_INVALID_ARG;
  void *scratch = nullptr;
  if ((rc = static_scratch(&scratch))) return rc;
  const MtpModule one{*w, k_cache, v_cache};
  Draft D;
  rc = prepare_draft(dims, &one, 1, h, last_tok, ctx_len, k, T, mode, u_draft, draft_tok, draft_logits, scratch,
                     MTP_STATIC_SCRATCH_BYTES, false, DraftOpts{}, &D, true);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the status word and the LM-head ticket counter (the first two aligned
  // slots) must start at zero
  cudaError_t e = cudaMemsetAsync(scratch, 0, 2 * kAlign, s);
  if (e == cudaSuccess) e = run_draft(D, s);
  if (e == cudaSuccess && status)
    e = cudaMemcpyAsync(status, D.c.status, sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_rc(e);
}

size_t spec_verify_workspace_size(int B, int k, int V) {
  if (B < 1 || k < 1 || k > 8 || V < 1) return 0;
  return kAlign + up(verify_state_bytes(B, k, V));
}

int spec_verify_dynamic(int B, int k, int V, float T, int mode, const float *target_logits,
                        const float *draft_logits, const int32_t *draft_tok, const int32_t *k_eff,
                        const float *u_accept, const float *u_final, int32_t *out_tok, int32_t *accept_len,
                        int32_t *num_accepted, void *ws, size_t ws_bytes, mtp_stream_t stream) {
  VerifyArgs a{};
  if (!aligned16(ws) || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MTP_ERR_INVALID_ARG;
  if (ws_bytes < kAlign) return MTP_ERR_WORKSPACE;
  int rc = prepare_verify(B, k, V, T, mode, target_logits, draft_logits, draft_tok, u_accept, u_final, out_tok,
                          accept_len, num_accepted, static_cast<char *>(ws) + kAlign, ws_bytes - kAlign, true, k_eff,
                          &a);
  if (rc) return rc;
  a.status = static_cast<int *>(ws);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  NvtxRange r("spec verify");
  cudaError_t e = timed(MTP_KC_VERIFY, s, [&] { return launch_verify(a, s, false); });
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_rc(e);
}

int spec_verify(int B, int k, int V, float T, int mode, const float *target_logits, const float *draft_logits,
                const int32_t *draft_tok, const float *u_accept, const float *u_final, int32_t *out_tok,
                int32_t *accept_len, int32_t *num_accepted, void *ws, size_t ws_bytes, mtp_stream_t stream) {
  return spec_verify_dynamic(B, k, V, T, mode, target_logits, draft_logits, draft_tok, nullptr, u_accept, u_final,
                             out_tok, accept_len, num_accepted, ws, ws_bytes, stream);
}

// spec_step over modules, with the dynamic draft length when k_eff is given.
static int step_call(const MtpDims *dims, const MtpModule *modules, int n_modules, const void *h,
                     const int32_t *last_tok, const int32_t *ctx_len, int k, float T, int mode, const DraftOpts &o,
                     const float *u_draft, const float *target_logits, const float *u_accept, const float *u_final,
                     int32_t *draft_tok, float *draft_logits, int32_t *out_tok, int32_t *accept_len,
                     int32_t *num_accepted, void *ws, size_t ws_bytes, mtp_stream_t stream) {
  Draft D;
  int rc = prepare_draft(dims, modules, n_modules, h, last_tok, ctx_len, k, T, mode, u_draft, draft_tok,
                         draft_logits, ws, ws_bytes, mode == MTP_STOCHASTIC, o, &D);
  if (rc) return rc;
  VerifyArgs a{};
  const WsLayout L = draft_layout(*dims, k);
  rc = prepare_verify(dims->B, k, dims->V, T, mode, target_logits, D.c.logits, draft_tok, u_accept, u_final, out_tok,
                      accept_len, num_accepted, static_cast<char *>(ws) + L.vstate, L.total - L.vstate, false, o.k_eff,
                      &a);
  if (rc) return rc;
  a.status = D.c.status;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = run_draft(D, s);
  if (e == cudaSuccess) {
    NvtxRange r("spec verify");
    e = timed(MTP_KC_VERIFY, s, [&] { return launch_verify(a, s, use_pdl()); });
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_rc(e);
}

int spec_step_modules(const MtpDims *dims, const MtpModule *modules, int n_modules, const void *h,
                      const int32_t *last_tok, const int32_t *ctx_len, int k, float T, int mode,
                      const float *u_draft, const float *target_logits, const float *u_accept,
                      const float *u_final, int32_t *draft_tok, float *draft_logits, int32_t *out_tok,
                      int32_t *accept_len, int32_t *num_accepted, void *ws, size_t ws_bytes, mtp_stream_t stream) {
  return step_call(dims, modules, n_modules, h, last_tok, ctx_len, k, T, mode, DraftOpts{}, u_draft, target_logits,
                   u_accept, u_final, draft_tok, draft_logits, out_tok, accept_len, num_accepted, ws, ws_bytes,
                   stream);
}

int spec_step_reduced(const MtpDims *dims, const MtpWeights *w, const void *head_rows, const int32_t *vocab_map,
                      int n_draft_vocab, const void *h, const int32_t *last_tok, void *k_cache, void *v_cache,
                      const int32_t *ctx_len, int k, float T, int mode, const float *u_draft,
                      const float *target_logits, const float *u_accept, const float *u_final, int32_t *draft_tok,
                      float *draft_logits, int32_t *out_tok, int32_t *accept_len, int32_t *num_accepted, void *ws,
                      size_t ws_bytes, mtp_stream_t stream) {
  if (!w || !vocab_map) return MTP_ERR_INVALID_ARG;
  const MtpModule one{*w, k_cache, v_cache};
  DraftOpts o;
  o.head = head_rows;
  o.vmap = vocab_map;
  o.Vd = n_draft_vocab;
  return step_call(dims, &one, 1, h, last_tok, ctx_len, k, T, mode, o, u_draft, target_logits, u_accept, u_final,
                   draft_tok, draft_logits, out_tok, accept_len, num_accepted, ws, ws_bytes, stream);
}

int spec_step_dynamic(const MtpDims *dims, const MtpWeights *w, const void *h, const int32_t *last_tok,
                      void *k_cache, void *v_cache, const int32_t *ctx_len, int k, float T, int mode, float stop_p,
                      const float *u_draft, const float *target_logits, const float *u_accept,
                      const float *u_final, int32_t *draft_tok, float *draft_logits, int32_t *k_eff,
                      int32_t *out_tok, int32_t *accept_len, int32_t *num_accepted, void *ws, size_t ws_bytes,
                      mtp_stream_t stream) {
  if (!w || !k_eff) return MTP_ERR_INVALID_ARG;
  const MtpModule one{*w, k_cache, v_cache};
  DraftOpts o;
  o.stop_p = stop_p;
  o.k_eff = k_eff;
  return step_call(dims, &one, 1, h, last_tok, ctx_len, k, T, mode, o, u_draft, target_logits, u_accept, u_final,
                   draft_tok, draft_logits, out_tok, accept_len, num_accepted, ws, ws_bytes, stream);
}

int spec_step(const MtpDims *dims, const MtpWeights *w, const void *h, const int32_t *last_tok, void *k_cache,
              void *v_cache, const int32_t *ctx_len, int k, float T, int mode, const float *u_draft,
              const float *target_logits, const float *u_accept, const float *u_final, int32_t *draft_tok,
              float *draft_logits, int32_t *out_tok, int32_t *accept_len, int32_t *num_accepted, void *ws,
              size_t ws_bytes, mtp_stream_t stream) {
  if (!w) return MTP_ERR_INVALID_ARG;
  const MtpModule one{*w, k_cache, v_cache};
  return spec_step_modules(dims, &one, 1, h, last_tok, ctx_len, k, T, mode, u_draft, target_logits, u_accept,
                           u_final, draft_tok, draft_logits, out_tok, accept_len, num_accepted, ws, ws_bytes, stream);
}

size_t spec_verify_fused_workspace_size(int B, int k, int V, int d, int mode) {
  if (!fused_shape_ok(B, k, V, d) || (mode != MTP_GREEDY && mode != MTP_STOCHASTIC)) return 0;
  if (mode == MTP_STOCHASTIC && (long long)B * k * ((V + 255) / 256) >= (1ll << 31)) return 0;
  return fused_workspace_bytes(B, k, V, d, mode);
}

int spec_verify_fused(int B, int k, int V, int d, float T, int mode, const void *head, const void *target_hidden,
                      const float *draft_logits, const int32_t *draft_tok, const float *u_accept,
                      const float *u_final, int32_t *out_tok, int32_t *accept_len, int32_t *num_accepted, void *ws,
                      size_t ws_bytes, mtp_stream_t stream) {
  if (!fused_shape_ok(B, k, V, d)) return MTP_ERR_INVALID_ARG;
  if (mode != MTP_GREEDY && mode != MTP_STOCHASTIC) return MTP_ERR_INVALID_ARG;
  if (mode == MTP_STOCHASTIC && !(T > 0.f && T < 1e30f)) return MTP_ERR_INVALID_ARG;
  // the draft statistics' warps claim (row, 256-token tile) items from a
  // 32-bit counter: past 2^31 items it could wrap before the last claim
  if (mode == MTP_STOCHASTIC && (long long)B * k * ((V + 255) / 256) >= (1ll << 31)) return MTP_ERR_UNSUPPORTED_SHAPE;
  const void *ptrs[] = {head, target_hidden, draft_tok, out_tok, accept_len, num_accepted, ws};
  for (const void *p : ptrs)
    if (!aligned16(p)) return MTP_ERR_INVALID_ARG;
  if (mode == MTP_STOCHASTIC && (!aligned16(draft_logits) || !aligned16(u_accept) || !aligned16(u_final)))
    return MTP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MTP_ERR_INVALID_ARG;
  if (ws_bytes < fused_workspace_bytes(B, k, V, d, mode)) return MTP_ERR_WORKSPACE;
  if (!tc_available()) return MTP_ERR_CUDA;
  DevInfo di;
  int rc = device_info(&di);
  if (rc) return rc;
  FusedCall fc{};
  fc.B = B; fc.k = k; fc.V = V; fc.d = d; fc.mode = mode; fc.T = T;
  fc.head = head; fc.hidden = target_hidden; fc.draft = draft_logits; fc.draft_tok = draft_tok;
  fc.u_accept = u_accept; fc.u_final = u_final;
  fc.out_tok = out_tok; fc.accept_len = accept_len; fc.num_accepted = num_accepted;
  fc.ws = ws;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  NvtxRange r("spec verify fused");
  cudaError_t e = timed(MTP_KC_VERIFY, s, [&] { return launch_fused_verify(fc, s, use_pdl()); });
  if (e == cudaSuccess) e = cudaGetLastError();
  return cuda_rc(e);
}

int mtp_get_status(const void *ws, mtp_stream_t stream, int32_t *status) {
  if (!ws || !status) return MTP_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return MTP_ERR_CUDA;
  *status = v;
  return MTP_OK;
}

int mtp_clear_status(void *ws, mtp_stream_t stream) {
  if (!ws) return MTP_ERR_INVALID_ARG;
  return cuda_rc(cudaMemsetAsync(ws, 0, sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream)));
}

const char *mtp_error_string(int code) {
  switch (code) {
    case MTP_OK: return "ok";
    case MTP_ERR_INVALID_ARG: return "invalid argument";
    case MTP_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MTP_ERR_WORKSPACE: return "workspace too small";
    case MTP_ERR_CUDA: return "CUDA error";
    case MTP_ERR_SCRATCH_LIMIT: return "problem needs more scratch than MTP_STATIC_SCRATCH_BYTES";
    default: return "unknown error";
  }
}

int mtp_profiler_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof.on = on != 0;
  for (int i = 0; i < MTP_KC_COUNT; ++i) g_prof.used[i] = 0;
  return MTP_OK;
}

int mtp_profiler_read(int kernel_class, double *total_ms, int64_t *launches) {
  if (kernel_class < 0 || kernel_class >= MTP_KC_COUNT || !total_ms || !launches) return MTP_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  double t = 0.0;
  auto &v = g_prof.ev[kernel_class];
  for (size_t i = 0; i < g_prof.used[kernel_class]; ++i) {
    if (cudaEventSynchronize(v[2 * i + 1]) != cudaSuccess) return MTP_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, v[2 * i], v[2 * i + 1]) != cudaSuccess) return MTP_ERR_CUDA;
    t += ms;
  }
  *total_ms = t;
  *launches = (int64_t)g_prof.used[kernel_class];
  return MTP_OK;
}

int64_t mtp_launch_count(void) { return (int64_t)g_launches.load(); }

int mtp_trace_read(MtpTraceEntry *entries, int max_entries) {
#ifndef MTP_TRACE
  (void)entries;
  (void)max_entries;
  return MTP_ERR_UNSUPPORTED_SHAPE;
#else
  if (max_entries < 0 || (max_entries > 0 && !entries)) return MTP_ERR_INVALID_ARG;
  using Collector = int (*)(mtp::TraceRec *, int);
  static const Collector collectors[] = {mtp::trace_collect_draft, mtp::trace_collect_attn_tc,
                                         mtp::trace_collect_verify,
                                         mtp::trace_collect_verify_split, mtp::trace_collect_tc,
                                         mtp::trace_collect_fused, mtp::trace_collect_chain,
                                         mtp::trace_collect_diag};
  static mtp::TraceRec recs[mtp::kTraceSlots];
  int n = 0;
  for (Collector col : collectors) {
    const int got = col(recs, mtp::kTraceSlots);
    if (got < 0) return MTP_ERR_CUDA;
    for (int i = 0; i < got && n < max_entries; ++i, ++n) {
      entries[n].launch = recs[i].grid;
      entries[n].kind = recs[i].kind;
      entries[n].reserved = 0;
      entries[n].t_start_ns = ~recs[i].nstart;
      entries[n].t_dep_ns = recs[i].ndep ? ~recs[i].ndep : 0ull;
      entries[n].t_end_ns = recs[i].end;
      for (int m = 0; m < 4; ++m) entries[n].t_mark_ns[m] = recs[i].mark[m];
    }
  }
  return n;
#endif
}

}  // extern "C"
