// Internal interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Plain structs of pointers and sizes, passed by value to
// the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mtp {

// Everything one depth of the draft chain reads or writes.
struct DraftCtx {
  // shape
  int B, d, Hq, Hkv, Dh, F, V, Lmax, k, j, mode;
  int jc;                 // this depth's cache row past ctx_len: depths of this call
                          // that ran the same module before it (j with one module)
  float eps, T;
  // weights (bf16)
  const uint16_t *E, *fc, *wq, *wk, *wv, *wo, *wgate, *wup, *wdown;
  const uint16_t *g_emb, *g_hid, *g_attn, *g_mlp, *g_final;
  // the draft's vocabulary head: E itself, or the Vd rows of a reduced draft
  // vocabulary with the full-vocabulary id of each (vmap null: head = E, Vd = V)
  const uint16_t *head;
  const int *vmap;
  int Vd;
  // caller inputs
  const uint16_t *h;      // [B, d] trunk hidden state
  const int *last_tok;    // [B]
  const int *ctx_len;     // [B]
  const float *u_draft;   // [B, k]
  uint16_t *kc, *vc;      // [B, Hkv, Lmax, Dh]
  // outputs
  int *draft_tok;         // [B, k]
  float *logits;          // [B, k, V] or null (greedy without logits)
  // dynamic draft length (null k_eff: off): sequence b keeps the drafts before
  // its first depth whose draft confidence is below stop_p
  int *k_eff;             // [B] drafts kept (k until the sequence stops)
  unsigned *n_active;     // sequences still drafting (workspace)
  float stop_p;
  // workspace
  int *status;
  unsigned *lm_cnt;       // 1 ticket counter
  float *x0, *x1, *x2;    // [B, d]
  float *q, *o;           // [B, Hq*Dh]
  float *act;             // [B, F]
  float *lm_part;         // [B, lm_grid, 4]
  int lm_grid;            // CTAs of the LM-head launch
  int lm_rpc;             // vocabulary rows per LM-head CTA
  int zero_counters;      // this launch clears the ticket counters first
  // sequences longest context first (batches on the tensor-core path; null:
  // index order): the attention's clusters are scheduled in this order
  int *seq_order;         // [B]
};

enum GemvOp { OP_FC = 0, OP_QKV = 1, OP_WO = 2, OP_GATEUP = 3, OP_DOWN = 4, OP_LMHEAD = 5 };

// How one weight-streaming GEMV launch is cut up.
struct GemvPlan {
  int op;
  int N;             // virtual rows
  int K;             // columns
  int P;             // column pieces per row (divides the warps per CTA)
  int PC;            // columns per piece (multiple of 8)
  int nv;            // 16-byte vectors per lane per piece = ceil(PC / 256)
  int rows_per_cta;  // contiguous rows per CTA (even for the gate/up pair layout)
  int grid;          // CTAs
  int bg;            // batch rows per group (activation registers per lane)
  int ngroups;       // batch groups = ceil(B / bg)
  int stages;        // TMA ring depth per warp
  int pre;           // stages requested before the wait for the previous kernel (the rest after the activations)
  int factor;        // the norm's scale applied to the finished dot products (else to the inputs)
  size_t smem;       // dynamic shared memory bytes
};

constexpr int kGemvWarps = 8;
constexpr int kMaxLmGrid = 2048;  // LM-head CTAs at most: the workspace holds that many partials per sequence
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kAttnThreads = 288;  // 8 compute warps and a K/V streaming warp
constexpr int kMaxGroup = 8;        // Hq / Hkv

GemvPlan plan_gemv(int op, int N, int K, int B, int num_sms);

// Several GEMV ops in one cooperative launch (chain.cu): ops[o] runs op
// ops[o].op of context c[ops[o].ctx] with plan ops[o].g, a grid barrier between
// consecutive ops; the barrier after op select_after picks the draft token.
constexpr int kMaxChainOps = 8;
constexpr size_t kChainSmemCap = 110 * 1024;  // per CTA: two CTAs per SM
struct ChainOp {
  int op, ctx;
  GemvPlan g;
};
struct ChainArgs {
  DraftCtx c[2];
  ChainOp ops[kMaxChainOps];
  int nops, select_after;
  int ring_bytes, part_floats, ys_floats;  // set by launch_chain
  unsigned *bar;  // [0] arrivals, [1] generation: workspace words, zero before the first use
  int *status;
};
bool chain_op_ok(const GemvPlan &g);
cudaError_t launch_chain(ChainArgs a, cudaStream_t s);
cudaError_t launch_gemv(const DraftCtx &c, const GemvPlan &g, cudaStream_t s, bool pdl);
cudaError_t launch_attention(const DraftCtx &c, int cluster, cudaStream_t s, bool pdl);
// p[0 .. n) = v (a reduced draft vocabulary's logits: -inf at the other ids)
cudaError_t launch_fill(float *p, size_t n, float v, cudaStream_t s, bool pdl);
size_t attention_smem_bytes(int Dh);
int attention_cluster_size(int ctx_max, int pairs, int num_sms, int max_cluster, bool tc);
// Tensor-core decode attention (GQA groups of 2..16, head size 64 or 128).
bool attention_tc_shape_ok(const DraftCtx &c);
cudaError_t launch_attention_tc(const DraftCtx &c, int cluster, cudaStream_t s, bool pdl);

// Tensor-core path of the draft chain (batches of several sequences).
struct MtpShape {
  int B, d, Hq, Hkv, Dh, F, V;
};
struct TcSizes {
  int rows;            // activation rows: the batch padded to the MMA N
  int kmax;            // activation row length: max K over the GEMMs
  size_t part_floats;  // split-K partials / LM-head logits scratch
};
struct TcBufs {
  uint16_t *a[3];  // [rows, kmax] bf16 terms hi, mid, lo of the next GEMM's input
  int rows, kmax;
  float *part;
  size_t part_floats;
};
bool tc_shape_ok(const MtpShape &s);  // the workspace holds the tensor-core buffers
bool tc_available();                  // the driver can encode tensor maps
TcSizes tc_sizes(const MtpShape &s);
cudaError_t tc_set_attributes();
cudaError_t run_block_pre_tc(const DraftCtx &c, const TcBufs &t, cudaStream_t s, bool pdl);
cudaError_t run_block_post_tc(const DraftCtx &c, const TcBufs &t, cudaStream_t s, bool pdl);
cudaError_t run_lmhead_tc(const DraftCtx &c, const TcBufs &t, cudaStream_t s, bool pdl);

// Verification launch.
struct VerifyPlan {
  int NS;          // 512-element sub-chunks per logit row
  int C;           // CTAs per cluster: each owns C-th of every row's sub-chunks
  int G;           // clusters
  int lookahead;   // items a cluster claims ahead of the one it streams
  unsigned total;  // work items: one per position of one sequence
};

// A sequence's first rejection, for the residual draw of verify_split.cu.
struct alignas(16) SplitRec {
  float Mt, iZt, Ml, iZl;  // target / draft row max and inverse partition sum
  int j, flags, pad0, pad1;
};

struct VerifyArgs {
  int B, k, V, mode;
  float T;
  const float *target;   // [B, k+1, V]
  const float *draft;    // [B, k, V]
  const int *draft_tok;  // [B, k]
  const int *k_eff;      // [B] drafts kept per sequence, or null (all k)
  const float *u_accept; // [B, k]
  const float *u_final;  // [B]
  int *out_tok;          // [B, k+1]
  int *accept_len;       // [B]
  int *num_accepted;     // [B]
  int *status;
  // state in the workspace: zero before the first call, left zero by each call
  unsigned *ctl;         // [0] claim counter, [1] CTAs finished
  unsigned *hint;        // [B] k + 1 - (earliest position known to reject), or 0
  unsigned long long *rec;  // [B, k+1] per position: flags | token << 32, 0 until written
  VerifyPlan p;
  // the ticketed stochastic kernel (verify_split.cu), when split is set
  int split;
  int snch;                // 32768-element chunks a row
  int sNA, sNB, sD;        // statistics / residual items a sequence; lag of the residual group in sequences
  int shint;               // L2 policy: 0 normal; 1 pair rows evict_last, the rest evict_first; 2 pair rows normal
  unsigned *sseq;          // [B, 4] statistics arrivals, residual arrivals, decision, -- (state: zero, left zero)
  SplitRec *srec;          // [B] the rejection each sequence's residual items draw from
  float2 *spart;           // [B, 2k+1, snch] chunk (max, sum of exp2)
  double *cmass;           // [B, snch] residual chunk masses
  float *smass;            // [B, snch, 64] residual masses of the chunks' 512-element sub-chunks
};

size_t verify_state_bytes(int B, int k, int V);
void verify_bind_state(VerifyArgs &a, void *state);
bool plan_verify(int B, int k, int V, VerifyPlan *p);
cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t s, bool pdl);
cudaError_t verify_set_attributes();
int split_chunks(int V);
bool split_shape_ok(int B, int k, int V);
size_t split_state_bytes(int B, int k, int V);
void split_bind_state(VerifyArgs &a, void *state, int lag_items);
cudaError_t launch_verify_split(const VerifyArgs &a, cudaStream_t s, bool pdl);

// Verification from the target's hidden states (fused.cu).
struct FusedCall {
  int B, k, V, d, mode;
  float T;
  const void *head;       // [V, d] bf16
  const void *hidden;     // [B (k+1), d] bf16
  const float *draft;     // [B, k, V] (stochastic)
  const int *draft_tok;   // [B, k]
  const float *u_accept;  // [B, k]
  const float *u_final;   // [B]
  int *out_tok, *accept_len, *num_accepted;
  void *ws;               // fused_workspace_bytes(), 256-byte aligned; starts with the status word
};
bool fused_shape_ok(int B, int k, int V, int d);
size_t fused_workspace_bytes(int B, int k, int V, int d, int mode);
cudaError_t fused_set_attributes();
cudaError_t launch_fused_verify(const FusedCall &fc, cudaStream_t s, bool pdl);

// Launch-trace record (a build with MTP_TRACE; common.cuh): start and
// dependency times stored complemented, so that atomicMax keeps the earliest.
struct TraceRec {
  unsigned long long grid, nstart, ndep, end;
  unsigned long long mark[4];  // the last CTA to reach each of a kernel's intermediate marks
  int kind, pad[3];
};
constexpr int kTraceSlots = 4096;
// record kinds: the MTP_TK_* values of the public header
constexpr int kTkGemv = 0, kTkAttn = 10, kTkAttnTc = 11, kTkVerify = 20, kTkVerifySplit = 21, kTkTcGemm = 30,
              kTkTcAux = 31, kTkFusedGemm = 40, kTkFusedAux = 41, kTkChain = 50;

// bookkeeping shared with api.cu
void note_launch();
// Unique id of the calling thread's current CUDA context (0 if there is none):
// kernel attributes and device addresses are set up again when it changes.
unsigned long long context_id();

}  // namespace mtp
