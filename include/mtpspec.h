/*
 * mtpspec -- the hot path of MTP speculative decoding on one GB300 (sm_103a):
 * a single Multi-Token-Prediction draft block chained k times, then
 * verification of the k drafted tokens against the target's distributions.
 *
 * Sources (web pages; section names as printed on them):
 *  [P1] "Optimize vLLM speculative decoding with FastMTP heads"
 *  [P2] "Faster Rollouts with MTP Speculative Decoding"
 *  [P3] "Speculative Decoding and MTP: Why Guessing Is Free"
 *  [P4] "The Tiny Draft Model Hidden Inside Qwen"
 *
 * Conventions shared by every entry point
 *  - Every array argument is a DEVICE pointer owned by the caller, aligned to
 *    16 bytes; the workspace is aligned to 256 bytes.  Nothing here allocates
 *    or frees device memory.
 *  - Calls are asynchronous on the given stream (a cudaStream_t; NULL is the
 *    legacy default stream).  They return MTP_OK or a negative MTP_ERR_* code
 *    for errors the host can see (bad argument, unsupported shape, workspace too
 *    small, failed launch).  Conditions only the device can see (a token id out
 *    of range, a context length past the cache, a non-finite logit row, a
 *    bounded wait that ran out) set bits of a status word inside the workspace;
 *    mtp_get_status() reads it.
 *  - A workspace must be zero-filled (cudaMemset) before its first use.  It
 *    holds the status word and the verifier's work counters and tickets, which
 *    every call leaves at zero for the next one; zero it again after a call
 *    that set MTP_STATUS_TIMEOUT.  Calls that share a workspace must not
 *    overlap in time.
 *  - Random draws use caller-supplied uniforms in [0, 1), so every result is a
 *    deterministic function of the inputs, bit for bit from run to run.
 *  - bf16 means IEEE binary32's upper 16 bits (the storage type of the weights,
 *    the trunk hidden state and the KV cache).  Logits are float32.
 */
#ifndef MTPSPEC_H
#define MTPSPEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *mtp_stream_t; /* identical to cudaStream_t */

/* Host-visible return codes. */
enum {
    MTP_OK = 0,
    MTP_ERR_INVALID_ARG = -1,       /* null / misaligned pointer, k outside 1..8, T <= 0, ... */
    MTP_ERR_UNSUPPORTED_SHAPE = -2, /* dims the kernels do not implement (see MtpDims) */
    MTP_ERR_WORKSPACE = -3,         /* workspace smaller than the *_workspace_size() answer */
    MTP_ERR_CUDA = -4,              /* a CUDA runtime call or launch failed */
    MTP_ERR_SCRATCH_LIMIT = -5      /* mtp_draft_noalloc: the problem needs more
                                       than MTP_STATIC_SCRATCH_BYTES of scratch */
};

/* Bits of the device status word (sticky until mtp_clear_status()). */
enum {
    MTP_STATUS_TIMEOUT = 1,    /* a bounded wait gave up; results of that call are invalid */
    MTP_STATUS_BAD_TOKEN = 2,  /* a token id outside [0, V); token 0 was used instead */
    MTP_STATUS_BAD_CTX = 4,    /* ctx_len[b] < 0 or ctx_len[b] + k > Lmax; clamped */
    MTP_STATUS_NONFINITE = 8,  /* a logit row without a finite maximum */
    MTP_STATUS_BOUNDS = 16     /* only a library built with MTP_BOUNDS: an index outside
                                  its buffer was found and that access skipped */
};

typedef enum { MTP_GREEDY = 0, MTP_STOCHASTIC = 1 } MtpMode;

/*
 * Shape of the draft module and of the batch.  [P4] "The Tiny Draft Model
 * Hidden Inside Qwen", opening section: the module is one input projection
 * mtp.fc, one full-attention transformer block and three normalisation weights,
 * and it reuses the trunk's token embedding.
 *   B     sequences in the batch (>= 1)
 *   d     hidden width (multiple of 8)
 *   Hq    query heads; Hkv key/value heads (Hq % Hkv == 0, Hq / Hkv <= 8)
 *   Dh    head size: 32, 64 or 128
 *   F     SwiGLU inner width (multiple of 8)
 *   V     vocabulary size (>= 1; any value)
 *   Lmax  KV-cache capacity per sequence (positions)
 *   rms_eps  RMSNorm epsilon: rms(v) = v / sqrt(mean(v^2) + eps)
 */
typedef struct {
    int32_t B, d, Hq, Hkv, Dh, F, V, Lmax;
    float rms_eps;
} MtpDims;

/*
 * Weights, all bf16 row-major [out, in], no biases.  E [V, d] is the shared
 * embedding AND the vocabulary head ([P1] "Key features": full-vocabulary head
 * shared with the verifier; [P4] opening section: no second embedding table).
 *   fc [d, 2d] applied to [rms(E[tok]) * g_emb ; rms(x) * g_hid]
 *   wq [Hq*Dh, d], wk [Hkv*Dh, d], wv [Hkv*Dh, d], wo [d, Hq*Dh]
 *   wgate [F, d], wup [F, d], wdown [d, F]                     (SwiGLU)
 *   g_emb, g_hid, g_attn, g_mlp, g_final [d]                   (norm gains)
 */
typedef struct {
    const void *E, *fc, *wq, *wk, *wv, *wo, *wgate, *wup, *wdown;
    const void *g_emb, *g_hid, *g_attn, *g_mlp, *g_final;
} MtpWeights;

/* Bytes of workspace mtp_draft / spec_step need for these dims and depth k
 * (0 if the arguments are invalid). */
size_t mtp_workspace_size(const MtpDims *dims, int k);

/*
 * mtp_draft -- run the MTP module k times in a chain ([P4] "One step deeper
 * than the main model" and "What vLLM and SGLang do with the weights"; [P1]
 * "Why fine-tune a single MTP head": the same module is applied autoregressively,
 * fed its own output hidden state and the token it just drafted).
 *
 * Depth j = 0..k-1 computes, per sequence b:
 *   u  = [rms(E[tok]) * g_emb ; rms(x) * g_hid];  x0 = fc u
 *   n  = rms(x0) * g_attn;  q = wq n;  K/V rows wk n, wv n stored (bf16) at
 *        position ctx_len[b] + j of the cache
 *   o  = softmax attention of q over cache positions 0 .. ctx_len[b] + j
 *        (query head h uses kv head h / (Hq/Hkv); scale 1/sqrt(Dh))
 *   x1 = x0 + wo o;  x2 = x1 + wdown(silu(wgate rms(x1)*g_mlp) * wup rms(x1)*g_mlp)
 *   logits = E (rms(x2) * g_final)
 *   draft token: argmax (lowest index on ties) if greedy; else the inverse-CDF
 *   draw of softmax(logits / T) at u_draft[b, j]
 * with x = h, tok = last_tok at depth 0 and x = x2, tok = the new draft after.
 *
 *   h         [B, d] bf16 trunk hidden state h_t
 *   last_tok  [B] int32, the token the trunk just produced
 *   k_cache, v_cache  [B, Hkv, Lmax, Dh] bf16; rows [0, ctx_len[b]) hold the
 *             context.  Rows ctx_len[b] .. ctx_len[b]+k-1 are overwritten with
 *             the drafts' keys/values; ctx_len is not changed (after verifying,
 *             the caller advances it by num_accepted + 1: rejected rows are
 *             simply overwritten next step).  Requires ctx_len[b] + k <= Lmax.
 *   ctx_len   [B] int32
 *   k         draft depth, 1..8;  T  temperature (> 0; ignored when greedy)
 *   u_draft   [B, k] float32 uniforms (may be NULL when greedy)
 *   draft_tok [B, k] int32 output
 *   draft_logits [B, k, V] float32 output, or NULL when greedy
 *   ws, ws_bytes  workspace of at least mtp_workspace_size(dims, k) bytes
 * Returns MTP_OK or MTP_ERR_*.
 */
int mtp_draft(const MtpDims *dims, const MtpWeights *w, const void *h,
              const int32_t *last_tok, void *k_cache, void *v_cache,
              const int32_t *ctx_len, int k, float T, int mode,
              const float *u_draft, int32_t *draft_tok, float *draft_logits,
              void *ws, size_t ws_bytes, mtp_stream_t stream);

/*
 * mtp_draft_noalloc -- mtp_draft without a caller-supplied workspace and
 * without allocating: its scratch is a fixed device array of
 * MTP_STATIC_SCRATCH_BYTES that is part of the library's image.  The pages
 * describe no such call; it exists for callers that cannot hand over device
 * memory: a host engine that has already given all free HBM to its KV-cache
 * pool (a cudaMalloc would then fail, and it synchronises the device in any
 * case), or code embedded in another runtime that passes in a stream but no
 * allocator.
 *
 * Arguments and results as mtp_draft, except:
 *   status  optional device int32: if not NULL, the status word (MTP_STATUS_*
 *           bits) of this call is copied there, on the stream, after the chain.
 * Limits: the call keeps no logits and no verifier state in its scratch, so it
 * needs mtp_workspace_size(dims, k) less those two regions: the activations,
 * the LM-head partials and, for batches of 5 or more, the tensor-core buffers.
 * That must not exceed MTP_STATIC_SCRATCH_BYTES (else MTP_ERR_SCRATCH_LIMIT,
 * nothing launched).  At d = 4096, V = 151936 and F = 12288 a batch of up to 4
 * sequences fits (about 0.17 MB per sequence); at d = 256 batches of 3 fit at
 * any vocabulary size.  The first call on a device does that device's set-up
 * (it loads the library's device image and looks up the scratch array's
 * address), so make it before any stream capture; the lookup is made again
 * when the device's context has changed (after cudaDeviceReset, for one).
 * Each call zeroes the scratch's status word and counters on the stream
 * before the chain.  There is one scratch array per device: calls that
 * overlap in time on the same device (two streams, or two host threads) race
 * on it and must be serialised by the caller.
 */
#define MTP_STATIC_SCRATCH_BYTES ((size_t)4 << 20)
int mtp_draft_noalloc(const MtpDims *dims, const MtpWeights *w, const void *h,
                      const int32_t *last_tok, void *k_cache, void *v_cache,
                      const int32_t *ctx_len, int k, float T, int mode,
                      const float *u_draft, int32_t *draft_tok, float *draft_logits,
                      int32_t *status, mtp_stream_t stream);

/* Bytes of workspace spec_verify needs (0 if the arguments are invalid). */
size_t spec_verify_workspace_size(int B, int k, int V);

/*
 * spec_verify -- accept or reject k drafts per sequence against the target
 * ([P4] "How the draft becomes real output": longest agreeing prefix, then the
 * corrected replacement at the first rejection; [P3] "Speculative decoding:
 * draft, then verify" and "It's exact, not approximate").
 *
 * Greedy: draft j+1 is accepted while it equals argmax(target row j) (lowest
 * index on ties); the emitted token after the accepted prefix is argmax of the
 * first disagreeing row (or of row k when all k agree).  Equals plain greedy.
 *
 * Stochastic, with p_j = softmax(target_j / T), q_j = softmax(draft_j / T) and
 * d = draft_tok[b, j]: accept iff u_accept[b, j] * q_j(d) < p_j(d), i.e. with
 * probability min(1, p/q); at the first rejection r emit the inverse-CDF draw at
 * u_final[b] of max(0, p_r - q_r) (of p_r if that is identically zero); if all
 * k are accepted emit the draw at u_final[b] of p_k (the bonus token).
 *
 *   target_logits [B, k+1, V] float32;  draft_logits [B, k, V] float32 (NULL ok
 *   when greedy);  draft_tok [B, k] int32;  u_accept [B, k], u_final [B] float32
 *   (NULL ok when greedy)
 *   out_tok [B, k+1] int32: accepted drafts then the emitted token, -1 padded
 *   accept_len [B] int32 = tokens emitted (1 .. k+1); num_accepted [B] = accept_len - 1
 */
int spec_verify(int B, int k, int V, float T, int mode,
                const float *target_logits, const float *draft_logits,
                const int32_t *draft_tok, const float *u_accept, const float *u_final,
                int32_t *out_tok, int32_t *accept_len, int32_t *num_accepted,
                void *ws, size_t ws_bytes, mtp_stream_t stream);

/*
 * spec_step -- mtp_draft followed by spec_verify on the same stream, with the
 * kernels of the two chained back to back.  Arguments as above; draft_logits
 * may be NULL in either mode (stochastic mode then keeps them in the
 * workspace, which mtp_workspace_size() already counts).
 */
int spec_step(const MtpDims *dims, const MtpWeights *w, const void *h,
              const int32_t *last_tok, void *k_cache, void *v_cache,
              const int32_t *ctx_len, int k, float T, int mode,
              const float *u_draft, const float *target_logits,
              const float *u_accept, const float *u_final,
              int32_t *draft_tok, float *draft_logits,
              int32_t *out_tok, int32_t *accept_len, int32_t *num_accepted,
              void *ws, size_t ws_bytes, mtp_stream_t stream);

/*
 * Distinct modules per depth.  [P1] "What is multi-token prediction?": a
 * model trained with MTP carries D sequential modules, one per additional
 * future token, chained so that each takes the previous one's output hidden
 * state; every module has its own transformer block and input projection and
 * shares the embedding and the output head with the main model.  [P1] "Why
 * fine-tune a single MTP head": DeepSeek-V3 trains D distinct modules, while
 * engines usually keep one and reuse it -- mtp_draft's case.
 *
 * One module: its weights and its own K/V cache (its block has its own
 * attention).  `modules` is a HOST array of n_modules such structs, 1 <=
 * n_modules <= k; every pointer inside is a device pointer as for mtp_draft.
 * Depth j runs module m = min(j, n_modules - 1): n_modules = 1 is mtp_draft's
 * single module applied k times, n_modules = k gives every depth its own
 * module, and in between the last module serves the remaining depths.  Depth j
 * stores its K/V row at position ctx_len[b] + jc of module m's cache and
 * attends over that cache's positions 0 .. ctx_len[b] + jc, where jc = j - m
 * is the number of earlier depths of this call that ran module m (jc = j with
 * one module, 0 with one module per depth).  Each module's E is its embedding
 * and vocabulary head; pass the same E in every module for the shared head of
 * the pages.  Everything else, the outputs and the workspace
 * (mtp_workspace_size(dims, k)) are as for mtp_draft / spec_step.
 */
typedef struct {
    MtpWeights w;
    void *k_cache, *v_cache; /* [B, Hkv, Lmax, Dh] bf16, this module's own */
} MtpModule;

int mtp_draft_modules(const MtpDims *dims, const MtpModule *modules, int n_modules,
                      const void *h, const int32_t *last_tok, const int32_t *ctx_len,
                      int k, float T, int mode, const float *u_draft,
                      int32_t *draft_tok, float *draft_logits,
                      void *ws, size_t ws_bytes, mtp_stream_t stream);

int spec_step_modules(const MtpDims *dims, const MtpModule *modules, int n_modules,
                      const void *h, const int32_t *last_tok, const int32_t *ctx_len,
                      int k, float T, int mode, const float *u_draft,
                      const float *target_logits, const float *u_accept,
                      const float *u_final, int32_t *draft_tok, float *draft_logits,
                      int32_t *out_tok, int32_t *accept_len, int32_t *num_accepted,
                      void *ws, size_t ws_bytes, mtp_stream_t stream);

/*
 * Dynamic draft length.  [P2] "Faster Rollouts with MTP Speculative
 * Decoding", section "What's Next", names it without a rule; the rule here:
 * the draft confidence of depth j is the largest probability of the
 * distribution its token is taken from (softmax(logits / T) when stochastic,
 * softmax(logits) when greedy).  Sequence b keeps the drafts before its first
 * depth j whose confidence is below stop_p: k_eff[b] = j, or k if none is
 * (stop_p = 0 never stops; stop_p > 1 stops at depth 0, a plain decoding
 * step).  The stop depends only on the draft, so the stochastic output keeps
 * the target's distribution exactly.
 *
 * mtp_draft_dynamic: mtp_draft plus k_eff [B] int32 (device, output).  Drafts
 *   and logits at depths >= k_eff[b] are unspecified.  Once every sequence of
 *   the batch has stopped, the later depths' weight-streaming kernels (batches
 *   of up to 4) return after their first copies land, so a stopped chain does
 *   not stream the remaining depths' weights.
 * spec_verify_dynamic: spec_verify where sequence b is verified over its
 *   drafts 0 .. k_eff[b]-1 only, the bonus row being target row k_eff[b];
 *   k_eff [B] int32 (device, input; clamped to 0..k; NULL: k for all).
 *   accept_len[b] is then in 1 .. k_eff[b]+1.
 * spec_step_dynamic: the two in one call, k_eff written by the draft and read
 *   by the verification.
 * stop_p must be finite and >= 0 (else MTP_ERR_INVALID_ARG).
 */
int mtp_draft_dynamic(const MtpDims *dims, const MtpWeights *w, const void *h,
                      const int32_t *last_tok, void *k_cache, void *v_cache,
                      const int32_t *ctx_len, int k, float T, int mode, float stop_p,
                      const float *u_draft, int32_t *draft_tok, float *draft_logits,
                      int32_t *k_eff, void *ws, size_t ws_bytes, mtp_stream_t stream);

int spec_verify_dynamic(int B, int k, int V, float T, int mode,
                        const float *target_logits, const float *draft_logits,
                        const int32_t *draft_tok, const int32_t *k_eff,
                        const float *u_accept, const float *u_final,
                        int32_t *out_tok, int32_t *accept_len, int32_t *num_accepted,
                        void *ws, size_t ws_bytes, mtp_stream_t stream);

int spec_step_dynamic(const MtpDims *dims, const MtpWeights *w, const void *h,
                      const int32_t *last_tok, void *k_cache, void *v_cache,
                      const int32_t *ctx_len, int k, float T, int mode, float stop_p,
                      const float *u_draft, const float *target_logits,
                      const float *u_accept, const float *u_final,
                      int32_t *draft_tok, float *draft_logits, int32_t *k_eff,
                      int32_t *out_tok, int32_t *accept_len, int32_t *num_accepted,
                      void *ws, size_t ws_bytes, mtp_stream_t stream);

/*
 * Reduced draft vocabulary.  [P1] "How FastMTP-style fine-tuning works in
 * Speculators" (its note on the full-vocabulary head) and "What's next?" name
 * FR-Spec-style frequency-ranked draft-vocabulary reduction, to shrink the cost
 * of each recursive step, without a rule.  The
 * rule here: the draft head is N rows of E chosen by the caller (in FR-Spec,
 * the N most frequent tokens).
 *   head_rows  [N, d] bf16: those rows, gathered once by the caller
 *              (head_rows[i] = E[vocab_map[i]])
 *   vocab_map  [N] int32: the vocabulary id of each head row; distinct ids in
 *              [0, V) (an id outside it sets MTP_STATUS_BAD_TOKEN)
 *   n_draft_vocab = N, 128 <= N <= V
 * The draft distribution is q = softmax over the N head logits (zero outside
 * the N ids); the draft token is vocab_map of the argmax / inverse-CDF draw
 * over the N rows in row order.  The token embedding still reads E.
 * draft_logits [B, k, V] stays in full-vocabulary layout: the N logits at
 * their ids and -inf at every other id, so spec_verify (q = 0 there) needs
 * nothing new and stays exact.  Everything else is as for mtp_draft /
 * spec_step.
 */
int mtp_draft_reduced(const MtpDims *dims, const MtpWeights *w,
                      const void *head_rows, const int32_t *vocab_map, int n_draft_vocab,
                      const void *h, const int32_t *last_tok, void *k_cache, void *v_cache,
                      const int32_t *ctx_len, int k, float T, int mode,
                      const float *u_draft, int32_t *draft_tok, float *draft_logits,
                      void *ws, size_t ws_bytes, mtp_stream_t stream);

int spec_step_reduced(const MtpDims *dims, const MtpWeights *w,
                      const void *head_rows, const int32_t *vocab_map, int n_draft_vocab,
                      const void *h, const int32_t *last_tok, void *k_cache, void *v_cache,
                      const int32_t *ctx_len, int k, float T, int mode,
                      const float *u_draft, const float *target_logits,
                      const float *u_accept, const float *u_final,
                      int32_t *draft_tok, float *draft_logits,
                      int32_t *out_tok, int32_t *accept_len, int32_t *num_accepted,
                      void *ws, size_t ws_bytes, mtp_stream_t stream);

/*
 * Verification from the target's hidden states.  [P4] "How the draft becomes
 * real output": the target runs once over every candidate position and its
 * own vocabulary head gives its distribution at each of them.  This call
 * takes what that head consumes -- the target's final hidden state after its
 * final norm, one row per position -- together with the head itself, and
 * forms the target logits t = head . h inside the verification (bf16
 * operands, fp32 accumulation on the tensor cores), so that the [B, k+1, V]
 * logits never have to be written by one kernel and read back by another.
 * The decisions are spec_verify's, same rule, same uniforms.
 *
 *   d             hidden width (multiple of 8)
 *   head          [V, d] bf16: the target's vocabulary head (with the pages'
 *                 shared head, the embedding matrix E of MtpWeights)
 *   target_hidden [B, k+1, d] bf16: row (b, j) is the head's input at
 *                 position j of sequence b (after the context and the first j
 *                 drafts)
 *   draft_logits, draft_tok, u_accept, u_final, out_tok, accept_len,
 *   num_accepted  as spec_verify (the draft logits, u_accept and u_final may
 *                 be NULL when greedy)
 *   ws, ws_bytes  workspace of at least spec_verify_fused_workspace_size()
 *                 bytes, 256-byte aligned; its first word is the status word
 *                 (mtp_get_status).  Greedy keeps only per-(row, 256-token
 *                 tile) partials there; stochastic also keeps the target's
 *                 fp32 logits, since its one residual draw per sequence needs
 *                 every element of the first rejecting row.
 * Returns MTP_OK or MTP_ERR_*; stochastic calls with B * k * ceil(V / 256) of
 * 2^31 or more return MTP_ERR_UNSUPPORTED_SHAPE (and the workspace size 0).  A
 * draft token outside [0, V) is never accepted and sets MTP_STATUS_BAD_TOKEN.
 */
size_t spec_verify_fused_workspace_size(int B, int k, int V, int d, int mode);

int spec_verify_fused(int B, int k, int V, int d, float T, int mode,
                      const void *head, const void *target_hidden,
                      const float *draft_logits, const int32_t *draft_tok,
                      const float *u_accept, const float *u_final,
                      int32_t *out_tok, int32_t *accept_len, int32_t *num_accepted,
                      void *ws, size_t ws_bytes, mtp_stream_t stream);

/* Wait for the stream, then copy the workspace's status word (MTP_STATUS_* bits)
 * to *status.  Returns MTP_OK or MTP_ERR_*. */
int mtp_get_status(const void *ws, mtp_stream_t stream, int32_t *status);

/* Zero the status word (asynchronously, on the stream). */
int mtp_clear_status(void *ws, mtp_stream_t stream);

/*
 * Diagnostics.  Runs the library's two bounded mbarrier waits (the spinning
 * and the parked form) on a barrier phase that no thread ever completes.
 * Each gives up after the wait limit (2 s), sets MTP_STATUS_TIMEOUT in
 * *status and returns; the context stays usable.
 *   status  device int32, 4-byte aligned, owned by the caller; bits are OR-ed
 *           in, never cleared here.
 * Asynchronous on the stream (about 2 s of GPU time).  Returns MTP_OK,
 * MTP_ERR_INVALID_ARG (null or misaligned status) or MTP_ERR_CUDA.
 */
int mtp_selftest_wait_timeout(int32_t *status, mtp_stream_t stream);

/* Human-readable text for an MTP_ERR_* code. */
const char *mtp_error_string(int code);

/*
 * Instrumentation.  mtp_profiler_enable(1) makes later calls record a CUDA
 * event pair around every launch of the kernel classes below (this splits the
 * programmatic launch chain at those points, so time steps with it off);
 * mtp_profiler_read() waits for the events and returns the summed time and the
 * launch count since the last enable.  mtp_launch_count() counts every kernel
 * this library has launched in the process.
 */
enum { MTP_KC_LMHEAD = 0, MTP_KC_VERIFY = 1, MTP_KC_ATTN = 2, MTP_KC_GEMV = 3, MTP_KC_COUNT = 4 };
int mtp_profiler_enable(int on);
int mtp_profiler_read(int kernel_class, double *total_ms, int64_t *launches);
int64_t mtp_launch_count(void);

/*
 * Launch trace, for the library built with MTP_TRACE (build variant "trace",
 * loaded by the binding when MTP_LIB_VARIANT=trace).  Every kernel records,
 * on the GPU's global nanosecond timer, when its first CTA started, when the
 * first CTA got past its wait for the previous kernel (programmatic dependent
 * launch; 0 where the kernel does not record it), when the last CTA reached
 * each of up to four intermediate points of the kernel (the GEMV: activations
 * loaded, last weight piece used, epilogue done; tensor-core attention: query
 * staged, last tile done, CTA merged, cluster combined) and when the last CTA
 * finished.  Unlike the event profiler above it leaves the launch chain
 * intact, so it shows the live overlap of the chained kernels.
 *
 * mtp_trace_read() copies up to max_entries records (in no particular order)
 * into `entries` (host memory, owned by the caller) and clears the device
 * buffers.  Call it once the traced work has completed (after a device or
 * stream synchronisation).  A buffer holds 4096 launches per source file; a
 * later launch can overwrite an unread record of one 4096 launches earlier.
 * Returns the number of records written (>= 0), MTP_ERR_INVALID_ARG for a
 * null buffer with max_entries > 0, MTP_ERR_UNSUPPORTED_SHAPE from a library
 * built without MTP_TRACE, or MTP_ERR_CUDA.
 */
enum {
    MTP_TK_GEMV = 0,        /* + the op: 0 input projection, 1 QKV, 2 output projection,
                               3 gate/up, 4 down, 5 LM head */
    MTP_TK_ATTN = 10,       /* CUDA-core decode attention */
    MTP_TK_ATTN_TC = 11,    /* tensor-core decode attention */
    MTP_TK_VERIFY = 20,     /* cluster verification kernel */
    MTP_TK_VERIFY_SPLIT = 21, /* ticketed stochastic verification kernel */
    MTP_TK_TC_GEMM = 30,    /* tcgen05 GEMM of the batched path */
    MTP_TK_TC_AUX = 31,     /* the batched path's prologue / select / scatter kernels */
    MTP_TK_FUSED_GEMM = 40, /* spec_verify_fused: head GEMM */
    MTP_TK_FUSED_AUX = 41,  /* spec_verify_fused: draft statistics, decisions and draws */
    MTP_TK_CHAIN = 50       /* chain launch of several GEMV ops */
};
typedef struct MtpTraceEntry {
    uint64_t launch;      /* the launch's grid id */
    int32_t kind;         /* MTP_TK_* */
    int32_t reserved;
    uint64_t t_start_ns;  /* first CTA started */
    uint64_t t_dep_ns;    /* first CTA past its wait for the previous kernel, or 0 */
    uint64_t t_end_ns;    /* last CTA finished */
    uint64_t t_mark_ns[4]; /* the last CTA to reach each of the kernel's intermediate marks, or 0 */
} MtpTraceEntry;
int mtp_trace_read(MtpTraceEntry *entries, int max_entries);

#ifdef __cplusplus
}
#endif
#endif /* MTPSPEC_H */
