"""Seeded synthetic inputs for the draft + verify path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it.  Every tensor comes from its own numpy PCG64 stream, derived
from (seed, tensor name, chunk index), so the values do not depend on how many
threads generate them or in which order tensors are requested.

Shapes follow the pages' models: hidden 4096-5120, 32-40 query heads over 8 KV
heads of size 128, SwiGLU FFN 12288-17408, vocabularies of 151936 and 256000,
contexts up to 16384 tokens, draft depths 1-5 with k = 3 the default ("Faster
Rollouts with MTP Speculative Decoding", section "Enabling MTP"; "Optimize vLLM
speculative decoding with FastMTP heads", section "Stitch and serve").  No
dataset is involved: the pages' GSM8K / DAPO workloads are represented only by
their sequence lengths.

bf16 tensors are returned as their raw bit patterns in ``numpy.uint16`` arrays.
"""

import zlib
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace  # noqa: F401 (replace is re-exported)

import numpy as np
import torch

GREEDY = 0
STOCHASTIC = 1

_CHUNK = 1 << 24  # elements per independent sub-stream


@dataclass(frozen=True)
class Workload:
    """One synthetic workload.

    ctx is either a single context length or an inclusive (lo, hi) range from
    which each sequence's length is drawn uniformly.  target_std / draft_std
    describe the logits used when the target (and, for verify-only workloads,
    the draft) logits are drawn directly.  draft_noise_std0 is the standard
    deviation of the noise separating target from draft logits at position 0;
    it grows by ``noise_growth`` per position.
    """
    name: str
    B: int
    k: int
    V: int
    d: int = 0
    Hq: int = 0
    Hkv: int = 0
    Dh: int = 0
    F: int = 0
    ctx: object = 16
    T: float = 1.0
    mode: int = GREEDY
    eps: float = 1e-6
    w_std: float = 0.02
    target_std: float = 4.0
    draft_noise_std0: float = 1.0
    noise_growth: float = 1.0
    verify_only: bool = False
    fused: bool = False          # verification from the target's hidden states
    seed: int = 1000
    notes: str = field(default="", compare=False)

    @property
    def ctx_max(self):
        return self.ctx[1] if isinstance(self.ctx, tuple) else self.ctx

    @property
    def Lmax(self):
        return self.ctx_max + self.k


# The five workloads.  Seeds are 1000 + the workload's index.
TINY = Workload(
    "tiny_b1_d64_v1000", B=1, k=3, V=1000, d=64, Hq=2, Hkv=2, Dh=32, F=256, ctx=16,
    T=1.0, mode=GREEDY, target_std=4.0, draft_noise_std0=1.0, seed=1001,
    notes="fp32 master weights N(0,0.02) rounded to bf16 for the GPU; tied embedding/head")
SINGLE_GREEDY = Workload(
    "single_greedy_b1_d4096_v151936_ctx4096", B=1, k=3, V=151936, d=4096, Hq=32, Hkv=8,
    Dh=128, F=12288, ctx=4096, T=1.0, mode=GREEDY, target_std=4.0, seed=1002)
BATCHED_STOCHASTIC = Workload(
    "batched_stochastic_b64_d4096_v151936_ctx1024-8192", B=64, k=3, V=151936, d=4096,
    Hq=32, Hkv=8, Dh=128, F=12288, ctx=(1024, 8192), T=1.0, mode=STOCHASTIC,
    draft_noise_std0=0.75, noise_growth=1.5, seed=1003)
VERIFY_SWEEP = Workload(
    "verify_sweep_b256_v151936", B=256, k=3, V=151936, T=1.0, mode=STOCHASTIC,
    target_std=4.0, draft_noise_std0=1.5, verify_only=True, seed=1004)
DEEP_CHAIN = Workload(
    "deep_chain_b32_k5_d5120_v256000_ctx16384", B=32, k=5, V=256000, d=5120, Hq=40,
    Hkv=8, Dh=128, F=17408, ctx=16384, T=0.7, mode=STOCHASTIC,
    draft_noise_std0=0.75, noise_growth=1.5, seed=1005)

# Verification from the target's hidden states at the batched workload's shape:
# 64 sequences, k = 3 (256 verified positions), hidden 4096, vocabulary 151936.
FUSED_VERIFY = Workload(
    "fused_verify_b64_k3_d4096_v151936", B=64, k=3, V=151936, d=4096, T=1.0, mode=STOCHASTIC,
    draft_noise_std0=0.3, verify_only=True, fused=True, seed=1006)

WORKLOADS = {w.name: w for w in (TINY, SINGLE_GREEDY, BATCHED_STOCHASTIC, VERIFY_SWEEP, DEEP_CHAIN, FUSED_VERIFY)}


def with_k(w, k):
    """The same workload at another draft depth (the verify sweep runs k = 1..5)."""
    return replace(w, k=k, name="%s_k%d" % (w.name.split("_k")[0], k))


# ----------------------------------------------------------------------------
# random streams

def _stream(seed, name, chunk):
    ss = np.random.SeedSequence(entropy=seed, spawn_key=(zlib.crc32(name.encode()), chunk))
    return np.random.Generator(np.random.PCG64(ss))


def _fill(seed, name, n, draw):
    """Fill n values chunk by chunk, each chunk from its own stream."""
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def work(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        out[lo:hi] = draw(_stream(seed, name, c), hi - lo)

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(max_workers=8) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def normal(seed, name, shape, std=1.0, mean=0.0):
    """float32 N(mean, std^2) of the given shape."""
    n = int(np.prod(shape))
    x = _fill(seed, name, n, lambda g, m: g.standard_normal(m, dtype=np.float32))
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return x.reshape(shape)


def uniform(seed, name, shape):
    """float32 U[0, 1) of the given shape."""
    n = int(np.prod(shape))
    return _fill(seed, name, n, lambda g, m: g.random(m, dtype=np.float32)).reshape(shape)


def integers(seed, name, shape, lo, hi):
    """int32 uniform on the inclusive range [lo, hi]."""
    g = _stream(seed, name, 0)
    return g.integers(lo, hi + 1, size=shape, dtype=np.int64).astype(np.int32)


def to_bf16_bits(x):
    """float32 -> bf16 bit patterns (round to nearest even), via torch's cast."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------------------------
# workload pieces

WEIGHT_NAMES = ("E", "fc", "wq", "wk", "wv", "wo", "wgate", "wup", "wdown")
GAIN_NAMES = ("g_emb", "g_hid", "g_attn", "g_mlp", "g_final")


def weight_shapes(w):
    d, Hq, Hkv, Dh, F, V = w.d, w.Hq, w.Hkv, w.Dh, w.F, w.V
    return {
        "E": (V, d), "fc": (d, 2 * d), "wq": (Hq * Dh, d), "wk": (Hkv * Dh, d),
        "wv": (Hkv * Dh, d), "wo": (d, Hq * Dh), "wgate": (F, d), "wup": (F, d),
        "wdown": (d, F),
    }


def make_weights(w, master=False):
    """Weights of the draft module: matrices N(0, w_std^2), gains 1 + N(0, w_std^2).

    Returns a dict of bf16 bit arrays; with master=True also a dict of the
    float32 values they were rounded from.
    """
    bits, full = {}, {}
    for name, shape in weight_shapes(w).items():
        x = normal(w.seed, "w." + name, shape, std=w.w_std)
        bits[name] = to_bf16_bits(x)
        if master:
            full[name] = x
    for name in GAIN_NAMES:
        x = normal(w.seed, "w." + name, (w.d,), std=w.w_std, mean=1.0)
        bits[name] = to_bf16_bits(x)
        if master:
            full[name] = x
    return (bits, full) if master else bits


def make_module_weights(w, m, E=None):
    """Weights of module m of a chain of distinct modules, as bf16 bits.

    Module 0 is make_weights' module.  Module m >= 1 draws its own input
    projection, block and gains from streams named "w<m>.<name>"; the embedding
    and vocabulary head E is shared, so every module returns module 0's E (drawn
    again unless the caller passes it in).
    """
    if m == 0:
        return make_weights(w)
    if E is None:
        E = to_bf16_bits(normal(w.seed, "w.E", weight_shapes(w)["E"], std=w.w_std))
    bits = {"E": E}
    for name, shape in weight_shapes(w).items():
        if name != "E":
            bits[name] = to_bf16_bits(normal(w.seed, "w%d.%s" % (m, name), shape, std=w.w_std))
    for name in GAIN_NAMES:
        bits[name] = to_bf16_bits(normal(w.seed, "w%d.%s" % (m, name), (w.d,), std=w.w_std, mean=1.0))
    return bits


def make_draft_vocab(w, n):
    """A reduced draft vocabulary of n distinct ids in [0, V), in a seeded random
    order (the order of the draft head's rows), and the head: those rows of E,
    as bf16 bits.  Stands in for FR-Spec's most frequent tokens: synthetic
    weights have no token frequencies."""
    g = _stream(w.seed, "draft_vocab", 0)
    vmap = g.permutation(w.V)[:n].astype(np.int32)
    E = to_bf16_bits(normal(w.seed, "w.E", weight_shapes(w)["E"], std=w.w_std))
    return vmap, np.ascontiguousarray(E[vmap])


def make_module_cache(w, m):
    """K/V caches [B, Hkv, Lmax, Dh] bf16 N(0,1) of module m (m = 0: make_context's)."""
    shape = (w.B, w.Hkv, w.Lmax, w.Dh)
    suffix = "" if m == 0 else str(m)
    return (to_bf16_bits(normal(w.seed, "k_cache" + suffix, shape)),
            to_bf16_bits(normal(w.seed, "v_cache" + suffix, shape)))


def make_context(w):
    """Per-step inputs of the drafter.

    h [B,d] bf16 N(0,1); last_tok [B] int32; ctx_len [B] int32; the K and V
    caches [B, Hkv, Lmax, Dh] bf16 N(0,1) (every row random, including the rows
    past each sequence's context, which the kernels must never read).
    """
    B = w.B
    if isinstance(w.ctx, tuple):
        ctx_len = integers(w.seed, "ctx_len", (B,), w.ctx[0], w.ctx[1])
    else:
        ctx_len = np.full((B,), w.ctx, dtype=np.int32)
    shape = (B, w.Hkv, w.Lmax, w.Dh)
    return {
        "h": to_bf16_bits(normal(w.seed, "h", (B, w.d))),
        "last_tok": integers(w.seed, "last_tok", (B,), 0, w.V - 1),
        "ctx_len": ctx_len,
        "k_cache": to_bf16_bits(normal(w.seed, "k_cache", shape)),
        "v_cache": to_bf16_bits(normal(w.seed, "v_cache", shape)),
    }


def make_uniforms(w):
    """u_draft [B,k], u_accept [B,k], u_final [B]: float32 U[0,1)."""
    return {
        "u_draft": uniform(w.seed, "u_draft", (w.B, w.k)),
        "u_accept": uniform(w.seed, "u_accept", (w.B, w.k)),
        "u_final": uniform(w.seed, "u_final", (w.B,)),
    }


def target_logits(w):
    """Target logits [B, k+1, V] float32 N(0, target_std^2), independent of the draft."""
    return normal(w.seed, "target", (w.B, w.k + 1, w.V), std=w.target_std)


def draft_noise(w, positions):
    """Noise [B, positions, V] float32; position j has std draft_noise_std0 * growth^j."""
    z = normal(w.seed, "noise", (w.B, positions, w.V))
    for j in range(positions):
        z[:, j] *= np.float32(w.draft_noise_std0 * (w.noise_growth ** j))
    return z


def fused_inputs(w):
    """Inputs of a verification from hidden states: head [V, d] bf16 N(0, w_std^2)
    (the shared embedding of this seed), hidden [B, k+1, d] bf16 N(0, 1), the
    draft's noise [B, k, V] float32 N(0, draft_noise_std0^2) and the uniforms.
    The consumer forms draft = head . hidden + noise for the k draft
    positions, and draws the draft tokens from q."""
    out = {"head": to_bf16_bits(normal(w.seed, "w.E", (w.V, w.d), std=w.w_std)),
           "hidden": to_bf16_bits(normal(w.seed, "hidden_target", (w.B, w.k + 1, w.d))),
           "noise": normal(w.seed, "noise", (w.B, w.k, w.V), std=w.draft_noise_std0)}
    out.update(make_uniforms(w))
    return out


def verify_inputs(w):
    """Verify-only workload: target ~ N(0, target_std^2), draft = target + noise.

    Returns target [B,k+1,V], draft [B,k,V] float32 and the uniforms.  Draft
    tokens are not drawn here: choosing them from the draft distribution is part
    of the method and is done by whoever consumes these inputs.
    """
    t = target_logits(w)
    dl = t[:, :w.k] + draft_noise(w, w.k)
    out = {"target_logits": t, "draft_logits": dl}
    out.update(make_uniforms(w))
    return out
