"""ctypes binding of libmtpspec (include/mtpspec.h).

Argument marshalling only: every step of the path runs in the CUDA library.
Tensors are torch CUDA tensors; their device pointers are passed through the
C ABI unchanged.  If the library is missing or cannot be loaded this module
raises: there is no fallback implementation.
"""

import ctypes
import os

import torch

from .build import library_path

GREEDY = 0
STOCHASTIC = 1

KC_LMHEAD, KC_VERIFY, KC_ATTN, KC_GEMV = 0, 1, 2, 3

STATUS_TIMEOUT = 1
STATUS_BAD_TOKEN = 2
STATUS_BAD_CTX = 4
STATUS_NONFINITE = 8
STATUS_BOUNDS = 16


class MtpError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (what, _lib().mtp_error_string(code).decode(), code))


class MtpDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("d", ctypes.c_int32), ("Hq", ctypes.c_int32),
                ("Hkv", ctypes.c_int32), ("Dh", ctypes.c_int32), ("F", ctypes.c_int32),
                ("V", ctypes.c_int32), ("Lmax", ctypes.c_int32), ("rms_eps", ctypes.c_float)]


WEIGHT_FIELDS = ("E", "fc", "wq", "wk", "wv", "wo", "wgate", "wup", "wdown",
                 "g_emb", "g_hid", "g_attn", "g_mlp", "g_final")


class MtpWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


class MtpModule(ctypes.Structure):
    _fields_ = [("w", MtpWeights), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p)]


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        lib = library_path()
        if not os.path.exists(lib):
            raise RuntimeError("%s is not built; run __graft_entry__.build() (or build(variant=...) for "
                               "MTP_LIB_VARIANT)" % lib)
        L = ctypes.CDLL(lib)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.mtp_workspace_size.argtypes = [ctypes.POINTER(MtpDims), I]
        L.mtp_workspace_size.restype = Z
        L.mtp_draft.argtypes = [ctypes.POINTER(MtpDims), ctypes.POINTER(MtpWeights), P, P, P, P, P, I, F, I,
                                P, P, P, P, Z, P]
        L.mtp_draft.restype = I
        L.mtp_draft_noalloc.argtypes = [ctypes.POINTER(MtpDims), ctypes.POINTER(MtpWeights), P, P, P, P, P, I,
                                        F, I, P, P, P, P, P]
        L.mtp_draft_noalloc.restype = I
        L.spec_verify_workspace_size.argtypes = [I, I, I]
        L.spec_verify_workspace_size.restype = Z
        L.spec_verify.argtypes = [I, I, I, F, I, P, P, P, P, P, P, P, P, P, Z, P]
        L.spec_verify.restype = I
        L.spec_step.argtypes = [ctypes.POINTER(MtpDims), ctypes.POINTER(MtpWeights), P, P, P, P, P, I, F, I,
                                P, P, P, P, P, P, P, P, P, P, Z, P]
        L.spec_step.restype = I
        L.mtp_draft_modules.argtypes = [ctypes.POINTER(MtpDims), ctypes.POINTER(MtpModule), I, P, P, P, I, F, I,
                                        P, P, P, P, Z, P]
        L.mtp_draft_modules.restype = I
        L.spec_step_modules.argtypes = [ctypes.POINTER(MtpDims), ctypes.POINTER(MtpModule), I, P, P, P, I, F, I,
                                        P, P, P, P, P, P, P, P, P, P, Z, P]
        L.spec_step_modules.restype = I
        L.mtp_draft_dynamic.argtypes = [ctypes.POINTER(MtpDims), ctypes.POINTER(MtpWeights), P, P, P, P, P, I, F,
                                        I, F, P, P, P, P, P, Z, P]
        L.mtp_draft_dynamic.restype = I
        L.spec_verify_dynamic.argtypes = [I, I, I, F, I, P, P, P, P, P, P, P, P, P, P, Z, P]
        L.spec_verify_dynamic.restype = I
        L.spec_step_dynamic.argtypes = [ctypes.POINTER(MtpDims), ctypes.POINTER(MtpWeights), P, P, P, P, P, I, F,
                                        I, F, P, P, P, P, P, P, P, P, P, P, P, Z, P]
        L.spec_step_dynamic.restype = I
        L.mtp_draft_reduced.argtypes = [ctypes.POINTER(MtpDims), ctypes.POINTER(MtpWeights), P, P, I, P, P, P, P,
                                        P, I, F, I, P, P, P, P, Z, P]
        L.mtp_draft_reduced.restype = I
        L.spec_step_reduced.argtypes = [ctypes.POINTER(MtpDims), ctypes.POINTER(MtpWeights), P, P, I, P, P, P, P,
                                        P, I, F, I, P, P, P, P, P, P, P, P, P, P, Z, P]
        L.spec_step_reduced.restype = I
        L.spec_verify_fused_workspace_size.argtypes = [I, I, I, I, I]
        L.spec_verify_fused_workspace_size.restype = Z
        L.spec_verify_fused.argtypes = [I, I, I, I, F, I, P, P, P, P, P, P, P, P, P, P, Z, P]
        L.spec_verify_fused.restype = I
        L.mtp_get_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_int32)]
        L.mtp_get_status.restype = I
        L.mtp_clear_status.argtypes = [P, P]
        L.mtp_clear_status.restype = I
        L.mtp_selftest_wait_timeout.argtypes = [P, P]
        L.mtp_selftest_wait_timeout.restype = I
        L.mtp_error_string.argtypes = [I]
        L.mtp_error_string.restype = ctypes.c_char_p
        L.mtp_profiler_enable.argtypes = [I]
        L.mtp_profiler_enable.restype = I
        L.mtp_profiler_read.argtypes = [I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)]
        L.mtp_profiler_read.restype = I
        L.mtp_launch_count.argtypes = []
        L.mtp_launch_count.restype = ctypes.c_int64
        L.mtp_trace_read.argtypes = [P, I]
        L.mtp_trace_read.restype = I
        _LIB = L
    return _LIB


def library():
    """The loaded ctypes library (loads it on first use)."""
    return _lib()


def _ptr(t, name, dtype=None, numel=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if numel is not None and t.numel() < numel:
        raise ValueError("%s has %d elements, needs %d" % (name, t.numel(), numel))
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def make_dims(B, d, Hq, Hkv, Dh, F, V, Lmax, eps=1e-6):
    return MtpDims(B, d, Hq, Hkv, Dh, F, V, Lmax, eps)


def make_weights(w):
    """MtpWeights from a dict of bf16 CUDA tensors keyed by WEIGHT_FIELDS."""
    return MtpWeights(*[_ptr(w[n], n, torch.bfloat16) for n in WEIGHT_FIELDS])


def make_modules(modules):
    """A ctypes array of MtpModule from (weights dict, k_cache, v_cache) triples;
    the caches are bf16 CUDA tensors [B, Hkv, Lmax, Dh]."""
    arr = (MtpModule * len(modules))()
    for i, (w, kc, vc) in enumerate(modules):
        arr[i] = MtpModule(make_weights(w), _ptr(kc, "k_cache", torch.bfloat16),
                           _ptr(vc, "v_cache", torch.bfloat16))
    return arr


def workspace_size(dims, k):
    return int(_lib().mtp_workspace_size(ctypes.byref(dims), int(k)))


def verify_workspace_size(B, k, V):
    return int(_lib().spec_verify_workspace_size(int(B), int(k), int(V)))


def alloc_workspace(nbytes, device=None):
    """A 256-byte aligned uint8 CUDA buffer of at least nbytes."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def mtp_draft(dims, weights, h, last_tok, k_cache, v_cache, ctx_len, k, T, mode, u_draft,
              draft_tok, draft_logits, ws, stream=None):
    B, V = dims.B, dims.V
    rc = _lib().mtp_draft(
        ctypes.byref(dims), ctypes.byref(weights), _ptr(h, "h", torch.bfloat16, B * dims.d),
        _ptr(last_tok, "last_tok", torch.int32, B), _ptr(k_cache, "k_cache", torch.bfloat16),
        _ptr(v_cache, "v_cache", torch.bfloat16), _ptr(ctx_len, "ctx_len", torch.int32, B), int(k),
        float(T), int(mode), _ptr(u_draft, "u_draft", torch.float32, B * k),
        _ptr(draft_tok, "draft_tok", torch.int32, B * k),
        _ptr(draft_logits, "draft_logits", torch.float32, B * k * V),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream))
    if rc != 0:
        raise MtpError(rc, "mtp_draft")


def mtp_draft_noalloc(dims, weights, h, last_tok, k_cache, v_cache, ctx_len, k, T, mode, u_draft,
                      draft_tok, draft_logits, status=None, stream=None):
    """mtp_draft on the library's static scratch (no workspace argument)."""
    B, V = dims.B, dims.V
    rc = _lib().mtp_draft_noalloc(
        ctypes.byref(dims), ctypes.byref(weights), _ptr(h, "h", torch.bfloat16, B * dims.d),
        _ptr(last_tok, "last_tok", torch.int32, B), _ptr(k_cache, "k_cache", torch.bfloat16),
        _ptr(v_cache, "v_cache", torch.bfloat16), _ptr(ctx_len, "ctx_len", torch.int32, B), int(k),
        float(T), int(mode), _ptr(u_draft, "u_draft", torch.float32, B * k),
        _ptr(draft_tok, "draft_tok", torch.int32, B * k),
        _ptr(draft_logits, "draft_logits", torch.float32, B * k * V),
        _ptr(status, "status", torch.int32, 1), _stream(stream))
    if rc != 0:
        raise MtpError(rc, "mtp_draft_noalloc")


def spec_verify(B, k, V, T, mode, target_logits, draft_logits, draft_tok, u_accept, u_final,
                out_tok, accept_len, num_accepted, ws, stream=None):
    rc = _lib().spec_verify(
        int(B), int(k), int(V), float(T), int(mode),
        _ptr(target_logits, "target_logits", torch.float32, B * (k + 1) * V),
        _ptr(draft_logits, "draft_logits", torch.float32, B * k * V),
        _ptr(draft_tok, "draft_tok", torch.int32, B * k),
        _ptr(u_accept, "u_accept", torch.float32, B * k), _ptr(u_final, "u_final", torch.float32, B),
        _ptr(out_tok, "out_tok", torch.int32, B * (k + 1)), _ptr(accept_len, "accept_len", torch.int32, B),
        _ptr(num_accepted, "num_accepted", torch.int32, B),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream))
    if rc != 0:
        raise MtpError(rc, "spec_verify")


def spec_step(dims, weights, h, last_tok, k_cache, v_cache, ctx_len, k, T, mode, u_draft,
              target_logits, u_accept, u_final, draft_tok, draft_logits, out_tok, accept_len,
              num_accepted, ws, stream=None):
    B, V = dims.B, dims.V
    rc = _lib().spec_step(
        ctypes.byref(dims), ctypes.byref(weights), _ptr(h, "h", torch.bfloat16, B * dims.d),
        _ptr(last_tok, "last_tok", torch.int32, B), _ptr(k_cache, "k_cache", torch.bfloat16),
        _ptr(v_cache, "v_cache", torch.bfloat16), _ptr(ctx_len, "ctx_len", torch.int32, B), int(k),
        float(T), int(mode), _ptr(u_draft, "u_draft", torch.float32, B * k),
        _ptr(target_logits, "target_logits", torch.float32, B * (k + 1) * V),
        _ptr(u_accept, "u_accept", torch.float32, B * k), _ptr(u_final, "u_final", torch.float32, B),
        _ptr(draft_tok, "draft_tok", torch.int32, B * k),
        _ptr(draft_logits, "draft_logits", torch.float32, B * k * V),
        _ptr(out_tok, "out_tok", torch.int32, B * (k + 1)), _ptr(accept_len, "accept_len", torch.int32, B),
        _ptr(num_accepted, "num_accepted", torch.int32, B),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream))
    if rc != 0:
        raise MtpError(rc, "spec_step")


def mtp_draft_modules(dims, modules, h, last_tok, ctx_len, k, T, mode, u_draft, draft_tok, draft_logits,
                      ws, stream=None):
    """mtp_draft over distinct modules: `modules` from make_modules(); depth j
    runs module min(j, len(modules) - 1)."""
    B, V = dims.B, dims.V
    rc = _lib().mtp_draft_modules(
        ctypes.byref(dims), modules, len(modules), _ptr(h, "h", torch.bfloat16, B * dims.d),
        _ptr(last_tok, "last_tok", torch.int32, B), _ptr(ctx_len, "ctx_len", torch.int32, B), int(k),
        float(T), int(mode), _ptr(u_draft, "u_draft", torch.float32, B * k),
        _ptr(draft_tok, "draft_tok", torch.int32, B * k),
        _ptr(draft_logits, "draft_logits", torch.float32, B * k * V),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream))
    if rc != 0:
        raise MtpError(rc, "mtp_draft_modules")


def spec_step_modules(dims, modules, h, last_tok, ctx_len, k, T, mode, u_draft, target_logits, u_accept,
                      u_final, draft_tok, draft_logits, out_tok, accept_len, num_accepted, ws, stream=None):
    """spec_step over distinct modules (see mtp_draft_modules)."""
    B, V = dims.B, dims.V
    rc = _lib().spec_step_modules(
        ctypes.byref(dims), modules, len(modules), _ptr(h, "h", torch.bfloat16, B * dims.d),
        _ptr(last_tok, "last_tok", torch.int32, B), _ptr(ctx_len, "ctx_len", torch.int32, B), int(k),
        float(T), int(mode), _ptr(u_draft, "u_draft", torch.float32, B * k),
        _ptr(target_logits, "target_logits", torch.float32, B * (k + 1) * V),
        _ptr(u_accept, "u_accept", torch.float32, B * k), _ptr(u_final, "u_final", torch.float32, B),
        _ptr(draft_tok, "draft_tok", torch.int32, B * k),
        _ptr(draft_logits, "draft_logits", torch.float32, B * k * V),
        _ptr(out_tok, "out_tok", torch.int32, B * (k + 1)), _ptr(accept_len, "accept_len", torch.int32, B),
        _ptr(num_accepted, "num_accepted", torch.int32, B),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream))
    if rc != 0:
        raise MtpError(rc, "spec_step_modules")


def mtp_draft_dynamic(dims, weights, h, last_tok, k_cache, v_cache, ctx_len, k, T, mode, stop_p, u_draft,
                      draft_tok, draft_logits, k_eff, ws, stream=None):
    """mtp_draft with the dynamic draft length: k_eff [B] int32 receives the
    drafts each sequence keeps (its first depth of confidence below stop_p)."""
    B, V = dims.B, dims.V
    rc = _lib().mtp_draft_dynamic(
        ctypes.byref(dims), ctypes.byref(weights), _ptr(h, "h", torch.bfloat16, B * dims.d),
        _ptr(last_tok, "last_tok", torch.int32, B), _ptr(k_cache, "k_cache", torch.bfloat16),
        _ptr(v_cache, "v_cache", torch.bfloat16), _ptr(ctx_len, "ctx_len", torch.int32, B), int(k),
        float(T), int(mode), float(stop_p), _ptr(u_draft, "u_draft", torch.float32, B * k),
        _ptr(draft_tok, "draft_tok", torch.int32, B * k),
        _ptr(draft_logits, "draft_logits", torch.float32, B * k * V), _ptr(k_eff, "k_eff", torch.int32, B),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream))
    if rc != 0:
        raise MtpError(rc, "mtp_draft_dynamic")


def spec_verify_dynamic(B, k, V, T, mode, target_logits, draft_logits, draft_tok, k_eff, u_accept, u_final,
                        out_tok, accept_len, num_accepted, ws, stream=None):
    """spec_verify over each sequence's kept drafts (k_eff [B] int32, or None for k)."""
    rc = _lib().spec_verify_dynamic(
        int(B), int(k), int(V), float(T), int(mode),
        _ptr(target_logits, "target_logits", torch.float32, B * (k + 1) * V),
        _ptr(draft_logits, "draft_logits", torch.float32, B * k * V),
        _ptr(draft_tok, "draft_tok", torch.int32, B * k), _ptr(k_eff, "k_eff", torch.int32, B),
        _ptr(u_accept, "u_accept", torch.float32, B * k), _ptr(u_final, "u_final", torch.float32, B),
        _ptr(out_tok, "out_tok", torch.int32, B * (k + 1)), _ptr(accept_len, "accept_len", torch.int32, B),
        _ptr(num_accepted, "num_accepted", torch.int32, B),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream))
    if rc != 0:
        raise MtpError(rc, "spec_verify_dynamic")


def spec_step_dynamic(dims, weights, h, last_tok, k_cache, v_cache, ctx_len, k, T, mode, stop_p, u_draft,
                      target_logits, u_accept, u_final, draft_tok, draft_logits, k_eff, out_tok, accept_len,
                      num_accepted, ws, stream=None):
    """spec_step with the dynamic draft length (see mtp_draft_dynamic)."""
    B, V = dims.B, dims.V
    rc = _lib().spec_step_dynamic(
        ctypes.byref(dims), ctypes.byref(weights), _ptr(h, "h", torch.bfloat16, B * dims.d),
        _ptr(last_tok, "last_tok", torch.int32, B), _ptr(k_cache, "k_cache", torch.bfloat16),
        _ptr(v_cache, "v_cache", torch.bfloat16), _ptr(ctx_len, "ctx_len", torch.int32, B), int(k),
        float(T), int(mode), float(stop_p), _ptr(u_draft, "u_draft", torch.float32, B * k),
        _ptr(target_logits, "target_logits", torch.float32, B * (k + 1) * V),
        _ptr(u_accept, "u_accept", torch.float32, B * k), _ptr(u_final, "u_final", torch.float32, B),
        _ptr(draft_tok, "draft_tok", torch.int32, B * k),
        _ptr(draft_logits, "draft_logits", torch.float32, B * k * V), _ptr(k_eff, "k_eff", torch.int32, B),
        _ptr(out_tok, "out_tok", torch.int32, B * (k + 1)), _ptr(accept_len, "accept_len", torch.int32, B),
        _ptr(num_accepted, "num_accepted", torch.int32, B),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream))
    if rc != 0:
        raise MtpError(rc, "spec_step_dynamic")


def mtp_draft_reduced(dims, weights, head_rows, vocab_map, h, last_tok, k_cache, v_cache, ctx_len, k, T, mode,
                      u_draft, draft_tok, draft_logits, ws, stream=None):
    """mtp_draft over a reduced draft vocabulary: head_rows [N, d] bf16 (rows
    vocab_map of E), vocab_map [N] int32."""
    B, V, N = dims.B, dims.V, int(vocab_map.numel())
    rc = _lib().mtp_draft_reduced(
        ctypes.byref(dims), ctypes.byref(weights), _ptr(head_rows, "head_rows", torch.bfloat16, N * dims.d),
        _ptr(vocab_map, "vocab_map", torch.int32, N), N, _ptr(h, "h", torch.bfloat16, B * dims.d),
        _ptr(last_tok, "last_tok", torch.int32, B), _ptr(k_cache, "k_cache", torch.bfloat16),
        _ptr(v_cache, "v_cache", torch.bfloat16), _ptr(ctx_len, "ctx_len", torch.int32, B), int(k),
        float(T), int(mode), _ptr(u_draft, "u_draft", torch.float32, B * k),
        _ptr(draft_tok, "draft_tok", torch.int32, B * k),
        _ptr(draft_logits, "draft_logits", torch.float32, B * k * V),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream))
    if rc != 0:
        raise MtpError(rc, "mtp_draft_reduced")


def spec_step_reduced(dims, weights, head_rows, vocab_map, h, last_tok, k_cache, v_cache, ctx_len, k, T, mode,
                      u_draft, target_logits, u_accept, u_final, draft_tok, draft_logits, out_tok, accept_len,
                      num_accepted, ws, stream=None):
    """spec_step over a reduced draft vocabulary (see mtp_draft_reduced)."""
    B, V, N = dims.B, dims.V, int(vocab_map.numel())
    rc = _lib().spec_step_reduced(
        ctypes.byref(dims), ctypes.byref(weights), _ptr(head_rows, "head_rows", torch.bfloat16, N * dims.d),
        _ptr(vocab_map, "vocab_map", torch.int32, N), N, _ptr(h, "h", torch.bfloat16, B * dims.d),
        _ptr(last_tok, "last_tok", torch.int32, B), _ptr(k_cache, "k_cache", torch.bfloat16),
        _ptr(v_cache, "v_cache", torch.bfloat16), _ptr(ctx_len, "ctx_len", torch.int32, B), int(k),
        float(T), int(mode), _ptr(u_draft, "u_draft", torch.float32, B * k),
        _ptr(target_logits, "target_logits", torch.float32, B * (k + 1) * V),
        _ptr(u_accept, "u_accept", torch.float32, B * k), _ptr(u_final, "u_final", torch.float32, B),
        _ptr(draft_tok, "draft_tok", torch.int32, B * k),
        _ptr(draft_logits, "draft_logits", torch.float32, B * k * V),
        _ptr(out_tok, "out_tok", torch.int32, B * (k + 1)), _ptr(accept_len, "accept_len", torch.int32, B),
        _ptr(num_accepted, "num_accepted", torch.int32, B),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream))
    if rc != 0:
        raise MtpError(rc, "spec_step_reduced")


def fused_workspace_size(B, k, V, d, mode):
    return int(_lib().spec_verify_fused_workspace_size(int(B), int(k), int(V), int(d), int(mode)))


def spec_verify_fused(B, k, V, d, T, mode, head, target_hidden, draft_logits, draft_tok, u_accept, u_final,
                      out_tok, accept_len, num_accepted, ws, stream=None):
    """spec_verify from the target's hidden states: head [V, d] bf16 (the
    target's vocabulary head) and target_hidden [B, k+1, d] bf16 (what the head
    consumes at each position) instead of target logits."""
    rc = _lib().spec_verify_fused(
        int(B), int(k), int(V), int(d), float(T), int(mode), _ptr(head, "head", torch.bfloat16, V * d),
        _ptr(target_hidden, "target_hidden", torch.bfloat16, B * (k + 1) * d),
        _ptr(draft_logits, "draft_logits", torch.float32, B * k * V),
        _ptr(draft_tok, "draft_tok", torch.int32, B * k),
        _ptr(u_accept, "u_accept", torch.float32, B * k), _ptr(u_final, "u_final", torch.float32, B),
        _ptr(out_tok, "out_tok", torch.int32, B * (k + 1)), _ptr(accept_len, "accept_len", torch.int32, B),
        _ptr(num_accepted, "num_accepted", torch.int32, B),
        _ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream))
    if rc != 0:
        raise MtpError(rc, "spec_verify_fused")


def get_status(ws, stream=None):
    v = ctypes.c_int32(0)
    rc = _lib().mtp_get_status(_ptr(ws, "ws"), _stream(stream), ctypes.byref(v))
    if rc != 0:
        raise MtpError(rc, "mtp_get_status")
    return int(v.value)


def clear_status(ws, stream=None):
    rc = _lib().mtp_clear_status(_ptr(ws, "ws"), _stream(stream))
    if rc != 0:
        raise MtpError(rc, "mtp_clear_status")


def selftest_wait_timeout(status, stream=None):
    """Run the library's bounded waits on a phase nothing completes: they give
    up after the wait limit and OR MTP_STATUS_TIMEOUT into status (device int32)."""
    rc = _lib().mtp_selftest_wait_timeout(_ptr(status, "status", torch.int32, 1), _stream(stream))
    if rc != 0:
        raise MtpError(rc, "mtp_selftest_wait_timeout")


def profiler_enable(on=True):
    _lib().mtp_profiler_enable(1 if on else 0)


def profiler_read(kernel_class):
    ms = ctypes.c_double(0.0)
    n = ctypes.c_int64(0)
    rc = _lib().mtp_profiler_read(int(kernel_class), ctypes.byref(ms), ctypes.byref(n))
    if rc != 0:
        raise MtpError(rc, "mtp_profiler_read")
    return float(ms.value), int(n.value)


def launch_count():
    return int(_lib().mtp_launch_count())


class MtpTraceEntry(ctypes.Structure):
    _fields_ = [("launch", ctypes.c_uint64), ("kind", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("t_start_ns", ctypes.c_uint64), ("t_dep_ns", ctypes.c_uint64), ("t_end_ns", ctypes.c_uint64),
                ("t_mark_ns", ctypes.c_uint64 * 4)]


TRACE_KIND_NAMES = {0: "gemv input projection", 1: "gemv QKV", 2: "gemv output projection", 3: "gemv gate/up",
                    4: "gemv down", 5: "gemv LM head", 10: "attention", 11: "attention (tensor cores)",
                    20: "verify (cluster)", 21: "verify (ticketed)", 30: "tc GEMM", 31: "tc prologue/select",
                    40: "fused verify GEMM", 41: "fused verify aux (stats, decisions, draws)", 50: "chain"}


def trace_read(max_entries=16384):
    """The launch-trace records since the last read (library built with
    MTP_TRACE), as dicts sorted by start time.  Call after synchronising."""
    buf = (MtpTraceEntry * max_entries)()
    n = _lib().mtp_trace_read(ctypes.cast(buf, ctypes.c_void_p), max_entries)
    if n < 0:
        raise MtpError(n, "mtp_trace_read")
    out = [dict(launch=e.launch, kind=e.kind, name=TRACE_KIND_NAMES.get(e.kind, str(e.kind)),
                start=e.t_start_ns, dep=e.t_dep_ns, end=e.t_end_ns, marks=list(e.t_mark_ns)) for e in buf[:n]]
    return sorted(out, key=lambda r: r["start"])
