"""Device-resident inputs, outputs and workspace for one workload.

Holds torch CUDA tensors only (PyTorch is used for device memory and streams)
and forwards every computation to the C-ABI calls in ``binding``.
"""

import numpy as np
import torch

from . import binding as bd


def to_device_bf16(bits, device="cuda"):
    """bf16 bit patterns (numpy uint16) -> torch.bfloat16 CUDA tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_device(x, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


CANARY_BYTES = 4096
CANARY_BYTE = 0xA5


class Guarded:
    """Device buffers with CANARY_BYTES of a fixed byte pattern on both sides.

    alloc() returns the usable (zeroed, contiguous) middle part; check() raises
    if any kernel wrote into a guard band.  The middle starts CANARY_BYTES past
    the allocation, so it keeps the allocation's 256-byte alignment."""

    def __init__(self, device="cuda"):
        self.device = device
        self.bufs = []

    def alloc(self, name, numel, dtype):
        es = torch.empty(0, dtype=dtype).element_size()
        pad = CANARY_BYTES // es
        buf = torch.empty(int(numel) + 2 * pad, dtype=dtype, device=self.device)
        buf.view(torch.uint8).fill_(CANARY_BYTE)
        mid = buf[pad:pad + int(numel)]
        mid.zero_()
        self.bufs.append((name, buf, pad, int(numel)))
        return mid

    def check(self):
        for name, buf, pad, n in self.bufs:
            raw = buf.view(torch.uint8)
            nb = pad * buf.element_size()
            head = raw[:nb]
            tail = raw[raw.numel() - nb:]
            bad_h = int((head != CANARY_BYTE).sum().item())
            bad_t = int((tail != CANARY_BYTE).sum().item())
            if bad_h or bad_t:
                raise AssertionError("%s: %d bytes written before and %d after the buffer" % (name, bad_h, bad_t))


class DraftModule:
    """The MTP module's weights on the device plus the per-step buffers.

    extra_modules: weights (bf16 bits) of further distinct modules for depths 1,
    2, ... (the chain then runs mtp_draft_modules / spec_step_modules); their E
    is not uploaded again, every module uses this one's.
    """

    def __init__(self, w, weights_bits, device="cuda", k=None, extra_modules=()):
        self.w = w
        self.k = w.k if k is None else k
        self.device = device
        self.weights = {n: to_device_bf16(weights_bits[n], device) for n in bd.WEIGHT_FIELDS}
        self.extra = []
        for bits in extra_modules:
            wd = {n: to_device_bf16(bits[n], device) for n in bd.WEIGHT_FIELDS if n != "E"}
            wd["E"] = self.weights["E"]
            self.extra.append(wd)
        self.mods = None
        self.dims = bd.make_dims(w.B, w.d, w.Hq, w.Hkv, w.Dh, w.F, w.V, w.ctx_max + self.k, w.eps)
        self.wptr = bd.make_weights(self.weights)
        # outputs and workspace inside canary bands (check_canaries)
        self.guard = Guarded(device)
        g = self.guard
        self.ws = g.alloc("workspace", max(256, bd.workspace_size(self.dims, self.k)), torch.uint8)
        B, k, V = w.B, self.k, w.V
        self.draft_tok = g.alloc("draft_tok", B * k, torch.int32)
        self.draft_logits = g.alloc("draft_logits", B * k * V, torch.float32)
        self.out_tok = g.alloc("out_tok", B * (k + 1), torch.int32)
        self.accept_len = g.alloc("accept_len", B, torch.int32)
        self.num_accepted = g.alloc("num_accepted", B, torch.int32)

    def set_context(self, ctx, extra_caches=()):
        """Upload h, last_tok, ctx_len and the K/V caches (numpy from workloads);
        extra_caches: (k_cache, v_cache) of each extra module."""
        self.h = to_device_bf16(ctx["h"], self.device)
        self.last_tok = to_device(ctx["last_tok"].astype(np.int32), self.device)
        self.ctx_len = to_device(ctx["ctx_len"].astype(np.int32), self.device)
        self.k_cache = to_device_bf16(ctx["k_cache"], self.device)
        self.v_cache = to_device_bf16(ctx["v_cache"], self.device)
        if self.extra:
            if len(extra_caches) != len(self.extra):
                raise ValueError("one (k_cache, v_cache) pair per extra module")
            self.extra_caches = [(to_device_bf16(kc, self.device), to_device_bf16(vc, self.device))
                                 for kc, vc in extra_caches]
            self.mods = bd.make_modules([(self.weights, self.k_cache, self.v_cache)] +
                                        [(wd, kc, vc) for wd, (kc, vc) in zip(self.extra, self.extra_caches)])

    def draft(self, T, mode, u_draft=None, logits=True, stream=None):
        lg = self.draft_logits if logits else None
        if self.mods is not None:
            bd.mtp_draft_modules(self.dims, self.mods, self.h, self.last_tok, self.ctx_len, self.k, T, mode,
                                 u_draft, self.draft_tok, lg, self.ws, stream)
            return
        bd.mtp_draft(self.dims, self.wptr, self.h, self.last_tok, self.k_cache, self.v_cache,
                     self.ctx_len, self.k, T, mode, u_draft, self.draft_tok, lg, self.ws, stream)

    def step(self, T, mode, target_logits, u_draft=None, u_accept=None, u_final=None,
             logits=True, stream=None):
        lg = self.draft_logits if logits else None
        if self.mods is not None:
            bd.spec_step_modules(self.dims, self.mods, self.h, self.last_tok, self.ctx_len, self.k, T, mode,
                                 u_draft, target_logits, u_accept, u_final, self.draft_tok, lg, self.out_tok,
                                 self.accept_len, self.num_accepted, self.ws, stream)
            return
        bd.spec_step(self.dims, self.wptr, self.h, self.last_tok, self.k_cache, self.v_cache,
                     self.ctx_len, self.k, T, mode, u_draft, target_logits, u_accept, u_final,
                     self.draft_tok, lg, self.out_tok, self.accept_len, self.num_accepted, self.ws, stream)

    def step_dynamic(self, T, mode, stop_p, target_logits, u_draft=None, u_accept=None, u_final=None,
                     logits=True, stream=None):
        """spec_step with the dynamic draft length; self.k_eff receives the drafts kept."""
        if not hasattr(self, "k_eff"):
            self.k_eff = self.guard.alloc("k_eff", self.w.B, torch.int32)
        bd.spec_step_dynamic(self.dims, self.wptr, self.h, self.last_tok, self.k_cache, self.v_cache,
                             self.ctx_len, self.k, T, mode, stop_p, u_draft, target_logits, u_accept, u_final,
                             self.draft_tok, self.draft_logits if logits else None, self.k_eff, self.out_tok,
                             self.accept_len, self.num_accepted, self.ws, stream)

    def set_draft_vocab(self, vmap, head_bits):
        """Draft over a reduced vocabulary from now on: vmap [N] ids, head [N, d] bf16 bits."""
        self.vmap = to_device(np.asarray(vmap, dtype=np.int32), self.device)
        self.head = to_device_bf16(head_bits, self.device)

    def step_reduced(self, T, mode, target_logits, u_draft=None, u_accept=None, u_final=None, logits=True,
                     stream=None):
        bd.spec_step_reduced(self.dims, self.wptr, self.head, self.vmap, self.h, self.last_tok, self.k_cache,
                             self.v_cache, self.ctx_len, self.k, T, mode, u_draft, target_logits, u_accept,
                             u_final, self.draft_tok, self.draft_logits if logits else None, self.out_tok,
                             self.accept_len, self.num_accepted, self.ws, stream)

    def status(self, stream=None):
        return bd.get_status(self.ws, stream)

    def check_canaries(self):
        """Raise if any call wrote outside an output or the workspace."""
        torch.cuda.synchronize()
        self.guard.check()


class Verifier:
    """Buffers for spec_verify on B sequences of depth k over V tokens."""

    def __init__(self, B, k, V, device="cuda"):
        self.B, self.k, self.V = B, k, V
        self.guard = Guarded(device)
        g = self.guard
        self.ws = g.alloc("workspace", max(256, bd.verify_workspace_size(B, k, V)), torch.uint8)
        self.out_tok = g.alloc("out_tok", B * (k + 1), torch.int32)
        self.accept_len = g.alloc("accept_len", B, torch.int32)
        self.num_accepted = g.alloc("num_accepted", B, torch.int32)

    def __call__(self, T, mode, target_logits, draft_logits, draft_tok, u_accept=None, u_final=None,
                 stream=None):
        bd.spec_verify(self.B, self.k, self.V, T, mode, target_logits, draft_logits, draft_tok,
                       u_accept, u_final, self.out_tok, self.accept_len, self.num_accepted, self.ws,
                       stream)

    def check_canaries(self):
        torch.cuda.synchronize()
        self.guard.check()

    def results(self):
        torch.cuda.synchronize()
        return (self.out_tok.view(self.B, self.k + 1).cpu().numpy(), self.accept_len.cpu().numpy(),
                self.num_accepted.cpu().numpy())


class FusedVerifier:
    """Buffers for spec_verify_fused on B sequences of depth k over V tokens
    with hidden width d (outputs and workspace inside canary bands)."""

    def __init__(self, B, k, V, d, mode, device="cuda"):
        self.B, self.k, self.V, self.d, self.mode = B, k, V, d, mode
        self.guard = Guarded(device)
        g = self.guard
        self.ws = g.alloc("workspace", max(256, bd.fused_workspace_size(B, k, V, d, mode)), torch.uint8)
        self.out_tok = g.alloc("out_tok", B * (k + 1), torch.int32)
        self.accept_len = g.alloc("accept_len", B, torch.int32)
        self.num_accepted = g.alloc("num_accepted", B, torch.int32)

    def __call__(self, T, head, target_hidden, draft_logits, draft_tok, u_accept=None, u_final=None, stream=None):
        bd.spec_verify_fused(self.B, self.k, self.V, self.d, T, self.mode, head, target_hidden, draft_logits,
                             draft_tok, u_accept, u_final, self.out_tok, self.accept_len, self.num_accepted, self.ws,
                             stream)

    def check_canaries(self):
        torch.cuda.synchronize()
        self.guard.check()

    def results(self):
        torch.cuda.synchronize()
        return (self.out_tok.view(self.B, self.k + 1).cpu().numpy(), self.accept_len.cpu().numpy(),
                self.num_accepted.cpu().numpy())
