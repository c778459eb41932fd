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
        self.ws = bd.alloc_workspace(bd.workspace_size(self.dims, self.k), device)
        B, k, V = w.B, self.k, w.V
        self.draft_tok = torch.zeros(B * k, dtype=torch.int32, device=device)
        self.draft_logits = torch.zeros(B * k * V, dtype=torch.float32, device=device)
        self.out_tok = torch.zeros(B * (k + 1), dtype=torch.int32, device=device)
        self.accept_len = torch.zeros(B, dtype=torch.int32, device=device)
        self.num_accepted = torch.zeros(B, dtype=torch.int32, device=device)

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
            self.k_eff = torch.zeros(self.w.B, dtype=torch.int32, device=self.device)
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


class Verifier:
    """Buffers for spec_verify on B sequences of depth k over V tokens."""

    def __init__(self, B, k, V, device="cuda"):
        self.B, self.k, self.V = B, k, V
        self.ws = bd.alloc_workspace(bd.verify_workspace_size(B, k, V), device)
        self.out_tok = torch.zeros(B * (k + 1), dtype=torch.int32, device=device)
        self.accept_len = torch.zeros(B, dtype=torch.int32, device=device)
        self.num_accepted = torch.zeros(B, dtype=torch.int32, device=device)

    def __call__(self, T, mode, target_logits, draft_logits, draft_tok, u_accept=None, u_final=None,
                 stream=None):
        bd.spec_verify(self.B, self.k, self.V, T, mode, target_logits, draft_logits, draft_tok,
                       u_accept, u_final, self.out_tok, self.accept_len, self.num_accepted, self.ws,
                       stream)

    def results(self):
        torch.cuda.synchronize()
        return (self.out_tok.view(self.B, self.k + 1).cpu().numpy(), self.accept_len.cpu().numpy(),
                self.num_accepted.cpu().numpy())
