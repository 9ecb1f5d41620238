"""Device-side batch holder: the input tensors of one packed batch, its output tensors and
its workspace, with one method that enqueues spec_verify on a stream.

Plumbing only (PyTorch for device memory and copies); all verification work happens in
libspecverify.so through the binding in this package.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import sv_workspace_bytes, spec_verify, spec_verify_lazy, spec_verify_onehot


def _t(a: Optional[np.ndarray], device, dtype=None):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


class DeviceBatch:
    """Inputs, outputs and workspace of one batch, resident on a CUDA device."""

    def __init__(self, *, target_logits, draft_probs, draft_tokens, num_drafts, row_offsets, k_max,
                 temperature, top_k, top_p, presence, frequency, greedy, uniforms, want_pq=True, prior=None):
        self.target_logits = target_logits
        self.draft_probs = draft_probs
        self.draft_tokens = draft_tokens
        self.num_drafts = num_drafts
        self.row_offsets = row_offsets
        self.k_max = int(k_max)
        self.temperature, self.top_k, self.top_p = temperature, top_k, top_p
        self.presence, self.frequency, self.greedy = presence, frequency, greedy
        self.uniforms = uniforms
        self.prior = prior          # None or (prior_offsets, prior_tokens, prior_counts)
        dev = target_logits.device
        R, V = target_logits.shape
        B = num_drafts.numel()
        self.B, self.R, self.V, self.D = B, R, V, R - B
        self.out_tokens = torch.empty((B, self.k_max + 1), dtype=torch.int32, device=dev)
        self.accept_len = torch.empty(B, dtype=torch.int32, device=dev)
        self.out_pq = torch.empty((max(self.D, 0), 2), dtype=torch.float32, device=dev) if want_pq else None
        self.workspace = torch.empty(sv_workspace_bytes(B, R, V), dtype=torch.uint8, device=dev)

    @staticmethod
    def logits_tensor(w_logits: np.ndarray, dtype: str, device) -> torch.Tensor:
        if dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(w_logits).view(np.int16)).to(device).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(w_logits, dtype=np.float32)).to(device)

    @classmethod
    def from_host(cls, w, device="cuda", want_pq=True) -> "DeviceBatch":
        """From a host workload (numpy arrays laid out as the C ABI expects)."""
        return cls(target_logits=cls.logits_tensor(w.target_logits, w.dtype, device),
                   draft_probs=_t(w.draft_probs.reshape(-1, w.V) if w.draft_probs.size else
                                  np.zeros((0, w.V), np.float32), device, torch.float32),
                   draft_tokens=_t(w.draft_tokens, device, torch.int32),
                   num_drafts=_t(w.num_drafts, device, torch.int32),
                   row_offsets=_t(w.row_offsets, device, torch.int32),
                   k_max=w.k_max,
                   temperature=_t(w.temperature, device, torch.float32),
                   top_k=_t(w.top_k, device, torch.int32),
                   top_p=_t(w.top_p, device, torch.float32),
                   presence=_t(w.presence, device, torch.float32),
                   frequency=_t(w.frequency, device, torch.float32),
                   greedy=_t(w.greedy, device, torch.uint8),
                   uniforms=_t(w.uniforms, device, torch.float32), want_pq=want_pq,
                   prior=None if getattr(w, "prior_offsets", None) is None else
                   (_t(w.prior_offsets, device, torch.int32), _t(w.prior_tokens, device, torch.int32),
                    _t(w.prior_counts, device, torch.int32)))

    def run(self, stream=None, target_logits=None, draft_probs=None, onehot=False, lazy=False) -> None:
        """Enqueue one verification (optionally on other copies of the two large inputs).
        onehot=True runs the one-hot-draft scheme, which reads no draft_probs; lazy=True runs
        spec_verify_lazy (no row after a request's first rejection is read)."""
        if onehot:
            spec_verify_onehot(self.target_logits if target_logits is None else target_logits,
                               self.draft_tokens, self.num_drafts, self.row_offsets, self.k_max,
                               self.temperature, self.top_k, self.top_p, self.presence, self.frequency,
                               self.greedy, self.uniforms, self.out_tokens, self.accept_len, self.out_pq,
                               self.workspace, stream, self.prior)
            return
        (spec_verify_lazy if lazy else spec_verify)(
                    self.target_logits if target_logits is None else target_logits,
                    self.draft_probs if draft_probs is None else draft_probs,
                    self.draft_tokens, self.num_drafts, self.row_offsets, self.k_max,
                    self.temperature, self.top_k, self.top_p, self.presence, self.frequency, self.greedy,
                    self.uniforms, self.out_tokens, self.accept_len, self.out_pq, self.workspace, stream,
                    self.prior)

    def results(self) -> dict:
        torch.cuda.synchronize(self.target_logits.device)
        out = dict(out_tokens=self.out_tokens.cpu().numpy(), accept_len=self.accept_len.cpu().numpy())
        if self.out_pq is not None:
            out["pq"] = self.out_pq.cpu().numpy()
        return out


def bound_call(db: "DeviceBatch", stream, target_logits=None, draft_probs=None, onehot=False, lazy=False):
    """A zero-argument callable that enqueues spec_verify (spec_verify_onehot with onehot=True,
    spec_verify_lazy with lazy=True) for `db` with every pointer already marshalled (for tight
    timing loops; argument checks happen once, here)."""
    from . import SV_BF16, SV_F32, SV_OK, SvError, SvParams, lib
    tl = db.target_logits if target_logits is None else target_logits
    dp = db.draft_probs if draft_probs is None else draft_probs
    # one checked call validates shapes and pointers
    if onehot:
        spec_verify_onehot(tl, db.draft_tokens, db.num_drafts, db.row_offsets, db.k_max, db.temperature, db.top_k,
                           db.top_p, db.presence, db.frequency, db.greedy, db.uniforms, db.out_tokens,
                           db.accept_len, db.out_pq, db.workspace, stream, db.prior)
    else:
        (spec_verify_lazy if lazy else spec_verify)(
            tl, dp, db.draft_tokens, db.num_drafts, db.row_offsets, db.k_max, db.temperature, db.top_k, db.top_p,
            db.presence, db.frequency, db.greedy, db.uniforms, db.out_tokens, db.accept_len, db.out_pq,
            db.workspace, stream, db.prior)
    p = lambda t: None if t is None else t.data_ptr()
    ho, ht, hc = db.prior if db.prior is not None else (None, None, None)
    params = SvParams(p(db.temperature), p(db.top_k), p(db.top_p), p(db.presence), p(db.frequency), p(db.greedy),
                      p(ho), p(ht), p(hc), 0 if ht is None else ht.numel())
    head = (p(tl), SV_BF16 if tl.dtype == torch.bfloat16 else SV_F32) + (() if onehot else (p(dp),))
    args = head + (p(db.draft_tokens), p(db.num_drafts), p(db.row_offsets), db.B, db.k_max, db.V, db.R, params,
                   p(db.uniforms), p(db.out_tokens), p(db.accept_len), p(db.out_pq), p(db.workspace),
                   db.workspace.numel(), getattr(stream, "cuda_stream", stream))
    f = lib().spec_verify_onehot if onehot else (lib().spec_verify_lazy if lazy else lib().spec_verify)

    def call():
        st = f(*args)
        if st != SV_OK:
            raise SvError(st, "spec_verify")
    return call
