"""GB300 (sm_103a) batched speculative-decoding verification.

A thin ctypes binding over the C ABI in include/spec_verify.h: every call here marshals
torch tensors (device memory and streams only) into pointers and sizes and calls the CUDA
library libspecverify.so, which does all of the work.  There is no CPU fallback: loading
fails loudly when the library is missing.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libspecverify.so")

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_WORKSPACE, SV_ERR_CUDA, SV_ERR_UNSUPPORTED, SV_ERR_DEVICE_DATA = range(6)
SV_F32, SV_BF16 = 0, 1
DEV_ERRORS = {0: "ok", 1: "bad layout", 2: "bad token", 3: "bad temperature", 4: "bad top_p",
              5: "bad uniform", 6: "bad penalty", 7: "timeout", 8: "bad history"}


class SvParams(C.Structure):
    _fields_ = [("temperature", C.c_void_p), ("top_k", C.c_void_p), ("top_p", C.c_void_p),
                ("presence_penalty", C.c_void_p), ("frequency_penalty", C.c_void_p), ("greedy", C.c_void_p),
                ("prior_offsets", C.c_void_p), ("prior_tokens", C.c_void_p), ("prior_counts", C.c_void_p),
                ("prior_len", C.c_int32)]


class SvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {lib().sv_status_string(status).decode()} (status {status})")
        self.status = status


_lib = None


def lib():
    """The loaded CUDA library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        l = C.CDLL(LIB_PATH)
        l.sv_workspace_bytes.restype = C.c_size_t
        l.sv_workspace_bytes.argtypes = [C.c_int32, C.c_int32, C.c_int32]
        l.spec_verify.restype = C.c_int
        l.spec_verify.argtypes = [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                  C.c_int32, C.c_int32, C.c_int32, C.c_int32, SvParams, C.c_void_p,
                                  C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]
        l.spec_verify_lazy.restype = C.c_int
        l.spec_verify_lazy.argtypes = l.spec_verify.argtypes
        l.spec_verify_onehot.restype = C.c_int
        l.spec_verify_onehot.argtypes = [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p,
                                         C.c_int32, C.c_int32, C.c_int32, C.c_int32, SvParams, C.c_void_p,
                                         C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]
        l.spec_verify_static.restype = C.c_int
        l.spec_verify_static.argtypes = [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                         C.c_int32, C.c_int32, C.c_int32, C.c_int32, SvParams, C.c_void_p,
                                         C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
        l.spec_rollback.restype = C.c_int
        l.spec_rollback.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]
        l.sv_read_device_error.restype = C.c_int
        l.sv_read_device_error.argtypes = [C.c_void_p, C.POINTER(C.c_int32), C.POINTER(C.c_int32)]
        l.sv_set_test_withhold.restype = C.c_int
        l.sv_set_test_withhold.argtypes = [C.c_int32]
        l.sv_set_phase_events.restype = C.c_int
        l.sv_set_phase_events.argtypes = [C.c_void_p, C.c_void_p]
        l.sv_prefer_lazy.restype = C.c_int32
        l.sv_prefer_lazy.argtypes = [C.c_int32, C.c_int32, C.c_int32, C.c_int, C.c_float]
        l.sv_status_string.restype = C.c_char_p
        l.sv_status_string.argtypes = [C.c_int]
        _lib = l
    return _lib


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _check(t, name, dtype=None, numel=None):
    import torch
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")


def sv_workspace_bytes(B: int, total_rows: int, V: int) -> int:
    return int(lib().sv_workspace_bytes(B, total_rows, V))


def sv_prefer_lazy(B: int, total_rows: int, V: int, dtype, row0_reject_share: float) -> bool:
    """Whether spec_verify_lazy is expected to beat spec_verify on this batch, given the expected
    share of requests whose draft 0 is rejected.  dtype: SV_BF16 / SV_F32 or a torch dtype."""
    if not isinstance(dtype, int):
        import torch
        dtype = SV_BF16 if dtype == torch.bfloat16 else SV_F32 if dtype == torch.float32 else -1
    r = int(lib().sv_prefer_lazy(B, total_rows, V, dtype, row0_reject_share))
    if r < 0:
        raise SvError(SV_ERR_INVALID_ARG, "sv_prefer_lazy")
    return r == 1


def _checked_args(target_logits, draft_probs, draft_tokens, num_drafts, row_offsets, k_max, temperature, top_k,
                  top_p, presence_penalty, frequency_penalty, greedy, uniforms, out_tokens, accept_len, out_pq,
                  workspace, prior=None):
    """Checks the tensors of one verify call; returns (dtype code, B, V, R, SvParams).
    prior is None or (prior_offsets [B+1], prior_tokens [H], prior_counts [H]) int32."""
    import torch
    R, V = target_logits.shape
    B = num_drafts.numel()
    D = R - B
    if target_logits.dtype == torch.bfloat16:
        dt = SV_BF16
    elif target_logits.dtype == torch.float32:
        dt = SV_F32
    else:
        raise ValueError("target_logits must be bfloat16 or float32")
    _check(target_logits, "target_logits")
    _check(draft_probs, "draft_probs", torch.float32, D * V)
    _check(draft_tokens, "draft_tokens", torch.int32, D)
    _check(num_drafts, "num_drafts", torch.int32, B)
    _check(row_offsets, "row_offsets", torch.int32, B + 1)
    _check(temperature, "temperature", torch.float32, B)
    _check(top_k, "top_k", torch.int32, B)
    _check(top_p, "top_p", torch.float32, B)
    _check(presence_penalty, "presence_penalty", torch.float32, B)
    _check(frequency_penalty, "frequency_penalty", torch.float32, B)
    _check(greedy, "greedy", torch.uint8, B)
    _check(uniforms, "uniforms", torch.float32, R * 2)
    _check(out_tokens, "out_tokens", torch.int32, B * (k_max + 1))
    _check(accept_len, "accept_len", torch.int32, B)
    _check(out_pq, "out_pq", torch.float32, D * 2)
    _check(workspace, "workspace")
    ho = ht = hc = None
    H = 0
    if prior is not None:
        ho, ht, hc = prior
        H = ht.numel()
        _check(ho, "prior_offsets", torch.int32, B + 1)
        _check(ht, "prior_tokens", torch.int32, H)
        _check(hc, "prior_counts", torch.int32, H)
    params = SvParams(_ptr(temperature), _ptr(top_k), _ptr(top_p), _ptr(presence_penalty),
                      _ptr(frequency_penalty), _ptr(greedy), _ptr(ho), _ptr(ht), _ptr(hc), H)
    return dt, B, V, R, params


def spec_verify(target_logits, draft_probs, draft_tokens, num_drafts, row_offsets, k_max: int,
                temperature, top_k, top_p, presence_penalty, frequency_penalty, greedy, uniforms,
                out_tokens, accept_len, out_pq, workspace, stream=None, prior=None) -> None:
    """Verify a batch of drafts (see include/spec_verify.h for the layout and semantics).

    target_logits [R, V] bf16 or fp32; draft_probs [R-B, V] fp32; draft_tokens [R-B] int32;
    num_drafts [B] int32; row_offsets [B+1] int32 or None (uniform layout);
    per-request params [B]; uniforms [R, 2] fp32; outputs out_tokens [B, k_max+1] int32,
    accept_len [B] int32, out_pq [R-B, 2] fp32 or None; workspace uint8 device tensor;
    prior: None or (prior_offsets [B+1], prior_tokens [H], prior_counts [H]) int32, the
    requests' prior history for the penalties.
    """
    dt, B, V, R, params = _checked_args(target_logits, draft_probs, draft_tokens, num_drafts, row_offsets, k_max,
                                        temperature, top_k, top_p, presence_penalty, frequency_penalty, greedy,
                                        uniforms, out_tokens, accept_len, out_pq, workspace, prior)
    st = lib().spec_verify(_ptr(target_logits), dt, _ptr(draft_probs), _ptr(draft_tokens), _ptr(num_drafts),
                           _ptr(row_offsets), B, k_max, V, R, params, _ptr(uniforms), _ptr(out_tokens),
                           _ptr(accept_len), _ptr(out_pq), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _stream(stream))
    if st != SV_OK:
        raise SvError(st, "spec_verify")


def spec_verify_lazy(target_logits, draft_probs, draft_tokens, num_drafts, row_offsets, k_max: int,
                     temperature, top_k, top_p, presence_penalty, frequency_penalty, greedy, uniforms,
                     out_tokens, accept_len, out_pq, workspace, stream=None, prior=None) -> None:
    """spec_verify that reads each request's rows 1..k only when its draft 0 was kept (the rows
    after a first rejection are never read); same arguments and results as spec_verify."""
    dt, B, V, R, params = _checked_args(target_logits, draft_probs, draft_tokens, num_drafts, row_offsets, k_max,
                                        temperature, top_k, top_p, presence_penalty, frequency_penalty, greedy,
                                        uniforms, out_tokens, accept_len, out_pq, workspace, prior)
    st = lib().spec_verify_lazy(_ptr(target_logits), dt, _ptr(draft_probs), _ptr(draft_tokens), _ptr(num_drafts),
                                _ptr(row_offsets), B, k_max, V, R, params, _ptr(uniforms), _ptr(out_tokens),
                                _ptr(accept_len), _ptr(out_pq), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    if st != SV_OK:
        raise SvError(st, "spec_verify_lazy")


def spec_verify_onehot(target_logits, draft_tokens, num_drafts, row_offsets, k_max: int, temperature, top_k,
                       top_p, presence_penalty, frequency_penalty, greedy, uniforms, out_tokens, accept_len,
                       out_pq, workspace, stream=None, prior=None) -> None:
    """Verify drafts proposed as one-hot (argmax) tokens: every row is sampled with slot 1 of
    its uniforms and the drafts are kept while they equal the samples; no q is read (see
    include/spec_verify.h).  Arguments as spec_verify without draft_probs; out_pq receives
    (p(x_i), 1)."""
    dt, B, V, R, params = _checked_args(target_logits, None, draft_tokens, num_drafts, row_offsets, k_max,
                                        temperature, top_k, top_p, presence_penalty, frequency_penalty, greedy,
                                        uniforms, out_tokens, accept_len, out_pq, workspace, prior)
    st = lib().spec_verify_onehot(_ptr(target_logits), dt, _ptr(draft_tokens), _ptr(num_drafts),
                                  _ptr(row_offsets), B, k_max, V, R, params, _ptr(uniforms), _ptr(out_tokens),
                                  _ptr(accept_len), _ptr(out_pq), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream))
    if st != SV_OK:
        raise SvError(st, "spec_verify_onehot")


def spec_rollback(kv_seq_len, accept_len, num_drafts, workspace, stream=None) -> None:
    """kv_seq_len[b] <- kv_seq_len[b] - (k_b + 1) + 1 + accept_len[b], in place on the device."""
    import torch
    B = kv_seq_len.numel()
    _check(kv_seq_len, "kv_seq_len", torch.int32, B)
    _check(accept_len, "accept_len", torch.int32, B)
    _check(num_drafts, "num_drafts", torch.int32, B)
    _check(workspace, "workspace")
    st = lib().spec_rollback(_ptr(kv_seq_len), _ptr(accept_len), _ptr(num_drafts), B, _ptr(workspace),
                             _stream(stream))
    if st != SV_OK:
        raise SvError(st, "spec_rollback")


def sv_read_device_error(workspace):
    """(code, first_bad_request) of the workspace's sticky device-data error word (syncs)."""
    code, bad = C.c_int32(0), C.c_int32(-1)
    st = lib().sv_read_device_error(_ptr(workspace), C.byref(code), C.byref(bad))
    if st not in (SV_OK, SV_ERR_DEVICE_DATA):
        raise SvError(st, "sv_read_device_error")
    return int(code.value), int(bad.value)
