"""The library's per-context state: a context created again on the same device (after
cudaDeviceReset, which ends only this process's context) must work like the first one.

The stream kernel needs more than the default 48 KB of dynamic shared memory at V = 128256,
and that opt-in belongs to the kernel in one context.  A library that remembered it per
process would skip it in the new context and fail the launch; the same would happen for a
second device in one process.  The check runs in a child process that touches the GPU only
through the library and the CUDA runtime (no PyTorch), so the reset disturbs nothing else.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import ctypes as C, sys
import numpy as np
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import sv_workloads as W
import speculative_decoding_verification_12_gb300 as sv
import oracle
from sv_parity import compare

lib = sv.lib()
rt = C.CDLL("libcudart.so.13")          # the runtime the library itself loaded
H2D, D2H = 1, 2


def call(w):
    held = []

    def up(a):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        p = C.c_void_p()
        assert rt.cudaMalloc(C.byref(p), C.c_size_t(max(a.nbytes, 16))) == 0
        assert rt.cudaMemcpy(p, a.ctypes.data_as(C.c_void_p), C.c_size_t(a.nbytes), H2D) == 0
        held.append(p)
        return p.value

    B, k, V, R = w.B, w.k_max, w.V, w.total_rows
    ws_bytes = lib.sv_workspace_bytes(B, R, V)
    ws = C.c_void_p()
    assert rt.cudaMalloc(C.byref(ws), C.c_size_t(ws_bytes)) == 0
    out = up(np.full((B, k + 1), -7, np.int32))
    acc = up(np.full(B, -7, np.int32))
    prm = sv.SvParams(up(w.temperature), up(w.top_k), up(w.top_p), up(w.presence), up(w.frequency),
                      up(w.greedy), None, None, None, 0)
    st = lib.spec_verify(up(w.target_logits), sv.SV_BF16, up(w.draft_probs), up(w.draft_tokens),
                         up(w.num_drafts), None, B, k, V, R, prm, up(w.uniforms), out, acc, None, ws,
                         ws_bytes, None)
    assert st == sv.SV_OK, ("spec_verify", st)
    assert rt.cudaDeviceSynchronize() == 0
    o_tok = np.empty((B, k + 1), np.int32)
    o_acc = np.empty(B, np.int32)
    assert rt.cudaMemcpy(o_tok.ctypes.data_as(C.c_void_p), C.c_void_p(out), C.c_size_t(o_tok.nbytes), D2H) == 0
    assert rt.cudaMemcpy(o_acc.ctypes.data_as(C.c_void_p), C.c_void_p(acc), C.c_size_t(o_acc.nbytes), D2H) == 0
    for p in held + [ws]:
        rt.cudaFree(p)
    return {"out_tokens": o_tok, "accept_len": o_acc}


w = W.random_batch(31, B=6, k_max=3, V=128256, dtype="bf16", greedy_frac=0.3)
first = call(w)
assert rt.cudaDeviceReset() == 0         # a new context on the same device from here on
second = call(w)
assert np.array_equal(first["out_tokens"], second["out_tokens"])
assert np.array_equal(first["accept_len"], second["accept_len"])
print(compare(w, second, oracle.verify(w)))
print("context ok")
'''


def test_new_context_on_the_same_device():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    oracle.build()
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "context ok" in r.stdout, r.stdout + r.stderr
