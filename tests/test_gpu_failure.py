"""Failure detection on the GPU without a GPU fault.

Every wait of the streaming kernel is bounded (2 s).  The testing aid sv_set_test_withhold
makes one CTA's scheduler withhold a work unit -- a flag that nothing else sets -- so the
copy and reduction warps waiting for it give up.  The call must still complete: SV_DEV_TIMEOUT
in the workspace's error word, -1 for every request's outputs, and a device that the next call
uses normally.
"""
import numpy as np
import pytest

import sv_workloads as W
from sv_parity import compare

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_12_gb300 as sv
    sv.lib()
    return sv


@pytest.mark.parametrize("onehot", [False, True])
def test_bounded_wait_runs_out(sv, oracle_lib, onehot):
    from speculative_decoding_verification_12_gb300.batch import DeviceBatch
    # 16-byte aligned rows (V * 2 bytes = 40000): the two-kernel path whose waits are bounded
    w = W.random_batch(33, B=16, k_max=3, V=20000, dtype="bf16", greedy_frac=0.3)
    db = DeviceBatch.from_host(w, "cuda", want_pq=True)
    lib = sv.lib()
    assert lib.sv_set_test_withhold(1) == sv.SV_OK
    try:
        db.run(onehot=onehot)
        torch.cuda.synchronize()
    finally:
        lib.sv_set_test_withhold(0)
    g = db.results()
    code, _ = sv.sv_read_device_error(db.workspace)
    assert code == 7, code
    assert (g["accept_len"] == -1).all() and (g["out_tokens"] == -1).all()
    # the context is intact: the same batch verifies normally
    db.run(onehot=onehot)
    g2 = db.results()
    assert sv.sv_read_device_error(db.workspace)[0] == 0
    compare(w, g2, oracle_lib.verify(w, onehot=onehot))
