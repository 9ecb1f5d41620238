"""Failure detection on the GPU without a GPU fault.

Every wait of the streaming kernel is bounded (2 s).  The testing aid sv_set_test_withhold
makes one CTA's scheduler withhold a work unit -- a flag that nothing else sets -- so the
copy and reduction warps waiting for it give up.  The call must still complete, with
SV_DEV_TIMEOUT in the workspace's error word and a device that the next call uses normally.
Which requests get -1 outputs depends on how the call selects rows: a one-pass call over more
rows than the select kernel holds at once selects each row as soon as it is streamed, so only
the requests with a row that was not streamed fail and the others must match the oracle; a
smaller one-pass call selects once the whole stream is done and fails every request, as does
the lazy call for every request it had not decided.
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


@pytest.mark.parametrize("size", ["one_wave", "many_rows"])
@pytest.mark.parametrize("scheme", ["accept", "onehot", "lazy"])
def test_bounded_wait_runs_out(sv, oracle_lib, scheme, size):
    from speculative_decoding_verification_12_gb300.batch import DeviceBatch
    onehot, lazy = scheme == "onehot", scheme == "lazy"
    # 16-byte aligned rows: the two-kernel path whose waits are bounded.  many_rows: 1600 rows,
    # more than the select kernel holds at once on a GB300 (9 per SM, 152 SMs)
    if size == "one_wave":
        w = W.random_batch(33, B=16, k_max=3, V=20000, dtype="bf16", greedy_frac=0.3)
    else:
        w = W.random_batch(34, B=400, k_max=3, V=2048, dtype="bf16", greedy_frac=0.3)
    per_row = size == "many_rows" and not lazy and w.total_rows > 9 * torch.cuda.get_device_properties(0).multi_processor_count
    db = DeviceBatch.from_host(w, "cuda", want_pq=True)
    lib = sv.lib()
    assert lib.sv_set_test_withhold(1) == sv.SV_OK
    try:
        db.run(onehot=onehot, lazy=lazy)
        torch.cuda.synchronize()
    finally:
        lib.sv_set_test_withhold(0)
    g = db.results()
    code, _ = sv.sv_read_device_error(db.workspace)
    assert code == 7, code
    o = oracle_lib.verify(w, onehot=onehot)
    failed = g["accept_len"] == -1
    assert failed.any()
    assert (g["out_tokens"][failed] == -1).all()
    if per_row:
        # only the requests of the withheld CTA's rows fail
        assert failed.sum() < w.B
        compare(w, g, o, requests=np.flatnonzero(~failed))
    else:
        assert failed.all()
    # the context is intact: the same batch verifies normally
    db.run(onehot=onehot, lazy=lazy)
    g2 = db.results()
    assert sv.sv_read_device_error(db.workspace)[0] == 0
    compare(w, g2, o, pq_on_path=lazy)
