"""spec_verify_static (the entry point whose workspace is a device array inside the library)
against spec_verify with a caller-provided workspace, through the C ABI.

Kept in a file of its own that sorts last, so that it runs both alone and after every other
GPU test in the same process (the array is shared by every call on the device).
"""
import ctypes as C

import numpy as np
import pytest

import sv_workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

# out_pq of the two entry points must agree to within this relative error (both run the same
# kernels on the same inputs, so in practice they agree bit for bit)
PQ_RTOL = 1e-6


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_12_gb300 as sv
    sv.lib()
    return sv


def _static_call(sv, db):
    """One spec_verify_static call on the tensors of a DeviceBatch; returns its outputs."""
    from speculative_decoding_verification_12_gb300 import SvParams, SV_BF16, SV_F32
    p = lambda t: None if t is None else t.data_ptr()
    out_tokens = torch.full_like(db.out_tokens, -7)
    accept_len = torch.full_like(db.accept_len, -7)
    out_pq = torch.full_like(db.out_pq, float("nan"))
    params = SvParams(p(db.temperature), p(db.top_k), p(db.top_p), p(db.presence), p(db.frequency), p(db.greedy))
    dt = SV_BF16 if db.target_logits.dtype == torch.bfloat16 else SV_F32
    st = sv.lib().spec_verify_static(p(db.target_logits), dt, p(db.draft_probs), p(db.draft_tokens),
                                     p(db.num_drafts), p(db.row_offsets), db.B, db.k_max, db.V, db.R, params,
                                     p(db.uniforms), p(out_tokens), p(accept_len), p(out_pq),
                                     torch.cuda.current_stream().cuda_stream)
    assert st == sv.SV_OK, sv.lib().sv_status_string(st)
    torch.cuda.synchronize()
    return out_tokens.cpu().numpy(), accept_len.cpu().numpy(), out_pq.cpu().numpy()


@pytest.mark.parametrize("seed,dtype,varlen", [(3, "bf16", True), (4, "f32", False)])
def test_static_matches_workspace_call(sv, seed, dtype, varlen):
    from speculative_decoding_verification_12_gb300.batch import DeviceBatch
    w = W.random_batch(seed, B=40, k_max=5, V=6000, dtype=dtype, varlen=varlen, greedy_frac=0.3)
    db = DeviceBatch.from_host(w, "cuda", want_pq=True)
    db.run()
    torch.cuda.synchronize()
    ref_tok = db.out_tokens.cpu().numpy()
    ref_acc = db.accept_len.cpu().numpy()
    ref_pq = db.out_pq.cpu().numpy()
    # two calls in a row: the second starts from whatever the first left in the shared array
    for _ in range(2):
        tok, acc, pq = _static_call(sv, db)
        np.testing.assert_array_equal(acc, ref_acc)
        np.testing.assert_array_equal(tok, ref_tok)
        np.testing.assert_allclose(pq, ref_pq, rtol=PQ_RTOL, atol=0.0, equal_nan=True)


def test_static_rejects_batches_beyond_the_array(sv):
    """A batch whose workspace exceeds the array is refused before anything is enqueued."""
    from speculative_decoding_verification_12_gb300 import SvParams
    limit = 32 << 20
    B, R, V = 1024, 8192, 128256
    assert sv.sv_workspace_bytes(B, R, V) > limit
    params = SvParams(None, None, None, None, None, None)
    st = sv.lib().spec_verify_static(None, 0, None, None, None, None, B, 7, V, R, params, None, None, None, None,
                                     None)
    assert st == sv.SV_ERR_WORKSPACE
