"""The C-ABI library loads and exports every entry point include/*.h declares; host-side
argument checks reject bad calls before anything is enqueued (no GPU work here)."""
import ctypes as C
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libsv():
    from speculative_decoding_verification_12_gb300 import build
    build.build()
    import speculative_decoding_verification_12_gb300 as sv
    return sv


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\**\s*([A-Za-z_]\w*)\s*\(", src, flags=re.M):
            if m.group(1) not in ("if", "while", "for", "switch", "return", "sizeof"):
                names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    assert declared_functions() >= {"sv_workspace_bytes", "spec_verify", "spec_rollback", "sv_read_device_error",
                                    "sv_status_string"}


def test_every_declared_symbol_is_exported(libsv):
    l = libsv.lib()
    for name in declared_functions():
        assert hasattr(l, name), f"{name} declared in include/ but not exported"


def test_workspace_size(libsv):
    assert libsv.sv_workspace_bytes(0, 5, 10) == 0
    assert libsv.sv_workspace_bytes(2, 1, 10) == 0
    a = libsv.sv_workspace_bytes(256, 1280, 128256)
    b = libsv.sv_workspace_bytes(512, 2560, 151936)
    assert 0 < a < b and a % 256 == 0
    # per row: statistics, a kept list and 12 bytes per (padded) 256-token segment; per
    # request: a counter and the history index (a word per segment, a mask bit per segment)
    nsegp = ((128256 + 255) // 256 + 31) // 32 * 32
    assert a < 1280 * (4096 + 12 * nsegp) + 256 * (64 + 4 * (nsegp + 1) + nsegp // 8) + 65536


def test_host_checks_reject_bad_calls(libsv):
    l = libsv.lib()
    P = libsv.SvParams(1, 1, 1, None, None, 1)   # non-null placeholders; never dereferenced
    ws = C.c_void_p(256)
    base = dict(tl=C.c_void_p(16), dt=libsv.SV_BF16, dp=C.c_void_p(16), tok=C.c_void_p(16), nd=C.c_void_p(16),
                ro=None, B=2, k=4, V=100, R=10, u=C.c_void_p(16), ot=C.c_void_p(16), al=C.c_void_p(16))

    def call(**kw):
        a = dict(base, **kw)
        return l.spec_verify(a["tl"], a["dt"], a["dp"], a["tok"], a["nd"], a["ro"], a["B"], a["k"], a["V"], a["R"],
                             a.get("P", P), a["u"], a["ot"], a["al"], None, a.get("ws", ws), a.get("wsb", 1 << 30),
                             None)

    assert call(B=0) == libsv.SV_ERR_INVALID_ARG
    assert call(V=0) == libsv.SV_ERR_INVALID_ARG
    assert call(k=65, R=2 * 66) == libsv.SV_ERR_UNSUPPORTED
    assert call(V=(1 << 21) + 1) == libsv.SV_ERR_UNSUPPORTED
    assert call(dt=7) == libsv.SV_ERR_INVALID_ARG
    assert call(R=11) == libsv.SV_ERR_INVALID_ARG            # uniform layout needs R = B (k+1)
    assert call(tl=None) == libsv.SV_ERR_INVALID_ARG
    assert call(dp=None) == libsv.SV_ERR_INVALID_ARG
    assert call(P=libsv.SvParams(None, 1, 1, None, None, 1)) == libsv.SV_ERR_INVALID_ARG
    # a history needs all three arrays and a length >= 0
    assert call(P=libsv.SvParams(1, 1, 1, None, None, 1, 16, None, 16, 4)) == libsv.SV_ERR_INVALID_ARG
    assert call(P=libsv.SvParams(1, 1, 1, None, None, 1, 16, 16, 16, -1)) == libsv.SV_ERR_INVALID_ARG
    assert call(ws=C.c_void_p(257)) == libsv.SV_ERR_WORKSPACE
    assert call(wsb=100) == libsv.SV_ERR_WORKSPACE
    # the one-hot entry point: the same host checks, without draft_probs

    def call1(**kw):
        a = dict(base, **kw)
        return l.spec_verify_onehot(a["tl"], a["dt"], a["tok"], a["nd"], a["ro"], a["B"], a["k"], a["V"], a["R"],
                                    a.get("P", P), a["u"], a["ot"], a["al"], None, a.get("ws", ws),
                                    a.get("wsb", 1 << 30), None)

    assert call1(B=0) == libsv.SV_ERR_INVALID_ARG
    assert call1(k=65, R=2 * 66) == libsv.SV_ERR_UNSUPPORTED
    assert call1(R=11) == libsv.SV_ERR_INVALID_ARG
    assert call1(tok=None) == libsv.SV_ERR_INVALID_ARG        # drafts are still needed
    assert call1(u=None) == libsv.SV_ERR_INVALID_ARG
    assert call1(wsb=100) == libsv.SV_ERR_WORKSPACE
    assert l.spec_rollback(None, C.c_void_p(16), C.c_void_p(16), 4, ws, None) == libsv.SV_ERR_INVALID_ARG
    assert l.sv_status_string(libsv.SV_ERR_WORKSPACE) == b"workspace too small or misaligned"
    # the measurement hook takes both events or neither (nothing is recorded by these calls)
    assert l.sv_set_phase_events(C.c_void_p(16), None) == libsv.SV_ERR_INVALID_ARG
    assert l.sv_set_phase_events(None, C.c_void_p(16)) == libsv.SV_ERR_INVALID_ARG
    assert l.sv_set_phase_events(None, None) == libsv.SV_OK


def test_prefer_lazy_choice(libsv):
    """sv_prefer_lazy on the measured batch shapes (bf16 unless noted).  Both calls were timed
    on a GB300 with the share of requests rejecting draft 0 set to 0, 1/4, 1/2, 3/4 and 1: the
    lazy call won on the 64-request V=32000 batch only at share 1; on the 256-request V=128256
    batch from about 3/4 on; on the ragged 512-request V=151936 batch from about 1/4 on (by 25 us
    at 0.44); and on the 1024-request fp32 batch at its natural share (about 0.26)."""
    pick = libsv.sv_prefer_lazy
    for share in (0.0, 0.5, 0.75, 0.95):
        assert not pick(64, 384, 32000, libsv.SV_BF16, share)
    assert pick(64, 384, 32000, libsv.SV_BF16, 1.0)
    assert not pick(256, 1280, 128256, libsv.SV_BF16, 0.5)
    assert pick(256, 1280, 128256, libsv.SV_BF16, 0.9)
    assert not pick(512, 2510, 151936, libsv.SV_BF16, 0.1)
    assert pick(512, 2510, 151936, libsv.SV_BF16, 0.44)
    assert pick(1024, 8192, 128256, libsv.SV_F32, 0.26)
    assert not pick(1024, 8192, 128256, libsv.SV_F32, 0.01)
    # one switch from the one-pass call to the lazy call as the share grows
    for shape in ((64, 384, 32000), (256, 1280, 128256), (512, 2510, 151936), (1024, 8192, 128256)):
        got = [pick(*shape, libsv.SV_BF16, s / 100) for s in range(101)]
        assert got == sorted(got), shape
    # fp32 rows skip twice the bytes of bf16 rows
    assert pick(256, 1280, 128256, libsv.SV_F32, 0.5) and not pick(256, 1280, 128256, libsv.SV_BF16, 0.5)
    l = libsv.lib()
    assert l.sv_prefer_lazy(0, 10, 100, libsv.SV_BF16, 0.5) == -1
    assert l.sv_prefer_lazy(4, 3, 100, libsv.SV_BF16, 0.5) == -1
    assert l.sv_prefer_lazy(4, 20, 0, libsv.SV_BF16, 0.5) == -1
    assert l.sv_prefer_lazy(4, 20, 100, 7, 0.5) == -1
    assert l.sv_prefer_lazy(4, 20, 100, libsv.SV_BF16, 1.5) == -1
    assert l.sv_prefer_lazy(4, 20, 100, libsv.SV_BF16, float("nan")) == -1
    with pytest.raises(libsv.SvError):
        pick(4, 20, 100, libsv.SV_BF16, -0.1)


def test_package_has_no_cpu_fallback():
    """The binding never imports the oracle or a CPU implementation."""
    pkg = os.path.join(ROOT, "speculative_decoding_verification_12_gb300")
    for f in glob.glob(os.path.join(pkg, "*.py")):
        src = open(f).read()
        assert "import oracle" not in src and "from oracle" not in src, f
