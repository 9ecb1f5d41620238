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


def test_package_has_no_cpu_fallback():
    """The binding never imports the oracle or a CPU implementation."""
    pkg = os.path.join(ROOT, "speculative_decoding_verification_12_gb300")
    for f in glob.glob(os.path.join(pkg, "*.py")):
        src = open(f).read()
        assert "import oracle" not in src and "from oracle" not in src, f
