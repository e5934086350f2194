"""The C-ABI library: it loads, exports what include/bwd.h declares, its host
codebook builder agrees with the oracle bit for bit, and it rejects bad
arguments on the host before touching a GPU."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_wise_dynamic_gb300 import build as b

    b.build()
    from block_wise_dynamic_gb300 import _abi

    return _abi.load()


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(bwd_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("bwd_quantize_blockwise", "bwd_dequantize_blockwise", "bwd_adam8bit_step",
                 "bwd_adam8bit_step_multi", "bwd_build_map", "bwd_state_init"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


@pytest.mark.parametrize("kind,signed", [(0, True), (1, False)])
def test_host_builder_matches_oracle_bitwise(lib, kind, signed):
    m = np.empty(256, np.float32)
    t = np.empty(255, np.float32)
    assert lib.bwd_build_map(kind, m.ctypes.data, t.ctypes.data) == 0
    assert np.array_equal(m.view(np.uint32), oracle.dynamic_map(signed).view(np.uint32))
    assert np.array_equal(t.view(np.uint32), oracle.thresholds(signed).view(np.uint32))
    assert lib.bwd_build_map(kind, None, None) == 0


def test_num_blocks(lib):
    for n, nb in [(0, 0), (1, 1), (2047, 1), (2048, 1), (2049, 2), (6_738_415_616, 3_290_242)]:
        assert lib.bwd_num_blocks(n) == nb
    assert lib.bwd_num_blocks(-1) == -1


def test_status_strings(lib):
    assert lib.bwd_status_string(0) == b"ok"
    assert lib.bwd_status_string(1) == b"invalid argument"
    assert lib.bwd_status_string(99) == b"unknown status"


def test_bad_arguments_are_rejected_on_the_host(lib):
    from block_wise_dynamic_gb300._abi import AdamHParams

    fake = ctypes.c_void_p(0x1000)  # never dereferenced: rejected first
    assert lib.bwd_build_map(7, None, None) == 1
    assert lib.bwd_quantize_blockwise(fake, -1, 0, fake, fake, None) == 1
    assert lib.bwd_quantize_blockwise(fake, 10, 5, fake, fake, None) == 1
    assert lib.bwd_quantize_blockwise(None, 10, 0, fake, fake, None) == 1
    assert b"NULL" in lib.bwd_last_error()
    assert lib.bwd_dequantize_blockwise(fake, None, 10, 0, fake, None) == 1
    assert lib.bwd_state_init(fake, fake, None, fake, 10, None) == 1
    # n == 0 is a no-op that succeeds without a device
    assert lib.bwd_quantize_blockwise(None, 0, 0, None, None, None) == 0
    assert lib.bwd_dequantize_blockwise(None, None, 0, 1, None, None) == 0
    assert lib.bwd_state_init(None, None, None, None, 0, None) == 0

    hp = AdamHParams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1)
    step = lib.bwd_adam8bit_step
    assert step(fake, fake, 0, fake, fake, fake, fake, 0, ctypes.byref(hp), None) == 0
    assert step(fake, fake, 7, fake, fake, fake, fake, 10, ctypes.byref(hp), None) == 2
    assert step(fake, fake, 0, fake, fake, fake, fake, 10, None, None) == 1
    for bad in (AdamHParams(1e-3, 0.9, 0.999, 1e-8, 0.0, 0),      # step 0
                AdamHParams(1e-3, 1.0, 0.999, 1e-8, 0.0, 1),      # beta1 = 1
                AdamHParams(1e-3, 0.9, -0.1, 1e-8, 0.0, 1),       # beta2 < 0
                AdamHParams(float("nan"), 0.9, 0.999, 1e-8, 0.0, 1),
                AdamHParams(1e-3, 0.9, 0.999, -1.0, 0.0, 1),      # eps < 0
                AdamHParams(1e-3, 0.9, 0.999, 1e-8, -0.01, 1),    # negative weight decay
                AdamHParams(1e-3, 0.9, 0.999, 1e-8, float("inf"), 1)):
        assert step(fake, fake, 0, fake, fake, fake, fake, 10, ctypes.byref(bad), None) == 1
    assert step(None, fake, 0, fake, fake, fake, fake, 10, ctypes.byref(hp), None) == 1

    multi = lib.bwd_adam8bit_step_multi
    assert multi(0, None, None, 0, None, None, None, None, None, ctypes.byref(hp), None) == 0
    assert multi(-1, None, None, 0, None, None, None, None, None, ctypes.byref(hp), None) == 1
    assert multi(2, None, None, 0, None, None, None, None, None, ctypes.byref(hp), None) == 1
    arr = (ctypes.c_void_p * 2)(0x1000, 0x2000)
    nul = (ctypes.c_void_p * 2)(0x1000, None)
    ns = (ctypes.c_int64 * 2)(5, 7)
    neg = (ctypes.c_int64 * 2)(5, -7)
    assert multi(2, arr, arr, 0, arr, arr, arr, arr, neg, ctypes.byref(hp), None) == 1
    assert multi(2, arr, nul, 0, arr, arr, arr, arr, ns, ctypes.byref(hp), None) == 1
    assert b"tensor 1" in lib.bwd_last_error()


def test_embedding_xavier_bound_matches_oracle(lib):
    from oracle import stable_embedding as se

    for v, d in [(32000, 4096), (50304, 1024), (7, 5), (1, 1)]:
        assert np.float32(lib.bwd_embedding_xavier_bound(v, d)).view(np.uint32) == se.xavier_bound(v, d).view(np.uint32)
    assert lib.bwd_embedding_xavier_bound(0, 5) == -1.0
    assert lib.bwd_embedding_xavier_bound(5, 0) == -1.0


def test_embedding_bad_arguments_are_rejected_on_the_host(lib):
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: rejected first
    init = lib.bwd_embedding_init
    assert init(fake, 0, 4, fake, None) == 1
    assert init(fake, 4, 0, fake, None) == 1
    assert init(None, 4, 4, fake, None) == 1
    assert init(fake, 2 ** 40, 2 ** 40, fake, None) == 1     # V * D overflows
    fwd = lib.bwd_embedding_forward
    ok = dict(ids=fake, t=10, w=fake, v=100, d=64, g=fake, b=fake, eps=1e-5, y=fake)

    def f(**kw):
        a = {**ok, **kw}
        return fwd(a["ids"], a["t"], a["w"], a["v"], a["d"], a["g"], a["b"], a["eps"], a["y"], None, None, None)

    assert f(t=-1) == 1
    assert f(v=0) == 1
    assert f(d=0) == 1
    assert f(eps=-1.0) == 1
    assert f(eps=float("inf")) == 1
    assert f(eps=float("nan")) == 1
    assert f(ids=None) == 1 and f(w=None) == 1 and f(g=None) == 1 and f(b=None) == 1 and f(y=None) == 1
    assert f(t=2 ** 62, d=64) == 1                          # T * D overflows
    assert f(t=0, ids=None, w=None, y=None) == 0            # no tokens: no-op without a device
    bwd = lib.bwd_embedding_backward
    args = [fake, 10, fake, 100, 64, fake, fake, fake, fake, fake, fake, fake, None]
    for i in (0, 2, 5, 6, 7, 8, 9, 10, 11):                 # every pointer argument
        a = list(args)
        a[i] = None
        assert bwd(*a) == 1
    a = list(args)
    a[1] = -5
    assert bwd(*a) == 1
    a = [None] * 13
    a[1], a[3], a[4] = 0, 100, 64
    assert bwd(*a) == 0


def test_pointers_misaligned_for_their_element_size_are_rejected(lib):
    from block_wise_dynamic_gb300._abi import AdamHParams

    ok, odd = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1001)
    assert lib.bwd_quantize_blockwise(odd, 10, 0, ok, ok, None) == 1
    assert b"aligned" in lib.bwd_last_error()
    assert lib.bwd_dequantize_blockwise(ok, ok, 10, 0, odd, None) == 1
    assert lib.bwd_state_init(ok, odd, ok, ok, 10, None) == 1
    hp = AdamHParams(1e-3, 0.9, 0.999, 1e-8, 0.0, 1)
    assert lib.bwd_adam8bit_step(odd, ok, 0, ok, ok, ok, ok, 10, ctypes.byref(hp), None) == 1
    two = ctypes.c_void_p(0x1002)  # fine for bf16, not for fp32
    assert lib.bwd_adam8bit_step(ok, two, 0, ok, ok, ok, ok, 10, ctypes.byref(hp), None) == 1
    assert lib.bwd_embedding_forward(ctypes.c_void_p(0x1004), 10, ok, 100, 64, ok, ok, 1e-5, ok, None, None,
                                     None) == 1
    assert lib.bwd_embedding_init(ok, 4, 4, two, None) == 1


def test_missing_library_fails_loudly():
    """Without the built library every call raises ImportError: there is no
    CPU fallback behind the package's functions."""
    import subprocess
    import sys

    code = (
        "import block_wise_dynamic_gb300._abi as a\n"
        "a.LIB_PATH = '/nonexistent/libbwd.so'\n"
        "import block_wise_dynamic_gb300 as m\n"
        "from block_wise_dynamic_gb300 import embedding as emb\n"
        "for call in (lambda: m.build_map('signed'), lambda: emb.xavier_bound(10, 10)):\n"
        "    try:\n"
        "        call()\n"
        "    except ImportError as err:\n"
        "        assert 'no fallback' in str(err)\n"
        "    else:\n"
        "        raise SystemExit('no ImportError')\n"
        "print('ok')\n"
    )
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
