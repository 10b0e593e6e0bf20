"""CPU checks of the C library: it builds, loads, exports every function the header
declares, and rejects bad host-side arguments synchronously (no kernel is launched)."""
import ctypes
import os
import re

import pytest

from tests.helpers import ensure_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(simsd_\w+)\s*\(", text, re.M):
            names.append(m.group(1))
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    ensure_library()
    import diffusion_speculative_verify_gb300 as pkg
    return pkg.load_library()


def test_header_declares_the_three_calls():
    names = _declared_functions()
    for n in ("simsd_build_layout", "simsd_verify_attention", "simsd_accept",
              "simsd_verify_attention_workspace", "simsd_accept_workspace"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    names = _declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), n
    import diffusion_speculative_verify_gb300 as pkg
    assert set(pkg.EXPORTED) == set(names)


def test_status_strings_and_version(lib):
    import diffusion_speculative_verify_gb300 as pkg
    assert pkg.simsd_status_str(0) == "SIMSD_OK"
    assert pkg.simsd_status_str(3) == "SIMSD_ERR_WORKSPACE"
    assert pkg.simsd_status_str(99) == "SIMSD_ERR_UNKNOWN"
    assert pkg.simsd_version() == 300


def test_host_argument_errors_return_status(lib):
    # nothing below reaches a kernel launch
    assert lib.simsd_build_layout(None, None, 4, 0, None, None, None, None) == 1
    assert lib.simsd_build_layout(None, None, 4, 33, None, None, None, None) == 1
    assert lib.simsd_build_layout(None, None, 4, 4, None, None, None, None) == 1
    assert lib.simsd_build_layout(None, None, 0, 4, None, None, None, None) == 0
    assert lib.simsd_build_layout_ex(None, None, 0, 4, 1, None, None, None, None) == 0
    assert lib.simsd_build_layout_ex(None, None, 0, 4, 2, None, None, None, None) == 1
    assert lib.simsd_build_layout_ex(None, None, 4, 4, 1, None, None, None, None) == 1
    # temperature 0 (greedy) is accepted, a negative one is not; gamma > B is invalid
    args = [None] * 4 + [2, 4, 4, 100, 0.0, 0, 0] + [None] * 4 + [None, 0, None, None]
    assert lib.simsd_accept(*args) == 1          # null pointers
    args[8] = -1.0
    assert lib.simsd_accept(*args) == 1
    args[8] = 1.0
    args[6] = 5
    assert lib.simsd_accept(*args) == 1
    args[6] = 4
    assert lib.simsd_accept(*args) == 1          # null pointers
    assert lib.simsd_accept_workspace(2, 4, 4, 100) > 0
    assert lib.simsd_accept_workspace(2, 4, 5, 100) == 0
    # the logit-type entries: an unknown type is invalid; batch 0 with a known one is a no-op
    ex = [None, None, 1, None, None, 0, 4, 4, 100, 1.0, 0, 0] + [None] * 5 + [0, None, None]
    assert lib.simsd_accept_ex(*ex) == 0
    ex[2] = 2
    assert lib.simsd_accept_ex(*ex) == 1
    ex[2], ex[5] = 1, 2
    assert lib.simsd_accept_ex(*ex) == 1          # null pointers
    cx = [None, 1, None, None, None, 0, 4, 4, 100, 1.0, 0, 0] + [None] * 5 + [0, None, None]
    assert lib.simsd_accept_coupled_ex(*cx) == 0
    cx[1] = 7
    assert lib.simsd_accept_coupled_ex(*cx) == 1
    cx[1], cx[5] = 0, 2
    assert lib.simsd_accept_coupled_ex(*cx) == 1  # null pointers
    # the expected accepted-prefix estimator: T > 0, beta >= 0, a known mode and type
    kx = [None, 0, None, 0, 4, 4, 100, 1.0, 1, 0.5, 1.0, None, None, None, 0, None, None]
    assert lib.simsd_expected_prefix(*kx) == 0    # batch 0: nothing to do
    for i, bad in ((7, 0.0), (7, -1.0), (10, -0.5), (8, 2), (1, 3), (9, float("nan"))):
        k2 = list(kx)
        k2[i] = bad
        assert lib.simsd_expected_prefix(*k2) == 1, (i, bad)
    kx[3] = 2
    assert lib.simsd_expected_prefix(*kx) == 1    # null pointers
    assert lib.simsd_expected_prefix_workspace(2, 4, 4, 100) >= 256
    assert lib.simsd_expected_prefix_workspace(2, 4, 5, 100) == 0


def test_attention_parameter_checks(lib):
    import diffusion_speculative_verify_gb300 as pkg
    p = pkg.AttnParams()
    p.dtype, p.batch, p.B, p.Hq, p.Hkv, p.D = 0, 1, 4, 4, 1, 64
    p.rope_theta = 1e4
    assert lib.simsd_verify_attention_workspace(ctypes.byref(p)) > 0
    assert lib.simsd_verify_attention(ctypes.byref(p), None, 0, None) == 1  # null pointers
    p.Hq = 3
    assert lib.simsd_verify_attention(ctypes.byref(p), None, 0, None) == 1
    p.Hq, p.D = 4, 96
    assert lib.simsd_verify_attention(ctypes.byref(p), None, 0, None) == 2
    p.D, p.B = 64, 40
    assert lib.simsd_verify_attention(ctypes.byref(p), None, 0, None) == 1
    p.B, p.rope_theta = 4, 0.0
    assert lib.simsd_verify_attention(ctypes.byref(p), None, 0, None) == 1


def test_noalloc_accept_returns_the_status_of_accept(lib):
    # the allocation-free entry runs simsd_accept's argument checks first and in the same
    # order, so a bad argument gives the same status even for sizes beyond its fixed scratch
    big = [1 << 16, 32, 32, 1000]   # batch, B, gamma, V: a plan larger than the fixed array
    for temperature in (float("nan"), -1.0):
        a = [None] * 4 + big + [temperature, 0, 0] + [None] * 4 + [None, 0, None, None]
        n = [None] * 4 + big + [temperature, 0, 0] + [None] * 4 + [None, None]
        assert lib.simsd_accept(*a) == 1
        assert lib.simsd_accept_noalloc(*n) == 1
    n = [None] * 4 + [0, 4, 4, 100, 1.0, 0, 0] + [None] * 4 + [None, None]
    assert lib.simsd_accept_noalloc(*n) == 0      # batch 0: nothing to do
    n[4] = 2
    assert lib.simsd_accept_noalloc(*n) == 1      # null pointers
    n[6] = 5
    assert lib.simsd_accept_noalloc(*n) == 1      # gamma > B
