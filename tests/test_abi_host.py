"""Host-only checks of the C ABI (no GPU needed): the library loads, exports every symbol the public
header declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

from fp8_causal_prefill_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load_library()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "zyfa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zyfa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_abi():
    assert _declared_functions() == sorted(api.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_status_strings(lib):
    for code, name in api.STATUS.items():
        assert lib.zyfa_status_string(code).decode() == name
    assert lib.zyfa_status_string(99).decode() == "ZYFA_ERR_UNKNOWN"


def test_kernel_launch_count(lib):
    assert api.zyfa_kernel_launches(1, 32768, 32) == 1
    assert api.zyfa_kernel_launches(1, 0, 32) == 0


A = 1 << 20  # a 16-byte aligned fake address; validation rejects the calls before any dereference


@pytest.mark.parametrize("args,expect", [
    (dict(B=0), 1), (dict(H=0), 1), (dict(H_kv=0), 1), (dict(S=-1), 1),
    (dict(H=6, H_kv=4), 1), (dict(dtype=7), 1),
    (dict(scale=-1.0), 1), (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(D_qk=96, D_v=96), 2), (dict(D_qk=128, D_v=64), 2), (dict(D_qk=256, D_v=256), 2),
    (dict(q=A + 1), 3), (dict(k=A + 8), 3), (dict(v=A + 4), 3), (dict(out=A + 2), 3),
    (dict(q=0), 1), (dict(out=0), 1),
    (dict(S=0), 0), (dict(S=0, q=0, k=0, v=0, out=0), 0),
])
def test_argument_validation(lib, args, expect):
    a = dict(q=A, k=A, v=A, out=A, B=1, S=100, H=4, H_kv=2, D_qk=128, D_v=128, scale=0.0, dtype=0)
    a.update(args)
    st = api.zyfa_attn_fwd_causal(a["q"], a["k"], a["v"], a["out"], a["B"], a["S"], a["H"], a["H_kv"], a["D_qk"],
                                  a["D_v"], a["scale"], a["dtype"])
    assert st == expect, (args, api.STATUS.get(st))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(api, "_LIB_PATH", str(tmp_path / "libzyfa.so"))
    monkeypatch.setattr(api, "_lib", None)
    with pytest.raises(api.ZyfaError):
        api.load_library()


def test_options_validation(lib):
    import ctypes as ct
    bad_mode = api.FwdOptions(7, 0, None)
    st = lib.zyfa_attn_fwd_causal_ex(16, 16, 16, 16, 1, 8, 2, 2, 128, 128, 0.0, 0, None, None, None,
                                     ct.byref(bad_mode), None)
    assert st == 1
    bad_flag = api.FwdOptions(0, 2, None)
    st = lib.zyfa_attn_fwd_causal_ex(16, 16, 16, 16, 1, 8, 2, 2, 128, 128, 0.0, 0, None, None, None,
                                     ct.byref(bad_flag), None)
    assert st == 1
    odd_lse = api.FwdOptions(0, 0, 18)
    st = lib.zyfa_attn_fwd_causal_ex(16, 16, 16, 16, 1, 8, 2, 2, 128, 128, 0.0, 0, None, None, None,
                                     ct.byref(odd_lse), None)
    assert st == 3
    # S == 0 with valid options returns OK without touching the device
    for mode in (api.ZYFA_P_LEAN, api.ZYFA_P_EXACT, api.ZYFA_P_EXACT_NO_BLOCK_SCALE):
        ok = api.FwdOptions(mode, 1, None)
        assert lib.zyfa_attn_fwd_causal_ex(16, 16, 16, 16, 1, 0, 2, 2, 128, 128, 0.0, 0, None, None, None,
                                           ct.byref(ok), None) == 0
    bad_mode = api.FwdOptions(3, 0, None)
    assert lib.zyfa_attn_fwd_causal_ex(16, 16, 16, 16, 1, 0, 2, 2, 128, 128, 0.0, 0, None, None, None,
                                       ct.byref(bad_mode), None) == 1
