"""The C-ABI boundary, checked without a GPU.

* the shared library builds, loads, and exports every function that
  include/*.h declares (and the binding wraps exactly those);
* every argument error is reported with its status code before any CUDA
  call or launch (the pointers below are never dereferenced);
* valid calls on a machine without a usable sm_103 device fail loudly with a
  status code instead of computing anything elsewhere.

A call that passes every argument check would launch a kernel on the fake
pointers wherever an sm_103 device is present, so such tests are skipped
there: this file is for the host without a GPU.
"""
import ctypes
import os
import re

import pytest

import exact_attention_74_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("fa.h", "fa_testing.h")]
P = 0x10000          # a 16-byte aligned fake device address (never dereferenced)


def _has_sm103():
    try:
        import torch
        return torch.cuda.is_available() and torch.cuda.get_device_capability() == (10, 3)
    except Exception:
        return False


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fa.library_path):
        from exact_attention_74_gb300 import _build
        _build.build()
    return fa.library()


def _declared():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text))
    return names


def test_headers_declare_the_entry_points():
    names = _declared()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_bytes", "fa_get_last_device_status",
              "fa_status_string", "fa_fwd_ex", "fa_set_wait_timeout_ns"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    declared = _declared()
    assert declared == set(fa.EXPORTED_SYMBOLS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert fa.fa_status_string(fa.FA_OK) == "ok"
    for code in range(1, 7):
        assert fa.fa_status_string(code) not in ("ok", "unknown status")
    assert fa.fa_status_string(99) == "unknown status"


def _fwd(**over):
    a = dict(Q=P, K=P, V=P, O=P, LSE=P, B=1, H=1, N_q=128, N_kv=128, d=128, causal=0, scale=0.088)
    a.update(over)
    return fa.fa_fwd(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["N_q"],
                     a["N_kv"], a["d"], a["causal"], a["scale"], 0)


@pytest.mark.parametrize("over,code", [
    (dict(Q=None), fa.FA_ERR_INVALID), (dict(K=None), fa.FA_ERR_INVALID),
    (dict(V=None), fa.FA_ERR_INVALID), (dict(O=None), fa.FA_ERR_INVALID),
    (dict(LSE=None), fa.FA_ERR_INVALID),
    (dict(B=0), fa.FA_ERR_INVALID), (dict(H=0), fa.FA_ERR_INVALID),
    (dict(N_q=0), fa.FA_ERR_INVALID), (dict(N_kv=-5), fa.FA_ERR_INVALID),
    (dict(causal=2), fa.FA_ERR_INVALID), (dict(scale=0.0), fa.FA_ERR_INVALID),
    (dict(scale=-1.0), fa.FA_ERR_INVALID), (dict(scale=float("nan")), fa.FA_ERR_INVALID),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED), (dict(d=512), fa.FA_ERR_UNSUPPORTED),
    (dict(d=32), fa.FA_ERR_UNSUPPORTED),
    (dict(Q=P + 8), fa.FA_ERR_ALIGN), (dict(K=P + 2), fa.FA_ERR_ALIGN),
    (dict(V=P + 4), fa.FA_ERR_ALIGN), (dict(O=P + 8), fa.FA_ERR_ALIGN),
    (dict(LSE=P + 2), fa.FA_ERR_ALIGN),
])
def test_fwd_argument_errors(lib, over, code):
    assert _fwd(**over) == code


def test_fwd_ex_knob_errors(lib):
    def call(tau, emu):
        return fa.fa_fwd_ex(P, P, P, P, P, 1, 1, 64, 64, 64, 0, 0.125, tau, emu, 0)
    assert call(-1.0, -1) == fa.FA_ERR_INVALID
    assert call(17.0, -1) == fa.FA_ERR_INVALID
    assert call(float("nan"), -1) == fa.FA_ERR_INVALID
    assert call(8.0, 4) == fa.FA_ERR_INVALID
    assert call(8.0, 32) == fa.FA_ERR_INVALID


@pytest.mark.skipif(_has_sm103(), reason="would launch on the fake pointers")
def test_lse_needs_only_4_byte_alignment(lib):
    # passes every argument check, then fails only on the device check here
    st = _fwd(LSE=P + 4)
    assert st != fa.FA_ERR_ALIGN


def test_workspace_bytes(lib):
    # fp32 dQ accumulator + two fp32 row vectors padded to 128 rows + one counter per
    # 128-row tile + the ticket word, each part rounded up to 256 B
    assert fa.fa_bwd_workspace_bytes(2, 16, 8192, 8192, 128) == \
        2 * 16 * 8192 * (128 * 4 + 2 * 4) + 2 * 16 * 64 * 4 + 256
    assert fa.fa_bwd_workspace_bytes(1, 1, 3, 5, 64) == 768 + 2 * 512 + 256 + 256
    assert fa.fa_bwd_workspace_bytes(3, 1, 130, 5, 128) == 3 * 130 * 128 * 4 + 2 * 3 * 256 * 4 + 256 + 256
    assert fa.fa_bwd_workspace_bytes(1, 1, 0, 5, 64) == 0
    assert fa.fa_bwd_workspace_bytes(1, 1, 3, 5, 80) == 0
    assert fa.fa_bwd_workspace_bytes(1, 1, 3, 5, 256) == 0     # forward only at d = 256


def _bwd(ws_bytes=None, **over):
    a = dict(Q=P, K=P, V=P, O=P, dO=P, LSE=P, dQ=P, dK=P, dV=P, B=1, H=2, N_q=100, N_kv=90,
             d=64, causal=1, scale=0.125, ws=P)
    a.update(over)
    need = fa.fa_bwd_workspace_bytes(a["B"], a["H"], a["N_q"], a["N_kv"], a["d"])
    return fa.fa_bwd(a["Q"], a["K"], a["V"], a["O"], a["dO"], a["LSE"], a["dQ"], a["dK"], a["dV"],
                     a["B"], a["H"], a["N_q"], a["N_kv"], a["d"], a["causal"], a["scale"],
                     a["ws"], need if ws_bytes is None else ws_bytes, 0)


@pytest.mark.parametrize("over,code", [
    (dict(dO=None), fa.FA_ERR_INVALID), (dict(dQ=None), fa.FA_ERR_INVALID),
    (dict(dK=None), fa.FA_ERR_INVALID), (dict(dV=None), fa.FA_ERR_INVALID),
    (dict(LSE=None), fa.FA_ERR_INVALID), (dict(N_kv=0), fa.FA_ERR_INVALID),
    (dict(causal=-1), fa.FA_ERR_INVALID), (dict(d=100), fa.FA_ERR_UNSUPPORTED),
    (dict(d=256, ws_bytes=1 << 20), fa.FA_ERR_UNSUPPORTED),
    (dict(dO=P + 2), fa.FA_ERR_ALIGN), (dict(dK=P + 8), fa.FA_ERR_ALIGN),
    (dict(ws=None), fa.FA_ERR_WORKSPACE), (dict(ws=P + 16), fa.FA_ERR_ALIGN),
])
def test_bwd_argument_errors(lib, over, code):
    assert _bwd(**over) == code


def test_bwd_workspace_too_small(lib):
    need = fa.fa_bwd_workspace_bytes(1, 2, 100, 90, 64)
    assert _bwd(ws_bytes=need - 1) == fa.FA_ERR_WORKSPACE


def test_timeout_setting_bounds(lib):
    assert fa.fa_set_wait_timeout_ns(10) == fa.FA_ERR_INVALID
    assert fa.fa_set_wait_timeout_ns(10 ** 12) == fa.FA_ERR_INVALID
    assert fa.fa_set_wait_timeout_ns(10 ** 9) == fa.FA_OK


def test_testing_entry_point_argument_errors(lib):
    assert fa.fa_test_exp2(P, P, -1, 0, 0) == fa.FA_ERR_INVALID
    assert fa.fa_test_exp2(P, P, 10, 2, 0) == fa.FA_ERR_INVALID
    assert fa.fa_test_exp2(None, None, 0, 0, 0) == fa.FA_OK     # empty: launches nothing
    assert fa.fa_test_mma_tile(P, P, P, 96, 0, 0) == fa.FA_ERR_INVALID
    assert fa.fa_test_mma_tile(P, P, P, 64, 6, 0) == fa.FA_ERR_INVALID
    assert fa.fa_test_mma_tile(P, P, P, 64, -1, 0) == fa.FA_ERR_INVALID
    assert fa.fa_test_mma_tile(P + 8, P, P, 64, 0, 0) == fa.FA_ERR_ALIGN
    assert fa.fa_test_mma_pair(P, P, P, 96, 0, 0) == fa.FA_ERR_INVALID
    assert fa.fa_test_mma_pair(P, P, P, 64, 4, 0) == fa.FA_ERR_INVALID
    assert fa.fa_test_mma_pair(P, P, P, 64, -1, 0) == fa.FA_ERR_INVALID
    assert fa.fa_test_mma_pair(P, P + 8, P, 128, 0, 0) == fa.FA_ERR_ALIGN
    assert fa.fa_test_wait_timeout(5, 0) == fa.FA_ERR_INVALID


@pytest.mark.skipif(_has_sm103(), reason="only meaningful without an sm_103 device")
def test_valid_call_without_device_fails_loudly(lib):
    st = _fwd()
    assert st in (fa.FA_ERR_CUDA, fa.FA_ERR_UNSUPPORTED)
    assert fa.fa_get_last_device_status(0) in (fa.FA_ERR_CUDA, fa.FA_ERR_UNSUPPORTED)


def test_bwd_ex_deterministic_flag(lib):
    need = fa.fa_bwd_workspace_bytes(1, 2, 100, 90, 64)
    for bad in (-1, 2):
        assert fa.fa_bwd_ex(P, P, P, P, P, P, P, P, P, 1, 2, 100, 90, 64, 1, 0.125, bad, P, need, 0) \
            == fa.FA_ERR_INVALID
    # argument errors are fa_bwd's
    assert fa.fa_bwd_ex(P, P, P, P, P, P, P, P, P, 1, 2, 100, 90, 96, 1, 0.125, 1, P, need, 0) \
        == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_bwd_ex(P, P, P, P, P, P, P, P, P, 1, 2, 100, 90, 64, 1, 0.125, 1, P, need - 1, 0) \
        == fa.FA_ERR_WORKSPACE


def test_bwd_pair_argument_errors(lib):
    need = fa.fa_bwd_workspace_bytes(1, 2, 100, 90, 64)

    def call(d=64, ws=P, nbytes=need, dQ=P, causal=1, K=P):
        return fa.fa_bwd_pair(P, K, P, P, P, P, dQ, P, P, 1, 2, 100, 90, d, causal, 0.125, ws, nbytes, 0)

    # the pair kernel covers d = 64 only; the other argument errors are fa_bwd's
    assert call(d=128, nbytes=fa.fa_bwd_workspace_bytes(1, 2, 100, 90, 128)) == fa.FA_ERR_UNSUPPORTED
    assert call(d=256, nbytes=1 << 20) == fa.FA_ERR_UNSUPPORTED
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED
    assert call(dQ=None) == fa.FA_ERR_INVALID
    assert call(causal=2) == fa.FA_ERR_INVALID
    assert call(K=P + 8) == fa.FA_ERR_ALIGN
    assert call(ws=None) == fa.FA_ERR_WORKSPACE
    assert call(nbytes=need - 1) == fa.FA_ERR_WORKSPACE


def test_fp8_workspace_bytes(lib):
    # Q, K and V codes (rows padded to 128), the Q and K multipliers, the
    # block and head maxima of |V|, each rounded up to 256 bytes
    B, H, nq, nk = 2, 3, 200, 130
    r = lambda x: (x + 255) // 256 * 256
    want = (r(6 * 256 * 128) + r(6 * 256 * 128) + r(6 * 256 * 128) + r(6 * 2 * 4) + r(6 * 2 * 4)
            + r(6 * 2 * 4) + r(6 * 4))
    assert fa.fa_fwd_fp8_workspace_bytes(B, H, nq, nk, 128) == want
    assert fa.fa_fwd_fp8_workspace_bytes(B, H, nq, nk, 64) == 0
    want256 = (r(6 * 256 * 256) * 3 + r(6 * 2 * 4) * 3 + r(6 * 4))
    assert fa.fa_fwd_fp8_workspace_bytes(B, H, nq, nk, 256) == want256
    assert fa.fa_fwd_fp8_workspace_bytes(B, H, 0, nk, 128) == 0


def _fp8(ws_bytes=None, **over):
    a = dict(Q=P, K=P, V=P, O=P, LSE=P, B=1, H=2, N_q=100, N_kv=90, d=128, causal=0, scale=0.088,
             signs=[1, 2, 3, 4], ws=P)
    a.update(over)
    need = fa.fa_fwd_fp8_workspace_bytes(a["B"], a["H"], a["N_q"], a["N_kv"], 128)
    return fa.fa_fwd_fp8(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["N_q"], a["N_kv"],
                         a["d"], a["causal"], a["scale"], a["signs"], a["ws"],
                         need if ws_bytes is None else ws_bytes, 0)


@pytest.mark.parametrize("over,code", [
    (dict(Q=None), fa.FA_ERR_INVALID), (dict(LSE=None), fa.FA_ERR_INVALID),
    (dict(N_q=0), fa.FA_ERR_INVALID), (dict(causal=3), fa.FA_ERR_INVALID),
    (dict(scale=-1.0), fa.FA_ERR_INVALID), (dict(d=64), fa.FA_ERR_UNSUPPORTED),
    (dict(d=512), fa.FA_ERR_UNSUPPORTED), (dict(V=P + 8), fa.FA_ERR_ALIGN),
    (dict(ws=None), fa.FA_ERR_WORKSPACE), (dict(ws_bytes=1024), fa.FA_ERR_WORKSPACE),
    (dict(ws=P + 128), fa.FA_ERR_ALIGN),
])
def test_fp8_argument_errors(lib, over, code):
    assert _fp8(**over) == code


def test_fp8_signs_must_cover_d(lib):
    # d = 256 reads 8 sign words; the binding refuses a shorter list before
    # any call (the C side cannot know the length of a host array)
    with pytest.raises(ValueError):
        fa.fa_fwd_fp8(P, P, P, P, P, 1, 2, 100, 90, 256, 0, 0.06, [1, 2, 3, 4], P, 1 << 20, 0)
