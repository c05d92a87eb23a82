"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device memory.

Such callers (code handed only its input and output buffers by a host
framework, request paths where allocation is forbidden because it can fail
or synchronise the device) cannot pass fa_bwd a workspace.  fa_bwd_noalloc
uses scratch the library reserves when it is loaded instead.  These tests
call it through the C ABI and compare it with fa_bwd given its own workspace,
within the same 1e-2 relative-RMS tolerance the backward parity tests use,
on consecutive calls (the scratch keeps the previous call's contents, so
every call must clear what it needs).  The file is named to run last.
"""
import math

import numpy as np
import pytest

import exact_attention_74_gb300 as fa
import fa_inputs
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch
    assert torch.cuda.is_available()
    fa.library()
    return torch


def _problem(torch, B, H, N, d, causal, seed):
    w = fa_inputs.Workload(f"noalloc B{B}H{H}N{N}d{d}", B, H, N, N, d, causal, 1.0 / math.sqrt(d), seed)
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)
    q, k, v, do = (gu.dev_bf16(x) for x in (qb, kb, vb, dob))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    assert fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                     B, H, N, N, d, int(causal), w.scale, 0) == fa.FA_OK
    return w, (q, k, v, o, do, lse)


def _grads(torch, w, t, noalloc):
    q, k, v, o, do, lse = t
    dq, dk, dv = (torch.full_like(x, float("nan")) for x in (q, k, v))
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, w.N_q, w.N_kv, w.d, int(w.causal), w.scale)
    if noalloc:
        st = fa.fa_bwd_noalloc(*args, 0)
    else:
        need = fa.fa_bwd_workspace_bytes(w.B, w.H, w.N_q, w.N_kv, w.d)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        st = fa.fa_bwd(*args, ws.data_ptr(), need, 0)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    assert fa.fa_get_last_device_status(0) == fa.FA_OK
    return [gu.to_f64(x) for x in (dq, dk, dv)]


def test_noalloc_matches_fa_bwd_on_consecutive_calls(torch):
    # two calls in a row on one problem, then a call on a different, smaller
    # problem that reuses the scratch left behind by the larger one
    for (B, H, N, d, causal, seed, calls) in ((1, 4, 1000, 128, True, 71, 2), (2, 2, 300, 64, False, 72, 1)):
        w, t = _problem(torch, B, H, N, d, causal, seed)
        ref = _grads(torch, w, t, noalloc=False)
        assert fa.fa_bwd_workspace_bytes(B, H, N, N, d) <= fa.FA_BWD_NOALLOC_MAX_WORKSPACE
        for _ in range(calls):
            got = _grads(torch, w, t, noalloc=True)
            for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
                assert np.all(np.isfinite(g)), name
                assert gu.rel_rms(g, r) <= gu.GRAD_REL_RMS, (name, gu.rel_rms(g, r))


def test_noalloc_rejects_problems_beyond_its_scratch(torch):
    B, H, N, d = 1, 64, 1024, 128
    assert fa.fa_bwd_workspace_bytes(B, H, N, N, d) > fa.FA_BWD_NOALLOC_MAX_WORKSPACE
    x = torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    p = x.data_ptr()
    assert fa.fa_bwd_noalloc(p, p, p, p, p, lse.data_ptr(), p, p, p, B, H, N, N, d, 0, 0.088, 0) \
        == fa.FA_ERR_WORKSPACE
    # other argument errors are fa_bwd's own
    assert fa.fa_bwd_noalloc(p, p, p, p, p, lse.data_ptr(), p, p, p, 1, 1, 64, 64, 96, 0, 0.1, 0) \
        == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_get_last_device_status(0) == fa.FA_OK
