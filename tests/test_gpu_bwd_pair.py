"""Backward on pairs of CTAs (fa_bwd_pair, d = 64) against the fp64 oracle.

The pair kernel shares every product between two thread blocks of a cluster
(256 keys per pair, B operands split between the blocks, dQ summed over the
pair's 256 keys before it is added into the workspace).  These tests run it
on the same inputs and bounds as the single-block backward: the GPU
forward's own O and LSE in, dQ, dK, dV within 1e-2 relative RMS of the exact
gradients, every element compared on the small and ragged problems (odd and
even numbers of key tiles, so that the last pair's second block holds no keys
or only some; odd numbers of query tiles, so that the last dQ product has
one query tile), whole sampled heads at the full-size d = 64 workload.
Outputs start as NaN inside guard bands and the workspace as garbage.
"""
import math

import numpy as np
import pytest

import exact_attention_74_gb300 as fa
import fa_inputs
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch
    assert torch.cuda.is_available()
    fa.library()
    return torch


def _forward(torch, w, qb, kb, vb):
    B, H, N_q, d = qb.shape
    N_kv = kb.shape[2]
    q, k, v = (gu.dev_bf16(x) for x in (qb, kb, vb))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N_q), dtype=torch.float32, device="cuda")
    st = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                   B, H, N_q, N_kv, d, int(w.causal), w.scale, 0)
    assert st == fa.FA_OK
    return q, k, v, o, lse


def _backward(torch, w, t, do, pair=True):
    q, k, v, o, lse = t
    B, H, N_q, d = q.shape
    N_kv = k.shape[2]
    dq = gu.Guarded((B, H, N_q, d), torch.bfloat16)
    dk = gu.Guarded((B, H, N_kv, d), torch.bfloat16)
    dv = gu.Guarded((B, H, N_kv, d), torch.bfloat16)
    need = fa.fa_bwd_workspace_bytes(B, H, N_q, N_kv, d)
    ws = gu.Guarded((need,), torch.uint8)
    ws.view.fill_(0xFF)
    fn = fa.fa_bwd_pair if pair else fa.fa_bwd
    st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
            dq.view.data_ptr(), dk.view.data_ptr(), dv.view.data_ptr(), B, H, N_q, N_kv, d, int(w.causal),
            w.scale, ws.view.data_ptr(), need, 0)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    assert fa.fa_get_last_device_status(0) == fa.FA_OK
    for g in (dq, dk, dv):
        assert g.guards_intact()
    return gu.to_f64(dq.view), gu.to_f64(dk.view), gu.to_f64(dv.view)


def _check(got, ref, what, tol=gu.GRAD_REL_RMS):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert np.all(np.isfinite(g)), f"{what}: non-finite {name}"
        e = gu.rel_rms(g, r)
        assert e <= tol, f"{what}: {name} rel-RMS {e:.3e} > {tol:.3e}"


def _wl(B, H, N_q, N_kv, causal, seed=7, kind="iid"):
    return fa_inputs.Workload(f"pair B{B}H{H}q{N_q}kv{N_kv}c{int(causal)}", B, H, N_q, N_kv, 64, causal,
                              1.0 / math.sqrt(64), seed, kind)


def full_compare(torch, w):
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)
    t = _forward(torch, w, qb, kb, vb)
    got = _backward(torch, w, t, gu.dev_bf16(dob))
    q, k, v, do = (fa_inputs.bf16_bits_to_f64(x) for x in (qb, kb, vb, dob))
    ref = oracle.attention_backward(q, k, v, do, causal=w.causal, scale=w.scale)
    _check(got, ref, w.name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [1, 17, 128, 129, 255, 256, 300, 384, 512, 640, 1000])
def test_ragged_square(torch, causal, n):
    full_compare(torch, _wl(1, 2, n, n, causal, seed=n + 3))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nkv", [(100, 300), (300, 100), (1, 513), (513, 1), (256, 384), (384, 256),
                                    (128, 640), (640, 128)])
def test_ragged_rectangular(torch, causal, nq, nkv):
    full_compare(torch, _wl(2, 1, nq, nkv, causal, seed=nq * 5 + nkv))


@pytest.mark.parametrize("causal", [False, True])
def test_many_heads(torch, causal):
    """B*H = 600 heads of 200 rows: many clusters, heads interleaved in a wave."""
    full_compare(torch, _wl(2, 300, 200, 200, causal, seed=31))


@pytest.mark.parametrize("causal", [False, True])
def test_agrees_with_single_block_backward(torch, causal):
    """Same inputs through fa_bwd and fa_bwd_pair: the two differ only in the
    order of fp32 additions (dQ is summed over 256 keys before its reduce-add),
    so they agree far below the tolerance against the oracle."""
    w = _wl(2, 3, 1024, 1024, causal, seed=5)
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)
    t = _forward(torch, w, qb, kb, vb)
    do = gu.dev_bf16(dob)
    a = _backward(torch, w, t, do, pair=True)
    b = _backward(torch, w, t, do, pair=False)
    for name, x, y in zip(("dQ", "dK", "dV"), a, b):
        e = gu.rel_rms(x, y)
        print(f"{w.name}: {name} pair vs single-block rel-RMS {e:.2e}")
        assert e <= 2e-3, f"{name}: {e:.3e}"
    # dK and dV are the same products over the same query tiles in the same
    # order (the pair only splits B's columns between the blocks): identical
    for name, x, y in zip(("dK", "dV"), a[1:], b[1:]):
        assert np.array_equal(x, y), f"{name}: pair and single-block results differ"


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes_against_single_block(torch, seed):
    """Seeded random shapes (batch, heads, query and key lengths, mask): the
    pair backward against the single-block one on the same inputs, dK and dV
    bit for bit, dQ within the reordering of its fp32 additions; and every
    gradient against the oracle on one head."""
    rng = np.random.default_rng(1000 + seed)
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 5))
    causal = bool(rng.integers(0, 2))
    N_q = int(rng.integers(1, 1300))
    N_kv = N_q if rng.integers(0, 2) else int(rng.integers(1, 1300))
    w = _wl(B, H, N_q, N_kv, causal, seed=2000 + seed)
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)
    t = _forward(torch, w, qb, kb, vb)
    do = gu.dev_bf16(dob)
    a = _backward(torch, w, t, do, pair=True)
    b = _backward(torch, w, t, do, pair=False)
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2]), w.name
    assert gu.rel_rms(a[0], b[0]) <= 1e-4, w.name
    bi, hi = B - 1, H - 1
    q, k, v, dO = (fa_inputs.bf16_bits_to_f64(x[bi, hi]) for x in (qb, kb, vb, dob))
    ref = oracle.head_backward(q, k, v, dO, causal=causal, scale=w.scale)
    _check((a[0][bi, hi], a[1][bi, hi], a[2][bi, hi]), ref, f"{w.name} b{bi} h{hi}")


def test_two_streams_at_once(torch):
    """Two pair calls on different streams (own workspaces, inputs and
    outputs) overlapping on the device: both equal to the same call made
    alone, dK and dV bit for bit (their order is fixed), dQ within the
    reordering of its fp32 additions."""
    ws_ = [_wl(1, 8, 2048, 2048, False, seed=71), _wl(1, 8, 2048, 2048, True, seed=72)]
    runs = []
    for w in ws_:
        qb, kb, vb = fa_inputs.make_qkv(w)
        t = _forward(torch, w, qb, kb, vb)
        do = gu.dev_bf16(fa_inputs.make_dout(w))
        runs.append((w, t, do, _backward(torch, w, t, do)))
    streams = [torch.cuda.Stream() for _ in runs]
    outs = []
    torch.cuda.synchronize()
    for (w, t, do, _), st in zip(runs, streams):
        q, k, v, o, lse = t
        B, H, N, d = q.shape
        dq, dk, dv = (torch.empty_like(x) for x in (q, k, v))
        need = fa.fa_bwd_workspace_bytes(B, H, N, N, d)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        with torch.cuda.stream(st):
            ws.fill_(0xFF)
            r = fa.fa_bwd_pair(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                               lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, N, d,
                               int(w.causal), w.scale, ws.data_ptr(), need, st.cuda_stream)
        assert r == fa.FA_OK
        outs.append((dq, dk, dv, ws))
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status(0) == fa.FA_OK
    for (w, _, _, alone), (dq, dk, dv, _) in zip(runs, outs):
        got = [gu.to_f64(x) for x in (dq, dk, dv)]
        assert np.array_equal(got[1], alone[1]) and np.array_equal(got[2], alone[2]), w.name
        assert gu.rel_rms(got[0], alone[0]) <= 1e-4, w.name


@pytest.mark.parametrize("causal", [False, True])
def test_full_size(torch, causal):
    """The d = 64 workload B2 H16 N8192 at full size: dQ, dK, dV of four whole
    heads (both batches, first and last heads among them) against the
    oracle's exact gradients."""
    w = fa_inputs.WORKLOADS["hdim64_8k"].with_(causal=causal)
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)
    t = _forward(torch, w, qb, kb, vb)
    dq, dk, dv = _backward(torch, w, t, gu.dev_bf16(dob))
    for b, h in ((0, 0), (0, 9), (1, 4), (1, 15)):
        q, k, v, do = (fa_inputs.bf16_bits_to_f64(x[b, h]) for x in (qb, kb, vb, dob))
        ref = oracle.head_backward(q, k, v, do, causal=w.causal, scale=w.scale)
        _check((dq[b, h], dk[b, h], dv[b, h]), ref, f"{w.name} c{int(causal)} b{b} h{h}")
