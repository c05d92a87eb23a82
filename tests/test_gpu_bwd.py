"""Backward parity: fa_bwd (through the C ABI) against the fp64 oracle's exact gradients.

The GPU backward consumes the GPU forward's own bf16 O and fp32 LSE; the
oracle differentiates <dO, O> at the same bf16 inputs in float64.  dQ, dK and
dV must each lie within 1e-2 relative RMS.  Small and ragged problems are
compared over every element; the full-size backward workload (B=2, H=16,
N=8192, d=128, causal) runs at full size and is compared on whole sampled
heads.  Outputs start as NaN inside guard bands, and the workspace starts
as garbage, so unwritten elements, stray writes and a missing clear all show.
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


def run_fwd_bwd(torch, w, qb, kb, vb, dob, fwd_out=None):
    B, H, N_q, d = qb.shape
    N_kv = kb.shape[2]
    q, k, v, do = (gu.dev_bf16(x) for x in (qb, kb, vb, dob))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N_q), dtype=torch.float32, device="cuda")
    st = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                   B, H, N_q, N_kv, d, int(w.causal), w.scale, 0)
    assert st == fa.FA_OK
    if fwd_out is not None:
        fwd_out.extend([gu.to_f64(o), lse.cpu().numpy().astype(np.float64)])
    dq = gu.Guarded((B, H, N_q, d), torch.bfloat16)
    dk = gu.Guarded((B, H, N_kv, d), torch.bfloat16)
    dv = gu.Guarded((B, H, N_kv, d), torch.bfloat16)
    need = fa.fa_bwd_workspace_bytes(B, H, N_q, N_kv, d)
    ws = gu.Guarded((need,), torch.uint8)
    ws.view.fill_(0xFF)                                   # garbage (NaN patterns) on entry
    st = fa.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                   lse.data_ptr(), dq.view.data_ptr(), dk.view.data_ptr(), dv.view.data_ptr(),
                   B, H, N_q, N_kv, d, int(w.causal), w.scale, ws.view.data_ptr(), need, 0)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    assert fa.fa_get_last_device_status(0) == fa.FA_OK
    for g in (dq, dk, dv):
        assert g.guards_intact()
    return gu.to_f64(dq.view), gu.to_f64(dk.view), gu.to_f64(dv.view)


def check_grads(got, ref, what, tols=(gu.GRAD_REL_RMS,) * 3):
    for name, g, r, tol in zip(("dQ", "dK", "dV"), got, ref, tols):
        assert np.all(np.isfinite(g)), f"{what}: non-finite {name}"
        e = gu.rel_rms(g, r)
        assert e <= tol, f"{what}: {name} rel-RMS {e:.3e} > {tol:.3e}"


def full_compare(torch, w):
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)
    got = run_fwd_bwd(torch, w, qb, kb, vb, dob)
    q, k, v, do = (fa_inputs.bf16_bits_to_f64(x) for x in (qb, kb, vb, dob))
    ref = oracle.attention_backward(q, k, v, do, causal=w.causal, scale=w.scale)
    check_grads(got, ref, w.name)


def _wl(B, H, N_q, N_kv, d, causal, seed=11, kind="iid"):
    return fa_inputs.Workload(f"bwd B{B}H{H}q{N_q}kv{N_kv}d{d}c{int(causal)}", B, H, N_q, N_kv, d,
                              causal, 1.0 / math.sqrt(d), seed, kind)


def test_many_heads(torch):
    """B*H = 80,000 heads (more than a grid's y or z extent) of 5 query rows
    and 7 keys, causal: every gradient of every head compared."""
    full_compare(torch, _wl(2, 40000, 5, 7, 64, True, seed=42))


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_d64(torch, causal):
    full_compare(torch, fa_inputs.WORKLOADS["tiny_causal" if causal else "tiny"])


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n", [1, 17, 128, 129, 300, 640])
def test_ragged_square(torch, d, causal, n):
    full_compare(torch, _wl(1, 2, n, n, d, causal, seed=n + d))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nkv", [(100, 300), (300, 100), (1, 513), (513, 1), (256, 384)])
def test_ragged_rectangular(torch, d, causal, nq, nkv):
    full_compare(torch, _wl(2, 1, nq, nkv, d, causal, seed=nq * 3 + nkv))


@pytest.mark.parametrize("causal", [False, True])
def test_medium_multi_head(torch, causal):
    full_compare(torch, _wl(2, 3, 1024, 1024, 128, causal, seed=5))


def test_stress_inputs_from_saved_outputs(torch):
    """Near-one-hot rows: both sides get the oracle's O (rounded to bf16) and LSE (fp32).

    There dP - D nearly cancels, so the gradient depends on the saved O's
    rounding; comparing against the exact gradient would measure the bf16
    storage of O rather than the kernel.  Here the oracle applies the same
    saved-output formulas to the same saved inputs.
    """
    w = fa_inputs.WORKLOADS["stress_8k"].with_(B=1, H=2, N_q=1024, N_kv=1024)
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)
    q, k, v, do = (fa_inputs.bf16_bits_to_f64(x) for x in (qb, kb, vb, dob))
    o_ref, lse_ref = oracle.attention_forward(q, k, v, causal=w.causal, scale=w.scale)
    ob = fa_inputs.f32_to_bf16_bits(o_ref.astype(np.float32))
    lse32 = lse_ref.astype(np.float32)
    B, H, N, d = qb.shape
    tq, tk, tv, tdo, to = (gu.dev_bf16(x) for x in (qb, kb, vb, dob, ob))
    tl = torch.from_numpy(lse32).cuda()
    dq, dk, dv = (torch.empty_like(tq) for _ in range(3))
    need = fa.fa_bwd_workspace_bytes(B, H, N, N, d)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = fa.fa_bwd(tq.data_ptr(), tk.data_ptr(), tv.data_ptr(), to.data_ptr(), tdo.data_ptr(), tl.data_ptr(),
                   dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, N, d, 1, w.scale,
                   ws.data_ptr(), need, 0)
    assert st == fa.FA_OK and fa.fa_get_last_device_status(0) == fa.FA_OK
    o_saved = fa_inputs.bf16_bits_to_f64(ob)
    lse_saved = lse32.astype(np.float64)
    for h in range(H):
        ref = oracle.head_backward_from_saved(q[0, h], k[0, h], v[0, h], o_saved[0, h], do[0, h],
                                              lse_saved[0, h], causal=True, scale=w.scale)
        tols = [max(gu.GRAD_REL_RMS, 2 * 2.0 ** -9 / math.sqrt(3) * c)
                for c in _conditioning(q[0, h], k[0, h], v[0, h], o_saved[0, h], do[0, h],
                                       lse_saved[0, h], w.scale)]
        check_grads((gu.to_f64(dq)[0, h], gu.to_f64(dk)[0, h], gu.to_f64(dv)[0, h]), ref,
                    f"stress h{h}", tols)


def _conditioning(q, k, v, o, do, lse, scale):
    """Frobenius condition numbers ||(|A||B|)|| / ||A B|| of the three gradient products.

    The kernel stores P and dS in bf16 (unit roundoff 2^-9, RMS 2^-9/sqrt(3)
    for round-to-nearest) before the dV, dK and dQ products; the relative RMS
    error those roundings cause grows with this ratio, which is large when
    sum_j dS_ij nearly cancels against keys with a large common component.
    """
    n = q.shape[0]
    s = scale * q @ k.T
    s = np.where(np.tril(np.ones((n, k.shape[0]))) > 0, s, -np.inf)
    p = np.exp(s - lse[:, None])
    ds = p * (do @ v.T - np.sum(do * o, axis=1)[:, None])
    def kappa(a, b):
        return np.linalg.norm(np.abs(a) @ np.abs(b)) / np.linalg.norm(a @ b)
    return kappa(ds, k), kappa(ds.T, q), kappa(p.T, do)


def test_full_size_backward(torch):
    """The backward workload B2 H16 N8192 d128 causal at full size: its
    forward (O, LSE) on sampled rows of all 32 heads under the stated bounds
    and the per-element arithmetic bound, then dQ, dK, dV of 8 whole heads
    (both batches, first and last heads among them) against the oracle's exact
    gradients."""
    w = fa_inputs.WORKLOADS["bwd_8k"]
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)
    fwd_out = []
    dq, dk, dv = run_fwd_bwd(torch, w, qb, kb, vb, dob, fwd_out)
    o, lse = fwd_out
    rng = np.random.default_rng(w.seed + 99)
    got, ref, got_l, ref_l, sps = [], [], [], [], []
    for b in range(w.B):
        for h in range(w.H):
            rows = gu.sample_rows(w.N_q, 32, rng)
            o_ref, lse_ref, sp = gu.oracle_rows(qb, kb, vb, b, h, rows, True, w.scale, with_spread=True)
            got.append(o[b, h][rows]); ref.append(o_ref); sps.append(sp)
            got_l.append(lse[b, h][rows]); ref_l.append(lse_ref)
    gu.assert_o_lse(np.concatenate(got), np.concatenate(got_l), np.concatenate(ref), np.concatenate(ref_l),
                    f"{w.name} forward (32 heads x 40 rows)", spread_=np.concatenate(sps))
    for b, h in ((0, 0), (0, 5), (0, 10), (0, 15), (1, 0), (1, 6), (1, 13), (1, 15)):
        q, k, v, do = (fa_inputs.bf16_bits_to_f64(x[b, h]) for x in (qb, kb, vb, dob))
        ref = oracle.head_backward(q, k, v, do, causal=w.causal, scale=w.scale)
        check_grads((dq[b, h], dk[b, h], dv[b, h]), ref, f"{w.name} b{b} h{h}")


@pytest.mark.parametrize("causal", [False, True])
def test_many_heads_d64(torch, causal):
    """d = 64 on B*H = 600 heads of 200 rows: many CTAs of the unordered d = 64
    kernel in flight, heads interleaved in a wave, a ragged last tile."""
    full_compare(torch, _wl(2, 300, 200, 200, 64, causal, seed=31))


@pytest.mark.parametrize("causal", [False, True])
def test_full_size_d64(torch, causal):
    """The d = 64 workload B2 H16 N8192 at full size through fa_bwd (the
    unordered d = 64 kernel: every intermediate in its own tensor-memory
    columns, products on two issuing threads): dQ, dK, dV of four whole heads
    (both batches, first and last heads among them) against the oracle's exact
    gradients."""
    w = fa_inputs.WORKLOADS["hdim64_8k"].with_(causal=causal)
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)
    dq, dk, dv = run_fwd_bwd(torch, w, qb, kb, vb, dob)
    for b, h in ((0, 0), (0, 9), (1, 4), (1, 15)):
        q, k, v, do = (fa_inputs.bf16_bits_to_f64(x[b, h]) for x in (qb, kb, vb, dob))
        ref = oracle.head_backward(q, k, v, do, causal=w.causal, scale=w.scale)
        check_grads((dq[b, h], dk[b, h], dv[b, h]), ref, f"{w.name} c{int(causal)} b{b} h{h}")


# ----------------------------------------------------------- deterministic mode

def _bwd_ex(torch, w, t, deterministic):
    q, k, v, o, do, lse = t
    dq, dk, dv = (torch.full_like(x, float("nan")) for x in (q, k, v))
    need = fa.fa_bwd_workspace_bytes(w.B, w.H, w.N_q, w.N_kv, w.d)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)
    st = fa.fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                      dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, w.N_q, w.N_kv, w.d,
                      int(w.causal), w.scale, deterministic, ws.data_ptr(), need, 0)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    assert fa.fa_get_last_device_status(0) == fa.FA_OK
    return dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nkv", [(1000, 1000), (700, 300), (300, 700)])
def test_deterministic_bitwise_repeatable_and_exact(torch, d, causal, nq, nkv):
    w = _wl(2, 3, nq, nkv, d, causal, seed=nq + 7 * nkv + d)
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)
    q, k, v, do = (gu.dev_bf16(x) for x in (qb, kb, vb, dob))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, nq), dtype=torch.float32, device="cuda")
    assert fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                     w.B, w.H, nq, nkv, d, int(causal), w.scale, 0) == fa.FA_OK
    t = (q, k, v, o, do, lse)
    a = _bwd_ex(torch, w, t, 1)
    b = _bwd_ex(torch, w, t, 1)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    ref = oracle.attention_backward(*(fa_inputs.bf16_bits_to_f64(x) for x in (qb, kb, vb, dob)),
                                    causal=causal, scale=w.scale)
    check_grads([gu.to_f64(x) for x in a], ref, f"deterministic {w.name}")


@pytest.mark.parametrize("d", [64, 128])
def test_deterministic_head_groups(torch, d):
    """Without a mask the fixed-order mode dispatches heads in groups of 16,
    interleaved key tile by key tile; 22 heads make one full group and one
    of 6, and 700 keys six key tiles: every head compared, bit-identical
    across calls."""
    w = _wl(2, 11, 700, 700, d, False, seed=97 + d)
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)
    q, k, v, do = (gu.dev_bf16(x) for x in (qb, kb, vb, dob))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N_q), dtype=torch.float32, device="cuda")
    assert fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                     w.B, w.H, w.N_q, w.N_kv, d, 0, w.scale, 0) == fa.FA_OK
    t = (q, k, v, o, do, lse)
    a = _bwd_ex(torch, w, t, 1)
    b = _bwd_ex(torch, w, t, 1)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    ref = oracle.attention_backward(*(fa_inputs.bf16_bits_to_f64(x) for x in (qb, kb, vb, dob)),
                                    causal=False, scale=w.scale)
    check_grads([gu.to_f64(x) for x in a], ref, f"deterministic {w.name}")


def test_deterministic_full_size_noncausal(torch):
    """The bench workload (64 heads: four groups of 16) in the fixed-order
    mode: bit-identical across four calls, and two heads against the oracle."""
    w = fa_inputs.WORKLOADS["fwd_4k"]
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)
    q, k, v, do = (gu.dev_bf16(x) for x in (qb, kb, vb, dob))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N_q), dtype=torch.float32, device="cuda")
    assert fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                     w.B, w.H, w.N_q, w.N_kv, w.d, 0, w.scale, 0) == fa.FA_OK
    t = (q, k, v, o, do, lse)
    a = _bwd_ex(torch, w, t, 1)
    for _ in range(3):
        b = _bwd_ex(torch, w, t, 1)
        for x, y in zip(a, b):
            assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    for bi, hi in ((0, 0), (3, 15)):
        q64, k64, v64, do64 = (fa_inputs.bf16_bits_to_f64(x[bi, hi]) for x in (qb, kb, vb, dob))
        ref = oracle.head_backward(q64, k64, v64, do64, causal=False, scale=w.scale)
        check_grads([gu.to_f64(x)[bi, hi] for x in a], ref, f"deterministic fwd_4k b{bi} h{hi}")


def test_deterministic_full_size_causal(torch):
    w = fa_inputs.WORKLOADS["bwd_8k"]
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)
    q, k, v, do = (gu.dev_bf16(x) for x in (qb, kb, vb, dob))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N_q), dtype=torch.float32, device="cuda")
    assert fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                     w.B, w.H, w.N_q, w.N_kv, w.d, 1, w.scale, 0) == fa.FA_OK
    t = (q, k, v, o, do, lse)
    a = _bwd_ex(torch, w, t, 1)
    for _ in range(3):
        b = _bwd_ex(torch, w, t, 1)
        for x, y in zip(a, b):
            assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    got = [gu.to_f64(x) for x in a]
    for bi, hi in ((0, 0), (0, 11), (1, 5), (1, 15)):
        q64, k64, v64, do64 = (fa_inputs.bf16_bits_to_f64(x[bi, hi]) for x in (qb, kb, vb, dob))
        ref = oracle.head_backward(q64, k64, v64, do64, causal=True, scale=w.scale)
        check_grads([g[bi, hi] for g in got], ref, f"deterministic bwd_8k b{bi} h{hi}")


def test_deterministic_beside_a_concurrent_kernel(torch):
    """The fixed-order backward while another stream keeps SMs busy with long
    forward launches of this library: its thread blocks then start in an
    order the hardware picks around the other kernel's.  Every wait must
    still end (FA_OK), and the gradients must equal, bit for bit, those of a
    call with the GPU to itself."""
    w = _wl(2, 8, 2048, 2048, 128, False, seed=123)
    qb, kb, vb = fa_inputs.make_qkv(w)
    dob = fa_inputs.make_dout(w)
    q, k, v, do = (gu.dev_bf16(x) for x in (qb, kb, vb, dob))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N_q), dtype=torch.float32, device="cuda")
    assert fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                     w.B, w.H, w.N_q, w.N_kv, w.d, 0, w.scale, 0) == fa.FA_OK
    solo = _bwd_ex(torch, w, (q, k, v, o, do, lse), 1)
    # the other kernel: forward launches on 2 x 16 heads of 8192 rows (~1 ms each)
    bq = torch.randn((2, 16, 8192, 128), device="cuda").to(torch.bfloat16)
    bo = torch.empty_like(bq)
    bl = torch.empty((2, 16, 8192), dtype=torch.float32, device="cuda")
    need = fa.fa_bwd_workspace_bytes(w.B, w.H, w.N_q, w.N_kv, w.d)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    s_other, s_bwd = torch.cuda.Stream(), torch.cuda.Stream()
    for rep in range(3):
        dq, dk, dv = (torch.full_like(x, float("nan")) for x in (q, k, v))
        for _ in range(4):
            assert fa.fa_fwd(bq.data_ptr(), bq.data_ptr(), bq.data_ptr(), bo.data_ptr(), bl.data_ptr(),
                             2, 16, 8192, 8192, 128, 0, 0.088, s_other.cuda_stream) == fa.FA_OK
        st = fa.fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                          dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, w.N_q, w.N_kv, w.d, 0,
                          w.scale, 1, ws.data_ptr(), need, s_bwd.cuda_stream)
        assert st == fa.FA_OK
        torch.cuda.synchronize()
        assert fa.fa_get_last_device_status(0) == fa.FA_OK, f"rep {rep}: a wait ran out"
        for x, y in zip((dq, dk, dv), solo):
            assert torch.equal(x.view(torch.int16), y.view(torch.int16)), f"rep {rep}"


def test_d64_backward_and_d256_forward_on_two_streams(torch):
    """The unordered d = 64 backward (two issuing threads) and the d = 256
    forward (two issuing threads) running at the same time on two streams, each
    equal to the same call made alone: O, dK and dV bit for bit, dQ within the
    reordering of its fp32 additions."""
    w64 = _wl(2, 8, 2048, 2048, 64, True, seed=81)
    w256 = _wl(1, 8, 2048, 2048, 256, False, seed=82)
    ins = {}
    for w in (w64, w256):
        qb, kb, vb = fa_inputs.make_qkv(w)
        ins[w.d] = tuple(gu.dev_bf16(x) for x in (qb, kb, vb)) + (gu.dev_bf16(fa_inputs.make_dout(w)),)
    q, k, v, do = ins[64]
    o64, lse64 = fa.forward(q, k, v, causal=True)
    alone_bwd = fa.backward(q, k, v, o64, do, lse64, causal=True)
    q2, k2, v2, _ = ins[256]
    alone_fwd, _ = fa.forward(q2, k2, v2)
    torch.cuda.synchronize()
    ws = torch.empty(fa.fa_bwd_workspace_bytes(2, 8, 2048, 2048, 64), dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(3):
        with torch.cuda.stream(s1):
            got_bwd = fa.backward(q, k, v, o64, do, lse64, causal=True, workspace=ws, stream=s1)
        with torch.cuda.stream(s2):
            got_fwd, _ = fa.forward(q2, k2, v2, stream=s2)
        torch.cuda.synchronize()
        assert fa.fa_get_last_device_status(0) == fa.FA_OK
        assert torch.equal(got_fwd.view(torch.int16), alone_fwd.view(torch.int16))
        for name, x, y in zip(("dQ", "dK", "dV"), got_bwd, alone_bwd):
            if name == "dQ":
                assert gu.rel_rms(gu.to_f64(x), gu.to_f64(y)) <= 1e-4
            else:
                assert torch.equal(x.view(torch.int16), y.view(torch.int16)), name
