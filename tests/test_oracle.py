"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: closed
forms worked by hand, invariants of the softmax definition, a brute-force
pure-Python restatement, PyTorch's math SDPA in float64 (the MATH backend named
in "FlashAttention: GPUメモリ階層を活用したアテンション最適化の分析" §11.2),
finite differences, and the printed exp2 coefficients.  The cases are chosen
so that a dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one of them (see the planted-mistake tests at the end).
"""
import json
import math
import os

import numpy as np
import pytest

import fa_inputs
import oracle
from oracle import attention as orc

pytestmark = pytest.mark.oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, *shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------- forward pins

@pytest.mark.parametrize("causal", [False, True])
def test_rows_sum_to_one(causal):
    rng = np.random.default_rng(1)
    q, k = _rand(rng, 37, 16), _rand(rng, 53, 16)
    p, _, _ = orc.softmax_probs(q, k, causal=causal, scale=0.3)
    assert np.max(np.abs(p.sum(axis=1) - 1.0)) <= 1e-12
    if causal:
        assert np.all(p[np.triu_indices(37, 1, 53)] == 0.0)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_returns_that_row(causal):
    rng = np.random.default_rng(2)
    q, k = _rand(rng, 1, 1, 40, 8), _rand(rng, 1, 1, 40, 8)
    row = _rand(rng, 8)
    v = np.broadcast_to(row, (1, 1, 40, 8)).copy()
    o, _ = oracle.attention_forward(q, k, v, causal=causal, scale=0.5)
    assert np.max(np.abs(o - row)) <= 1e-12


def test_single_key():
    rng = np.random.default_rng(3)
    q, k, v = _rand(rng, 1, 2, 9, 6), _rand(rng, 1, 2, 1, 6), _rand(rng, 1, 2, 1, 6)
    for causal in (False, True):
        o, lse = oracle.attention_forward(q, k, v, causal=causal, scale=0.7)
        assert np.max(np.abs(o - v)) <= 1e-12
        expect = 0.7 * np.einsum("bhnd,bhd->bhn", q, k[:, :, 0])
        assert np.max(np.abs(lse - expect)) <= 1e-12


def test_key_value_permutation_invariance():
    rng = np.random.default_rng(4)
    q, k, v = _rand(rng, 2, 2, 17, 8), _rand(rng, 2, 2, 23, 8), _rand(rng, 2, 2, 23, 8)
    perm = rng.permutation(23)
    o1, l1 = oracle.attention_forward(q, k, v, causal=False, scale=0.4)
    o2, l2 = oracle.attention_forward(q, k[:, :, perm], v[:, :, perm], causal=False, scale=0.4)
    assert np.max(np.abs(o1 - o2)) <= 1e-12
    assert np.max(np.abs(l1 - l2)) <= 1e-12


def _hadamard(n):
    h = np.array([[1.0]])
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


@pytest.mark.parametrize("which", ["qr", "hadamard"])
@pytest.mark.parametrize("causal", [False, True])
def test_orthogonal_rotation_invariance(which, causal):
    """(QM)(KM)^T = QK^T for orthogonal M (incoherent processing, FlashAttention-3 notes §技術 3)."""
    rng = np.random.default_rng(5)
    d = 16
    q, k, v = _rand(rng, 1, 2, 30, d), _rand(rng, 1, 2, 30, d), _rand(rng, 1, 2, 30, d)
    if which == "qr":
        m, _ = np.linalg.qr(rng.standard_normal((d, d)))
    else:
        m = (_hadamard(d) * rng.choice([-1.0, 1.0], size=d)[None, :]) / math.sqrt(d)
    assert np.max(np.abs(m @ m.T - np.eye(d))) <= 1e-12
    o1, l1 = oracle.attention_forward(q, k, v, causal=causal, scale=0.25)
    o2, l2 = oracle.attention_forward(q @ m, k @ m, v, causal=causal, scale=0.25)
    assert np.max(np.abs(o1 - o2)) <= 1e-11
    assert np.max(np.abs(l1 - l2)) <= 1e-11


def test_closed_form_two_keys():
    """s = [0, ln 3] -> P = [1/4, 3/4], LSE = ln 4 (worked by hand from the definition)."""
    q = np.array([[[[math.log(3.0)]]]])
    k = np.array([[[[0.0], [1.0]]]])
    v = np.array([[[[2.0, -1.0], [6.0, 3.0]]]])
    p, _, _ = orc.softmax_probs(q[0, 0], k[0, 0], causal=False, scale=1.0)
    assert np.allclose(p, [[0.25, 0.75]], atol=1e-15, rtol=0)
    o, lse = oracle.attention_forward(q, k, v, causal=False, scale=1.0)
    assert np.allclose(o[0, 0, 0], [0.25 * 2 + 0.75 * 6, 0.25 * -1 + 0.75 * 3], atol=1e-14, rtol=0)
    assert abs(lse[0, 0, 0] - math.log(4.0)) <= 1e-15


def test_closed_form_zero_queries():
    """Q = 0 -> every score 0 -> O = mean of V over the allowed keys, LSE = ln(count)."""
    rng = np.random.default_rng(6)
    q = np.zeros((1, 1, 12, 4))
    k, v = _rand(rng, 1, 1, 12, 4), _rand(rng, 1, 1, 12, 4)
    o, lse = oracle.attention_forward(q, k, v, causal=False, scale=1.0)
    assert np.max(np.abs(o[0, 0] - v[0, 0].mean(axis=0))) <= 1e-14
    assert np.max(np.abs(lse - math.log(12))) <= 1e-14
    o, lse = oracle.attention_forward(q, k, v, causal=True, scale=1.0)
    for i in range(12):
        assert np.max(np.abs(o[0, 0, i] - v[0, 0, :i + 1].mean(axis=0))) <= 1e-14
        assert abs(lse[0, 0, i] - math.log(i + 1)) <= 1e-14


def test_causal_first_row_sees_only_key_zero():
    rng = np.random.default_rng(7)
    q, k, v = _rand(rng, 1, 1, 5, 3), _rand(rng, 1, 1, 5, 3), _rand(rng, 1, 1, 5, 3)
    o, lse = oracle.attention_forward(q, k, v, causal=True, scale=1.3)
    assert np.max(np.abs(o[0, 0, 0] - v[0, 0, 0])) <= 1e-15
    assert abs(lse[0, 0, 0] - 1.3 * q[0, 0, 0] @ k[0, 0, 0]) <= 1e-14


def _brute(q, k, v, causal, scale):
    """Triple loop with math.exp: the standard attention of §2.1, one element at a time."""
    n_q, d = len(q), len(q[0])
    n_kv = len(k)
    out, lses = [], []
    for i in range(n_q):
        keys = [j for j in range(n_kv) if (not causal or j <= i)]
        s = {j: scale * sum(q[i][c] * k[j][c] for c in range(d)) for j in keys}
        mx = max(s.values())
        w = {j: math.exp(s[j] - mx) for j in keys}
        tot = sum(w.values())
        out.append([sum(w[j] / tot * v[j][c] for j in keys) for c in range(len(v[0]))])
        lses.append(mx + math.log(tot))
    return np.array(out), np.array(lses)


@pytest.mark.parametrize("n_q,n_kv,d,causal", [
    (1, 1, 1, False), (5, 5, 3, False), (5, 5, 3, True), (8, 3, 4, True),
    (3, 8, 4, True), (7, 6, 2, False), (8, 8, 4, True)])
def test_brute_force_tiny(n_q, n_kv, d, causal):
    rng = np.random.default_rng(100 + n_q * 10 + n_kv + d)
    q, k, v = _rand(rng, n_q, d), _rand(rng, n_kv, d), _rand(rng, n_kv, d)
    o, lse = orc.head_forward(q, k, v, causal=causal, scale=0.9)
    ob, lb = _brute(q.tolist(), k.tolist(), v.tolist(), causal, 0.9)
    assert np.max(np.abs(o - ob)) <= 1e-13
    assert np.max(np.abs(lse - lb)) <= 1e-13


# ------------------------------------------------------- library cross-check

torch = pytest.importorskip("torch")


def _sdpa(q, k, v, causal, scale):
    import torch.nn.functional as F
    from torch.nn.attention import SDPBackend, sdpa_kernel
    with sdpa_kernel(SDPBackend.MATH):
        return F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale)


@pytest.mark.parametrize("n_q,n_kv,causal", [(33, 33, False), (33, 33, True),
                                             (20, 45, True), (45, 20, True), (64, 17, False)])
def test_against_torch_math_sdpa_float64(n_q, n_kv, causal):
    rng = np.random.default_rng(8)
    q, k, v = _rand(rng, 2, 3, n_q, 16), _rand(rng, 2, 3, n_kv, 16), _rand(rng, 2, 3, n_kv, 16)
    do = _rand(rng, 2, 3, n_q, 16)
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    to = _sdpa(tq, tk, tv, causal, 0.3)
    to.backward(torch.tensor(do))
    o, _ = oracle.attention_forward(q, k, v, causal=causal, scale=0.3)
    assert np.max(np.abs(o - to.detach().numpy())) <= 1e-12
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal=causal, scale=0.3)
    assert np.max(np.abs(dq - tq.grad.numpy())) <= 1e-11
    assert np.max(np.abs(dk - tk.grad.numpy())) <= 1e-11
    assert np.max(np.abs(dv - tv.grad.numpy())) <= 1e-11


def test_lse_against_torch_logsumexp():
    rng = np.random.default_rng(9)
    q, k, v = _rand(rng, 1, 2, 19, 8), _rand(rng, 1, 2, 31, 8), _rand(rng, 1, 2, 31, 8)
    for causal in (False, True):
        s = 0.5 * torch.tensor(q) @ torch.tensor(k).transpose(-1, -2)
        if causal:
            s = s.masked_fill(~torch.ones(19, 31, dtype=torch.bool).tril(), float("-inf"))
        ref = torch.logsumexp(s, dim=-1).numpy()
        _, lse = oracle.attention_forward(q, k, v, causal=causal, scale=0.5)
        assert np.max(np.abs(lse - ref)) <= 1e-12


# -------------------------------------------------------------- backward pins

def test_backward_finite_differences():
    rng = np.random.default_rng(10)
    q, k, v, do = (_rand(rng, 12, 5) for _ in range(4))
    for causal in (False, True):
        dq, dk, dv = orc.head_backward(q, k, v, do, causal=causal, scale=0.8)

        def loss(qq, kk, vv):
            o, _ = orc.head_forward(qq, kk, vv, causal=causal, scale=0.8)
            return float(np.sum(o * do))

        h = 1e-6
        for name, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            for idx in [(0, 0), (3, 2), (11, 4), (7, 1)]:
                a_p, a_m = arr.copy(), arr.copy()
                a_p[idx] += h
                a_m[idx] -= h
                args_p = {"q": q, "k": k, "v": v}
                args_m = dict(args_p)
                args_p[name], args_m[name] = a_p, a_m
                fd = (loss(**{"qq": args_p["q"], "kk": args_p["k"], "vv": args_p["v"]}) -
                      loss(**{"qq": args_m["q"], "kk": args_m["k"], "vv": args_m["v"]})) / (2 * h)
                assert abs(fd - grad[idx]) <= 1e-7, (name, idx, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_sum_identities(causal):
    rng = np.random.default_rng(11)
    q, k, v, do = (_rand(rng, 2, 2, 29, 8) for _ in range(4))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal=causal, scale=0.35)
    # rows of P sum to one -> sum_j dV_j = sum_i dO_i
    assert np.max(np.abs(dv.sum(axis=2) - do.sum(axis=2))) <= 1e-11
    # O is unchanged by a common shift of all keys -> sum_j dK_j = 0
    assert np.max(np.abs(dk.sum(axis=2))) <= 1e-11


def test_backward_identical_keys_give_zero_dq():
    rng = np.random.default_rng(12)
    q, v, do = _rand(rng, 1, 1, 14, 6), _rand(rng, 1, 1, 14, 6), _rand(rng, 1, 1, 14, 6)
    k = np.broadcast_to(_rand(rng, 6), (1, 1, 14, 6)).copy()
    for causal in (False, True):
        dq, _, _ = oracle.attention_backward(q, k, v, do, causal=causal, scale=0.6)
        assert np.max(np.abs(dq)) <= 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_backward_from_saved_outputs_equals_exact_gradient(causal):
    """Fed the exact O and LSE, the saved-output backward is the exact gradient."""
    rng = np.random.default_rng(16)
    q, k, v, do = _rand(rng, 40, 8), _rand(rng, 40, 8), _rand(rng, 40, 8), _rand(rng, 40, 8)
    o, lse = orc.head_forward(q, k, v, causal=causal, scale=0.45)
    a = orc.head_backward_from_saved(q, k, v, o, do, lse, causal=causal, scale=0.45)
    b = orc.head_backward(q, k, v, do, causal=causal, scale=0.45)
    for x, y in zip(a, b):
        assert np.max(np.abs(x - y)) <= 1e-12
    # and it really uses the given O: a shifted O changes dQ and dK but not dV
    a2 = orc.head_backward_from_saved(q, k, v, o + 0.01, do, lse, causal=causal, scale=0.45)
    assert np.max(np.abs(a2[0] - a[0])) > 1e-6 and np.max(np.abs(a2[2] - a[2])) <= 1e-12


# ------------------------------------------------ tiled algorithm equivalence

@pytest.mark.parametrize("tau", [0.0, 8.0, math.inf])
@pytest.mark.parametrize("causal", [False, True])
def test_online_softmax_equals_definition(tau, causal):
    """The recurrences of §6.2 with conditional rescaling are exact for any tau."""
    rng = np.random.default_rng(13)
    q, k, v = _rand(rng, 150, 32), _rand(rng, 300, 32), _rand(rng, 300, 32)
    q[:, 3] *= 6.0   # wide logit spread so the maximum moves between blocks
    k[:, 3] *= 6.0
    o1, l1 = orc.head_forward(q, k, v, causal=causal, scale=0.2)
    o2, l2 = orc.online_softmax_forward(q, k, v, causal=causal, scale=0.2,
                                        block_kv=64, tau=tau)
    assert np.max(np.abs(o1 - o2)) <= 1e-12
    assert np.max(np.abs(l1 - l2)) <= 1e-12


def test_stress_recipe_moves_the_running_max():
    """The stress inputs make the row max jump by more than tau=8 (log2) many times."""
    w = fa_inputs.WORKLOADS["stress_8k"].with_(B=1, H=1, N_q=1024, N_kv=1024)
    qb, kb, _ = fa_inputs.make_qkv(w)
    q = fa_inputs.bf16_bits_to_f64(qb)[0, 0]
    k = fa_inputs.bf16_bits_to_f64(kb)[0, 0]
    t = w.scale / math.log(2.0) * (q[-64:] @ k.T)
    blk_max = np.stack([t[:, j:j + 128].max(axis=1) for j in range(0, 1024, 128)], axis=1)
    run = np.maximum.accumulate(blk_max, axis=1)
    jumps = np.sum(np.diff(run, axis=1) > 8.0, axis=1)
    assert jumps.mean() >= 1.0


# ------------------------------------------------------------------- exp2

def test_exp2_poly_matches_printed_coefficients():
    with open(os.path.join(GOLDEN, "exp2_poly.json")) as f:
        g = json.load(f)
    assert tuple(g["p"]) == oracle.EXP2_POLY


def test_exp2_cubic_error_bound_dense_grid():
    """Max relative error of the printed cubic over x in [-126, 8] is below 2e-4."""
    x = np.linspace(-126.0, 8.0, 2_000_001)
    f = np.linspace(0.0, 1.0, 1_000_001, endpoint=False)
    for xs in (x, f, f - 7.0):
        rel = np.abs(oracle.exp2_cubic(xs) / np.exp2(xs) - 1.0)
        assert rel.max() <= 2e-4
    # 2^n is exact at integers (p0 = 1), and the worst case sits near f -> 1
    ints = np.arange(-126, 9, dtype=np.float64)
    assert np.array_equal(oracle.exp2_cubic(ints), np.exp2(ints))
    rel = np.abs(oracle.exp2_cubic(f) / np.exp2(f) - 1.0)
    assert 0.9e-4 <= rel.max() <= 1.1e-4


# ------------------------------------------------------- input generator pins

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(14)
    x = (rng.standard_normal(100_000) * np.exp(rng.uniform(-20, 20, 100_000))).astype(np.float32)
    x[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]   # ties to even
    ours = fa_inputs.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = fa_inputs.bf16_bits_to_f64(ours)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).double().numpy())


# ----------------------------------- planted mistakes: the pins are sensitive

def test_planted_mistakes_are_caught(monkeypatch):
    """Mutate the oracle on the CPU and check that a pin above fails."""
    rng = np.random.default_rng(15)
    q, k, v = _rand(rng, 6, 3), _rand(rng, 6, 3), _rand(rng, 6, 3)
    ob, lb = _brute(q.tolist(), k.tolist(), v.tolist(), True, 0.9)

    # (a) transposed operand in O = P V
    real = orc.softmax_probs
    monkeypatch.setattr(orc, "softmax_probs",
                        lambda *a, **kw: (lambda r: (r[0].T.copy(), r[1], r[2]))(real(*a, **kw)))
    o, _ = orc.head_forward(q, k, v, causal=True, scale=0.9)
    assert np.max(np.abs(o - ob)) > 1e-3
    monkeypatch.undo()

    # (b) a causal mask off by one (j < i instead of j <= i) changes row results
    s = 0.9 * q @ k.T
    s_bad = np.where(np.arange(6)[None, :] < np.arange(6)[:, None] + 2, s, -np.inf)
    lse_bad = np.log(np.exp(s_bad).sum(axis=1))
    assert np.max(np.abs(lse_bad - lb)) > 1e-3

    # (c) Horner with the coefficients reversed breaks the exp2 bound
    f = np.linspace(0, 1, 1001, endpoint=False)
    rel = np.abs(oracle.exp2_cubic(f, poly=oracle.EXP2_POLY[::-1]) / np.exp2(f) - 1)
    assert rel.max() > 2e-4
    # (d) round-to-nearest range reduction (f in [-0.5, 0.5)) breaks it too
    rel = np.abs(np.ldexp(np.polyval(oracle.EXP2_POLY[::-1], f - 0.5), 0) / np.exp2(f - 0.5) - 1)
    assert rel.max() > 2e-4
