"""Plain fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The library never calls it; it shares no
code, constant or helper with the CUDA path.

Pages followed (cited by title and section):

* [FA]  "FlashAttention: GPUメモリ階層を活用したアテンション最適化の分析"
        (youngju.dev) -- §2.1 standard attention, §6.1 safe softmax,
        §6.2 online softmax, §6.3 rescaling identity, §7.2 recomputation,
        §8.1 deferred normalisation, §11.3 causal mask as ``tril``.
* [FA4] "論文解説: FlashAttention-4 — Algorithm and Kernel Pipelining
        Co-Design for Asymmetric Hardware Scaling" (0h-n0.github.io) --
        ソフトウェア指数関数エミュレーション (exp2 emulation),
        条件付きオンラインsoftmaxリスケーリング (conditional rescaling).

Every function here is the plain definition written out, with S and P
materialised, except ``online_softmax_forward`` (an fp64 restatement of the
tiled algorithm, used only to show the tiled recurrences are exact) and
``exp2_cubic`` (the emulation's own steps).  Readings of the pages where they
are silent or garbled:

* Causal masking is top-left aligned: query i may attend key j iff j <= i
  (the square ``tril`` mask of [FA] §11.3, extended to N_q != N_kv).
* LSE is the natural-log log-sum-exp of the scaled scores, fp32 on the GPU.
* The backward pass is the exact gradient of <dO, O> at the given inputs
  ([FA] §7.2 only says S and P are recomputed from the saved statistics);
  ``head_backward_from_saved`` is the same computation driven by a given
  (saved, possibly rounded) O and LSE, which is what a backward kernel
  receives.
* Conditional rescaling keeps a reference maximum m_ref per row; P is
  2^(t - m_ref) while the row max has not risen more than tau above m_ref
  (so P may reach 2^tau); when it has, O and l are multiplied by
  2^(m_ref - m_new) and m_ref becomes m_new ([FA4] 条件付き... whose
  "otherwise" branch is internally inconsistent as printed).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "head_forward", "attention_forward", "attention_backward", "head_backward",
    "head_backward_from_saved",
    "online_softmax_forward", "exp2_cubic", "EXP2_POLY", "softmax_probs",
]

# Cubic coefficients for 2^f on f in [0, 1), as printed in [FA4]
# ソフトウェア指数関数エミュレーション, step 2.
EXP2_POLY = (1.0, 0.6951, 0.2276, 0.0771)


def _row_block(n_kv: int) -> int:
    # Bound the materialised score block to ~2^22 doubles (32 MB).
    return max(1, min(1024, (1 << 22) // max(1, n_kv)))


def softmax_probs(q, k, *, causal: bool, scale: float, rows=None):
    """P = softmax(scale * q k^T) for one head, materialised ([FA] §2.1, §6.1).

    q: [n, d] float64, k: [N_kv, d] float64.  ``rows`` gives each q row's
    query index (default 0..n-1), used only by the causal mask.
    Returns (P [n, N_kv], m [n], l [n]) where m is the row max of the scaled
    scores over the allowed keys and l = sum_j exp(s_ij - m_i).
    """
    n, n_kv = q.shape[0], k.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows)
    s = scale * (q @ k.T)
    if causal:
        allowed = np.arange(n_kv)[None, :] <= rows[:, None]
        s = np.where(allowed, s, -np.inf)
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])          # masked entries: exp(-inf) = 0
    l = e.sum(axis=1)
    return e / l[:, None], m, l


def head_forward(q, k, v, *, causal: bool, scale: float, rows=None):
    """O and LSE for one head (float64): O = P v, LSE = m + ln l.

    [FA] §2.1 (S = QK^T, P = softmax(S), O = PV) with the safe softmax of
    §6.1; the LSE is the statistic saved for the backward pass (§7.2).
    """
    n = q.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows)
    o = np.empty((n, v.shape[1]))
    lse = np.empty(n)
    rb = _row_block(k.shape[0])
    for r0 in range(0, n, rb):
        sl = slice(r0, min(n, r0 + rb))
        p, m, l = softmax_probs(q[sl], k, causal=causal, scale=scale, rows=rows[sl])
        o[sl] = p @ v
        lse[sl] = m + np.log(l)
    return o, lse


def attention_forward(q, k, v, *, causal: bool, scale: float):
    """Batched oracle forward: q [B,H,N_q,d], k/v [B,H,N_kv,d] float64.

    Returns O [B,H,N_q,d] and LSE [B,H,N_q], both float64.
    """
    B, H, n_q, d = q.shape
    o = np.empty((B, H, n_q, v.shape[3]))
    lse = np.empty((B, H, n_q))
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = head_forward(q[b, h], k[b, h], v[b, h],
                                              causal=causal, scale=scale)
    return o, lse


def head_backward(q, k, v, do, *, causal: bool, scale: float):
    """Exact gradients of L = <dO, O> for one head (float64).

    With P the softmax probabilities ([FA] §2.1) and D_i = sum_c dO_ic O_ic:
    dV = P^T dO, dP = dO V^T, dS = P o (dP - D), dQ = scale dS K,
    dK = scale dS^T Q.  S and P are recomputed row block by row block, the
    recomputation of [FA] §7.2; O is this oracle's own float64 output.
    """
    n = q.shape[0]
    o, _ = head_forward(q, k, v, causal=causal, scale=scale)
    D = np.sum(do * o, axis=1)
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rb = _row_block(k.shape[0])
    for r0 in range(0, n, rb):
        sl = slice(r0, min(n, r0 + rb))
        p, _, _ = softmax_probs(q[sl], k, causal=causal, scale=scale,
                                rows=np.arange(sl.start, sl.stop))
        dv += p.T @ do[sl]
        dp = do[sl] @ v.T
        ds = p * (dp - D[sl, None])
        dq[sl] = scale * (ds @ k)
        dk += scale * (ds.T @ q[sl])
    return dq, dk, dv


def attention_backward(q, k, v, do, *, causal: bool, scale: float):
    """Batched oracle backward; returns (dQ, dK, dV) float64, same shapes as q, k, v."""
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    B, H = q.shape[:2]
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = head_backward(
                q[b, h], k[b, h], v[b, h], do[b, h], causal=causal, scale=scale)
    return dq, dk, dv


def head_backward_from_saved(q, k, v, o, do, lse, *, causal: bool, scale: float):
    """Gradients for one head from saved forward outputs (float64).

    The recomputation contract of [FA] §7.2 taken literally: the forward
    saved O and the row statistics (here the natural-log LSE), and the
    backward rebuilds P = exp(scale q k^T - LSE) from them instead of
    renormalising.  With D_i = sum_c dO_ic o_ic for the GIVEN o:
    dV = P^T dO, dS = P o (dO V^T - D), dQ = scale dS K, dK = scale dS^T Q.
    Fed this oracle's own O and LSE it equals ``head_backward``; fed a rounded
    O (as a bf16 forward output would be) it gives what a backward pass
    computes from that O.
    """
    n, n_kv = q.shape[0], k.shape[0]
    D = np.sum(do * o, axis=1)
    dq = np.empty_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    rb = _row_block(n_kv)
    for r0 in range(0, n, rb):
        sl = slice(r0, min(n, r0 + rb))
        s = scale * (q[sl] @ k.T)
        if causal:
            rows = np.arange(sl.start, sl.stop)
            s = np.where(np.arange(n_kv)[None, :] <= rows[:, None], s, -np.inf)
        p = np.exp(s - lse[sl, None])
        dv += p.T @ do[sl]
        ds = p * (do[sl] @ v.T - D[sl, None])
        dq[sl] = scale * (ds @ k)
        dk += scale * (ds.T @ q[sl])
    return dq, dk, dv


def online_softmax_forward(q, k, v, *, causal: bool, scale: float,
                           block_kv: int = 128, tau: float = 8.0):
    """Tiled online-softmax forward for one head, float64, in base 2.

    The running statistics of [FA] §6.2 (row max m, row sum l, output
    accumulator) updated one key block at a time, with the conditional
    rescaling of [FA4] 条件付きオンラインsoftmaxリスケーリング: the
    accumulator and l are rescaled only when the block's row max exceeds the
    reference max by more than ``tau`` (log2 units); the normalisation by l
    is deferred to the end ([FA] §8.1).  ``tau = 0`` is the ordinary online
    softmax; ``tau = inf`` never rescales after the first block.

    Returns (O [n, d], LSE [n]) -- equal to ``head_forward`` up to rounding,
    which is what makes the tiled algorithm exact ([FA] §6.3).
    """
    n, n_kv = q.shape[0], k.shape[0]
    log2e = 1.0 / math.log(2.0)
    m_ref = np.full(n, -np.inf)
    l = np.zeros(n)
    acc = np.zeros((n, v.shape[1]))
    rows = np.arange(n)
    for j0 in range(0, n_kv, block_kv):
        cols = np.arange(j0, min(n_kv, j0 + block_kv))
        t = (scale * log2e) * (q @ k[cols].T)          # scores in log2 units
        if causal:
            t = np.where(cols[None, :] <= rows[:, None], t, -np.inf)
        m_blk = t.max(axis=1)
        m_new = np.maximum(m_ref, m_blk)
        jump = np.isneginf(m_ref) & np.isfinite(m_new)
        with np.errstate(invalid="ignore"):
            jump |= (m_new - m_ref) > tau
        alpha = np.where(jump, np.exp2(np.where(jump, m_ref - m_new, 0.0)), 1.0)
        acc *= alpha[:, None]
        l *= alpha
        m_ref = np.where(jump, m_new, m_ref)
        with np.errstate(invalid="ignore"):
            p = np.where(np.isneginf(t), 0.0, np.exp2(t - m_ref[:, None]))
        l += p.sum(axis=1)
        acc += p @ v[cols]
    o = acc / l[:, None]
    lse = math.log(2.0) * (m_ref + np.log2(l))
    return o, lse


def exp2_cubic(x, poly=EXP2_POLY):
    """2^x by the emulation of [FA4] ソフトウェア指数関数エミュレーション, in float64.

    Range reduction n = floor(x), f = x - n in [0, 1); 2^f from the cubic
    p0 + p1 f + p2 f^2 + p3 f^3 evaluated by Horner's rule (three
    multiply-adds); the result is the cubic scaled by 2^n (the step the page
    performs by shifting n into the float's exponent field).
    """
    x = np.asarray(x, dtype=np.float64)
    n = np.floor(x)
    f = x - n
    p0, p1, p2, p3 = poly
    poly_f = ((p3 * f + p2) * f + p1) * f + p0
    return np.ldexp(poly_f, n.astype(np.int64))
