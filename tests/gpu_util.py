"""Helpers shared by the GPU parity tests (device tensors, guard bands, metrics).

The tolerances are the ones fixed for this library: O max-abs error <= 1e-2
and relative RMS <= 5e-3, LSE max-abs error <= 1e-3, dQ/dK/dV relative RMS
<= 1e-2, emulated 2^x max relative error <= 2e-4.  Relative RMS is
||x - ref||_2 / ||ref||_2 over the compared elements.

``assert_o_lse`` applies those bounds exactly as stated; every test of the
five stated workloads (and every other forward test at head dimension 64 or
128) uses it.  The one place where no bf16 output can meet 1e-2 is an exact
value with no bf16 number within 1e-2 of it (possible only for |O| >= 4,
where bf16 values lie 0.031 apart): such an element must equal the exact
value correctly rounded to bf16, and the check reports how many there were.
Only the extra tests whose exact outputs routinely leave bf16's reach of 1e-2
(|O| up to 4.7 at head dimension 256 on the stress inputs, tens on the
outlier inputs) use ``assert_o_lse_bf16`` instead: there each element must
lie within half a bf16 step of its exact value's binade plus the kernel's
arithmetic budget (below), or within 1e-2.

The arithmetic budget.  The kernels form O = sum_j p^_j v_j / L with the
unnormalised weights p^_j rounded to bf16 (the operand type of the P V
product; bf16 carries 8 significant bits, so each rounding is within 2^-8
relative) and L their fp32 sum corrected for each key block's largest
weight.  Writing O for the exact output and A_ic = sum_j P_ij |v_jc - O_ic|
(P the exact probabilities), the rounding of the weights moves O_ic by at
most 2^-8 (A_ic + |O_ic|); a quarter more covers fp32 accumulation, fp32
scores and the emulated exponentials (relative error 1e-4).
``o_element_bound`` adds half a bf16 step of the binade of |O| + budget for
the final rounding to bf16.  This per-element bound is also asserted on top
of the stated tolerances wherever the oracle can afford A (whole small
problems and sampled rows of the large ones): it is the precise form of
"within about one bf16 step of the rounded exact value", which does not hold
element by element on its own -- on rows whose output nearly cancels (|O|
far below A) the rounding of the bf16 weights alone is many steps of the
small result.
"""
import numpy as np

import fa_inputs
from oracle import attention as orc

O_MAX_ABS = 1e-2
O_REL_RMS = 5e-3
LSE_MAX_ABS = 1e-3
GRAD_REL_RMS = 1e-2
P_ROUNDING = 2.0 ** -8 * 1.25       # the budget's factor on A + |O| (see the module docstring)


def torch():
    import torch as t
    return t


def dev_bf16(bits):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to("cuda").view(t.bfloat16)


class Guarded:
    """A device buffer with all-ones (NaN for floats) guard bands of 256 bytes
    on each side of the usable view, which keeps the view 256-byte aligned."""

    def __init__(self, shape, dtype):
        t = torch()
        n = int(np.prod(shape))
        self.g = 256 // t.empty((), dtype=dtype).element_size()
        self.raw = t.empty(n + 2 * self.g, dtype=dtype, device="cuda")
        self._bits().fill_(-1 if self.raw.dtype != t.uint8 else 255)
        self.view = self.raw[self.g:self.g + n].view(shape)

    def _bits(self):
        t = torch()
        return self.raw.view({t.bfloat16: t.int16, t.float32: t.int32}.get(self.raw.dtype, self.raw.dtype))

    def guards_intact(self):
        t = torch()
        b = self._bits()
        g = t.cat([b[:self.g], b[-self.g:]])
        return bool((g == (255 if self.raw.dtype == t.uint8 else -1)).all().item())


def to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def rel_rms(x, ref):
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


# ------------------------------------------------------------ bf16 arithmetic

def half_step(x):
    """Half the bf16 spacing of the binade holding |x|: 2^(e - 8) for |x| in [2^e, 2^(e+1))."""
    a = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -126)
    e = np.floor(np.log2(a))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def bf16_round(x):
    """x (float64) rounded to the nearest bf16 value, ties to even, returned as float64."""
    x = np.asarray(x, dtype=np.float64)
    step = 2.0 * half_step(x)
    return np.round(x / step) * step


def _bf16_key(x):
    """Monotone integer position of bf16 values (exactly representable float64 input)."""
    bits = fa_inputs.f32_to_bf16_bits(np.asarray(x, dtype=np.float32)).astype(np.int64)
    mag = bits & 0x7FFF
    return np.where(bits & 0x8000, -mag, mag)


def ulp_stats(o, o_ref):
    """(largest number of bf16 steps between o and the bf16-rounded exact value,
    fraction of elements within one step)."""
    d = np.abs(_bf16_key(o) - _bf16_key(bf16_round(o_ref)))
    return int(d.max()), float(np.mean(d <= 1))


def o_element_bound(o_ref, spread):
    """Per-element bound on |O_kernel - O|: the weights' rounding budget
    P_ROUNDING * (A + |O|) plus half a bf16 step of |O| + budget."""
    budget = P_ROUNDING * (spread + np.abs(o_ref))
    return budget + half_step(np.abs(o_ref) + budget)


def spread(q, k, v, o_ref, causal, scale, rows=None):
    """A_ic = sum_j P_ij |v_jc - O_ic| for one head (float64), P from the oracle."""
    n = q.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows)
    out = np.empty_like(o_ref)
    chunk = max(1, (1 << 23) // max(1, k.shape[0] * v.shape[1]))
    for r0 in range(0, n, chunk):
        sl = slice(r0, min(n, r0 + chunk))
        p, _, _ = orc.softmax_probs(q[sl], k, causal=causal, scale=scale, rows=rows[sl])
        out[sl] = np.einsum("rj,rjc->rc", p, np.abs(v[None, :, :] - o_ref[sl, None, :]))
    return out


# ---------------------------------------------------------------- the checks

def _check_lse(lse, lse_ref, what, lse_rel):
    assert np.all(np.isfinite(lse)), f"{what}: non-finite LSE"
    e_lse = float(np.max(np.abs(lse - lse_ref)))
    assert np.all(np.abs(lse - lse_ref) <= LSE_MAX_ABS + lse_rel * np.abs(lse_ref)), \
        f"{what}: LSE max-abs {e_lse:.3e}"
    return e_lse


def assert_o_lse(o, lse, o_ref, lse_ref, what="", spread_=None):
    """The stated bounds as written: O max-abs <= 1e-2, O relative RMS <=
    5e-3, LSE max-abs <= 1e-3; with ``spread_`` (A, same shape as O) also the
    per-element arithmetic bound.  Returns (O max-abs, O rel-RMS, LSE
    max-abs, max bf16 steps from the rounded exact value, fraction within one)."""
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    err = np.abs(o - o_ref)
    e_max = float(np.max(err))
    e_rms = rel_rms(o, o_ref)
    # elements whose exact value has no bf16 number within 1e-2 (|O| >= 4):
    # there the output must be that value correctly rounded
    rounded = bf16_round(o_ref)
    beyond = np.abs(rounded - o_ref) > O_MAX_ABS
    bad = (err > O_MAX_ABS) & ~(beyond & (o == rounded))
    worst = int(np.argmax(np.where(bad, err, -1.0)))
    assert not bad.any(), \
        f"{what}: O max-abs {err.flat[worst]:.3e} (|O| {np.abs(o_ref).flat[worst]:.3f} there)"
    e_in = float(np.max(np.where(beyond, 0.0, err)))
    assert e_rms <= O_REL_RMS, f"{what}: O rel-RMS {e_rms:.3e}"
    if spread_ is not None:
        _assert_element_bound(err, o_ref, spread_, what)
    e_lse = _check_lse(lse, lse_ref, what, 0.0)
    steps, within1 = ulp_stats(o, o_ref)
    print(f"{what}: O max-abs {e_max:.2e} ({e_in:.2e} where bf16 can reach 1e-2; {int(beyond.sum())} elements "
          f"beyond bf16's reach, each correctly rounded) rel-RMS {e_rms:.2e} LSE max-abs {e_lse:.2e} "
          f"bf16 steps from rounded exact: max {steps}, {100 * within1:.2f}% within 1")
    return e_max, e_rms, e_lse, steps, within1


def _assert_element_bound(err, o_ref, spread_, what):
    bound = o_element_bound(o_ref, spread_)
    over = err - bound
    i = int(np.argmax(over))
    assert over.flat[i] <= 0.0, \
        (f"{what}: O error {err.flat[i]:.3e} above the per-element arithmetic bound {bound.flat[i]:.3e} "
         f"(|O| {abs(o_ref.flat[i]):.4f}, A {spread_.flat[i]:.4f})")


def assert_o_lse_bf16(o, lse, o_ref, lse_ref, spread_, what="", lse_rel=0.0):
    """The reading for exact outputs beyond bf16's reach of 1e-2: each element
    within max(1e-2, the per-element arithmetic bound); relative RMS <= 5e-3;
    LSE within 1e-3 (+ lse_rel |LSE|)."""
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    err = np.abs(o - o_ref)
    bound = np.maximum(O_MAX_ABS, o_element_bound(o_ref, spread_))
    over = err - bound
    i = int(np.argmax(over))
    assert over.flat[i] <= 0.0, \
        (f"{what}: O error {err.flat[i]:.3e} above max(1e-2, arithmetic bound {bound.flat[i]:.3e}) "
         f"(|O| {abs(o_ref.flat[i]):.4f}, A {spread_.flat[i]:.4f})")
    e_rms = rel_rms(o, o_ref)
    assert e_rms <= O_REL_RMS, f"{what}: O rel-RMS {e_rms:.3e}"
    e_lse = _check_lse(lse, lse_ref, what, lse_rel)
    steps, within1 = ulp_stats(o, o_ref)
    print(f"{what}: O max-abs {float(err.max()):.2e} (|O| up to {float(np.abs(o_ref).max()):.2f}) rel-RMS "
          f"{e_rms:.2e} LSE max-abs {e_lse:.2e} bf16 steps: max {steps}, {100 * within1:.2f}% within 1")
    return float(err.max()), e_rms, e_lse, steps, within1


def sample_rows(n, k, rng):
    """Rows to compare at full size: the first and last rows, tile edges, random rows."""
    fixed = {0, 1, n - 1, n - 2, min(127, n - 1), min(128, n - 1), min(255, n - 1), min(256, n - 1)}
    rnd = set(rng.choice(n, size=min(n, k), replace=False).tolist())
    return np.array(sorted(fixed | rnd))


def oracle_rows(qb, kb, vb, b, h, rows, causal, scale, with_spread=False):
    q = fa_inputs.bf16_bits_to_f64(qb[b, h][rows])
    k = fa_inputs.bf16_bits_to_f64(kb[b, h])
    v = fa_inputs.bf16_bits_to_f64(vb[b, h])
    o, lse = orc.head_forward(q, k, v, causal=causal, scale=scale, rows=rows)
    if not with_spread:
        return o, lse
    return o, lse, spread(q, k, v, o, causal, scale, rows=rows)
