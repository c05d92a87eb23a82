"""Helpers shared by the GPU parity tests (device tensors, guard bands, metrics).

The tolerances are the ones fixed for this library: O max-abs error <= 1e-2
and relative RMS <= 5e-3, LSE max-abs error <= 1e-3, dQ/dK/dV relative RMS
<= 1e-2, emulated 2^x max relative error <= 2e-4.  Relative RMS is
||x - ref||_2 / ||ref||_2 over the compared elements.  O is bf16, whose step
exceeds 1e-2 once |O| >= 1.28 (0.0156 on [2, 4), 0.031 on [4, 8)): there
each element must instead lie within one bf16 step (2^-7 |O|) of the exact
value, the closest any bf16 output can be guaranteed to come.
"""
import numpy as np

import fa_inputs
from oracle import attention as orc

O_MAX_ABS = 1e-2
O_REL_RMS = 5e-3
LSE_MAX_ABS = 1e-3
GRAD_REL_RMS = 1e-2


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


def assert_o_lse(o, lse, o_ref, lse_ref, what=""):
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    assert np.all(np.isfinite(lse)), f"{what}: non-finite LSE"
    err = np.abs(o - o_ref)
    e_max = float(np.max(err))
    e_rms = rel_rms(o, o_ref)
    e_lse = float(np.max(np.abs(lse - lse_ref)))
    bound = np.maximum(O_MAX_ABS, 2.0 ** -7 * np.abs(o_ref))
    worst = int(np.argmax(err - bound))
    assert np.all(err <= bound), \
        f"{what}: O max-abs {e_max:.3e} (|O| {np.abs(o_ref).flat[worst]:.3f} where the bound is exceeded)"
    assert e_rms <= O_REL_RMS, f"{what}: O rel-RMS {e_rms:.3e}"
    assert e_lse <= LSE_MAX_ABS, f"{what}: LSE max-abs {e_lse:.3e}"
    return e_max, e_rms, e_lse


def sample_rows(n, k, rng):
    """Rows to compare at full size: the first and last rows, tile edges, random rows."""
    fixed = {0, 1, n - 1, n - 2, min(127, n - 1), min(128, n - 1), min(255, n - 1), min(256, n - 1)}
    rnd = set(rng.choice(n, size=min(n, k), replace=False).tolist())
    return np.array(sorted(fixed | rnd))


def oracle_rows(qb, kb, vb, b, h, rows, causal, scale):
    q = fa_inputs.bf16_bits_to_f64(qb[b, h][rows])
    k = fa_inputs.bf16_bits_to_f64(kb[b, h])
    v = fa_inputs.bf16_bits_to_f64(vb[b, h])
    return orc.head_forward(q, k, v, causal=causal, scale=scale, rows=rows)
