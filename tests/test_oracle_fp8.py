"""Pins of the 8-bit forward's definition (``oracle/fp8.py``).

Each check ties the oracle to something other than itself: PyTorch's
float8_e4m3fn conversion (the OCP e4m3 format), scipy's Hadamard matrix, the
orthogonality identity the method rests on ("FlashAttention-3: Fast and
Accurate Attention with Asynchrony and Low-precision" 技術 3: multiplying Q
and K by the same orthogonal matrix leaves Q K^T unchanged), and the plain
attention oracle on inputs that the quantisation reproduces exactly.  A
wrong block size, a missing 1/d, a transposed Hadamard stage or a wrong
rounding mode fails one of them.
"""
import numpy as np
import pytest

from oracle import attention as orc
from oracle import fp8 as o8

pytestmark = pytest.mark.oracle


def _grid_values():
    """Every finite e4m3 value, and midpoints between neighbours."""
    pos = [m * 2.0 ** -9 for m in range(8)]                         # subnormals and 0
    pos += [(1 + m / 8) * 2.0 ** e for e in range(-6, 9) for m in range(8)]
    pos = np.array(sorted(set(v for v in pos if v <= 448.0)))
    mids = (pos[1:] + pos[:-1]) / 2
    return pos, mids


def test_e4m3_round_matches_float8_e4m3fn():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    pos, mids = _grid_values()
    x = np.concatenate([pos, -pos, mids, -mids, rng.standard_normal(20000) * 30,
                        rng.uniform(-2.0 ** -5, 2.0 ** -5, 5000)])
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn)
    assert np.array_equal(o8.e4m3_round(x.astype(np.float32)), ref.to(torch.float64).numpy())
    assert np.array_equal(o8.e4m3_codes(x.astype(np.float32)), ref.view(torch.uint8).numpy())


def test_e4m3_ties_to_even_and_saturates():
    # 1 + 1/16 lies halfway between 1 and 1 + 1/8: ties go to the even mantissa (1)
    assert o8.e4m3_round(np.array([1.0625, 1.1875, 448.0, 460.0, 1e6, -1e6]))[:6].tolist() == \
        [1.0, 1.25, 448.0, 448.0, 448.0, -448.0]
    assert o8.e4m3_codes(np.array([448.0, -448.0, 1000.0, 0.0, 2.0 ** -9])).tolist() == \
        [0x7E, 0xFE, 0x7E, 0x00, 0x01]


@pytest.mark.parametrize("d", [128, 256])
def test_fwht_is_the_sylvester_hadamard_product(d):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = scipy_linalg.hadamard(d).astype(np.float64)
    rng = np.random.default_rng(6)
    xi = rng.integers(-8, 9, size=(5, d)).astype(np.float32)      # exact in fp32
    assert np.array_equal(o8.fwht_f32(xi).astype(np.float64), xi.astype(np.float64) @ H)
    x = rng.standard_normal((7, d)).astype(np.float32)
    assert np.max(np.abs(o8.fwht_f32(x) - x.astype(np.float64) @ H)) < 1e-4 * d / 128


def test_sign_vector_reads_bit_c_of_word_c_over_32():
    # channel 37 is bit 5 of word 1; channel 255 bit 31 of word 7
    words = [0] * 8
    words[1] = 1 << 5
    words[7] = 1 << 31
    v = o8.sign_vector(words, 256)
    assert np.flatnonzero(v < 0).tolist() == [37, 255]


@pytest.mark.parametrize("d", [128, 256])
def test_incoherent_processing_keeps_qk_up_to_d(d):
    rng = np.random.default_rng(7)
    q, k = rng.standard_normal((2, 64, d))
    signs = rng.integers(0, 2 ** 32, size=d // 32, dtype=np.uint64)
    D = o8.sign_vector(signs, d).astype(np.float64)
    assert set(np.unique(D)) == {-1.0, 1.0}
    import scipy.linalg
    H = scipy.linalg.hadamard(d).astype(np.float64)
    # (Q D H)(K D H)^T = Q D H H^T D K^T = d Q K^T
    lhs = (q * D) @ H @ ((k * D) @ H).T
    assert np.max(np.abs(lhs - d * q @ k.T)) < 1e-9 * d
    # and the oracle's fp32 path agrees up to fp32 rounding
    got = o8.incoherent(q, signs).astype(np.float64) @ o8.incoherent(k, signs).astype(np.float64).T
    assert np.max(np.abs(got - d * q @ k.T)) / np.max(np.abs(q @ k.T)) < 1e-3 * d / 128


def _exact_inputs(rng, B, H, N, d, block_scale):
    """Values on the e4m3 grid whose every quantisation block has amax 448 * 2^-k:
    the multiplier is a power of two and the codes are the values themselves."""
    pos, _ = _grid_values()
    x = rng.choice(np.concatenate([pos, -pos]), size=(B, H, N, d))
    nb = (N + 127) // 128
    for b in range(nb):
        sl = slice(128 * b, min(N, 128 * b + 128))
        x[:, :, sl] *= block_scale[b % len(block_scale)]
        x[:, :, sl.start, 0] = 448.0 * block_scale[b % len(block_scale)]   # the block's amax
    return x


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward_without_rounding_is_plain_attention(causal):
    """Blocks with different powers of two as amax: a per-tensor scale, a wrong
    block size or a wrong multiplier would change the codes and fail."""
    rng = np.random.default_rng(8)
    q = _exact_inputs(rng, 1, 2, 300, 128, [1.0, 0.25, 2.0 ** -5])
    k = _exact_inputs(rng, 1, 2, 300, 128, [0.5, 1.0, 0.125])
    v = _exact_inputs(rng, 1, 2, 300, 128, [1.0])
    v[:, :, 0, 0] = 448.0                                 # per-head amax of V
    scale = 2.0 ** -7
    o, lse, parts = o8.fp8_forward(q, k, v, causal, scale, signs=None)
    o_ref, lse_ref = orc.attention_forward(q, k, v, causal=causal, scale=scale)
    assert np.max(np.abs(o - o_ref)) < 1e-12 and np.max(np.abs(lse - lse_ref)) < 1e-12
    assert parts["inv_q"][0].tolist() == [1.0, 4.0, 32.0]
    assert parts["inv_k"][0].tolist() == [2.0, 1.0, 8.0]


@pytest.mark.parametrize("d", [128, 256])
def test_fp8_forward_with_signs_uses_scale_over_d_any_d(d):
    """As below, at both head dimensions of the 8-bit path."""
    rng = np.random.default_rng(12)
    q, k, v = (rng.standard_normal((1, 1, 160, d)) for _ in range(3))
    signs = rng.integers(0, 2 ** 32, size=d // 32, dtype=np.uint64)
    o, lse, _ = o8.fp8_forward(q, k, v, False, d ** -0.5, signs=signs)
    o_ref, lse_ref = orc.attention_forward(q, k, v, causal=False, scale=d ** -0.5)
    assert np.max(np.abs(lse - lse_ref)) < 0.05
    assert np.sqrt(np.mean((o - o_ref) ** 2)) / np.sqrt(np.mean(o_ref ** 2)) < 0.1


def test_fp8_forward_with_signs_uses_scale_over_d():
    """With incoherent processing the 8-bit scores are d times the plain ones;
    dropping the 1/d (or applying it without the transform) moves the LSE by
    log(d)-sized amounts, far outside this bound."""
    rng = np.random.default_rng(9)
    q = rng.standard_normal((1, 1, 200, 128))
    k = rng.standard_normal((1, 1, 200, 128))
    v = rng.standard_normal((1, 1, 200, 128))
    signs = rng.integers(0, 2 ** 32, size=4, dtype=np.uint64)
    o, lse, _ = o8.fp8_forward(q, k, v, False, 128 ** -0.5, signs=signs)
    o_ref, lse_ref = orc.attention_forward(q, k, v, causal=False, scale=128 ** -0.5)
    # only the 8-bit rounding separates them (e4m3: 2^-4 relative per value)
    assert np.max(np.abs(lse - lse_ref)) < 0.05
    assert np.sqrt(np.mean((o - o_ref) ** 2)) / np.sqrt(np.mean(o_ref ** 2)) < 0.1


def test_incoherent_processing_lowers_the_error_on_outlier_inputs():
    """The error claim of the same page (数値誤差: incoherent processing gives a
    lower RMSE than plain FP8 when a few channels carry large outliers)."""
    rng = np.random.default_rng(10)
    shape = (1, 2, 256, 128)
    def draw():
        return rng.standard_normal(shape) + rng.standard_normal(shape) * 10.0 * (rng.random(shape) < 0.001)
    q, k, v = draw(), draw(), draw()
    o_ref, _ = orc.attention_forward(q, k, v, causal=False, scale=128 ** -0.5)
    o_plain, _, _ = o8.fp8_forward(q, k, v, False, 128 ** -0.5, signs=None)
    signs = rng.integers(0, 2 ** 32, size=4, dtype=np.uint64)
    o_inc, _, _ = o8.fp8_forward(q, k, v, False, 128 ** -0.5, signs=signs)
    rmse = lambda o: float(np.sqrt(np.mean((o - o_ref) ** 2)))
    assert rmse(o_inc) < rmse(o_plain)


def test_per_head_scale_is_one_block_spanning_the_head():
    """qk_block=None (one scale per head) equals block quantisation with a
    block as long as the sequence, and differs from 128-row blocks when the
    blocks' ranges differ."""
    rng = np.random.default_rng(11)
    q = rng.standard_normal((1, 2, 256, 128))
    q[:, :, 128:] *= 1e-3                     # second block far smaller than the first
    k, v = rng.standard_normal((2, 1, 2, 256, 128))
    o_t, lse_t, p_t = o8.fp8_forward(q, k, v, False, 0.1, qk_block=None)
    o_b, lse_b, p_b = o8.fp8_forward(q, k, v, False, 0.1, qk_block=256)
    assert np.array_equal(o_t, o_b) and np.array_equal(lse_t, lse_b)
    assert np.array_equal(p_t["inv_q"], p_b["inv_q"][:, 0])
    _, _, p_128 = o8.fp8_forward(q, k, v, False, 0.1)
    assert not np.array_equal(p_128["q8"], p_t["q8"])
