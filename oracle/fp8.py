"""The 8-bit forward's definition, on the CPU -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The library never calls it; it shares no
code, constant or helper with the CUDA path.

Follows "FlashAttention-3: Fast and Accurate Attention with Asynchrony and
Low-precision" (notes.yuuk.io), 技術 3: Q, K and V are held in 8-bit floating
point with one scale per block, and before quantisation Q and K are both
multiplied by one random orthogonal matrix M = D H (D a diagonal of random
signs, H the Hadamard matrix), which leaves Q K^T unchanged and spreads an
outlier channel over all channels ("incoherent processing").  The pages fix
neither the 8-bit format, the block size, how a scale is chosen, nor the
order of the Hadamard transform; the readings taken here:

* Format: e4m3 (OCP FP8 E4M3: 4 exponent bits with bias 7, 3 mantissa bits,
  no infinities, largest finite 448), values rounded to nearest (ties to
  even) and saturated to +-448.
* Q and K: one scale per 128-row block of each (batch, head); V: one scale
  per (batch, head).  A block's multiplier is inv = 448 / amax in fp32 (1 for
  an all-zero block), so the largest magnitude maps to 448; code =
  e4m3(fp32(x * inv)).
* H is the Sylvester Hadamard matrix (entries +-1, unnormalised, H H^T = d I)
  applied to each row of Q and K by the butterfly of stages h = 1, 2, 4, ...,
  d/2 in fp32, after negating the channels whose sign bit is set.  With the
  unnormalised H, Q' K'^T = d Q K^T, so the logit scale is divided by d.
* The attention itself is exact (fp64) on the dequantised values: S =
  scale' (Q8 / inv_q)(K8 / inv_k)^T, softmax, O = P (V8 / inv_v), LSE.  The
  GPU path also rounds P to e4m3 for the P V product; that rounding is part
  of the tolerance, not of the definition.

Every arithmetic step that decides a code (the butterfly, the block maximum,
the multiplier, the product x * inv) is done in fp32 in the order stated, so
that the codes are the same as the GPU's, bit for bit.
"""
from __future__ import annotations

import numpy as np

from .attention import attention_forward

E4M3_MAX = 448.0
BLOCK = 128


def e4m3_round(x: np.ndarray) -> np.ndarray:
    """Nearest e4m3 value (ties to even), saturated to +-448, as float64."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    m, e = np.frexp(a)                       # a = m 2^e, m in [0.5, 1)
    # the leading bit is 2^(e-1); three mantissa bits below it; subnormals
    # (leading bit below 2^-6) share the step 2^-9
    step = np.exp2(np.maximum(e - 1, -6) - 3)
    r = np.round(a / step) * step            # numpy rounds halves to even
    r = np.minimum(r, E4M3_MAX)
    return np.where(np.signbit(x), -r, r)


def e4m3_codes(x: np.ndarray) -> np.ndarray:
    """The 8-bit codes of e4m3_round(x): sign, 4-bit exponent (bias 7), 3-bit mantissa."""
    v = e4m3_round(x)
    a = np.abs(v)
    m, e = np.frexp(a)
    normal = a >= 2.0 ** -6
    exp_field = np.where(normal, e - 1 + 7, 0)
    man = np.where(normal, a / np.exp2(e - 1) - 1.0, a / 2.0 ** -6) * 8.0
    code = (exp_field.astype(np.int64) << 3) | np.rint(man).astype(np.int64)
    code = np.where(a == 0, 0, code)
    return (code | (np.signbit(v).astype(np.int64) << 7)).astype(np.uint8)


def fwht_f32(x: np.ndarray) -> np.ndarray:
    """x H along the last axis (Sylvester order, unnormalised), butterflies in fp32."""
    y = np.array(x, dtype=np.float32)
    d = y.shape[-1]
    h = 1
    while h < d:
        z = y.reshape(y.shape[:-1] + (d // (2 * h), 2, h))
        a, b = z[..., 0, :].copy(), z[..., 1, :].copy()
        z[..., 0, :] = a + b
        z[..., 1, :] = a - b
        y = z.reshape(y.shape)
        h *= 2
    return y


def sign_vector(signs, d: int) -> np.ndarray:
    """+-1 per channel from d/32 32-bit words (bit c of word c // 32 set: negate)."""
    w = np.asarray(signs, dtype=np.uint64)
    bits = (w[np.arange(d) // 32] >> (np.arange(d) % 32).astype(np.uint64)) & 1
    return np.where(bits == 1, -1.0, 1.0).astype(np.float32)


def incoherent(x: np.ndarray, signs) -> np.ndarray:
    """Rows of x (fp32) times D H: channels negated where the sign bit is set, then H."""
    x32 = np.asarray(x, dtype=np.float32)
    return fwht_f32(x32 * sign_vector(signs, x32.shape[-1]))


def quantize(x: np.ndarray, block: int | None) -> tuple[np.ndarray, np.ndarray]:
    """e4m3 codes' values of fp32 x [BH, N, d] and the multipliers inv.

    block = 128: one multiplier per 128-row block of each leading index
    (rows past N count as zeros); None: one per leading index.
    """
    x32 = np.asarray(x, dtype=np.float32)
    BH, N, d = x32.shape
    if block is None:
        amax = np.max(np.abs(x32), axis=(1, 2), keepdims=True)
        per_row = lambda a: a
    else:
        nb = (N + block - 1) // block
        pad = np.zeros((BH, nb * block, d), dtype=np.float32)
        pad[:, :N] = x32
        amax = np.max(np.abs(pad.reshape(BH, nb, block, d)), axis=(2, 3))        # [BH, nb]
        per_row = lambda a: np.repeat(a, block, axis=1)[:, :N, None]
    amax = amax.astype(np.float32)
    inv = np.where(amax > 0, np.float32(E4M3_MAX) / np.where(amax > 0, amax, np.float32(1)),
                   np.float32(1)).astype(np.float32)
    y = (x32 * per_row(inv).astype(np.float32)).astype(np.float32)
    return e4m3_round(y), (inv.reshape(BH, -1) if block is not None else inv.reshape(BH))


def fp8_forward(q, k, v, causal: bool, scale: float, signs=None, qk_block: int | None = BLOCK):
    """O, LSE of exact attention on the 8-bit inputs, and the codes' parts.

    q, k, v: the bf16 inputs' values [B, H, N, d] (float64, exact).  signs:
    d/32 words for incoherent processing, or None for plain quantisation.
    qk_block: rows per Q/K scale (128, the block quantisation), or None for
    one scale per (batch, head) -- the per-tensor baseline of the same page's
    error table, which the library does not implement.
    Returns (O, LSE, parts) with parts = dict of the quantised values
    q8, k8, v8 ([B*H, N, d]) and multipliers inv_q, inv_k ([B*H, blocks] or
    [B*H]), inv_v ([B*H]).
    """
    B, H, N_q, d = q.shape
    N_kv = k.shape[2]
    q32 = np.asarray(q, dtype=np.float32).reshape(B * H, N_q, d)
    k32 = np.asarray(k, dtype=np.float32).reshape(B * H, N_kv, d)
    v32 = np.asarray(v, dtype=np.float32).reshape(B * H, N_kv, d)
    s = scale
    if signs is not None:
        q32, k32 = incoherent(q32, signs), incoherent(k32, signs)
        s = scale / d                        # (Q D H)(K D H)^T = d Q K^T
    q8, inv_q = quantize(q32, qk_block)
    k8, inv_k = quantize(k32, qk_block)
    v8, inv_v = quantize(v32, None)
    if qk_block is None:
        qd = q8 / inv_q.astype(np.float64)[:, None, None]
        kd = k8 / inv_k.astype(np.float64)[:, None, None]
    else:
        qd = q8 / np.repeat(inv_q.astype(np.float64), qk_block, axis=1)[:, :N_q, None]
        kd = k8 / np.repeat(inv_k.astype(np.float64), qk_block, axis=1)[:, :N_kv, None]
    vd = v8 / inv_v.astype(np.float64)[:, None, None]
    o, lse = attention_forward(qd.reshape(B, H, N_q, d), kd.reshape(B, H, N_kv, d),
                               vd.reshape(B, H, N_kv, d), causal=causal, scale=s)
    parts = dict(q8=q8, k8=k8, v8=v8, inv_q=inv_q, inv_k=inv_k, inv_v=inv_v)
    return o, lse, parts
