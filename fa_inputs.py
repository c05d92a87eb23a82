"""Seeded synthetic inputs for exact attention, shared by the CUDA-path tests,
the bench and the oracle's tests.

This module holds no attention arithmetic.  It draws random numbers, rounds
them to bf16 (round-to-nearest-even) and lays them out as ``[B, H, N, d]``
with ``d`` innermost.  Both sides of every parity check consume the same bf16
bit patterns: the CUDA path as ``torch.bfloat16`` device tensors, the oracle
as exactly-upcast float64 arrays.

Workload recipes (the shapes follow the benchmark settings of
"FlashAttention-3: Fast and Accurate Attention with Asynchrony and
Low-precision", §実験設定, and the hdim 128/64, seqlen 8192 rows of
"論文解説: FlashAttention-4 — Algorithm and Kernel Pipelining Co-Design for
Asymmetric Hardware Scaling", 実験結果):

* ``iid``     -- every element N(0, 1).
* ``stress``  -- Q, K iid N(0, 1); channels {0, 32, 64, 96} multiplied by 20
  in both Q and K (outlier channels); channel d-1 of Q set to 1 and channel
  d-1 of key j set to ``drift * j / (N_kv * scale)``, so the logits carry a
  term that rises by ``drift`` (natural-log units) across the keys and the
  running row maximum keeps rising.
* ``outlier`` -- N(0, 1) + N(0, 100) * Bernoulli(0.001) per element, the
  distribution of the numerical-error experiment of the FlashAttention-3
  notes (§数値誤差実験).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = [
    "f32_to_bf16_bits", "bf16_bits_to_f32", "bf16_bits_to_f64",
    "Workload", "WORKLOADS", "sweep_workloads", "make_qkv", "make_dout",
]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float64."""
    return bf16_bits_to_f32(bits).astype(np.float64)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: sizes, mask, softmax scale, input recipe, seed."""
    name: str
    B: int
    H: int
    N_q: int
    N_kv: int
    d: int
    causal: bool
    scale: float
    seed: int
    kind: str = "iid"          # "iid" | "stress" | "outlier"
    drift: float = 256.0       # stress only: logit rise across the keys

    def fwd_flops(self) -> float:
        """4*B*H*N_q*N_kv*d, halved when causal (the reporting convention)."""
        f = 4.0 * self.B * self.H * self.N_q * self.N_kv * self.d
        return f / 2 if self.causal else f

    def bwd_flops(self) -> float:
        return 2.5 * self.fwd_flops()

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _wl(name, B, H, N, d, causal, seed, kind="iid"):
    return Workload(name, B, H, N, N, d, causal, 1.0 / math.sqrt(d), seed, kind)


# The five workloads: tiny d=64; B4 H16 N4096 d128; the 16k-token sequence
# sweep; the rescaling stress case; the backward case.  Seed base 20260 + index.
WORKLOADS = {
    "tiny": _wl("tiny", 1, 1, 256, 64, False, 20261),
    "tiny_causal": _wl("tiny_causal", 1, 1, 256, 64, True, 20261),
    "fwd_4k": _wl("fwd_4k", 4, 16, 4096, 128, False, 20262),
    "fwd_4k_causal": _wl("fwd_4k_causal", 4, 16, 4096, 128, True, 20262),
    "stress_8k": _wl("stress_8k", 2, 16, 8192, 128, True, 20264, "stress"),
    "bwd_8k": _wl("bwd_8k", 2, 16, 8192, 128, True, 20265),
    # 16k tokens at head dimension 256 (FlashAttention-3's largest, where
    # its 8-bit measurements centre), scale 1/16
    "hdim64_8k": Workload("hdim64_8k", 2, 16, 8192, 8192, 64, False, 0.125, 20266),
    "hdim256_8k": Workload("hdim256_8k", 2, 16, 8192, 8192, 256, False, 1.0 / 16.0, 20267),
    "hdim256_8k_causal": Workload("hdim256_8k_causal", 2, 16, 8192, 8192, 256, True, 1.0 / 16.0, 20267),
}


def sweep_workloads(causal: bool):
    """16384 tokens per batch: N in {1k..32k}, B = 16384 // N (B = 1 at 32k)."""
    out = []
    for n in (1024, 2048, 4096, 8192, 16384, 32768):
        b = max(1, 16384 // n)
        out.append(_wl(f"sweep_{n}{'_causal' if causal else ''}", b, 16, n, 128,
                       causal, 20263))
    return out


def _normal(rng, shape):
    return rng.standard_normal(size=shape, dtype=np.float32)


def make_qkv(w: Workload):
    """Return (q, k, v) as uint16 bf16 bit arrays of shape [B, H, N, d]."""
    qs = (w.B, w.H, w.N_q, w.d)
    ks = (w.B, w.H, w.N_kv, w.d)
    rq = np.random.default_rng(w.seed)
    rk = np.random.default_rng(w.seed + 1)
    rv = np.random.default_rng(w.seed + 2)
    if w.kind == "iid":
        q, k, v = _normal(rq, qs), _normal(rk, ks), _normal(rv, ks)
    elif w.kind == "outlier":
        q, k, v = (_outlier(r, s) for r, s in ((rq, qs), (rk, ks), (rv, ks)))
    elif w.kind == "stress":
        q, k, v = _normal(rq, qs), _normal(rk, ks), _normal(rv, ks)
        for c in (0, 32, 64, 96):
            if c < w.d - 1:
                q[..., c] *= 20.0
                k[..., c] *= 20.0
        q[..., w.d - 1] = 1.0
        j = np.arange(w.N_kv, dtype=np.float64)
        k[..., w.d - 1] = (w.drift * j / (w.N_kv * w.scale)).astype(np.float32)
    else:
        raise ValueError(f"unknown input kind {w.kind!r}")
    return f32_to_bf16_bits(q), f32_to_bf16_bits(k), f32_to_bf16_bits(v)


def make_dout(w: Workload):
    """dO for the backward pass: iid N(0, 1), seed base + 3, bf16 bits."""
    r = np.random.default_rng(w.seed + 3)
    return f32_to_bf16_bits(_normal(r, (w.B, w.H, w.N_q, w.d)))


def _outlier(rng, shape):
    base = rng.standard_normal(size=shape, dtype=np.float32)
    big = rng.standard_normal(size=shape, dtype=np.float32) * 10.0
    hit = rng.random(size=shape, dtype=np.float32) < 0.001
    return base + np.where(hit, big, np.float32(0.0))
