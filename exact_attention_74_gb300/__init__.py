"""Exact attention on one NVIDIA GB300 (sm_103a): Python binding of the C ABI.

The functions with C names (``fa_fwd``, ``fa_fwd_ex``, ``fa_bwd``,
``fa_bwd_workspace_bytes``, ``fa_get_last_device_status``,
``fa_set_wait_timeout_ns``, ``fa_status_string`` and the ``fa_test_*``
entry points) marshal plain integers (device pointers, sizes) into the shared
library ``lib/libfa_gb300.so`` and return its status code.  ``forward`` and
``backward`` are thin conveniences over them for ``torch`` tensors
``[B, H, N, d]`` bf16 on the current CUDA device and stream; every step of the
computation runs in the library's kernels.  There is no fallback: if the
library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "FA_OK", "FA_ERR_INVALID", "FA_ERR_UNSUPPORTED", "FA_ERR_ALIGN", "FA_ERR_WORKSPACE",
    "FA_ERR_CUDA", "FA_ERR_TIMEOUT", "FAError", "library", "library_path",
    "fa_fwd", "fa_fwd_ex", "fa_fwd_fp8", "fa_fwd_fp8_workspace_bytes", "forward_fp8", "fa_bwd", "fa_bwd_workspace_bytes", "fa_get_last_device_status",
    "fa_bwd_noalloc", "FA_BWD_NOALLOC_MAX_WORKSPACE", "fa_bwd_ex", "fa_bwd_pair",
    "fa_set_wait_timeout_ns", "fa_status_string", "fa_test_exp2", "fa_test_mma_tile", "fa_test_mma_pair",
    "fa_test_mma_fp8", "fa_test_wait_timeout", "forward", "backward", "EXPORTED_SYMBOLS",
]

FA_OK, FA_ERR_INVALID, FA_ERR_UNSUPPORTED, FA_ERR_ALIGN = 0, 1, 2, 3
FA_ERR_WORKSPACE, FA_ERR_CUDA, FA_ERR_TIMEOUT = 4, 5, 6

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "lib", "libfa_gb300.so")

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_ll, _ull = ctypes.c_longlong, ctypes.c_ulonglong

# name -> (restype, argtypes), one line per declaration in include/fa.h and
# include/fa_testing.h
_SIGNATURES = {
    "fa_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp]),
    "fa_fwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _f, _i, _vp]),
    "fa_fwd_fp8_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "fa_fwd_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp]),
    "fa_bwd_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "fa_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                    _i, _i, _i, _i, _i, _i, _f, _vp, _sz, _vp]),
    "fa_bwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                       _i, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
    "fa_bwd_pair": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                         _i, _i, _i, _i, _i, _i, _f, _vp, _sz, _vp]),
    "fa_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                            _i, _i, _i, _i, _i, _i, _f, _vp]),
    "fa_get_last_device_status": (_i, [_vp]),
    "fa_set_wait_timeout_ns": (_i, [_ull]),
    "fa_status_string": (ctypes.c_char_p, [_i]),
    "fa_test_exp2": (_i, [_vp, _vp, _ll, _i, _vp]),
    "fa_test_mma_tile": (_i, [_vp, _vp, _vp, _i, _i, _vp]),
    "fa_test_mma_pair": (_i, [_vp, _vp, _vp, _i, _i, _vp]),
    "fa_test_mma_fp8": (_i, [_vp, _vp, _vp, _vp, _i, _vp]),
    "fa_test_wait_timeout": (_i, [_ull, _vp]),
}
EXPORTED_SYMBOLS = tuple(_SIGNATURES)

_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: status {status} ({fa_status_string(status)})")
        self.status = status


def library() -> ctypes.CDLL:
    """Load the shared library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(f"CUDA library not built: {library_path} is missing "
                               "(run __graft_entry__.build() or python -m exact_attention_74_gb300._build)")
        lib = ctypes.CDLL(library_path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _call(name, *args):
    return getattr(library(), name)(*args)


def fa_fwd(Q, K, V, O, LSE, B, H, N_q, N_kv, d, causal, scale, stream=0):
    return _call("fa_fwd", Q, K, V, O, LSE, B, H, N_q, N_kv, d, causal, scale, stream)


def fa_fwd_ex(Q, K, V, O, LSE, B, H, N_q, N_kv, d, causal, scale, tau, emu_per_32, stream=0):
    return _call("fa_fwd_ex", Q, K, V, O, LSE, B, H, N_q, N_kv, d, causal, scale, tau,
                 emu_per_32, stream)


def fa_fwd_fp8_workspace_bytes(B, H, N_q, N_kv, d):
    return _call("fa_fwd_fp8_workspace_bytes", B, H, N_q, N_kv, d)


def fa_fwd_fp8(Q, K, V, O, LSE, B, H, N_q, N_kv, d, causal, scale, signs, workspace, workspace_bytes,
               stream=0):
    """signs: None, or d/32 32-bit words (a sequence of ints, or a pointer)."""
    if signs is not None and not isinstance(signs, (int, ctypes.c_void_p)):
        if d in (128, 256) and len(signs) < d // 32:      # other d: the call answers UNSUPPORTED
            raise ValueError(f"signs: need d/32 = {d // 32} words, got {len(signs)}")
        signs = (ctypes.c_uint * len(signs))(*[int(x) & 0xffffffff for x in signs])
    return _call("fa_fwd_fp8", Q, K, V, O, LSE, B, H, N_q, N_kv, d, causal, scale, signs, workspace,
                 workspace_bytes, stream)


def fa_bwd_workspace_bytes(B, H, N_q, N_kv, d):
    return _call("fa_bwd_workspace_bytes", B, H, N_q, N_kv, d)


def fa_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N_q, N_kv, d, causal, scale,
           workspace, workspace_bytes, stream=0):
    return _call("fa_bwd", Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N_q, N_kv, d, causal, scale,
                 workspace, workspace_bytes, stream)


def fa_bwd_ex(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N_q, N_kv, d, causal, scale,
              deterministic, workspace, workspace_bytes, stream=0):
    return _call("fa_bwd_ex", Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N_q, N_kv, d, causal, scale,
                 deterministic, workspace, workspace_bytes, stream)


def fa_bwd_pair(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N_q, N_kv, d, causal, scale,
                workspace, workspace_bytes, stream=0):
    """fa_bwd at d = 64 on pairs of thread blocks sharing 256-key products."""
    return _call("fa_bwd_pair", Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N_q, N_kv, d, causal, scale,
                 workspace, workspace_bytes, stream)


# Bytes of scratch fa_bwd_noalloc can use (FA_BWD_NOALLOC_MAX_WORKSPACE in fa.h).
FA_BWD_NOALLOC_MAX_WORKSPACE = 16 << 20


def fa_bwd_noalloc(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N_q, N_kv, d, causal, scale, stream=0):
    """fa_bwd without a workspace argument, for callers that cannot allocate device memory."""
    return _call("fa_bwd_noalloc", Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N_q, N_kv, d, causal,
                 scale, stream)


def fa_get_last_device_status(stream=0):
    return _call("fa_get_last_device_status", stream)


def fa_set_wait_timeout_ns(ns):
    return _call("fa_set_wait_timeout_ns", ns)


def fa_status_string(status):
    return _call("fa_status_string", status).decode()


def fa_test_exp2(x, y, n, mode, stream=0):
    return _call("fa_test_exp2", x, y, n, mode, stream)


def fa_test_mma_tile(A, B, C, K, mode, stream=0):
    return _call("fa_test_mma_tile", A, B, C, K, mode, stream)


def fa_test_mma_pair(A, B, C, K, mode, stream=0):
    return _call("fa_test_mma_pair", A, B, C, K, mode, stream)


def fa_test_mma_fp8(A, B, C, A_codes, mode, stream=0):
    return _call("fa_test_mma_fp8", A, B, C, A_codes, mode, stream)


def fa_test_wait_timeout(timeout_ns, stream=0):
    return _call("fa_test_wait_timeout", timeout_ns, stream)


# ------------------------------------------------------- torch conveniences

def _stream_handle(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(t, shape, name):
    import torch
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != shape:
        raise ValueError(f"{name}: need a contiguous CUDA bf16 tensor of shape {shape}, "
                         f"got {t.dtype} {tuple(t.shape)} on {t.device}")


def forward(q, k, v, causal=False, scale=None, out=None, lse=None, stream=None,
            tau=None, emu_per_32=None):
    """O, LSE = attention(q, k, v) for bf16 tensors [B, H, N, d] on the GPU."""
    import torch
    B, H, N_q, d = q.shape
    N_kv = k.shape[2]
    _check(q, (B, H, N_q, d), "q")
    _check(k, (B, H, N_kv, d), "k")
    _check(v, (B, H, N_kv, d), "v")
    scale = d ** -0.5 if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N_q), dtype=torch.float32, device=q.device)
    s = _stream_handle(stream)
    if tau is None and emu_per_32 is None:
        st = fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                    B, H, N_q, N_kv, d, int(causal), scale, s)
    else:
        st = fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                       B, H, N_q, N_kv, d, int(causal), scale,
                       8.0 if tau is None else float(tau),
                       -1 if emu_per_32 is None else int(emu_per_32), s)
    if st != FA_OK:
        raise FAError(st, "fa_fwd")
    return out, lse


def forward_fp8(q, k, v, causal=False, scale=None, signs=None, out=None, lse=None, stream=None,
                workspace=None):
    """O, LSE on 8-bit copies of q, k, v (bf16 [B, H, N, d], d in {128, 256}, on the GPU).

    signs: None, or d / 32 32-bit words for incoherent processing; see fa_fwd_fp8."""
    import torch
    B, H, N_q, d = q.shape
    N_kv = k.shape[2]
    _check(q, (B, H, N_q, d), "q")
    _check(k, (B, H, N_kv, d), "k")
    _check(v, (B, H, N_kv, d), "v")
    scale = d ** -0.5 if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N_q), dtype=torch.float32, device=q.device)
    need = fa_fwd_fp8_workspace_bytes(B, H, N_q, N_kv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    st = fa_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N_q,
                    N_kv, d, int(causal), scale, signs, workspace.data_ptr(), workspace.numel(),
                    _stream_handle(stream))
    if st != FA_OK:
        raise FAError(st, "fa_fwd_fp8")
    return out, lse


def backward(q, k, v, o, do, lse, causal=False, scale=None, stream=None, workspace=None,
             deterministic=False, pair=False):
    """dQ, dK, dV for bf16 tensors [B, H, N, d] and fp32 LSE [B, H, N_q].

    pair=True runs fa_bwd_pair (d = 64 only; not with deterministic)."""
    import torch
    B, H, N_q, d = q.shape
    N_kv = k.shape[2]
    for t, n, name in ((q, N_q, "q"), (k, N_kv, "k"), (v, N_kv, "v"), (o, N_q, "o"), (do, N_q, "do")):
        _check(t, (B, H, n, d), name)
    scale = d ** -0.5 if scale is None else float(scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    need = fa_bwd_workspace_bytes(B, H, N_q, N_kv, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr())
    ws = (workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if pair:
        if deterministic:
            raise ValueError("pair=True has no fixed-order mode")
        st = fa_bwd_pair(*ptrs, B, H, N_q, N_kv, d, int(causal), scale, *ws)
    else:
        st = fa_bwd_ex(*ptrs, B, H, N_q, N_kv, d, int(causal), scale, int(deterministic), *ws)
    if st != FA_OK:
        raise FAError(st, "fa_bwd_pair" if pair else "fa_bwd")
    return dq, dk, dv
