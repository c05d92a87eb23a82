"""The device-memory check at the C-ABI boundary, on a GPU.

Every entry point refuses, with FA_ERR_INVALID and before building a tensor
map or launching anything, a tensor or workspace pointer whose memory the
current device cannot address as device memory.  The refused case here is
pinned host memory (from torch's pin_memory, i.e. cudaHostAlloc): it is
host memory that a kernel could still reach on this machine, so even a
regression of the check could not fault.  The accepted case is every other
GPU test, whose buffers are torch device allocations (views into them at
256-byte offsets included).
"""
import pytest

import exact_attention_74_gb300 as fa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch
    assert torch.cuda.is_available()
    fa.library()
    return torch


def _tensors(torch, B=1, H=2, N=256, d=128):
    dev = [torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda") for _ in range(8)]
    lse = torch.zeros((B, H, N), dtype=torch.float32, device="cuda")
    pinned = torch.zeros((B, H, N, d), dtype=torch.bfloat16).pin_memory()
    pinned_lse = torch.zeros((B, H, N), dtype=torch.float32).pin_memory()
    return dev, lse, pinned, pinned_lse


def test_forward_refuses_pinned_host_memory(torch):
    B, H, N, d = 1, 2, 256, 128
    (q, k, v, o, *_), lse, pinned, pinned_lse = _tensors(torch, B, H, N, d)
    p = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr()]
    assert fa.fa_fwd(*p, B, H, N, N, d, 0, 0.088, 0) == fa.FA_OK
    for i in range(5):
        bad = list(p)
        bad[i] = pinned_lse.data_ptr() if i == 4 else pinned.data_ptr()
        assert fa.fa_fwd(*bad, B, H, N, N, d, 0, 0.088, 0) == fa.FA_ERR_INVALID, i
    ws_bytes = fa.fa_fwd_fp8_workspace_bytes(B, H, N, N, d)
    ws_host = torch.empty(ws_bytes + 256, dtype=torch.uint8).pin_memory()
    base = (ws_host.data_ptr() + 255) // 256 * 256
    assert fa.fa_fwd_fp8(*p, B, H, N, N, d, 0, 0.088, None, base, ws_bytes, 0) == fa.FA_ERR_INVALID
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status(0) == fa.FA_OK


def test_backward_refuses_pinned_host_memory(torch):
    B, H, N, d = 1, 2, 256, 128
    (q, k, v, o, do, dq, dk, dv), lse, pinned, pinned_lse = _tensors(torch, B, H, N, d)
    need = fa.fa_bwd_workspace_bytes(B, H, N, N, d)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    p = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
         dq.data_ptr(), dk.data_ptr(), dv.data_ptr()]
    assert fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                     B, H, N, N, d, 0, 0.088, 0) == fa.FA_OK
    assert fa.fa_bwd(*p, B, H, N, N, d, 0, 0.088, ws.data_ptr(), need, 0) == fa.FA_OK
    for i in range(9):
        bad = list(p)
        bad[i] = pinned_lse.data_ptr() if i == 5 else pinned.data_ptr()
        assert fa.fa_bwd(*bad, B, H, N, N, d, 0, 0.088, ws.data_ptr(), need, 0) == fa.FA_ERR_INVALID, i
        assert fa.fa_bwd_noalloc(*bad, B, H, N, N, d, 0, 0.088, 0) == fa.FA_ERR_INVALID, i
    ws_host = torch.empty(need + 256, dtype=torch.uint8).pin_memory()
    base = (ws_host.data_ptr() + 255) // 256 * 256
    assert fa.fa_bwd(*p, B, H, N, N, d, 0, 0.088, base, need, 0) == fa.FA_ERR_INVALID
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status(0) == fa.FA_OK
