"""Device building blocks on the GPU, each against the CPU.

* both 2^x paths on a dense grid: the FMA-pipe cubic within 2e-4 of exact
  2^x (the bound fixed for the emulation) and within fp32 rounding of the
  oracle's float64 restatement of the same steps;
* one TMA-loaded tcgen05 tile product in each operand form the attention
  kernels use (both operands K-major; B N-major; A from tensor memory);
* the watchdog: a wait that nothing satisfies runs out, the status reads
  FA_ERR_TIMEOUT, and the context keeps working.
"""
import numpy as np
import pytest

import exact_attention_74_gb300 as fa
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch
    assert torch.cuda.is_available()
    fa.library()
    return torch


def _exp2(torch, x, mode):
    xd = torch.from_numpy(x.astype(np.float32)).cuda()
    yd = torch.empty_like(xd)
    assert fa.fa_test_exp2(xd.data_ptr(), yd.data_ptr(), xd.numel(), mode, 0) == fa.FA_OK
    torch.cuda.synchronize()
    return yd.cpu().numpy().astype(np.float64)


def test_exp2_emulation_error_bound(torch):
    x = np.concatenate([np.linspace(-126.0, 8.0, 2_000_001),
                        np.linspace(-1.0, 1.0, 400_001),
                        np.arange(-126, 9, dtype=np.float64)]).astype(np.float32).astype(np.float64)
    y = _exp2(torch, x, 1)
    rel = np.abs(y / np.exp2(x) - 1.0)
    assert rel.max() <= 2e-4, rel.max()
    # the same steps in float64 (oracle): agreement up to fp32 rounding
    ref = oracle.exp2_cubic(x)
    assert np.max(np.abs(y / ref - 1.0)) <= 2e-6
    # exact powers of two at integers
    ints = np.arange(-126, 9, dtype=np.float64)
    assert np.array_equal(_exp2(torch, ints, 1), np.exp2(ints))


def test_exp2_hardware_unit(torch):
    x = np.linspace(-126.0, 8.0, 1_000_001).astype(np.float32).astype(np.float64)
    y = _exp2(torch, x, 0)
    assert np.max(np.abs(y / np.exp2(x) - 1.0)) <= 1e-6


def test_exp2_masked_input_is_negligible(torch):
    y = _exp2(torch, np.array([-np.inf, -1e30, -200.0]), 1)
    assert np.all(y <= 2.0 ** -125)
    y = _exp2(torch, np.array([-np.inf]), 0)
    assert y[0] == 0.0


@pytest.mark.parametrize("K", [64, 128])
@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4, 5])
def test_mma_tile(torch, K, mode):
    rng = np.random.default_rng(1000 + K + mode)
    a_bits = fa_inputs_bits(rng, (K, 128) if mode & 4 else (128, K))
    b_bits = fa_inputs_bits(rng, (K, 128) if mode & 1 else (128, K))
    A, B = gu.dev_bf16(a_bits), gu.dev_bf16(b_bits)
    C = torch.full((128, 128), float("nan"), dtype=torch.float32, device="cuda")
    assert fa.fa_test_mma_tile(A.data_ptr(), B.data_ptr(), C.data_ptr(), K, mode, 0) == fa.FA_OK
    assert fa.fa_get_last_device_status(0) == fa.FA_OK
    a = gu.fa_inputs.bf16_bits_to_f64(a_bits)
    b = gu.fa_inputs.bf16_bits_to_f64(b_bits)
    a = a.T if mode & 4 else a
    ref = a @ b if mode & 1 else a @ b.T
    got = C.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - ref)) <= 1e-4 * np.max(np.abs(ref)) + 1e-5


@pytest.mark.parametrize("K", [64, 128])
@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_mma_pair(torch, K, mode):
    """One 256 x 128 x K product shared by the two CTAs of a cluster
    (cta_group::2): rows 0-127 of A and C in CTA 0, 128-255 in CTA 1, B's N
    columns split between them; A from shared or tensor memory, B K- or
    N-major."""
    rng = np.random.default_rng(2000 + K + mode)
    a_bits = fa_inputs_bits(rng, (256, K))
    b_bits = fa_inputs_bits(rng, (K, 128) if mode & 1 else (128, K))
    A, B = gu.dev_bf16(a_bits), gu.dev_bf16(b_bits)
    C = torch.full((256, 128), float("nan"), dtype=torch.float32, device="cuda")
    assert fa.fa_test_mma_pair(A.data_ptr(), B.data_ptr(), C.data_ptr(), K, mode, 0) == fa.FA_OK
    assert fa.fa_get_last_device_status(0) == fa.FA_OK
    a = gu.fa_inputs.bf16_bits_to_f64(a_bits)
    b = gu.fa_inputs.bf16_bits_to_f64(b_bits)
    ref = a @ b if mode & 1 else a @ b.T
    got = C.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(got - ref)) <= 1e-4 * np.max(np.abs(ref)) + 1e-5


def fa_inputs_bits(rng, shape):
    return gu.fa_inputs.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def test_watchdog_times_out_without_hanging(torch):
    assert fa.fa_get_last_device_status(0) == fa.FA_OK
    assert fa.fa_test_wait_timeout(20_000_000, 0) == fa.FA_OK      # 20 ms
    assert fa.fa_get_last_device_status(0) == fa.FA_ERR_TIMEOUT
    assert fa.fa_get_last_device_status(0) == fa.FA_OK            # read clears it
    # the context is still usable
    x = torch.ones(16, device="cuda")
    assert float((x * 2).sum().item()) == 32.0


@pytest.mark.parametrize("mode", [0, 1])
def test_mma_fp8_tile(torch, mode):
    """e4m3 rounding on the device (nearest even) and one kind::f8f6f4 tile
    product, A from shared or tensor memory, against PyTorch's float8_e4m3fn
    conversion and an fp64 product of the decoded values."""
    rng = np.random.default_rng(811 + mode)
    A = (rng.standard_normal((128, 128)) * np.exp(rng.uniform(-6, 5, (128, 128)))).astype(np.float32)
    B = (rng.standard_normal((128, 128)) * 4.0).astype(np.float32)
    A = np.clip(A, -440.0, 440.0)        # saturation is checked below, separately
    A[0, :8] = [0.0, -0.0, 1.0, -1.0, 0.0625, 1.0 / 512, 3.0 / 1024, 448.0]
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    c = torch.full((128, 128), float("nan"), device="cuda")
    codes = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    assert fa.fa_test_mma_fp8(a.data_ptr(), b.data_ptr(), c.data_ptr(), codes.data_ptr(), mode, 0) == fa.FA_OK
    assert fa.fa_get_last_device_status(0) == fa.FA_OK
    ref_a = torch.from_numpy(A).to(torch.float8_e4m3fn)
    ref_b = torch.from_numpy(B).to(torch.float8_e4m3fn)
    got = codes.cpu()
    assert torch.equal(got, ref_a.view(torch.uint8)), "e4m3 codes differ from float8_e4m3fn"
    expect = ref_a.to(torch.float64).numpy() @ ref_b.to(torch.float64).numpy().T
    out = c.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(out))
    assert np.max(np.abs(out - expect)) <= 1e-5 * (1.0 + np.max(np.abs(expect)))


def test_e4m3_saturates(torch):
    A = np.zeros((128, 128), dtype=np.float32)
    A[0, :4] = [1000.0, -1000.0, 449.0, 464.0]
    B = np.zeros((128, 128), dtype=np.float32)
    a, b = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    c = torch.empty((128, 128), device="cuda")
    codes = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    assert fa.fa_test_mma_fp8(a.data_ptr(), b.data_ptr(), c.data_ptr(), codes.data_ptr(), 0, 0) == fa.FA_OK
    got = codes.cpu().numpy()[0, :4]
    assert list(got) == [0x7E, 0xFE, 0x7E, 0x7E]      # +-448, the largest finite e4m3
