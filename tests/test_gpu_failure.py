"""The bounded-wait failure path on the GPU, made to run out on purpose.

With the test flags TQ_GEMV_TEST_STALL / TQ_GEMM_TEST_STALL the first CTA of
the launch never issues one of its copies (a barrier phase that nothing
completes) and every bounded wait of that launch gives up after about 20 ms.
No trap, no fault and no endless wait is involved: the kernel records the
event, winds down, and the host reads the status.  The tests then check that
the context is still usable -- the next clean launch reproduces a clean
result bit for bit."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ternary_weight_fwht128_gb300 as tq
from ternary_weight_fwht128_gb300 import synth
from tq_testutil import to_dev_bf16

pytestmark = pytest.mark.gpu

TQ_GEMV_TEST_STALL = 0x100
TQ_GEMM_TEST_STALL = 0x100


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tq.lib()
    torch.cuda.set_device(0)


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("N,K,M,fmt", [(27648, 5120, 1, tq.TQ_PACK_2BIT), (5120, 27648, 4, tq.TQ_PACK_BASE3)])
def test_gemv_stall_reports_timeout_then_recovers(N, K, M, fmt):
    assert tq.gemv_path(N, K, M, fmt) == tq.TQ_GEMV_TENSOR_MEMORY
    W = synth.weights(N, K, 61, dtype="bf16")
    c2, c3, s = tq.quantize_pack(to_dev_bf16(W), fmt)
    codes = c2 if fmt == tq.TQ_PACK_2BIT else c3
    x = to_dev_bf16(synth.activations(M, K, 62))
    ref = tq.gemv(codes, s, x, K, fmt)
    tq.device_fault()  # clean so far
    L = tq.lib()
    y = torch.zeros(M, N, device="cuda")
    st = L.tq_gemv_ex(codes.data_ptr(), codes.stride(0), fmt, s.data_ptr(), s.stride(0), N, K, x.data_ptr(),
                      x.stride(0), M, y.data_ptr(), y.stride(0), TQ_GEMV_TEST_STALL, _stream())
    assert st == tq.TQ_OK, tq.status_string(st)
    assert L.tq_device_fault() == tq.TQ_ERR_TIMEOUT
    assert L.tq_device_fault() == tq.TQ_OK  # read and cleared
    y2 = tq.gemv(codes, s, x, K, fmt)
    tq.device_fault()
    assert torch.equal(y2, ref)


def test_gemv_stall_needs_the_tensor_memory_kernel():
    """The mma.sync kernel has no waits to stall: the flag is refused there."""
    N, K, M = 96, 262144, 16
    assert tq.gemv_path(N, K, M) == tq.TQ_GEMV_MMA_SYNC
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    p = dummy.data_ptr()
    st = tq.lib().tq_gemv_ex(p, K // 4, tq.TQ_PACK_2BIT, p, K // 128, N, K, p, K, M, p, N, TQ_GEMV_TEST_STALL,
                             _stream())
    assert st == tq.TQ_ERR_UNSUPPORTED


@pytest.mark.parametrize("N,K,M", [(2048, 1280, 512), (5120, 5120, 2048)])
def test_gemm_stall_reports_timeout_then_recovers(N, K, M):
    W = synth.weights(N, K, 71, dtype="bf16")
    c2, _, s = tq.quantize_pack(to_dev_bf16(W), tq.TQ_PACK_2BIT)
    x = to_dev_bf16(synth.activations(M, K, 72))
    ws = torch.empty(tq.gemm_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    ref = tq.gemm(c2, s, x, K, workspace=ws)
    tq.gemm_check_range(ws)
    L = tq.lib()
    y = torch.zeros(M, N, device="cuda")
    st = L.tq_gemm_ex(c2.data_ptr(), c2.stride(0), tq.TQ_PACK_2BIT, s.data_ptr(), s.stride(0), N, K, x.data_ptr(),
                      x.stride(0), M, y.data_ptr(), y.stride(0), ws.data_ptr(), ws.numel(), TQ_GEMM_TEST_STALL,
                      _stream())
    assert st == tq.TQ_OK, tq.status_string(st)
    assert L.tq_gemm_check_range(ws.data_ptr(), _stream()) == tq.TQ_ERR_TIMEOUT
    assert L.tq_device_fault() == tq.TQ_OK  # the GEMM reports through its workspace
    y2 = tq.gemm(c2, s, x, K, workspace=ws)
    tq.gemm_check_range(ws)
    assert torch.equal(y2, ref)


@pytest.mark.parametrize("scale_exp", [110, -110])
def test_gemv_reports_activations_out_of_range(scale_exp):
    """A group of x whose rotation lies beyond what the e4m3 pieces represent
    (|x'| >= 2^108, or a positive max below 2^-93) is recorded, and
    tq_device_fault reports TQ_ERR_RANGE once; the next clean call is clean."""
    N, K, M = 27648, 5120, 1
    assert tq.gemv_path(N, K, M) == tq.TQ_GEMV_TENSOR_MEMORY
    W = synth.weights(N, K, 81, dtype="bf16")
    c2, _, s = tq.quantize_pack(to_dev_bf16(W), tq.TQ_PACK_2BIT)
    xb = synth.activations(M, K, 82)
    x = to_dev_bf16(xb).float()
    x[:, 256:384] *= 2.0 ** scale_exp
    x = x.to(torch.bfloat16)
    tq.device_fault()
    tq.gemv(c2, s, x, K)
    assert tq.lib().tq_device_fault() == tq.TQ_ERR_RANGE
    tq.gemv(c2, s, to_dev_bf16(xb), K)
    assert tq.lib().tq_device_fault() == tq.TQ_OK


@pytest.mark.parametrize("N,K,M", [(5120, 27648, 1), (27648, 5120, 2)])
def test_gemv_rotate_next_stall_reports_timeout_then_recovers(N, K, M):
    """The chained form (rank 0 of each cluster reduces every row): the
    stalled CTA is rank 0 of the first cluster, which its peers push all
    their rows into; the launch still winds down, reports TQ_ERR_TIMEOUT, and
    the next clean call reproduces y and x' bit for bit."""
    W = synth.weights(N, K, 91, dtype="bf16")
    c2, _, s = tq.quantize_pack(to_dev_bf16(W), tq.TQ_PACK_2BIT)
    x = to_dev_bf16(synth.activations(M, K, 92))
    ref_y, ref_xn = tq.gemv_rotate_next(c2, s, x, K)
    tq.device_fault()
    y, xn = tq.gemv_rotate_next(c2, s, x, K, flags=TQ_GEMV_TEST_STALL)
    torch.cuda.synchronize()
    assert tq.lib().tq_device_fault() == tq.TQ_ERR_TIMEOUT
    y2, xn2 = tq.gemv_rotate_next(c2, s, x, K)
    tq.device_fault()
    assert torch.equal(y2, ref_y) and torch.equal(xn2, ref_xn)
