"""tq_gemm_noalloc: the prefill GEMM for callers that cannot allocate device
memory (it takes its workspace from a fixed scratch array inside the library).

Called through the C ABI on two calls in a row, each compared with tq_gemm on
the same inputs within the tolerance the parity tests use.  This file is
collected last, so a run that stops at the first failure has already run every
other test; it also passes alone in a fresh process (the first call on the
device does the one-time set-up)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import ternary_weight_fwht128_gb300 as tq
from ternary_weight_fwht128_gb300 import synth
from tq_testutil import check_y, to_dev_bf16

pytestmark = pytest.mark.gpu


def test_gemm_noalloc_matches_gemm_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    L = tq.lib()
    N, K, M = 1000, 1280, 300
    W = synth.weights(N, K, 77, dtype="bf16")
    c2, _, s = tq.quantize_pack(to_dev_bf16(W), tq.TQ_PACK_2BIT)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        x = to_dev_bf16(synth.activations(M, K, 100 + call))
        ref = tq.gemm(c2, s, x, K, tq.TQ_PACK_2BIT)
        y = torch.full((M, N), float("nan"), device="cuda")
        st = L.tq_gemm_noalloc(c2.data_ptr(), c2.stride(0), tq.TQ_PACK_2BIT, s.data_ptr(), s.stride(0), N, K,
                               x.data_ptr(), x.stride(0), M, y.data_ptr(), y.stride(0), stream)
        assert st == tq.TQ_OK, tq.status_string(st)
        torch.cuda.synchronize()
        check_y(y.cpu().numpy(), ref.cpu().numpy().astype(np.float64), f"no-alloc call {call}")

