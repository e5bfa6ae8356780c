"""The allocation-free few-row GEMM entry point.

Some callers of this library cannot allocate device memory for it: their heap
belongs to another allocator that must stay its only owner, or they run on a
path that must never enter the driver's allocation code. They call
fk_gemm_bf16_splitk_noalloc, which keeps the split-K partial sums and arrival
counters in a fixed array inside the library instead of a caller buffer. Its
results must equal those of fk_gemm_bf16_splitk with a caller buffer, call
after call (the array keeps the previous call's contents), and shapes whose
scratch would not fit must be refused before anything runs.

This file is collected last, so a run that stops at the first failure has run
every other test first; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from helpers import err_scale, to_dev_bf16

pytestmark = pytest.mark.gpu


def _noalloc(fk, x, w, fp32):
    import torch
    P, K = x.shape
    N = w.shape[0]
    y = torch.empty((P, N), dtype=torch.float32 if fp32 else torch.bfloat16, device="cuda")
    lib = fk.load()
    st = lib.fk_gemm_bf16_splitk_noalloc(x.data_ptr(), w.data_ptr(), P, K, N, y.data_ptr(), 1 if fp32 else 0,
                                         torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.fk_last_error().decode()
    return y


# two calls in a row with different inputs: the first takes the fused
# last-CTA reduction (<= 8 rows), the second the separate reduction kernel
@pytest.mark.parametrize("order", [0, 1])
def test_noalloc_matches_caller_scratch(fk, order):
    import torch
    lib = fk.load()
    assert lib.fk_gemm_bf16_splitk_noalloc_limit() == 8 << 20
    cases = [(1, 4096, 14336, True, 31), (16, 4096, 4096, False, 32)]
    if order:
        cases = cases[::-1]
    for P, K, N, fp32, s in cases:
        assert lib.fk_gemm_bf16_splitk_scratch_bytes(P, K, N) <= lib.fk_gemm_bf16_splitk_noalloc_limit()
        xb = synth.normal_bf16(synth.SEED_GEMM_X, s, (P, K), 1.0)
        wb = synth.normal_bf16(synth.SEED_WEIGHTS, s, (N, K), 0.02)
        x, w = to_dev_bf16(xb), to_dev_bf16(wb)
        want = fk.gemm_splitk(x, w, out_fp32=fp32)
        got = _noalloc(fk, x, w, fp32)
        torch.cuda.synchronize()
        ref = want.float().cpu().numpy()
        assert err_scale(got.float().cpu().numpy(), ref) < (2e-5 if fp32 else 6e-3)
        assert torch.equal(got, want)  # same kernel, same split plan: bitwise equal
        # and both against the float64 oracle, within the GEMM tests' gate
        exact = oracle.gemm(oracle.bf16_to_f64(xb), oracle.bf16_to_f64(wb))
        assert err_scale(got.float().cpu().numpy(), exact) < (2e-5 if fp32 else 6e-3)


def test_noalloc_refuses_oversized_scratch(fk):
    import torch
    lib = fk.load()
    P, K, N = 64, 4096, 128256  # needs ~32 MB of partial sums
    assert lib.fk_gemm_bf16_splitk_scratch_bytes(P, K, N) > lib.fk_gemm_bf16_splitk_noalloc_limit()
    x = torch.zeros((P, K), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    y = torch.full((P, N), 7.0, dtype=torch.float32, device="cuda")
    st = lib.fk_gemm_bf16_splitk_noalloc(x.data_ptr(), w.data_ptr(), P, K, N, y.data_ptr(), 1,
                                         torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 9, st  # FK_ERR_WORKSPACE, nothing launched
    assert b"scratch" in lib.fk_last_error()
    assert torch.all(y == 7.0)
