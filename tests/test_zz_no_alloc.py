"""The allocation-free decode-attention entry point.

Callers that cannot give the library a scratch buffer (their device memory is
owned by another allocator, or their path must not enter the driver's
allocation code) use fk_attention_decode_noalloc, whose split-KV partials live
in a fixed array inside the library. Its results must equal those of
fk_attention_decode with a caller buffer. Two calls in a row with different
inputs check that the array's leftover contents from the first call do not
leak into the second. Runs last so that a stop-at-first-failure run has run
everything else first; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

import synth
from helpers import to_dev_bf16

pytestmark = pytest.mark.gpu


def _call_noalloc(fk, q, k, v, ctx, window, out):
    import torch
    B, Hkv, cap, hd = k.shape
    Hq = q.shape[1] // hd
    lib = fk.load()
    st = lib.fk_attention_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, Hq, Hkv, hd, cap, ctx, window,
                                         out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.fk_last_error().decode()


@pytest.mark.parametrize("B,Hq,Hkv,hd,ctx,window", [(32, 32, 8, 128, 2048, 0), (1, 16, 8, 256, 1500, 1024)])
def test_noalloc_matches_scratch_entry_point(fk, B, Hq, Hkv, hd, ctx, window):
    import torch
    lib = fk.load()
    assert lib.fk_attention_decode_noalloc_limit() == 4 << 20
    for call, seed in enumerate((11, 12)):  # two calls in a row, different inputs
        cap = (ctx + 3 + 63) // 64 * 64
        q = to_dev_bf16(synth.normal_bf16(seed, 1, (B, Hq * hd), 1.0))
        k = to_dev_bf16(synth.normal_bf16(seed, 2, (B, Hkv, cap, hd), 1.0))
        v = to_dev_bf16(synth.normal_bf16(seed, 3, (B, Hkv, hd, cap), 1.0))  # transposed values
        want = fk.attention_decode(q, k, v, ctx - call, window)
        got = torch.empty_like(q)
        _call_noalloc(fk, q, k, v, ctx - call, window, got)
        torch.cuda.synchronize()
        torch.testing.assert_close(got.float(), want.float(), atol=1e-3, rtol=4e-3)
        assert torch.equal(got, want)  # same kernel, same split plan: bitwise equal


def test_noalloc_rejects_oversize(fk):
    import torch
    lib = fk.load()
    B, Hq, Hkv, hd, ctx = 256, 64, 8, 256, 4096   # partials far above the 4 MiB array
    assert lib.fk_attention_decode_scratch_bytes(B, Hq, Hkv, hd, ctx) > lib.fk_attention_decode_noalloc_limit()
    q = torch.zeros((B, Hq * hd), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((1, 16), dtype=torch.bfloat16, device="cuda")  # never read: rejected before launch
    out = torch.empty_like(q)
    st = lib.fk_attention_decode_noalloc(q.data_ptr(), kv.data_ptr(), kv.data_ptr(), B, Hq, Hkv, hd, ctx, ctx, 0,
                                         out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 9  # FK_ERR_WORKSPACE
    assert b"fixed" in lib.fk_last_error()
