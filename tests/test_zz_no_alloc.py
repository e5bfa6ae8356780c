"""The allocation-free decode-attention entry point.

Callers that cannot give the library a scratch buffer (their device memory is
owned by another allocator, or their path must not enter the driver's
allocation code) use fk_attention_decode_noalloc. The decode kernel merges its
split partials inside a thread-block cluster, so the entry point needs no
device memory at all; its results must equal those of fk_attention_decode with
a caller buffer, call after call and for any size. Runs last so that a
stop-at-first-failure run has run everything else first; it also passes alone
in a fresh process.
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
    assert lib.fk_attention_decode_noalloc_limit() == 0  # nothing reserved
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


def test_noalloc_large_batch(fk):
    """A batch whose split partials would take megabytes in global memory."""
    import torch
    B, Hq, Hkv, hd, ctx = 64, 32, 8, 128, 1000
    cap = 1024
    q = to_dev_bf16(synth.normal_bf16(21, 1, (B, Hq * hd), 1.0))
    k = to_dev_bf16(synth.normal_bf16(21, 2, (B, Hkv, cap, hd), 1.0))
    v = to_dev_bf16(synth.normal_bf16(21, 3, (B, Hkv, hd, cap), 1.0))
    want = fk.attention_decode(q, k, v, ctx, 0)
    got = torch.empty_like(q)
    _call_noalloc(fk, q, k, v, ctx, 0, got)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
