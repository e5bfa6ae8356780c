"""Attention kernels against the oracle's attention ("N7 · model/forward-parity",
Thm 1: causal GQA attention; sliding window of the Gemma-style local layers)."""
import math

import numpy as np
import pytest

import oracle
import synth
from helpers import to_dev_bf16

pytestmark = pytest.mark.gpu


def _case(B, Hq, Hkv, hd, cap, seed):
    """q [B, Hq*hd]; k [B, Hkv, cap, hd]; v transposed [B, Hkv, hd, cap]."""
    q = synth.normal_bf16(seed, 1, (B, Hq * hd), 1.0)
    k = synth.normal_bf16(seed, 2, (B, Hkv, cap, hd), 1.0)
    v = synth.normal_bf16(seed, 3, (B, Hkv, hd, cap), 1.0)
    return q, k, v


@pytest.mark.parametrize("B,Hq,Hkv,hd,ctx,window", [
    (1, 4, 1, 64, 1, 0), (3, 9, 3, 64, 77, 0), (2, 32, 8, 128, 2049, 0), (32, 32, 8, 128, 300, 0),
    (1, 16, 8, 256, 1500, 1024), (2, 2, 1, 256, 40, 16), (4, 8, 8, 128, 1025, 0)])
def test_decode_attention_vs_oracle(fk, B, Hq, Hkv, hd, ctx, window):
    import torch
    cap = (ctx + 5 + 63) // 64 * 64
    q, k, v = _case(B, Hq, Hkv, hd, cap, seed=B * 100 + hd)
    out = fk.attention_decode(to_dev_bf16(q), to_dev_bf16(k), to_dev_bf16(v), ctx, window)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().reshape(B, Hq, hd)
    qf, kf, vf = (oracle.bf16_to_f64(a) for a in (q, k, v))
    for b in range(B):
        ref = oracle.attention(qf[b].reshape(1, Hq, hd), kf[b, :, :ctx].transpose(1, 0, 2),
                               vf[b, :, :, :ctx].transpose(2, 0, 1), np.array([ctx - 1]), np.arange(ctx), window,
                               1.0 / math.sqrt(hd))[0]
        # bf16 output rounding (2^-9 relative) on values of size <= max|v|
        np.testing.assert_allclose(got[b], ref, atol=1e-3, rtol=4e-3)
