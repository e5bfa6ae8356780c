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
    (1, 16, 8, 256, 1500, 1024), (2, 2, 1, 256, 40, 16), (4, 8, 8, 128, 1025, 0),
    # a cluster of 16 splits with fewer tiles than splits (window start mid-tile),
    # and a 2-split cluster over a ragged last tile
    (1, 8, 1, 128, 3000, 700), (1, 4, 4, 64, 130, 0)])
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


@pytest.mark.parametrize("B,S,pos0,Hq,Hkv,hd,window,ramp", [
    (1, 1024, 0, 4, 1, 128, 0, True), (2, 600, 0, 8, 2, 128, 0, False), (1, 700, 0, 4, 2, 64, 0, True),
    (1, 300, 200, 4, 1, 128, 0, True), (1, 900, 0, 4, 1, 128, 256, True), (1, 260, 0, 2, 1, 256, 64, False)])
def test_prefill_attention_vs_oracle(fk, B, S, pos0, Hq, Hkv, hd, window, ramp):
    """Prefill attention against the oracle. With ``ramp`` the keys grow along
    the sequence, so each query row's running maximum keeps rising from one
    key block to the next and the lazy O rescale of the tensor-core kernel runs
    many times."""
    import torch
    kv_len = pos0 + S
    cap = (kv_len + 63) // 64 * 64
    q = synth.normal_bf16(7, 11, (B * S, Hq * hd), 1.0)
    kf = synth.bf16_bits_to_f32(synth.normal_bf16(7, 12, (B, Hkv, cap, hd), 1.0))
    if ramp:  # scores grow ~linearly with the key position
        kf = kf * 0.25 + (np.arange(cap) / 64.0)[None, None, :, None].astype(np.float32)
    k = synth.f32_to_bf16_bits(kf)
    v = synth.normal_bf16(7, 13, (B, Hkv, hd, cap), 1.0)
    out = fk.attention_prefill(to_dev_bf16(q), to_dev_bf16(k), to_dev_bf16(v), S, pos0, window)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().reshape(B, S, Hq, hd)
    qf, kk, vv = (oracle.bf16_to_f64(a) for a in (q, k, v))
    qf = qf.reshape(B, S, Hq, hd)
    for b in range(B):
        ref = oracle.attention(qf[b], kk[b, :, :kv_len].transpose(1, 0, 2), vv[b, :, :, :kv_len].transpose(2, 0, 1),
                               pos0 + np.arange(S), np.arange(kv_len), window, 1.0 / math.sqrt(hd))
        # P is rounded to bf16 for the PV product (2^-9 relative) and the output to bf16
        np.testing.assert_allclose(got[b], ref, atol=1e-2, rtol=1e-2)


def _ring(a, cap, axis):
    """A linear cache [.., positions, ..] laid into a ring of cap slots along
    `axis` (position p in slot p mod cap; later positions overwrite earlier)."""
    n = a.shape[axis]
    shape = list(a.shape)
    shape[axis] = cap
    r = np.zeros(shape, dtype=a.dtype)
    for p in range(n):
        idx = [slice(None)] * a.ndim
        idx[axis] = p % cap
        src = [slice(None)] * a.ndim
        src[axis] = p
        r[tuple(idx)] = a[tuple(src)]
    return r


@pytest.mark.parametrize("B,Hq,Hkv,hd,ctx,window,cap", [(1, 8, 2, 128, 1000, 300, 320), (2, 4, 1, 64, 777, 64, 64),
                                                        (1, 16, 8, 256, 1500, 1024, 1088)])
def test_decode_attention_ring_cache(fk, B, Hq, Hkv, hd, ctx, window, cap):
    """Decode attention over a sliding-window ring (ctx beyond cap): the same
    result as the oracle's attention over the last `window` keys."""
    import torch
    q, k, v = _case(B, Hq, Hkv, hd, ctx, seed=B * 31 + hd)
    kr, vr = _ring(k, cap, 2), _ring(v, cap, 3)
    out = fk.attention_decode(to_dev_bf16(q), to_dev_bf16(kr), to_dev_bf16(vr), ctx, window)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().reshape(B, Hq, hd)
    qf, kf, vf = (oracle.bf16_to_f64(a) for a in (q, k, v))
    for b in range(B):
        ref = oracle.attention(qf[b].reshape(1, Hq, hd), kf[b].transpose(1, 0, 2), vf[b].transpose(2, 0, 1),
                               np.array([ctx - 1]), np.arange(ctx), window, 1.0 / math.sqrt(hd))[0]
        np.testing.assert_allclose(got[b], ref, atol=1e-3, rtol=4e-3)


@pytest.mark.parametrize("S,pos0,hd,window,cap", [(64, 960, 128, 256, 320), (100, 700, 64, 60, 192)])
def test_prefill_attention_ring_cache(fk, S, pos0, hd, window, cap):
    """Prefill chunk at positions beyond the ring's capacity: the window plus
    the chunk fit (window + S - 1 <= cap)."""
    import torch
    B, Hq, Hkv = 1, 4, 2
    kv_len = pos0 + S
    q = synth.normal_bf16(5, 11, (B * S, Hq * hd), 1.0)
    k = synth.normal_bf16(5, 12, (B, Hkv, kv_len, hd), 1.0)
    v = synth.normal_bf16(5, 13, (B, Hkv, hd, kv_len), 1.0)
    kr, vr = _ring(k, cap, 2), _ring(v, cap, 3)
    out = fk.attention_prefill(to_dev_bf16(q), to_dev_bf16(kr), to_dev_bf16(vr), S, pos0, window)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().reshape(B, S, Hq, hd)
    qf, kk, vv = (oracle.bf16_to_f64(a) for a in (q, k, v))
    ref = oracle.attention(qf.reshape(B, S, Hq, hd)[0], kk[0].transpose(1, 0, 2), vv[0].transpose(2, 0, 1),
                           pos0 + np.arange(S), np.arange(kv_len), window, 1.0 / math.sqrt(hd))
    np.testing.assert_allclose(got[0], ref, atol=1e-2, rtol=1e-2)
