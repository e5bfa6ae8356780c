"""Op hooks against the oracle, element by element ("N9 · metalgemm", Thm 1:
op-level parity of each device op, not only of the chain).

* fk_op_rmsnorm vs oracle.rmsnorm ("N7 · model/forward-parity", Thm 1).
* fk_op_rope vs oracle.rope_apply (+ oracle.rmsnorm for QK-norm): llama3
  scaling, QK-norm, local/global bases, cache placement of k and of the
  transposed v ("N7", Thm 1 RoPE; Thm 2 QK-norm and rope scaling axes).
* fk_op_head_argmax vs the oracle head (+ softcap), with the argmax and the
  top-2 margin checked exactly on the device's own fp32 logits, including
  exact ties ("N7", Thm 3: the near-tie flip that motivates the margin).

Tolerances: every output is bf16 or fp32 computed in fp32 from bf16 inputs.
A bf16 store rounds to 2^-9 relative; fp32 sums over <= 4096 terms add far
less than that.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import to_dev_bf16, weights_to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,hidden", [(1, 64), (7, 576), (33, 4096), (130, 3840), (5, 8192), (3, 16384)])
def test_op_rmsnorm(fk, rows, hidden):
    import torch
    x = synth.normal_f32(3, rows, (rows, hidden), 1.0) * np.float32(3.0)
    wb = synth.normal_bf16(3, 100 + rows, (hidden,), 0.1, 1.0)
    eps = 1e-6
    out = fk.rmsnorm(torch.from_numpy(x).cuda(), to_dev_bf16(wb), eps)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    ref = oracle.rmsnorm(x.astype(np.float64), oracle.bf16_to_f64(wb), eps)
    np.testing.assert_allclose(got, ref, rtol=2.0 ** -8, atol=1e-6)


def _rope_case(cfg, B, S, pos0, seed):
    Hq, Hkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    qkv = synth.normal_bf16(seed, 1, (B * S, (Hq + 2 * Hkv) * hd), 1.0)
    return qkv


@pytest.mark.parametrize("kind,layer,B,S,pos0", [("llama3", 0, 2, 70, 0), ("llama3", 1, 1, 33, 100),
                                                 ("gemma", 0, 2, 40, 5), ("gemma", 2, 1, 64, 64),
                                                 ("llama", 1, 3, 9, 17)])
def test_op_rope(fk, kind, layer, B, S, pos0):
    import torch
    cfg = synth.small_config(kind)
    wb = synth.make_weights(cfg, norm_mode="random")
    model = fk.Model(cfg, weights_to_dev(wb), max_positions=256)
    Hq, Hkv, hd = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    qkv_bits = _rope_case(cfg, B, S, pos0, seed=11 + layer)
    cap = (pos0 + S + 63) // 64 * 64
    qkv = to_dev_bf16(qkv_bits)
    kc = torch.zeros((B, Hkv, cap, hd), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros((B, Hkv, hd, cap), dtype=torch.bfloat16, device="cuda")
    model.rope(layer, qkv, B, S, pos0, kc, vc)
    torch.cuda.synchronize()
    x = oracle.bf16_to_f64(qkv_bits).reshape(B, S, Hq + 2 * Hkv, hd)
    q, k, v = x[:, :, :Hq], x[:, :, Hq:Hq + Hkv], x[:, :, Hq + Hkv:]
    if cfg.qk_norm:
        q = oracle.rmsnorm(q, oracle.bf16_to_f64(wb[f"L{layer}.q_norm"]), cfg.rms_eps)
        k = oracle.rmsnorm(k, oracle.bf16_to_f64(wb[f"L{layer}.k_norm"]), cfg.rms_eps)
    pos = np.broadcast_to(pos0 + np.arange(S), (B, S))
    f = oracle.rope_inv_freq(cfg, cfg.kinds()[layer])
    q_ref, k_ref = oracle.rope_apply(q, pos, f), oracle.rope_apply(k, pos, f)
    got = qkv.float().cpu().numpy().reshape(B, S, Hq + 2 * Hkv, hd)
    tol = dict(rtol=2.0 ** -8, atol=2e-3)
    np.testing.assert_allclose(got[:, :, :Hq], q_ref, **tol)
    kg, vg = kc.float().cpu().numpy(), vc.float().cpu().numpy()
    np.testing.assert_allclose(kg[:, :, pos0:pos0 + S].transpose(0, 2, 1, 3), k_ref, **tol)
    np.testing.assert_array_equal(vg[:, :, :, pos0:pos0 + S].transpose(0, 3, 1, 2), v)  # moved, not rounded
    # nothing written outside [pos0, pos0 + S)
    assert not kg[:, :, :pos0].any() and not kg[:, :, pos0 + S:].any()
    assert not vg[:, :, :, :pos0].any() and not vg[:, :, :, pos0 + S:].any()


@pytest.mark.parametrize("kind,rows", [("gemma", 5), ("llama3", 70), ("llama", 1), ("llama", 130)])
def test_op_head_argmax(fk, kind, rows):
    import torch
    cfg = synth.small_config(kind)
    wb = synth.make_weights(cfg, norm_mode="random")
    model = fk.Model(cfg, weights_to_dev(wb), max_positions=64)
    ub = synth.normal_bf16(5, rows, (rows, cfg.hidden), 1.0 if kind != "gemma" else 40.0)
    out = model.head_argmax(to_dev_bf16(ub))
    torch.cuda.synchronize()
    z = out["logits"].cpu().numpy()
    head = wb["embed"] if cfg.tied else wb["lm_head"]
    zr = oracle.gemm(oracle.bf16_to_f64(ub), oracle.bf16_to_f64(head))
    if cfg.final_softcap > 0:
        zr = oracle.softcap(zr, cfg.final_softcap)
    np.testing.assert_allclose(z, zr, rtol=1e-5, atol=1e-5 * np.max(np.abs(zr)))
    if cfg.final_softcap > 0:
        assert np.max(np.abs(z)) < cfg.final_softcap and np.max(np.abs(zr)) > 0.5 * cfg.final_softcap
    # argmax and margin exactly on the device's own logits
    am, mg = out["argmax"].cpu().numpy(), out["margin"].cpu().numpy()
    np.testing.assert_array_equal(am, np.argmax(z, axis=-1))
    part = np.sort(z, axis=-1)
    np.testing.assert_array_equal(mg, (part[:, -1] - part[:, -2]).astype(np.float32))
    decided = oracle.top2_margin(zr) > 1e-3
    np.testing.assert_array_equal(am[decided], oracle.argmax_first(zr)[decided])


def test_op_head_argmax_exact_ties(fk):
    """Duplicate head rows give bit-identical logits: the lowest index wins and
    the margin is exactly 0 (lowest-index rule of the argmax reading)."""
    import torch
    cfg = synth.small_config("llama3")  # untied head
    wb = synth.make_weights(cfg, norm_mode="random")
    head = wb["lm_head"].copy()
    big = synth.normal_bf16(9, 9, (cfg.hidden,), 0.5)
    for j in (900, 17, 513):  # the same large row at three indices
        head[j] = big
    wb["lm_head"] = head
    model = fk.Model(cfg, weights_to_dev(wb), max_positions=64)
    ub = np.stack([big, big, synth.normal_bf16(9, 10, (cfg.hidden,), 1.0)])  # u aligned with the row: it wins
    out = model.head_argmax(to_dev_bf16(ub))
    torch.cuda.synchronize()
    am, mg = out["argmax"].cpu().numpy(), out["margin"].cpu().numpy()
    assert am[0] == 17 and am[1] == 17 and mg[0] == 0.0 and mg[1] == 0.0
    z = out["logits"].cpu().numpy()
    assert z[0, 17] == z[0, 513] == z[0, 900]


def test_forward_and_session_margins(fk):
    """The margins of fk_forward, fk_session_prefill and fk_decode_step equal
    the top-1 minus top-2 value of the logits each call writes."""
    import torch
    cfg = synth.small_config("gemma")
    wb = synth.make_weights(cfg, norm_mode="random")
    model = fk.Model(cfg, weights_to_dev(wb), max_positions=64)
    ids = synth.make_ids(cfg, 2, 20)
    out = model.forward(ids, margin=True)
    torch.cuda.synchronize()
    z = out["logits"].cpu().numpy()
    part = np.sort(z, axis=-1)
    np.testing.assert_array_equal(out["margin"].cpu().numpy(), (part[:, -1] - part[:, -2]).astype(np.float32))
    sess = model.session(2, 40)
    zl = torch.empty((2, cfg.vocab), dtype=torch.float32, device="cuda")
    nx = torch.empty((2,), dtype=torch.int32, device="cuda")
    mg = torch.empty((2,), dtype=torch.float32, device="cuda")
    sess.prefill(ids, logits=zl, next_ids=nx, margin=mg)
    for step in range(4):
        torch.cuda.synchronize()
        zz = zl.cpu().numpy()
        p = np.sort(zz, axis=-1)
        np.testing.assert_array_equal(mg.cpu().numpy(), (p[:, -1] - p[:, -2]).astype(np.float32))
        np.testing.assert_array_equal(nx.cpu().numpy(), np.argmax(zz, axis=-1))
        sess.decode(None, logits=zl, next_ids=nx, margin=mg)  # graph replay from the second step on
