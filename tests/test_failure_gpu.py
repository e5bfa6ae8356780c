"""Failure detection on the device, without faulting it.

A bounded pipeline wait that runs out must end the kernel with a status the
host can read, and leave the context (and the library's split-K counters)
usable: the test arms no pipeline stage for the consumers of the op-level
skinny GEMM (a barrier nothing completes), with a 2 ms wait limit, then checks
that fk_sync_status reports FK_DEVERR_PIPE_TIMEOUT and that the next normal
call is correct. Host-visible session errors ("pegainfer issue #878",
Proposed Plan: ids bounds-checked before upload, geometry from the config)
are checked through a small model.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from helpers import err_scale, to_dev_bf16, weights_to_dev

pytestmark = pytest.mark.gpu


def _gemm_case(P, K, N, s):
    xb = synth.normal_bf16(synth.SEED_GEMM_X, 40 + s, (P, K), 1.0)
    wb = synth.normal_bf16(synth.SEED_WEIGHTS, 40 + s, (N, K), 0.02)
    return xb, wb, oracle.gemm(oracle.bf16_to_f64(xb), oracle.bf16_to_f64(wb))


@pytest.mark.parametrize("P,K,N", [(1, 4096, 4096), (16, 1024, 512)])
def test_op_pipeline_timeout_is_reported_and_recovers(fk, P, K, N):
    import torch
    lib = fk.load()
    xb, wb, ref = _gemm_case(P, K, N, P)
    x, w = to_dev_bf16(xb), to_dev_bf16(wb)
    assert fk.op_sync_status()[0] == 0
    assert lib.fk_debug_set_op_pipe_fault(1, 2000) == 0
    try:
        fk.gemm_splitk(x, w, out_fp32=True)
        st, flags = fk.op_sync_status(timeout_ms=20000)
    finally:
        assert lib.fk_debug_set_op_pipe_fault(0, 0) == 0
    assert st == 7 and flags & fk.DEVERR_PIPE_TIMEOUT, (st, flags)
    assert fk.op_sync_status() == (0, 0)  # read and cleared
    # the context, the kernel and its arrival counters are fine afterwards
    for _ in range(2):
        y = fk.gemm_splitk(x, w, out_fp32=True)
        torch.cuda.synchronize()
        assert err_scale(y.cpu().numpy(), ref) < 2e-5
    assert fk.op_sync_status() == (0, 0)


def _small_model(fk, max_positions=64):
    cfg = synth.small_config("llama")
    wb = synth.make_weights(cfg, norm_mode="random")
    return cfg, fk.Model(cfg, weights_to_dev(wb), max_positions=max_positions)


def test_session_context_full(fk):
    cfg, model = _small_model(fk)
    sess = model.session(2, 20)
    ids = synth.make_ids(cfg, 2, 15)
    sess.prefill(ids)
    with pytest.raises(fk.FkError) as ei:
        sess.prefill(synth.make_ids(cfg, 2, 6, stream=1))  # 15 + 6 > 20
    assert ei.value.status == 4
    assert sess.length == 15  # nothing was appended
    for _ in range(5):
        sess.decode()
    with pytest.raises(fk.FkError) as ei:
        sess.decode()
    assert ei.value.status == 4 and sess.length == 20
    with pytest.raises(fk.FkError) as ei:
        model.forward(synth.make_ids(cfg, 1, 65))  # beyond max_positions
    assert ei.value.status == 4


def test_workspace_and_argument_errors(fk):
    import torch
    cfg, model = _small_model(fk)
    lib = fk.load()
    ids = np.ascontiguousarray(synth.make_ids(cfg, 1, 8))
    need = lib.fk_forward_workspace_bytes(model.handle, 1, 8)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = fk.fk_forward(model.handle, ids.ctypes.data, 0, 1, 8, ws.data_ptr(), need - 256, 0, 0, 0, 0, 0)
    assert st == 9  # FK_ERR_WORKSPACE
    sb = lib.fk_session_bytes(model.handle, 1, 32, 32)
    mem = torch.empty(sb, dtype=torch.uint8, device="cuda")
    h = ctypes.c_void_p()
    assert lib.fk_session_create(model.handle, 1, 32, 32, mem.data_ptr(), sb - 1, ctypes.byref(h)) == 9
    assert lib.fk_session_create(model.handle, 1, 32, 32, mem.data_ptr() + 16, sb, ctypes.byref(h)) == 1
    sess = model.session(1, 32)
    with pytest.raises(fk.FkError) as ei:
        sess.decode()  # nothing to feed back yet
    assert ei.value.status == 1
    bad = ids.copy()
    bad[0, 2] = -1
    with pytest.raises(fk.FkError) as ei:
        sess.prefill(bad)
    assert ei.value.status == 3 and sess.length == 0
    st, flags = model.sync_status()
    assert st == 0 and flags == 0
