"""On-device log-softmax and top-k against the oracle's readouts
("pegainfer issue #878", Acceptance Criteria: log-probabilities at each
position's top-64 ids over the 262144-word vocabulary).

The device computes on fp32 logits; the oracle's log_softmax and topk_ids run
in float64 on the same values. Ids are compared exactly (value descending,
ties to the lower id); log-probabilities within 2e-5 (fp32 sums of up to
262144 terms below 1 and one fp32 subtraction).
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


def _rows(R, V, seed, scale):
    return synth.normal_f32(seed, R, (R, V), 1.0) * np.float32(scale)


@pytest.mark.parametrize("R,V,k,scale", [(1, 262144, 64, 2.0), (37, 262144, 64, 5.0), (300, 49152, 64, 1.0),
                                         (5, 1000, 128, 3.0), (3, 64, 64, 1.0), (2, 128256, 1, 8.0)])
def test_logsoftmax_topk_vs_oracle(fk, R, V, k, scale):
    import torch
    z = _rows(R, V, seed=61, scale=scale)
    out = fk.logsoftmax_topk(torch.from_numpy(z).cuda(), k=k, logprobs=True)
    torch.cuda.synchronize()
    zd = z.astype(np.float64)
    want_ids = oracle.topk_ids(zd, k)
    lp = oracle.log_softmax(zd)
    np.testing.assert_array_equal(out["ids"].cpu().numpy(), want_ids)
    np.testing.assert_allclose(out["top_logprobs"].cpu().numpy(), np.take_along_axis(lp, want_ids, -1), atol=2e-5)
    np.testing.assert_allclose(out["logprobs"].cpu().numpy(), lp, atol=2e-5)
    lse = np.max(zd, -1) + np.log(np.sum(np.exp(zd - np.max(zd, -1, keepdims=True)), -1))
    np.testing.assert_allclose(out["lse"].cpu().numpy(), lse, atol=2e-5)


def test_logsoftmax_topk_ties_at_the_boundary(fk):
    """Equal values straddling the k-th place: the lower ids are taken, and
    the order among equal values is by id."""
    import torch
    V, k = 262144, 64
    z = _rows(4, V, seed=62, scale=1.0)
    z[0, [5, 70000, 123, 262143, 9999]] = 50.0        # five equal maxima
    z[1, np.arange(0, V, 4096)] = 20.0                 # 64 equal values exactly fill k
    z[2, np.arange(7, V, 2048)] = 20.0                 # 128 equal values: only the 64 lowest ids
    z[3, :] = 0.25                                     # a constant row
    out = fk.logsoftmax_topk(torch.from_numpy(z).cuda(), k=k)
    torch.cuda.synchronize()
    ids = out["ids"].cpu().numpy()
    np.testing.assert_array_equal(ids, oracle.topk_ids(z.astype(np.float64), k))
    assert list(ids[0, :5]) == [5, 123, 9999, 70000, 262143]
    assert list(ids[2]) == list(range(7, V, 2048))[:64]
    assert list(ids[3]) == list(range(64))
    np.testing.assert_allclose(out["top_logprobs"].cpu().numpy()[3], -np.log(V), atol=2e-5)


def test_logsoftmax_topk_rejects_bad_k(fk):
    import torch
    z = torch.zeros((2, 100), dtype=torch.float32, device="cuda")
    for k in (0, 101, 129):
        with pytest.raises(fk.FkError) as ei:
            fk.logsoftmax_topk(z, k=k)
        assert ei.value.status == 1
