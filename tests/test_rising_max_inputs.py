"""The inputs of the GPU rescale tests take the branch they are meant to take.

For every case of ``rising_max`` the oracle's score matrix (float64, on the
same rounded inputs the GPU reads) is replayed through the lazy rescale rule
of the tensor-core forward: "fires" cases must make some row move its
reference maximum after its first key tile (the in-place rescale of the
accumulator), "mixed" rows must put rows that do and rows that do not into
one warp, and "below" cases must keep every row on its first reference while
forming weights above 2^7 against it.  No GPU is needed."""

import numpy as np
import pytest
import torch

import oracle
import rising_max as rm
from parity import default_scale

DTYPES = [torch.bfloat16, torch.float16]


def _check(scores_by_head, rows, expect):
    fired_all, peak_all = [], []
    for s in scores_by_head:
        fired, peak = rm.lazy_rescale_events(s)
        fired_all.append(fired)
        peak_all.append(peak)
        if expect == "fires" and rows == "mixed":
            # some 32-row warp holds a row that rescales and one that does not
            n = len(fired) // 32 * 32
            w = (fired[:n] > 0).reshape(-1, 32)
            assert (w.any(1) & ~w.all(1)).any()
    fired, peak = np.concatenate(fired_all), np.concatenate(peak_all)
    if expect == "fires":
        assert fired.sum() > 0
    else:
        assert fired.sum() == 0
        assert peak.max() > 2.0 ** 7
    assert peak.max() <= 2.0 ** rm.THRESHOLD_LOG2


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "f16"])
@pytest.mark.parametrize("case", rm.DENSE_CASES, ids=rm.case_id)
def test_dense_case_premise(case, dtype):
    profile, step, rows, sigma_k, shape, causal, expect = case
    if shape[2] > 1000 and dtype == torch.float16:
        pytest.skip("one dtype is enough for the long case's premise")
    scale = default_scale(shape[-1])
    q, k, _, _ = rm.dense(shape, dtype, scale, profile, step, rows, sigma_k)
    qn, kn = q.double().numpy(), k.double().numpy()
    heads = [oracle.score_matrix(qn[b, h], kn[b, h], scale, causal)
             for b in range(shape[0]) for h in range(shape[1])]
    _check(heads, rows, expect)


@pytest.mark.parametrize("case", rm.PACKED_CASES, ids=rm.case_id)
def test_packed_case_premise(case):
    profile, step, rows, sigma_k, H, D, causal, expect = case
    scale = default_scale(D)
    q, k, _, _, cu = rm.packed(rm.PACKED_LENGTHS, H, D, torch.bfloat16, scale, profile, step, rows, sigma_k)
    qn, kn = q.double().numpy(), k.double().numpy()
    seqs = []
    for s in range(len(rm.PACKED_LENGTHS)):
        a, b = int(cu[s]), int(cu[s + 1])
        if b - a >= 2 * rm.TILE:  # sequences with a later tile
            seqs += [oracle.score_matrix(qn[h, a:b], kn[h, a:b], scale, causal) for h in range(H)]
    # rows of one warp belong to one sequence only when it starts on a tile
    # boundary; check the warp mix on the first sequence alone
    _check(seqs[:1], rows, expect)
    _check(seqs, "n/a", expect)


def test_helper_levels_and_gains():
    """The planted channel: levels step by the requested rise, gains follow the pattern."""
    scale = default_scale(128)
    q, k, _, _ = rm.dense((1, 1, 600, 128), torch.float32, scale, "ramp", 12.0, "mixed", 1.0)
    step = np.diff(k[0, 0, ::128, 0].double().numpy()) * scale * rm.GAIN / np.log(2.0)
    np.testing.assert_allclose(step, 12.0, rtol=1e-6)
    assert q[0, 0, :6, 0].tolist() == [4.0, 0.0, -4.0, 4.0, 0.0, -4.0]
    _, k2, _, _ = rm.dense((1, 1, 600, 128), torch.float32, scale, "last", 12.0, "odd_tiles", 1.0)
    assert (k2[0, 0, :512, 0] == 0).all() and (k2[0, 0, 512:, 0] > 0).all()
