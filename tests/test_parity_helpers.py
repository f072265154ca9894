"""The whole-row top-k comparison of tests/parity.py accepts the oracle's own
selection and rejects planted mistakes (CPU only)."""
import numpy as np
import pytest

import parity


def _rows(orc, Q=3, n=700, k=64, seed=0):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(4 * n)[:n] for _ in range(Q)]).astype(np.int64)
    x = rng.standard_normal((Q, n))
    ref = np.empty((Q, k), np.int32)
    for r in range(Q):
        ref[r], _, _ = orc.topk(ids[r], x[r], k)
    sc = np.full((Q, k), -np.inf, np.float32)
    for r in range(Q):
        lut = dict(zip(ids[r].tolist(), x[r].tolist()))
        sc[r, :] = [lut[int(i)] for i in ref[r]]
    return ids, x, ref, sc


def test_accepts_oracle_selection(orc):
    ids, x, ref, sc = _rows(orc)
    assert parity.assert_topk_rows_parity(ref, sc, ref, ids, x) == 0


@pytest.mark.parametrize("mistake", ["swap_id", "wrong_score", "unsorted", "non_candidate", "short", "pad"])
def test_rejects_planted_mistakes(orc, mistake):
    ids, x, ref, sc = _rows(orc, seed=3)
    got, gs = ref.copy(), sc.copy()
    r = 1
    if mistake == "swap_id":  # the worst candidate instead of the best
        best = int(np.argmax(x[r]))
        worst = int(ids[r, np.argmin(x[r])])
        sel = sorted(set(got[r].tolist()) - {int(ids[r, best])} | {worst})
        got[r] = sel
        lut = dict(zip(ids[r].tolist(), x[r].tolist()))
        gs[r] = [lut[i] for i in sel]
    elif mistake == "wrong_score":
        gs[r, 5] += 0.01
    elif mistake == "unsorted":
        got[r, [2, 3]] = got[r, [3, 2]]
        gs[r, [2, 3]] = gs[r, [3, 2]]
    elif mistake == "non_candidate":
        got[r, -1] = 4 * ids.shape[1] + 7
    elif mistake == "short":
        got[r, -1] = -1
        gs[r, -1] = -np.inf
    elif mistake == "pad":
        got = np.concatenate([got, np.zeros((got.shape[0], 1), np.int32)], axis=1)
        ref2 = np.concatenate([ref, -np.ones((ref.shape[0], 1), np.int32)], axis=1)
        gs = np.concatenate([gs, np.full((gs.shape[0], 1), -np.inf, np.float32)], axis=1)
        with pytest.raises(AssertionError):
            parity.assert_topk_rows_parity(got, gs, ref2, ids, x)
        return
    with pytest.raises(AssertionError):
        parity.assert_topk_rows_parity(got, gs, ref, ids, x)
