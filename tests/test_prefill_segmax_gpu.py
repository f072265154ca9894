"""Prefill top-k rows long enough for the segment-pruned select (at least 2k
segments of 32 chunks below the causal limit), against the oracle: the pruned
path itself, each of its fallbacks (too few segments, more segments than the
select holds, a candidate list that overflows on clustered scores), rows of
negative scores, rows of exact ties and rows with NaN and infinite scores."""
import numpy as np
import pytest

import parity
from test_prefill_gpu import check, run_prefill, small

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return torch, torch.device("cuda:0")


def mixed_positions(T, S, seed):
    """Half the tokens see every chunk; the others stop at a random limit
    (some below 64k chunks, where rows fall back to the whole-row select,
    many inside a segment, so the last segment is partial)."""
    rng = np.random.default_rng(seed)
    pos = 4 * S + 17 + np.arange(T, dtype=np.int64)
    cut = rng.integers(0, 4 * S, size=T // 2)
    pos[1::2][: len(cut)] = cut
    return pos


@pytest.mark.parametrize("T,S,k", [(8, 40000, 512), (24, 20000, 64), (16, 8191, 100), (7, 2048, 1),
                                   (5, 100000, 300), (3, 150000, 512)])
def test_segmax_rows_match_oracle(torch_dev, orc, T, S, k):
    """(3, 150000, 512) has more segments (4688) than the select holds, so
    its full rows take the whole-row select inside the same kernel."""
    torch, dev = torch_dev
    q, w, pos, K = small(T, S, seed=T * 13 + S, pos=mixed_positions(T, S, seed=S))
    idx, sc = run_prefill(torch, dev, q, w, pos, K, k)
    check(orc, q, w, pos, K, idx, sc, k)


def test_segmax_clustered_scores(torch_dev, orc):
    """Chunks ordered by token 0's score (ascending), and token 1 with token
    0's query and negated weights (its scores descend along the row).  Token
    0's largest segment entries all sit at the end of the row, so nearly every
    score of the last k segments passes the bound and the candidate list
    overflows (the whole-row fallback); token 1's cluster at the start."""
    torch, dev = torch_dev
    T, S, k = 4, 30000, 256
    q, w, pos, K = small(T, S, seed=77)
    lg = orc.prefill_logits(q[:1], w[:1], pos[:1], K)[0]
    K = np.ascontiguousarray(K[np.argsort(lg, kind="stable")])
    q[1] = q[0]
    w[1] = -w[0]
    idx, sc = run_prefill(torch, dev, q, w, pos, K, k)
    check(orc, q, w, pos, K, idx, sc, k)


def test_segmax_negative_scores(torch_dev, orc):
    """Non-positive head weights make every score <= 0: every segment entry is
    negative, so the bound on a segment is +0, every segment is listed and
    the candidate list overflows (the whole-row fallback)."""
    torch, dev = torch_dev
    T, S, k = 6, 20000, 64
    q, w, pos, K = small(T, S, seed=91)
    w = -np.abs(w)
    idx, sc = run_prefill(torch, dev, q, w, pos, K, k)
    check(orc, q, w, pos, K, idx, sc, k)
    assert (sc <= 0).all()


def test_segmax_exact_ties(torch_dev, orc):
    """q = 0 gives every chunk the score 0: all 3000 scores are candidates
    (within the list), and the ties go to the lowest chunk ids."""
    torch, dev = torch_dev
    T, S, k = 3, 3000, 40
    q, w, pos, K = small(T, S, seed=5)
    q = np.zeros_like(q)
    idx, sc = run_prefill(torch, dev, q, w, pos, K, k)
    check(orc, q, w, pos, K, idx, sc, k)
    assert (idx == np.arange(k, dtype=np.int32)[None, :]).all()
    assert (sc == 0).all()


def test_segmax_nonfinite_scores(torch_dev, orc):
    """Three chunk keys with +inf in one element.  Their dots are ±inf, so
    with mixed-sign head weights (tokens 0-2) their score is NaN in every row
    (ranked as -inf: never selected while finite scores remain), and with
    non-negative weights (tokens 3-5) +inf (selected first).  The segments
    holding them carry NaN / +inf entries through the pruned select.  Token 6
    has a NaN head weight, so every score of its row is NaN: all of them tie
    at -inf and the lowest chunk ids are selected."""
    torch, dev = torch_dev
    T, S, k = 7, 20000, 64
    q, w, pos, K = small(T, S, seed=123)
    K = K.copy()
    special = [5, 4100, 13377]
    K[special, 0] = 0x7F80  # bf16 +inf
    w = w.copy()
    w[3:6] = np.abs(w[3:6])
    w[6, 0] = np.nan
    idx, sc = run_prefill(torch, dev, q, w, pos, K, k)
    ref_idx, _ = orc.prefill_topk(q, w, pos, K, k=k)
    assert (ref_idx[6] == np.arange(k)).all() and (idx[6] == np.arange(k)).all()
    assert np.all(~(sc[6] > -np.inf))  # NaN scores rank as -inf
    for t in range(6):
        x = {int(i): orc.score_bf16(q[t], w[t], K[int(i)]) for i in set(idx[t]) | set(ref_idx[t]) if i >= 0}
        if t < 3:
            assert all(np.isnan(orc.score_bf16(q[t], w[t], K[s])) for s in special)
            assert not set(special) & set(int(i) for i in idx[t])
        else:
            assert all(np.isposinf(orc.score_bf16(q[t], w[t], K[s])) for s in special)
            assert set(special) <= set(int(i) for i in idx[t])
        got, ref = set(int(i) for i in idx[t]), set(int(i) for i in ref_idx[t])
        assert list(idx[t]) == sorted(got) and len(got) == k
        finite_ref = [x[i] for i in ref if np.isfinite(x[i])]
        kth = min(finite_ref)
        for i in got ^ ref:  # only near-ties at the k-th score may differ
            assert np.isfinite(x[i]) and abs(x[i] - kth) <= parity.tol(kth), (t, i, x[i], kth)
        for j, i in enumerate(idx[t]):
            if np.isfinite(x[int(i)]):
                parity.assert_logits_close([sc[t, j]], [x[int(i)]], what="top-k scores")
            else:
                assert sc[t, j] == x[int(i)]
