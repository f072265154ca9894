"""Prefill top-k rows long enough for the segment-pruned select (at least 2k
segments of 32 chunks below the causal limit), against the oracle: the pruned
path itself, each of its fallbacks (too few segments, more segments than the
select holds, a candidate list that overflows on clustered scores), rows of
negative scores and rows of exact ties."""
import numpy as np
import pytest

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
