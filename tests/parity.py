"""Parity rules between the CUDA path and the oracle.

Floating point: pre-sigmoid logits agree within |diff| <= 1e-3 * (|ref| + 1)
for bf16 keys and 4e-2 * (|ref| + 1) for E4M3 keys.  Integer results (mask
bits, top-k id sets) must be bit-exact, except for chunks whose oracle logit
lies within that tolerance of the decision point (0 for the mask, the k-th
score for a top-k), where either decision is correct.
"""
import numpy as np

REL_BF16 = 1e-3
REL_FP8 = 4e-2


def tol(ref, fp8=False):
    return (REL_FP8 if fp8 else REL_BF16) * (np.abs(ref) + 1.0)


def assert_logits_close(got, ref, fp8=False, what="logits"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bad = ~(np.abs(got - ref) <= tol(ref, fp8))
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; "
                           f"worst at {np.unravel_index(np.argmax(np.abs(got - ref) / tol(ref, fp8)), ref.shape)}")
    return float((np.abs(got - ref) / (np.abs(ref) + 1)).max()) if ref.size else 0.0


def mask_bits(mask_words, S):
    """[B, words] uint32 -> [B, S] bool (bit s & 31 of word s >> 5)."""
    m = np.ascontiguousarray(np.asarray(mask_words).view(np.uint32))
    bits = np.unpackbits(m.view(np.uint8), bitorder="little").reshape(m.shape[0], -1)
    return bits[:, :S].astype(bool), bits[:, S:].astype(bool)


def assert_mask_parity(got_words, ref_maxlogit, S, thr_logit=0.0, fp8=False):
    """got_words [B, words]; ref_maxlogit [B, S] = max_l x (oracle, fp64)."""
    bits, tail = mask_bits(got_words, S)
    assert not tail.any(), "mask bits past S are set"
    want = ref_maxlogit >= thr_logit
    diff = bits != want
    exempt = np.abs(ref_maxlogit - thr_logit) <= tol(ref_maxlogit, fp8)
    bad = diff & ~exempt
    assert not bad.any(), f"mask differs at {int(bad.sum())} chunks outside the tolerance band, e.g. {np.argwhere(bad)[:3]}"
    return int((diff & exempt).sum())


def assert_topk_parity(got_idx, ref_idx, score_of, k, fp8=False, got_scores=None):
    """One row.  got_idx/ref_idx [k] int32 (ascending, -1 padded);
    score_of(id) -> oracle fp64 score of a candidate id."""
    got_idx = [int(i) for i in got_idx]
    ref_idx = [int(i) for i in ref_idx]
    n_ref = sum(1 for i in ref_idx if i >= 0)
    n_got = sum(1 for i in got_idx if i >= 0)
    assert n_got == n_ref, f"selected {n_got} ids, oracle {n_ref}"
    sel = got_idx[:n_got]
    assert sel == sorted(sel) and len(set(sel)) == n_got, "ids not strictly ascending"
    assert all(i == -1 for i in got_idx[n_got:]), "padding must be -1"
    g, r = set(sel), set(ref_idx[:n_ref])
    if g == r:
        exempt = 0
    else:
        kth = min(score_of(i) for i in r)
        for i in g ^ r:
            x = score_of(i)
            assert abs(x - kth) <= tol(kth, fp8), f"id {i} (score {x}) differs, k-th score {kth}"
        exempt = len(g ^ r)
    if got_scores is not None:
        gs = np.asarray(got_scores[:n_got], dtype=np.float64)
        ref = np.array([score_of(i) for i in sel])
        assert_logits_close(gs, ref, fp8, "top-k scores")
        assert np.all(np.isneginf(np.asarray(got_scores[n_got:], dtype=np.float64)))
    return exempt


def assert_topk_rows_parity(got_idx, got_scores, ref_idx, cand_ids, cand_x, fp8=False):
    """Whole rows at once.  got_idx / ref_idx [Q, k] int32 (ascending, -1
    padded); got_scores [Q, k] fp32 or None; cand_ids [Q, n] int64 candidate
    ids of each row (-1 = no candidate) and cand_x [Q, n] their oracle fp64
    scores.  Every selected id must be a candidate, the id sets may differ
    only inside the tolerance band around the oracle's k-th score, and every
    returned score must match the oracle's score of its id.  Returns the
    number of ids exempted by the band."""
    got_idx = np.asarray(got_idx)
    ref_idx = np.asarray(ref_idx)
    exempt = 0
    for r in range(got_idx.shape[0]):
        n_ref = int((ref_idx[r] >= 0).sum())
        n_got = int((got_idx[r] >= 0).sum())
        assert n_got == n_ref, f"row {r}: selected {n_got} ids, oracle {n_ref}"
        sel = got_idx[r, :n_got].astype(np.int64)
        assert (got_idx[r, n_got:] == -1).all(), f"row {r}: padding must be -1"
        assert n_got == 0 or (np.diff(sel) > 0).all(), f"row {r}: ids not strictly ascending"
        ids = np.asarray(cand_ids[r], dtype=np.int64)
        xs = np.asarray(cand_x[r], dtype=np.float64)
        keep = ids >= 0
        ids, xs = ids[keep], xs[keep]
        order = np.argsort(ids, kind="stable")
        ids, xs = ids[order], xs[order]
        pos = np.searchsorted(ids, sel)
        assert n_got == 0 or ((pos < len(ids)) & (ids[np.minimum(pos, len(ids) - 1)] == sel)).all(), \
            f"row {r}: a selected id is not a candidate"
        x_sel = xs[pos] if n_got else np.empty(0)
        ref_sel = ref_idx[r, :n_ref].astype(np.int64)
        diff = np.setxor1d(sel, ref_sel)
        if diff.size:
            kth = xs[np.searchsorted(ids, ref_sel)].min()
            x_diff = xs[np.searchsorted(ids, diff)]
            bad = ~(np.abs(x_diff - kth) <= tol(kth, fp8))
            assert not bad.any(), (f"row {r}: ids {diff[bad][:4]} (scores {x_diff[bad][:4]}) differ from the "
                                   f"oracle's set outside the band around its k-th score {kth}")
            exempt += int(diff.size)
        if got_scores is not None:
            gs = np.asarray(got_scores[r], dtype=np.float64)
            assert_logits_close(gs[:n_got], x_sel, fp8, f"row {r} top-k scores")
            assert np.isneginf(gs[n_got:]).all(), f"row {r}: score padding must be -inf"
    return exempt
