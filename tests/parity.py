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
