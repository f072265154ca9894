"""Pins of the CPU oracle to facts outside the oracle itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with a value fixed by the pages, by a published format
definition, by mathematics (closed forms, identities, invariants) or by brute
force on tiny inputs.  ``test_oracle_pins.py`` runs them against the oracle;
``test_oracle_mutants.py`` plants single mistakes into a copy of the oracle's
source and checks that at least one pin catches each of them.
"""
from __future__ import annotations

import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# helpers (input construction only)
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(a) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bit patterns (inputs for pins)."""
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f64(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rank_key_sorted(ids, x):
    """Brute force: all candidates ordered by (x desc, id asc); NaN as -inf."""
    xs = [(-math.inf if math.isnan(v) else v) for v in x]
    return sorted(zip(ids, xs), key=lambda t: (-t[1], t[0]))


def expected_topk(ids, x, k):
    order = rank_key_sorted(list(ids), list(x))
    chosen = sorted(i for i, _ in order[:k])
    return chosen + [-1] * (k - len(chosen))


# ---------------------------------------------------------------------------
# element decoding
# ---------------------------------------------------------------------------

def pin_bf16_decode(orc):
    """bf16 is the top half of binary32: all 65536 codes vs numpy's view."""
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.bf16(codes)
    want = bf16_bits_to_f64(codes)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), f"bf16 decode differs at {np.nonzero(~same)[0][:5]}"


def pin_e4m3_golden(orc):
    """OCP OFP8 E4M3 table values (tests/golden/e4m3_ocp.txt)."""
    with open(os.path.join(GOLDEN, "e4m3_ocp.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for code, val in rows:
        got = orc.e4m3([int(code, 16)])[0]
        want = float(val)
        if math.isnan(want):
            assert math.isnan(got), f"{code}: {got} should be NaN"
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), f"{code}: {got} != {want}"


def pin_e4m3_all_codes_vs_torch(orc):
    """All 256 E4M3 codes vs PyTorch's float8_e4m3fn (an independent decoder)."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.e4m3(codes)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), f"e4m3 decode differs at codes {np.nonzero(~same)[0][:5]}"


def pin_fp8_dequant_is_fp32_product(orc):
    """compressed_k dequant = fp8.float() * scale in fp32: with n_h = d = 1,
    q = 1, w = 1 the score is exactly the fp32 product (when positive)."""
    q = f32_to_bf16_bits(np.array([[1.0]], dtype=np.float32))
    w = np.array([1.0], dtype=np.float32)
    for code, scale in [(0x3F, 0.1), (0x01, 3.0), (0x7E, 1e-3), (0x26, 7.25)]:
        val = {0x3F: 1.875, 0x01: 2.0 ** -9, 0x7E: 448.0, 0x26: 0.21875}[code]
        want = float(np.float32(val) * np.float32(scale))
        got = orc.score_fp8(q, w, np.array([code], dtype=np.uint8), scale)
        assert got == want, f"code {code:#x} scale {scale}: {got} != {want}"


# ---------------------------------------------------------------------------
# score: closed forms and identities
# ---------------------------------------------------------------------------

def pin_score_scalar(orc):
    """n_h = d = 1: x = w * max(0, q*k)."""
    bf = lambda v: f32_to_bf16_bits(np.array(v, dtype=np.float32))
    cases = [(2.0, 3.0, 0.5, 3.0), (2.0, -3.0, 0.5, 0.0), (-2.0, -3.0, 0.5, 3.0),
             (2.0, 3.0, -0.5, -3.0), (0.0, 5.0, 1.0, 0.0), (1.5, 0.25, 4.0, 1.5)]
    for qv, kv, wv, want in cases:
        got = orc.score_bf16(bf([[qv]]), np.array([wv], np.float32), bf([kv]))
        assert got == want, f"q={qv} k={kv} w={wv}: {got} != {want}"


def pin_score_unit_vectors(orc):
    """q_h = c_h e_{pi(h)}, k = e_j: x = w_h max(0, c_h) for the head with
    pi(h) = j, else 0.  Catches head/dim transposes and w misalignment."""
    n_h, d = 4, 8
    pi = [5, 2, 7, 0]
    c = [1.0, 2.0, -1.0, 4.0]
    w = np.array([0.5, 0.25, 2.0, -1.0], dtype=np.float32)
    qf = np.zeros((n_h, d), np.float32)
    for h in range(n_h):
        qf[h, pi[h]] = c[h]
    q = f32_to_bf16_bits(qf)
    for j in range(d):
        k = f32_to_bf16_bits(np.eye(d, dtype=np.float32)[j])
        want = 0.0
        for h in range(n_h):
            if pi[h] == j:
                want = float(w[h]) * max(0.0, c[h])
        got = orc.score_bf16(q, w, k)
        assert got == want, f"e_{j}: {got} != {want}"


def pin_score_antisymmetry(orc):
    """ReLU(v) - ReLU(-v) = v, so x(q) - x(-q) = sum_h w_h (q_h . k) = k . (Q^T w),
    evaluated here by a matrix product in a different association."""
    rng = np.random.default_rng(7)
    for n_h, d in [(64, 128), (3, 5), (1, 128)]:
        for _ in range(3):
            q = f32_to_bf16_bits(rng.standard_normal((n_h, d)).astype(np.float32))
            k = f32_to_bf16_bits((rng.standard_normal(d) / 11).astype(np.float32))
            w = rng.standard_normal(n_h).astype(np.float32)
            qneg = q ^ np.uint16(0x8000)
            lhs = orc.score_bf16(q, w, k) - orc.score_bf16(qneg, w, k)
            rhs = float(bf16_bits_to_f64(k) @ (bf16_bits_to_f64(q).T @ w.astype(np.float64)))
            assert abs(lhs - rhs) <= 1e-10 * (1 + abs(rhs)), f"{lhs} vs {rhs}"


def pin_score_homogeneity(orc):
    """Positive homogeneity: x(2q) = 2 x(q) and x(q; 2w) = 2 x(q; w) exactly."""
    rng = np.random.default_rng(11)
    q = f32_to_bf16_bits(rng.standard_normal((64, 128)).astype(np.float32))
    k = f32_to_bf16_bits((rng.standard_normal(128) / 11).astype(np.float32))
    w = rng.standard_normal(64).astype(np.float32)
    x = orc.score_bf16(q, w, k)
    q2 = f32_to_bf16_bits(bf16_bits_to_f64(q).astype(np.float32) * 2)
    assert orc.score_bf16(q2, w, k) == 2 * x
    assert orc.score_bf16(q, (w * 2).astype(np.float32), k) == 2 * x


def pin_score_relu_negative(orc):
    """All head dots negative -> x = 0 for any w; sigma(0) = 0.5 is resident."""
    q = f32_to_bf16_bits(np.abs(np.random.default_rng(3).standard_normal((64, 128))).astype(np.float32) + 0.01)
    k = f32_to_bf16_bits(-np.full(128, 0.05, np.float32))
    w = np.random.default_rng(4).standard_normal(64).astype(np.float32)
    x = orc.score_bf16(q, w, k)
    assert x == 0.0, x
    mask, maxsig = orc.memindex_select(np.array([[[x]]]), 0.5)
    assert mask[0, 0] == 1 and maxsig[0, 0] == 0.5


def pin_fp8_scale_invariance(orc):
    """Doubling the chunk scale and halving w leaves every score unchanged."""
    rng = np.random.default_rng(5)
    q = f32_to_bf16_bits(rng.standard_normal((64, 128)).astype(np.float32))
    w = rng.standard_normal(64).astype(np.float32)
    k8 = rng.integers(0, 256, 128).astype(np.uint8)
    k8[(k8 & 0x7F) == 0x7F] = 0x11
    a = orc.score_fp8(q, w, k8, 0.0123)
    b = orc.score_fp8(q, (w / 2).astype(np.float32), k8, np.float32(0.0123) * 2)
    assert a == b, (a, b)


# ---------------------------------------------------------------------------
# sigmoid, threshold, union
# ---------------------------------------------------------------------------

def pin_sigmoid_closed_forms(orc):
    assert orc.sigmoid(0.0) == 0.5
    assert abs(orc.sigmoid(math.log(3.0)) - 0.75) < 1e-15
    assert abs(orc.sigmoid(-math.log(3.0)) - 0.25) < 1e-15
    assert abs(orc.sigmoid(-40.0) - math.exp(-40.0) / (1 + math.exp(-40.0))) < 1e-30


def pin_threshold_boundary(orc):
    """sigma(x) >= 0.5 <=> x >= 0 (inclusive); other thresholds via logit."""
    x = np.array([[[-1.0, 0.0, 1.0, -1e-12, 3.0, -5.0, 1e-12]]])
    mask, _ = orc.memindex_select(x, 0.5)
    assert mask[0, 0] == 0b1010110, bin(mask[0, 0])
    lg = math.log(3.0)
    x = np.array([[[lg + 1e-9, lg - 1e-9, 0.0]]])
    mask, _ = orc.memindex_select(x, 0.75)
    assert mask[0, 0] == 0b001, bin(mask[0, 0])


def pin_union_invariants(orc):
    """Mask = OR of per-layer masks = 1(max_l x >= 0); permuting layers changes
    nothing; maxsig = max_l sigma(x_l); bits past S are zero."""
    rng = np.random.default_rng(9)
    B, L, S = 2, 3, 101
    x = rng.standard_normal((B, L, S)) * 2
    x[0, 1, 7] = 0.0
    mask, maxsig = orc.memindex_select(x, 0.5)
    per = [orc.memindex_select(x[:, l:l + 1, :], 0.5)[0] for l in range(L)]
    assert (mask == (per[0] | per[1] | per[2])).all()
    perm, _ = orc.memindex_select(x[:, ::-1, :].copy(), 0.5)
    assert (perm == mask).all()
    words = (S + 31) // 32
    want = np.zeros((B, words), np.uint32)
    for b in range(B):
        for s in range(S):
            if x[b, :, s].max() >= 0:
                want[b, s >> 5] |= np.uint32(1 << (s & 31))
    assert (mask == want).all()
    sig = 1 / (1 + np.exp(-x))
    assert np.allclose(maxsig, sig.max(axis=1), rtol=0, atol=1e-15)


def pin_memindex_logits_layout(orc):
    """orc_memindex_logits places layer l / request b at x[b, l] (checked with
    per-element single-chunk scores on distinct layers)."""
    rng = np.random.default_rng(13)
    B, L, S, n_h, d = 2, 3, 5, 4, 8
    q = f32_to_bf16_bits(rng.standard_normal((B, L, n_h, d)).astype(np.float32))
    w = rng.standard_normal((B, L, n_h)).astype(np.float32)
    K = f32_to_bf16_bits(rng.standard_normal((B, L, S, d)).astype(np.float32))
    x = orc.memindex_logits(q, w, K)
    for b in range(B):
        for l in range(L):
            for s in range(S):
                qd = bf16_bits_to_f64(q[b, l])
                kd = bf16_bits_to_f64(K[b, l, s])
                want = float(np.sum(w[b, l].astype(np.float64) * np.maximum(qd @ kd, 0)))
                assert abs(x[b, l, s] - want) <= 1e-12 * (1 + abs(want))


# ---------------------------------------------------------------------------
# top-k
# ---------------------------------------------------------------------------

def pin_topk_bruteforce(orc):
    """Top-k with heavy ties vs a brute-force ordering by (x desc, id asc);
    output sorted by id, padded with -1; every chosen beats every other."""
    rng = np.random.default_rng(17)
    for n, k in [(0, 8), (1, 8), (5, 8), (8, 8), (17, 8), (40, 8), (300, 64)]:
        ids = rng.permutation(1000)[:n].astype(np.int64)
        x = rng.integers(-3, 4, n).astype(np.float64)
        if n > 3:
            x[2] = np.nan
            x[3] = -np.inf
        idx, sc, m = orc.topk(ids, x, k)
        assert m == min(n, k)
        assert list(idx) == expected_topk(ids, x, k), (n, k)
        chosen = set(int(i) for i in idx if i >= 0)
        xs = {int(i): (-math.inf if math.isnan(v) else v) for i, v in zip(ids, x)}
        for a in chosen:
            for b in set(xs) - chosen:
                assert (xs[a], -a) > (xs[b], -b)


def pin_topk_512_random(orc):
    rng = np.random.default_rng(19)
    n, k = 4096, 512
    ids = np.arange(n, dtype=np.int64)
    x = np.round(rng.standard_normal(n), 2)
    idx, _, m = orc.topk(ids, x, k)
    assert m == k
    assert list(idx) == expected_topk(ids, x, k)


# ---------------------------------------------------------------------------
# paged (Level-2) top-k
# ---------------------------------------------------------------------------

def _paged_case(rng, Q=3, R=5, n_pages=9, page=4, n_h=3, d=8):
    P = Q * R + 2
    q = f32_to_bf16_bits(rng.standard_normal((Q, n_h, d)).astype(np.float32))
    w = rng.standard_normal((Q, n_h)).astype(np.float32)
    k8 = rng.integers(0, 256, (P, page, d)).astype(np.uint8)
    k8[(k8 & 0x7F) == 0x7F] = 0x33
    scale = (rng.random((P, page)) + 0.1).astype(np.float32)
    phys = rng.permutation(P)[: Q * R].reshape(Q, R).astype(np.int32)
    logical = np.stack([rng.permutation(n_pages)[:R] for _ in range(Q)]).astype(np.int32)
    return q, w, k8, scale, phys, logical, n_pages, page


def pin_paged_mode_a(orc):
    """Mode A (non-resident logits at -inf over the full logical chunk range):
    paged top-k = brute-force top-k over all n_pages*page logical chunks of a
    dense, scattered copy of the resident keys."""
    rng = np.random.default_rng(23)
    for k in (6, 40):
        q, w, k8, scale, phys, logical, n_pages, page = _paged_case(rng)
        idx, _ = orc.paged_topk(q, w, k8, scale, phys, logical, k=k)
        Q, R = phys.shape
        for qi in range(Q):
            dense = np.full(n_pages * page, -math.inf)
            for j in range(R):
                for o in range(page):
                    dense[logical[qi, j] * page + o] = orc.score_fp8(q[qi], w[qi], k8[phys[qi, j], o],
                                                                     scale[phys[qi, j], o])
            resident = [lp * page + o for lp in sorted(set(logical[qi].tolist())) for o in range(page)]
            want = expected_topk(resident, [dense[i] for i in resident], k)
            assert list(idx[qi]) == want, qi


def pin_paged_bf16_pool_mode_a(orc):
    """A pool of bf16 keys: the paged top-k equals the brute-force top-k over
    a dense copy of the listed pages' keys scored by the Memory Indexer's
    logits (orc_memindex_logits, pinned on its own), with the chunks of
    unlisted pages excluded; n_res, a resident mask and the remap follow the
    E4M3 pool's rules."""
    rng = np.random.default_rng(31)
    Q, R, n_pages, page, n_h, d = 3, 5, 9, 4, 3, 8
    P = Q * R + 2
    q = f32_to_bf16_bits(rng.standard_normal((Q, n_h, d)).astype(np.float32))
    w = rng.standard_normal((Q, n_h)).astype(np.float32)
    kbf = f32_to_bf16_bits(rng.standard_normal((P, page, d)).astype(np.float32))
    phys = rng.permutation(P)[: Q * R].reshape(Q, R).astype(np.int32)
    logical = np.stack([rng.permutation(n_pages)[:R] for _ in range(Q)]).astype(np.int32)
    n_res = np.array([5, 2, 0], dtype=np.int32)
    for k in (6, 40):
        idx, sc, lg = orc.paged_topk_bf16(q, w, kbf, phys, logical, n_res=n_res, k=k, want_logits=True)
        for qi in range(Q):
            dense = np.zeros((1, 1, n_pages * page, d), np.uint16)
            for j in range(n_res[qi]):
                dense[0, 0, logical[qi, j] * page:(logical[qi, j] + 1) * page] = kbf[phys[qi, j]]
            x = orc.memindex_logits(q[qi][None, None], w[qi][None, None], dense)[0, 0]
            listed = [int(lp) * page + o for lp in sorted(logical[qi, :n_res[qi]].tolist()) for o in range(page)]
            want = expected_topk(listed, [x[i] for i in listed], k)
            assert list(idx[qi]) == want, qi
            got = [float(v) for v, i in zip(sc[qi], idx[qi]) if i >= 0]
            assert got == [float(x[i]) for i in idx[qi] if i >= 0]
            for j in range(n_res[qi]):  # logits in table order
                assert np.array_equal(lg[qi, j * page:(j + 1) * page],
                                      x[logical[qi, j] * page:(logical[qi, j] + 1) * page])
    # a resident mask and the remap: the same selection rules as the E4M3 pool
    mask = np.packbits(rng.random((Q, 64)) < 0.5, axis=-1, bitorder="little").view("<u4").reshape(Q, 2)
    for id_mode in (0, 1):
        idx, _ = orc.paged_topk_bf16(q, w, kbf, phys, logical, k=40, res_mask=mask, id_mode=id_mode)
        for qi in range(Q):
            dense = np.zeros((1, 1, n_pages * page, d), np.uint16)
            for j in range(R):
                dense[0, 0, logical[qi, j] * page:(logical[qi, j] + 1) * page] = kbf[phys[qi, j]]
            x = orc.memindex_logits(q[qi][None, None], w[qi][None, None], dense)[0, 0]
            bits = np.unpackbits(mask[qi].view(np.uint8), bitorder="little")
            cand = [int(lp) * page + o for lp in sorted(logical[qi].tolist()) for o in range(page)
                    if bits[int(lp) * page + o]]
            want = expected_topk(cand, [x[i] for i in cand], 40)
            if id_mode == 1:
                cell = {int(logical[qi, j]) * page + o: int(phys[qi, j]) * page + o for j in range(R)
                        for o in range(page)}
                want = [cell[i] if i >= 0 else -1 for i in want]  # in the order of the logical ids
            assert list(idx[qi]) == want, (qi, id_mode)


def pin_paged_resident_mask_and_remap(orc):
    """Level 2 inside the resident set ([RM] Level 2; [FM] sec. 6 Mode A):
    with a chunk-level resident mask (shared by groups of queries, ragged mask
    rows) only resident chunks are candidates; fewer than k -> all of them,
    padded.  The fused remap emits reserve cells phys*page + o, ranked and
    ordered by those ids.  Brute force over per-chunk scores."""
    rng = np.random.default_rng(29)
    q, w, k8, scale, phys, logical, n_pages, page = _paged_case(rng, Q=4)
    Q, R = phys.shape
    n_chunks = n_pages * page
    for mask_ld in ((n_chunks + 31) // 32, 1):  # a short row: words past it read as 0
        bits = rng.random((2, mask_ld * 32)) < 0.45
        mask = np.packbits(bits, axis=-1, bitorder="little").view("<u4").reshape(2, mask_ld)
        for k in (3, 40):
            for id_mode in (0, 1):
                idx, sc = orc.paged_topk(q, w, k8, scale, phys, logical, k=k, res_mask=mask, mask_group=2,
                                         id_mode=id_mode)
                for qi in range(Q):
                    ids, xs, cell = [], [], {}
                    for j in range(R):
                        for o in range(page):
                            c = int(logical[qi, j]) * page + o
                            cell[c] = int(phys[qi, j]) * page + o
                            if c < mask_ld * 32 and bits[qi // 2, c]:
                                ids.append(c)
                                xs.append(orc.score_fp8(q[qi], w[qi], k8[phys[qi, j], o], scale[phys[qi, j], o]))
                    want = expected_topk(ids, xs, k)
                    if id_mode:
                        want = [cell[c] if c >= 0 else -1 for c in want]
                    assert list(idx[qi]) == want, (mask_ld, k, id_mode, qi)
    ones = np.full((Q, (n_chunks + 31) // 32), 0xFFFFFFFF, np.uint32)
    a, _ = orc.paged_topk(q, w, k8, scale, phys, logical, k=10, res_mask=ones)
    b, _ = orc.paged_topk(q, w, k8, scale, phys, logical, k=10)
    assert (a == b).all(), "an all-resident mask must equal no mask"
    zero = np.zeros((Q, 2), np.uint32)
    a, sc = orc.paged_topk(q, w, k8, scale, phys, logical, k=10, res_mask=zero)
    assert (a == -1).all() and np.isneginf(sc).all(), "an empty resident set selects nothing"


def pin_paged_row_order_and_nres(orc):
    """Page-table row order does not matter; n_res limits the pages used."""
    rng = np.random.default_rng(29)
    q, w, k8, scale, phys, logical, n_pages, page = _paged_case(rng, Q=2, R=6)
    idx, sc = orc.paged_topk(q, w, k8, scale, phys, logical, k=10)
    perm = rng.permutation(phys.shape[1])
    idx2, sc2 = orc.paged_topk(q, w, k8, scale, phys[:, perm].copy(), logical[:, perm].copy(), k=10)
    assert (idx == idx2).all() and np.array_equal(sc, sc2)
    n_res = np.array([2, 0], np.int32)
    idx3, _ = orc.paged_topk(q, w, k8, scale, phys, logical, n_res=n_res, k=10)
    allowed = {int(logical[0, j]) * page + o for j in range(2) for o in range(page)}
    got = [int(i) for i in idx3[0] if i >= 0]
    assert len(got) == 2 * page and set(got) <= allowed
    assert (idx3[1] == -1).all()


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------

def pin_prefill_causal(orc):
    """Candidates of a query at position pos are chunks s < min(S, pos // 4)
    (chunk s covers tokens 4s..4s+3): brute force over tiny inputs."""
    rng = np.random.default_rng(31)
    T, S, n_h, d, k = 9, 23, 2, 8, 5
    q = f32_to_bf16_bits(rng.standard_normal((T, n_h, d)).astype(np.float32))
    w = rng.standard_normal((T, n_h)).astype(np.float32)
    K = f32_to_bf16_bits(rng.standard_normal((S, d)).astype(np.float32))
    pos = np.array([0, 3, 4, 7, 8, 22, 40, 91, 1000], np.int64)
    idx, _ = orc.prefill_topk(q, w, pos, K, ratio=4, k=k)
    for t in range(T):
        lim = min(S, int(pos[t]) // 4)
        assert orc.causal_limit(int(pos[t]), S, 4) == lim
        xs = [orc.score_bf16(q[t], w[t], K[s]) for s in range(lim)]
        assert list(idx[t]) == expected_topk(list(range(lim)), xs, k), t
    assert (idx[0] == -1).all() and (idx[1] == -1).all()
    assert list(idx[2]) == [0, -1, -1, -1, -1]


def pin_prefill_logits(orc):
    """The prefill scores are the definition element by element: each finite
    entry equals the single-score routine (n_h heads, one key), every entry at
    or past the causal limit is -inf, and the scores' own top-k (by score desc,
    id asc) is the prefill top-k."""
    rng = np.random.default_rng(37)
    T, S, n_h, d, k = 7, 19, 3, 8, 4
    q = f32_to_bf16_bits(rng.standard_normal((T, n_h, d)).astype(np.float32))
    w = rng.standard_normal((T, n_h)).astype(np.float32)
    K = f32_to_bf16_bits(rng.standard_normal((S, d)).astype(np.float32))
    pos = np.array([0, 5, 12, 33, 75, 76, 400], np.int64)
    y = orc.prefill_logits(q, w, pos, K, ratio=4)
    idx, _ = orc.prefill_topk(q, w, pos, K, ratio=4, k=k)
    for t in range(T):
        lim = min(S, int(pos[t]) // 4)
        assert np.all(np.isneginf(y[t, lim:]))
        for s in range(lim):
            assert y[t, s] == orc.score_bf16(q[t], w[t], K[s])
        assert list(idx[t]) == expected_topk(list(range(lim)), list(y[t, :lim]), k), t


# ---------------------------------------------------------------------------
# planted construction (the generator's promise, checked through the oracle)
# ---------------------------------------------------------------------------

def pin_planted_tiny(orc):
    """Tiny workload (1 query, S=4096, 12% planted): planted chunks score far
    above the cold ones (~+50 vs N(-1.3, 1.9^2)), so every planted chunk is
    resident and, being fewer than 512, all are in the top-512."""
    import gen
    cfg = gen.TINY
    q, w, hot = gen.memindex_qw(cfg)
    K = gen.memindex_keys_host(cfg, hot)
    x = orc.memindex_logits(q, w, K)
    mask, _ = orc.memindex_select(x, 0.5)
    pl = gen.planted(cfg, 0, 0)
    n_pl = int(pl.sum())
    assert 0.10 * cfg.S < n_pl < 0.14 * cfg.S, n_pl
    bits = np.unpackbits(mask.view(np.uint8), bitorder="little")[: cfg.S].astype(bool)
    assert bits[pl].all()
    assert x[0, 0, pl].min() > 20 and x[0, 0, ~pl].max() < 20
    cold = x[0, 0, ~pl]
    assert -1.6 < cold.mean() < -1.0 and 1.6 < cold.std() < 2.2, (cold.mean(), cold.std())
    idx, _, m = orc.topk(np.arange(cfg.S), x[0, 0], 512)
    assert m == 512 and set(np.nonzero(pl)[0]) <= set(idx.tolist())


def pin_memindex_fp8_equals_bf16_on_exact_keys(orc):
    """Keys that E4M3 and bf16 both represent exactly, at scale 1, give the
    same logits through the compressed-key path as through the bf16 path (an
    identity between two decoders); doubling the scale equals doubling the
    keys (x is positively homogeneous in k); layout: every (b, l, s) lands in
    its own slot."""
    rng = np.random.default_rng(31)
    B, L, S, n_h, d = 2, 3, 7, 5, 16
    q = f32_to_bf16_bits(rng.standard_normal((B, L, n_h, d)).astype(np.float32))
    w = rng.standard_normal((B, L, n_h)).astype(np.float32)
    codes = rng.integers(0, 256, (B, L, S, d)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x40  # no NaN codes
    vals = orc.e4m3(codes.reshape(-1)).reshape(codes.shape)  # exact in bf16 too (3 mantissa bits)
    kb = f32_to_bf16_bits(vals.astype(np.float32))
    ones = np.ones((B, L, S), np.float32)
    x8 = orc.memindex_logits_fp8(q, w, codes, ones)
    xb = orc.memindex_logits(q, w, kb)
    assert np.array_equal(x8, xb), np.abs(x8 - xb).max()
    x2 = orc.memindex_logits_fp8(q, w, codes, 2 * ones)
    assert np.array_equal(x2, 2 * x8)
    # a distinct scale per (b, l, s) multiplies exactly that slot's keys
    sc = (2.0 ** rng.integers(-3, 4, (B, L, S))).astype(np.float32)
    xs = orc.memindex_logits_fp8(q, w, codes, sc)
    for b in range(B):
        for l in range(L):
            for s in range(S):
                kk = f32_to_bf16_bits((vals[b, l, s] * sc[b, l, s]).astype(np.float32))
                assert xs[b, l, s] == orc.score_bf16(q[b, l], w[b, l], kk), (b, l, s)


def pin_unpack_compressed_k(orc):
    """[RM] "compressed_k format": a chunk is 132 bytes, [:128] E4M3 codes and
    [128:132] an fp32 scale.  Rows built field by field with a numpy record
    type (an independent construction) unpack to their fields; IEEE-754
    binary32 fixes 1.0 as bytes 00 00 80 3f and -2.5 as 00 00 20 c0 in
    little-endian order."""
    rng = np.random.default_rng(41)
    n, d = 37, 128
    rec = np.zeros(n, dtype=np.dtype([("k", np.uint8, (d,)), ("s", "<f4")]))
    assert rec.dtype.itemsize == d + 4
    rec["k"] = rng.integers(0, 256, (n, d))
    rec["s"] = rng.standard_normal(n).astype(np.float32)
    rec["s"][0], rec["s"][1] = 1.0, -2.5
    ck = rec.view(np.uint8).reshape(n, d + 4)
    assert list(ck[0, d:]) == [0x00, 0x00, 0x80, 0x3F] and list(ck[1, d:]) == [0x00, 0x00, 0x20, 0xC0]
    k8, sc = orc.unpack_compressed_k(ck)
    assert np.array_equal(k8, rec["k"]) and np.array_equal(sc.view(np.uint32), rec["s"].view(np.uint32))
    # a [B, L, S, 132] block unpacks row by row
    k8b, scb = orc.unpack_compressed_k(ck[:36].reshape(2, 3, 6, d + 4))
    assert k8b.shape == (2, 3, 6, d) and np.array_equal(k8b.reshape(36, d), rec["k"][:36])
    assert np.array_equal(scb.reshape(36), rec["s"][:36])


def pin_ensemble_closed_forms(orc):
    """[RM] "Joint checkpoint + ensemble": max (the union) or mean of the
    per-layer sigmoid scores.  sigma(0) = 1/2 and sigma(ln 3) = 3/4, so layers
    with logits (0, ln 3) ensemble to 3/4 by max and 5/8 by mean (the sigmoid
    of the mean logit would be 0.634); sigma(a) + sigma(-a) = 1 gives a mean
    of 1/2 for (a, -a); an ensembled score equal to the threshold is resident
    (the threshold test is inclusive); one layer makes both modes sigma(x); the max mode is
    the union rule; the mean lies between the smallest and largest layer
    score and does not depend on layer order."""
    x = np.array([[[0.0], [math.log(3.0)]]])  # B=1, L=2, S=1
    _, emax = orc.memindex_ensemble(x, 0)
    _, emean = orc.memindex_ensemble(x, 1)
    assert abs(emax[0, 0] - 0.75) < 1e-15 and abs(emean[0, 0] - 0.625) < 1e-15, (emax, emean)
    for thr, want in ((0.62, 1), (0.63, 0)):
        m, _ = orc.memindex_ensemble(x, 1, thr)
        assert int(m[0, 0]) & 1 == want
    z = np.zeros((1, 2, 3))  # sigma(0) = 1/2 exactly: the inclusive threshold keeps it
    for mode in (0, 1):
        m, e = orc.memindex_ensemble(z, mode, 0.5)
        assert np.all(e == 0.5) and int(m[0, 0]) == 0b111, (mode, e, m)
    a = np.array([[[7.25, -3.0], [-7.25, 3.0]]])
    _, e = orc.memindex_ensemble(a, 1)
    assert np.all(np.abs(e - 0.5) < 1e-15)
    rng = np.random.default_rng(43)
    x1 = rng.normal(0, 3, (2, 1, 50))
    for mode in (0, 1):
        _, e1 = orc.memindex_ensemble(x1, mode)
        assert np.all(np.abs(e1 - 1 / (1 + np.exp(-x1[:, 0]))) < 1e-15)
    xr = rng.normal(0, 3, (3, 4, 77))
    m0, e0 = orc.memindex_ensemble(xr, 0, 0.6)
    ms, es = orc.memindex_select(xr, 0.6)
    assert np.array_equal(m0, ms) and np.array_equal(e0, es)
    m1, e1 = orc.memindex_ensemble(xr, 1, 0.6)
    sig = 1 / (1 + np.exp(-xr))
    assert np.all(e1 <= sig.max(axis=1) + 1e-15) and np.all(e1 >= sig.min(axis=1) - 1e-15)
    m2, e2 = orc.memindex_ensemble(xr[:, ::-1], 1, 0.6)
    assert np.allclose(e2, e1, rtol=0, atol=1e-15)
    bits = np.unpackbits(m1.view(np.uint8), bitorder="little").reshape(3, -1)[:, :77].astype(bool)
    assert np.array_equal(bits, e1 >= 0.6)


# ---------------------------------------------------------------------------
# query projection chain ([RM] "Retriever architecture", "Hyperparameters")
# ---------------------------------------------------------------------------

def pin_rmsnorm_closed_forms(orc):
    """RMSNorm divides by the root mean square: (3, 4) has mean square 12.5,
    so with unit gain and eps = 0 it maps to (3, 4) / sqrt(12.5); a constant
    vector maps to +-1; scaling the input does not change the output (eps = 0);
    the gain multiplies element by element; eps sits inside the root."""
    one = f32_to_bf16_bits(np.ones(2, np.float32))
    y = orc.rmsnorm(np.array([3.0, 4.0]), one, eps=0.0)
    assert np.allclose(y, np.array([3.0, 4.0]) / math.sqrt(12.5), rtol=1e-15)
    g8 = f32_to_bf16_bits(np.ones(8, np.float32))
    assert np.allclose(orc.rmsnorm(np.full(8, -2.5), g8, eps=0.0), -1.0, rtol=1e-15)
    rng = np.random.default_rng(51)
    x = rng.standard_normal(64)
    g = f32_to_bf16_bits(rng.standard_normal(64).astype(np.float32))
    y1 = orc.rmsnorm(x, g, eps=0.0)
    assert np.allclose(orc.rmsnorm(7.5 * x, g, eps=0.0), y1, rtol=1e-13)
    ones = f32_to_bf16_bits(np.ones(64, np.float32))
    assert np.allclose(y1, orc.rmsnorm(x, ones, eps=0.0) * bf16_bits_to_f64(g), rtol=1e-15)
    # eps inside the root: mean square 1 with eps = 3 halves the output
    assert np.allclose(orc.rmsnorm(np.ones(4), f32_to_bf16_bits(np.ones(4, np.float32)), eps=3.0), 0.5, rtol=1e-15)


def pin_yarn_frequencies(orc):
    """YaRN's NTK-by-parts frequencies at the pages' hyperparameters (64
    rotary dims, base 160000, factor 16, original length 65536, beta 32 / 1):
    pair 0 (theta = 1) turns 65536 / 2 pi times in the original context, far
    above beta_fast, and keeps its frequency; the slowest pairs turn less than
    once and are divided by the factor; factor 1 leaves every frequency at
    base^(-2i/64); the scale theta'/theta never leaves [1/16, 1], decreases
    with i, and is linear in the number of turns r inside the blend region."""
    f = [orc.yarn_freq(i) for i in range(32)]
    th = [160000.0 ** (-2.0 * i / 64) for i in range(32)]
    assert f[0] == 1.0
    turns = [65536 * t / (2 * math.pi) for t in th]
    ratio = [a / b for a, b in zip(f, th)]
    for i in range(32):
        assert 1 / 16 - 1e-15 <= ratio[i] <= 1 + 1e-15
        if turns[i] >= 32:
            assert abs(ratio[i] - 1) < 1e-15
        if turns[i] <= 1:
            assert abs(ratio[i] - 1 / 16) < 1e-15
    assert all(ratio[i] >= ratio[i + 1] - 1e-15 for i in range(31))
    blend = [i for i in range(32) if 1 < turns[i] < 32]
    assert len(blend) >= 3
    i0, i1, i2 = blend[0], blend[len(blend) // 2], blend[-1]
    slope01 = (ratio[i1] - ratio[i0]) / (turns[i1] - turns[i0])
    slope12 = (ratio[i2] - ratio[i1]) / (turns[i2] - turns[i1])
    assert abs(slope01 - slope12) < 1e-12 and abs(slope01 - (1 - 1 / 16) / 31) < 1e-12
    assert all(abs(orc.yarn_freq(i, factor=1.0) - th[i]) <= 1e-15 * th[i] for i in range(32))


def pin_rope_rotation(orc):
    """Rotary embedding on the last 64 of 128 entries: position 0 is the
    identity; the first 64 entries never change; each rotary pair keeps its
    length; positions add (rotating by p1 then p2 equals rotating by p1 + p2);
    the unit vector on entry 64 (pair 0, frequency 1) lands on
    (cos p, sin p) in entries 64 and 65."""
    rng = np.random.default_rng(53)
    x = rng.standard_normal(128)
    assert np.array_equal(orc.rope_yarn(x, 0), x)
    y = orc.rope_yarn(x, 12345)
    assert np.array_equal(y[:64], x[:64])
    assert np.allclose(np.hypot(y[64::2], y[65::2]), np.hypot(x[64::2], x[65::2]), rtol=1e-13)
    assert np.allclose(orc.rope_yarn(orc.rope_yarn(x, 700), 1234), orc.rope_yarn(x, 1934), rtol=0, atol=1e-11)
    e = np.zeros(128)
    e[64] = 1.0
    for p in (1, 7, 100000):
        z = orc.rope_yarn(e, p)
        assert abs(z[64] - math.cos(p)) < 1e-12 and abs(z[65] - math.sin(p)) < 1e-12
        assert np.count_nonzero(z) <= 2


def pin_hadamard_transform(orc):
    """The normalised Walsh-Hadamard transform equals scipy's Sylvester
    Hadamard matrix divided by sqrt(n) (a library routine), is its own
    inverse, keeps lengths, and maps e_0 to the constant 1/sqrt(n)."""
    from scipy.linalg import hadamard
    n = 128
    rng = np.random.default_rng(57)
    x = rng.standard_normal(n)
    assert np.allclose(orc.hadamard(x), hadamard(n) @ x / math.sqrt(n), rtol=0, atol=1e-12)
    assert np.allclose(orc.hadamard(orc.hadamard(x)), x, rtol=0, atol=1e-12)
    assert abs(np.linalg.norm(orc.hadamard(x)) - np.linalg.norm(x)) < 1e-12
    e0 = np.zeros(n)
    e0[0] = 1.0
    assert np.allclose(orc.hadamard(e0), 1 / math.sqrt(n), rtol=1e-15)


def pin_query_chain_composition(orc):
    """The chain is the composition of its steps in the pages' order: Linear
    (weights [out, in]) -> RMSNorm -> Linear -> per-head rotary -> per-head
    Hadamard; the head weights are a Linear of the hidden state times
    head_dim^-1/2 n_h^-1/2 (here 1 / sqrt(16 * 3)).  Matrix products from
    numpy, the steps from their pinned oracle functions."""
    rng = np.random.default_rng(59)
    T, dim, r, n_h, hd = 3, 24, 16, 3, 16
    hidden = f32_to_bf16_bits(rng.standard_normal((T, dim)).astype(np.float32))
    wa = f32_to_bf16_bits((rng.standard_normal((r, dim)) / 5).astype(np.float32))
    gn = f32_to_bf16_bits(rng.uniform(0.5, 1.5, r).astype(np.float32))
    wb = f32_to_bf16_bits((rng.standard_normal((n_h * hd, r)) / 4).astype(np.float32))
    wp = f32_to_bf16_bits(rng.standard_normal((n_h, dim)).astype(np.float32))
    pos = np.array([0, 17, 262143], dtype=np.int64)
    rope = dict(rope_dim=8, base=10000.0, factor=4.0, orig_len=64.0, beta_fast=8.0, beta_slow=1.0)
    q, w = orc.query_chain(hidden, wa, gn, wb, wp, pos, n_h=n_h, head_dim=hd, eps=1e-6, **rope)
    h = bf16_bits_to_f64(hidden)
    for t in range(T):
        a = bf16_bits_to_f64(wa) @ h[t]
        c = orc.rmsnorm(a, gn, eps=1e-6)
        u = (bf16_bits_to_f64(wb) @ c).reshape(n_h, hd)
        for hh in range(n_h):
            want = orc.hadamard(orc.rope_yarn(u[hh], int(pos[t]), **rope))
            assert np.allclose(q[t, hh], want, rtol=1e-12, atol=1e-12), (t, hh)
        assert np.allclose(w[t], bf16_bits_to_f64(wp) @ h[t] / math.sqrt(hd * n_h), rtol=1e-12)


# ---------------------------------------------------------------------------
# page recall (densest resident pages)
# ---------------------------------------------------------------------------

def _recall_bruteforce(mask_row, S, kmax, sink, recent, page=64):
    """Resident set as a Python set, densities by counting, order by sorting."""
    resident = {s for s in range(S) if (int(mask_row[s >> 5]) >> (s & 31)) & 1}
    resident |= set(range(min(sink, S)))
    resident |= set(range(max(S - recent, 0), S))
    n_pages = (S + page - 1) // page
    dens = [sum(1 for s in range(p * page, min((p + 1) * page, S)) if s in resident) for p in range(n_pages)]
    order = sorted((p for p in range(n_pages) if dens[p] > 0), key=lambda p: (-dens[p], p))
    chosen = sorted(order[:kmax])
    return (chosen + [-1] * (kmax - len(chosen)), [dens[p] for p in chosen] + [-1] * (kmax - len(chosen)),
            len(chosen))


def pin_page_recall_bruteforce(orc):
    """[RM] Level 1 resident set (threshold + recent + sink) and the KMAX
    densest 64-chunk pages: brute force over small random masks, with partial
    last pages, ties in density and forced sink / recency chunks."""
    rng = np.random.default_rng(17)
    for S in (1, 63, 64, 65, 200, 777, 1024):
        words = (S + 31) // 32
        for density_p in (0.02, 0.3, 0.9):
            bits = rng.random((3, words * 32)) < density_p
            bits[:, S:] = False  # bits past S are zero by contract
            mask = np.packbits(bits.reshape(3, words, 32)[:, :, ::-1], axis=-1, bitorder="big")
            mask = mask.reshape(3, words, 4)[:, :, ::-1].copy().view(np.uint32).reshape(3, words)
            for kmax in (1, 3, 16):
                sink, recent = int(rng.integers(0, 70)), int(rng.integers(0, 90))
                pages, dens, n = orc.page_recall(mask, S, kmax, sink=sink, recent=recent)
                for b in range(3):
                    wp, wd, wn = _recall_bruteforce(mask[b], S, kmax, sink, recent)
                    assert list(pages[b]) == wp and list(dens[b]) == wd and n[b] == wn, (S, kmax, b)


def pin_page_recall_closed_forms(orc):
    """Closed forms: an empty resident set recalls nothing; an all-resident
    history of P full pages plus a partial page of r chunks has densities
    64 ... 64, r; the recency tail alone recalls exactly the last pages."""
    S = 64 * 5 + 17
    words = (S + 31) // 32
    zero = np.zeros((1, words), np.uint32)
    pages, dens, n = orc.page_recall(zero, S, 8)
    assert n[0] == 0 and (pages == -1).all() and (dens == -1).all()
    ones = np.full((1, words), 0xFFFFFFFF, np.uint32)
    ones[0, -1] = (1 << (S % 32)) - 1  # bits past S are zero
    pages, dens, n = orc.page_recall(ones, S, 8)
    assert n[0] == 6 and list(pages[0]) == [0, 1, 2, 3, 4, 5, -1, -1] and list(dens[0][:6]) == [64] * 5 + [17]
    pages, dens, n = orc.page_recall(ones, S, 5)  # the partial page loses
    assert list(pages[0]) == [0, 1, 2, 3, 4]
    pages, dens, n = orc.page_recall(zero, S, 8, sink=S)  # the sink covers everything
    assert n[0] == 6 and list(dens[0][:6]) == [64] * 5 + [17]
    pages, dens, n = orc.page_recall(zero, S, 8, recent=17 + 64)  # the last page and a half
    assert list(pages[0][:2]) == [4, 5] and list(dens[0][:2]) == [64, 17] and n[0] == 2
    pages, dens, n = orc.page_recall(zero, S, 8, sink=1, recent=1)
    assert list(pages[0][:2]) == [0, 5] and list(dens[0][:2]) == [1, 1] and n[0] == 2


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
