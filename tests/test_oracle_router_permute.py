"""Pins of the oracle's router (S1/S2) and permutation (S4): brute force on tiny
inputs, engineered exact ties, closed forms and invariants."""
import itertools
import math

import numpy as np
import pytest

from oracle import permute as P
from oracle import router as R


def _brute_topk(row, k):
    """Best ordered k-tuple by exhaustive search: the lexicographically largest
    sequence of (logit, -index) keys over all ordered k-subsets."""
    best, best_key = None, None
    for tup in itertools.permutations(range(len(row)), k):
        key = [(row[e], -e) for e in tup]
        if best_key is None or key > best_key:
            best, best_key = tup, key
    return list(best)


def test_topk_brute_force_tiny():
    rng = np.random.default_rng(10)
    for _ in range(60):
        E = int(rng.integers(2, 8))
        k = int(rng.integers(1, min(E, 3) + 1))
        l = np.round(rng.standard_normal((1, E)) * 2) / 2  # coarse: many exact ties
        idx = R.topk_full_sort(l, k)
        assert list(idx[0]) == _brute_topk(list(l[0]), k)


def test_topk_exact_ties_go_to_lower_index():
    rng = np.random.default_rng(11)
    H, E = 64, 16
    Wr = rng.standard_normal((E, H)) * 0.02
    Wr[9] = Wr[2]       # duplicate router rows -> identical logits for experts 2 and 9
    Wr[15] = Wr[4]
    x = rng.standard_normal((200, H))
    l = R.router_logits(x, Wr)
    idx = R.topk_full_sort(l, 6)
    for t in range(len(x)):
        sel = list(idx[t])
        for lo, hi in ((2, 9), (4, 15)):
            if hi in sel:
                assert lo in sel and sel.index(lo) < sel.index(hi)


def test_topk_properties_large():
    rng = np.random.default_rng(12)
    l = rng.standard_normal((500, 512))
    idx = R.topk_full_sort(l, 10)
    for t in range(0, 500, 7):
        sel = idx[t]
        assert len(set(sel)) == 10
        rest = np.setdiff1d(np.arange(512), sel)
        assert l[t, sel].min() >= l[t, rest].max()
        assert np.all(np.diff(l[t, sel]) <= 0)


def test_weights_sum_to_one_and_match_restricted_softmax():
    rng = np.random.default_rng(13)
    l = rng.standard_normal((300, 64)) * 3
    idx, w = R.route(l, 5)
    assert np.max(np.abs(w.sum(axis=1) - 1)) <= 1e-15
    # full softmax over all experts, restricted to the picks and renormalised
    full = np.exp(l - l.max(axis=1, keepdims=True))
    full = full / full.sum(axis=1, keepdims=True)
    restricted = np.take_along_axis(full, idx.astype(np.int64), axis=1)
    restricted = restricted / restricted.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(w, restricted, rtol=1e-13, atol=0)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_logits_exact_sums():
    rng = np.random.default_rng(14)
    x = rng.standard_normal((3, 128)).astype(np.float32)
    Wr = (rng.standard_normal((8, 128)) * 0.02).astype(np.float32)
    b = rng.standard_normal(8).astype(np.float32)
    l = R.router_logits(x, Wr, b)
    for t in range(3):
        for e in range(8):
            exact = math.fsum([float(x[t, h]) * float(Wr[e, h]) for h in range(128)]) + float(b[e])
            assert abs(l[t, e] - exact) <= 1e-14 * (1 + abs(exact))


def test_near_tie_flags():
    l = np.array([[3.0, 2.0, 2.0 + 1e-6, 0.0, -1.0]])
    assert R.near_tie_tokens(l, 2, 2.0 ** -12)[0]
    assert not R.near_tie_tokens(np.array([[3.0, 2.0, 1.0, 0.0]]), 2, 2.0 ** -12)[0]


def _brute_permute(idx, E):
    flat = [int(e) for e in np.asarray(idx).reshape(-1)]
    counts = [flat.count(e) for e in range(E)]
    offsets = [0]
    for c in counts:
        offsets.append(offsets[-1] + c)
    perm = sorted(range(len(flat)), key=lambda p: (flat[p], p))
    return counts, offsets, perm


@pytest.mark.parametrize("T,E,k", [(1, 16, 2), (5, 8, 3), (37, 32, 4), (200, 64, 6), (0, 8, 2)])
def test_permutation_brute_force_and_invariants(T, E, k):
    rng = np.random.default_rng(T * 1000 + E)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), np.int64)
    counts, offsets, perm, inv = P.permute(idx, E)
    bc, bo, bp = _brute_permute(idx, E)
    assert list(counts) == bc and list(offsets) == bo and list(perm) == bp
    assert counts.sum() == T * k and offsets[E] == T * k
    np.testing.assert_array_equal(inv[perm], np.arange(T * k))
    # inside an expert, pairs are in token order
    flat = idx.reshape(-1)
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg // k) > 0)


# ----------------------------------------------------------- route-tail skip

def test_route_tail_skip_brute_force():
    """The skip keeps ranks < r and resident experts; the kept weights are the
    full top-k softmax restricted to the kept picks and renormalised (an
    independent route to the same numbers); dropped picks are -1 with weight 0."""
    rng = np.random.default_rng(7)
    l = rng.normal(size=(40, 12))
    k = 5
    resident = np.zeros(12, dtype=np.uint8)
    resident[[2, 7]] = 1
    idx_full, w_full = R.route(l, k)
    for keep, res in ((1, None), (3, None), (2, resident), (5, None), (5, resident)):
        idx, w = R.route(l, k, keep=keep, resident=res)
        for t in range(l.shape[0]):
            order = sorted(range(12), key=lambda e: (-l[t, e], e))[:k]   # brute force
            kept = [j for j in range(k) if j < keep or (res is not None and res[order[j]])]
            for j in range(k):
                if j in kept:
                    assert idx[t, j] == order[j]
                    assert w[t, j] == pytest.approx(w_full[t, j] / w_full[t, kept].sum(), rel=1e-13)
                else:
                    assert idx[t, j] == -1 and w[t, j] == 0.0
            assert w[t].sum() == pytest.approx(1.0, abs=1e-15)
        if keep >= k:
            np.testing.assert_array_equal(idx, idx_full)
            np.testing.assert_array_equal(w, w_full)


def test_permutation_leaves_out_dropped_pairs():
    idx = np.array([[3, 1, -1], [1, -1, -1], [0, 3, 2]], dtype=np.int32)
    counts, offsets, perm, inv = P.permute(idx, 4)
    np.testing.assert_array_equal(counts, [1, 2, 1, 2])
    np.testing.assert_array_equal(offsets, [0, 1, 3, 4, 6])
    # live pair ids by (expert, pair id): e0: 6; e1: 1, 3; e2: 8; e3: 0, 7
    np.testing.assert_array_equal(perm, [6, 1, 3, 8, 0, 7])
    np.testing.assert_array_equal(inv, [4, 1, -1, 2, -1, -1, 0, 5, 3])
