"""Pins for the oracle's top-k routing and its expert sort.

Routing is checked by brute force over all k-subsets (and all group subsets for
grouped selection) on tiny E, by invariants (renormalised weights sum to 1, or
to routed_scaling), and against torch.softmax / torch.sigmoid.  The sort is
checked against numpy's stable argsort and np.bincount, and permute followed by
unpermute must be the identity.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle


def distinct_logits(rng, T, E):
    # a random permutation of well separated values per row: no ties, no rounding near-ties
    base = np.stack([rng.permutation(E) for _ in range(T)]).astype(np.float32)
    return (base * 0.37 - 1.0 + rng.uniform(0, 0.05, size=(T, E))).astype(np.float32)


@pytest.mark.parametrize("E,k", [(4, 1), (4, 2), (6, 3), (8, 2), (8, 5)])
def test_softmax_topk_brute_force(E, k):
    rng = np.random.default_rng(E * 10 + k)
    logits = distinct_logits(rng, 40, E)
    ids, w = oracle.route(logits, k, renormalize=True)
    for t in range(logits.shape[0]):
        best = max(itertools.combinations(range(E), k), key=lambda c: sum(float(logits[t, e]) for e in c))
        assert set(ids[t].tolist()) == set(best)
        # chosen in descending logit order
        assert np.all(np.diff(logits[t, ids[t]]) < 0)
    sel = torch.from_numpy(np.take_along_axis(logits, ids, axis=1)).double()
    ref = torch.softmax(sel, dim=1).numpy()
    assert np.allclose(w, ref, rtol=1e-6, atol=0)
    assert np.allclose(w.astype(np.float64).sum(axis=1), 1.0, atol=1e-6)


def test_softmax_without_renormalize_uses_all_experts():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((30, 16)).astype(np.float32)
    ids, w = oracle.route(logits, 4, renormalize=False)
    full = torch.softmax(torch.from_numpy(logits).double(), dim=1).numpy()
    assert np.allclose(w, np.take_along_axis(full, ids, axis=1), rtol=1e-6, atol=0)
    assert np.all(w.sum(axis=1) < 1.0)


def test_ties_resolve_to_lower_index():
    logits = np.zeros((3, 8), dtype=np.float32)
    logits[1, 5] = 1.0
    logits[2, :] = [0, 2, 2, 0, 2, 0, 0, 2]
    ids, w = oracle.route(logits, 3, renormalize=True)
    assert ids[0].tolist() == [0, 1, 2]
    assert ids[1].tolist() == [5, 0, 1]
    assert ids[2].tolist() == [1, 2, 4]
    assert np.allclose(w[0], 1 / 3)


def test_sigmoid_ungrouped_without_bias_is_topk_of_logits():
    rng = np.random.default_rng(2)
    logits = distinct_logits(rng, 50, 32)
    ids, w = oracle.route(logits, 6, True, scoring=oracle.SIGMOID, routed_scaling=2.5)
    ids_s, _ = oracle.route(logits, 6, True)                       # softmax order = logit order
    assert np.array_equal(ids, ids_s)
    sig = torch.sigmoid(torch.from_numpy(np.take_along_axis(logits, ids, axis=1)).double())
    sig = sig.float().double()                                      # scores are fp32 values
    ref = (sig / sig.sum(dim=1, keepdim=True) * 2.5).numpy()
    assert np.allclose(w, ref, rtol=1e-6, atol=0)
    assert np.allclose(w.astype(np.float64).sum(axis=1), 2.5, atol=1e-5)


def test_sigmoid_without_renormalize_weights_are_scores():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((20, 16)).astype(np.float32)
    ids, w = oracle.route(logits, 3, False, scoring=oracle.SIGMOID, routed_scaling=1.5)
    sig = torch.sigmoid(torch.from_numpy(logits).double()).float().double().numpy()
    assert np.allclose(w, np.take_along_axis(sig, ids, axis=1) * 1.5, rtol=1e-6, atol=0)


def _sig32(l):
    return torch.sigmoid(torch.from_numpy(np.asarray(l, dtype=np.float32)).double()).float().numpy()


@pytest.mark.parametrize("E,n_group,topk_group,k", [(8, 4, 2, 2), (8, 4, 2, 3), (12, 3, 2, 4), (8, 2, 1, 2)])
def test_grouped_selection_brute_force(E, n_group, topk_group, k):
    rng = np.random.default_rng(E + n_group + topk_group + k)
    logits = distinct_logits(rng, 60, E)
    bias = (rng.standard_normal(E) * 0.05).astype(np.float32)
    ids, w = oracle.route(logits, k, True, scoring=oracle.SIGMOID, bias=bias, n_group=n_group,
                          topk_group=topk_group, routed_scaling=1.0)
    G = E // n_group
    for t in range(logits.shape[0]):
        s = _sig32(logits[t])
        b = (s + bias).astype(np.float32)
        gscore = [float(np.float32(sum(sorted(b[g * G:(g + 1) * G].tolist(), reverse=True)[:2])))
                  for g in range(n_group)]
        best_groups = max(itertools.combinations(range(n_group), topk_group),
                          key=lambda c: sum(gscore[g] for g in c))
        allowed = [e for g in best_groups for e in range(g * G, (g + 1) * G)]
        best = max(itertools.combinations(allowed, k), key=lambda c: sum(float(b[e]) for e in c))
        assert set(ids[t].tolist()) == set(best), t
        # weights use the unbiased scores
        sel = s[ids[t]].astype(np.float64)
        assert np.allclose(w[t], sel / sel.sum(), rtol=1e-6)


def test_grouped_selection_single_group_equals_ungrouped():
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((40, 16)).astype(np.float32)
    bias = (rng.standard_normal(16) * 0.01).astype(np.float32)
    a = oracle.route(logits, 4, True, scoring=oracle.SIGMOID, bias=bias, n_group=1)
    b = oracle.route(logits, 4, True, scoring=oracle.SIGMOID, bias=bias, n_group=4, topk_group=4)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_route_rejects_bad_arguments():
    l = np.zeros((2, 8), dtype=np.float32)
    for kw in [dict(topk=9), dict(topk=0), dict(topk=2, n_group=3, scoring=oracle.SIGMOID),
               dict(topk=2, n_group=2, topk_group=3, scoring=oracle.SIGMOID),
               dict(topk=2, n_group=2, topk_group=1)]:
        with pytest.raises(ValueError):
            oracle.route(l, **kw)


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (16, 2, 4), (100, 8, 32), (513, 6, 64)])
def test_permute_against_stable_argsort(T, k, E):
    rng = np.random.default_rng(T)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    offsets, sorted_, pos = oracle.permute(ids, E)
    flat = ids.reshape(-1)
    counts = np.bincount(flat, minlength=E)
    assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    assert np.array_equal(sorted_, np.argsort(flat, kind="stable"))
    # unpermute(permute(x)) == x
    assert np.array_equal(sorted_[pos], np.arange(T * k))
    x = rng.standard_normal((T * k, 3))
    assert np.array_equal(x[sorted_][pos], x)


def test_permute_skewed_and_empty_experts():
    ids = np.array([[3, 3], [3, 0], [3, 3]], dtype=np.int32)
    offsets, sorted_, pos = oracle.permute(ids, 6)
    assert offsets.tolist() == [0, 1, 1, 1, 6, 6, 6]
    assert sorted_.tolist() == [3, 0, 1, 2, 4, 5]
    assert pos.tolist() == [1, 2, 3, 0, 4, 5]
