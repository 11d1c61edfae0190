"""Pins for the oracle's router top-k and softmax (CPU only): a hand-worked
example (tests/golden/router_example.txt), brute-force checks of the
selection on random and tie-heavy logits, and softmax closed forms."""

import os

import numpy as np

from oracle.router import router_topk

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "router_example.txt")


def _golden():
    d = {}
    for line in open(GOLDEN):
        line = line.split("#")[0].split()
        if line:
            d[line[0]] = np.array([float(v) for v in line[1:]])
    return d


def test_router_worked_example():
    g = _golden()
    ids, w = router_topk(g["logits"][None, :], 3)
    assert ids[0].tolist() == g["ids"].astype(int).tolist()
    assert np.allclose(w[0], g["weights"], rtol=0, atol=5e-9)
    ids, w = router_topk(g["logits"][None, :], 3, bias=g["bias"])
    assert ids[0].tolist() == g["ids_bias"].astype(int).tolist()
    assert np.allclose(w[0], g["weights_bias"], rtol=0, atol=5e-9)


def _brute_force_check(logits, bias, k, ids):
    """Every selected expert beats every unselected one, the selection is in
    descending score and equal scores go to the lower index, by exhaustive
    pairwise comparison in float32."""
    lg = np.asarray(logits, np.float32)
    sc = lg if bias is None else (lg + np.asarray(bias, np.float32)).astype(np.float32)
    T, E = lg.shape
    for t in range(T):
        sel = [int(e) for e in ids[t]]
        assert len(set(sel)) == k
        better = lambda a, b: sc[t, a] > sc[t, b] or (sc[t, a] == sc[t, b] and a < b)
        for i in range(k - 1):
            assert better(sel[i], sel[i + 1])
        for e in range(E):
            if e not in sel:
                assert better(sel[-1], e)


def test_router_selection_brute_force_random_and_ties():
    rng = np.random.default_rng(31)
    logits = rng.standard_normal((40, 24)).astype(np.float32)
    bias = rng.uniform(-1, 1, 24).astype(np.float32)
    for b in (None, bias):
        ids, _ = router_topk(logits, 5, bias=b)
        _brute_force_check(logits, b, 5, ids)
    # heavy ties: values on a coarse grid
    tied = rng.integers(-2, 3, (40, 24)).astype(np.float32)
    ids, _ = router_topk(tied, 6)
    _brute_force_check(tied, None, 6, ids)


def test_router_softmax_closed_forms():
    # equal selected logits -> 1/k each; weights sum to 1; a shared column of 1
    ids, w = router_topk(np.zeros((3, 10), np.float32), 4, shared_expert=10)
    assert np.array_equal(w[:, :4], np.full((3, 4), 0.25))
    assert np.all(ids[:, 4] == 10) and np.all(w[:, 4] == 1.0)
    assert ids[:, :4].tolist() == [[0, 1, 2, 3]] * 3
    rng = np.random.default_rng(32)
    lg = rng.standard_normal((50, 64)).astype(np.float32) * 3
    ids, w = router_topk(lg, 6)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    # ratio of two weights = exp(difference of their logits)
    sel = np.take_along_axis(lg, ids, 1).astype(np.float64)
    assert np.allclose(w[:, 0] / w[:, 1], np.exp(sel[:, 0] - sel[:, 1]), rtol=1e-12)
