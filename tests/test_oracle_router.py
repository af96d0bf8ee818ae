"""Pins for the oracle's router: group-limited top-k selection and routing weights.

The rule (page "Nemotron Is Not One Circuit", section "The Router Is A
Deterministic Algorithm"): sigmoid scores s; biased score c = s + b chooses;
equal groups scored by the sum of their two largest c; keep the best
topk_group groups; top-K of c among survivors; weights are the unbiased s of
the chosen experts, normalised, times routed_scaling_factor; ties to the lower
expert id (section "The C Kernel Contract").
"""
import itertools
import os

import numpy as np
import pytest

from oracle import moe_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _brute_force(c, n_group, topk_group, top_k):
    """Independent statement of the rule as two combinatorial maximisations
    (valid for distinct values): the kept groups are the topk_group-subset with
    the largest total group score, and the chosen experts are the top_k-subset
    of the kept experts with the largest total biased score; slots are then
    listed by decreasing c."""
    E = len(c)
    gsz = E // n_group
    groups = [list(range(g * gsz, (g + 1) * gsz)) for g in range(n_group)]
    gscore = []
    for g in groups:
        vals = [float(c[e]) for e in g]
        # largest sum of any two distinct members = sum of the two largest
        gscore.append(max(np.float32(vals[i]) + np.float32(vals[j])
                          for i, j in itertools.combinations(range(len(vals)), 2)))
    best_groups = max(itertools.combinations(range(n_group), topk_group),
                      key=lambda sub: sum(float(gscore[g]) for g in sub))
    cand = [e for g in best_groups for e in groups[g]]
    best = max(itertools.combinations(cand, top_k), key=lambda sub: sum(float(c[e]) for e in sub))
    return sorted(best, key=lambda e: -float(c[e]))


@pytest.mark.parametrize("seed", range(40))
def test_selection_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    n_group = int(rng.choice([1, 2, 3, 4]))
    gsz = int(rng.integers(2, 4))
    E = n_group * gsz
    topk_group = int(rng.integers(1, n_group + 1))
    top_k = int(rng.integers(1, min(4, topk_group * gsz) + 1))
    s = rng.uniform(0.05, 0.95, E).astype(np.float32)
    b = rng.uniform(-0.1, 0.1, E).astype(np.float32)
    c = (s + b).astype(np.float32)
    assert len(set(c.tolist())) == E
    got = O.select_token(s, b, n_group, topk_group, top_k).tolist()
    want = _brute_force(c, n_group, topk_group, top_k)
    assert got == want


def test_single_group_is_plain_topk_by_stable_sort():
    rng = np.random.default_rng(7)
    for _ in range(50):
        s = rng.uniform(0, 1, 128).astype(np.float32)
        s[rng.integers(0, 128, 10)] = s[3]          # plant ties
        b = np.zeros(128, dtype=np.float32)
        want = np.argsort(-s.astype(np.float64), kind="stable")[:6]
        assert O.select_token(s, b, 1, 1, 6).tolist() == want.tolist()


def test_batched_selection_equals_per_token_selection():
    rng = np.random.default_rng(8)
    for E, G, TG, K in [(128, 1, 1, 6), (128, 8, 3, 6), (512, 8, 4, 22), (16, 4, 2, 3)]:
        s = rng.uniform(0, 1, (64, E)).astype(np.float32)
        s[:, 5] = s[:, 9]                           # ties inside a group
        b = rng.uniform(-0.1, 0.1, E).astype(np.float32)
        batch = O.select_batch(s, b, G, TG, K)
        for t in range(64):
            assert batch[t].tolist() == O.select_token(s[t], b, G, TG, K).tolist()


def test_token_choice_fixture_from_the_page():
    rows, hist = [], None
    for line in open(os.path.join(GOLD, "token_choice_top2.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        if f[0] == "histogram":
            hist = [int(v) for v in f[1:]]
        else:
            rows.append(([float(v) for v in f[1:5]], [int(v) for v in f[5:7]]))
    counts = np.zeros(4, dtype=int)
    for aff, want in rows:
        got = O.select_token(np.array(aff, dtype=np.float32), None, 1, 1, 2).tolist()
        assert got == want
        counts[got] += 1
    assert counts.tolist() == hist


def test_group_score_is_top_two_sum_not_max():
    # group 0: c = [0.9, 0.0] (max 0.9, top-2 sum 0.9); group 1: [0.6, 0.5]
    # (max 0.6, top-2 sum 1.1).  Keeping one group must keep group 1.
    s = np.array([0.9, 0.0, 0.6, 0.5], dtype=np.float32)
    assert O.select_token(s, None, 2, 1, 1).tolist() == [2]


def test_masked_group_cannot_contribute_its_best_expert():
    # expert 0 has the largest score but its group loses on top-2 sum
    s = np.array([0.95, 0.01, 0.02, 0.6, 0.59, 0.58], dtype=np.float32)
    assert O.select_token(s, None, 2, 1, 2).tolist() == [3, 4]


def test_ties_go_to_the_lower_expert_and_the_lower_group():
    s = np.full(8, 0.5, dtype=np.float32)
    assert O.select_token(s, None, 1, 1, 3).tolist() == [0, 1, 2]
    # equal group scores: groups 0 and 1 tie, keep group 0
    assert O.select_token(s, None, 4, 1, 2).tolist() == [0, 1]
    s2 = np.array([0.1, 0.7, 0.7, 0.2], dtype=np.float32)
    assert O.select_token(s2, None, 1, 1, 2).tolist() == [1, 2]


def test_bias_moves_the_choice_but_not_the_weights():
    s = np.array([0.50, 0.49, 0.30, 0.20], dtype=np.float32)
    b = np.array([0.0, 0.0, 0.3, 0.0], dtype=np.float32)
    ids0 = O.select_token(s, None, 1, 1, 2)
    ids1 = O.select_token(s, b, 1, 1, 2)
    assert ids0.tolist() == [0, 1] and ids1.tolist() == [2, 0]
    w1 = O.routing_weights(s, ids1, 1, 2.5)
    # weights come from the unbiased scores: 0.30 and 0.50, normalised, x 2.5
    np.testing.assert_allclose(w1, np.array([0.30, 0.50]) / 0.80 * 2.5, rtol=1e-6)


def test_weights_sum_to_the_scaling_factor_and_stay_in_range():
    rng = np.random.default_rng(11)
    for rsf in (1.0, 2.5, 5.0):
        s = O.sigmoid_scores(rng.standard_normal((200, 64)).astype(np.float32))
        ids, w = O.route(s, rng.uniform(-0.1, 0.1, 64).astype(np.float32), 8, 4, 6, 1, rsf)
        np.testing.assert_allclose(w.sum(axis=1), rsf, rtol=1e-12)
        assert np.all(w > 0) and np.all(w <= rsf)
        for t in range(200):
            assert len(set(ids[t].tolist())) == 6
    # without normalisation the weights are the raw scores times the factor
    ids, w = O.route(s, None, 1, 1, 4, 0, 2.0)
    np.testing.assert_allclose(w, 2.0 * s[np.arange(200)[:, None], ids].astype(np.float64))


def test_constant_bias_shift_keeps_choice_when_margins_are_large():
    rng = np.random.default_rng(12)
    s = O.sigmoid_scores(rng.standard_normal((300, 128)).astype(np.float32))
    b = rng.uniform(-0.1, 0.1, 128).astype(np.float32)
    ids_a, w_a = O.route(s, b, 1, 1, 6, 1, 2.5)
    ids_b, w_b = O.route(s, (b + np.float32(0.25)).astype(np.float32), 1, 1, 6, 1, 2.5)
    margin = O.boundary_margin(s, b, ids_a)
    safe = margin > 1e-5
    assert safe.mean() > 0.95
    assert np.array_equal(ids_a[safe], ids_b[safe])
    assert np.array_equal(w_a[safe], w_b[safe])


def test_sigmoid_scores_match_scipy_expit_rounded_to_fp32():
    scipy_special = pytest.importorskip("scipy.special")
    z = np.linspace(-30, 30, 10001).astype(np.float32)
    want = scipy_special.expit(z.astype(np.float64)).astype(np.float32)
    assert np.array_equal(O.sigmoid_scores(z), want)
