"""Pins for the sampling oracle (CPU only).

The pages fix the output law, not a procedure's intermediate numbers, so the pins are:
* lossless output: 10^6 seeded rounds on a 16-token vocabulary reproduce P (chi-square, p > 0.01),
  for identical rows (the whole emitted stream is i.i.d. P) and for per-position rows (the first
  emitted token of a round is distributed as P_1);
* mean tokens per round = (1 - a^(g+1)) / (1 - a) with a = sum min(P, Q);
* an exact-law brute force on V = 3, gamma = 2 (draft tokens enumerated with their draft
  probabilities, accept uniforms split at their thresholds, the final uniform on a fine grid);
* closed-form special cases (Q = P, disjoint supports, one-hot P, one-hot Q) and invariants;
* greedy chain vs the target's own greedy continuation, and the hand-worked tree fixture.
"""

import json
import os

import numpy as np
import pytest
from scipy import stats
from scipy.special import softmax as sp_softmax

from oracle import sample as osm


def _logits_from_probs(p):
    with np.errstate(divide="ignore"):
        return np.where(p > 0, np.log(p), -1e4).astype(np.float32)


def _rand_probs(rng, V, alpha=1.0):
    return rng.dirichlet(np.full(V, alpha))


def _draw_tokens(rng, Q, size):
    """x ~ Q by inverse CDF on a fresh uniform (harness-side draft sampler)."""
    c = np.cumsum(Q)
    c[-1] = 1.0
    return np.searchsorted(c, rng.random(size), side="right").astype(np.int32)


def _rounds_iid(P, Q, gamma, n, seed):
    rng = np.random.default_rng(seed)
    V = len(P)
    tl = np.broadcast_to(_logits_from_probs(P), (n, gamma + 1, V)).copy()
    dl = np.broadcast_to(_logits_from_probs(Q), (n, gamma, V)).copy()
    x = _draw_tokens(rng, Q, (n, gamma))
    u = rng.random((n, gamma + 1), dtype=np.float32)
    return tl, dl, x, u


def test_chi_square_stream_is_target_distribution_iid_rows():
    V, gamma, n = 16, 4, 1_000_000
    rng = np.random.default_rng(1234)
    P = _rand_probs(rng, V)
    Q = _rand_probs(rng, V)
    tl, dl, x, u = _rounds_iid(P, Q, gamma, n, seed=99)
    P = sp_softmax(tl[0, 0].astype(np.float64))     # the law the fp32 logits actually encode
    out, nacc, _ = osm.spec_sample_chain(tl, dl, x, u)
    toks = out[out >= 0]
    assert len(toks) == int((nacc + 1).sum())
    counts = np.bincount(toks, minlength=V)
    chi2, p = stats.chisquare(counts, P * counts.sum())
    assert p > 0.01, (chi2, p)


def test_chi_square_first_token_per_position_rows():
    V, gamma, n = 16, 4, 1_000_000
    rng = np.random.default_rng(4321)
    Ps = [_rand_probs(rng, V) for _ in range(gamma + 1)]
    Qs = [_rand_probs(rng, V, 0.5) for _ in range(gamma)]
    tl = np.stack([_logits_from_probs(p) for p in Ps])[None].repeat(n, 0)
    dl = np.stack([_logits_from_probs(q) for q in Qs])[None].repeat(n, 0)
    r2 = np.random.default_rng(77)
    x = np.stack([_draw_tokens(r2, Qs[i], n) for i in range(gamma)], axis=1)
    u = r2.random((n, gamma + 1), dtype=np.float32)
    out, _, _ = osm.spec_sample_chain(tl, dl, x, u)
    P1 = sp_softmax(tl[0, 0].astype(np.float64))
    counts = np.bincount(out[:, 0], minlength=V)
    chi2, p = stats.chisquare(counts, P1 * n)
    assert p > 0.01, (chi2, p)


def test_mean_tokens_per_round_matches_closed_form():
    V, gamma, n = 16, 4, 400_000
    rng = np.random.default_rng(55)
    P = _rand_probs(rng, V)
    Q = 0.6 * P + 0.4 * _rand_probs(rng, V)
    tl, dl, x, u = _rounds_iid(P, Q, gamma, n, seed=56)
    Pf = sp_softmax(tl[0, 0].astype(np.float64))
    Qf = sp_softmax(dl[0, 0].astype(np.float64))
    alpha = osm.acceptance_rate(Pf, Qf)
    E = osm.expected_tokens_per_round(alpha, gamma)
    _, nacc, _ = osm.spec_sample_chain(tl, dl, x, u)
    emitted = nacc + 1
    se = emitted.std() / np.sqrt(n)
    assert abs(emitted.mean() - E) < 4 * se, (emitted.mean(), E, se)
    assert 0.5 < alpha < 0.95


def test_expected_tokens_formula_values():
    assert osm.expected_tokens_per_round(0.0, 5) == 1.0
    assert osm.expected_tokens_per_round(1.0, 5) == 6.0
    assert np.isclose(osm.expected_tokens_per_round(0.5, 2), 1.75)   # 1 + 1/2 + 1/4


def test_exact_law_brute_force_small_vocab():
    """V = 3, gamma = 2: enumerate draft tokens (weight Q_1(x1) Q_2(x2)), split each accept
    uniform at min(1, P/Q) into its two pieces (exact), and put the final uniform on a 2^16
    midpoint grid.  The law of the first emitted token must be P_1, the law of the second given
    an accepted first must be P_2, and E[len] = 1 + a1 + a1 a2."""
    V, gamma, G = 3, 2, 1 << 16
    Ps = [np.array([0.5, 0.3, 0.2]), np.array([0.1, 0.6, 0.3]), np.array([0.25, 0.25, 0.5])]
    Qs = [np.array([0.2, 0.2, 0.6]), np.array([0.5, 0.4, 0.1])]
    tl = np.stack([_logits_from_probs(p) for p in Ps])
    dl = np.stack([_logits_from_probs(q) for q in Qs])
    Pf = [sp_softmax(r.astype(np.float64)) for r in tl]
    Qf = [sp_softmax(r.astype(np.float64)) for r in dl]
    ug = ((np.arange(G) + 0.5) / G).astype(np.float32)
    cases_x, cases_u, weights = [], [], []
    for x1 in range(V):
        for x2 in range(V):
            wx = Qf[0][x1] * Qf[1][x2]
            pieces = []
            for i, xi in enumerate((x1, x2)):
                a = min(1.0, Pf[i][xi] / Qf[i][xi])
                pieces.append([(a / 2, a), ((1 + a) / 2, 1 - a)] if a < 1 else [(0.5, 1.0)])
            for (u1, w1) in pieces[0]:
                for (u2, w2) in pieces[1]:
                    if w1 * w2 == 0:
                        continue
                    cases_x.append(np.tile([x1, x2], (G, 1)))
                    cases_u.append(np.stack([np.full(G, u1, np.float32), np.full(G, u2, np.float32), ug], 1))
                    weights.append(np.full(G, wx * w1 * w2 / G))
    x = np.concatenate(cases_x).astype(np.int32)
    u = np.concatenate(cases_u)
    w = np.concatenate(weights)
    n = len(w)
    out, nacc, _ = osm.spec_sample_chain(np.broadcast_to(tl, (n,) + tl.shape),
                                         np.broadcast_to(dl, (n,) + dl.shape), x, u)
    assert np.isclose(w.sum(), 1.0)
    first = np.bincount(out[:, 0], weights=w, minlength=V)
    assert np.allclose(first, Pf[0], atol=1e-4), (first, Pf[0])
    for a in range(V):
        sel = (nacc >= 1) & (out[:, 0] == a)
        if w[sel].sum() > 1e-9:
            second = np.bincount(out[sel, 1], weights=w[sel], minlength=V) / w[sel].sum()
            assert np.allclose(second, Pf[1], atol=1e-4), (a, second)
    a1 = np.minimum(Pf[0], Qf[0]).sum()
    a2 = np.minimum(Pf[1], Qf[1]).sum()
    assert np.isclose((w * (nacc + 1)).sum(), 1 + a1 + a1 * a2, atol=1e-9)


def test_equal_draft_and_target_accepts_everything_and_bonus_is_last_row():
    V, gamma, n = 8, 3, 20000
    rng = np.random.default_rng(3)
    P = _rand_probs(rng, V)
    tl = np.broadcast_to(_logits_from_probs(P), (n, gamma + 1, V)).copy()
    Plast = _rand_probs(rng, V)
    tl[:, gamma] = _logits_from_probs(Plast)
    dl = tl[:, :gamma].copy()
    x = _draw_tokens(rng, P, (n, gamma))
    u = rng.random((n, gamma + 1), dtype=np.float32)
    out, nacc, _ = osm.spec_sample_chain(tl, dl, x, u)
    assert np.all(nacc == gamma)
    assert np.array_equal(out[:, :gamma], x)
    bonus = np.bincount(out[:, gamma], minlength=V) / n
    assert np.allclose(bonus, sp_softmax(tl[0, gamma].astype(np.float64)), atol=0.015)


def test_disjoint_supports_reject_first_and_resample_from_target():
    V, gamma, n = 8, 4, 20000
    P = np.array([0.4, 0.3, 0.2, 0.1, 0, 0, 0, 0])
    Q = np.array([0, 0, 0, 0, 0.25, 0.25, 0.25, 0.25])
    tl, dl, x, u = _rounds_iid(P, Q, gamma, n, seed=8)
    out, nacc, _ = osm.spec_sample_chain(tl, dl, x, u)
    assert np.all(nacc == 0)
    assert np.all(out[:, 1:] == -1)
    freq = np.bincount(out[:, 0], minlength=V) / n
    assert np.allclose(freq, P, atol=0.015)


def test_one_hot_target_reduces_to_greedy_decode():
    V, gamma, n = 32, 4, 2000
    rng = np.random.default_rng(10)
    tl = rng.standard_normal((n, gamma + 1, V)).astype(np.float32)
    a = rng.integers(V, size=(n, gamma + 1))
    np.put_along_axis(tl, a[..., None], 1e3, axis=-1)          # P one-hot at a in float64
    dl = rng.standard_normal((n, gamma, V)).astype(np.float32)
    x = np.where(rng.random((n, gamma)) < 0.7, a[:, :gamma], rng.integers(V, size=(n, gamma))).astype(np.int32)
    u = rng.random((n, gamma + 1), dtype=np.float32)
    out_s, k_s, _ = osm.spec_sample_chain(tl, dl, x, u)
    out_g, k_g = osm.greedy_chain(tl, x)
    assert np.array_equal(k_s, k_g)
    assert np.array_equal(out_s, out_g)


def test_one_hot_draft_accepts_with_probability_target_mass():
    # Q one-hot at x: the accept test u * 1 < P(x) passes for a fraction P(x) of uniforms
    V, G = 6, 1 << 14
    P = np.array([0.05, 0.15, 0.3, 0.2, 0.1, 0.2])
    tl = np.broadcast_to(_logits_from_probs(P), (G, 2, V)).copy()
    dl = np.full((G, 1, V), -1e4, dtype=np.float32)
    dl[:, 0, 2] = 0.0
    x = np.full((G, 1), 2, dtype=np.int32)
    ug = ((np.arange(G) + 0.5) / G).astype(np.float32)
    u = np.stack([ug, np.full(G, 0.5, np.float32)], axis=1)
    _, nacc, _ = osm.spec_sample_chain(tl, dl, x, u)
    Pf = sp_softmax(tl[0, 0].astype(np.float64))
    assert abs(nacc.mean() - Pf[2]) <= 1.0 / G


def test_zero_residual_falls_back_to_target_row():
    # P == Q with a draft token of zero mass under both: the test u * 0 < 0 fails, the
    # residual is identically zero and the draw comes from P itself.
    V, G = 5, 4096
    P = np.array([0.1, 0.2, 0.3, 0.4, 0.0])
    tl = np.broadcast_to(_logits_from_probs(P), (G, 2, V)).copy()
    dl = tl[:, :1].copy()
    x = np.full((G, 1), 4, dtype=np.int32)
    ug = ((np.arange(G) + 0.5) / G).astype(np.float32)
    u = np.stack([np.full(G, 0.3, np.float32), ug], axis=1)
    out, nacc, _ = osm.spec_sample_chain(tl, dl, x, u)
    assert np.all(nacc == 0)
    freq = np.bincount(out[:, 0], minlength=V) / G
    assert np.allclose(freq, sp_softmax(tl[0, 0].astype(np.float64)), atol=2.0 / G)


def test_invariants_on_random_rounds():
    rng = np.random.default_rng(12)
    B, gamma, V = 3000, 5, 40
    tl = (2 * rng.standard_normal((B, gamma + 1, V))).astype(np.float32)
    dl = (tl[:, :gamma] + rng.standard_normal((B, gamma, V))).astype(np.float32)
    x = rng.integers(V, size=(B, gamma)).astype(np.int32)
    u = rng.random((B, gamma + 1), dtype=np.float32)
    out, nacc, _ = osm.spec_sample_chain(tl, dl, x, u)
    assert np.all((nacc >= 0) & (nacc <= gamma))
    P = sp_softmax(tl.astype(np.float64), axis=-1)
    Q = sp_softmax(dl.astype(np.float64), axis=-1)
    for b in range(B):
        k = nacc[b]
        assert np.all(out[b, : k + 1] >= 0) and np.all(out[b, k + 1:] == -1)
        assert np.array_equal(out[b, :k], x[b, :k])
        for i in range(min(k + 1, gamma)):
            if P[b, i, x[b, i]] >= Q[b, i, x[b, i]]:
                assert i < k, "a draft with P >= Q must be accepted"


def test_bad_token_marks_row():
    tl = np.zeros((2, 3, 4), np.float32)
    dl = np.zeros((2, 2, 4), np.float32)
    x = np.array([[0, 1], [1, 7]], np.int32)
    u = np.full((2, 3), 0.5, np.float32)
    out, nacc, _ = osm.spec_sample_chain(tl, dl, x, u)
    assert nacc[1] == -1 and np.all(out[1] == -1)
    assert nacc[0] == 2


def test_greedy_chain_reproduces_target_greedy_continuation():
    rng = np.random.default_rng(13)
    B, gamma, V = 50, 4, 100
    tl = rng.standard_normal((B, gamma + 1, V)).astype(np.float32)
    a = np.argmax(tl, -1)
    out, k = osm.greedy_chain(tl, a[:, :gamma].astype(np.int32))
    assert np.all(k == gamma) and np.array_equal(out, a)
    x = a[:, :gamma].copy()
    x[:, 2] = (x[:, 2] + 1) % V
    out, k = osm.greedy_chain(tl, x.astype(np.int32))
    assert np.all(k == 2) and np.array_equal(out[:, :3], a[:, :3]) and np.all(out[:, 3:] == -1)


def test_tree_greedy_hand_worked_fixture(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "tree_greedy_small.json")))
    parent = np.array(g["parent"])
    for case in g["cases"]:
        tl = np.array(case["logits"], np.float32)[None]
        tok = np.array(case["tokens"], np.int32)[None]
        out, nodes, nacc = osm.tree_greedy(tl, tok, parent)
        assert out[0].tolist() == case["out_tokens"]
        assert nodes[0].tolist()[: len(case["path_nodes"])] == case["path_nodes"]
        assert nacc[0] == case["num_accepted"]


def test_chain_shaped_tree_equals_greedy_chain():
    rng = np.random.default_rng(14)
    B, N, V = 40, 6, 30
    tl = rng.standard_normal((B, N, V)).astype(np.float32)
    a = np.argmax(tl, -1)
    tok = np.zeros((B, N), np.int32)
    tok[:, 1:] = np.where(rng.random((B, N - 1)) < 0.7, a[:, :-1], rng.integers(V, size=(B, N - 1)))
    parent = np.arange(-1, N - 1)
    out_t, _, k_t = osm.tree_greedy(tl, tok, parent, out_cols=N)
    out_c, k_c = osm.greedy_chain(tl, tok[:, 1:])
    assert np.array_equal(k_t, k_c)
    assert np.array_equal(out_t, out_c)


def test_near_threshold_flag():
    # u exactly at P/Q +- 1e-7 is flagged; far away it is not
    V = 4
    P = np.array([0.4, 0.3, 0.2, 0.1])
    Q = np.array([0.1, 0.2, 0.3, 0.4])
    tl = _logits_from_probs(P)[None, None].repeat(2, 1)
    dl = _logits_from_probs(Q)[None, None]
    Pf = sp_softmax(tl[0, 0].astype(np.float64))
    Qf = sp_softmax(dl[0, 0].astype(np.float64))
    ratio = Pf[3] / Qf[3]
    x = np.array([[3]], np.int32)
    near_u = np.array([[np.float32(ratio), 0.5]], np.float32)
    far_u = np.array([[0.9, 0.5]], np.float32)
    _, _, f1 = osm.spec_sample_chain(tl, dl, x, near_u)
    _, _, f2 = osm.spec_sample_chain(tl, dl, x, far_u)
    assert f1[0] and not f2[0]


def test_outcome_validity_accepts_own_outcome_and_only_it_away_from_thresholds():
    """chain_outcome_valid: the oracle's own outcome is always valid; for a sequence with no near
    decision, changing the count by one or the emitted token by one makes it invalid."""
    rng = np.random.default_rng(31)
    B, gamma, V = 400, 3, 12
    tl = (2 * rng.standard_normal((B, gamma + 1, V))).astype(np.float32)
    dl = (tl[:, :gamma] + rng.standard_normal((B, gamma, V))).astype(np.float32)
    Q = sp_softmax(dl.astype(np.float64), axis=-1)
    x = np.stack([_draw_tokens(rng, Q[b, i], ()) for b in range(B) for i in range(gamma)]).reshape(B, gamma)
    u = rng.random((B, gamma + 1), dtype=np.float32)
    out, nacc, near = osm.spec_sample_chain(tl, dl, x, u)
    assert np.all(osm.chain_outcome_valid(tl, dl, x, u, out, nacc))
    far = np.nonzero(~near)[0]
    assert len(far) > 300
    for b in far:
        k, y = int(nacc[b]), int(out[b, nacc[b]])
        for y2 in (y - 1, y + 1):
            if 0 <= y2 < V:
                o2 = out[b:b + 1].copy()
                o2[0, k] = y2
                assert not osm.chain_outcome_valid(tl[b:b + 1], dl[b:b + 1], x[b:b + 1], u[b:b + 1], o2, nacc[b:b + 1])[0]
        for k2 in (k - 1, k + 1):
            if 0 <= k2 <= gamma:
                o2 = np.full((1, gamma + 1), -1, np.int32)
                o2[0, :k2] = x[b, :k2]
                # every token is tried at the new count: none may be valid
                for y2 in range(V):
                    o2[0, k2] = y2
                    assert not osm.chain_outcome_valid(tl[b:b + 1], dl[b:b + 1], x[b:b + 1], u[b:b + 1], o2,
                                                       np.array([k2]))[0]


def test_outcome_validity_lets_near_decisions_go_either_way():
    # draw: uniform P over 4 tokens, every draft accepted (Q = P), u R = 0.5 = C(1) exactly: the
    # exact rule gives y = 2, and y = 1 lies on the other side of the step
    V, gamma = 4, 1
    tl = np.zeros((1, gamma + 1, V), np.float32)
    dl = np.zeros((1, gamma, V), np.float32)
    x = np.array([[0]], np.int32)
    u = np.array([[0.3, 0.5]], np.float32)
    out, nacc, near = osm.spec_sample_chain(tl, dl, x, u)
    assert nacc[0] == 1 and out[0, 1] == 2 and near[0]
    for y, ok in ((0, False), (1, True), (2, True), (3, False)):
        o = np.array([[0, y]], np.int32)
        assert osm.chain_outcome_valid(tl, dl, x, u, o, nacc)[0] == ok, y
    # accept test: P(x)/Q(x) = 0.5 and u = 0.5 (rejected by the strict test, but near): both counts
    P = np.array([0.25, 0.25, 0.25, 0.25])
    Qd = np.array([0.5, 0.5 / 3, 0.5 / 3, 0.5 / 3])
    tl = _logits_from_probs(P)[None, None].repeat(2, 1)
    dl = _logits_from_probs(Qd)[None, None]
    ratio = sp_softmax(tl[0, 0].astype(np.float64))[0] / sp_softmax(dl[0, 0].astype(np.float64))[0]
    u = np.array([[np.float32(ratio), 0.9]], np.float32)
    out, nacc, near = osm.spec_sample_chain(tl, dl, x, u)
    assert near[0]
    # the count the exact rule did not take, with the draw its residual row gives
    k2 = 1 - int(nacc[0])
    u_draw = np.array([[0.0, 0.9]], np.float32) if k2 == 1 else np.array([[0.99, 0.9]], np.float32)
    o2, n2, _ = osm.spec_sample_chain(tl, dl, x, u_draw)
    assert n2[0] == k2
    assert osm.chain_outcome_valid(tl, dl, x, u, out, nacc)[0]
    assert osm.chain_outcome_valid(tl, dl, x, u, o2, n2)[0]


def test_outcome_validity_bad_token_row():
    tl = np.zeros((1, 3, 4), np.float32)
    dl = np.zeros((1, 2, 4), np.float32)
    x = np.array([[1, 9]], np.int32)
    u = np.full((1, 3), 0.5, np.float32)
    assert osm.chain_outcome_valid(tl, dl, x, u, np.full((1, 3), -1, np.int32), np.array([-1]))[0]
    assert not osm.chain_outcome_valid(tl, dl, x, u, np.array([[1, 2, -1]], np.int32), np.array([1]))[0]
