"""Pins for the stochastic tree rule of the sampling oracle (CPU only).

* hand-worked cases (tests/golden/tree_stochastic_small.json);
* a chain-shaped tree reduces exactly to the chain sampler (itself pinned in test_oracle_sample);
* the rule leaves the target distribution unchanged: with children drawn from the draft
  distribution, the first emitted token follows the root's target distribution, and after an
  accepted child the next token follows that child's (Monte Carlo, 6-sigma bounds);
* the residual after i rejections against one draft distribution Q is max(P - c_i Q, 0)
  normalised, with c_0 = 0 and c_{i+1} = c_i + sum max(P - c_i Q, 0) (the form the GPU kernel
  evaluates without storing a residual vector).
"""

import json
import os

import numpy as np
import pytest

from oracle import sample as osm
from workloads import gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tree_stochastic_small.json")


def _rows(p, n):
    return np.tile(np.log(np.asarray(p, dtype=np.float64)).astype(np.float32), (1, n, 1))


def test_golden_cases():
    g = json.load(open(GOLDEN))
    for case in g["cases"]:
        parent = np.array(case["parent"])
        N = len(parent)
        out, nodes, k, near = osm.tree_stochastic(_rows(g["P"], N), _rows(g["Q"], N), np.array([case["tokens"]]),
                                                  parent, np.array([case["uniforms"]], dtype=np.float32))
        assert list(out[0]) == case["out"], case["name"]
        assert list(nodes[0]) == case["nodes"], case["name"]
        assert k[0] == case["k"] and not near[0], case["name"]


def test_chain_shaped_tree_equals_chain_sampler():
    """Node i's only child is i + 1: draft row i is the chain's draft row for position i + 1, the
    child tests use the chain's uniforms u_1..u_gamma and the final draw its u_{gamma+1}."""
    B, gamma, V = 200, 5, 60
    rng = np.random.default_rng(7)
    t = (2.0 * rng.standard_normal((B, gamma + 1, V))).astype(np.float32)
    d = (t[:, :gamma] + 0.7 * rng.standard_normal((B, gamma, V))).astype(np.float32)
    x = np.array([[rng.choice(V, p=osm.softmax64(d[b, i])) for i in range(gamma)] for b in range(B)], dtype=np.int32)
    u = rng.random((B, gamma + 1), dtype=np.float32)
    out_c, k_c, near_c = osm.spec_sample_chain(t, d, x, u)
    parent = np.arange(-1, gamma, dtype=np.int32)
    tok = np.concatenate([np.zeros((B, 1), np.int32), x], axis=1)
    u_tree = np.concatenate([u[:, gamma:], u[:, :gamma]], axis=1)
    d_tree = np.concatenate([d, np.zeros((B, 1, V), np.float32)], axis=1)   # the leaf's row is not read
    out_t, nodes, k_t, near_t = osm.tree_stochastic(t, d_tree, tok, parent, u_tree)
    ok = ~(near_c | near_t)
    assert ok.sum() > 150
    assert np.array_equal(out_t[ok], out_c[ok]) and np.array_equal(k_t[ok], k_c[ok])
    assert all(list(nodes[b, :k_t[b]]) == list(range(1, k_t[b] + 1)) for b in range(B))


def _draw_children(rng, Q, parent, tok_row):
    for c in range(1, len(parent)):
        tok_row[c] = rng.choice(len(Q[parent[c]]), p=Q[parent[c]])


def test_target_distribution_is_preserved():
    """Root with 3 children, each with 2 children; children drawn i.i.d. from the parent's draft
    distribution.  First emitted token ~ P_root; given that child c was accepted, the next token
    ~ P_c (every depth-1 row is the same P1 here)."""
    V, n = 4, 60000
    P0 = np.array([0.1, 0.4, 0.3, 0.2]); Q0 = np.array([0.4, 0.1, 0.25, 0.25])
    P1 = np.array([0.6, 0.1, 0.1, 0.2]); Q1 = np.array([0.1, 0.5, 0.2, 0.2])
    parent = np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3])
    N = len(parent)
    Ps = [P0] + [P1] * 3 + [P1] * 6
    Qs = [Q0] + [Q1] * 3 + [Q1] * 6
    t = np.log(np.array(Ps))[None].astype(np.float32)
    d = np.log(np.array(Qs))[None].astype(np.float32)
    Pn = [osm.softmax64(t[0, i]) for i in range(N)]
    Qn = [osm.softmax64(d[0, i]) for i in range(N)]
    rng = np.random.default_rng(11)
    first = np.zeros(V)
    second = np.zeros(V)
    tok = np.zeros((1, N), dtype=np.int32)
    for _ in range(n):
        _draw_children(rng, Qn, parent, tok[0])
        u = rng.random((1, N), dtype=np.float32)
        out, nodes, k, _ = osm.tree_stochastic(t, d, tok, parent, u)
        first[out[0, 0]] += 1
        if k[0] >= 1:
            second[out[0, 1]] += 1
    for freq, P, m in ((first, Pn[0], n), (second, Pn[1], second.sum())):
        f = freq / m
        assert np.all(np.abs(f - P) <= 6 * np.sqrt(P * (1 - P) / m) + 1e-4), (f, P)


def test_residual_closed_form():
    rng = np.random.default_rng(3)
    for _ in range(20):
        V = 50
        P = osm.softmax64(2 * rng.standard_normal(V))
        Q = osm.softmax64(2 * rng.standard_normal(V))
        R, c = P.copy(), 0.0
        for _ in range(6):
            Nc = np.maximum(P - c * Q, 0).sum()
            assert np.allclose(R, np.maximum(P - c * Q, 0) / Nc, rtol=1e-9, atol=1e-15)
            r = np.maximum(R - Q, 0)
            if r.sum() <= 1e-12:
                break
            R, c = r / r.sum(), c + Nc
