"""Pins for the fused LM-head + greedy oracle (CPU only): brute-force dot products, planted
argmaxes that the greedy rules must follow through (chain: every draft accepted; tree: the
first-child chain), and the near-tie flag on constructed ties."""

import numpy as np

from oracle import lmhead as ol
from oracle import sample as osm
from workloads import gen


def test_logits_brute_force():
    rng = np.random.default_rng(1)
    h = rng.standard_normal((2, 3, 5))
    w = rng.standard_normal((7, 5))
    lg = ol.lmhead_logits(h, w)
    for b in range(2):
        for r in range(3):
            for v in range(7):
                assert abs(lg[b, r, v] - sum(h[b, r, k] * w[v, k] for k in range(5))) < 1e-12


def test_planted_chain_accepts_every_draft():
    """Row i's argmax is the planted token of row i + 1, so all gamma drafts are accepted and the
    emitted token is the argmax of the last row."""
    B, gamma, d, V = 6, 4, 512, 3000
    inp = gen.lmhead_inputs(B, gamma + 1, d, V, 11, plant=1.0)
    out, k, near = ol.lmhead_greedy_chain(inp["hidden"], inp["weight"], inp["tokens"][:, 1:])
    lg = ol.lmhead_logits(inp["hidden"], inp["weight"])
    assert not near.any()
    assert np.all(k == gamma)
    for b in range(B):
        assert list(out[b, :gamma]) == list(inp["tokens"][b, 1:])
        assert out[b, gamma] == int(np.argmax(lg[b, gamma]))


def test_planted_tree_follows_first_children():
    parent = gen.random_tree(21, 4, 3, 2)
    first = {}
    for c in range(1, len(parent)):
        first.setdefault(int(parent[c]), c)
    chain = [0]
    while chain[-1] in first:
        chain.append(first[chain[-1]])
    inp = gen.lmhead_inputs(4, len(parent), 512, 3000, 12, plant=1.0, parent=parent)
    out, nodes, k, near = ol.lmhead_tree_greedy(inp["hidden"], inp["weight"], inp["tokens"], parent)
    assert not near.any()
    assert np.all(k == len(chain) - 1)
    for b in range(4):
        assert list(nodes[b, :k[b]]) == chain[1:]
        assert list(out[b, :k[b]]) == [int(inp["tokens"][b, c]) for c in chain[1:]]


def test_near_flag_on_ties():
    h = np.array([[[1.0, 2.0]]])
    w = np.array([[1.0, 1.0], [3.0, 0.0], [0.0, 0.0]])   # logits 3, 3, 0: an exact tie
    lg = ol.lmhead_logits(h, w)
    assert ol.near_rows(h, w, lg)[0, 0]
    w2 = np.array([[1.0, 1.0], [30.0, 0.0], [0.0, 0.0]])  # 3 vs 30
    assert not ol.near_rows(h, w2, ol.lmhead_logits(h, w2))[0, 0]
    # the greedy rule on a tie picks the smallest id (osm.argmax_rows)
    assert osm.argmax_rows(lg)[0, 0] == 0


def test_near_band_grows_with_the_hidden_size():
    """The near-tie band is the worst-case relative error of a d-term fp32 sum, d * 2^-24, never
    below the d = 4096 floor: a gap of 1e-3 of the magnitude is near at d = 65 536 (band 3.9e-3)
    but not at d = 64 (floor 2.5e-4)."""
    for d, expect in ((64, False), (65536, True)):
        h = np.zeros((1, 1, d))
        h[0, 0, 0] = 1.0
        w = np.zeros((3, d))
        w[0, 0], w[1, 0] = 1.0, 1.0 - 1e-3        # logits 1 and 0.999, sum |terms| = 1.999
        lg = ol.lmhead_logits(h, w)
        assert bool(ol.near_rows(h, w, lg)[0, 0]) is expect


def test_grid_inputs_give_order_free_fp32_logits():
    """The exact-grid inputs of the stochastic LM-head tests: any summation order of the fp32
    products gives the same logits as the float64 product, so a GPU kernel's fp32 logits must
    equal the oracle's bit for bit.  Checked here with two unrelated orders (a float32 matmul and
    a reversed running float32 sum) for the largest and smallest hidden sizes used."""
    for d, V in ((4096, 64), (64, 96)):
        inp = gen.lmhead_grid_inputs(2, 3, d, V, 41)
        ref = ol.lmhead_logits(inp["hidden"], inp["weight"])
        mm = (inp["hidden"] @ inp["weight"].T).astype(np.float64)
        assert np.array_equal(mm, ref)
        h, w = inp["hidden"][1, 2], inp["weight"][V - 1]
        acc = np.float32(0)
        for k in range(d - 1, -1, -1):
            acc = np.float32(acc + h[k] * w[k])
        assert float(acc) == ref[1, 2, V - 1]
        assert 1.0 < ref.std() < 3.0
        assert np.all(gen.round_bf16(inp["hidden"]) == inp["hidden"])
        assert np.all(gen.round_bf16(inp["weight"]) == inp["weight"])


def test_grid_inputs_planted_drafts_have_mass_in_both_models():
    """The planted draft tokens of the grid inputs sit where both softmaxes put real mass, so the
    accept test is exercised both ways (the chain is then a non-trivial sample of the rule)."""
    inp = gen.lmhead_grid_inputs(40, 5, 256, 3000, 7)
    lg = ol.lmhead_logits(inp["hidden"], inp["weight"])
    _, k, _ = osm.spec_sample_chain(lg.astype(np.float32), inp["draft_logits"], inp["tokens"], inp["uniforms"])
    counts = np.bincount(k, minlength=5)
    assert counts[0] > 0 and counts[4] > 0 and counts[1:4].sum() > 0
