"""Pins for the attention oracle (CPU only).

Each check ties ``oracle.attn`` to something other than itself: hand-enumerated visible sets
(tests/golden/visible_sets.json), closed forms with hand-computed values, the window = full
context equivalence, chain-shaped tree = chain verify, the page's roll-based draft cache vs the
ring layout, key-permutation invariance and planted needles.
"""

import json
import os

import numpy as np
import pytest

from oracle import attn as oa
from workloads import gen


def _one_hot_readout(L, D):
    """K = 0 (all scores equal) and V = identity rows: o[d] = 1/|S| for d in the visible set S."""
    k = np.zeros((1, 1, L, D))
    v = np.zeros((1, 1, L, D))
    for t in range(L):
        v[0, 0, t, t] = 1.0
    return k, v


def _visible_from_output(o_row):
    nz = np.nonzero(np.abs(o_row) > 1e-12)[0]
    assert np.allclose(o_row[nz], 1.0 / len(nz))
    return [int(i) for i in nz]


def test_chain_visible_sets_match_hand_enumeration(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "visible_sets.json")))["chain"]
    L, nq, D = g["L"], g["nq"], 16
    k, v = _one_hot_readout(L, D)
    q = np.random.default_rng(0).standard_normal((1, nq, 1, D))
    o = oa.verify_attn(q, k, v, np.array([L]))
    for j in range(nq):
        assert _visible_from_output(o[0, j, 0]) == g["rows"][j]


def test_tree_visible_sets_match_hand_enumeration(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "visible_sets.json")))["tree"]
    L, parent, D = g["L"], np.array(g["parent"]), 16
    N = len(parent)
    k, v = _one_hot_readout(L, D)
    q = np.random.default_rng(1).standard_normal((1, N, 1, D))
    o = oa.verify_attn(q, k, v, np.array([L]), tree_parent=parent)
    for i in range(N):
        assert _visible_from_output(o[0, i, 0]) == g["rows"][i]


def test_window_slots_match_hand_enumeration(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "visible_sets.json")))["window"]
    for case in g["cases"]:
        assert list(oa.window_slots(case["pos"], g["W"])) == case["slots"]


def test_softmax_weights_closed_form():
    # scores log(w) with w = 1, 2, 3, 4 and v_t = (t, 1): o = (sum w_t t / sum w_t, 1) = (20/10, 1)
    w = np.array([1.0, 2.0, 3.0, 4.0])
    keys = np.stack([np.log(w), np.zeros(4)], axis=1)
    vals = np.stack([np.arange(4.0), np.ones(4)], axis=1)
    o = oa.attend(np.array([1.0, 0.0]), keys, vals, scale=1.0)
    assert np.allclose(o, [2.0, 1.0], rtol=0, atol=1e-15)


def test_default_scale_is_inverse_sqrt_head_dim():
    # D = 4: q . k1 = 2 ln 2, scaled by 1/2 -> ln 2, so key 1 weighs twice key 0
    D = 4
    q = np.array([[[[2.0, 0, 0, 0]]]])                 # [1, nq=1, Hq=1, D]
    k = np.zeros((1, 1, 2, D))
    k[0, 0, 1, 0] = np.log(2.0)
    v = np.zeros((1, 1, 2, D))
    v[0, 0, 0, 1] = 3.0
    v[0, 0, 1, 2] = 3.0
    o = oa.verify_attn(q, k, v, np.array([2]))
    assert np.allclose(o[0, 0, 0], [0.0, 1.0, 2.0, 0.0], atol=1e-14)


def test_gqa_head_mapping_is_contiguous_groups():
    B, nq, Hq, Hkv, D, L = 1, 2, 8, 2, 4, 6
    q = np.random.default_rng(2).standard_normal((B, nq, Hq, D))
    k = np.random.default_rng(3).standard_normal((B, Hkv, L, D))
    v = np.zeros((B, Hkv, L, D))
    v[0, 0] = 10.0
    v[0, 1] = 11.0
    o = oa.verify_attn(q, k, v, np.array([L]))
    for h in range(Hq):
        assert np.allclose(o[0, :, h], 10.0 + h // (Hq // Hkv))


def test_closed_forms_equal_keys_one_key_constant_values():
    rng = np.random.default_rng(4)
    D, L, nq = 8, 9, 3
    q = rng.standard_normal((1, nq, 1, D))
    # all keys equal -> o = mean of visible values
    k = np.tile(rng.standard_normal(D), (1, 1, L, 1))
    v = rng.standard_normal((1, 1, L, D))
    o = oa.verify_attn(q, k, v, np.array([L]))
    for j in range(nq):
        assert np.allclose(o[0, j, 0], v[0, 0, : L - nq + j + 1].mean(axis=0), atol=1e-14)
    # one visible key -> o = v of that key (chain row 0 with L = nq)
    k = rng.standard_normal((1, 1, nq, D))
    v = rng.standard_normal((1, 1, nq, D))
    o = oa.verify_attn(q, k, v, np.array([nq]))
    assert np.allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-15)
    # constant values -> o = that constant, whatever the scores
    v = np.full((1, 1, L, D), 0.375)
    k = rng.standard_normal((1, 1, L, D)) * 5
    o = oa.verify_attn(q, k, v, np.array([L]))
    assert np.allclose(o, 0.375, atol=1e-14)


def test_chain_shaped_tree_equals_chain_verify():
    rng = np.random.default_rng(5)
    B, nq, Hq, Hkv, D = 2, 5, 4, 2, 16
    kv_len = np.array([40, 23])
    q = rng.standard_normal((B, nq, Hq, D))
    k = rng.standard_normal((B, Hkv, 40, D))
    v = rng.standard_normal((B, Hkv, 40, D))
    chain = oa.verify_attn(q, k, v, kv_len)
    parent = np.arange(-1, nq - 1)
    tree = oa.verify_attn(q, k, v, kv_len, tree_parent=parent)
    assert np.allclose(chain, tree, atol=1e-14)


def test_window_equals_full_attention_when_window_covers_context():
    # W >= context: the draft window sees everything the full-context (single-query) verify sees
    rng = np.random.default_rng(6)
    B, Hq, Hkv, D, W = 2, 4, 2, 8, 16
    pos = np.array([9, 16])
    k_ring = rng.standard_normal((B, Hkv, W, D))
    v_ring = rng.standard_normal((B, Hkv, W, D))
    q = rng.standard_normal((B, Hq, D))
    o_win, _, _ = oa.draft_window_attn(q, k_ring, v_ring, pos)
    o_full = oa.verify_attn(q[:, None], k_ring, v_ring, pos)
    assert np.allclose(o_win, o_full[:, 0], atol=1e-14)


def test_ring_layout_matches_roll_cache_over_a_long_stream():
    # the page's shift-left cache and slot = t mod W hold the same token set; attention over a key
    # set does not depend on the order of the keys
    rng = np.random.default_rng(7)
    Hq, Hkv, D, W, T = 4, 2, 8, 5, 23
    roll = oa.RollWindowCache(W, Hkv, D)
    k_ring = np.full((1, Hkv, W, D), np.nan)
    v_ring = np.full((1, Hkv, W, D), np.nan)
    for t in range(T):
        kt = rng.standard_normal((Hkv, D))
        vt = rng.standard_normal((Hkv, D))
        q = rng.standard_normal((1, Hq, D))
        roll.append(kt, vt)
        o_ring, k_ring, v_ring = oa.draft_window_attn(q, k_ring, v_ring, np.array([t + 1]),
                                                      k_new=kt[None], v_new=vt[None])
        kk, vv = roll.get_kv()
        for h in range(Hq):
            g = h // (Hq // Hkv)
            ref = oa.attend(q[0, h], kk[g], vv[g], 1.0 / np.sqrt(D))
            assert np.allclose(o_ring[0, h], ref, atol=1e-13), (t, h)


@pytest.mark.parametrize("W,S", [(5, 1), (8, 4), (6, 5), (12, 4)])
def test_sink_ring_matches_sink_roll_cache_over_a_long_stream(W, S):
    # attention sinks ([MagicDec] Best Practices §1): slot-mapped ring vs the independently laid
    # out shift-left cache with the first S tokens kept in front
    rng = np.random.default_rng(17 + W + S)
    Hq, Hkv, D, T = 4, 2, 8, 3 * W + 7
    roll = oa.SinkRollCache(W, S, Hkv, D)
    k_ring = np.full((1, Hkv, W, D), np.nan)
    v_ring = np.full((1, Hkv, W, D), np.nan)
    for t in range(T):
        kt = rng.standard_normal((Hkv, D))
        vt = rng.standard_normal((Hkv, D))
        q = rng.standard_normal((1, Hq, D))
        roll.append(kt, vt)
        o_ring, k_ring, v_ring = oa.draft_window_attn(q, k_ring, v_ring, np.array([t + 1]),
                                                      k_new=kt[None], v_new=vt[None], n_sinks=S)
        kk, vv = roll.get_kv()
        assert kk.shape[1] == min(t + 1, W)
        for h in range(Hq):
            g = h // (Hq // Hkv)
            ref = oa.attend(q[0, h], kk[g], vv[g], 1.0 / np.sqrt(D))
            assert np.allclose(o_ring[0, h], ref, atol=1e-13), (t, h)


def test_sink_slots_hold_the_visible_tokens_by_simulation():
    # write token ids into a physical slot array by the slot rule and read back the visible set
    for W, S in ((7, 0), (7, 3), (4, 1), (9, 8)):
        slots = [-1] * W
        for pos in range(1, 5 * W):
            slots[oa.token_slot(pos - 1, W, S)] = pos - 1
            held = sorted(slots[s] for s in oa.window_slots(pos, W, S))
            expect = list(range(pos)) if pos <= W else list(range(S)) + list(range(pos - (W - S), pos))
            assert held == expect, (W, S, pos)
    # no sinks: the plain ring
    for pos in range(1, 30):
        assert list(oa.window_slots(pos, 8, 0)) == sorted({t % 8 for t in range(max(0, pos - 8), pos)})


def test_context_key_permutation_invariance():
    rng = np.random.default_rng(8)
    B, nq, Hq, Hkv, D, L = 1, 3, 2, 1, 8, 30
    q = rng.standard_normal((B, nq, Hq, D))
    k = rng.standard_normal((B, Hkv, L, D))
    v = rng.standard_normal((B, Hkv, L, D))
    perm = np.concatenate([rng.permutation(L - nq), np.arange(L - nq, L)])
    o1 = oa.verify_attn(q, k, v, np.array([L]))
    o2 = oa.verify_attn(q, k[:, :, perm], v[:, :, perm], np.array([L]))
    assert np.allclose(o1, o2, atol=1e-13)


def test_planted_needle_dominates_and_trap_is_ignored():
    B, nq, Hq, Hkv, D = 1, 4, 2, 1, 32
    kv_len = np.array([50])
    inp = gen.attn_inputs(B, Hq, Hkv, D, nq, kv_len, 50, "f32", seed=11, tail_fill="zero")
    inp = gen.plant_chain_needles(inp, nq, "f32", seed=11, strength=12.0)
    k, v, q = inp["k"], inp["v"], inp["q"]
    o = oa.verify_attn(q, k, v, kv_len)
    # row 0 / head 0: the hit key dominates; the trap at L - nq + 1 is invisible to row 0
    s = k[0, 0, :47] @ q[0, 0, 0] / np.sqrt(D)
    hit = int(np.argmax(s))
    assert s[hit] - np.sort(s)[-2] > 20
    assert np.allclose(o[0, 0, 0], v[0, 0, hit], atol=1e-6)
    trap = 50 - nq + 1
    assert np.linalg.norm(o[0, 0, 0] - v[0, 0, trap]) > 1.0


def test_nan_tail_slots_are_never_read():
    B, nq, Hq, Hkv, D = 2, 5, 4, 2, 16
    kv_len = np.array([33, 20])
    inp = gen.attn_inputs(B, Hq, Hkv, D, nq, kv_len, 40, "bf16", seed=12, tail_fill="nan")
    o = oa.verify_attn(inp["q"], inp["k"], inp["v"], kv_len)
    assert np.all(np.isfinite(o))


def test_dense_masked_formulation_brute_force():
    """Brute force with the page's 2D boolean mask formulation: build the full [nq, L] mask and
    take a masked softmax over a dense score matrix (scipy), for chain and tree."""
    from scipy.special import softmax
    rng = np.random.default_rng(9)
    Hq, Hkv, D, L = 4, 2, 8, 20
    parent = np.array([-1, 0, 0, 1, 2, 2])
    for tree in (None, parent):
        nq = 5 if tree is None else len(parent)
        q = rng.standard_normal((1, nq, Hq, D))
        k = rng.standard_normal((1, Hkv, L, D))
        v = rng.standard_normal((1, Hkv, L, D))
        mask = np.zeros((nq, L), dtype=bool)
        mask[:, : L - nq] = True
        for i in range(nq):
            if tree is None:
                mask[i, L - nq: L - nq + i + 1] = True
            else:
                j = i
                while j >= 0:
                    mask[i, L - nq + j] = True
                    j = tree[j]
        o = oa.verify_attn(q, k, v, np.array([L]), tree_parent=tree)
        for h in range(Hq):
            g = h // (Hq // Hkv)
            S = (q[0, :, h] @ k[0, g].T) / np.sqrt(D)
            S = np.where(mask, S, -np.inf)
            ref = softmax(S, axis=1) @ v[0, g]
            assert np.allclose(o[0, :, h], ref, atol=1e-13)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_generators_round_to_storage(dtype):
    x = gen.store(np.random.default_rng(0).standard_normal(1000).astype(np.float32), dtype)
    if dtype == "bf16":
        assert np.all((x.view(np.uint32) & 0xFFFF) == 0)
    # round-to-nearest-even on an exact tie: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7
    assert gen.round_bf16(np.array([1.0 + 2 ** -8], dtype=np.float32))[0] == 1.0
    assert gen.round_bf16(np.array([1.0 + 3 * 2 ** -8], dtype=np.float32))[0] == 1.0 + 2 ** -6


def test_bf16_rounding_matches_torch_and_handles_specials():
    """The generator's bf16 rounding against PyTorch's float32 -> bfloat16 conversion (round to
    nearest even) on random values of every magnitude, exact ties, +-0, +-inf, subnormals and NaN,
    in an array longer than one internal block."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2 ** 32, size=(1 << 22) + 1000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32).copy()
    special = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1.0 + 2 ** -8, -(1.0 + 3 * 2 ** -8), 1e-40, -1e-40,
                        3.4028235e38], dtype=np.float32)
    x[:len(special)] = special
    got = gen.round_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    nan = np.isnan(x)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_append_places_rows_by_hand():
    """Two sequences, 2 kv heads, nq = 2: sequence 0 (kv_len 5) gets its rows at positions 3 and 4
    of each head; sequence 1 (kv_len 1 < nq) is left untouched."""
    B, Hkv, Lmax, D, nq = 2, 2, 6, 3, 2
    k = np.zeros((B, Hkv, Lmax, D))
    v = -np.ones((B, Hkv, Lmax, D))
    k_new = np.arange(B * nq * Hkv * D, dtype=np.float64).reshape(B, nq, Hkv, D) + 1.0
    v_new = 100.0 + k_new
    k2, v2 = oa.append_new_tokens(k, v, np.array([5, 1]), k_new, v_new)
    # sequence 0, head g, position 3 + j holds k_new[0, j, g]; written out element by element
    assert list(k2[0, 0, 3]) == [1.0, 2.0, 3.0] and list(k2[0, 1, 3]) == [4.0, 5.0, 6.0]
    assert list(k2[0, 0, 4]) == [7.0, 8.0, 9.0] and list(k2[0, 1, 4]) == [10.0, 11.0, 12.0]
    assert list(v2[0, 1, 4]) == [110.0, 111.0, 112.0]
    untouched = np.ones((B, Hkv, Lmax), dtype=bool)
    untouched[0, :, 3:5] = False
    assert np.all(k2[untouched] == 0.0) and np.all(v2[untouched] == -1.0)
    assert np.all(k == 0.0) and np.all(v == -1.0)          # inputs not modified


@pytest.mark.parametrize("tree", [False, True])
def test_append_then_verify_equals_verify_on_the_written_cache(tree):
    """Poison the nq tail positions with NaN, append the true rows, verify: the same output as
    verifying the intact cache (ties the append to the pinned verify oracle)."""
    B, Hq, Hkv, D, Lmax = 2, 8, 2, 16, 90
    parent = gen.random_tree(9, 3, 3, 11) if tree else None
    nq = 9 if tree else 4
    kv_len = np.array([70, 90], dtype=np.int32)
    inp = gen.attn_inputs(B, Hq, Hkv, D, nq, kv_len, Lmax, "f32", 5)
    k_new = np.stack([inp["k"][b][:, kv_len[b] - nq:kv_len[b]].transpose(1, 0, 2) for b in range(B)])
    v_new = np.stack([inp["v"][b][:, kv_len[b] - nq:kv_len[b]].transpose(1, 0, 2) for b in range(B)])
    k_bad, v_bad = inp["k"].copy(), inp["v"].copy()
    for b in range(B):
        k_bad[b, :, kv_len[b] - nq:kv_len[b]] = np.nan
        v_bad[b, :, kv_len[b] - nq:kv_len[b]] = np.nan
    k2, v2 = oa.append_new_tokens(k_bad, v_bad, kv_len, k_new, v_new)
    ref = oa.verify_attn(inp["q"], inp["k"], inp["v"], kv_len, tree_parent=parent)
    got = oa.verify_attn(inp["q"], k2, v2, kv_len, tree_parent=parent)
    assert np.array_equal(got, ref)
