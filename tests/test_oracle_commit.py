"""Pins for the commit (rollback) oracle: the chain rule as arithmetic on the verified window,
the tree rule tied to the chain rule on chain-shaped trees, and -- independently of the copy
code -- attention equivalence: after compaction, the accepted path's last node attending over the
committed prefix sees exactly what it saw in tree verification."""

import numpy as np
import pytest

from oracle import attn as oa
from oracle import commit as oc
from oracle import sample as osm
from workloads import gen


def test_chain_commit_keeps_the_accepted_prefix():
    nq, Lmax = 5, 100
    kv_len = np.array([50, 50, 50, 5, 4, 101, 60])
    k = np.array([0, 2, 4, 1, 1, 0, -1])
    new, flag = oc.chain_commit(kv_len, nq, k, Lmax)
    # positions 45..49 were verified: the last committed token (45) plus k accepted drafts stay
    assert list(new[:4]) == [46, 48, 50, 2]
    assert list(flag) == [False, False, False, False, True, True, True]
    assert new[4] == 4 and new[5] == 101 and new[6] == 60      # flagged rows unchanged
    # a bad count (> gamma) is flagged too
    _, f2 = oc.chain_commit(np.array([50]), nq, np.array([5]), Lmax)
    assert f2[0]


def test_tree_commit_of_a_chain_shaped_tree_is_the_chain_commit():
    rng = np.random.default_rng(3)
    B, Hkv, D, N, Lmax = 3, 2, 8, 6, 40
    parent = np.arange(-1, N - 1)
    kv_len = np.array([30, 6, 40])
    k_cache = rng.standard_normal((B, Hkv, Lmax, D))
    v_cache = rng.standard_normal((B, Hkv, Lmax, D))
    acc = np.array([0, 3, 5])
    path = np.full((B, N), -1)
    for b in range(B):
        path[b, :acc[b]] = np.arange(1, acc[b] + 1)          # depth j+1 is node j+1
    k2, v2, new, flag = oc.tree_commit(k_cache, v_cache, kv_len, N, path, acc)
    ref, _ = oc.chain_commit(kv_len, N, acc, Lmax)
    assert np.array_equal(new, ref) and not flag.any()
    assert np.array_equal(k2, k_cache) and np.array_equal(v2, v_cache)   # nothing moves
    assert list(parent) == [-1, 0, 1, 2, 3, 4]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_compacted_path_attends_like_the_tree_verify(seed):
    """Attention equivalence through the independent verify oracle: node n_k of the accepted path
    sees the context plus its ancestors in tree verification; after compaction the same keys are
    the committed prefix, so single-query attention at the new last position gives the same row."""
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, D, N, V = 3, 4, 2, 16, 12, 50
    parent = gen.random_tree(N, 4, 3, 100 + seed)
    depth = osm.tree_depths(parent)
    kv_len = np.array([40, 25, 12])
    Lmax = 48
    q = rng.standard_normal((B, N, Hq, D))
    k_cache = rng.standard_normal((B, Hkv, Lmax, D))
    v_cache = rng.standard_normal((B, Hkv, Lmax, D))
    o_tree = oa.verify_attn(q, k_cache, v_cache, kv_len, tree_parent=parent)
    # an accepted path per sequence: the root path of a random node
    path = np.full((B, N), -1)
    acc = np.zeros(B, dtype=np.int64)
    last = np.zeros(B, dtype=np.int64)
    for b in range(B):
        node = int(rng.integers(N))
        chain = oa.ancestors(parent, node)            # root .. node
        nodes = [m for m in chain if m != 0]
        acc[b] = len(nodes)
        path[b, :len(nodes)] = nodes
        last[b] = node
        assert acc[b] == depth[node]
    k2, v2, new, flag = oc.tree_commit(k_cache, v_cache, kv_len, N, path, acc)
    assert not flag.any()
    for b in range(B):
        L2 = int(new[b])
        for h in range(Hq):
            g = h // (Hq // Hkv)
            ref = o_tree[b, int(last[b]), h]
            got = oa.attend(q[b, int(last[b]), h], k2[b, g, :L2], v2[b, g, :L2], 1.0 / np.sqrt(D))
            assert np.allclose(got, ref, atol=1e-12), (b, h)
    # keys outside the verified window never move
    for b in range(B):
        base = int(kv_len[b]) - N
        assert np.array_equal(k2[b][:, :base + 1], k_cache[b][:, :base + 1])


def test_tree_commit_brute_force_token_lists():
    """Tiny brute force: caches whose rows are the token ids themselves; the committed prefix must
    read context, root, then the path's node ids in depth order."""
    N, Lmax, ctx = 7, 20, 5
    parent = np.array([-1, 0, 0, 1, 1, 3, 2])
    L = ctx + N
    k_cache = np.zeros((1, 1, Lmax, 1))
    k_cache[0, 0, :L, 0] = np.concatenate([np.arange(100, 100 + ctx), np.arange(N)])
    for leaf in range(N):
        chain = [m for m in oa.ancestors(parent, leaf) if m != 0]
        path = np.full((1, N), -1)
        path[0, :len(chain)] = chain
        k2, _, new, _ = oc.tree_commit(k_cache, k_cache, np.array([L]), N, path, np.array([len(chain)]))
        got = list(k2[0, 0, :int(new[0]), 0].astype(int))
        assert got == list(range(100, 100 + ctx)) + [0] + chain


def test_tree_commit_flags_bad_inputs():
    k = np.zeros((4, 1, 10, 2))
    path = np.array([[1, 2], [1, -1], [1, 5], [1, 2]])
    _, _, new, flag = oc.tree_commit(k, k, np.array([12, 10, 10, 10]), 3, path, np.array([2, -1, 2, 3]))
    # kv_len > Lmax; a bad count; a node id outside [1, N); a count above the row (and above N - 1)
    assert list(flag) == [True, True, True, True] and list(new) == [12, 10, 10, 10]
