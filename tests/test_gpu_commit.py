"""GPU parity: spec_commit (the rollback after verification) against the CPU oracle.

Chain commit is integer arithmetic on kv_len; tree commit moves K/V rows, so both must be
bit-exact: lengths, moved rows, and every row outside the moved range untouched."""

import numpy as np
import pytest

from oracle import attn as oa
from oracle import commit as oc
from oracle import sample as osm
from workloads import gen
from workloads.configs import CONFIGS

from .helpers import to_dev, to_np, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verify_attn_gb300 as sv
    sv.lib()
    return sv


def test_chain_commit_lengths_and_flags(sv):
    nq, Lmax = 5, 70000
    kv_len = np.array([65536, 65536, 65536, 5, 4, 70001, 300, 300], dtype=np.int32)
    nacc = np.array([0, 2, 4, 1, 1, 0, -1, 5], dtype=np.int32)
    dl, dk = to_dev(kv_len, "i32"), to_dev(nacc, "i32")
    ws = sv.spec_commit(sv.SPEC_COMMIT_CHAIN, dl, dk, nq)
    torch_mod().cuda.synchronize()
    ref, flag = oc.chain_commit(kv_len, nq, nacc, 2 ** 31 - 1)
    assert np.array_equal(to_np(dl), ref.astype(np.int32))
    assert sv.read_status(ws) & (1 | 4) == (1 | 4)   # a bad length and a bad count were flagged
    assert list(flag) == [False, False, False, False, True, False, True, True]


def _random_paths(parent, B, rng):
    N = len(parent)
    path = np.full((B, N - 1), -1, dtype=np.int32)
    acc = np.zeros(B, dtype=np.int32)
    for b in range(B):
        node = int(rng.integers(N))
        nodes = [m for m in oa.ancestors(parent, node) if m != 0]
        path[b, :len(nodes)] = nodes
        acc[b] = len(nodes)
    return path, acc


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f32", 64), ("bf16", 64)])
def test_tree_commit_moves_the_accepted_path(sv, dtype, D):
    torch = torch_mod()
    cfg = CONFIGS["medusa-tree-8k"]
    N, Hkv = cfg.tree_nodes, cfg.Hkv
    parent = gen.random_tree(N, cfg.tree_max_depth, cfg.tree_max_children, cfg.seed)
    rng = np.random.default_rng(5)
    B, Lmax = 6, 700
    kv_len = np.array([600, 64, 700, 65, 300, 200], dtype=np.int32)
    k = gen.store(rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float32), dtype)
    v = gen.store(rng.standard_normal((B, Hkv, Lmax, D)).astype(np.float32), dtype)
    path, acc = _random_paths(parent, B, rng)
    acc[5] = -1                                    # a sequence the sampler flagged
    dk, dv = to_dev(k, dtype), to_dev(v, dtype)
    dl = to_dev(kv_len, "i32")
    ws = sv.spec_commit(sv.SPEC_COMMIT_TREE, dl, to_dev(acc, "i32"), N, k=dk, v=dv,
                        path_nodes=to_dev(path, "i32"))
    torch.cuda.synchronize()
    k2, v2, ref_len, flag = oc.tree_commit(k, v, kv_len, N, path, acc)
    assert np.array_equal(to_np(dl), ref_len.astype(np.int32))
    assert np.array_equal(to_np(dk), k2.astype(np.float32))
    assert np.array_equal(to_np(dv), v2.astype(np.float32))
    assert list(flag) == [False] * 5 + [True]
    assert sv.read_status(ws) & 4


def test_tree_round_verify_sample_commit(sv):
    """One Medusa-style round on the device (tree verify, greedy tree selection, commit) against the
    oracle's; then the deepest accepted node's query over the committed cache reproduces its tree
    verify output (attention equivalence, checked on the GPU with a single-query verify)."""
    torch = torch_mod()
    cfg = CONFIGS["medusa-tree-8k"]
    N, Hq, Hkv, D, V = cfg.tree_nodes, cfg.Hq, cfg.Hkv, cfg.D, 4096
    parent = gen.random_tree(N, cfg.tree_max_depth, cfg.tree_max_children, cfg.seed)
    B = 3
    kv_len = np.array([900, 400, 1100], dtype=np.int32)
    Lmax = 1200
    inp = gen.attn_inputs(B, Hq, Hkv, D, N, kv_len, Lmax, "bf16", 77)
    smp = gen.tree_sample_inputs(B, parent, V, 78)
    dq, dk, dv = to_dev(inp["q"], "bf16"), to_dev(inp["k"], "bf16"), to_dev(inp["v"], "bf16")
    dl = to_dev(kv_len, "i32")
    o = torch.empty((B, N, Hq, D), dtype=torch.float32, device="cuda")
    sv.spec_verify_attn(dq, dk, dv, dl, o, tree_parent=parent)
    depth = int(osm.tree_depths(parent).max())
    out = torch.full((B, depth + 1), -7, dtype=torch.int32, device="cuda")
    nodes = torch.full((B, depth + 1), -7, dtype=torch.int32, device="cuda")
    nacc = torch.empty((B,), dtype=torch.int32, device="cuda")
    sv.spec_sample(sv.SPEC_SAMPLE_TREE_GREEDY, to_dev(smp["target_logits"]), out, nacc,
                   draft_tokens=to_dev(smp["node_tokens"], "i32"), tree_parent=parent, out_path_nodes=nodes)
    ref_out, ref_nodes, ref_k = osm.tree_greedy(smp["target_logits"], smp["node_tokens"], parent, depth + 1)
    assert np.array_equal(to_np(nacc), ref_k) and np.array_equal(to_np(nodes), ref_nodes)
    sv.spec_commit(sv.SPEC_COMMIT_TREE, dl, nacc, N, k=dk, v=dv, path_nodes=nodes)
    torch.cuda.synchronize()
    k2, v2, ref_len, _ = oc.tree_commit(inp["k"], inp["v"], kv_len, N, ref_nodes, ref_k)
    new_len = to_np(dl)
    assert np.array_equal(new_len, ref_len.astype(np.int32))
    assert np.array_equal(to_np(dk), k2.astype(np.float32), equal_nan=True)   # NaN past kv_len
    assert np.array_equal(to_np(dv), v2.astype(np.float32), equal_nan=True)
    # the deepest accepted node, re-queried over the committed prefix on the GPU
    o_tree = to_np(o)
    for b in range(B):
        last = int(ref_nodes[b, ref_k[b] - 1]) if ref_k[b] > 0 else 0
        q1 = dq[b:b + 1, last:last + 1].contiguous()
        o1 = torch.empty((1, 1, Hq, D), dtype=torch.float32, device="cuda")
        sv.spec_verify_attn(q1, dk[b:b + 1], dv[b:b + 1], dl[b:b + 1], o1)
        torch.cuda.synchronize()
        assert np.max(np.abs(to_np(o1)[0, 0] - o_tree[b, last])) <= 2e-3, b
