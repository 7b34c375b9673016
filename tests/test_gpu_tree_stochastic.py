"""GPU parity: spec_sample(SPEC_SAMPLE_TREE) -- stochastic tree acceptance -- against the oracle.

Token decisions are compared exactly on every sequence whose decisions the oracle does not mark
as lying within 1e-6 of a threshold (fp32/float-float on the GPU, fp64 in the oracle)."""

import json
import os

import numpy as np
import pytest

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


def _gpu(sv, inp, parent, cols):
    torch = torch_mod()
    B = inp["target_logits"].shape[0]
    out = torch.full((B, cols), -7, dtype=torch.int32, device="cuda")
    nodes = torch.full((B, cols), -7, dtype=torch.int32, device="cuda")
    nacc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    sv.spec_sample(sv.SPEC_SAMPLE_TREE, to_dev(inp["target_logits"]), out, nacc,
                   draft_logits=to_dev(inp["draft_logits"]), draft_tokens=to_dev(inp["node_tokens"], "i32"),
                   uniforms=to_dev(inp["uniforms"]), tree_parent=parent, out_path_nodes=nodes, workspace=ws)
    torch.cuda.synchronize()
    return to_np(out), to_np(nodes), to_np(nacc), sv.read_status(ws)


def _compare(sv, inp, parent, min_ok):
    cols = int(osm.tree_depths(parent).max()) + 1
    out, nodes, nacc, st = _gpu(sv, inp, parent, cols)
    r_out, r_nodes, r_k, near = osm.tree_stochastic(inp["target_logits"], inp["draft_logits"], inp["node_tokens"],
                                                    parent, inp["uniforms"], cols)
    ok = ~near
    assert ok.sum() >= min_ok
    assert np.array_equal(nacc[ok], r_k[ok])
    assert np.array_equal(out[ok], r_out[ok]) and np.array_equal(nodes[ok], r_nodes[ok])
    return r_k, st


def test_medusa_tree_config(sv):
    """The Medusa tree workload's shape: 64 nodes, depth <= 4, V = 32 000, draft correlated 0.8."""
    cfg = CONFIGS["medusa-tree-8k"]
    parent = gen.random_tree(cfg.tree_nodes, cfg.tree_max_depth, cfg.tree_max_children, cfg.seed)
    inp = gen.tree_stochastic_inputs(24, parent, cfg.vocab, cfg.seed)
    k, st = _compare(sv, inp, parent, 22)
    assert st == 0 and k.max() >= 1


@pytest.mark.parametrize("V,corr", [(64, 0.9), (1024, 0.5), (4100, 0.95)])
def test_many_small_trees(sv, V, corr):
    """Many sequences over small random trees: rejections, residual draws and deep acceptances,
    vocabularies with a ragged last chunk of the final scan."""
    parent = gen.random_tree(17, 5, 3, V)
    inp = gen.tree_stochastic_inputs(300, parent, V, V + 1, draft_corr=corr)
    k, st = _compare(sv, inp, parent, 280)
    assert st == 0 and k.min() == 0 and k.max() >= 2


def test_golden_cases(sv, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "tree_stochastic_small.json")))
    for case in g["cases"]:
        parent = np.array(case["parent"])
        N = len(parent)
        pad = lambda p: np.concatenate([np.log(np.array(p, np.float64)), [-1e30]]).astype(np.float32)  # V = 4
        inp = dict(target_logits=np.tile(pad(g["P"]), (1, N, 1)), draft_logits=np.tile(pad(g["Q"]), (1, N, 1)),
                   node_tokens=np.array([case["tokens"]], np.int32),
                   uniforms=np.array([case["uniforms"]], np.float32))
        out, nodes, nacc, st = _gpu(sv, inp, parent, len(case["out"]))
        assert out[0].tolist() == case["out"] and nodes[0].tolist() == case["nodes"] and nacc[0] == case["k"], case


def test_bad_child_token_flagged(sv):
    parent = gen.random_tree(9, 3, 3, 4)
    inp = gen.tree_stochastic_inputs(3, parent, 256, 6)
    inp["node_tokens"][1, 5] = 256
    out, nodes, nacc, st = _gpu(sv, inp, parent, int(osm.tree_depths(parent).max()) + 1)
    assert nacc[1] == -1 and np.all(out[1] == -1) and st & 4
    r_out, _, r_k, near = osm.tree_stochastic(inp["target_logits"], inp["draft_logits"], inp["node_tokens"], parent,
                                              inp["uniforms"])
    assert r_k[1] == -1
    for b in (0, 2):
        if not near[b]:
            assert nacc[b] == r_k[b] and np.array_equal(out[b], r_out[b])
