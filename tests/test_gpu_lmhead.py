"""GPU parity: spec_lmhead_sample -- the LM-head projection fused with greedy or stochastic chain /
tree verification -- against the oracle.

The GPU accumulates bf16 products in fp32; the oracle takes the exact float64 dot products.  Token
decisions are compared exactly on every sequence none of whose consulted rows the oracle marks as
near-tied (top two logits within the fp32 accumulation bound of a d-term dot product of each
other); the near-tied ones are only checked for validity.

The stochastic modes run on exact-grid inputs (``workloads.gen.lmhead_grid_inputs``): every fp32
partial sum of those dot products is exact, so the GPU's logits must equal the oracle's bit for
bit, and the sampled outcomes are then held to spec_sample's own bar (exact wherever no decision
lies within 1e-6 of its threshold, valid elsewhere)."""

import numpy as np
import pytest

from oracle import lmhead as ol
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


def _gpu(sv, mode, hidden, weight, tokens, cols, parent=None):
    torch = torch_mod()
    B = hidden.shape[0]
    out = torch.full((B, cols), -7, dtype=torch.int32, device="cuda")
    nodes = torch.full((B, cols), -7, dtype=torch.int32, device="cuda")
    nacc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    need = sv.spec_lmhead_sample_workspace(mode, hidden, weight)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    sv.spec_lmhead_sample(mode, hidden, weight, out, nacc, draft_tokens=tokens, tree_parent=parent,
                          out_path_nodes=nodes if parent is not None else None, workspace=ws)
    torch.cuda.synchronize()
    return to_np(out), to_np(nodes), to_np(nacc), sv.read_status(ws)


def _chain(sv, inp, gamma, min_ok, drafts=None):
    drafts = inp["tokens"][:, 1:gamma + 1] if drafts is None else drafts
    h, w = to_dev(inp["hidden"], "bf16"), to_dev(inp["weight"], "bf16")
    tok = to_dev(drafts, "i32") if gamma > 0 else None
    out, _, nacc, st = _gpu(sv, sv.SPEC_SAMPLE_CHAIN_GREEDY, h, w, tok, gamma + 1)
    r_out, r_k, near = ol.lmhead_greedy_chain(inp["hidden"], inp["weight"], drafts)
    ok = ~near
    assert st == 0
    assert ok.sum() >= min_ok
    assert np.array_equal(nacc[ok], r_k[ok])
    assert np.array_equal(out[ok], r_out[ok])
    _valid_chain(inp, drafts, out, nacc, ~ok)
    return r_k


def _valid_chain(inp, drafts, out, nacc, which):
    """Near-tied sequences: every accepted draft and the emitted token are within the fp32 bound
    of their row's maximum."""
    if not which.any():
        return
    lg = ol.lmhead_logits(inp["hidden"][which], inp["weight"])
    for i, b in enumerate(np.nonzero(which)[0]):
        k = int(nacc[b])
        assert 0 <= k <= drafts.shape[1]
        assert list(out[b, :k]) == list(drafts[b, :k])
        for r in range(k + 1):
            t = int(out[b, r])
            assert lg[i, r].max() - lg[i, r, t] <= 1e-3 * np.abs(lg[i, r]).max() + 1e-6


def _tree(sv, inp, parent, min_ok):
    cols = int(osm.tree_depths(parent).max()) + 1
    h, w = to_dev(inp["hidden"], "bf16"), to_dev(inp["weight"], "bf16")
    out, nodes, nacc, st = _gpu(sv, sv.SPEC_SAMPLE_TREE_GREEDY, h, w, to_dev(inp["tokens"], "i32"), cols, parent)
    r_out, r_nodes, r_k, near = ol.lmhead_tree_greedy(inp["hidden"], inp["weight"], inp["tokens"], parent, cols)
    ok = ~near
    assert st == 0
    assert ok.sum() >= min_ok
    assert np.array_equal(nacc[ok], r_k[ok])
    assert np.array_equal(out[ok], r_out[ok]) and np.array_equal(nodes[ok], r_nodes[ok])
    return r_k


def test_chain_small_ragged_vocab(sv):
    """8 vocabulary tiles, the last one 104 entries long; d = 128 (two K chunks)."""
    inp = gen.lmhead_inputs(3, 5, 128, 1000, 301)
    k = _chain(sv, inp, 4, 3)
    assert k.max() >= 1


def test_chain_llama3_8b_lm_head(sv):
    """LLaMA-3-8B's LM head (d 4096, V 128 256), batch 8, gamma 4: the full-size launch."""
    cfg = CONFIGS["llama3-8b-layer"]
    inp = gen.lmhead_inputs(cfg.B, cfg.gamma + 1, 4096, cfg.vocab, cfg.seed)
    k = _chain(sv, inp, cfg.gamma, cfg.B - 1)
    assert k.max() >= 2


def test_chain_gamma_zero(sv):
    """No drafts: the emitted token is row 0's argmax; V = 130 leaves a 2-entry last tile."""
    inp = gen.lmhead_inputs(2, 1, 64, 130, 302)
    k = _chain(sv, inp, 0, 2)
    assert np.all(k == 0)


def test_chain_many_tiles_per_cta(sv):
    """230 vocabulary tiles (V = 29 435, a ragged last tile), d = 1024 (four K groups of four
    chunks), 40 rows: more tiles than SMs, so CTAs take two tiles each in one pass."""
    inp = gen.lmhead_inputs(8, 5, 1024, 29435, 312)
    k = _chain(sv, inp, 4, 6)
    assert k.max() >= 1


def test_chain_many_tiles_several_passes(sv):
    """600 vocabulary tiles (V = 76 797), d = 256 (two K groups), 160 rows: three tiles fill TMEM,
    so a CTA's four tiles take two passes (the hidden rows staged once per pass)."""
    inp = gen.lmhead_inputs(32, 5, 256, 76797, 313)
    k = _chain(sv, inp, 4, 23)
    assert k.max() >= 1


def test_chain_256_rows(sv):
    """B * (gamma + 1) = 255 hidden rows: the widest accumulator (N = 256), two tiles per pass."""
    inp = gen.lmhead_inputs(51, 5, 64, 300, 303)
    _chain(sv, inp, 4, 48)


def test_chain_longest_gamma(sv):
    """gamma = 32, the longest chain the ABI takes (33 rows per sequence, 231 rows in all)."""
    inp = gen.lmhead_inputs(7, 33, 128, 1000, 310, plant=0.9)
    k = _chain(sv, inp, 32, 6)
    assert k.max() >= 3


def test_largest_hidden_size(sv):
    """d = 65 536, the largest hidden size the ABI takes (1024 K chunks per tile).  The worst-case
    fp32 band grows with d, so every row gets a planted winner (margin ~3 sqrt(d) against N(0, 1)
    logits): sequence 0 accepts both drafts, sequence 1 has its second draft replaced and rejects
    it; every consulted row must then be outside the band."""
    d, V = 65536, 300
    inp = gen.lmhead_inputs(2, 3, d, V, 311, plant=1.0)
    w, tok = inp["weight"].copy(), inp["tokens"].copy()
    planted = {int(t) for t in tok[:, 1:].ravel()}
    free = [t for t in range(V) if t not in planted]
    for b in range(2):   # the last row's winner (no draft follows it)
        w[free[b]] = gen.store(inp["hidden"][b, 2] * np.float32(3.0 / np.sqrt(d)), "bf16")
    tok[1, 2] = free[2]
    k = _chain(sv, dict(hidden=inp["hidden"], weight=w, tokens=tok), 2, 2)
    assert list(k) == [2, 1]


def test_chain_planted_at_tile_edges(sv):
    """Drafts planted at vocabulary ids 127, 128 and V - 1 (the last and first entries of tiles
    and the last entry of the ragged tile), in every position of the chain."""
    gamma, d, V = 3, 256, 1001
    base = gen.lmhead_inputs(1, gamma + 1, d, V, 304, plant=0.0)
    for order in ([127, 128, V - 1], [V - 1, 127, 128], [128, V - 1, 127]):
        w = base["weight"].copy()
        tok = base["tokens"].copy()
        for i, t in enumerate(order):
            w[t] = gen.store(base["hidden"][0, i] * np.float32(3.0 / np.sqrt(d)), "bf16")
            tok[0, i + 1] = t
        k = _chain(sv, dict(hidden=base["hidden"], weight=w, tokens=tok), gamma, 1)
        assert k[0] == gamma


def test_exact_tie_goes_to_smaller_id(sv):
    """Two identical weight rows in different tiles (and CTAs): the smaller id wins."""
    torch = torch_mod()
    d, V = 128, 2048
    inp = gen.lmhead_inputs(1, 1, d, V, 305, plant=0.0)
    w = inp["weight"].copy()
    row = gen.store(inp["hidden"][0, 0] * np.float32(3.0 / np.sqrt(d)), "bf16")
    w[1700] = row
    w[300] = row
    h, wd = to_dev(inp["hidden"], "bf16"), to_dev(w, "bf16")
    out, _, nacc, st = _gpu(sv, sv.SPEC_SAMPLE_CHAIN_GREEDY, h, wd, None, 1)
    assert st == 0 and nacc[0] == 0 and out[0, 0] == 300
    del torch


def test_zero_logits_tie_to_id_zero(sv):
    """An all-zero hidden row makes every logit +0 or -0 (products of zero with weights of either
    sign): all equal, so the argmax is id 0 -- a signed-zero order would pick some +0 instead."""
    torch = torch_mod()
    d, V = 64, 700
    w = gen.lmhead_inputs(1, 1, d, V, 309, plant=0.0)["weight"]
    h = np.zeros((2, 1, d), dtype=np.float32)
    out, _, nacc, st = _gpu(sv, sv.SPEC_SAMPLE_CHAIN_GREEDY, to_dev(h, "bf16"), to_dev(w, "bf16"), None, 1)
    assert st == 0 and list(nacc) == [0, 0] and list(out[:, 0]) == [0, 0]
    assert int(np.argmax(ol.lmhead_logits(h, w)[0, 0])) == 0
    del torch


def test_tree_medusa_lm_head(sv):
    """Vicuna-7B-sized LM head (d 4096, V 32 000) over the Medusa tree (64 nodes), batch 4:
    256 hidden rows."""
    cfg = CONFIGS["medusa-tree-8k"]
    parent = gen.random_tree(cfg.tree_nodes, cfg.tree_max_depth, cfg.tree_max_children, cfg.seed)
    inp = gen.lmhead_inputs(cfg.B, len(parent), 4096, cfg.vocab, cfg.seed, parent=parent)
    k = _tree(sv, inp, parent, cfg.B - 1)
    assert k.max() >= 2


@pytest.mark.parametrize("N,depth,ch,B,d,V", [(9, 3, 3, 5, 192, 777), (2, 1, 1, 1, 64, 129), (1, 0, 0, 3, 64, 50)])
def test_tree_small(sv, N, depth, ch, B, d, V):
    parent = gen.random_tree(N, depth, ch, 306 + N) if N > 1 else np.array([-1], dtype=np.int32)
    inp = gen.lmhead_inputs(B, N, d, V, 307 + N, parent=parent)
    _tree(sv, inp, parent, B - 1)


def test_bad_token_flagged(sv):
    torch = torch_mod()
    inp = gen.lmhead_inputs(3, 4, 64, 500, 308)
    drafts = inp["tokens"][:, 1:].copy()
    drafts[1, 2] = 500
    h, w = to_dev(inp["hidden"], "bf16"), to_dev(inp["weight"], "bf16")
    out, _, nacc, st = _gpu(sv, sv.SPEC_SAMPLE_CHAIN_GREEDY, h, w, to_dev(drafts, "i32"), 4)
    assert st == sv.SPEC_STATUS_BAD_TOKEN
    assert nacc[1] == -1 and np.all(out[1] == -1)
    r_out, r_k, near = ol.lmhead_greedy_chain(inp["hidden"][[0, 2]], inp["weight"], drafts[[0, 2]])
    for i, b in enumerate((0, 2)):
        if not near[i]:
            assert nacc[b] == r_k[i] and list(out[b]) == list(r_out[i])
    del torch


def _stochastic(sv, mode, inp, parent=None, take_logits=True):
    """One stochastic fused call on the grid inputs; returns the outputs, the status word and the
    logits the GEMM wrote (None unless taken through out_logits)."""
    torch = torch_mod()
    B, R, _ = inp["hidden"].shape
    V = inp["weight"].shape[0]
    tree = parent is not None
    cols = int(osm.tree_depths(parent).max()) + 1 if tree else R
    h, w = to_dev(inp["hidden"], "bf16"), to_dev(inp["weight"], "bf16")
    out = torch.full((B, cols), -7, dtype=torch.int32, device="cuda")
    nodes = torch.full((B, cols), -7, dtype=torch.int32, device="cuda")
    nacc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    lg = torch.full((B, R, V), float("nan"), dtype=torch.float32, device="cuda") if take_logits else None
    need = sv.spec_lmhead_sample_workspace(mode, h, w, lg)
    ws = torch.full((need,), 0xA5, dtype=torch.uint8, device="cuda")   # stale bytes: the call clears what it needs
    sv.spec_lmhead_sample(mode, h, w, out, nacc, draft_tokens=to_dev(inp["tokens"], "i32"), tree_parent=parent,
                          out_path_nodes=nodes if tree else None, workspace=ws,
                          draft_logits=to_dev(inp["draft_logits"]), uniforms=to_dev(inp["uniforms"]), out_logits=lg)
    torch.cuda.synchronize()
    return to_np(out), to_np(nodes), to_np(nacc), sv.read_status(ws), None if lg is None else to_np(lg)


def _stochastic_chain(sv, inp, min_ok, take_logits=True):
    """Grid inputs make every fp32 logit exact, so the GPU's logits equal the oracle's float64 ones
    bit for bit and the sampling decisions must agree wherever the oracle marks none near."""
    out, _, nacc, st, lg = _stochastic(sv, sv.SPEC_SAMPLE_CHAIN, inp, take_logits=take_logits)
    ref = ol.lmhead_logits(inp["hidden"], inp["weight"])
    if lg is not None:
        assert np.array_equal(lg.astype(np.float64), ref)
    t = ref.astype(np.float32)
    r_out, r_k, near = osm.spec_sample_chain(t, inp["draft_logits"], inp["tokens"], inp["uniforms"])
    ok = ~near
    assert st == 0
    assert ok.sum() >= min_ok
    assert np.array_equal(nacc[ok], r_k[ok]) and np.array_equal(out[ok], r_out[ok])
    if near.any():
        assert osm.chain_outcome_valid(t[near], inp["draft_logits"][near], inp["tokens"][near],
                                       inp["uniforms"][near], out[near], nacc[near]).all()
    return r_k


def _stochastic_tree(sv, inp, parent, min_ok, take_logits=True):
    out, nodes, nacc, st, lg = _stochastic(sv, sv.SPEC_SAMPLE_TREE, inp, parent, take_logits=take_logits)
    ref = ol.lmhead_logits(inp["hidden"], inp["weight"])
    if lg is not None:
        assert np.array_equal(lg.astype(np.float64), ref)
    cols = out.shape[1]
    r_out, r_nodes, r_k, near = osm.tree_stochastic(ref.astype(np.float32), inp["draft_logits"], inp["tokens"],
                                                    parent, inp["uniforms"], cols)
    ok = ~near
    assert st == 0
    assert ok.sum() >= min_ok
    assert np.array_equal(nacc[ok], r_k[ok])
    assert np.array_equal(out[ok], r_out[ok]) and np.array_equal(nodes[ok], r_nodes[ok])
    for b in np.nonzero(near)[0]:       # near: the path must still be a parent chain of drafts
        k = int(nacc[b])
        assert 0 <= k < cols
        prev = 0
        for j in range(k):
            n = int(nodes[b, j])
            assert parent[n] == prev and out[b, j] == inp["tokens"][b, n]
            prev = n
    return r_k


def test_stochastic_chain_llama3_8b_lm_head(sv):
    """LLaMA-3-8B's LM head (d 4096, V 128 256), batch 8, gamma 4, on exact-grid inputs: the
    projected logits match bit for bit and the sampled outcome matches the oracle's."""
    cfg = CONFIGS["llama3-8b-layer"]
    inp = gen.lmhead_grid_inputs(cfg.B, cfg.gamma + 1, 4096, cfg.vocab, cfg.seed)
    k = _stochastic_chain(sv, inp, int(np.ceil(0.7 * cfg.B)))
    assert k.max() >= 1


def test_stochastic_chain_magicdec_batch(sv):
    """The MagicDec batch (32 sequences x 5 rows = 160 hidden rows: three accumulator passes) over
    the LLaMA-3 vocabulary, logits handed out: the shape of the bench's LM-head record."""
    cfg = CONFIGS["magicdec-64k"]
    inp = gen.lmhead_grid_inputs(cfg.B, cfg.gamma + 1, 4096, cfg.vocab, cfg.seed)
    # over 128 256 tokens the residual's CDF steps are ~1e-5 of its mass apart, so a draw lands
    # within the 1e-6 band of a step for up to a quarter of the sequences (checked for validity)
    k = _stochastic_chain(sv, inp, int(np.ceil(0.7 * cfg.B)))
    assert k.min() == 0 and k.max() >= 2


@pytest.mark.parametrize("B,gamma,d,V,take", [(50, 4, 256, 3000, True), (40, 5, 128, 1004, False),
                                              (7, 32, 64, 2048, True), (3, 1, 192, 2052, False)])
def test_stochastic_chain_shapes(sv, B, gamma, d, V, take):
    """Both sampling paths (V <= 2048: one warp per sequence; above: the statistics pass), a
    ragged last vocabulary tile, the longest chain, logits kept in the workspace or handed out."""
    inp = gen.lmhead_grid_inputs(B, gamma + 1, d, V, 320 + gamma)
    k = _stochastic_chain(sv, inp, B - 2, take_logits=take)
    if B >= 40:
        assert k.min() == 0 and k.max() >= 2


def test_stochastic_tree_medusa_lm_head(sv):
    """Vicuna-7B-sized LM head (d 4096, V 32 000) over the Medusa tree (64 nodes), batch 4: the
    256-row accumulator, logits bit for bit, the tree walk against the oracle."""
    cfg = CONFIGS["medusa-tree-8k"]
    parent = gen.random_tree(cfg.tree_nodes, cfg.tree_max_depth, cfg.tree_max_children, cfg.seed)
    inp = gen.lmhead_grid_inputs(cfg.B, len(parent), 4096, cfg.vocab, cfg.seed, parent=parent)
    _stochastic_tree(sv, inp, parent, cfg.B - 1)


@pytest.mark.parametrize("N,B,d,V,take", [(20, 12, 128, 1004, True), (9, 25, 64, 4100, False), (1, 3, 64, 96, True)])
def test_stochastic_tree_shapes(sv, N, B, d, V, take):
    parent = gen.random_tree(N, 4, 3, 330 + N) if N > 1 else np.array([-1], dtype=np.int32)
    inp = gen.lmhead_grid_inputs(B, N, d, V, 331 + N, parent=parent)
    k = _stochastic_tree(sv, inp, parent, B - 2, take_logits=take)
    if N > 1:
        assert k.max() >= 1


def test_stochastic_bad_token_flagged(sv):
    """A draft token outside [0, V) in one sequence: that sequence reports -1, the others match."""
    inp = gen.lmhead_grid_inputs(4, 4, 64, 500, 340)
    inp["tokens"][2, 1] = 500
    out, _, nacc, st, lg = _stochastic(sv, sv.SPEC_SAMPLE_CHAIN, inp)
    assert st == sv.SPEC_STATUS_BAD_TOKEN
    assert nacc[2] == -1 and np.all(out[2] == -1)
    keep = [0, 1, 3]
    ref = ol.lmhead_logits(inp["hidden"], inp["weight"]).astype(np.float32)
    r_out, r_k, near = osm.spec_sample_chain(ref[keep], inp["draft_logits"][keep], inp["tokens"][keep],
                                             inp["uniforms"][keep])
    for i, b in enumerate(keep):
        if not near[i]:
            assert nacc[b] == r_k[i] and list(out[b]) == list(r_out[i])
