"""GPU parity: spec_sample through the C ABI against the CPU oracle.

Accepted counts and emitted token ids must be bit-exact given the same uniforms, except in
sequences where the oracle reports a decision within 1e-6 of its threshold.  Those are counted and
reported separately, and their outcome must still be one the rule gives with the near decisions
taken either way.  Both the one-warp-per-sequence small-vocabulary path and the chunked
large-vocabulary path are covered, with ragged vocabulary tails and the batches the bench times.
"""

import numpy as np
import pytest
from scipy import stats
from scipy.special import softmax as sp_softmax

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


def gpu_chain(sv, inp, mode=None, diag=False):
    torch = torch_mod()
    mode = sv.SPEC_SAMPLE_CHAIN if mode is None else mode
    tl = to_dev(inp["target_logits"])
    B, rows, V = tl.shape
    dl = to_dev(inp["draft_logits"]) if mode == sv.SPEC_SAMPLE_CHAIN else None
    x = to_dev(inp["draft_tokens"], "i32")
    u = to_dev(inp["uniforms"]) if mode == sv.SPEC_SAMPLE_CHAIN else None
    out = torch.full((B, rows), -7, dtype=torch.int32, device=tl.device)
    nacc = torch.full((B,), -7, dtype=torch.int32, device=tl.device)
    ws = torch.zeros(sv.spec_sample_workspace(mode, tl), dtype=torch.uint8, device=tl.device)
    sv.spec_sample(mode, tl, out, nacc, draft_logits=dl, draft_tokens=x, uniforms=u, workspace=ws)
    torch.cuda.synchronize()
    res = (to_np(out), to_np(nacc), sv.read_status(ws))
    if diag:
        # the finish kernel's launch shape (byte 4 of the workspace): CTAs per sequence, and bit 8
        # when the draw re-reads the residual row instead of scanning kept values
        w = int(ws[4:8].view(torch.int32).item())
        res = res + ({"ctas_per_sequence": w & 0xFF, "rereads_residual": bool(w & 0x100)},)
    return res


# Sequences with a decision within 1e-6 of its threshold, as a share of a batch: with V = 128 256
# and logits of standard deviation 2 the final draw's band (1e-6 R on each side of a CDF step) holds
# about 15 % of the draws (5 of 32, 0 of 16 and 14 of 100 sequences in the bench-shaped batches);
# twice that leaves room for batch-to-batch spread and still fails a band that swallowed the draws.
MAX_NEAR_FRAC = 0.3


def compare_chain(inp, out, nacc, what, max_near_frac=MAX_NEAR_FRAC):
    """Bit-exact outside the near-threshold band; inside it (a decision within 1e-6 of its
    threshold, which fp32 kernels and the fp64 oracle may round to different sides), the outcome
    must still be one the rule gives with those decisions taken either way (oracle
    chain_outcome_valid).  Counts are printed and returned."""
    ref_out, ref_k, near = osm.spec_sample_chain(inp["target_logits"], inp["draft_logits"],
                                                 inp["draft_tokens"], inp["uniforms"])
    far = ~near
    bad_k = np.nonzero((nacc != ref_k) & far)[0]
    bad_t = np.nonzero(np.any(out != ref_out, axis=1) & far)[0]
    assert len(bad_k) == 0, f"{what}: accepted counts differ at {bad_k[:10]} ({nacc[bad_k[:5]]} vs {ref_k[bad_k[:5]]})"
    assert len(bad_t) == 0, f"{what}: tokens differ at {bad_t[:10]}"
    idx = np.nonzero(near)[0]
    if len(idx):
        ok = osm.chain_outcome_valid(inp["target_logits"][idx], inp["draft_logits"][idx], inp["draft_tokens"][idx],
                                     inp["uniforms"][idx], out[idx], nacc[idx])
        assert np.all(ok), f"{what}: near-threshold sequences {idx[~ok][:10]} have outcomes no rounding explains"
    near_match = int(np.sum(near & (nacc == ref_k) & np.all(out == ref_out, axis=1)))
    print(f"{what}: {len(near)} sequences, {int(near.sum())} near-threshold (all valid; {near_match} of them "
          f"identical to the oracle's own outcome)")
    assert near.mean() <= max_near_frac, f"{what}: {near.sum()} near-threshold sequences"
    return int(near.sum())


def test_tiny_config(sv):
    cfg = CONFIGS["tiny"]
    inp = gen.chain_sample_inputs(64, cfg.gamma, cfg.vocab, cfg.seed, cfg.target_sigma, cfg.draft_noise_sigma)
    out, nacc, st = gpu_chain(sv, inp)
    assert st == 0
    compare_chain(inp, out, nacc, "tiny")


@pytest.mark.parametrize("name,B", [("llama3-8b-layer", 8), ("magicdec-64k", 6), ("llama3-70b-layer", 5)])
def test_large_vocab_configs(sv, name, B):
    cfg = CONFIGS[name]
    inp = gen.chain_sample_inputs(B, cfg.gamma, cfg.vocab, cfg.seed, cfg.target_sigma, cfg.draft_noise_sigma,
                                  cfg.draft_corr)
    out, nacc, st = gpu_chain(sv, inp)
    assert st == 0
    compare_chain(inp, out, nacc, name)


@pytest.mark.parametrize("name,B,cs,rereads", [
    ("magicdec-64k", 32, 4, False),      # the MagicDec bench batch: 4 CTAs per sequence, values kept
    ("llama3-70b-layer", 16, 4, False),  # the 70B bench batch (gamma 6, correlated draft): sixteen
                                         # 8-CTA clusters are not all resident at once, so 4 CTAs
    ("llama3-8b-layer", 50, 2, True),    # 2 CTAs per sequence, 126 slabs each: re-reads the row
    ("llama3-8b-layer", 100, 1, True),   # more sequences than 152 / 2 SMs: one CTA per sequence,
                                         # 251 slabs, the draw re-reads the residual row
])
def test_bench_batches_full_vocab(sv, name, B, cs, rereads):
    """Stochastic chain at V = 128 256 with the batches the bench times.  The finish kernel's
    cluster size depends on B, so each case asserts which configuration it exercised."""
    cfg = CONFIGS[name]
    inp = gen.chain_sample_inputs(B, cfg.gamma, cfg.vocab, cfg.seed + B, cfg.target_sigma, cfg.draft_noise_sigma,
                                  cfg.draft_corr)
    out, nacc, st, shape = gpu_chain(sv, inp, diag=True)
    assert st == 0
    assert shape == {"ctas_per_sequence": cs, "rereads_residual": rereads}, shape
    compare_chain(inp, out, nacc, f"{name} B={B}")


@pytest.mark.parametrize("V", [2052, 5000, 8196, 40000])
def test_ragged_vocab_tails(sv, V):
    inp = gen.chain_sample_inputs(24, 3, V, 100 + V, 2.0, 1.0)
    out, nacc, st = gpu_chain(sv, inp)
    assert st == 0
    compare_chain(inp, out, nacc, f"V={V}")


@pytest.mark.parametrize("B", [3, 17, 40, 100])
def test_batch_sizes(sv, B):
    """Batches from a few sequences (eight CTAs share a sequence's vocabulary) to more sequences
    than SMs (one CTA per sequence)."""
    inp = gen.chain_sample_inputs(B, 3, 20000, 300 + B, 2.0, 1.0)
    out, nacc, st = gpu_chain(sv, inp)
    assert st == 0
    compare_chain(inp, out, nacc, f"B={B}")


@pytest.mark.parametrize("V", [16, 64, 1024, 2048])
def test_small_vocab_path(sv, V):
    inp = gen.chain_sample_inputs(3000, 4, V, 200 + V, 2.0, 0.5)
    out, nacc, st = gpu_chain(sv, inp)
    assert st == 0
    compare_chain(inp, out, nacc, f"small V={V}")


def test_chi_square_one_million_rounds_on_gpu(sv):
    """10^6 rounds on a 16-token vocabulary: bit-exact against the oracle outside the band, and the
    emitted stream of the GPU itself follows P (chi-square p > 0.01); mean tokens per round within
    4 standard errors of (1 - a^(g+1)) / (1 - a)."""
    V, gamma, n = 16, 4, 1_000_000
    rng = np.random.default_rng(2024)
    P = rng.dirichlet(np.ones(V))
    Q = 0.5 * P + 0.5 * rng.dirichlet(np.ones(V))
    tl = np.broadcast_to(np.log(P).astype(np.float32), (n, gamma + 1, V)).copy()
    dl = np.broadcast_to(np.log(Q).astype(np.float32), (n, gamma, V)).copy()
    c = np.cumsum(Q)
    c[-1] = 1.0
    x = np.searchsorted(c, rng.random((n, gamma)), side="right").astype(np.int32)
    u = rng.random((n, gamma + 1), dtype=np.float32)
    inp = dict(target_logits=tl, draft_logits=dl, draft_tokens=x, uniforms=u)
    out, nacc, st = gpu_chain(sv, inp)
    assert st == 0
    near = compare_chain(inp, out, nacc, "chi2")
    Pf = sp_softmax(tl[0, 0].astype(np.float64))
    Qf = sp_softmax(dl[0, 0].astype(np.float64))
    toks = out[out >= 0]
    counts = np.bincount(toks, minlength=V)
    _, p = stats.chisquare(counts, Pf * counts.sum())
    assert p > 0.01, p
    E = osm.expected_tokens_per_round(osm.acceptance_rate(Pf, Qf), gamma)
    emitted = nacc + 1
    assert abs(emitted.mean() - E) < 4 * emitted.std() / np.sqrt(n)
    print(f"chi2 p={p:.3f} near-threshold={near}")


def test_bad_tokens_flagged(sv):
    for V in (1024, 8192):
        inp = gen.chain_sample_inputs(4, 3, V, 5, 2.0, 1.0)
        inp["draft_tokens"][1, 2] = V
        inp["draft_tokens"][3, 0] = -1
        out, nacc, st = gpu_chain(sv, inp)
        assert st & 4
        assert nacc[1] == -1 and nacc[3] == -1 and np.all(out[1] == -1) and np.all(out[3] == -1)
        ok = [0, 2]
        ref_out, ref_k, near = osm.spec_sample_chain(inp["target_logits"][ok], inp["draft_logits"][ok],
                                                     inp["draft_tokens"][ok], inp["uniforms"][ok])
        assert np.array_equal(nacc[ok][~near], ref_k[~near])


def test_equal_rows_accept_all_and_disjoint_reject(sv):
    B, gamma, V = 500, 4, 4096
    r = np.random.default_rng(3)
    t = (2 * r.standard_normal((B, gamma + 1, V))).astype(np.float32)
    x = r.integers(V, size=(B, gamma)).astype(np.int32)
    u = r.random((B, gamma + 1), dtype=np.float32)
    inp = dict(target_logits=t, draft_logits=t[:, :gamma].copy(), draft_tokens=x, uniforms=u)
    out, nacc, _ = gpu_chain(sv, inp)
    assert np.all(nacc == gamma)
    compare_chain(inp, out, nacc, "Q == P")


@pytest.mark.parametrize("V", [1024, 128256])
def test_greedy_chain(sv, V):
    B, gamma = 16, 5
    r = np.random.default_rng(V)
    t = (2 * r.standard_normal((B, gamma + 1, V))).astype(np.float32)
    a = np.argmax(t, -1)
    x = np.where(r.random((B, gamma)) < 0.8, a[:, :gamma], r.integers(V, size=(B, gamma))).astype(np.int32)
    inp = dict(target_logits=t, draft_tokens=x)
    out, nacc, st = gpu_chain(sv, inp, mode=sv.SPEC_SAMPLE_CHAIN_GREEDY)
    ref_out, ref_k = osm.greedy_chain(t, x)
    assert st == 0
    assert np.array_equal(nacc, ref_k) and np.array_equal(out, ref_out)


@pytest.mark.parametrize("V", [1024, 5120])
def test_greedy_rows_of_all_neg_inf(sv, V):
    """A row whose logits are all -inf ties everywhere: its argmax is id 0 (ties to the smallest
    id), as in the oracle, on the one-warp path (V 1024) and the item path (V 5120); a row with -inf
    everywhere but one finite logit picks that one."""
    B, gamma = 3, 3
    r = np.random.default_rng(7)
    t = (2 * r.standard_normal((B, gamma + 1, V))).astype(np.float32)
    t[0, 0] = -np.inf                       # row 1 of sequence 0: no finite logit
    t[1, 2] = -np.inf                       # sequence 1, row 3: one finite logit, late in the row
    t[1, 2, V - 3] = -5.0
    t[2, :] = -np.inf                       # every row of sequence 2
    x = np.argmax(t[:, :gamma], -1).astype(np.int32)
    x[0, 0] = 0
    inp = dict(target_logits=t, draft_tokens=x)
    out, nacc, st = gpu_chain(sv, inp, mode=sv.SPEC_SAMPLE_CHAIN_GREEDY)
    ref_out, ref_k = osm.greedy_chain(t, x)
    assert st == 0
    assert np.array_equal(nacc, ref_k) and np.array_equal(out, ref_out)
    assert ref_k[2] == gamma and ref_out[2].tolist() == [0] * (gamma + 1)
    parent = np.array([-1, 0, 0, 1], np.int32)
    tok = np.zeros((B, 4), np.int32)
    tok[:, 1:] = r.integers(V, size=(B, 3))
    tok[2, 1] = 0
    tok[2, 3] = 0
    o, nodes, k = _gpu_tree(sv, t, tok, parent, 3)
    r_o, r_nodes, r_k = osm.tree_greedy(t, tok, parent, 3)
    assert np.array_equal(k, r_k) and np.array_equal(o, r_o) and np.array_equal(nodes, r_nodes)
    assert r_k[2] == 2


def _gpu_tree(sv, tl, tok, parent, out_cols):
    torch = torch_mod()
    tld = to_dev(tl)
    B = tl.shape[0]
    out = torch.full((B, out_cols), -7, dtype=torch.int32, device=tld.device)
    nodes = torch.full((B, out_cols), -7, dtype=torch.int32, device=tld.device)
    nacc = torch.full((B,), -7, dtype=torch.int32, device=tld.device)
    sv.spec_sample(sv.SPEC_SAMPLE_TREE_GREEDY, tld, out, nacc, draft_tokens=to_dev(tok, "i32"),
                   tree_parent=parent, out_path_nodes=nodes)
    torch.cuda.synchronize()
    return to_np(out), to_np(nodes), to_np(nacc)


def test_tree_greedy_medusa_config(sv):
    cfg = CONFIGS["medusa-tree-8k"]
    parent = gen.random_tree(cfg.tree_nodes, cfg.tree_max_depth, cfg.tree_max_children, cfg.seed)
    inp = gen.tree_sample_inputs(cfg.B, parent, cfg.vocab, cfg.seed)
    depth = osm.tree_depths(parent)
    cols = int(depth.max()) + 1
    out, nodes, nacc = _gpu_tree(sv, inp["target_logits"], inp["node_tokens"], parent, cols)
    r_out, r_nodes, r_nacc = osm.tree_greedy(inp["target_logits"], inp["node_tokens"], parent, cols)
    assert np.array_equal(nacc, r_nacc) and np.array_equal(out, r_out) and np.array_equal(nodes, r_nodes)
    assert r_nacc.max() >= 1  # the planted matches make some paths longer than zero


def test_tree_greedy_small_vocab_and_golden(sv, golden_dir):
    import json
    import os
    g = json.load(open(os.path.join(golden_dir, "tree_greedy_small.json")))
    parent = np.array(g["parent"])
    # pad V = 5 to a multiple of 4 with very low logits (they never win an argmax)
    for case in g["cases"]:
        tl = np.full((1, len(parent), 8), -1e30, np.float32)
        tl[0, :, :5] = np.array(case["logits"], np.float32)
        out, nodes, nacc = _gpu_tree(sv, tl, np.array(case["tokens"], np.int32)[None], parent, 3)
        assert out[0].tolist() == case["out_tokens"]
        assert nacc[0] == case["num_accepted"]


def test_host_validation_rejects_before_launch(sv):
    torch = torch_mod()
    tl = torch.zeros((2, 3, 1022), device="cuda")   # V % 4 != 0
    out = torch.zeros((2, 3), dtype=torch.int32, device="cuda")
    nacc = torch.zeros((2,), dtype=torch.int32, device="cuda")
    with pytest.raises(sv.SpecError) as e:
        sv.spec_sample(sv.SPEC_SAMPLE_CHAIN_GREEDY, tl, out, nacc, draft_tokens=out[:, :2])
    assert e.value.status in (sv.SPEC_ERR_UNSUPPORTED, sv.SPEC_ERR_INVALID_ARG)


def test_status_cleared_by_the_next_call(sv):
    """With V > 2048 the statistics kernel clears the call's status word itself (no memset before
    it): a call that flags SPEC_STATUS_BAD_TOKEN, then a clean call on the same workspace (filled
    with ones before the first), reads 0."""
    torch = torch_mod()
    V = 8192
    good = gen.chain_sample_inputs(4, 3, V, 5, 2.0, 1.0)
    bad = {k: v.copy() for k, v in good.items()}
    bad["draft_tokens"][1, 2] = V
    tl = to_dev(good["target_logits"])
    ws = torch.full((sv.spec_sample_workspace(sv.SPEC_SAMPLE_CHAIN, tl),), 255, dtype=torch.uint8, device=tl.device)
    out = torch.empty((4, 4), dtype=torch.int32, device=tl.device)
    nacc = torch.empty((4,), dtype=torch.int32, device=tl.device)
    for inp, want in ((bad, 4), (good, 0)):
        sv.spec_sample(sv.SPEC_SAMPLE_CHAIN, to_dev(inp["target_logits"]), out, nacc,
                       draft_logits=to_dev(inp["draft_logits"]), draft_tokens=to_dev(inp["draft_tokens"], "i32"),
                       uniforms=to_dev(inp["uniforms"]), workspace=ws)
        torch.cuda.synchronize()
        assert sv.read_status(ws) == want
