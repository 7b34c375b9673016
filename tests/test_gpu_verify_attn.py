"""GPU parity: spec_verify_attn (chain and tree) through the C ABI against the CPU oracle.

Sizes the oracle finishes in seconds still span several 64-key tiles, several CTAs per sequence
and ragged tails; K/V slots past kv_len hold NaN; planted needles make mask leaks visible.  The
full-size workloads are checked on every (sequence, KV head) segment: the first, the last and one
middle query row, every head of the group.
"""

import numpy as np
import pytest

from oracle import attn as oa
from workloads import gen
from workloads.configs import CONFIGS

from .helpers import assert_attn_close, to_dev, to_np, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verify_attn_gb300 as sv
    sv.lib()
    return sv


def run_verify(sv, inp, kv_dtype, out_dtype="f32", tree_parent=None):
    torch = torch_mod()
    q = to_dev(inp["q"], kv_dtype)
    k = to_dev(inp["k"], kv_dtype)
    v = to_dev(inp["v"], kv_dtype)
    kv_len = to_dev(inp["kv_len"], "i32")
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16 if out_dtype == "bf16" else torch.float32,
                   device=q.device)
    ws = torch.empty(sv.spec_verify_attn_workspace(q, k, o), dtype=torch.uint8, device=q.device)
    sv.spec_verify_attn(q, k, v, kv_len, o, tree_parent=tree_parent, workspace=ws)
    torch.cuda.synchronize()
    return to_np(o), sv.read_status(ws)


def test_tiny_config_fp32(sv):
    cfg = CONFIGS["tiny"]
    kv_len = gen.kv_lengths(cfg.B, *cfg.ctx, cfg.seed)
    inp = gen.attn_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, cfg.nq, kv_len, int(kv_len.max()), "f32", cfg.seed)
    o, st = run_verify(sv, inp, "f32")
    ref = oa.verify_attn(inp["q"], inp["k"], inp["v"], kv_len)
    assert st == 0
    assert_attn_close(o, ref, "f32", what="tiny")


@pytest.mark.parametrize("name,B,lens", [
    ("llama3-8b-layer", 3, [1500, 2113, 777]),
    ("magicdec-64k", 2, [2600, 2600]),
    ("llama3-70b-layer", 2, [1900, 1023]),
])
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_chain_bf16_scaled(sv, name, B, lens, out_dtype):
    cfg = CONFIGS[name]
    kv_len = np.array(lens, dtype=np.int32)
    Lmax = int(kv_len.max()) + 37
    inp = gen.attn_inputs(B, cfg.Hq, cfg.Hkv, cfg.D, cfg.nq, kv_len, Lmax, "bf16", cfg.seed)
    inp = gen.plant_chain_needles(inp, cfg.nq, "bf16", cfg.seed)
    o, st = run_verify(sv, inp, "bf16", out_dtype)
    ref = oa.verify_attn(inp["q"], inp["k"], inp["v"], kv_len)
    assert st == 0
    assert_attn_close(o, ref, "bf16", out_dtype, what=name)


def test_tree_bf16_scaled(sv):
    cfg = CONFIGS["medusa-tree-8k"]
    parent = gen.random_tree(cfg.tree_nodes, cfg.tree_max_depth, cfg.tree_max_children, cfg.seed)
    kv_len = np.array([1100, 700], dtype=np.int32)
    inp = gen.attn_inputs(2, cfg.Hq, cfg.Hkv, cfg.D, cfg.nq, kv_len, 1200, "bf16", cfg.seed)
    inp = gen.plant_tree_needles(inp, parent, "bf16", cfg.seed)
    o, st = run_verify(sv, inp, "bf16", tree_parent=parent)
    ref = oa.verify_attn(inp["q"], inp["k"], inp["v"], kv_len, tree_parent=parent)
    assert st == 0
    assert_attn_close(o, ref, "bf16", what="tree")


@pytest.mark.parametrize("Hq,Hkv,nq,tree", [(64, 8, 20, False), (64, 8, 40, True), (32, 2, 9, True)])
def test_tensor_core_row_blocks(sv, Hq, Hkv, nq, tree):
    """More than 128 query rows per kv head (160, 320 and 144 rows: pairs of row blocks per CTA,
    one of them half empty for 320), with contexts long enough to split over many CTAs."""
    kv_len = np.array([3000, 1500], dtype=np.int32)
    parent = gen.random_tree(nq, 4, 8, 77) if tree else None
    inp = gen.attn_inputs(2, Hq, Hkv, 128, nq, kv_len, 3100, "bf16", 90 + nq)
    inp = gen.plant_tree_needles(inp, parent, "bf16", 91) if tree else gen.plant_chain_needles(inp, nq, "bf16", 91)
    o, st = run_verify(sv, inp, "bf16", tree_parent=parent)
    ref = oa.verify_attn(inp["q"], inp["k"], inp["v"], kv_len, tree_parent=parent)
    assert st == 0
    assert_attn_close(o, ref, "bf16", what=f"rows {nq * Hq // Hkv}")


@pytest.mark.parametrize("Hq,Hkv,nq,tree", [(64, 8, 32, False), (64, 8, 48, True), (32, 8, 64, True), (32, 1, 16, True)])
def test_pair_kernel_q_rows_by_tma(sv, Hq, Hkv, nq, tree):
    """Row counts that are whole multiples of 128 (256, 384, 256 and 512 rows), where the pair
    kernel takes the first part's Q rows by TMA: a chain mask, a 3-block launch whose last pair
    has one block entirely past the rows (its copy starts beyond the tensor and reads zeros), the
    Medusa shape, and G = 32 (boxes of 32 heads x 4 positions)."""
    kv_len = np.array([2900, 1400], dtype=np.int32)
    parent = gen.random_tree(nq, 5, 8, 78 + nq) if tree else None
    inp = gen.attn_inputs(2, Hq, Hkv, 128, nq, kv_len, 3000, "bf16", 95 + nq)
    inp = gen.plant_tree_needles(inp, parent, "bf16", 96) if tree else gen.plant_chain_needles(inp, nq, "bf16", 96)
    o, st = run_verify(sv, inp, "bf16", tree_parent=parent)
    ref = oa.verify_attn(inp["q"], inp["k"], inp["v"], kv_len, tree_parent=parent)
    assert st == 0
    assert_attn_close(o, ref, "bf16", what=f"rows {nq * Hq // Hkv}")


def test_chain_shaped_tree_matches_chain_on_gpu(sv):
    cfg = CONFIGS["llama3-8b-layer"]
    kv_len = np.array([640, 333], dtype=np.int32)
    inp = gen.attn_inputs(2, cfg.Hq, cfg.Hkv, cfg.D, cfg.nq, kv_len, 700, "bf16", 7)
    chain, _ = run_verify(sv, inp, "bf16")
    tree, _ = run_verify(sv, inp, "bf16", tree_parent=np.arange(-1, cfg.nq - 1))
    assert np.max(np.abs(chain - tree)) <= 1e-6


@pytest.mark.parametrize("D", [64, 128])
def test_head_dims_and_group_sizes(sv, D):
    kv_len = np.array([300, 129, 64], dtype=np.int32)
    for Hq, Hkv, nq in ((8, 8, 3), (16, 2, 2), (12, 4, 9)):
        inp = gen.attn_inputs(3, Hq, Hkv, D, nq, kv_len, 320, "bf16", 21 + Hq)
        o, st = run_verify(sv, inp, "bf16")
        ref = oa.verify_attn(inp["q"], inp["k"], inp["v"], kv_len)
        assert st == 0
        assert_attn_close(o, ref, "bf16", what=f"D{D} Hq{Hq} Hkv{Hkv} nq{nq}")


def test_fp32_tree_and_d128(sv):
    parent = np.array([-1, 0, 0, 1, 1, 2, 3, 3])
    kv_len = np.array([90, 40], dtype=np.int32)
    inp = gen.attn_inputs(2, 8, 2, 128, len(parent), kv_len, 96, "f32", 33)
    o, st = run_verify(sv, inp, "f32", tree_parent=parent)
    ref = oa.verify_attn(inp["q"], inp["k"], inp["v"], kv_len, tree_parent=parent)
    assert st == 0
    assert_attn_close(o, ref, "f32", what="fp32 tree")


def test_edge_no_context_and_bad_lengths(sv):
    # kv_len == nq (only the new tokens), and invalid lengths (< nq, > Lmax) -> zeros + status flag
    nq = 5
    kv_len = np.array([nq, 200, 3, 999], dtype=np.int32)
    Lmax = 256
    safe = np.minimum(np.maximum(kv_len, 0), Lmax)
    inp = gen.attn_inputs(4, 8, 2, 128, nq, safe, Lmax, "bf16", 44)
    inp["kv_len"] = kv_len
    o, st = run_verify(sv, inp, "bf16")
    assert st & 1, "SPEC_STATUS_BAD_KV_LEN expected"
    for b in (2, 3):
        assert np.all(o[b] == 0.0)
    for b in (0, 1):
        ref = oa.verify_attn(inp["q"][b:b + 1], inp["k"][b:b + 1], inp["v"][b:b + 1], kv_len[b:b + 1])
        assert_attn_close(o[b:b + 1], ref, "bf16", what=f"edge b{b}")


def test_single_query_single_key(sv):
    # nq = 1, kv_len = 1: the output is exactly v of the only key (bf16-exact, fp32 output)
    inp = gen.attn_inputs(1, 4, 1, 64, 1, np.array([1], np.int32), 8, "bf16", 55)
    o, _ = run_verify(sv, inp, "bf16")
    assert np.allclose(o[0, 0], np.repeat(inp["v"][0, 0, 0][None], 4, 0), atol=1e-6)


def _device_inputs(cfg, seed):
    """Full-size inputs generated on the device (seeded torch generator)."""
    torch = torch_mod()
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    kv_len = gen.kv_lengths(cfg.B, *cfg.ctx, cfg.seed)
    Lmax = int(kv_len.max())
    shape = (cfg.B, cfg.Hkv, Lmax, cfg.D)
    k = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    v = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    for b in range(cfg.B):
        k[b] = torch.randn(shape[1:], generator=g, device="cuda").to(torch.bfloat16)
        v[b] = torch.randn(shape[1:], generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn((cfg.B, cfg.nq, cfg.Hq, cfg.D), generator=g, device="cuda").to(torch.bfloat16)
    return q, k, v, kv_len


@pytest.mark.timeout(900)
@pytest.mark.parametrize("name", ["magicdec-64k", "llama3-70b-layer", "medusa-tree-8k", "llama3-8b-layer"])
def test_full_size_every_segment(sv, name):
    """The full-size workloads in the launch configuration the bench times, checked segment by
    segment: for EVERY (sequence, KV head) the first and the last query row (chain: the shortest
    and the longest causal range; tree: the root and the last node) for every query head of the
    group, and one row in between for one head, against the oracle's attention over that row's
    visible keys.
    Every stream-K part boundary of the launch lies inside some checked segment."""
    torch = torch_mod()
    cfg = CONFIGS[name]
    q, k, v, kv_len = _device_inputs(cfg, cfg.seed)
    parent = None
    if cfg.tree_nodes:
        parent = gen.random_tree(cfg.tree_nodes, cfg.tree_max_depth, cfg.tree_max_children, cfg.seed)
    o = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
    kvl = to_dev(kv_len, "i32")
    ws = torch.empty(sv.spec_verify_attn_workspace(q, k, o), dtype=torch.uint8, device="cuda")
    sv.spec_verify_attn(q, k, v, kvl, o, tree_parent=parent, workspace=ws)
    torch.cuda.synchronize()
    assert sv.read_status(ws) == 0
    rng = np.random.default_rng(cfg.seed)
    G, scale = cfg.G, 1.0 / np.sqrt(cfg.D)
    worst_abs, worst_rel, checked = 0.0, 0.0, 0
    for b in range(cfg.B):
        L = int(kv_len[b])
        rows = sorted({0, cfg.nq - 1, int(rng.integers(1, cfg.nq - 1))})
        qb = q[b].float().cpu().numpy().astype(np.float64)          # [nq, Hq, D]
        ob = o[b].cpu().numpy()
        for g in range(cfg.Hkv):
            kb = k[b, g, :L].float().cpu().numpy().astype(np.float64)
            vb = v[b, g, :L].float().cpu().numpy().astype(np.float64)
            for j in rows:
                if parent is None:   # the chain's visible set is the prefix 0 .. L - nq + j (a view)
                    n_vis = len(oa.chain_visible(L, cfg.nq, j))
                    kv_, vv_ = kb[:n_vis], vb[:n_vis]
                else:
                    vis = oa.tree_visible(L, parent, j)
                    kv_, vv_ = kb[vis], vb[vis]
                # every head of the group for the first and last rows, one for the middle row
                heads = range(g * G, (g + 1) * G) if j in (0, cfg.nq - 1) else [g * G + int(rng.integers(G))]
                for h in heads:
                    ref = oa.attend(qb[j, h], kv_, vv_, scale)
                    got = ob[j, h]
                    err = float(np.max(np.abs(got - ref)))
                    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
                    worst_abs, worst_rel = max(worst_abs, err), max(worst_rel, rel)
                    checked += 1
                    assert err <= 2e-2 and rel <= 1e-2, (name, b, g, j, h, err, rel)
    print(f"{name}: {checked} output rows checked, worst max-abs {worst_abs:.2e}, rel-L2 {worst_rel:.2e}")
    del k, v
    torch.cuda.empty_cache()


@pytest.mark.parametrize("case", ["llama3-8b-layer", "llama3-70b-layer", "medusa-tree-8k", "tiny"])
def test_fused_append(sv, case):
    """spec_verify_attn with k_new/v_new: the new tokens' rows land in the cache (bit-exact, NaN tail
    before the call), a sequence with an out-of-range kv_len is left alone and flagged, and the
    output equals the oracle's verify over the appended cache.  Covers the mma, tcgen05, pair and
    fp32 paths."""
    torch = torch_mod()
    cfg = CONFIGS[case]
    dtype = cfg.kv_dtype
    parent = gen.random_tree(cfg.tree_nodes, cfg.tree_max_depth, cfg.tree_max_children, cfg.seed) \
        if cfg.tree_nodes else None
    nq = cfg.nq
    kv_len = np.array([700, 333, nq - 1], dtype=np.int32)   # the last one is out of range
    B, Lmax = len(kv_len), 800
    inp = gen.attn_inputs(B, cfg.Hq, cfg.Hkv, cfg.D, nq, np.maximum(kv_len, nq), Lmax, dtype, cfg.seed + 3)
    rng = np.random.default_rng(cfg.seed + 4)
    k_new = gen.store(rng.standard_normal((B, nq, cfg.Hkv, cfg.D)).astype(np.float32), dtype)
    v_new = gen.store(rng.standard_normal((B, nq, cfg.Hkv, cfg.D)).astype(np.float32), dtype)
    k0, v0 = inp["k"].copy(), inp["v"].copy()
    for b in range(B):
        lo = max(int(kv_len[b]) - nq, 0)
        k0[b, :, lo:lo + nq] = np.nan                          # what the append must overwrite
        v0[b, :, lo:lo + nq] = np.nan
    dk, dv = to_dev(k0, dtype), to_dev(v0, dtype)
    q = to_dev(inp["q"], dtype)
    o = torch.full(q.shape, float("nan"), dtype=torch.float32, device=q.device)
    ws = torch.empty(sv.spec_verify_attn_workspace(q, dk, o), dtype=torch.uint8, device=q.device)
    sv.spec_verify_attn(q, dk, dv, to_dev(kv_len, "i32"), o, tree_parent=parent, workspace=ws,
                        k_new=to_dev(k_new, dtype), v_new=to_dev(v_new, dtype))
    torch.cuda.synchronize()
    k2, v2 = oa.append_new_tokens(k0, v0, kv_len, k_new, v_new)
    assert np.array_equal(to_np(dk), k2.astype(np.float32), equal_nan=True)
    assert np.array_equal(to_np(dv), v2.astype(np.float32), equal_nan=True)
    assert sv.read_status(ws) & 1                              # SPEC_STATUS_BAD_KV_LEN for b = 2
    ref = oa.verify_attn(inp["q"][:2], k2[:2], v2[:2], kv_len[:2], tree_parent=parent)
    assert_attn_close(to_np(o)[:2], ref, dtype, what=f"fused append {case}")
    assert np.all(to_np(o)[2] == 0.0)


@pytest.mark.parametrize("layout", ["bf16", "f32-offset"])
def test_tree_pair_output_layouts(sv, layout):
    """The pair kernel's merge stores 8-column row chunks with 16-byte stores where the output
    layout allows it and element stores otherwise: bf16 output, and an fp32 output view whose
    rows start 4 bytes past a 16-byte boundary (strides of a wider tensor)."""
    torch = torch_mod()
    cfg = CONFIGS["medusa-tree-8k"]
    parent = gen.random_tree(cfg.tree_nodes, cfg.tree_max_depth, cfg.tree_max_children, cfg.seed)
    kv_len = np.array([900, 611], dtype=np.int32)
    B, nq = 2, cfg.tree_nodes
    inp = gen.attn_inputs(B, cfg.Hq, cfg.Hkv, cfg.D, nq, kv_len, 1000, "bf16", cfg.seed + 9)
    q, k, v = to_dev(inp["q"], "bf16"), to_dev(inp["k"], "bf16"), to_dev(inp["v"], "bf16")
    if layout == "bf16":
        o = torch.full((B, nq, cfg.Hq, cfg.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        view = o
    else:
        o = torch.full((B, nq, cfg.Hq, cfg.D + 3), float("nan"), dtype=torch.float32, device="cuda")
        view = o[..., 1:cfg.D + 1]
    ws = torch.empty(sv.spec_verify_attn_workspace(q, k, view), dtype=torch.uint8, device="cuda")
    sv.spec_verify_attn(q, k, v, to_dev(kv_len, "i32"), view, tree_parent=parent, workspace=ws)
    torch.cuda.synchronize()
    ref = oa.verify_attn(inp["q"], inp["k"], inp["v"], kv_len, tree_parent=parent)
    assert sv.read_status(ws) == 0
    assert_attn_close(to_np(view.float()), ref, "bf16", "bf16" if layout == "bf16" else "f32", what=f"pair {layout}")
    if layout != "bf16":   # the padding columns around the view are untouched
        pad = to_np(o)[..., [0, cfg.D + 1, cfg.D + 2]]
        assert np.all(np.isnan(pad))
