"""GPU parity: spec_draft_window_attn (ring-buffer draft window) against the CPU oracle."""

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


def _run(sv, q, kr, vr, pos, kn, vn, dtype, n_sinks=0):
    torch = torch_mod()
    o = torch.full(q.shape, float("nan"), dtype=torch.float32, device=q.device)
    ws = torch.empty(sv.spec_draft_window_attn_workspace(q, kr, o), dtype=torch.uint8, device=q.device)
    sv.spec_draft_window_attn(q, kr, vr, pos, o, k_new=kn, v_new=vn, workspace=ws, n_sinks=n_sinks)
    torch.cuda.synchronize()
    return to_np(o), sv.read_status(ws)


@pytest.mark.parametrize("dtype,D,Hq,Hkv", [("bf16", 128, 32, 8), ("f32", 64, 4, 1), ("bf16", 64, 8, 2),
                                            ("bf16", 128, 24, 1), ("bf16", 128, 64, 1), ("f32", 128, 8, 8)])
def test_window_with_append_many_positions(sv, dtype, D, Hq, Hkv):
    """Group sizes 4..64 cover every partial kernel: mma.sync with 8, 4 and 2 key slices per
    tile, the fp32 kernel, and the tensor-core kernel (64 rows, separate append)."""
    W = 512
    pos = np.array([1, 100, 511, 512, 513, 1800, 70000], dtype=np.int32)
    B = len(pos)
    inp = gen.window_inputs(B, Hq, Hkv, D, W, pos, dtype, seed=5 + D)
    q, kr, vr = to_dev(inp["q"], dtype), to_dev(inp["k_ring"], dtype), to_dev(inp["v_ring"], dtype)
    kn, vn = to_dev(inp["k_new"], dtype), to_dev(inp["v_new"], dtype)
    o, st = _run(sv, q, kr, vr, to_dev(pos, "i32"), kn, vn, dtype)
    ref, k_after, v_after = oa.draft_window_attn(inp["q"], inp["k_ring"], inp["v_ring"], pos,
                                                 inp["k_new"], inp["v_new"])
    assert st == 0
    assert_attn_close(o, ref, dtype, what="window")
    # the append wrote the current token's slot and nothing else
    kr_np, vr_np = to_np(kr), to_np(vr)
    for b in range(B):
        s = (pos[b] - 1) % W
        assert np.array_equal(kr_np[b, :, s], k_after[b, :, s].astype(np.float32))
        assert np.array_equal(vr_np[b, :, s], v_after[b, :, s].astype(np.float32))
        other = [t for t in oa.window_slots(int(pos[b]), W) if t != s]
        assert np.array_equal(kr_np[b][:, other], inp["k_ring"][b][:, other])
        assert np.array_equal(vr_np[b][:, other], inp["v_ring"][b][:, other])


@pytest.mark.parametrize("W", [64, 512, 1024])
def test_window_full_batch_ring_sizes(sv, W):
    """The MagicDec draft shape at its full batch (32 sequences x 8 kv heads = 256 segments, two
    per SM) for rings of one, eight and sixteen 64-key tiles, with full rings and rings still
    filling (fewer tiles than the ring holds, so some of the first copies are never consumed)."""
    Hq, Hkv, D, B = 32, 8, 128, 32
    pos = np.random.default_rng(W).integers(1, 3 * W, size=B).astype(np.int32)
    pos[:4] = [1, W - 1, W, 70000]
    inp = gen.window_inputs(B, Hq, Hkv, D, W, pos, "bf16", seed=60 + W)
    q, kr, vr = to_dev(inp["q"], "bf16"), to_dev(inp["k_ring"], "bf16"), to_dev(inp["v_ring"], "bf16")
    kn, vn = to_dev(inp["k_new"], "bf16"), to_dev(inp["v_new"], "bf16")
    o, st = _run(sv, q, kr, vr, to_dev(pos, "i32"), kn, vn, "bf16")
    ref, k_after, v_after = oa.draft_window_attn(inp["q"], inp["k_ring"], inp["v_ring"], pos,
                                                 inp["k_new"], inp["v_new"])
    assert st == 0
    assert_attn_close(o, ref, "bf16", what=f"window W={W}")
    kr_np = to_np(kr)
    for b in range(B):
        s_ = (pos[b] - 1) % W
        assert np.array_equal(kr_np[b, :, s_], k_after[b, :, s_].astype(np.float32))


@pytest.mark.parametrize("D,Hq,Hkv,W", [(64, 32, 2, 100), (128, 16, 1, 200), (128, 64, 8, 72)])
def test_window_group_sizes_and_ragged_rings(sv, D, Hq, Hkv, W):
    """The per-segment window kernel at its largest GQA group (16 rows per kv head) and rings whose
    last 64-key tile runs past the ring (W = 100, 200: the copy reads zeros there, masked), with
    filling and full rings."""
    B = 12
    pos = np.array([1, 2, 63, 64, 65, W - 1, W, W + 1, 2 * W + 3, 5000, 70001, 3 * W], dtype=np.int32)
    inp = gen.window_inputs(B, Hq, Hkv, D, W, pos, "bf16", seed=70 + W)
    q, kr, vr = to_dev(inp["q"], "bf16"), to_dev(inp["k_ring"], "bf16"), to_dev(inp["v_ring"], "bf16")
    kn, vn = to_dev(inp["k_new"], "bf16"), to_dev(inp["v_new"], "bf16")
    o, st = _run(sv, q, kr, vr, to_dev(pos, "i32"), kn, vn, "bf16")
    ref, k_after, _ = oa.draft_window_attn(inp["q"], inp["k_ring"], inp["v_ring"], pos, inp["k_new"], inp["v_new"])
    assert st == 0
    assert_attn_close(o, ref, "bf16", what=f"window G={Hq // Hkv} W={W}")
    kr_np = to_np(kr)
    for b in range(B):
        s_ = (pos[b] - 1) % W
        assert np.array_equal(kr_np[b, :, s_], k_after[b, :, s_].astype(np.float32))


def test_magicdec_draft_round_four_steps(sv):
    """Four draft steps of a round, each appending one token, on the MagicDec window shape."""
    cfg = CONFIGS["magicdec-64k"]
    B, W = 6, cfg.window
    pos0 = np.array([65536, 65537, 300, 509, 512, 1024], dtype=np.int32)
    inp = gen.window_inputs(B, cfg.Hq, cfg.Hkv, cfg.D, W, pos0, "bf16", seed=cfg.seed)
    kr, vr = to_dev(inp["k_ring"], "bf16"), to_dev(inp["v_ring"], "bf16")
    k_ring, v_ring = inp["k_ring"], inp["v_ring"]
    r = np.random.default_rng(cfg.seed)
    for step in range(cfg.draft_steps):
        pos = pos0 + step
        q = gen.store(r.standard_normal((B, cfg.Hq, cfg.D)).astype(np.float32), "bf16")
        kn = gen.store(r.standard_normal((B, cfg.Hkv, cfg.D)).astype(np.float32), "bf16")
        vn = gen.store(r.standard_normal((B, cfg.Hkv, cfg.D)).astype(np.float32), "bf16")
        o, st = _run(sv, to_dev(q, "bf16"), kr, vr, to_dev(pos, "i32"), to_dev(kn, "bf16"), to_dev(vn, "bf16"), "bf16")
        ref, k_ring, v_ring = oa.draft_window_attn(q, k_ring, v_ring, pos, kn, vn)
        assert st == 0
        assert_attn_close(o, ref, "bf16", what=f"step {step}")


def test_window_without_append_and_bad_pos(sv):
    W, D, Hq, Hkv = 64, 128, 8, 2
    pos = np.array([0, 10, 64, 200], dtype=np.int32)
    inp = gen.window_inputs(4, Hq, Hkv, D, W, np.maximum(pos, 1), "bf16", seed=9)
    # without an append the current token must already be in its slot: fill slot (pos-1) mod W
    kr, vr = inp["k_ring"].copy(), inp["v_ring"].copy()
    for b in range(4):
        if pos[b] >= 1:
            kr[b, :, (pos[b] - 1) % W] = inp["k_new"][b]
            vr[b, :, (pos[b] - 1) % W] = inp["v_new"][b]
    o, st = _run(sv, to_dev(inp["q"], "bf16"), to_dev(kr, "bf16"), to_dev(vr, "bf16"), to_dev(pos, "i32"),
                 None, None, "bf16")
    assert st & 2, "SPEC_STATUS_BAD_POS expected for pos = 0"
    assert np.all(o[0] == 0.0)
    ref, _, _ = oa.draft_window_attn(inp["q"][1:], kr[1:], vr[1:], pos[1:])
    assert_attn_close(o[1:], ref, "bf16", what="no append")


def test_window_covering_context_equals_verify(sv):
    """W >= context: the window call equals single-query chain verify over the same keys."""
    torch = torch_mod()
    W, D, Hq, Hkv = 256, 128, 16, 4
    pos = np.array([256, 97], dtype=np.int32)
    inp = gen.window_inputs(2, Hq, Hkv, D, W, pos, "bf16", seed=12)
    kr, vr = inp["k_ring"].copy(), inp["v_ring"].copy()
    for b in range(2):
        kr[b, :, pos[b] - 1] = inp["k_new"][b]
        vr[b, :, pos[b] - 1] = inp["v_new"][b]
    o_win, _ = _run(sv, to_dev(inp["q"], "bf16"), to_dev(kr, "bf16"), to_dev(vr, "bf16"), to_dev(pos, "i32"),
                    None, None, "bf16")
    q4 = to_dev(inp["q"][:, None], "bf16")
    o_ver = torch.empty(q4.shape, dtype=torch.float32, device=q4.device)
    sv.spec_verify_attn(q4, to_dev(kr, "bf16"), to_dev(vr, "bf16"), to_dev(pos, "i32"), o_ver)
    torch.cuda.synchronize()
    # two different kernels (the window's per-segment kernel, the verify split-KV kernel) over the
    # same keys: each against the oracle's verify, and against each other, at the bf16 bars
    ref = oa.verify_attn(inp["q"][:, None], kr, vr, pos)[:, 0]
    assert_attn_close(o_win, ref, "bf16", what="window kernel vs verify oracle")
    assert_attn_close(to_np(o_ver)[:, 0], ref, "bf16", what="verify kernel vs verify oracle")
    assert_attn_close(o_win, to_np(o_ver)[:, 0].astype(np.float64), "bf16", what="window vs verify kernel")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_window_long_ring_split_over_ctas(sv, dtype):
    """A ring far longer than a CTA's share (W = 6000, one kv head) is split over many CTAs and
    merged; the new key then enters through the merge.  pos = 0 marks a bad sequence."""
    W, D, Hq, Hkv = 6000, 128, 4, 1
    pos = np.array([9001, 0, 4321], dtype=np.int32)
    inp = gen.window_inputs(3, Hq, Hkv, D, W, np.maximum(pos, 1), dtype, seed=21)
    q, kr, vr = to_dev(inp["q"], dtype), to_dev(inp["k_ring"], dtype), to_dev(inp["v_ring"], dtype)
    kn, vn = to_dev(inp["k_new"], dtype), to_dev(inp["v_new"], dtype)
    o, st = _run(sv, q, kr, vr, to_dev(pos, "i32"), kn, vn, dtype)
    assert st & 2, "SPEC_STATUS_BAD_POS expected for pos = 0"
    assert np.all(o[1] == 0.0)
    keep = [0, 2]
    ref, k_after, _ = oa.draft_window_attn(inp["q"][keep], inp["k_ring"][keep], inp["v_ring"][keep], pos[keep],
                                           inp["k_new"][keep], inp["v_new"][keep])
    assert_attn_close(o[keep], ref, dtype, what="long ring")
    kr_np = to_np(kr)
    for i, b in enumerate(keep):
        s = (pos[b] - 1) % W
        assert np.array_equal(kr_np[b, :, s], k_after[i, :, s].astype(np.float32))
    # the bad sequence's ring is untouched
    assert np.array_equal(kr_np[1], inp["k_ring"][1].astype(np.float32), equal_nan=True)


@pytest.mark.parametrize("dtype,D,Hq,Hkv,W,S", [("bf16", 128, 32, 8, 512, 4), ("f32", 64, 4, 1, 96, 4),
                                                ("bf16", 128, 64, 1, 256, 4), ("bf16", 128, 32, 8, 6000, 4),
                                                ("bf16", 64, 8, 2, 64, 63)])
def test_window_with_attention_sinks(sv, dtype, D, Hq, Hkv, W, S):
    """Attention sinks: the first S tokens keep their slots, the rest cycle through W - S slots.
    Covers every kernel path (direct and split mma.sync, fp32, tensor core with separate append)
    and positions before, at and far past the window size."""
    pos = np.array([1, 3, S, S + 1, W - 1, W, W + 1, 3 * W + 5, 70001], dtype=np.int32)
    B = len(pos)
    inp = gen.window_inputs(B, Hq, Hkv, D, W, pos, dtype, seed=40 + S)
    # unwritten slots (slot >= pos while pos <= W) hold NaN; with sinks slot s holds token s then
    kr0, vr0 = inp["k_ring"], inp["v_ring"]
    q, kr, vr = to_dev(inp["q"], dtype), to_dev(kr0, dtype), to_dev(vr0, dtype)
    kn, vn = to_dev(inp["k_new"], dtype), to_dev(inp["v_new"], dtype)
    o, st = _run(sv, q, kr, vr, to_dev(pos, "i32"), kn, vn, dtype, n_sinks=S)
    ref, k_after, v_after = oa.draft_window_attn(inp["q"], kr0, vr0, pos, inp["k_new"], inp["v_new"], n_sinks=S)
    assert st == 0
    assert_attn_close(o, ref, dtype, what=f"sinks S={S} W={W}")
    kr_np = to_np(kr)
    for b in range(B):
        s_ = oa.token_slot(int(pos[b]) - 1, W, S)
        assert np.array_equal(kr_np[b, :, s_], k_after[b, :, s_].astype(np.float32))
        other = [t for t in oa.window_slots(int(pos[b]), W, S) if t != s_]
        assert np.array_equal(kr_np[b][:, other], kr0[b][:, other])


def test_sink_window_round_matches_the_shift_left_cache(sv):
    """A stream of single-token draft steps with sinks against the page's shift-left cache with the
    first tokens kept in front, on the MagicDec window shape (W = 512, 4 sinks)."""
    torch = torch_mod()
    cfg = CONFIGS["magicdec-64k"]
    W, S, T = 64, 4, 150
    Hq, Hkv, D = cfg.Hq, cfg.Hkv, cfg.D
    r = np.random.default_rng(99)
    kr = torch.zeros((1, Hkv, W, D), dtype=torch.bfloat16, device="cuda")
    vr = torch.zeros_like(kr)
    roll = oa.SinkRollCache(W, S, Hkv, D)
    for t in range(T):
        kt = gen.store(r.standard_normal((Hkv, D)).astype(np.float32), "bf16")
        vt = gen.store(r.standard_normal((Hkv, D)).astype(np.float32), "bf16")
        q = gen.store(r.standard_normal((1, Hq, D)).astype(np.float32), "bf16")
        roll.append(kt.astype(np.float64), vt.astype(np.float64))
        if t % 7 != 6 and t != T - 1:
            o, st = _run(sv, to_dev(q, "bf16"), kr, vr, to_dev(np.array([t + 1], np.int32), "i32"),
                         to_dev(kt[None], "bf16"), to_dev(vt[None], "bf16"), "bf16", n_sinks=S)
            continue
        o, st = _run(sv, to_dev(q, "bf16"), kr, vr, to_dev(np.array([t + 1], np.int32), "i32"),
                     to_dev(kt[None], "bf16"), to_dev(vt[None], "bf16"), "bf16", n_sinks=S)
        kk, vv = roll.get_kv()
        ref = np.stack([oa.attend(q[0, h].astype(np.float64), kk[h // (Hq // Hkv)], vv[h // (Hq // Hkv)],
                                  1.0 / np.sqrt(D)) for h in range(Hq)])
        assert st == 0
        assert_attn_close(o, ref[None], "bf16", what=f"step {t}")


@pytest.mark.parametrize("layout", ["v_below_k", "heads_strided"])
def test_window_ring_layouts(sv, layout):
    """Where the rings lie decides how a tile is copied: K and V of a tile in one copy when each
    ring's heads are contiguous over the batch (the lower-addressed ring's tile landing first),
    one copy per ring otherwise.  v_below_k: both rings in one allocation with V first;
    heads_strided: each ring the first Hkv heads of a buffer with three more (batch stride is not
    Hkv head strides)."""
    torch = torch_mod()
    B, Hq, Hkv, D, W = 5, 32, 8, 128, 256
    pos = np.array([1, 77, 256, 257, 9000], dtype=np.int32)
    inp = gen.window_inputs(B, Hq, Hkv, D, W, pos, "bf16", seed=41)
    if layout == "v_below_k":
        buf = torch.empty((2, B, Hkv, W, D), dtype=torch.bfloat16, device="cuda")
        buf[0].copy_(to_dev(inp["v_ring"], "bf16"))
        buf[1].copy_(to_dev(inp["k_ring"], "bf16"))
        kr, vr = buf[1], buf[0]
    else:
        kb = torch.zeros((B, Hkv + 3, W, D), dtype=torch.bfloat16, device="cuda")
        vb = torch.zeros_like(kb)
        kb[:, :Hkv].copy_(to_dev(inp["k_ring"], "bf16"))
        vb[:, :Hkv].copy_(to_dev(inp["v_ring"], "bf16"))
        kr, vr = kb[:, :Hkv], vb[:, :Hkv]
    o, st = _run(sv, to_dev(inp["q"], "bf16"), kr, vr, to_dev(pos, "i32"), to_dev(inp["k_new"], "bf16"),
                 to_dev(inp["v_new"], "bf16"), "bf16")
    ref, k_after, v_after = oa.draft_window_attn(inp["q"], inp["k_ring"], inp["v_ring"], pos, inp["k_new"],
                                                 inp["v_new"])
    assert st == 0
    assert_attn_close(o, ref, "bf16", what=layout)
    kr_np, vr_np = to_np(kr), to_np(vr)
    for b in range(B):
        s = (pos[b] - 1) % W
        assert np.array_equal(kr_np[b, :, s], k_after[b, :, s].astype(np.float32))
        assert np.array_equal(vr_np[b, :, s], v_after[b, :, s].astype(np.float32))


def test_window_status_cleared_by_the_next_call(sv):
    """The draft window kernel clears the call's status word itself (no memset before it): a call
    that flags SPEC_STATUS_BAD_POS, then a clean call on the same workspace (filled with ones
    before the first), reads 0."""
    torch = torch_mod()
    B, Hq, Hkv, D, W = 2, 32, 8, 128, 64
    pos_bad, pos_ok = np.array([0, 10], np.int32), np.array([5, 10], np.int32)
    inp = gen.window_inputs(B, Hq, Hkv, D, W, np.maximum(pos_bad, 1), "bf16", seed=43)
    q, kr, vr = to_dev(inp["q"], "bf16"), to_dev(inp["k_ring"], "bf16"), to_dev(inp["v_ring"], "bf16")
    o = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    ws = torch.full((sv.spec_draft_window_attn_workspace(q, kr, o),), 255, dtype=torch.uint8, device=q.device)
    sv.spec_draft_window_attn(q, kr, vr, to_dev(pos_bad, "i32"), o, workspace=ws)
    torch.cuda.synchronize()
    assert sv.read_status(ws) == 2
    sv.spec_draft_window_attn(q, kr, vr, to_dev(pos_ok, "i32"), o, workspace=ws)
    torch.cuda.synchronize()
    assert sv.read_status(ws) == 0
