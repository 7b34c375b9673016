"""GPU test of the failure path: a bounded device wait that runs out returns a status instead of
hanging.

Every device-side wait of the bf16 attention kernels (the TMA ring's mbarriers, the tensor-core
hand-offs) gives up after about one second, sets SPEC_STATUS_TIMEOUT in the status word, stops
issuing work, waits (again bounded) for its own copies and MMAs in flight, frees its tensor memory
and returns.  The test hook SPEC_DEBUG_NO_LOADS makes the producers issue no copies at all, so the
first wait of every CTA runs out while nothing asynchronous is in flight: no fault, no trap and no
hang, only the status.  The next normal call on the same workspace must then be correct, which
shows the context and the workspace are still usable.

One case per kernel family: mma.sync (<= 32 query rows per KV head), tcgen05 (33-128 rows) and
the tcgen05 pair kernel (> 128 rows, a token tree).
"""

import time

import numpy as np
import pytest

from oracle import attn as oa
from workloads import gen

from .helpers import assert_attn_close, to_dev, to_np, torch_mod

pytestmark = [pytest.mark.gpu, pytest.mark.timeout(300)]

CASES = {
    # name: (Hq, Hkv, nq, tree, lens)
    "mma-chain": (32, 8, 5, False, [1500, 777]),
    "tcgen05-chain": (64, 8, 7, False, [1900, 1023]),
    "tcgen05-pair-tree": (32, 8, 64, True, [1100, 700]),
}


@pytest.mark.parametrize("case", list(CASES))
def test_wait_runs_out_then_next_call_is_correct(case):
    torch = torch_mod()
    import speculative_decoding_verify_attn_gb300 as sv
    Hq, Hkv, nq, tree, lens = CASES[case]
    parent = gen.random_tree(nq, 4, 8, 5) if tree else None
    kv_len = np.array(lens, dtype=np.int32)
    inp = gen.attn_inputs(len(lens), Hq, Hkv, 128, nq, kv_len, int(kv_len.max()) + 16, "bf16", 300 + nq)
    q, k, v = to_dev(inp["q"], "bf16"), to_dev(inp["k"], "bf16"), to_dev(inp["v"], "bf16")
    kvl = to_dev(kv_len, "i32")
    o = torch.full(q.shape, float("nan"), dtype=torch.float32, device=q.device)
    ws = torch.empty(sv.spec_verify_attn_workspace(q, k, o), dtype=torch.uint8, device=q.device)

    torch.cuda.synchronize()
    t0 = time.perf_counter()
    sv.spec_verify_attn(q, k, v, kvl, o, tree_parent=parent, workspace=ws, debug_flags=sv.SPEC_DEBUG_NO_LOADS)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    st = sv.read_status(ws)
    assert st & sv.SPEC_STATUS_TIMEOUT, f"{case}: status {st} after a call whose waits had to run out"
    # the limit is ~1 s per wait; every CTA gives up on its first one
    assert 0.5 < waited < 60.0, f"{case}: the failing call took {waited:.2f} s"

    o.fill_(float("nan"))
    sv.spec_verify_attn(q, k, v, kvl, o, tree_parent=parent, workspace=ws)
    torch.cuda.synchronize()
    assert sv.read_status(ws) == 0
    ref = oa.verify_attn(inp["q"], inp["k"], inp["v"], kv_len, tree_parent=parent)
    assert_attn_close(to_np(o), ref, "bf16", what=f"{case} after the timed-out call")
    print(f"{case}: timed-out call returned after {waited:.2f} s with status {st}")


def test_unknown_debug_flag_rejected_before_launch():
    torch = torch_mod()
    import speculative_decoding_verify_attn_gb300 as sv
    inp = gen.attn_inputs(1, 8, 2, 128, 2, np.array([64], np.int32), 64, "bf16", 1)
    q, k, v = to_dev(inp["q"], "bf16"), to_dev(inp["k"], "bf16"), to_dev(inp["v"], "bf16")
    o = torch.zeros(q.shape, dtype=torch.float32, device=q.device)
    with pytest.raises(sv.SpecError) as e:
        sv.spec_verify_attn(q, k, v, to_dev(inp["kv_len"], "i32"), o, debug_flags=2)
    assert e.value.status == sv.SPEC_ERR_INVALID_ARG
