"""GPU test of spec_verify_attn_noalloc, the verify-attention entry point for callers that cannot
allocate device memory on their hot path (an engine that gave all HBM to its KV cache and
weights at start-up, a plugin whose host framework owns every allocation, a loop that cannot
afford the device synchronisation of cudaMalloc/cudaFree).  It runs the same kernels as
spec_verify_attn with the library's fixed device scratch array in place of a caller workspace.

Its output must match spec_verify_attn's (within the attention parity tolerance) on two calls in
a row with different inputs, so that whatever the first call leaves in the shared array cannot
leak into the second.  This file sorts last so that a run stopping at the first failure has run
every other test first; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest

from workloads import gen
from workloads.configs import CONFIGS

from .helpers import assert_attn_close, to_dev, to_np, torch_mod

pytestmark = pytest.mark.gpu


def _inputs(seed, lens, tree=None):
    cfg = CONFIGS["llama3-8b-layer"]
    nq = cfg.nq if tree is None else len(tree)
    kv_len = np.array(lens, dtype=np.int32)
    inp = gen.attn_inputs(len(lens), cfg.Hq, cfg.Hkv, cfg.D, nq, kv_len, int(kv_len.max()) + 16, "bf16", seed)
    return {k_: to_dev(v_, "i32" if k_ == "kv_len" else "bf16") for k_, v_ in inp.items()}


def test_noalloc_matches_workspace_entry_on_two_calls():
    torch = torch_mod()
    import speculative_decoding_verify_attn_gb300 as sv
    tree = np.array([-1, 0, 0, 1, 2, 2, 3], dtype=np.int32)
    cases = [(_inputs(101, [1300, 2049, 640]), None), (_inputs(202, [777, 96]), tree)]
    refs = []
    for d, par in cases:
        o_ref = torch.empty(d["q"].shape, dtype=torch.float32, device=d["q"].device)
        sv.spec_verify_attn(d["q"], d["k"], d["v"], d["kv_len"], o_ref, tree_parent=par)
        refs.append(o_ref)
    torch.cuda.synchronize()
    outs = []
    for d, par in cases:   # two no-allocation calls in a row, different shapes and masks
        o = torch.full(d["q"].shape, float("nan"), dtype=torch.float32, device=d["q"].device)
        sv.spec_verify_attn_noalloc(d["q"], d["k"], d["v"], d["kv_len"], o, tree_parent=par)
        outs.append(o)
    torch.cuda.synchronize()
    for i, (o, o_ref) in enumerate(zip(outs, refs)):
        assert_attn_close(to_np(o), to_np(o_ref).astype(np.float64), "bf16", what=f"no-alloc call {i + 1}")


def test_noalloc_rejects_problems_beyond_its_scratch():
    import speculative_decoding_verify_attn_gb300 as sv
    from speculative_decoding_verify_attn_gb300.binding import SpecAttnArgs
    L = sv.lib()
    L.spec_verify_attn_noalloc.argtypes = [ctypes.POINTER(SpecAttnArgs), ctypes.c_void_p]
    L.spec_verify_attn_noalloc.restype = ctypes.c_int
    fake = 0x7f0000000000
    a = SpecAttnArgs(B=4096, Hq=64, Hkv=8, D=128, nq=7, q_dtype=1, kv_dtype=1, o_dtype=0, q=fake,
                     q_stride_b=7 * 64 * 128, q_stride_t=64 * 128, q_stride_h=128, k=fake, v=fake,
                     kv_stride_b=8 * 1024 * 128, kv_stride_h=1024 * 128, Lmax=1024, kv_len=fake,
                     o=fake, o_stride_b=7 * 64 * 128, o_stride_t=64 * 128, o_stride_h=128)
    assert L.spec_verify_attn_noalloc(ctypes.byref(a), None) == sv.binding.SPEC_ERR_SCRATCH_LIMIT
