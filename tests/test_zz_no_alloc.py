"""GPU test of spec_verify_attn_noalloc, the verify-attention entry point for callers that cannot
allocate device memory on their hot path (an engine that gave all HBM to its KV cache and
weights at start-up, a plugin whose host framework owns every allocation, a loop that cannot
afford the device synchronisation of cudaMalloc/cudaFree).  It runs the same kernels as
spec_verify_attn with the library's fixed device scratch array in place of a caller workspace.

Its output must match spec_verify_attn's (within the attention parity tolerance) and the CPU
oracle's on two calls in a row with different inputs, so that whatever the first call leaves in
the shared array cannot leak into the second; the outputs start as NaN, so a row the call did not
write (a sequence flagged in the status word, or a wait that ran out) fails the comparison.  A
child process then calls it in the primary context, in a second driver-API context and in the
primary context again: the scratch array has a different address in each context, so this
checks that no address is carried from one context to another.  This file sorts last so that a
run stopping at the first failure has run every other test first; it also passes on its own in
a fresh process.
"""

import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest

from oracle import attn as oa

from workloads import gen
from workloads.configs import CONFIGS

from .helpers import assert_attn_close, to_dev, to_np, torch_mod

pytestmark = pytest.mark.gpu


def _inputs(seed, lens, tree=None):
    cfg = CONFIGS["llama3-8b-layer"]
    nq = cfg.nq if tree is None else len(tree)
    kv_len = np.array(lens, dtype=np.int32)
    host = gen.attn_inputs(len(lens), cfg.Hq, cfg.Hkv, cfg.D, nq, kv_len, int(kv_len.max()) + 16, "bf16", seed)
    dev = {k_: to_dev(v_, "i32" if k_ == "kv_len" else "bf16") for k_, v_ in host.items()}
    return host, dev


def test_noalloc_matches_workspace_entry_and_oracle_on_two_calls():
    torch = torch_mod()
    import speculative_decoding_verify_attn_gb300 as sv
    tree = np.array([-1, 0, 0, 1, 2, 2, 3], dtype=np.int32)
    cases = [(_inputs(101, [1300, 2049, 640]), None), (_inputs(202, [777, 96], tree), tree)]
    refs = []
    for (_, d), par in cases:
        o_ref = torch.full(d["q"].shape, float("nan"), dtype=torch.float32, device=d["q"].device)
        sv.spec_verify_attn(d["q"], d["k"], d["v"], d["kv_len"], o_ref, tree_parent=par)
        refs.append(o_ref)
    torch.cuda.synchronize()
    outs = []
    for (_, d), par in cases:   # two no-allocation calls in a row, different shapes and masks
        o = torch.full(d["q"].shape, float("nan"), dtype=torch.float32, device=d["q"].device)
        sv.spec_verify_attn_noalloc(d["q"], d["k"], d["v"], d["kv_len"], o, tree_parent=par)
        outs.append(o)
    torch.cuda.synchronize()
    for i, (o, o_ref, ((h, _), par)) in enumerate(zip(outs, refs, cases)):
        assert_attn_close(to_np(o), to_np(o_ref).astype(np.float64), "bf16", what=f"no-alloc call {i + 1}")
        oracle = oa.verify_attn(h["q"], h["k"], h["v"], h["kv_len"], tree_parent=par)
        assert_attn_close(to_np(o), oracle, "bf16", what=f"no-alloc call {i + 1} vs oracle")


def test_noalloc_in_two_contexts_child_process():
    """Three calls in a fresh process: the primary context, a second driver-API context, the
    primary context again (tests/noalloc_context_child.py), each checked against the oracle."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "tests", "noalloc_context_child.py")], cwd=root,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().startswith("ok"), (r.returncode, r.stdout[-2000:], r.stderr[-2000:])


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
