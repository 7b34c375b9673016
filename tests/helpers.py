"""Shared test utilities: moving seeded NumPy inputs to the GPU and the parity checks."""

from __future__ import annotations

import numpy as np

# Attention parity bars: bf16 K/V max-abs 2e-2, fp32 max-abs 1e-4; relative L2 alongside, because
# N(0,1) data over long contexts gives outputs small enough to make the absolute bar vacuous.
ATOL = {"bf16": 2e-2, "f32": 1e-4}
RTOL_L2 = {"bf16": 1e-2, "f32": 1e-5}


def torch_mod():
    import torch
    return torch


def dev():
    return torch_mod().device("cuda", 0)


def to_dev(x: np.ndarray, dtype: str = "f32"):
    torch = torch_mod()
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    elif dtype == "i32":
        t = t.to(torch.int32)
    return t.to(dev())


def to_np(t) -> np.ndarray:
    torch = torch_mod()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def attn_errors(o_gpu: np.ndarray, o_ref: np.ndarray):
    o_gpu = np.asarray(o_gpu, dtype=np.float64)
    diff = o_gpu - o_ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    rel_l2 = float(np.linalg.norm(diff) / max(np.linalg.norm(o_ref), 1e-30))
    return max_abs, rel_l2


def assert_attn_close(o_gpu, o_ref, kv_dtype: str, out_dtype: str = "f32", what: str = ""):
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    max_abs, rel = attn_errors(o_gpu, o_ref)
    atol = ATOL[kv_dtype]
    rtol = RTOL_L2[kv_dtype]
    if out_dtype == "bf16":
        # storing the output in bf16 adds up to half an ulp of the output itself
        atol = max(atol, 2e-2)
        rtol = max(rtol, 1e-2)
    assert max_abs <= atol, f"{what}: max-abs {max_abs:.3e} > {atol}"
    assert rel <= rtol, f"{what}: rel-L2 {rel:.3e} > {rtol}"
    return max_abs, rel
