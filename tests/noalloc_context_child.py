"""Child process of tests/test_zz_no_alloc.py: spec_verify_attn_noalloc across two CUDA contexts.

A caller that drives the GPU through the driver API may own a context of its own besides the
device's primary context, and switch between them from call to call.  The scratch array of the
no-allocation entry point then has a different device address in each context, so the library
must look the address up in the context current at each call, never reuse one from another
context.  This script makes three calls -- in the primary context, in a context it creates, and in
the primary context again -- each on inputs it uploads into that context with plain driver-API
copies, and checks every output against the oracle.  It uses no PyTorch (whose own state belongs
to the primary context) and prints one line, "ok <worst max-abs error>", on success.

Run from the repository root: python tests/noalloc_context_child.py
"""

from __future__ import annotations

import ctypes
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import attn as oa  # noqa: E402
from speculative_decoding_verify_attn_gb300.binding import SPEC_BF16, SPEC_F32, SpecAttnArgs, lib  # noqa: E402
from workloads import gen  # noqa: E402

cu = ctypes.CDLL("libcuda.so.1")


def check(r, what):
    if r != 0:
        raise RuntimeError(f"{what} failed with CUresult {r}")


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of values that are already bf16-exact (the generator rounds them)."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


class DeviceBuffers:
    """Driver-API allocations of the current context, freed together."""

    def __init__(self):
        self.ptrs = []

    def upload(self, arr: np.ndarray) -> int:
        arr = np.ascontiguousarray(arr)
        p = ctypes.c_uint64(0)
        check(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(max(arr.nbytes, 16))), "cuMemAlloc")
        check(cu.cuMemcpyHtoD_v2(p, arr.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(arr.nbytes)), "cuMemcpyHtoD")
        self.ptrs.append(p.value)
        return p.value

    def alloc(self, nbytes: int) -> int:
        return self.upload(np.zeros(nbytes, np.uint8))

    def free(self):
        for p in self.ptrs:
            cu.cuMemFree_v2(ctypes.c_uint64(p))
        self.ptrs = []


def one_call(inp, kv_len, what):
    """Uploads the inputs into the current context, runs spec_verify_attn_noalloc there on the
    legacy default stream and returns the output."""
    B, nq, Hq, D = inp["q"].shape
    Hkv, Lmax = inp["k"].shape[1], inp["k"].shape[2]
    buf = DeviceBuffers()
    try:
        q = buf.upload(bf16_bits(inp["q"]))
        k = buf.upload(bf16_bits(inp["k"]))
        v = buf.upload(bf16_bits(inp["v"]))
        kl = buf.upload(kv_len.astype(np.int32))
        o_host = np.full((B, nq, Hq, D), np.nan, np.float32)
        o = buf.upload(o_host)
        a = SpecAttnArgs(B=B, Hq=Hq, Hkv=Hkv, D=D, nq=nq, q_dtype=SPEC_BF16, kv_dtype=SPEC_BF16, o_dtype=SPEC_F32,
                         q=q, q_stride_b=nq * Hq * D, q_stride_t=Hq * D, q_stride_h=D,
                         k=k, v=v, kv_stride_b=Hkv * Lmax * D, kv_stride_h=Lmax * D, Lmax=Lmax, kv_len=kl,
                         o=o, o_stride_b=nq * Hq * D, o_stride_t=Hq * D, o_stride_h=D)
        fn = lib().spec_verify_attn_noalloc
        fn.argtypes = [ctypes.POINTER(SpecAttnArgs), ctypes.c_void_p]
        fn.restype = ctypes.c_int
        st = fn(ctypes.byref(a), None)
        if st != 0:
            raise RuntimeError(f"{what}: spec_verify_attn_noalloc returned {st}")
        check(cu.cuCtxSynchronize(), f"{what}: cuCtxSynchronize")
        check(cu.cuMemcpyDtoH_v2(o_host.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(o),
                                 ctypes.c_size_t(o_host.nbytes)), "cuMemcpyDtoH")
        return o_host
    finally:
        buf.free()


def create_context(dev) -> ctypes.c_void_p:
    ctx = ctypes.c_void_p(0)
    if hasattr(cu, "cuCtxCreate_v2"):
        check(cu.cuCtxCreate_v2(ctypes.byref(ctx), ctypes.c_uint(0), dev), "cuCtxCreate")
    else:
        params = (ctypes.c_uint64 * 4)()   # CUctxCreateParams with every field zero
        check(cu.cuCtxCreate_v4(ctypes.byref(ctx), ctypes.byref(params), ctypes.c_uint(0), dev), "cuCtxCreate")
    # the new context was made current: take it off the stack until it is used
    popped = ctypes.c_void_p(0)
    check(cu.cuCtxPopCurrent_v2(ctypes.byref(popped)), "cuCtxPopCurrent")
    return ctx


def main() -> int:
    check(cu.cuInit(0), "cuInit")
    dev = ctypes.c_int(0)
    check(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
    primary = ctypes.c_void_p(0)
    check(cu.cuDevicePrimaryCtxRetain(ctypes.byref(primary), dev), "cuDevicePrimaryCtxRetain")
    own = create_context(dev)
    worst = 0.0
    try:
        cases = []
        for seed, lens in ((11, [900, 1333]), (12, [700, 64]), (13, [1500, 257])):
            kv_len = np.array(lens, dtype=np.int32)
            inp = gen.attn_inputs(len(lens), 32, 8, 128, 5, kv_len, int(kv_len.max()) + 8, "bf16", seed)
            cases.append((inp, kv_len))
        for (inp, kv_len), ctx, what in zip(cases, (primary, own, primary),
                                            ("primary context", "second context", "primary context again")):
            check(cu.cuCtxPushCurrent_v2(ctx), "cuCtxPushCurrent")
            try:
                o = one_call(inp, kv_len, what)
            finally:
                popped = ctypes.c_void_p(0)
                check(cu.cuCtxPopCurrent_v2(ctypes.byref(popped)), "cuCtxPopCurrent")
            ref = oa.verify_attn(inp["q"], inp["k"], inp["v"], kv_len)
            if not np.all(np.isfinite(o)):
                raise AssertionError(f"{what}: output rows left unwritten")
            err = float(np.max(np.abs(o - ref)))
            rel = float(np.linalg.norm(o - ref) / np.linalg.norm(ref))
            if err > 2e-2 or rel > 1e-2:
                raise AssertionError(f"{what}: max-abs {err:.3e}, rel-L2 {rel:.3e}")
            worst = max(worst, err)
    finally:
        cu.cuCtxDestroy_v2(own)
        cu.cuDevicePrimaryCtxRelease_v2(dev)
    print(f"ok {worst:.3e}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
