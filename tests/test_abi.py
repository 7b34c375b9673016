"""CPU checks of the C ABI: the library builds and loads, exports every function the header
declares, agrees with the binding on struct layouts, and rejects bad arguments on the host
before any launch (no GPU needed)."""

import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from speculative_decoding_verify_attn_gb300 import build, binding
    build.build()
    return binding.lib()


def header_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            txt = open(os.path.join(inc, fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(spec_\w+)\s*\(", txt, flags=re.M):
                names.add(m.group(1))
    return sorted(names)


def test_every_declared_symbol_is_exported(L):
    names = header_functions()
    assert len(names) >= 9, names
    for n in names:
        assert hasattr(L, n), f"missing export {n}"


def test_struct_layouts_match(L):
    from speculative_decoding_verify_attn_gb300 import binding as b
    assert L.spec_abi_struct_size(0) == ctypes.sizeof(b.SpecAttnArgs)
    assert L.spec_abi_struct_size(1) == ctypes.sizeof(b.SpecWindowArgs)
    assert L.spec_abi_struct_size(2) == ctypes.sizeof(b.SpecSampleArgs)
    assert L.spec_abi_struct_size(3) == ctypes.sizeof(b.SpecCommitArgs)
    assert L.spec_abi_struct_size(4) == ctypes.sizeof(b.SpecLmheadArgs)
    assert L.spec_abi_struct_size(5) == 0
    assert L.spec_abi_version() == 6
    assert L.spec_status_string(-3).decode().startswith("workspace")


FAKE = 0x7f0000000000  # never dereferenced: validation fails before any launch


def attn_args(**kw):
    from speculative_decoding_verify_attn_gb300.binding import SpecAttnArgs
    B, Hq, Hkv, D, nq, Lmax = 2, 8, 2, 128, 5, 1024
    d = dict(B=B, Hq=Hq, Hkv=Hkv, D=D, nq=nq, q_dtype=1, kv_dtype=1, o_dtype=0,
             q=FAKE, q_stride_b=nq * Hq * D, q_stride_t=Hq * D, q_stride_h=D,
             k=FAKE, v=FAKE + (1 << 30), kv_stride_b=Hkv * Lmax * D, kv_stride_h=Lmax * D,
             Lmax=Lmax, kv_len=FAKE, tree_parent=None, scale=0.0,
             o=FAKE, o_stride_b=nq * Hq * D, o_stride_t=Hq * D, o_stride_h=D,
             workspace=FAKE, workspace_bytes=1 << 40)
    d.update(kw)
    return SpecAttnArgs(**d)


def call_attn(L, a):
    return L.spec_verify_attn(ctypes.byref(a), None)


def test_verify_attn_host_validation(L):
    assert L.spec_verify_attn_workspace(ctypes.byref(attn_args())) > 0
    assert call_attn(L, attn_args(D=96)) == -2
    assert call_attn(L, attn_args(Hq=7)) == -1
    assert call_attn(L, attn_args(B=0)) == -1
    assert call_attn(L, attn_args(q=None)) == -1
    assert call_attn(L, attn_args(kv_len=None)) == -1
    assert call_attn(L, attn_args(k=FAKE + 8)) == -1                 # bf16 TMA base not 16-byte aligned
    assert call_attn(L, attn_args(kv_stride_h=1024 * 128 + 4)) == -1  # stride not a multiple of 8
    assert call_attn(L, attn_args(q_dtype=0)) == -2                   # mixed q / kv types
    assert call_attn(L, attn_args(workspace=None)) == -3
    assert call_attn(L, attn_args(workspace_bytes=16)) == -3
    assert call_attn(L, attn_args(workspace=FAKE + 8)) == -3
    assert call_attn(L, attn_args(scale=float("nan"))) == -1
    assert call_attn(L, attn_args(Lmax=3)) == -1                      # cache smaller than nq


def test_verify_attn_append_validation(L):
    """Fused append arguments are checked before any launch (the call would otherwise launch on
    the fake pointers, so only refusals are exercised here)."""
    nq, Hkv, D = 5, 2, 128
    ok = dict(k_new=FAKE + (2 << 30), v_new=FAKE + (3 << 30), new_stride_b=nq * Hkv * D, new_stride_t=Hkv * D,
              new_stride_h=D)
    assert call_attn(L, attn_args(**dict(ok, v_new=None))) == -1              # one without the other
    assert call_attn(L, attn_args(**dict(ok, k_new=FAKE + (2 << 30) + 2))) == -1  # not 16-byte aligned
    assert call_attn(L, attn_args(**dict(ok, new_stride_t=Hkv * D + 4))) == -1  # 8-byte stride multiple
    assert call_attn(L, attn_args(**dict(ok, new_stride_h=-D))) == -1
    assert call_attn(L, attn_args(**dict(ok, kv_dtype=0, q_dtype=0, k=FAKE + 4))) == -1  # f32 cache base


def test_tree_validation(L):
    for bad in ([0, 0, 1, 2, 3], [-1, 1, 0, 1, 2], [-1, 0, 5, 1, 2], [-1, 0, -1, 1, 2]):
        arr = np.array(bad, dtype=np.int32)
        a = attn_args(tree_parent=arr.ctypes.data)
        assert call_attn(L, a) == -1, bad
    big = np.array([-1] + list(range(64)), dtype=np.int32)   # 65 nodes
    a = attn_args(nq=65, tree_parent=big.ctypes.data, Hq=2, Hkv=2)
    assert call_attn(L, a) == -2


def window_args(**kw):
    from speculative_decoding_verify_attn_gb300.binding import SpecWindowArgs
    B, Hq, Hkv, D, W = 2, 8, 2, 128, 512
    d = dict(B=B, Hq=Hq, Hkv=Hkv, D=D, W=W, q_dtype=1, kv_dtype=1, o_dtype=0,
             q=FAKE, q_stride_b=Hq * D, q_stride_h=D, k_ring=FAKE, v_ring=FAKE,
             ring_stride_b=Hkv * W * D, ring_stride_h=W * D, pos=FAKE, k_new=None, v_new=None,
             new_stride_b=0, new_stride_h=0, scale=0.0, o=FAKE, o_stride_b=Hq * D, o_stride_h=D,
             workspace=FAKE, workspace_bytes=1 << 40)
    d.update(kw)
    return SpecWindowArgs(**d)


def test_window_host_validation(L):
    call = lambda a: L.spec_draft_window_attn(ctypes.byref(a), None)  # noqa: E731
    assert L.spec_draft_window_attn_workspace(ctypes.byref(window_args())) > 0
    assert call(window_args(W=0)) == -1
    assert call(window_args(pos=None)) == -1
    assert call(window_args(k_new=FAKE)) == -1         # k_new without v_new
    assert call(window_args(workspace_bytes=0)) == -3
    assert call(window_args(n_sinks=-1)) == -1
    assert call(window_args(n_sinks=window_args().W)) == -1   # at least one ring slot


def sample_args(**kw):
    from speculative_decoding_verify_attn_gb300.binding import SpecSampleArgs
    B, g, V = 4, 4, 128256
    d = dict(mode=0, B=B, n=g, V=V, target_logits=FAKE, tl_stride_b=(g + 1) * V,
             draft_logits=FAKE, dl_stride_b=g * V, draft_tokens=FAKE, tok_stride_b=g,
             tree_parent=None, uniforms=FAKE, u_stride_b=g + 1, out_cols=g + 1,
             out_tokens=FAKE, out_num_accepted=FAKE, out_path_nodes=None,
             workspace=FAKE, workspace_bytes=1 << 40)
    d.update(kw)
    return SpecSampleArgs(**d)


def test_sample_host_validation(L):
    call = lambda a: L.spec_sample(ctypes.byref(a), None)  # noqa: E731
    assert L.spec_sample_workspace(ctypes.byref(sample_args())) > 0
    assert call(sample_args(mode=7)) == -1
    assert call(sample_args(n=0)) == -2                  # stochastic chain needs gamma >= 1
    assert call(sample_args(n=33)) == -2
    assert call(sample_args(V=1022, tl_stride_b=5 * 1022, dl_stride_b=4 * 1022)) == -2
    assert call(sample_args(target_logits=FAKE + 4)) == -1
    assert call(sample_args(draft_logits=None)) == -1
    assert call(sample_args(uniforms=None)) == -1
    assert call(sample_args(out_cols=4)) == -1
    assert call(sample_args(workspace_bytes=100)) == -3
    parent = np.array([-1, 0, 0, 1, 1, 2], dtype=np.int32)
    tree = dict(mode=2, n=6, tree_parent=parent.ctypes.data, draft_logits=None, uniforms=None)
    assert call(sample_args(**tree, out_cols=2)) == -1    # depth 2 needs 3 output columns
    bad = np.array([-1, 0, 3, 1, 1, 2], dtype=np.int32)
    assert call(sample_args(**dict(tree, tree_parent=bad.ctypes.data), out_cols=3)) == -1


def commit_args(**kw):
    from speculative_decoding_verify_attn_gb300.binding import SpecCommitArgs
    a = SpecCommitArgs(mode=1, B=2, Hkv=2, D=128, nq=8, Lmax=100, kv_dtype=1, k=FAKE, v=FAKE,
                         kv_stride_b=2 * 100 * 128, kv_stride_h=100 * 128, kv_len=FAKE, num_accepted=FAKE,
                         path_nodes=FAKE, path_stride_b=8, path_cols=5, workspace=FAKE, workspace_bytes=256)
    for key, val in kw.items():
        setattr(a, key, val)
    return a


def test_commit_host_validation(L):
    call = lambda a: L.spec_commit(ctypes.byref(a), None)  # noqa: E731
    assert L.spec_commit_workspace(ctypes.byref(commit_args())) == 256
    assert call(commit_args(mode=5)) == -1
    assert call(commit_args(kv_len=None)) == -1
    assert call(commit_args(num_accepted=None)) == -1
    assert call(commit_args(path_nodes=None)) == -1
    assert call(commit_args(path_cols=0)) == -1
    assert call(commit_args(path_stride_b=4)) == -1           # rows of path_cols = 5 entries
    assert call(commit_args(nq=65)) == -2                     # trees of at most 64 nodes
    assert call(commit_args(Lmax=7)) == -1
    assert call(commit_args(kv_stride_h=100 * 128 + 1)) == -1  # bf16 rows must stay 4-byte aligned
    assert call(commit_args(D=3)) == -1
    assert call(commit_args(workspace_bytes=255)) == -3
    # chain mode needs no K/V at all; only its own fields are validated
    assert call(commit_args(mode=0, nq=0)) == -1


def lmhead_args(**kw):
    from speculative_decoding_verify_attn_gb300.binding import SpecLmheadArgs
    a = SpecLmheadArgs(mode=1, B=8, n=4, d=4096, V=128256, out_cols=5, hidden=FAKE, weight=FAKE + (1 << 30),
                       draft_tokens=FAKE, tok_stride_b=4, tree_parent=None, out_tokens=FAKE,
                       out_num_accepted=FAKE, out_path_nodes=None, workspace=FAKE, workspace_bytes=1 << 30)
    for key, val in kw.items():
        setattr(a, key, val)
    return a


def test_lmhead_host_validation(L):
    call = lambda a: L.spec_lmhead_sample(ctypes.byref(a), None)  # noqa: E731
    ws = L.spec_lmhead_sample_workspace(ctypes.byref(lmhead_args()))
    assert ws == 256 + 8 * 5 * 8                          # status + one 64-bit key per hidden row
    assert call(lmhead_args(mode=7)) == -1
    # stochastic modes: the logits (unless the caller takes them) and the sampling workspace follow
    sto = dict(mode=0, draft_logits=FAKE, dl_stride_b=4 * 128256, uniforms=FAKE, u_stride_b=5)
    ws0 = L.spec_lmhead_sample_workspace(ctypes.byref(lmhead_args(**sto)))
    logits = 8 * 5 * 128256 * 4
    ws0_own = L.spec_lmhead_sample_workspace(ctypes.byref(lmhead_args(**sto, out_logits=FAKE)))
    assert ws0 - ws0_own == logits and ws0_own > 768
    assert call(lmhead_args(**dict(sto, draft_logits=None))) == -1
    assert call(lmhead_args(**dict(sto, draft_logits=FAKE + 4))) == -1     # 16-byte aligned
    assert call(lmhead_args(**dict(sto, dl_stride_b=4 * 128256 + 2))) == -1
    assert call(lmhead_args(**dict(sto, uniforms=None))) == -1
    assert call(lmhead_args(**sto, out_logits=FAKE + 8)) == -1
    assert call(lmhead_args(**dict(sto, n=0), out_cols=1)) == -2           # a stochastic chain drafts
    assert call(lmhead_args(**dict(sto, V=1001))) == -2                    # V % 4
    assert call(lmhead_args(**dict(sto, V=(1 << 20) + 4))) == -2
    assert L.spec_lmhead_sample_workspace(ctypes.byref(lmhead_args(**dict(sto, V=1001)))) == 0
    assert call(lmhead_args(**sto, workspace_bytes=ws0 - 1)) == -3
    ptree = np.array([-1, 0, 0, 1, 1, 2], dtype=np.int32)
    assert L.spec_lmhead_sample_workspace(ctypes.byref(lmhead_args(**dict(sto, mode=3, n=6)))) > 8 * 6 * 128256 * 4
    assert call(lmhead_args(**dict(sto, mode=3, n=6, tree_parent=ptree.ctypes.data), out_cols=2)) == -1
    assert call(lmhead_args(n=33)) == -2
    assert call(lmhead_args(B=52, n=4)) == -2              # 260 hidden rows > 256
    assert call(lmhead_args(d=4000)) == -1                 # d a multiple of 64
    assert call(lmhead_args(d=0)) == -1
    assert call(lmhead_args(V=0)) == -1
    assert call(lmhead_args(V=(1 << 24) + 1)) == -2
    assert call(lmhead_args(hidden=FAKE + 8)) == -1
    assert call(lmhead_args(weight=None)) == -1
    assert call(lmhead_args(draft_tokens=None)) == -1
    assert call(lmhead_args(out_num_accepted=None)) == -1
    assert call(lmhead_args(out_cols=4)) == -1
    assert call(lmhead_args(workspace_bytes=ws - 1)) == -3
    parent = np.array([-1, 0, 0, 1, 1, 2], dtype=np.int32)
    tree = dict(mode=2, n=6, tree_parent=parent.ctypes.data, tok_stride_b=6)
    assert call(lmhead_args(**tree, out_cols=2)) == -1     # depth 2 needs 3 output columns
    bad = np.array([-1, 0, 3, 1, 1, 2], dtype=np.int32)
    assert call(lmhead_args(**dict(tree, tree_parent=bad.ctypes.data), out_cols=3)) == -1
    assert call(lmhead_args(mode=2, n=65, tok_stride_b=65, out_cols=64)) == -2


def test_header_is_plain_c():
    """include/spec_verify.h compiles as C99 (no C++ in the boundary) and as C++17."""
    import shutil
    import subprocess
    hdr = os.path.join(ROOT, "include", "spec_verify.h")
    for cc, std, lang in (("gcc", "-std=c99", "c"), ("g++", "-std=c++17", "c++")):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} not installed")
        r = subprocess.run([cc, std, "-Wall", "-Wextra", "-pedantic", "-fsyntax-only", "-x", lang, hdr],
                           capture_output=True, text=True)
        assert r.returncode == 0 and not r.stderr, r.stderr
