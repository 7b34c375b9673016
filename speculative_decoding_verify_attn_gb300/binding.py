"""Thin ctypes binding of libspecverify (include/spec_verify.h).

Same names as the C ABI; each function only marshals torch tensors into the argument struct
and calls the library.  Every step of the computation runs in the library's CUDA kernels.  There
is no fallback: if the shared library is missing or fails to load, every call raises.

Build the library first with ``python -m speculative_decoding_verify_attn_gb300.build`` (or
``__graft_entry__.build()``).
"""

from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, Structure, byref, c_float, c_int, c_int32, c_int64, c_size_t, c_void_p
from typing import Optional, Sequence

import numpy as np

from .build import LIBPATH

SPEC_OK = 0
SPEC_ERR_INVALID_ARG = -1
SPEC_ERR_UNSUPPORTED = -2
SPEC_ERR_WORKSPACE = -3
SPEC_ERR_CUDA = -4

SPEC_F32 = 0
SPEC_BF16 = 1

SPEC_STATUS_BAD_KV_LEN = 1
SPEC_STATUS_BAD_POS = 2
SPEC_STATUS_BAD_TOKEN = 4
SPEC_STATUS_TIMEOUT = 8

SPEC_DEBUG_NO_LOADS = 1

SPEC_COMMIT_CHAIN = 0
SPEC_COMMIT_TREE = 1
SPEC_SAMPLE_CHAIN = 0
SPEC_SAMPLE_CHAIN_GREEDY = 1
SPEC_SAMPLE_TREE_GREEDY = 2
SPEC_SAMPLE_TREE = 3


class SpecAttnArgs(Structure):
    _fields_ = [
        ("B", c_int32), ("Hq", c_int32), ("Hkv", c_int32), ("D", c_int32), ("nq", c_int32),
        ("q_dtype", c_int32), ("kv_dtype", c_int32), ("o_dtype", c_int32),
        ("q", c_void_p), ("q_stride_b", c_int64), ("q_stride_t", c_int64), ("q_stride_h", c_int64),
        ("k", c_void_p), ("v", c_void_p), ("kv_stride_b", c_int64), ("kv_stride_h", c_int64),
        ("Lmax", c_int32), ("reserved0", c_int32),
        ("kv_len", c_void_p), ("tree_parent", c_void_p),
        ("scale", c_float), ("debug_flags", c_int32),
        ("o", c_void_p), ("o_stride_b", c_int64), ("o_stride_t", c_int64), ("o_stride_h", c_int64),
        ("workspace", c_void_p), ("workspace_bytes", c_size_t),
        ("k_new", c_void_p), ("v_new", c_void_p),
        ("new_stride_b", c_int64), ("new_stride_t", c_int64), ("new_stride_h", c_int64),
    ]


class SpecWindowArgs(Structure):
    _fields_ = [
        ("B", c_int32), ("Hq", c_int32), ("Hkv", c_int32), ("D", c_int32), ("W", c_int32),
        ("q_dtype", c_int32), ("kv_dtype", c_int32), ("o_dtype", c_int32),
        ("q", c_void_p), ("q_stride_b", c_int64), ("q_stride_h", c_int64),
        ("k_ring", c_void_p), ("v_ring", c_void_p), ("ring_stride_b", c_int64), ("ring_stride_h", c_int64),
        ("pos", c_void_p),
        ("k_new", c_void_p), ("v_new", c_void_p), ("new_stride_b", c_int64), ("new_stride_h", c_int64),
        ("scale", c_float), ("n_sinks", c_int32),
        ("o", c_void_p), ("o_stride_b", c_int64), ("o_stride_h", c_int64),
        ("workspace", c_void_p), ("workspace_bytes", c_size_t),
    ]


class SpecCommitArgs(Structure):
    _fields_ = [
        ("mode", c_int32), ("B", c_int32), ("Hkv", c_int32), ("D", c_int32), ("nq", c_int32), ("Lmax", c_int32),
        ("kv_dtype", c_int32), ("path_cols", c_int32),
        ("k", c_void_p), ("v", c_void_p), ("kv_stride_b", c_int64), ("kv_stride_h", c_int64),
        ("kv_len", c_void_p), ("num_accepted", c_void_p), ("path_nodes", c_void_p), ("path_stride_b", c_int64),
        ("workspace", c_void_p), ("workspace_bytes", c_size_t),
    ]


class SpecSampleArgs(Structure):
    _fields_ = [
        ("mode", c_int32), ("B", c_int32), ("n", c_int32), ("V", c_int32),
        ("target_logits", c_void_p), ("tl_stride_b", c_int64),
        ("draft_logits", c_void_p), ("dl_stride_b", c_int64),
        ("draft_tokens", c_void_p), ("tok_stride_b", c_int64),
        ("tree_parent", c_void_p),
        ("uniforms", c_void_p), ("u_stride_b", c_int64),
        ("out_cols", c_int32), ("reserved0", c_int32),
        ("out_tokens", c_void_p), ("out_num_accepted", c_void_p), ("out_path_nodes", c_void_p),
        ("workspace", c_void_p), ("workspace_bytes", c_size_t),
    ]


class SpecLmheadArgs(Structure):
    _fields_ = [
        ("mode", c_int32), ("B", c_int32), ("n", c_int32), ("d", c_int32), ("V", c_int32),
        ("out_cols", c_int32),
        ("hidden", c_void_p), ("weight", c_void_p),
        ("draft_tokens", c_void_p), ("tok_stride_b", c_int64),
        ("tree_parent", c_void_p),
        ("out_tokens", c_void_p), ("out_num_accepted", c_void_p), ("out_path_nodes", c_void_p),
        ("workspace", c_void_p), ("workspace_bytes", c_size_t),
        ("draft_logits", c_void_p), ("dl_stride_b", c_int64),
        ("uniforms", c_void_p), ("u_stride_b", c_int64),
        ("out_logits", c_void_p),
    ]


class SpecError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {spec_status_string(status)} ({status})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (loaded once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIBPATH):
        raise RuntimeError(f"libspecverify is not built ({LIBPATH} missing); run "
                           "`python -m speculative_decoding_verify_attn_gb300.build`")
    L = ctypes.CDLL(LIBPATH)
    L.spec_verify_attn_workspace.argtypes = [POINTER(SpecAttnArgs)]
    L.spec_verify_attn_workspace.restype = c_size_t
    L.spec_verify_attn.argtypes = [POINTER(SpecAttnArgs), c_void_p]
    L.spec_verify_attn.restype = c_int
    L.spec_draft_window_attn_workspace.argtypes = [POINTER(SpecWindowArgs)]
    L.spec_draft_window_attn_workspace.restype = c_size_t
    L.spec_draft_window_attn.argtypes = [POINTER(SpecWindowArgs), c_void_p]
    L.spec_draft_window_attn.restype = c_int
    L.spec_sample_workspace.argtypes = [POINTER(SpecSampleArgs)]
    L.spec_sample_workspace.restype = c_size_t
    L.spec_sample.argtypes = [POINTER(SpecSampleArgs), c_void_p]
    L.spec_sample.restype = c_int
    L.spec_lmhead_sample_workspace.argtypes = [POINTER(SpecLmheadArgs)]
    L.spec_lmhead_sample_workspace.restype = c_size_t
    L.spec_lmhead_sample.argtypes = [POINTER(SpecLmheadArgs), c_void_p]
    L.spec_lmhead_sample.restype = c_int
    L.spec_commit_workspace.argtypes = [POINTER(SpecCommitArgs)]
    L.spec_commit_workspace.restype = c_size_t
    L.spec_commit.argtypes = [POINTER(SpecCommitArgs), c_void_p]
    L.spec_commit.restype = c_int
    L.spec_status_string.argtypes = [c_int]
    L.spec_status_string.restype = ctypes.c_char_p
    L.spec_abi_version.argtypes = []
    L.spec_abi_version.restype = c_int
    L.spec_abi_struct_size.argtypes = [c_int]
    L.spec_abi_struct_size.restype = c_size_t
    for i, cls in enumerate((SpecAttnArgs, SpecWindowArgs, SpecSampleArgs, SpecCommitArgs, SpecLmheadArgs)):
        if L.spec_abi_struct_size(i) != ctypes.sizeof(cls):
            raise RuntimeError(f"ABI mismatch for {cls.__name__}: library {L.spec_abi_struct_size(i)} "
                               f"bytes, binding {ctypes.sizeof(cls)}")
    _lib = L
    return L


def spec_status_string(status: int) -> str:
    return lib().spec_status_string(status).decode()


def spec_abi_version() -> int:
    return lib().spec_abi_version()


# ---------------------------------------------------------------------------- helpers
def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return SPEC_F32
    if t.dtype == torch.bfloat16:
        return SPEC_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (host buffers: copy them to the device first)")
        if t is not None and t.stride(-1) != 1:
            raise ValueError("innermost dimension must be contiguous")


def _stream_handle(stream) -> Optional[int]:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream if hasattr(s, "cuda_stream") else int(s)


def _workspace(nbytes: int, device, workspace):
    torch = _torch()
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace too small: need {nbytes} bytes")
        return workspace
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def _host_i32(seq: Optional[Sequence[int]]):
    if seq is None:
        return None, None
    arr = np.ascontiguousarray(np.asarray(seq, dtype=np.int32))
    return arr, arr.ctypes.data


# ---------------------------------------------------------------------------- attention
def verify_attn_args(q, k, v, kv_len, o, tree_parent=None, scale: float = 0.0, workspace=None,
                     k_new=None, v_new=None, debug_flags: int = 0):
    """Fill SpecAttnArgs from tensors (k_new, v_new [B, nq, Hkv, D] for the fused append, or
    None).  Returns (args, keepalive)."""
    B, nq, Hq, D = q.shape
    Hkv, Lmax = k.shape[1], k.shape[2]
    if k.stride(2) != D or v.stride(2) != D or tuple(k.stride()) != tuple(v.stride()):
        raise ValueError("K and V must share strides with token stride == head_dim")
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if k_new is not None:
        if tuple(k_new.shape) != (B, nq, Hkv, D) or tuple(k_new.stride()) != tuple(v_new.stride()):
            raise ValueError("k_new, v_new must be [B, nq, Hkv, D] with equal strides")
        if k_new.stride(3) != 1 or k_new.dtype != k.dtype or v_new.dtype != k.dtype:
            raise ValueError("k_new, v_new: innermost dim contiguous, cache dtype")
    parent_arr, parent_ptr = _host_i32(tree_parent)
    a = SpecAttnArgs(
        B=B, Hq=Hq, Hkv=Hkv, D=D, nq=nq,
        q_dtype=_dtype_code(q), kv_dtype=_dtype_code(k), o_dtype=_dtype_code(o),
        q=_ptr(q), q_stride_b=q.stride(0), q_stride_t=q.stride(1), q_stride_h=q.stride(2),
        k=_ptr(k), v=_ptr(v), kv_stride_b=k.stride(0), kv_stride_h=k.stride(1),
        Lmax=Lmax, kv_len=_ptr(kv_len), tree_parent=parent_ptr, scale=scale, debug_flags=debug_flags,
        o=_ptr(o), o_stride_b=o.stride(0), o_stride_t=o.stride(1), o_stride_h=o.stride(2),
        workspace=_ptr(workspace), workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size(),
    )
    if k_new is not None:
        a.k_new, a.v_new = _ptr(k_new), _ptr(v_new)
        a.new_stride_b, a.new_stride_t, a.new_stride_h = k_new.stride(0), k_new.stride(1), k_new.stride(2)
    return a, parent_arr


def spec_verify_attn_workspace(q, k, o, nq: Optional[int] = None) -> int:
    B, nq_, Hq, D = q.shape
    a = SpecAttnArgs(B=B, Hq=Hq, Hkv=k.shape[1], D=D, nq=nq or nq_, q_dtype=_dtype_code(q),
                     kv_dtype=_dtype_code(k), o_dtype=_dtype_code(o), Lmax=k.shape[2])
    return lib().spec_verify_attn_workspace(byref(a))


def spec_verify_attn(q, k, v, kv_len, o, *, tree_parent=None, scale: float = 0.0, workspace=None, stream=None,
                     k_new=None, v_new=None, debug_flags: int = 0):
    """Verify attention (chain if tree_parent is None, else tree; tree_parent is host data).

    q [B, nq, Hq, D]; k, v [B, Hkv, Lmax, D]; kv_len [B] int32 (device); o [B, nq, Hq, D].
    With k_new, v_new [B, nq, Hkv, D] the call first writes them into cache positions
    kv_len - nq .. kv_len - 1 (fused append).  debug_flags: SPEC_DEBUG_* test hooks (0 in normal
    use).  Writes o and returns it."""
    _check_cuda(q, k, v, kv_len, o)
    if k_new is not None:
        _check_cuda(k_new, v_new)
    need = spec_verify_attn_workspace(q, k, o)
    if need == 0:
        raise SpecError(SPEC_ERR_INVALID_ARG, "spec_verify_attn_workspace")
    ws = _workspace(need, q.device, workspace)
    a, keep = verify_attn_args(q, k, v, kv_len, o, tree_parent, scale, ws, k_new, v_new, debug_flags)
    st = lib().spec_verify_attn(byref(a), _stream_handle(stream))
    del keep
    if st != SPEC_OK:
        raise SpecError(st, "spec_verify_attn")
    return o


def window_attn_args(q, k_ring, v_ring, pos, o, k_new=None, v_new=None, scale: float = 0.0, workspace=None,
                     n_sinks: int = 0):
    B, Hq, D = q.shape
    Hkv, W = k_ring.shape[1], k_ring.shape[2]
    if k_ring.stride(2) != D or tuple(k_ring.stride()) != tuple(v_ring.stride()):
        raise ValueError("rings must share strides with token stride == head_dim")
    if k_new is not None and tuple(k_new.stride()) != tuple(v_new.stride()):
        raise ValueError("k_new and v_new must share strides")
    return SpecWindowArgs(
        B=B, Hq=Hq, Hkv=Hkv, D=D, W=W,
        q_dtype=_dtype_code(q), kv_dtype=_dtype_code(k_ring), o_dtype=_dtype_code(o),
        q=_ptr(q), q_stride_b=q.stride(0), q_stride_h=q.stride(1),
        k_ring=_ptr(k_ring), v_ring=_ptr(v_ring), ring_stride_b=k_ring.stride(0), ring_stride_h=k_ring.stride(1),
        pos=_ptr(pos),
        k_new=_ptr(k_new), v_new=_ptr(v_new),
        new_stride_b=0 if k_new is None else k_new.stride(0), new_stride_h=0 if k_new is None else k_new.stride(1),
        scale=scale, n_sinks=n_sinks,
        o=_ptr(o), o_stride_b=o.stride(0), o_stride_h=o.stride(1),
        workspace=_ptr(workspace), workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size(),
    )


def spec_draft_window_attn_workspace(q, k_ring, o) -> int:
    B, Hq, D = q.shape
    a = SpecWindowArgs(B=B, Hq=Hq, Hkv=k_ring.shape[1], D=D, W=k_ring.shape[2], q_dtype=_dtype_code(q),
                       kv_dtype=_dtype_code(k_ring), o_dtype=_dtype_code(o))
    return lib().spec_draft_window_attn_workspace(byref(a))


def spec_draft_window_attn(q, k_ring, v_ring, pos, o, *, k_new=None, v_new=None, scale: float = 0.0,
                           workspace=None, stream=None, n_sinks: int = 0):
    """Draft single-query attention over the ring window (appending k_new/v_new first if given).

    q [B, Hq, D]; k_ring, v_ring [B, Hkv, W, D] (updated in place when k_new is given);
    pos [B] int32 (device); o [B, Hq, D]; n_sinks attention-sink slots at the ring's front."""
    _check_cuda(q, k_ring, v_ring, pos, o, k_new, v_new)
    need = spec_draft_window_attn_workspace(q, k_ring, o)
    if need == 0:
        raise SpecError(SPEC_ERR_INVALID_ARG, "spec_draft_window_attn_workspace")
    ws = _workspace(need, q.device, workspace)
    a = window_attn_args(q, k_ring, v_ring, pos, o, k_new, v_new, scale, ws, n_sinks)
    st = lib().spec_draft_window_attn(byref(a), _stream_handle(stream))
    if st != SPEC_OK:
        raise SpecError(st, "spec_draft_window_attn")
    return o


# ---------------------------------------------------------------------------- sampling
def sample_args(mode, target_logits, out_tokens, out_num_accepted, *, draft_logits=None, draft_tokens=None,
                uniforms=None, tree_parent=None, out_path_nodes=None, workspace=None):
    B, rows, V = target_logits.shape
    n = rows if mode in (SPEC_SAMPLE_TREE_GREEDY, SPEC_SAMPLE_TREE) else rows - 1
    parent_arr, parent_ptr = _host_i32(tree_parent)
    for t in (target_logits, draft_logits):
        if t is not None and t.stride(1) != V:
            raise ValueError("logit rows must be contiguous with row stride V")
    a = SpecSampleArgs(
        mode=mode, B=B, n=n, V=V,
        target_logits=_ptr(target_logits), tl_stride_b=target_logits.stride(0),
        draft_logits=_ptr(draft_logits), dl_stride_b=0 if draft_logits is None else draft_logits.stride(0),
        draft_tokens=_ptr(draft_tokens), tok_stride_b=0 if draft_tokens is None else draft_tokens.stride(0),
        tree_parent=parent_ptr,
        uniforms=_ptr(uniforms), u_stride_b=0 if uniforms is None else uniforms.stride(0),
        out_cols=out_tokens.shape[1],
        out_tokens=_ptr(out_tokens), out_num_accepted=_ptr(out_num_accepted), out_path_nodes=_ptr(out_path_nodes),
        workspace=_ptr(workspace), workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size(),
    )
    return a, parent_arr


def spec_sample_workspace(mode, target_logits, tree_parent=None) -> int:
    B, rows, V = target_logits.shape
    n = rows if mode in (SPEC_SAMPLE_TREE_GREEDY, SPEC_SAMPLE_TREE) else rows - 1
    a = SpecSampleArgs(mode=mode, B=B, n=n, V=V)
    return lib().spec_sample_workspace(byref(a))


def spec_sample(mode, target_logits, out_tokens, out_num_accepted, *, draft_logits=None, draft_tokens=None,
                uniforms=None, tree_parent=None, out_path_nodes=None, workspace=None, stream=None):
    """Speculative sampling (SPEC_SAMPLE_CHAIN), greedy chain, greedy tree or stochastic tree
    (SPEC_SAMPLE_TREE) selection.

    target_logits [B, gamma+1 | N, V] fp32; draft_logits [B, gamma | N, V] fp32 (stochastic);
    draft_tokens [B, gamma] or node tokens [B, N] int32; uniforms [B, gamma+1 | N] fp32 (stochastic);
    tree_parent host [N] (tree); out_tokens [B, out_cols] int32; out_num_accepted [B] int32."""
    _check_cuda(target_logits, draft_logits, draft_tokens, uniforms, out_tokens, out_num_accepted, out_path_nodes)
    need = spec_sample_workspace(mode, target_logits, tree_parent)
    if need == 0:
        raise SpecError(SPEC_ERR_INVALID_ARG, "spec_sample_workspace")
    ws = _workspace(need, target_logits.device, workspace)
    a, keep = sample_args(mode, target_logits, out_tokens, out_num_accepted, draft_logits=draft_logits,
                          draft_tokens=draft_tokens, uniforms=uniforms, tree_parent=tree_parent,
                          out_path_nodes=out_path_nodes, workspace=ws)
    st = lib().spec_sample(byref(a), _stream_handle(stream))
    del keep
    if st != SPEC_OK:
        raise SpecError(st, "spec_sample")
    return out_tokens, out_num_accepted


def lmhead_args(mode, hidden, weight, out_tokens, out_num_accepted, *, draft_tokens=None, tree_parent=None,
                out_path_nodes=None, workspace=None, draft_logits=None, uniforms=None, out_logits=None):
    B, rows, d = hidden.shape
    V = weight.shape[0]
    n = rows if mode in (SPEC_SAMPLE_TREE_GREEDY, SPEC_SAMPLE_TREE) else rows - 1
    if not hidden.is_contiguous() or not weight.is_contiguous():
        raise ValueError("hidden [B, R, d] and weight [V, d] must be contiguous")
    if weight.shape[1] != d:
        raise ValueError("weight must be [V, d] with the hidden size d")
    parent_arr, parent_ptr = _host_i32(tree_parent)
    a = SpecLmheadArgs(
        mode=mode, B=B, n=n, d=d, V=V, out_cols=out_tokens.shape[1],
        hidden=_ptr(hidden), weight=_ptr(weight),
        draft_tokens=_ptr(draft_tokens), tok_stride_b=0 if draft_tokens is None else draft_tokens.stride(0),
        tree_parent=parent_ptr,
        out_tokens=_ptr(out_tokens), out_num_accepted=_ptr(out_num_accepted), out_path_nodes=_ptr(out_path_nodes),
        workspace=_ptr(workspace), workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size(),
        draft_logits=_ptr(draft_logits), dl_stride_b=0 if draft_logits is None else draft_logits.stride(0),
        uniforms=_ptr(uniforms), u_stride_b=0 if uniforms is None else uniforms.stride(0),
        out_logits=_ptr(out_logits),
    )
    return a, parent_arr


def spec_lmhead_sample_workspace(mode, hidden, weight, out_logits=None) -> int:
    B, rows, d = hidden.shape
    n = rows if mode in (SPEC_SAMPLE_TREE_GREEDY, SPEC_SAMPLE_TREE) else rows - 1
    a = SpecLmheadArgs(mode=mode, B=B, n=n, d=d, V=weight.shape[0], out_logits=_ptr(out_logits))
    return lib().spec_lmhead_sample_workspace(byref(a))


def spec_lmhead_sample(mode, hidden, weight, out_tokens, out_num_accepted, *, draft_tokens=None, tree_parent=None,
                       out_path_nodes=None, workspace=None, stream=None, draft_logits=None, uniforms=None,
                       out_logits=None):
    """The LM-head projection fused with verification.  Greedy modes (SPEC_SAMPLE_CHAIN_GREEDY,
    SPEC_SAMPLE_TREE_GREEDY): each row's logits hidden @ weight^T reduced to its argmax on the GPU,
    then the greedy rule.  Stochastic modes (SPEC_SAMPLE_CHAIN, SPEC_SAMPLE_TREE): the GEMM writes
    the fp32 logits (into out_logits if given, else the workspace) and spec_sample's kernels run on
    them in the same call.

    hidden [B, gamma+1 | N, d] bf16; weight [V, d] bf16; draft_tokens [B, gamma] or node tokens
    [B, N] int32; tree_parent host [N] (tree); out_tokens [B, out_cols] int32;
    out_num_accepted [B] int32; stochastic: draft_logits [B, gamma | N, V] fp32, uniforms
    [B, gamma+1 | N] fp32, out_logits [B, gamma+1 | N, V] fp32 (optional)."""
    _check_cuda(hidden, weight, draft_tokens, out_tokens, out_num_accepted, out_path_nodes, draft_logits, uniforms,
                out_logits)
    need = spec_lmhead_sample_workspace(mode, hidden, weight, out_logits)
    if need == 0:
        raise SpecError(SPEC_ERR_INVALID_ARG, "spec_lmhead_sample_workspace")
    ws = _workspace(need, hidden.device, workspace)
    a, keep = lmhead_args(mode, hidden, weight, out_tokens, out_num_accepted, draft_tokens=draft_tokens,
                          tree_parent=tree_parent, out_path_nodes=out_path_nodes, workspace=ws,
                          draft_logits=draft_logits, uniforms=uniforms, out_logits=out_logits)
    st = lib().spec_lmhead_sample(byref(a), _stream_handle(stream))
    del keep
    if st != SPEC_OK:
        raise SpecError(st, "spec_lmhead_sample")
    return out_tokens, out_num_accepted


def read_status(workspace) -> int:
    """The device status word (first 4 bytes of a workspace) after the stream is synchronized."""
    return int(workspace[:4].view(_torch().int32).item())


# ---------------------------------------------------------------------------- no-allocation verify
SPEC_ERR_SCRATCH_LIMIT = -6
_noalloc_fn = None


def spec_verify_attn_noalloc(q, k, v, kv_len, o, *, tree_parent=None, scale: float = 0.0, stream=None):
    """spec_verify_attn for callers that cannot allocate device memory: the library uses its own
    fixed 64 MiB device scratch array instead of a caller workspace, and nothing here allocates
    (no torch workspace either).  Calls on one device share that array, so calls whose kernels
    overlap on the GPU must not be issued; the first call in a context must precede any stream
    capture.  Writes o and returns it."""
    global _noalloc_fn
    _check_cuda(q, k, v, kv_len, o)
    if _noalloc_fn is None:
        fn = lib().spec_verify_attn_noalloc
        fn.argtypes = [POINTER(SpecAttnArgs), c_void_p]
        fn.restype = c_int
        _noalloc_fn = fn
    a, keep = verify_attn_args(q, k, v, kv_len, o, tree_parent, scale, None)
    st = _noalloc_fn(byref(a), _stream_handle(stream))
    del keep
    if st != SPEC_OK:
        raise SpecError(st, "spec_verify_attn_noalloc")
    return o


def commit_args(mode, kv_len, num_accepted, nq, *, k=None, v=None, path_nodes=None, workspace=None):
    B = kv_len.shape[0]
    a = SpecCommitArgs(mode=mode, B=B, nq=nq, kv_len=_ptr(kv_len), num_accepted=_ptr(num_accepted),
                       workspace=_ptr(workspace),
                       workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size())
    if k is not None:
        if k.stride(2) != k.shape[3] or tuple(k.stride()) != tuple(v.stride()):
            raise ValueError("k and v must share strides with token stride == head_dim")
        a.Hkv, a.Lmax, a.D = k.shape[1], k.shape[2], k.shape[3]
        a.kv_dtype = _dtype_code(k)
        a.k, a.v = _ptr(k), _ptr(v)
        a.kv_stride_b, a.kv_stride_h = k.stride(0), k.stride(1)
    else:
        a.Lmax = 2 ** 31 - 1
    if path_nodes is not None:
        a.path_nodes = _ptr(path_nodes)
        a.path_stride_b = path_nodes.stride(0)
        a.path_cols = path_nodes.shape[1]
    return a


def spec_commit(mode, kv_len, num_accepted, nq, *, k=None, v=None, path_nodes=None, workspace=None,
                stream=None):
    """Rollback after verification: kv_len [B] int32 (device, updated in place), num_accepted [B]
    int32 (device); SPEC_COMMIT_CHAIN needs nothing else; SPEC_COMMIT_TREE also moves the accepted
    path's K/V (k, v [B, Hkv, Lmax, D], path_nodes [B, path_cols] int32, e.g. spec_sample's
    out_path_nodes)."""
    _check_cuda(kv_len, num_accepted, k, v, path_nodes)
    ws = _workspace(256, kv_len.device, workspace)
    a = commit_args(mode, kv_len, num_accepted, nq, k=k, v=v, path_nodes=path_nodes, workspace=ws)
    st = lib().spec_commit(byref(a), _stream_handle(stream))
    if st != SPEC_OK:
        raise SpecError(st, "spec_commit")
    return ws

