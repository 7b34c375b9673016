"""Oracle: the rollback step after verification -- committing the accepted tokens' K/V.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"Speculative Decoding in LLM Serving Systems", Accepting and rejecting: once a draft token is
rejected, it and every later draft are discarded; "Guide to MagicDec", Solution §2 and
Implementation Step 3: the verified positions whose tokens were accepted stay in the target's
cache.  "Speculative Decoding & Medusa" §4: a token tree is verified in one pass, and the accepted
path is the prefix that continues.

Cache convention (the same as verify attention): sequence b's cache holds kv_len[b] keys; the nq
positions verified in the round are the last nq, kv_len[b] - nq .. kv_len[b] - 1.

Chain (nq = gamma + 1): position kv_len - nq holds the last committed token (the round's first
query) and the next gamma positions the drafts x_1..x_gamma.  With k accepted drafts the first
k + 1 verified positions stay; the emitted token after them has no K/V yet (the next round
verifies it).  New length: kv_len - nq + 1 + k.  Nothing moves.

Tree (nq = N nodes, node i at position kv_len - N + i, node 0 the root = the last committed
token): with the accepted path n_1, ..., n_k (depths 1..k, as spec_sample's tree mode reports
them), the root stays and the K/V of n_j move to position kv_len - N + j.  New length:
kv_len - N + 1 + k.

A sequence with num_accepted < 0 (a bad token id in the sampling step) or an out-of-range kv_len
is left unchanged and flagged.
"""

from __future__ import annotations

import numpy as np


def chain_commit(kv_len: np.ndarray, nq: int, num_accepted: np.ndarray, Lmax: int):
    """Returns (new kv_len [B], flags [B] bool = the sequence was left unchanged)."""
    kv_len = np.asarray(kv_len, dtype=np.int64)
    k = np.asarray(num_accepted, dtype=np.int64)
    out = kv_len.copy()
    flag = np.zeros(len(kv_len), dtype=bool)
    for b in range(len(kv_len)):
        if k[b] < 0 or k[b] > nq - 1 or kv_len[b] < nq or kv_len[b] > Lmax:
            flag[b] = True
            continue
        out[b] = kv_len[b] - nq + 1 + k[b]
    return out, flag


def tree_commit(k_cache: np.ndarray, v_cache: np.ndarray, kv_len: np.ndarray, N: int,
                path_nodes: np.ndarray, num_accepted: np.ndarray):
    """k_cache, v_cache [B, Hkv, Lmax, D]; path_nodes [B, path_cols] node ids (depth order); a count
    above path_cols or a node id outside [1, N) is flagged like a bad count.
    Returns (k, v, new kv_len, flags); inputs are not modified."""
    k_cache = np.array(k_cache, copy=True)
    v_cache = np.array(v_cache, copy=True)
    kv_len = np.asarray(kv_len, dtype=np.int64)
    acc = np.asarray(num_accepted, dtype=np.int64)
    Lmax = k_cache.shape[2]
    out = kv_len.copy()
    flag = np.zeros(len(kv_len), dtype=bool)
    for b in range(len(kv_len)):
        L, kb = int(kv_len[b]), int(acc[b])
        if kb < 0 or kb > N - 1 or kb > path_nodes.shape[1] or L < N or L > Lmax:
            flag[b] = True
            continue
        if any(not 1 <= int(path_nodes[b, j]) < N for j in range(kb)):
            flag[b] = True
            continue
        base = L - N
        src = [base + int(path_nodes[b, j]) for j in range(kb)]
        rows_k = k_cache[b][:, src].copy()   # gathered first: sources and destinations overlap
        rows_v = v_cache[b][:, src].copy()
        for j in range(kb):
            k_cache[b][:, base + 1 + j] = rows_k[:, j]
            v_cache[b][:, base + 1 + j] = rows_v[:, j]
        out[b] = base + 1 + kb
    return k_cache, v_cache, out, flag
