"""Oracle: attention over the KV cache for speculative verify and for the bounded draft window.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  float64 NumPy, one (sequence, head,
query row) at a time, exact max-subtracted softmax over the whole visible key set (no splitting).

Readings of the pages used here (the pages never write the attention formula):

* Attention is ``o = softmax(scale * q . k_t) @ v`` over the visible keys t, scale = D^-1/2
  unless given; Q and K arrive already position-encoded.
* Query head h reads KV head floor(h / G), G = Hq / Hkv (contiguous grouping).
* Chain verify ("Guide to MagicDec", Implementation Step 3: one target pass over prefix +
  drafts; "Speculative Decoding in LLM Serving Systems", The algorithm step 2): the nq = gamma+1
  new tokens are the last nq entries of the cache, and query row j sees keys 0 .. L - nq + j.
* Tree verify ("Speculative Decoding & Medusa", §4; "... LLM Serving Systems", Tree-based
  variants: each token attends only to its ancestors): node i sees the context keys
  [0, L - N) and the tree keys L - N + m for m in anc*(i) = {i, parent(i), ..., 0}.
* Draft window ("Guide to MagicDec", Solution §1 and Implementation Step 1): the draft attends
  to the last min(pos, W) tokens, token t stored in ring slot t mod W.
"""

from __future__ import annotations

import numpy as np


def attend(q: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float) -> np.ndarray:
    """Softmax attention of one query over an explicit key set (rows of ``keys``/``values``)."""
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    if keys.shape[0] == 0:
        return np.zeros(values.shape[-1], dtype=np.float64)
    s = (keys @ q) * scale
    m = np.max(s)
    w = np.exp(s - m)
    return (w @ values) / np.sum(w)


def default_scale(D: int, scale: float = 0.0) -> float:
    return float(scale) if scale else 1.0 / np.sqrt(D)


def ancestors(parent: np.ndarray, i: int) -> list:
    """anc*(i): node i and every node on its path to the root (parent[root] = -1)."""
    out = []
    j = int(i)
    while j >= 0:
        out.append(j)
        j = int(parent[j])
    return out


def chain_visible(L: int, nq: int, j: int) -> np.ndarray:
    """Key positions seen by chain query row j when the cache holds L entries, the last nq new."""
    return np.arange(0, L - nq + j + 1)


def tree_visible(L: int, parent: np.ndarray, i: int) -> np.ndarray:
    """Key positions seen by tree node i: the context plus the node's ancestors (and itself)."""
    N = len(parent)
    ctx = np.arange(0, L - N)
    tree = np.array(sorted(L - N + m for m in ancestors(parent, i)), dtype=np.int64)
    return np.concatenate([ctx, tree])


def verify_attn(q, k, v, kv_len, tree_parent=None, scale: float = 0.0) -> np.ndarray:
    """Verify attention, chain (``tree_parent is None``) or tree.

    q [B, nq, Hq, D]; k, v [B, Hkv, Lmax, D]; kv_len [B] (includes the nq new tokens).
    Returns o [B, nq, Hq, D] float64.
    """
    B, nq, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    sc = default_scale(D, scale)
    o = np.zeros((B, nq, Hq, D), dtype=np.float64)
    for b in range(B):
        L = int(kv_len[b])
        for j in range(nq):
            vis = chain_visible(L, nq, j) if tree_parent is None else tree_visible(L, tree_parent, j)
            for h in range(Hq):
                g = h // G
                o[b, j, h] = attend(q[b, j, h], k[b, g, vis], v[b, g, vis], sc)
    return o


def append_new_tokens(k, v, kv_len, k_new, v_new):
    """The verify step's append ("Speculative Decoding in LLM Serving Systems", The algorithm: the
    target pass over prefix + drafts extends the target cache; "Guide to MagicDec",
    Implementation Step 3): the nq new tokens' K/V rows ``k_new[b, j, g]`` go to cache position
    kv_len[b] - nq + j of head g.  k, v [B, Hkv, Lmax, D]; k_new, v_new [B, nq, Hkv, D].  A
    sequence with kv_len outside [nq, Lmax] is left as it is.  Returns new arrays."""
    k = np.array(k, copy=True)
    v = np.array(v, copy=True)
    nq, Lmax = k_new.shape[1], k.shape[2]
    for b in range(k.shape[0]):
        L = int(kv_len[b])
        if L < nq or L > Lmax:
            continue
        for j in range(nq):
            k[b, :, L - nq + j, :] = k_new[b, j]
            v[b, :, L - nq + j, :] = v_new[b, j]
    return k, v


def token_slot(t: int, W: int, n_sinks: int = 0) -> int:
    """Ring slot of token t ([MagicDec] Implementation Step 1, with the attention sinks of Best
    Practices §1): the first n_sinks tokens keep slots 0..n_sinks-1 for good; every later token t
    goes to slot n_sinks + (t - n_sinks) mod (W - n_sinks).  n_sinks = 0 is the plain ring."""
    t = int(t)
    if t < n_sinks:
        return t
    return n_sinks + (t - n_sinks) % (W - n_sinks)


def window_tokens(pos: int, W: int, n_sinks: int = 0) -> list:
    """Tokens the draft sees after pos tokens were written: all of them while pos <= W, else the
    n_sinks first ones and the W - n_sinks most recent ones."""
    pos = int(pos)
    if pos <= W:
        return list(range(pos))
    return list(range(n_sinks)) + list(range(pos - (W - n_sinks), pos))


def window_slots(pos: int, W: int, n_sinks: int = 0) -> np.ndarray:
    """Slots holding the visible tokens (for n_sinks = 0: {t mod W : pos - min(pos, W) <= t < pos})."""
    return np.array(sorted({token_slot(t, W, n_sinks) for t in window_tokens(pos, W, n_sinks)}), dtype=np.int64)


def ring_append(k_ring, v_ring, pos, k_new, v_new, n_sinks: int = 0):
    """Write the current token's K/V (token index pos[b]-1) into its slot.
    Returns new ring arrays (inputs are not modified)."""
    k_ring = np.array(k_ring, copy=True)
    v_ring = np.array(v_ring, copy=True)
    W = k_ring.shape[2]
    for b in range(k_ring.shape[0]):
        s = token_slot(int(pos[b]) - 1, W, n_sinks)
        k_ring[b, :, s] = k_new[b]
        v_ring[b, :, s] = v_new[b]
    return k_ring, v_ring


def draft_window_attn(q, k_ring, v_ring, pos, k_new=None, v_new=None, scale: float = 0.0, n_sinks: int = 0):
    """Single-query draft attention over the ring-buffer window.

    q [B, Hq, D]; k_ring, v_ring [B, Hkv, W, D]; pos [B] = tokens written including the current
    one.  If k_new/v_new [B, Hkv, D] are given they are appended first (slot of token pos-1).
    Returns (o [B, Hq, D] float64, k_ring, v_ring after the append).
    """
    if k_new is not None:
        k_ring, v_ring = ring_append(k_ring, v_ring, pos, k_new, v_new, n_sinks)
    B, Hq, D = q.shape
    Hkv, W = k_ring.shape[1], k_ring.shape[2]
    G = Hq // Hkv
    sc = default_scale(D, scale)
    o = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        slots = window_slots(int(pos[b]), W, n_sinks)
        for h in range(Hq):
            g = h // G
            o[b, h] = attend(q[b, h], k_ring[b, g, slots], v_ring[b, g, slots], sc)
    return o, k_ring, v_ring


class RollWindowCache:
    """The page's bounded draft cache as written there (Implementation Step 1): fill slots in
    order until full, then shift left by one and write the newest token into the last slot.
    Kept only as a second, independently laid-out model of the window for the ring tests."""

    def __init__(self, W: int, Hkv: int, D: int):
        self.W = W
        self.k = np.zeros((Hkv, W, D))
        self.v = np.zeros((Hkv, W, D))
        self.n = 0

    def append(self, k_tok: np.ndarray, v_tok: np.ndarray) -> None:
        if self.n < self.W:
            self.k[:, self.n] = k_tok
            self.v[:, self.n] = v_tok
            self.n += 1
        else:
            self.k = np.roll(self.k, -1, axis=1)
            self.v = np.roll(self.v, -1, axis=1)
            self.k[:, -1] = k_tok
            self.v[:, -1] = v_tok

    def get_kv(self):
        return self.k[:, : self.n], self.v[:, : self.n]


class SinkRollCache:
    """The page's shift-left draft cache with attention sinks: the first n_sinks tokens stay in
    front; behind them a FIFO of W - n_sinks slots filled in order, then shifted left by one per
    new token.  An independently laid-out model for the sink tests."""

    def __init__(self, W: int, n_sinks: int, Hkv: int, D: int):
        self.W, self.S = W, n_sinks
        self.sk = np.zeros((Hkv, 0, D))
        self.sv = np.zeros((Hkv, 0, D))
        self.fifo = RollWindowCache(W - n_sinks, Hkv, D)

    def append(self, k_tok: np.ndarray, v_tok: np.ndarray) -> None:
        if self.sk.shape[1] < self.S:
            self.sk = np.concatenate([self.sk, k_tok[:, None]], axis=1)
            self.sv = np.concatenate([self.sv, v_tok[:, None]], axis=1)
        else:
            self.fifo.append(k_tok, v_tok)

    def get_kv(self):
        fk, fv = self.fifo.get_kv()
        return np.concatenate([self.sk, fk], axis=1), np.concatenate([self.sv, fv], axis=1)
