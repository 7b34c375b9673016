"""Oracle: the LM-head projection fused with greedy verification.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"Speculative Decoding in LLM Serving Systems", The algorithm (and "Guide to MagicDec",
Implementation Step 3): one target forward over the drafted positions gives a next-token
distribution per position; its logits are the target's final hidden state at that position times
the LM-head (unembedding) matrix.  In the greedy modes (the temperature-0 limit of the accept
rule) only each row's argmax is used: the chain accepts drafts while they equal the argmax of
their row, the tree keeps the deepest node whose path matches its parents' argmaxes
(``oracle.sample.greedy_chain`` / ``tree_greedy``).

Here the logits are the plain matrix product in float64 of the stored (bf16-rounded) hidden
states and weights (a library matmul), followed by those greedy rules.  A row whose top two
logits lie within the fp32 accumulation error bound of a d-term dot product of each other is
marked ``near``: an fp32 kernel may pick either of them.
"""

from __future__ import annotations

import numpy as np

from . import sample as osm

# |fp32 sum - exact| <= d * 2^-24 * sum |terms| (worst case for d = 4096: 2.4e-4 sum |terms|);
# near_rows uses the larger of this floor and d * 2^-24 for the actual d
NEAR_REL = 2.5e-4


def lmhead_logits(hidden: np.ndarray, weight: np.ndarray, chunk: int = 8192) -> np.ndarray:
    """hidden [B, R, d], weight [V, d] (values as stored) -> logits [B, R, V] in float64.  The
    product is taken over blocks of ``chunk`` weight rows only to bound the float64 copy of the
    weight; every logit is the same d-term dot product either way."""
    h = np.asarray(hidden, np.float64)
    V = weight.shape[0]
    out = np.empty(h.shape[:-1] + (V,), np.float64)
    for v0 in range(0, V, chunk):
        out[..., v0:v0 + chunk] = h @ np.asarray(weight[v0:v0 + chunk], np.float64).T
    return out


def near_rows(hidden: np.ndarray, weight: np.ndarray, logits: np.ndarray, rel: float | None = None) -> np.ndarray:
    """[B, R] bool: the row's two largest logits differ by at most rel * (sum_k |h_k w_ak| +
    sum_k |h_k w_bk|), a and b the two top ids; rel defaults to max(NEAR_REL, d * 2^-24), the
    worst-case relative error of a d-term fp32 sum."""
    B, R, V = logits.shape
    if rel is None:
        rel = max(NEAR_REL, hidden.shape[-1] * 2.0 ** -24)
    top2 = np.argsort(-logits, axis=-1, kind="stable")[..., :2]
    h = np.abs(np.asarray(hidden, np.float64))
    near = np.zeros((B, R), dtype=bool)
    for b in range(B):
        for r in range(R):
            a, c = int(top2[b, r, 0]), int(top2[b, r, 1])
            wa = np.abs(np.asarray(weight[a], np.float64))
            wc = np.abs(np.asarray(weight[c], np.float64))
            bound = rel * (float(h[b, r] @ wa) + float(h[b, r] @ wc))
            near[b, r] = logits[b, r, a] - logits[b, r, c] <= bound
    return near


def lmhead_greedy_chain(hidden, weight, draft_tokens):
    """Greedy chain verify from hidden states: (out_tokens [B, gamma+1], num_accepted [B],
    near [B]); near marks a sequence with a near-tie in a row the rule looks at (rows 0..k)."""
    logits = lmhead_logits(hidden, weight)
    out, k = osm.greedy_chain(logits, draft_tokens)
    nr = near_rows(hidden, weight, logits)
    near = np.array([bool(nr[b, : max(int(k[b]), 0) + 1].any()) for b in range(len(k))])
    return out, k, near


def lmhead_tree_greedy(hidden, weight, node_tokens, parent, out_cols: int | None = None):
    """Greedy tree selection from hidden states: (out_tokens, out_path_nodes, num_accepted, near);
    near marks a sequence with a near-tie in a row the rule consults: the root's and every
    accepted node's (their argmaxes decide their children and the emitted token)."""
    logits = lmhead_logits(hidden, weight)
    out, nodes, k = osm.tree_greedy(logits, node_tokens, parent, out_cols)
    nr = near_rows(hidden, weight, logits)
    tok = np.asarray(node_tokens)
    a = np.argmax(logits, axis=-1)
    near = np.zeros(len(k), dtype=bool)
    for b in range(len(k)):
        acc = np.zeros(len(parent), dtype=bool)
        acc[0] = True
        for i in range(1, len(parent)):
            acc[i] = acc[int(parent[i])] and tok[b, i] == a[b, int(parent[i])]
        near[b] = bool(nr[b][acc].any())
    return out, nodes, k, near
