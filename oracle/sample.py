"""Oracle: the speculative-sampling step over the vocabulary (chain) and greedy chain/tree
acceptance.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  float64 NumPy from fp32 logits.

Notation: P = target distribution, Q = draft distribution (the "Speculative Decoding & Medusa"
page writes p = target, q = draft in §2; the UW CSE 599K notes swap the letters).

Chain, stochastic -- the rule of "Speculative Decoding & Medusa" §2 and "Speculative Decoding in
LLM Serving Systems", Accepting and rejecting; "Guide to MagicDec", Solution §2 equations:

1. P_i = softmax(target row i), Q_i = softmax(draft row i), max-subtracted, temperature 1.
2. Walk i = 1..gamma: accept x_i iff u_i * Q_i(x_i) < P_i(x_i) (accept with probability
   min(1, P/Q); strict "<" with u in [0, 1); division-free so Q_i(x_i) = 0 accepts iff
   P_i(x_i) > 0).  Stop at the first rejection; k = number accepted.
3. Residual row r = max(P_{k+1} - Q_{k+1}, 0) if k < gamma, else r = P_{gamma+1} (the free bonus
   token).  R = sum r; if R == 0 use r = P_{k+1}.
4. Inverse CDF in token-id order with u_{gamma+1}: y = min{y : C(y) > u_{gamma+1} * R},
   C(y) = sum_{z <= y} r_z; if no index qualifies (rounding), the largest y with r_y > 0.
5. Emit x_1..x_k, y (1 to gamma+1 tokens).

Greedy (temperature-0 limit): the draft token is accepted iff it equals the target row's argmax
(ties to the smallest id).  Tree greedy: a node is accepted iff its parent is accepted and its
token equals the argmax of its parent's row (the root, the last committed token, is accepted);
the deepest accepted node (ties to the smallest index) is chosen and its path plus the argmax of
its own row are emitted.
"""

from __future__ import annotations

import numpy as np

NEAR_BAND = 1e-6


def softmax64(logits: np.ndarray) -> np.ndarray:
    """Max-subtracted softmax over the last axis in float64."""
    x = np.asarray(logits, dtype=np.float64)
    m = np.max(x, axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def acceptance_rate(P: np.ndarray, Q: np.ndarray) -> float:
    """Probability that a draft x ~ Q passes the accept test: sum_x Q(x) min(1, P(x)/Q(x))
    = sum_x min(P(x), Q(x))."""
    return float(np.sum(np.minimum(P, Q)))


def expected_tokens_per_round(alpha: float, gamma: int) -> float:
    """Expected tokens emitted per round, (1 - alpha^(gamma+1)) / (1 - alpha)
    ("Speculative Decoding & Medusa", §1 formula block)."""
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)


def _leading_true(acc: np.ndarray) -> np.ndarray:
    """Per row, the number of leading True entries."""
    n = acc.shape[1]
    first_false = np.where(acc.all(axis=1), n, np.argmin(acc, axis=1))
    return first_false.astype(np.int64)


def spec_sample_chain(target_logits, draft_logits, draft_tokens, uniforms, band: float = NEAR_BAND,
                      batch_chunk: int = 65536):
    """Stochastic chain step, batched over sequences.

    target_logits [B, gamma+1, V], draft_logits [B, gamma, V] (fp32 values), draft_tokens
    [B, gamma] int, uniforms [B, gamma+1] in [0, 1).
    Returns (out_tokens [B, gamma+1] int32 padded with -1, num_accepted [B] int32 (-1 marks a
    draft token id outside [0, V)), near [B] bool: some decision lay within ``band`` of its
    threshold -- |u_i - P_i(x_i)/Q_i(x_i)| <= band for an evaluated accept test, or
    min_y |u*R - C(y)| <= band*R for the final draw).
    """
    B = target_logits.shape[0]
    outs, nacc, near = [], [], []
    for s in range(0, B, batch_chunk):
        o, n, f = _spec_sample_chain_block(target_logits[s:s + batch_chunk], draft_logits[s:s + batch_chunk],
                                           draft_tokens[s:s + batch_chunk], uniforms[s:s + batch_chunk], band)
        outs.append(o)
        nacc.append(n)
        near.append(f)
    return np.concatenate(outs), np.concatenate(nacc), np.concatenate(near)


def _spec_sample_chain_block(t, d, x, u, band):
    B, g1, V = t.shape
    gamma = g1 - 1
    rows = np.arange(B)
    x = np.asarray(x, dtype=np.int64).reshape(B, gamma)
    u = np.asarray(u, dtype=np.float32).astype(np.float64)
    bad = np.any((x < 0) | (x >= V), axis=1)
    xc = np.clip(x, 0, V - 1)

    P = softmax64(t)                       # [B, gamma+1, V]
    Q = softmax64(d)                       # [B, gamma, V]
    px = np.take_along_axis(P[:, :gamma], xc[..., None], axis=-1)[..., 0]
    qx = np.take_along_axis(Q, xc[..., None], axis=-1)[..., 0]
    acc = u[:, :gamma] * qx < px
    k = _leading_true(acc)

    # which accept tests were evaluated: i <= k (and i < gamma)
    evaluated = np.arange(gamma)[None, :] <= k[:, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(qx > 0, px / np.where(qx > 0, qx, 1.0), np.inf)
    near_acc = np.any(evaluated & (qx > 0) & (px > 0) & (np.abs(u[:, :gamma] - ratio) <= band), axis=1)

    kk = np.minimum(k, gamma - 1) if gamma > 0 else np.zeros_like(k)
    P_k = P[rows, k]                        # row k+1 in 1-based terms (row gamma+1 when k = gamma)
    if gamma > 0:
        Q_k = Q[rows, kk]
        r = np.where((k < gamma)[:, None], np.maximum(P_k - Q_k, 0.0), P_k)
    else:
        r = P_k
    R = r.sum(axis=1)
    r = np.where((R == 0)[:, None], P_k, r)
    R = r.sum(axis=1)
    C = np.cumsum(r, axis=1)
    thr = u[:, gamma] * R
    past = C > thr[:, None]
    any_past = past.any(axis=1)
    first_past = np.argmax(past, axis=1)
    last_pos = V - 1 - np.argmax((r > 0)[:, ::-1], axis=1)
    y = np.where(any_past, first_past, last_pos)
    near_draw = np.min(np.abs(C - thr[:, None]), axis=1) <= band * R

    out = np.full((B, gamma + 1), -1, dtype=np.int32)
    for b in range(B):
        if bad[b]:
            continue
        out[b, : k[b]] = x[b, : k[b]]
        out[b, k[b]] = y[b]
    nacc = np.where(bad, -1, k).astype(np.int32)
    near = (near_acc | near_draw) & ~bad
    return out, nacc, near


def chain_outcome_valid(target_logits, draft_logits, draft_tokens, uniforms, out_tokens, num_accepted,
                        band: float = NEAR_BAND) -> np.ndarray:
    """Per sequence: is (out_tokens, num_accepted) an outcome of the chain rule above once every
    decision whose exact value lies within ``band`` of its threshold may go either way?

    These are exactly the decisions ``spec_sample_chain`` flags as near: an evaluated accept test
    with |u_i - P_i(x_i)/Q_i(x_i)| <= band, and a final draw whose threshold u * R lies within
    band * R of a CDF step.  So for a sequence with no near decision only the outcome
    ``spec_sample_chain`` returns is valid, and for one with near decisions every outcome that
    rounding on either side of those thresholds can produce is.  Steps, for the claimed k:

    1. Accept tests 1..k must pass and test k+1 (if k < gamma) must fail, each unless near.
    2. The emitted row is x_1..x_k, then y, then -1 padding.
    3. With the residual row r of step 3 for this k (R = sum r, r = P_{k+1} if R = 0), y must hold
       mass (r_y > 0) and its CDF step [C(y-1), C(y)) must meet [u R - band R, u R + band R].
    A row with a draft token outside [0, V) is valid only as (-1 ..., num_accepted -1).
    """
    t = np.asarray(target_logits)
    d = np.asarray(draft_logits)
    B, g1, V = t.shape
    gamma = g1 - 1
    x = np.asarray(draft_tokens, dtype=np.int64).reshape(B, gamma)
    u = np.asarray(uniforms, dtype=np.float32).astype(np.float64)
    out = np.asarray(out_tokens)
    nacc = np.asarray(num_accepted)
    valid = np.zeros(B, dtype=bool)
    for b in range(B):
        k = int(nacc[b])
        if np.any((x[b] < 0) | (x[b] >= V)):
            valid[b] = k == -1 and bool(np.all(out[b] == -1))
            continue
        if not 0 <= k <= gamma:
            continue
        P = softmax64(t[b])
        Q = softmax64(d[b]) if gamma > 0 else None
        ok = True
        for i in range(min(k + 1, gamma)):          # tests 1..k+1 (0-based 0..k)
            px, qx = P[i, x[b, i]], Q[i, x[b, i]]
            accepted = u[b, i] * qx < px
            near = qx > 0 and px > 0 and abs(u[b, i] - px / qx) <= band
            if accepted != (i < k) and not near:
                ok = False
                break
        if not ok:
            continue
        if not (np.array_equal(out[b, :k], x[b, :k]) and np.all(out[b, k + 1:] == -1)):
            continue
        y = int(out[b, k])
        if k < gamma:
            r = np.maximum(P[k] - Q[k], 0.0)
        else:
            r = P[k]
        if r.sum() == 0:
            r = P[k]
        R = r.sum()
        if not 0 <= y < V or r[y] <= 0:
            continue
        C = np.cumsum(r)
        thr = u[b, gamma] * R
        lo = C[y - 1] if y > 0 else 0.0
        valid[b] = lo <= thr + band * R and C[y] > thr - band * R
    return valid


def argmax_rows(logits: np.ndarray) -> np.ndarray:
    """Argmax over the last axis, ties to the smallest index (NumPy returns the first maximum)."""
    return np.argmax(np.asarray(logits, dtype=np.float32), axis=-1).astype(np.int64)


def greedy_chain(target_logits, draft_tokens):
    """Greedy chain verify: accept x_i while x_i == argmax(target row i); then emit the argmax of
    the first unmatched row (or of row gamma+1).  Returns (out_tokens [B, gamma+1], num_accepted)."""
    B, g1, V = target_logits.shape
    gamma = g1 - 1
    x = np.asarray(draft_tokens, dtype=np.int64).reshape(B, gamma)
    bad = np.any((x < 0) | (x >= V), axis=1)
    a = argmax_rows(target_logits)          # [B, gamma+1]
    k = _leading_true(x == a[:, :gamma]) if gamma > 0 else np.zeros(B, dtype=np.int64)
    out = np.full((B, gamma + 1), -1, dtype=np.int32)
    for b in range(B):
        if bad[b]:
            continue
        out[b, : k[b]] = x[b, : k[b]]
        out[b, k[b]] = a[b, k[b]]
    return out, np.where(bad, -1, k).astype(np.int32)


def tree_depths(parent: np.ndarray) -> np.ndarray:
    depth = np.zeros(len(parent), dtype=np.int64)
    for i in range(1, len(parent)):
        depth[i] = depth[int(parent[i])] + 1
    return depth


def tree_greedy(target_logits, node_tokens, parent, out_cols: int | None = None):
    """Greedy longest-accepted-path selection over a token tree.

    target_logits [B, N, V] (row i = the target's next-token logits after node i),
    node_tokens [B, N], parent [N] (parent[0] = -1, parent[i] < i).
    Returns (out_tokens [B, out_cols], out_path_nodes [B, out_cols], num_accepted [B]); out_tokens
    holds the accepted path's tokens (depth 1..d) then the argmax of the deepest node's row;
    out_path_nodes holds the accepted nodes (depth 1..d); both padded with -1.
    """
    B, N, V = target_logits.shape
    depth = tree_depths(parent)
    if out_cols is None:
        out_cols = int(depth.max()) + 1
    tok = np.asarray(node_tokens, dtype=np.int64)
    a = argmax_rows(target_logits)          # [B, N]
    out = np.full((B, out_cols), -1, dtype=np.int32)
    nodes = np.full((B, out_cols), -1, dtype=np.int32)
    nacc = np.zeros(B, dtype=np.int32)
    for b in range(B):
        if np.any((tok[b, 1:] < 0) | (tok[b, 1:] >= V)):
            nacc[b] = -1
            continue
        accepted = np.zeros(N, dtype=bool)
        accepted[0] = True
        for i in range(1, N):
            p = int(parent[i])
            accepted[i] = accepted[p] and tok[b, i] == a[b, p]
        best = 0
        for i in range(N):
            if accepted[i] and depth[i] > depth[best]:
                best = i
        path = []
        j = best
        while j > 0:
            path.append(j)
            j = int(parent[j])
        path.reverse()
        for n_, node in enumerate(path):
            out[b, n_] = tok[b, node]
            nodes[b, n_] = node
        out[b, len(path)] = a[b, best]
        nacc[b] = len(path)
    return out, nodes, nacc


def tree_stochastic(target_logits, draft_logits, node_tokens, parent, uniforms, out_cols: int | None = None,
                    band: float = NEAR_BAND):
    """Stochastic acceptance over a token tree: multi-step speculative sampling.

    The pages name tree verification with sampling (SpecInfer, "Speculative Decoding in LLM
    Serving Systems", Tree-based variants) but do not state its rule; the reading used here
    applies the chain rule of "Speculative Decoding & Medusa" §2 to the children of one node in
    turn, each rejection replacing the target distribution by the normalised residual, as in the
    chain's resampling step:

    1. At node n (starting at the root, node 0, the last committed token): R = P_n =
       softmax(target row n); Q_n = softmax(draft row n), the distribution n's children were drawn
       from.
    2. For each child c of n in increasing index order, with token x_c: accept iff
       u_c * Q_n(x_c) < R(x_c) (u_c = uniforms[b, c]; division-free like the chain test).
       Accepted: emit x_c and continue at step 1 with n = c.  Rejected: R = max(R - Q_n, 0)
       normalised (R = P_n if that has no mass) and test the next child.
    3. When no child of n is accepted (a leaf included): draw y from R by inverse CDF in token-id
       order with u_0 = uniforms[b, 0] (node 0 has no accept test): y = min{y : C(y) > u_0},
       C the cumulative sum of R; if none qualifies (rounding), the largest y with R_y > 0.
       Emit y.

    target_logits, draft_logits [B, N, V] fp32 (rows of leaves are not read), node_tokens [B, N],
    parent [N], uniforms [B, N] in [0, 1).  Returns (out_tokens [B, out_cols], out_path_nodes
    [B, out_cols], num_accepted [B] (-1: a child token outside [0, V); nothing emitted),
    near [B] (an evaluated accept test with |u_c - R(x_c)/Q_n(x_c)| <= band, or a final draw
    with min_y |u_0 - C(y)| <= band)), padded with -1 like tree_greedy.
    """
    B, N, V = target_logits.shape
    depth = tree_depths(parent)
    if out_cols is None:
        out_cols = int(depth.max()) + 1
    tok = np.asarray(node_tokens, dtype=np.int64)
    u = np.asarray(uniforms, dtype=np.float32).astype(np.float64)
    children = [[] for _ in range(N)]
    for i in range(1, N):
        children[int(parent[i])].append(i)
    out = np.full((B, out_cols), -1, dtype=np.int32)
    nodes = np.full((B, out_cols), -1, dtype=np.int32)
    nacc = np.zeros(B, dtype=np.int32)
    near = np.zeros(B, dtype=bool)
    for b in range(B):
        if np.any((tok[b, 1:] < 0) | (tok[b, 1:] >= V)):
            nacc[b] = -1
            continue
        n, d = 0, 0
        while True:
            P = softmax64(target_logits[b, n])
            R = P
            moved = False
            if children[n]:
                Q = softmax64(draft_logits[b, n])
                for c in children[n]:
                    x = int(tok[b, c])
                    if Q[x] > 0 and R[x] > 0 and abs(u[b, c] - R[x] / Q[x]) <= band:
                        near[b] = True
                    if u[b, c] * Q[x] < R[x]:
                        out[b, d] = x
                        nodes[b, d] = c
                        d += 1
                        n = c
                        moved = True
                        break
                    r = np.maximum(R - Q, 0.0)
                    R = r / r.sum() if r.sum() > 0 else P
            if moved:
                continue
            C = np.cumsum(R)
            past = np.nonzero(C > u[b, 0])[0]
            y = int(past[0]) if len(past) else int(np.nonzero(R > 0)[0][-1])
            if np.min(np.abs(C - u[b, 0])) <= band:
                near[b] = True
            out[b, d] = y
            nacc[b] = d
            break
    return out, nodes, nacc, near
