"""Seeded host-side (NumPy) input generators.

Every array is drawn from ``numpy.random.default_rng([seed, sub])`` with a fixed sub-seed per
tensor, so any case can be replayed from (config, seed).  bf16 workloads are rounded to bf16
with round-to-nearest-even on the host; the returned float32 arrays hold exactly the values a
bf16 tensor holds, so the oracle sees the stored inputs and the tolerance measures kernel error
only.

None of the method's arithmetic is here.  Draft tokens x_i ~ softmax(draft logits) are drawn by
the Gumbel-max construction (argmax of logits plus Gumbel noise), which needs no softmax.
"""

from __future__ import annotations

import numpy as np

SUB = dict(q=1, k=2, v=3, kv_len=4, tree=5, target=6, draft=7, tokens=8, uniforms=9,
           ring_k=10, ring_v=11, new_k=12, new_v=13, pos=14, needles=15, gumbel=16, tree_tok=17,
           tree_gumbel=18)

BF16_NAN = np.float32(np.nan)


def rng_for(seed: int, what: str) -> np.random.Generator:
    return np.random.default_rng([int(seed), SUB[what]])


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); NaN stays NaN. Returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    src, dst = x.reshape(-1).view(np.uint32), out.reshape(-1).view(np.uint32)
    step = 1 << 22   # blocks bound the temporaries for weight-sized arrays
    for i in range(0, src.size, step):
        b = src[i:i + step]
        # 32-bit add wraps only for NaN bit patterns, which are restored below
        dst[i:i + step] = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    out[np.isnan(x)] = np.nan
    return out


def store(x: np.ndarray, dtype: str) -> np.ndarray:
    """Values as stored in a tensor of ``dtype`` ("f32" or "bf16"), as float32."""
    x = x.astype(np.float32)
    return round_bf16(x) if dtype == "bf16" else x


def kv_lengths(B: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """Per-sequence KV length uniform on the integers [lo, hi]."""
    if lo == hi:
        return np.full(B, lo, dtype=np.int32)
    return rng_for(seed, "kv_len").integers(lo, hi + 1, size=B).astype(np.int32)


def random_tree(N: int, max_depth: int, max_children: int, seed: int) -> np.ndarray:
    """parent[N] int32 with parent[0] = -1 and parent[i] < i.

    For i = 1..N-1 the parent is drawn uniformly among earlier nodes whose depth is below
    ``max_depth`` and which have fewer than ``max_children`` children.
    """
    r = rng_for(seed, "tree")
    parent = np.full(N, -1, dtype=np.int32)
    depth = np.zeros(N, dtype=np.int64)
    nchild = np.zeros(N, dtype=np.int64)
    for i in range(1, N):
        cands = [j for j in range(i) if depth[j] < max_depth and nchild[j] < max_children]
        if not cands:
            raise ValueError("tree capacity exhausted")
        p = cands[int(r.integers(len(cands)))]
        parent[i] = p
        depth[i] = depth[p] + 1
        nchild[p] += 1
    return parent


def attn_inputs(B: int, Hq: int, Hkv: int, D: int, nq: int, kv_len: np.ndarray, Lmax: int,
                dtype: str, seed: int, tail_fill: str = "nan") -> dict:
    """Q [B, nq, Hq, D], K/V [B, Hkv, Lmax, D] ~ N(0,1); K/V slots at or past kv_len[b] hold
    NaN (``tail_fill="nan"``) or zeros, so a kernel that reads unused cache slots shows it."""
    q = store(rng_for(seed, "q").standard_normal((B, nq, Hq, D), dtype=np.float32), dtype)
    k = store(rng_for(seed, "k").standard_normal((B, Hkv, Lmax, D), dtype=np.float32), dtype)
    v = store(rng_for(seed, "v").standard_normal((B, Hkv, Lmax, D), dtype=np.float32), dtype)
    fill = np.float32(np.nan) if tail_fill == "nan" else np.float32(0.0)
    for b in range(B):
        k[b, :, int(kv_len[b]):, :] = fill
        v[b, :, int(kv_len[b]):, :] = fill
    return dict(q=q, k=k, v=v, kv_len=np.asarray(kv_len, dtype=np.int32))


def _unit(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float64)
    return x / max(np.linalg.norm(x), 1e-30)


def plant_chain_needles(inp: dict, nq: int, dtype: str, seed: int, strength: float = 6.0) -> dict:
    """Plant keys that make mask mistakes visible (chain verify).

    Per (b, kv head g): a "hit" key at a position every row sees, aligned with the query of
    row 0 / head g*G, and for each row j < nq-1 a "trap" key at position L_b - nq + j + 1 (the
    first key row j must NOT see), aligned with that row's query.  A kernel that leaks the causal
    mask then puts a large weight on the trap's value row.
    """
    q, k = inp["q"], inp["k"]
    B, _, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    r = rng_for(seed, "needles")
    for b in range(B):
        L = int(inp["kv_len"][b])
        for g in range(Hkv):
            h = g * G
            if L - nq > 0:
                p = int(r.integers(0, L - nq))
                k[b, g, p] = strength * np.sqrt(D) * _unit(q[b, 0, h])
            for j in range(nq - 1):
                pos = L - nq + j + 1
                k[b, g, pos] = 1.5 * strength * np.sqrt(D) * _unit(q[b, j, h])
    inp["k"] = store(k, dtype)
    return inp


def plant_tree_needles(inp: dict, parent: np.ndarray, dtype: str, seed: int,
                       strength: float = 9.0) -> dict:
    """Plant tree traps: the key of tree node m is aligned with the query of a node i that is
    neither m nor a descendant of m, i.e. a node that must not see m."""
    q, k = inp["q"], inp["k"]
    B, N, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    r = rng_for(seed, "needles")
    anc = [set() for _ in range(N)]
    for i in range(N):
        j = i
        while j >= 0:
            anc[i].add(j)
            j = int(parent[j])
    for b in range(B):
        L = int(inp["kv_len"][b])
        for g in range(Hkv):
            for m in range(1, N):
                blind = [i for i in range(N) if m not in anc[i]]
                if not blind:
                    continue
                i = blind[int(r.integers(len(blind)))]
                k[b, g, L - N + m] = strength * np.sqrt(D) * _unit(q[b, i, g * G])
    inp["k"] = store(k, dtype)
    return inp


def window_inputs(B: int, Hq: int, Hkv: int, D: int, W: int, pos: np.ndarray, dtype: str,
                  seed: int) -> dict:
    """Draft-window inputs: q [B, Hq, D]; ring K/V [B, Hkv, W, D]; pos[b] = tokens written
    including the current one; new K/V [B, Hkv, D] for the current token.  Ring slots that no
    token has reached yet (slot >= pos[b] while pos[b] < W) hold NaN."""
    q = store(rng_for(seed, "q").standard_normal((B, Hq, D), dtype=np.float32), dtype)
    kr = store(rng_for(seed, "ring_k").standard_normal((B, Hkv, W, D), dtype=np.float32), dtype)
    vr = store(rng_for(seed, "ring_v").standard_normal((B, Hkv, W, D), dtype=np.float32), dtype)
    kn = store(rng_for(seed, "new_k").standard_normal((B, Hkv, D), dtype=np.float32), dtype)
    vn = store(rng_for(seed, "new_v").standard_normal((B, Hkv, D), dtype=np.float32), dtype)
    pos = np.asarray(pos, dtype=np.int32)
    for b in range(B):
        if pos[b] < W:
            kr[b, :, max(int(pos[b]) - 1, 0):, :] = np.nan
            vr[b, :, max(int(pos[b]) - 1, 0):, :] = np.nan
    return dict(q=q, k_ring=kr, v_ring=vr, k_new=kn, v_new=vn, pos=pos)


def gumbel_max_draw(logits: np.ndarray, r: np.random.Generator) -> np.ndarray:
    """One draw per row from softmax(logits) by the Gumbel-max construction: the argmax of
    logits + Gumbel(0,1) noise.  (Input generation only: this is how a draft model's sampler
    would pick x_i; the verify side never uses it.)"""
    u = r.random(logits.shape)
    u = np.clip(u, 1e-300, 1.0)
    gumbel = -np.log(-np.log(u))
    return np.argmax(logits.astype(np.float64) + gumbel, axis=-1).astype(np.int32)


def chain_sample_inputs(B: int, gamma: int, V: int, seed: int, target_sigma: float = 2.0,
                        draft_noise_sigma: float = 1.0, draft_corr: float = 0.0) -> dict:
    """target_logits [B, gamma+1, V], draft_logits [B, gamma, V] fp32, draft_tokens [B, gamma]
    drawn from the draft distributions, uniforms [B, gamma+1] in [0, 1) fp32."""
    z = rng_for(seed, "target").standard_normal((B, gamma + 1, V), dtype=np.float32)
    t = (target_sigma * z).astype(np.float32)
    eps = rng_for(seed, "draft").standard_normal((B, gamma, V), dtype=np.float32)
    if draft_corr > 0.0:
        d = target_sigma * (draft_corr * z[:, :gamma] + np.sqrt(1.0 - draft_corr ** 2) * eps)
    else:
        d = t[:, :gamma] + draft_noise_sigma * eps
    d = d.astype(np.float32)
    x = gumbel_max_draw(d, rng_for(seed, "gumbel"))
    u = rng_for(seed, "uniforms").random((B, gamma + 1), dtype=np.float32)
    return dict(target_logits=t, draft_logits=d, draft_tokens=x, uniforms=u)


def tree_sample_inputs(B: int, parent: np.ndarray, V: int, seed: int, target_sigma: float = 2.0,
                       p_match: float = 0.6, planted_logit: float = 30.0) -> dict:
    """target_logits [B, N, V] ~ N(0, sigma^2) and node_tokens [B, N].

    For each node with children, its first child's token is, with probability ``p_match``, a
    token whose logit in the parent's row is planted at ``planted_logit`` (far above any
    N(0, sigma^2) draw at these vocabulary sizes); the other children get random ids distinct
    from their siblings'."""
    N = len(parent)
    r = rng_for(seed, "tree_tok")
    t = (target_sigma * rng_for(seed, "target").standard_normal((B, N, V), dtype=np.float32)).astype(np.float32)
    tok = np.zeros((B, N), dtype=np.int32)
    children = [[] for _ in range(N)]
    for i in range(1, N):
        children[int(parent[i])].append(i)
    for b in range(B):
        tok[b, 0] = int(r.integers(V))
        for p in range(N):
            kids = children[p]
            if not kids:
                continue
            ids = r.choice(V, size=len(kids), replace=False).astype(np.int32)
            if r.random() < p_match:
                t[b, p, ids[0]] = np.float32(planted_logit)
            for c, tid in zip(kids, ids):
                tok[b, c] = tid
    return dict(target_logits=t, node_tokens=tok)


def tree_stochastic_inputs(B: int, parent: np.ndarray, V: int, seed: int, target_sigma: float = 2.0,
                           draft_corr: float = 0.8) -> dict:
    """Inputs of the stochastic tree step: target_logits, draft_logits [B, N, V] fp32 (draft
    correlated with target at ``draft_corr``), node_tokens [B, N] with each child's token drawn
    from its parent's draft row (Gumbel-max, i.i.d. per child; node 0's token is arbitrary),
    uniforms [B, N] in [0, 1) fp32."""
    N = len(parent)
    z = rng_for(seed, "target").standard_normal((B, N, V), dtype=np.float32)
    t = (target_sigma * z).astype(np.float32)
    eps = rng_for(seed, "draft").standard_normal((B, N, V), dtype=np.float32)
    d = (target_sigma * (draft_corr * z + np.sqrt(1.0 - draft_corr ** 2) * eps)).astype(np.float32)
    r = rng_for(seed, "tree_gumbel")
    tok = np.zeros((B, N), dtype=np.int32)
    for c in range(1, N):
        tok[:, c] = gumbel_max_draw(d[:, int(parent[c])], r)
    u = rng_for(seed, "uniforms").random((B, N), dtype=np.float32)
    return dict(target_logits=t, draft_logits=d, node_tokens=tok, uniforms=u)


def lmhead_inputs(B: int, R: int, d: int, V: int, seed: int, dtype: str = "bf16", plant: float = 0.6,
                  parent=None) -> dict:
    """Hidden states [B, R, d] ~ N(0, 1) and an LM-head weight [V, d] ~ N(0, 1/d) (stored as
    ``dtype``), with draft tokens [B, R] whose acceptance is non-trivial: with probability
    ``plant`` the token of row i + 1 (chain) or of each node's first child (tree, ``parent``
    given) gets a weight row proportional to the predecessor row's hidden state, which makes it
    that row's argmax."""
    r = rng_for(seed, "q")
    h = store(r.standard_normal((B, R, d), dtype=np.float32), dtype)
    w = rng_for(seed, "k").standard_normal((V, d), dtype=np.float32) / np.float32(np.sqrt(d))
    tok = rng_for(seed, "tokens").integers(0, V, size=(B, R)).astype(np.int32)
    pr = rng_for(seed, "tree_tok")
    used = set()
    if parent is not None:   # the first child of each node (planting siblings too would tie them)
        first = {}
        for c in range(1, R):
            first.setdefault(int(parent[c]), c)
        pairs = sorted((p_, c) for p_, c in first.items())
    else:
        pairs = [(i, i + 1) for i in range(R - 1)]
    for b in range(B):
        for src, dst in pairs:
            if pr.random() < plant:
                t = int(pr.integers(V))
                if t in used:
                    continue
                used.add(t)
                w[t] = h[b, src] * np.float32(3.0 / np.sqrt(d))
                tok[b, dst] = t
    return dict(hidden=h, weight=store(w, dtype), tokens=tok)


def lmhead_grid_inputs(B: int, R: int, d: int, V: int, seed: int, parent=None, plant: float = 0.85,
                       draft_sigma: float = 2.0) -> dict:
    """Inputs of the stochastic fused LM-head on an exact grid: every stored value is a small
    integer times a power of two, hidden = h_int * 2^-2 and weight = w_int * 2^-(s-2) with
    |h_int|, |w_int| <= 4 and s = floor(log2(4 sqrt(d))), so a logit is an integer times 2^-s of
    magnitude at most 16 d * 2^-s: every partial sum of a d-term dot product is exact in fp32
    (16 d < 2^24 for d <= 65 536), in any order.  The logits then spread about N(0, 1.7^2 .. 2.4^2).

    With probability ``plant`` the token of each chain row i + 1 (tree: each node's first child)
    is planted: a fresh vocabulary id whose weight row is +-4 on a random subset of coordinates
    (the signs of the source hidden row there, zero elsewhere) sized for a target logit near
    ln(V) + sigma_t^2 / 2 +- 2 (sigma_t the logits' spread), and whose draft logit in the source
    row is set near ln(V) + draft_sigma^2 / 2 +- 2, so that both distributions put real mass on
    it and the accept ratio spreads around 1.  Other draft
    tokens are drawn from their draft row by Gumbel-max.  Draft logits ~ N(0, draft_sigma^2)
    fp32.  Returns hidden [B, R, d], weight [V, d] (float32 holding bf16-exact values),
    draft_logits [B, R - 1 | R, V], tokens [B, R - 1 | R] (draft tokens; tree: node tokens with
    node 0's arbitrary), uniforms [B, R] (uniforms in [0, 1), fp32)."""
    s = int(np.floor(np.log2(4.0 * np.sqrt(d))))
    hi = rng_for(seed, "q").integers(-4, 5, size=(B, R, d), dtype=np.int8)
    wi = rng_for(seed, "k").integers(-4, 5, size=(V, d), dtype=np.int8)
    tree = parent is not None
    nd = R if tree else R - 1
    dl = (draft_sigma * rng_for(seed, "draft").standard_normal((B, nd, V), dtype=np.float32)).astype(np.float32)
    pr = rng_for(seed, "tree_tok")
    if tree:
        first = {}
        for c in range(1, R):
            first.setdefault(int(parent[c]), c)
        pairs = sorted((p_, c) for p_, c in first.items())
    else:
        pairs = [(i, i + 1) for i in range(R - 1)]
    planted = {}
    used = set()
    # ln V + sigma^2 / 2 is about the log of the softmax denominator of V N(0, sigma^2) logits
    sigma_t = (20.0 / 3.0) * np.sqrt(d) * 2.0 ** -s
    base_t, base_d = np.log(V) + sigma_t ** 2 / 2, np.log(V) + draft_sigma ** 2 / 2
    for b in range(B):
        for src, dst in pairs:
            if pr.random() >= plant:
                continue
            t = int(pr.integers(V))
            if t in used:
                continue
            used.add(t)
            # E|h_int| = 20/9: m coordinates at +-4 give a logit of about m * 4 * 20/9 * 2^-s
            want = base_t + pr.uniform(-2.0, 2.0)
            m = int(min(d, max(1, round(want * 2.0 ** s / (4.0 * 20.0 / 9.0)))))
            idx = pr.choice(d, size=m, replace=False)
            row = np.zeros(d, dtype=np.int8)
            row[idx] = 4 * np.sign(hi[b, src, idx]).astype(np.int8)
            wi[t] = row
            dl[b, src, t] = np.float32(base_d + pr.uniform(-2.0, 2.0))
            planted[(b, dst)] = t
    r = rng_for(seed, "gumbel")
    tok = np.zeros((B, nd), dtype=np.int32)
    for b in range(B):
        for j in range(nd):
            node = j if tree else j + 1          # the row whose token this is
            if tree and node == 0:
                tok[b, 0] = int(r.integers(V))
                continue
            src = int(parent[node]) if tree else node - 1
            if (b, node) in planted:
                tok[b, j] = planted[(b, node)]
            else:
                tok[b, j] = int(gumbel_max_draw(dl[b, src][None], r)[0])
    h = hi.astype(np.float32) * np.float32(0.25)
    w = np.empty((V, d), dtype=np.float32)
    step = 8192
    for v0 in range(0, V, step):
        w[v0:v0 + step] = wi[v0:v0 + step].astype(np.float32) * np.float32(2.0 ** -(s - 2))
    u = rng_for(seed, "uniforms").random((B, R), dtype=np.float32)
    return dict(hidden=h, weight=w, draft_logits=dl, tokens=tok, uniforms=u)
