"""The five workload configurations, by what they are and their sizes.

Each entry restates one workload shape: attention head layout, KV dtype, batch, context-length
distribution, chain length gamma (or tree size), vocabulary and logit distributions.  Seeds are
1000 + the entry's index, with fixed sub-seed offsets per tensor (see ``workloads.gen``).
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Tuple


@dataclass(frozen=True)
class WorkloadConfig:
    name: str
    index: int
    # attention
    B: int
    Hq: int
    Hkv: int
    D: int
    kv_dtype: str               # "f32" or "bf16"
    ctx: Tuple[int, int]        # kv_len drawn uniformly from [lo, hi] (inclusive); includes the nq new tokens
    gamma: int                  # chain draft length (nq = gamma + 1); 0 for tree workloads
    tree_nodes: int = 0         # N for tree verify (0 = chain)
    tree_max_depth: int = 0
    tree_max_children: int = 0
    window: int = 0             # draft ring-buffer size W (0 = no draft-window attention)
    draft_steps: int = 0        # draft window calls per round
    # sampling
    vocab: int = 0
    target_sigma: float = 2.0   # target logits ~ N(0, sigma^2)
    draft_noise_sigma: float = 0.0   # draft = target + N(0, noise^2)
    draft_corr: float = 0.0     # if > 0: draft = sigma * (corr * z + sqrt(1 - corr^2) * eps)
    sample_mode: str = "chain"  # "chain" (stochastic) or "tree_greedy"

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def nq(self) -> int:
        return self.tree_nodes if self.tree_nodes else self.gamma + 1

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def kv_bytes(self) -> int:
        return 4 if self.kv_dtype == "f32" else 2


CONFIGS = {
    # batch 1, 4/1 heads, d64, fp32 N(0,1), context 512, gamma 4; vocab 1024, target N(0,2), draft noise N(0,0.5)
    "tiny": WorkloadConfig(
        name="tiny", index=0, B=1, Hq=4, Hkv=1, D=64, kv_dtype="f32", ctx=(512, 512), gamma=4,
        vocab=1024, target_sigma=2.0, draft_noise_sigma=0.5),
    # LLaMA-3-8B-shaped layer: 32/8 x 128 bf16, batch 8, context U[16K, 32K], gamma 4, vocab 128256
    "llama3-8b-layer": WorkloadConfig(
        name="llama3-8b-layer", index=1, B=8, Hq=32, Hkv=8, D=128, kv_dtype="bf16",
        ctx=(16384, 32768), gamma=4, vocab=128256, target_sigma=2.0, draft_noise_sigma=1.0),
    # MagicDec long context: batch 32, context 64K, gamma 4 verify + 4 draft steps over a 512 ring
    "magicdec-64k": WorkloadConfig(
        name="magicdec-64k", index=2, B=32, Hq=32, Hkv=8, D=128, kv_dtype="bf16",
        ctx=(65536, 65536), gamma=4, window=512, draft_steps=4, vocab=128256,
        target_sigma=2.0, draft_noise_sigma=1.0),
    # Medusa-style tree: batch 4, context 8K incl. a 64-node tree (depth <= 4, branching <= 8), vocab 32000
    "medusa-tree-8k": WorkloadConfig(
        name="medusa-tree-8k", index=3, B=4, Hq=32, Hkv=8, D=128, kv_dtype="bf16",
        ctx=(8192, 8192), gamma=0, tree_nodes=64, tree_max_depth=4, tree_max_children=8,
        vocab=32000, target_sigma=2.0, sample_mode="tree_greedy"),
    # LLaMA-3-70B-shaped layer: 64/8 x 128 bf16, batch 16, context U[64K, 128K], gamma 6, corr 0.8 draft
    "llama3-70b-layer": WorkloadConfig(
        name="llama3-70b-layer", index=4, B=16, Hq=64, Hkv=8, D=128, kv_dtype="bf16",
        ctx=(65536, 131072), gamma=6, vocab=128256, target_sigma=2.0, draft_corr=0.8),
}


def get_config(name: str) -> WorkloadConfig:
    try:
        return CONFIGS[name]
    except KeyError as e:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(CONFIGS)}") from e


def scaled(cfg: WorkloadConfig, *, B: Optional[int] = None, ctx: Optional[Tuple[int, int]] = None,
           vocab: Optional[int] = None, **kw) -> WorkloadConfig:
    """A copy of ``cfg`` with smaller sizes (same heads, dtype, distributions) for oracle-sized tests."""
    d = dict(cfg.__dict__)
    if B is not None:
        d["B"] = B
    if ctx is not None:
        d["ctx"] = ctx
    if vocab is not None:
        d["vocab"] = vocab
    d.update(kw)
    return WorkloadConfig(**d)
