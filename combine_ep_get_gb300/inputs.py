"""Seeded synthetic inputs for MoE token dispatch / combine.

This module draws inputs only; it holds none of the method's arithmetic (no
routing layout, no copies, no casts of the method, no reductions).  It is the
one module that both the CUDA path's tests/benchmark and the CPU oracle's
tests use.

Every array comes from ``numpy.random.Generator(PCG64(seed))``:

* ``x``: standard normal fp32 rounded to bf16 (torch's CPU cast, ties to
  even), returned as uint16 bit patterns [T, H];
* ``topk_idx``: int64 [T, K], K distinct experts per token, drawn by
  Gumbel-top-k (``argsort`` of random keys), with -1 for masked entries;
* ``topk_weights``: fp32 softmax of standard-normal logits [T, K].

Routing recipes (the workload shapes):

* ``uniform``: K distinct experts uniform over E;
* ``zipf``: K distinct experts without replacement from popularity
  p_i ~ i^-s over a seeded permutation of the experts (Gumbel-top-k on log p);
* ``node_limited``: per token ``max_nodes`` distinct node groups uniform over
  R / ranks_per_node, then K distinct experts uniform among those groups'
  experts.

``mask_frac`` sets exactly floor(mask_frac * T * K) entries, chosen uniformly
without replacement, to -1.
"""
from dataclasses import dataclass
import numpy as np


@dataclass(frozen=True)
class Config:
    name: str
    T: int
    H: int
    E: int
    K: int
    R: int
    seed: int
    routing: str = "uniform"
    zipf_s: float = 1.2
    mask_frac: float = 0.0
    ranks_per_node: int = 0
    max_nodes: int = 0
    fp8: bool = False
    weighted: bool = False
    description: str = ""


# The five workloads: small parity case, DeepSeek-V3-shaped prefill, skewed
# routing, FP8 decode, large node-limited (hierarchical) routing.
CONFIGS = {
    "tiny": Config("tiny", T=128, H=256, E=16, K=4, R=4, seed=0,
                   description="T=128 H=256 E=16 K=4 R=4 uniform, identity expert"),
    "dsv3": Config("dsv3", T=4096, H=7168, E=256, K=8, R=8, seed=1,
                   description="DeepSeek-V3-shaped prefill T=4096 H=7168 E=256 K=8 R=8 bf16"),
    "skewed": Config("skewed", T=8192, H=7168, E=256, K=8, R=16, seed=2, routing="zipf",
                     zipf_s=1.2, mask_frac=0.05,
                     description="T=8192 H=7168 E=256 K=8 R=16 Zipf(1.2) routing, 5% masked"),
    "decode": Config("decode", T=128, H=7168, E=256, K=8, R=32, seed=3, fp8=True, weighted=True,
                     description="decode T=128 H=7168 E=256 K=8 R=32 FP8 dispatch, weighted combine"),
    "large": Config("large", T=32768, H=7168, E=256, K=8, R=64, seed=4, routing="node_limited",
                    ranks_per_node=8, max_nodes=4,
                    description="T=32768 H=7168 E=256 K=8 R=64, 8 ranks/node, <=4 nodes/token"),
}


def _bf16_bits(a32: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _softmax32(logits: np.ndarray) -> np.ndarray:
    m = logits.max(axis=1, keepdims=True)
    ex = np.exp(logits - m, dtype=np.float32)
    return (ex / ex.sum(axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)


def draw_topk(rng: np.random.Generator, T: int, E: int, K: int, routing: str = "uniform",
              zipf_s: float = 1.2, R: int = 1, ranks_per_node: int = 0,
              max_nodes: int = 0) -> np.ndarray:
    if T == 0:
        return np.zeros((0, K), np.int64)
    if routing == "uniform":
        keys = rng.random((T, E))
        return np.argsort(keys, axis=1, kind="stable")[:, :K].astype(np.int64)
    if routing == "zipf":
        perm = rng.permutation(E)
        p = np.arange(1, E + 1, dtype=np.float64) ** (-zipf_s)
        logp = np.empty(E)
        logp[perm] = np.log(p / p.sum())
        g = rng.gumbel(size=(T, E))
        keys = logp[None, :] + g
        return np.argsort(-keys, axis=1, kind="stable")[:, :K].astype(np.int64)
    if routing == "node_limited":
        nodes = R // ranks_per_node
        per_node = E // nodes
        node_keys = rng.random((T, nodes))
        chosen = np.argsort(node_keys, axis=1, kind="stable")[:, :max_nodes]      # [T, max_nodes]
        cand_keys = rng.random((T, max_nodes * per_node))
        pick = np.argsort(cand_keys, axis=1, kind="stable")[:, :K]              # [T, K]
        node_of = np.take_along_axis(chosen, pick // per_node, axis=1)
        return (node_of * per_node + pick % per_node).astype(np.int64)
    raise ValueError(routing)


def make_inputs(T: int, H: int, E: int, K: int, R: int, seed: int, routing: str = "uniform",
                zipf_s: float = 1.2, mask_frac: float = 0.0, ranks_per_node: int = 0,
                max_nodes: int = 0, with_x: bool = True) -> dict:
    rng = np.random.Generator(np.random.PCG64(seed))
    topk_idx = draw_topk(rng, T, E, K, routing, zipf_s, R, ranks_per_node, max_nodes)
    if mask_frac > 0 and T > 0:
        n_mask = int(np.floor(mask_frac * T * K))
        flat = rng.choice(T * K, size=n_mask, replace=False)
        topk_idx.reshape(-1)[flat] = -1
    logits = rng.standard_normal((T, K), dtype=np.float32)
    topk_weights = _softmax32(logits) if T > 0 else np.zeros((0, K), np.float32)
    out = dict(topk_idx=np.ascontiguousarray(topk_idx), topk_weights=topk_weights)
    if with_x:
        x32 = rng.standard_normal((T, H), dtype=np.float32)
        out["x_bits"] = _bf16_bits(x32)
    return out


def make_config(cfg, with_x: bool = True) -> dict:
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    d = make_inputs(cfg.T, cfg.H, cfg.E, cfg.K, cfg.R, cfg.seed, cfg.routing, cfg.zipf_s,
                    cfg.mask_frac, cfg.ranks_per_node, cfg.max_nodes, with_x=with_x)
    d["cfg"] = cfg
    return d


def make_rows(n: int, H: int, seed: int) -> np.ndarray:
    """Standard-normal bf16 rows [n, H] (uint16 bits): a stand-in expert output."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return _bf16_bits(rng.standard_normal((n, H), dtype=np.float32))
