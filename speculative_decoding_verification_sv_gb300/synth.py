"""Seeded synthetic inputs for the verify step, shaped like Qwen2.5-1.5B / 7B.

This module only draws random tensors and builds token trees; it holds none
of the verify step's arithmetic, and both the CUDA path (benchmark, tests) and
the CPU oracle (tests) take their inputs from it.

Workloads (one verify round each):
  0  1.5B shapes, 1 layer, t=2048, k=4, batch 1, greedy (acceptance planted at 0.55)
  1  1.5B shapes, 28 layers, t=4096, k=4, batch 1, greedy (planted at 0.52)
  2  sampled acceptance alone: batch 64, k=8, vocab 151936, temperature 1
  3  7B shapes, 28 layers, t=8192, k=8, batch 1 and 16, greedy and sampled
  4  7B shapes, token tree of 64 draft nodes, depth 8, branching 1..3, t=8192

Value distributions: Q, K/V cache, block K/V and hidden rows ~ N(0, 1) in bf16;
LM-head weights ~ N(0, 0.02^2) in bf16; sampled-mode target logits ~ N(0, 3^2)
in fp32; draft probabilities q = softmax(target logits + N(0, 1)); sampled
drafts are drawn from q.  Greedy drafts are planted: draft j equals the
argmax of its verifying row with the stated probability, else a uniformly
drawn different id.  Seeds: 0x53560000 + 16 * workload + tensor id.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np
import torch

SEED_BASE = 0x53560000


@dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    L: int            # layers
    B: int            # sequences
    Hq: int
    Hkv: int
    D: int
    H: int            # hidden size (LM-head input)
    V: int            # target vocab
    t: int            # committed context length
    k: int            # drafts per round (chain); tree: draft nodes
    mode: str         # "greedy" | "sampled"
    accept_rate: float = 0.55
    temperature: float = 1.0
    tree: bool = False
    tree_depth: int = 0
    Vq: Optional[int] = None   # draft vocab (<= V); None means V

    @property
    def R(self) -> int:
        return self.k + 1

    @property
    def T_cap(self) -> int:
        return ((self.t + self.R + 63) // 64) * 64 + 64

    @property
    def draft_vocab(self) -> int:
        return self.Vq if self.Vq is not None else self.V


QWEN15 = dict(Hq=12, Hkv=2, D=128, H=1536, V=151936)
QWEN7 = dict(Hq=28, Hkv=4, D=128, H=3584, V=152064)

WORKLOADS = {
    0: Workload(0, "qwen2.5-1.5b 1-layer verify t=2048 k=4 b=1 greedy", L=1, B=1, t=2048, k=4,
                mode="greedy", accept_rate=0.55, **QWEN15),
    1: Workload(1, "qwen2.5-1.5b 28-layer verify t=4096 k=4 b=1 greedy", L=28, B=1, t=4096, k=4,
                mode="greedy", accept_rate=0.52, **QWEN15),
    2: Workload(2, "sampled acceptance b=64 k=8 V=151936 T=1", L=0, B=64, Hq=0, Hkv=0, D=0, H=0,
                V=151936, t=0, k=8, mode="sampled"),
    3: Workload(3, "qwen2.5-7b 28-layer verify t=8192 k=8 b=1 greedy", L=28, B=1, t=8192, k=8,
                mode="greedy", accept_rate=0.55, **QWEN7),
    4: Workload(4, "qwen2.5-7b tree verify 64 nodes depth 8 t=8192 b=1 greedy", L=28, B=1, t=8192,
                k=64, mode="greedy", accept_rate=0.55, tree=True, tree_depth=8, **QWEN7),
}


def workload(wid: int, **overrides) -> Workload:
    w = WORKLOADS[wid]
    if not overrides:
        return w
    w = replace(w, **overrides)
    if "B" in overrides:   # keep the name true to the batch
        import re
        w = replace(w, name=re.sub(r"\bb=\d+", f"b={w.B}", w.name))
    return w


def seed_for(wid: int, tensor_id: int) -> int:
    return SEED_BASE + 16 * wid + tensor_id


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn_bf16(shape, seed: int, device="cpu", std: float = 1.0) -> torch.Tensor:
    g = _gen(device, seed)
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


# ----------------------------------------------------------------------------
# attention / KV inputs
# ----------------------------------------------------------------------------

@dataclass
class AttnInputs:
    q: torch.Tensor        # [L, B, R, Hq, D] bf16
    k_cache: torch.Tensor  # [L, B, Hkv, T_cap, D] bf16
    v_cache: torch.Tensor
    k_blk: torch.Tensor    # [L, B, Hkv, R, D] bf16
    v_blk: torch.Tensor
    length: torch.Tensor   # [B] int32 committed length t
    parent: Optional[torch.Tensor] = None  # [B, R] int32 (tree) or None (chain)


def attn_inputs(w: Workload, device="cpu", layers: Optional[int] = None, lengths=None,
                parent: Optional[torch.Tensor] = None) -> AttnInputs:
    L = w.L if layers is None else layers
    R, T_cap = w.R, w.T_cap
    q = randn_bf16((L, w.B, R, w.Hq, w.D), seed_for(w.wid, 1), device)
    kc = randn_bf16((L, w.B, w.Hkv, T_cap, w.D), seed_for(w.wid, 2), device)
    vc = randn_bf16((L, w.B, w.Hkv, T_cap, w.D), seed_for(w.wid, 3), device)
    kb = randn_bf16((L, w.B, w.Hkv, R, w.D), seed_for(w.wid, 4), device)
    vb = randn_bf16((L, w.B, w.Hkv, R, w.D), seed_for(w.wid, 5), device)
    if lengths is None:
        lengths = [w.t] * w.B
    ln = torch.tensor(lengths, dtype=torch.int32, device=device)
    return AttnInputs(q, kc, vc, kb, vb, ln, parent)


# ----------------------------------------------------------------------------
# LM head inputs
# ----------------------------------------------------------------------------

def lm_inputs(w: Workload, device="cpu", n_rows: Optional[int] = None):
    N = w.B * w.R if n_rows is None else n_rows
    hid = randn_bf16((N, w.H), seed_for(w.wid, 6), device)
    W = randn_bf16((w.H, w.V), seed_for(w.wid, 7), device, std=0.02)
    return hid, W


# ----------------------------------------------------------------------------
# drafts
# ----------------------------------------------------------------------------

def plant_chain_drafts(argmax_rows: np.ndarray, rate: float, V: int, seed: int,
                       pending: Optional[np.ndarray] = None) -> np.ndarray:
    """argmax_rows [B, R]: the argmax of every verify row (computed by the
    caller).  Returns tok [B, R]: tok[:, 0] the pending token, tok[:, j] = draft
    j, equal to argmax_rows[:, j-1] with probability `rate`, else a different
    uniformly drawn id."""
    rng = np.random.default_rng(seed)
    B, R = argmax_rows.shape
    tok = np.zeros((B, R), np.int32)
    tok[:, 0] = rng.integers(0, V, size=B) if pending is None else pending
    for b in range(B):
        for j in range(1, R):
            g = int(argmax_rows[b, j - 1])
            if rng.random() < rate:
                tok[b, j] = g
            else:
                x = int(rng.integers(0, V - 1))
                tok[b, j] = x if x < g else x + 1
    return tok


def plant_tree_drafts(argmax_rows: np.ndarray, parent: np.ndarray, rate: float, V: int,
                      seed: int) -> np.ndarray:
    """Tree version: node c's token equals the argmax of its parent's row with
    probability `rate`, else a different uniform id."""
    rng = np.random.default_rng(seed)
    B, R = argmax_rows.shape
    tok = np.zeros((B, R), np.int32)
    tok[:, 0] = rng.integers(0, V, size=B)
    for b in range(B):
        for c in range(1, R):
            g = int(argmax_rows[b, parent[b, c]])
            if rng.random() < rate:
                tok[b, c] = g
            else:
                x = int(rng.integers(0, V - 1))
                tok[b, c] = x if x < g else x + 1
    return tok


def random_tree(n_nodes: int, depth: int, max_children: int, seed: int) -> np.ndarray:
    """Random draft tree over n_nodes drafts plus the root: a spine of length
    `depth`, then children attached to uniformly chosen nodes of depth < depth
    with fewer than max_children children, relabelled in breadth-first order.
    Returns parent [n_nodes + 1] with parent[0] = -1 and parent[c] < c."""
    assert n_nodes >= depth
    rng = np.random.default_rng(seed)
    par = [-1]
    dep = [0]
    kids = [0]
    for i in range(1, depth + 1):   # spine
        par.append(i - 1)
        dep.append(i)
        kids.append(0)
        kids[i - 1] += 1
    while len(par) < n_nodes + 1:
        cand = [u for u in range(len(par)) if dep[u] < depth and kids[u] < max_children]
        u = int(cand[int(rng.integers(0, len(cand)))])
        par.append(u)
        dep.append(dep[u] + 1)
        kids.append(0)
        kids[u] += 1
    # breadth-first relabelling (children in creation order)
    order = [0]
    head = 0
    children = [[] for _ in par]
    for c in range(1, len(par)):
        children[par[c]].append(c)
    while head < len(order):
        order.extend(children[order[head]])
        head += 1
    new_id = {old: i for i, old in enumerate(order)}
    out = np.full(len(par), -1, np.int32)
    for old, new in new_id.items():
        out[new] = -1 if par[old] < 0 else new_id[par[old]]
    return out


def tree_depths(parent: np.ndarray) -> np.ndarray:
    d = np.zeros(len(parent), np.int32)
    for c in range(1, len(parent)):
        d[c] = d[parent[c]] + 1
    return d


# ----------------------------------------------------------------------------
# sampled-acceptance inputs
# ----------------------------------------------------------------------------

@dataclass
class SampleInputs:
    logits: torch.Tensor   # [B, R, V] fp32
    q: torch.Tensor        # [B, Rq, Vq] fp32
    tok: torch.Tensor      # [B, R] int32
    parent: Optional[torch.Tensor] = None


def sample_inputs(B: int, k: int, V: int, wid: int = 2, device="cpu", Vq: Optional[int] = None,
                  logit_std: float = 3.0, parent: Optional[np.ndarray] = None,
                  logits: Optional[torch.Tensor] = None) -> SampleInputs:
    """Target logits ~ N(0, logit_std^2) (unless given); q rows =
    softmax(logits + N(0, 1)) truncated to the draft vocab Vq and
    renormalised; drafts drawn from q with their own generator.  Chain:
    q has k rows (row u proposes draft u+1); tree (parent [R] given, shared by
    all sequences): q has R rows and the children of node u are drawn
    i.i.d. from q row u."""
    Vq = V if Vq is None else Vq
    R = k + 1 if parent is None else len(parent)
    if logits is None:
        g = _gen(device, seed_for(wid, 8))
        logits = torch.randn(B, R, V, generator=g, device=device, dtype=torch.float32) * logit_std
    g2 = _gen(device, seed_for(wid, 9))
    Rq = R - 1 if parent is None else R
    noisy = logits[:, :Rq, :Vq].float() + torch.randn(B, Rq, Vq, generator=g2, device=device,
                                                      dtype=torch.float32)
    q = torch.softmax(noisy, dim=-1).contiguous()
    g3 = _gen(device, seed_for(wid, 10))
    tok = torch.zeros(B, R, dtype=torch.int32, device=device)
    tok[:, 0] = torch.randint(0, V, (B,), generator=g3, device=device, dtype=torch.int32)
    if parent is None:
        if Rq > 0:
            draws = torch.multinomial(q.reshape(B * Rq, Vq), 1, generator=g3).reshape(B, Rq)
            tok[:, 1:] = draws.to(torch.int32)
        par_t = None
    else:
        draws = torch.multinomial(q.reshape(B * Rq, Vq), R, replacement=True,
                                  generator=g3).reshape(B, Rq, R)
        for c in range(1, R):
            tok[:, c] = draws[:, int(parent[c]), c].to(torch.int32)
        par_t = torch.tensor(np.tile(parent, (B, 1)), dtype=torch.int32, device=device)
    return SampleInputs(logits.contiguous(), q, tok, par_t)


# ----------------------------------------------------------------------------
# conversions used by both sides' callers
# ----------------------------------------------------------------------------

def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a tensor, as numpy uint16 (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
