"""Seeded synthetic workloads for one tree-speculative decoding step.

This module only draws numbers and moves them into place; it holds none of
the step's arithmetic (no softmax, top-k, scoring, masking, attention or
acceptance rule).  Both the CUDA path and the oracle consume what it makes.

The shapes follow the settings the EAGLE explainers describe: k=10 expanded
nodes, depth 6, m = 60 / 50 / 48 draft tokens for 7B / 13B / 70B targets
(EAGLE-2 explainer, section "動的ドラフトツリーの構築アルゴリズム" and the
vLLM settings paragraph), a GPT-OSS-20B-shaped high-concurrency setting at
depth 7 and c=64 (P-EAGLE note, sections on benchmarks and speculation
depth), plus a tiny case small enough for the fp64 oracle to check every
output.  No model weights or datasets exist here; draft and target logits,
queries and KV are random with the distributions below.

Draft row (one per [b, d, j]):  logit[t] = 4 * z_t - ln(rank(t) + 1), with
z ~ N(0, 1) i.i.d. and rank a per-row random permutation of the vocabulary,
so every row has a heavy head and a long tail, like a language model's.

Target row i (the target model's distribution after tree node i): the draft
row that node i was expanded with, plus sigma * N(0, 1) noise, when node i was
expanded; otherwise a fresh draft-distributed row plus the same noise.  Which
draft row belongs to which node is decided by the tree, so the caller passes
that map (`node_row`, -1 where the node was not expanded) in; this module only
gathers rows by it.
"""
from dataclasses import dataclass, field
import math

import numpy as np
import torch

from .philox import tree_uniforms


@dataclass(frozen=True)
class Workload:
    name: str
    B: int            # independent sequences
    V: int            # vocabulary
    D: int            # maximum tree depth
    k: int            # expansion width (top-k per node, top-k frontier)
    m: int            # draft tokens kept by the rerank (tree size without root)
    Hq: int           # query heads
    Hkv: int          # key/value heads
    dh: int           # head dimension
    L: int            # KV prefix length (max when ragged)
    L_min: int        # ragged prefixes: kv_len ~ U[L_min, L]; equal to L if fixed
    dtype: str        # "f32" or "bf16"
    sigma: float      # target noise scale
    modes: tuple      # verification modes exercised ("greedy", "sample")
    seed: int
    temperature: float = 1.0

    @property
    def n_nodes(self):
        return self.m + 1

    @property
    def n_candidates(self):
        return self.k + (self.D - 1) * self.k * self.k

    @property
    def rows_used(self):
        return 1 + (self.D - 1) * self.k

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


WORKLOADS = {
    "tiny": Workload("tiny", B=1, V=1000, D=3, k=4, m=10, Hq=4, Hkv=4, dh=64,
                     L=128, L_min=128, dtype="f32", sigma=0.5,
                     modes=("greedy", "sample"), seed=1000),
    "llama2-7b-b1": Workload("llama2-7b-b1", B=1, V=32000, D=6, k=10, m=60,
                             Hq=32, Hkv=32, dh=128, L=2048, L_min=2048,
                             dtype="bf16", sigma=0.5, modes=("greedy",), seed=1001),
    "llama2-13b-b8": Workload("llama2-13b-b8", B=8, V=32000, D=6, k=10, m=50,
                              Hq=40, Hkv=40, dh=128, L=4096, L_min=1024,
                              dtype="bf16", sigma=0.5, modes=("sample",), seed=1002),
    "llama2-70b-b16": Workload("llama2-70b-b16", B=16, V=32000, D=6, k=10, m=48,
                               Hq=64, Hkv=8, dh=128, L=4096, L_min=4096,
                               dtype="bf16", sigma=1.0, modes=("greedy", "sample"),
                               seed=1003),
    "gpt-oss-20b-b64": Workload("gpt-oss-20b-b64", B=64, V=201088, D=7, k=10, m=60,
                                Hq=64, Hkv=8, dh=64, L=8192, L_min=8192,
                                dtype="bf16", sigma=0.5, modes=("sample",), seed=1004),
}


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draft_like_rows(n_rows, V, seed, device="cpu", dtype=torch.float32,
                    row_block=256):
    """n_rows rows of 4*z - ln(rank+1), returned as `dtype` [n_rows, V].

    The values are computed in float32 and rounded once to `dtype`.
    """
    out = torch.empty((n_rows, V), dtype=dtype, device=device)
    g = _gen(seed, device)
    for r0 in range(0, n_rows, row_block):
        r1 = min(n_rows, r0 + row_block)
        z = torch.randn((r1 - r0, V), generator=g, device=device, dtype=torch.float32)
        rank = torch.argsort(torch.rand((r1 - r0, V), generator=g, device=device), dim=1)
        bias = torch.log1p(rank.to(torch.float32))
        out[r0:r1] = (4.0 * z - bias).to(dtype)
        del z, rank, bias
    return out


def draft_logits(w: Workload, device="cpu"):
    """Draft logits [B, D, k, V] in the workload's dtype.

    Row [b, d, j] is the draft head's output for the j-th expanded node of
    layer d of sequence b; row [b, 0, 0] is the root's.  Rows [b, 0, 1..k-1]
    are never read by the step and are filled like the others.
    """
    rows = draft_like_rows(w.B * w.D * w.k, w.V, w.seed, device, w.torch_dtype)
    return rows.view(w.B, w.D, w.k, w.V)


def target_logits(w: Workload, draft, node_row, device="cpu"):
    """Target logits [B, m+1, V] in the workload's dtype.

    node_row: int [B, m+1]; node_row[b, i] = d*k + j if tree node i was
    expanded with draft row [b, d, j], else -1.  Row i becomes that draft row
    (or a fresh draft-like row) plus sigma * N(0, 1), rounded once.
    """
    n = w.n_nodes
    node_row = torch.as_tensor(np.asarray(node_row), dtype=torch.int64, device=device)
    assert node_row.shape == (w.B, n)
    fresh = draft_like_rows(w.B * n, w.V, w.seed + 7919, device, torch.float32).view(w.B, n, w.V)
    g = _gen(w.seed + 104729, device)
    out = torch.empty((w.B, n, w.V), dtype=w.torch_dtype, device=device)
    flat = draft.reshape(w.B, w.D * w.k, w.V)
    for b in range(w.B):
        noise = torch.randn((n, w.V), generator=g, device=device, dtype=torch.float32)
        base = fresh[b].clone()
        has = node_row[b] >= 0
        if bool(has.any()):
            base[has] = flat[b, node_row[b][has]].to(torch.float32)
        out[b] = (base + w.sigma * noise).to(w.torch_dtype)
    return out


def kv_lengths(w: Workload):
    """Per-sequence prefix lengths, int32 [B]; U[L_min, L] when ragged."""
    if w.L_min == w.L:
        return np.full(w.B, w.L, dtype=np.int32)
    rng = np.random.default_rng(w.seed + 31)
    return rng.integers(w.L_min, w.L + 1, size=w.B).astype(np.int32)


def attention_inputs(w: Workload, device="cpu"):
    """Queries, KV prefix cache and tree KV, all N(0, 1) in the workload dtype.

    q       [B, m+1, Hq, dh]   one query per tree node (root = node 0)
    k_cache [B, Hkv, L, dh]    prefix keys; positions >= kv_len[b] are unused
    v_cache [B, Hkv, L, dh]
    k_tree  [B, Hkv, m+1, dh]  keys/values of the tree nodes themselves
    v_tree  [B, Hkv, m+1, dh]
    kv_len  int32 [B]
    """
    g = _gen(w.seed + 65537, device)
    n = w.n_nodes
    dt = w.torch_dtype

    def randn(*shape):
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(dt)

    q = randn(w.B, n, w.Hq, w.dh)
    k_cache = randn(w.B, w.Hkv, w.L, w.dh)
    v_cache = randn(w.B, w.Hkv, w.L, w.dh)
    k_tree = randn(w.B, w.Hkv, n, w.dh)
    v_tree = randn(w.B, w.Hkv, n, w.dh)
    kv_len = torch.as_tensor(kv_lengths(w), device=device)
    return dict(q=q, k_cache=k_cache, v_cache=v_cache, k_tree=k_tree,
                v_tree=v_tree, kv_len=kv_len)


def uniforms(w: Workload):
    """Verification uniforms, float32 [B, m+1, 2], from Philox4x32-10."""
    return tree_uniforms(w.seed, w.B, w.n_nodes)


def scaled(w: Workload, **changes):
    """A copy of a workload with some sizes changed (for small test cases)."""
    d = dict(w.__dict__)
    d.update(changes)
    return Workload(**d)


# ---------------------------------------------------------------------------
# static draft-tree templates (the EAGLE-1 style fixed tree is an input: the
# pages say only that it is chosen offline and applied to every input)
# ---------------------------------------------------------------------------

# A synthetic 60-node template for D = 6, k = 10: per depth, the number of
# children of that depth's nodes in node order (later nodes get none).
STATIC_SHAPE_60 = ([10], [5, 4, 3, 2, 1], [4, 3, 3, 2, 2, 1, 1, 1], [3, 2, 2, 1, 1, 1, 1],
                   [2, 1, 1, 1, 1], [1])


def static_template(shape=STATIC_SHAPE_60):
    """(parent, rank) int32 arrays of a template built from `shape`:
    shape[d][j] children (ranks 0..c-1) for the j-th node of depth d."""
    parent, rank = [-1], [0]
    level = [0]
    for counts in shape:
        nxt = []
        for j, c in enumerate(counts):
            for r in range(c):
                parent.append(level[j])
                rank.append(r)
                nxt.append(len(parent) - 1)
        level = nxt
    return np.array(parent, dtype=np.int32), np.array(rank, dtype=np.int32)
