"""Shared machinery of the GPU-vs-oracle parity tests.

Inputs come from the seeded generator (gen/), expected values from the
oracle (oracle/) only.  Where a CUDA stage needs an upstream result (a tree,
a mask), it is given the oracle's, so every stage is compared on identical
inputs; the end-to-end chain is checked separately.
"""
from dataclasses import dataclass, field

import numpy as np
import torch

import gen
from oracle import attn as oattn
from oracle import draft as odraft
from oracle import mask as omask
from oracle import tree as otree
from oracle import verify as over

CONF_RTOL = 1e-5          # softmax confidences, relative
LOGZ_TOL = 1e-5           # ln Z, relative to max(1, |ln Z|)
ATTN_TOL = {"bf16": 2e-2, "f32": 1e-4}   # absolute, against fp64
LSE_TOL = 1e-3


def f64(t):
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


@dataclass
class Case:
    w: gen.Workload
    oracle_seqs: list            # sequences the oracle computes fully
    attn_samples: object = None  # None = all outputs, else list of (b, i, h)
    attn_groups: list = field(default_factory=list)  # (b, KV head g): every node x grouped head compared
    device: str = "cuda"
    extra: dict = field(default_factory=dict)


def make_inputs(case):
    """Generate every input of the step for a case (on the case's device)."""
    w = case.w
    gen_dev = "cuda" if w.B * w.D * w.k * w.V > 50_000_000 else "cpu"
    draft = gen.draft_logits(w, device=gen_dev)
    return draft


def oracle_tree_stage(w, draft_cpu, seqs):
    """Oracle draft top-k + tree for the listed sequences."""
    tok = np.full((w.B, w.D, w.k, w.k), -1, dtype=np.int64)
    conf = np.zeros((w.B, w.D, w.k, w.k))
    stats = np.zeros((w.B, w.D, w.k, 2))
    trees = {}
    for b in seqs:
        t, c, s = odraft.draft_topk(draft_cpu[b:b + 1], w.k)
        tok[b], conf[b], stats[b] = t[0], c[0], s[0]
        c32 = np.nan_to_num(c[0]).astype(np.float32)
        trees[b] = otree.build_tree(t[0], c32, w.m, return_candidates=True)
        assert trees[b]["closure_added"] == []
    return tok, conf, stats, trees


def fill_trees(w, trees):
    """Node arrays [B, n] for every sequence; sequences the oracle did not
    build borrow a built tree (valid input for the later stages)."""
    keys = sorted(trees)
    out = {k_: np.zeros((w.B, w.n_nodes), dtype=np.int64) for k_ in ("tok", "parent", "row")}
    for b in range(w.B):
        t = trees[b] if b in trees else trees[keys[b % len(keys)]]
        out["tok"][b], out["parent"][b], out["row"][b] = t["tok"], t["parent"], t["row"]
    return out


def near_tie(tree, rel=1e-5):
    """True if two candidates near the selection boundaries of the oracle's
    build have scores within `rel` of each other (a float32 rounding of the
    confidences could then reorder them)."""
    C = tree["candidates"]
    vals = sorted((float(v) for v in C.score[1:]), reverse=True)
    vals = [v for v in vals if v > 0]
    for a, b in zip(vals, vals[1:]):
        if a - b <= rel * a:
            return True
    return False


def compare_draft(w, tok_g, conf_g, stats_g, tok_o, conf_o, stats_o, seqs):
    rows = odraft.used_rows(w.D, w.k)
    for b in seqs:
        for d, j in rows:
            assert (tok_g[b, d, j] == tok_o[b, d, j]).all(), (b, d, j)
            np.testing.assert_allclose(conf_g[b, d, j], conf_o[b, d, j], rtol=CONF_RTOL, atol=1e-30)
            assert stats_g[b, d, j, 0] == np.float32(stats_o[b, d, j, 0])
            lz = stats_o[b, d, j, 1]
            assert abs(stats_g[b, d, j, 1] - lz) <= LOGZ_TOL * max(1.0, abs(lz))


def compare_tree(got, want, mask_words=None):
    for key in ("tok", "parent", "depth", "src", "row"):
        assert (got[key] == want[key]).all(), key
    assert (got["score"] == want["score"]).all(), "score"
    if mask_words is not None:
        assert (mask_words == omask.pack_mask(omask.tree_mask(want["parent"]))).all(), "mask"


def attn_expected(case, ai_cpu, masks_bool):
    w = case.w
    scale = w.dh ** -0.5
    q, kc, vc = (f64(ai_cpu[k_]) for k_ in ("q", "k_cache", "v_cache"))
    kt, vt = f64(ai_cpu["k_tree"]), f64(ai_cpu["v_tree"])
    kv = ai_cpu["kv_len"].cpu().numpy()
    if case.attn_samples is None:
        return oattn.tree_attention(q, kc, vc, kv, kt, vt, masks_bool, scale)
    res = {}
    for (b, i, h) in case.attn_samples:
        res[(b, i, h)] = oattn.attention_row(q, kc, vc, kv, kt, vt, masks_bool, scale, b, i, h)
    return res


def check_walk(mode, acc_g, path_g, tok_g, acc_o, path_o, tok_o, r):
    """One sequence.  Greedy, and sampling without a flagged decision: exact.
    First flag at the bonus draw: path, accepted length and accepted tokens
    exact, the bonus one of the oracle's admissible tokens.  First flag at an
    accept test (two sides within 1e-5 of the row mass): exact up to that
    node.  Returns True when the comparison stopped at an accept test."""
    if mode == "greedy" or r.ambiguous is None:
        assert acc_g == acc_o, (acc_g, acc_o)
        assert (path_g == path_o).all()
        assert (tok_g == tok_o).all()
        return False
    pos = r.ambiguous[0]
    if r.ambiguous[1] == "bonus":
        assert acc_g == acc_o, (acc_g, acc_o)
        assert (path_g == path_o).all()
        assert (tok_g[:acc_o] == tok_o[:acc_o]).all()
        assert int(tok_g[acc_o]) in r.bonus_choices, (int(tok_g[acc_o]), r.bonus_choices)
        return False
    assert (path_g[:pos + 1] == path_o[:pos + 1]).all()
    return True


def compare_walk(w, mode, acc_g, path_g, tok_g, want, seqs):
    """Every sequence by check_walk; returns how many stopped at a flagged
    accept test."""
    acc_o, path_o, tok_o, walks = want
    n_amb = 0
    for b in seqs:
        try:
            n_amb += check_walk(mode, acc_g[b], path_g[b], tok_g[b], acc_o[b], path_o[b], tok_o[b], walks[b])
        except AssertionError as e:
            raise AssertionError(f"sequence {b}: {e}") from e
    return n_amb


def attn_group_expected(ai_cpu, masks_bool, b, g, G, scale):
    """The oracle's outputs for every (node, grouped head) of one sequence b
    and KV head g: out [n, G, dh] and lse [n, G]."""
    sl = slice(g * G, (g + 1) * G)
    q = f64(ai_cpu["q"][b:b + 1, :, sl])
    kc, vc = f64(ai_cpu["k_cache"][b:b + 1, g:g + 1]), f64(ai_cpu["v_cache"][b:b + 1, g:g + 1])
    kt, vt = f64(ai_cpu["k_tree"][b:b + 1, g:g + 1]), f64(ai_cpu["v_tree"][b:b + 1, g:g + 1])
    kv = ai_cpu["kv_len"].cpu().numpy()[b:b + 1]
    o, l = oattn.tree_attention(q, kc, vc, kv, kt, vt, masks_bool[b:b + 1], scale)
    return o[0], l[0]
