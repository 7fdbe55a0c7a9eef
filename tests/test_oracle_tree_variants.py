"""Pins for the oracle's ablation variants of the tree build.

[EAGLE-2] section "実験結果" (ablation table): "without the global acceptance
probability (confidence only)" and "without reranking".  Independent checks:
  * a tree worked by hand for each variant (tests/golden/hand_ablation.json),
    chosen so the four variants give four different trees;
  * best-first growth with V keys (written here, over the oracle's candidate
    table) reproduces the full method's top-m set and order, which is what
    makes the confidence-only rerank a generalisation of the full method;
  * without rerank, each depth's nodes are exactly that depth's k best keys;
  * node scores: the node's own confidence (confidence only) or the float32
    product along the root path (full);
  * structure: connected, parents first, |tree| = m+1, expanded parents.
"""
import json
import os

import numpy as np
import pytest

import gen
from oracle import draft as odraft
from oracle import tree as otree

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def hand():
    with open(os.path.join(GOLDEN, "hand_ablation.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("case", [c["name"] for c in hand()["cases"]])
def test_hand_worked_variants(case):
    h = hand()
    c = next(x for x in h["cases"] if x["name"] == case)
    out = otree.build_tree(np.array(h["tok"]), np.array(h["conf"], dtype=np.float32), c["m"], -1,
                           confidence_only=c["confidence_only"], rerank=c["rerank"])
    for key in ("tok", "parent", "depth", "src", "row"):
        assert list(out[key]) == c[key], key
    assert out["closure_added"] == []


def random_rows(seed, D=4, k=4, V=300):
    """Draft-like rows through the oracle's stage 1, as the step feeds stage 2."""
    w = gen.scaled(gen.WORKLOADS["tiny"], B=1, D=D, k=k, V=V, m=min(3 * k, k + (D - 1) * k * k), seed=seed)
    logits = gen.draft_logits(w).float().numpy()
    tok, conf, _ = odraft.draft_topk(logits, k)
    conf = np.where(np.isnan(conf), 0.0, conf).astype(np.float32)
    return tok[0], conf[0]


def path_product(out, tok, conf, i):
    v = np.float32(1.0)
    chain = []
    j = i
    while j > 0:
        chain.append(j)
        j = out["parent"][j]
    for j in reversed(chain):
        v = otree.fl32_mul(v, own_conf(out, tok, conf, j))
    return v


def own_conf(out, tok, conf, i):
    p = out["parent"][i]
    d, j = divmod(int(out["row"][p]), tok.shape[1])
    r = list(tok[d, j]).index(out["tok"][i])
    return conf[d, j, r]


def check_structure(out, m):
    par, dep = out["parent"], out["depth"]
    assert len(par) == m + 1 and par[0] == -1 and dep[0] == 0
    for i in range(1, m + 1):
        assert 0 <= par[i] < i
        assert dep[i] == dep[par[i]] + 1
        assert out["row"][par[i]] >= 0, "a parent must have been expanded"
    assert len(set(int(s) for s in out["src"])) == m + 1


@pytest.mark.parametrize("seed", [11, 12, 13, 14])
@pytest.mark.parametrize("conf_only,rerank", [(False, True), (True, True), (False, False), (True, False)])
def test_variant_structure_and_scores(seed, conf_only, rerank):
    tok, conf = random_rows(seed)
    D, k = tok.shape[0], tok.shape[1]
    m = 3 * k if rerank else D * k - 1
    out = otree.build_tree(tok, conf, m, -1, confidence_only=conf_only, rerank=rerank)
    check_structure(out, m)
    for i in range(1, m + 1):
        want = own_conf(out, tok, conf, i) if conf_only else path_product(out, tok, conf, i)
        assert out["score"][i] == np.float32(want)


@pytest.mark.parametrize("seed", [21, 22, 23])
def test_best_first_with_v_keys_is_top_m(seed):
    tok, conf = random_rows(seed)
    k = tok.shape[1]
    m = 3 * k
    full = otree.build_tree(tok, conf, m, -1, return_candidates=True)
    C = full["candidates"]
    inside, picks = {0}, []
    for _ in range(m):
        best = None
        for g in range(1, len(C)):
            if g in inside or C.parent[g] not in inside:
                continue
            if best is None or C.key(g) < C.key(best):
                best = g
        picks.append(best)
        inside.add(best)
    assert [0] + picks == list(full["src"])


@pytest.mark.parametrize("seed", [31, 32])
@pytest.mark.parametrize("conf_only", [False, True])
def test_no_rerank_layers_are_each_depths_best(seed, conf_only):
    tok, conf = random_rows(seed)
    D, k = tok.shape[0], tok.shape[1]
    out = otree.build_tree(tok, conf, D * k, -1, confidence_only=conf_only, rerank=False,
                           return_candidates=True)
    C = out["candidates"]
    for d in range(1, D + 1):
        layer = [g for g in range(1, len(C)) if C.depth[g] == d]
        best = sorted(layer, key=C.key)[:k]
        got = [int(g) for g, dep in zip(out["src"], out["depth"]) if dep == d]
        assert got == best
    # nodes appear depth by depth
    assert list(out["depth"]) == sorted(out["depth"])


def test_no_rerank_rejects_m_beyond_layers():
    tok, conf = random_rows(41)
    D, k = tok.shape[0], tok.shape[1]
    with pytest.raises(AssertionError):
        otree.build_tree(tok, conf, D * k + 1, -1, rerank=False)
