"""Pins for the oracle's EAGLE-1 static draft tree.

[EAGLE-2] sections "背景" and "EAGLE-1からの変更点": EAGLE-1 fixes the tree's
shape offline; only the tokens on it come from the draft.  Independent checks:
  * a template worked by hand (tests/golden/hand_static.json);
  * scores as explicit float32 products of the listed confidences;
  * invalid templates are rejected;
  * on generated templates: every node's token and confidence are found in
    its parent's draft row at the node's rank (the row looked up by an
    enumeration written here), depth = parent depth + 1.
"""
import json
import os

import numpy as np
import pytest

import gen
from oracle import draft as odraft
from oracle import static_tree as ost

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def product(cs):
    v = np.float32(1.0)
    for c in cs:
        v = np.float32(np.float64(v) * np.float64(np.float32(c)))
    return v


def test_hand_worked_static_tree():
    with open(os.path.join(GOLDEN, "hand_static.json")) as f:
        h = json.load(f)
    out = ost.build_static_tree(np.array(h["tok"]), np.array(h["conf"], dtype=np.float32),
                                h["parent"], h["rank"])
    e = h["expect"]
    assert list(out["tok"]) == e["tok"]
    assert list(out["depth"]) == e["depth"]
    assert list(out["row"]) == e["row"]
    assert list(out["parent"]) == h["parent"]
    assert list(out["score"]) == [product(cs) for cs in e["score_products"]]


@pytest.mark.parametrize("parent,rank,why", [
    ([0, 0], [0, 0], "root must have parent -1"),
    ([-1, 0, 2], [0, 0, 0], "parent after child"),
    ([-1, 0, 0], [0, 1, 1], "duplicate sibling rank"),
    ([-1, 0], [0, 2], "rank >= k"),
    ([-1, 0, 1, 2, 3], [0, 0, 0, 0, 0], "deeper than D"),
    ([-1, 0, 0, 0, 1, 2, 3], [0, 1, 0, 0, 0, 0, 0], "rank clash"),
])
def test_invalid_templates_rejected(parent, rank, why):
    tok = np.zeros((3, 2, 2), dtype=np.int64)
    conf = np.full((3, 2, 2), 0.5, dtype=np.float32)
    with pytest.raises(AssertionError):
        ost.build_static_tree(tok, conf, parent, rank)


def test_too_many_parents_at_one_depth():
    # k = 2 but three depth-1 nodes have children
    tok = np.zeros((3, 2, 2), dtype=np.int64)
    conf = np.full((3, 2, 2), 0.5, dtype=np.float32)
    parent = [-1, 0, 0, 1, 2, 0]
    rank = [0, 0, 1, 0, 0, 1]
    with pytest.raises(AssertionError):
        ost.build_static_tree(tok, conf, parent, rank)


def rows_by_enumeration(parent, k):
    """Draft row of every node with children: walk depth by depth, counting
    nodes with children in node order (written independently of the oracle)."""
    n = len(parent)
    kids = {i: [c for c in range(n) if parent[c] == i] for i in range(n)}
    depth = {0: 0}
    frontier = [0]
    while frontier:
        nxt = []
        for i in frontier:
            for c in kids[i]:
                depth[c] = depth[i] + 1
                nxt.append(c)
        frontier = sorted(nxt)
    rows = {0: (0, 0)}
    for d in sorted(set(depth.values()) - {0}):
        j = 0
        for i in range(n):
            if depth[i] == d and kids[i]:
                rows[i] = (d, j)
                j += 1
    return rows, depth


@pytest.mark.parametrize("shape,D,k", [
    (gen.STATIC_SHAPE_60, 6, 10),
    (([3], [2, 1], [1, 1]), 3, 3),
    (([8], [4, 2, 1], [3, 1], [2], [1], [1], [1]), 7, 8),
])
def test_generated_templates(shape, D, k):
    parent, rank = gen.static_template(shape)
    w = gen.scaled(gen.WORKLOADS["tiny"], B=1, D=D, k=k, V=256, m=len(parent) - 1, seed=77)
    logits = gen.draft_logits(w).float().numpy()
    tok, conf, _ = odraft.draft_topk(logits, k)
    tok, conf = tok[0], np.nan_to_num(conf[0]).astype(np.float32)
    out = ost.build_static_tree(tok, conf, parent, rank)
    rows, depth = rows_by_enumeration(list(parent), k)
    for i in range(1, len(parent)):
        d, j = rows[int(parent[i])]
        assert out["tok"][i] == tok[d, j, rank[i]]
        assert out["depth"][i] == depth[i] == out["depth"][parent[i]] + 1
        assert out["score"][i] == np.float32(np.float64(out["score"][parent[i]]) * np.float64(conf[d, j, rank[i]]))
    for i, (d, j) in rows.items():
        assert out["row"][i] == (0 if i == 0 else d * k + j)
