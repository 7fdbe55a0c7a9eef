"""Oracle: the EAGLE-1 static draft tree (test infrastructure only).

[EAGLE-2] sections "背景" and "EAGLE-1からの変更点": EAGLE-1 places its draft
tokens on a tree template fixed in advance (chosen offline) and applies the
same shape to every input; EAGLE-2 replaces only that choice of shape.  The
pages give no template, so the template is an input here.

Readings (the pages are silent on the encoding):
  * A template of n nodes is `parent` (parent[0] = -1 for the root, else
    0 <= parent[i] < i) and `rank` (0 <= rank[i] < k): node i is the
    rank[i]-th of its parent's top-k draft tokens.  Siblings have distinct
    ranks.
  * Draft rows as in the dynamic tree: the root's distribution is row [0, 0];
    the j-th node of depth d >= 1 that has children (j counted in node
    order) uses row [d, j], so a depth has at most k such nodes and they lie
    above depth D.
  * Node score: the product of the confidences along the root path, in
    float32 one factor at a time (the V of EAGLE-2, for information).
  * Outputs mirror the dynamic tree's: tok, parent, depth, score, src (the
    template index i), row (d*k + j for a node with children, root 0, else
    -1).
"""
import numpy as np

from .tree import fl32_mul


def template_rows(parent, k, D):
    """Depth of every node and the draft row slot of every node with
    children; asserts the template is valid for (k, D)."""
    parent = [int(p) for p in parent]
    n = len(parent)
    assert n >= 1 and parent[0] == -1, "node 0 is the root"
    depth = [0] * n
    for i in range(1, n):
        assert 0 <= parent[i] < i, "parents precede their children"
        depth[i] = depth[parent[i]] + 1
        assert depth[i] <= D, "template deeper than the draft rows"
    has_child = [False] * n
    for i in range(1, n):
        has_child[parent[i]] = True
    row = [-1] * n
    row[0] = 0
    count = {}
    for i in range(1, n):
        if has_child[i]:
            d = depth[i]
            j = count.get(d, 0)
            count[d] = j + 1
            assert d < D and j < k, "at most k nodes with children per depth, above depth D"
            row[i] = d * k + j
    return depth, row


def build_static_tree(tok, conf, parent, rank, root_token=-1):
    """tok int [D, k, k], conf fp32 [D, k, k] (one sequence's draft top-k);
    parent, rank: the template.  Returns the node arrays."""
    tok = np.asarray(tok)
    conf = np.asarray(conf, dtype=np.float32)
    D, k, _ = tok.shape
    n = len(parent)
    depth, row = template_rows(parent, k, D)
    sib = set()
    out_tok = [int(root_token)]
    score = [np.float32(1.0)]
    for i in range(1, n):
        p, r = int(parent[i]), int(rank[i])
        assert 0 <= r < k and (p, r) not in sib, "ranks in [0, k), distinct among siblings"
        sib.add((p, r))
        d, j = divmod(row[p], k)
        out_tok.append(int(tok[d, j, r]))
        score.append(fl32_mul(score[p], conf[d, j, r]))
    return dict(
        tok=np.array(out_tok, dtype=np.int64),
        parent=np.array(parent, dtype=np.int64),
        depth=np.array(depth, dtype=np.int64),
        score=np.array(score, dtype=np.float32),
        src=np.arange(n, dtype=np.int64),
        row=np.array(row, dtype=np.int64),
    )


def build_static_trees(tok, conf, parent, rank, root_tokens=None):
    """Batch version over tok/conf [B, D, k, k]; one template for all."""
    B = tok.shape[0]
    outs = [build_static_tree(tok[b], conf[b], parent, rank,
                              -1 if root_tokens is None else root_tokens[b]) for b in range(B)]
    return {key: np.stack([o[key] for o in outs]) for key in outs[0]}
