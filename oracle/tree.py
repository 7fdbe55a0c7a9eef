"""Oracle stage 2: global scores, frontier expansion, rerank, closure, order.

Follows [EAGLE-2] section "動的ドラフトツリーの構築アルゴリズム":
  * V_i, the global acceptance score of a draft token, is the product of the
    confidences c_j of every token on the path from the root to it (the
    V_i equation); the root has V = 1.
  * Expansion: at each depth the k nodes of that layer with the largest V
    are expanded, each getting its own top-k tokens as children (k = 10 in
    the paper's experiments).
  * Rerank: of all generated candidates the m with the largest V are kept
    (m = 60 / 50 / 48 for 7B / 13B / 70B targets).
  * Connectivity: ancestors of every kept token are added so the kept set is
    a connected tree.

Readings where the page leaves a point open:
  * Products are taken in float32 one factor at a time, V_child =
    fl32(V_parent * c), computed as the exact fp64 product of the two fp32
    values rounded once to fp32 (round to nearest even, subnormals kept).
  * Order among candidates ("key"): V descending, then the parent's global
    candidate id ascending, then token id ascending.  This is a total order.
  * Global candidate ids (gid): root 0; depth 1 gets 1..k in the root row's
    top-k order; deeper candidates are numbered depth by depth, by the rank j
    of their parent in that layer's expanded set, then by the child's rank
    in its parent's top-k list.
  * The j-th expanded node of layer d (in key order) is the one whose draft
    distribution is row [d, j].
  * Output order: root first, then the kept nodes in key order.
Because c <= 1, fl32(V * c) <= V, and a parent's gid is below its children's,
every ancestor precedes its descendants in key order, so the top-m set is
already closed and the closure step adds nothing; `build_tree` checks it.

Ablation variants ([EAGLE-2] section "実験結果", ablation table: "without the
global acceptance probability (confidence only)" and "without reranking"):
  * confidence_only: a candidate is ranked by its own confidence c instead
    of V, in the expansion and in the rerank.  Reading: c does not shrink
    along a path, so the m best keys need not form a connected tree; the
    rerank then grows the tree best-first, repeatedly adding the candidate
    with the greatest key among those whose parent is already in the tree.
    With V keys that is exactly the top-m set (ancestors outrank their
    descendants), so the full method is the same procedure.
  * rerank=False: the tree is the layers' selections E_1, E_2, ..., E_D in
    depth order, each layer's k greatest keys (E_D chosen the same way,
    although it is never expanded), truncated to m nodes; m <= D*k.
  * node score: the value the node was ranked by (V, or c when
    confidence_only).
"""
import numpy as np


def fl32_mul(a, b):
    """fl32(a * b) for float32 a, b: exact fp64 product, rounded once."""
    return np.float32(np.float64(np.float32(a)) * np.float64(np.float32(b)))


class Candidates:
    """Plain table of every node the expansion creates, indexed by gid."""

    def __init__(self, root_token):
        self.parent = [-1]
        self.token = [int(root_token)]
        self.depth = [0]
        self.score = [np.float32(1.0)]
        self.row = [0]          # draft row slot d*k + j if expanded, else -1

    def add(self, parent, token, conf, depth, confidence_only=False):
        self.parent.append(int(parent))
        self.token.append(int(token))
        self.depth.append(int(depth))
        self.score.append(np.float32(conf) if confidence_only
                          else fl32_mul(self.score[parent], conf))
        self.row.append(-1)
        return len(self.parent) - 1

    def key(self, g):
        """Sort key: ascending order of this tuple is the rank order."""
        return (-float(self.score[g]), self.parent[g], self.token[g])

    def __len__(self):
        return len(self.parent)


def build_tree(tok, conf, m, root_token=-1, return_candidates=False,
               confidence_only=False, rerank=True):
    """Build one sequence's draft tree.

    tok  int [D, k, k]   top-k token ids of each used draft row
    conf fp32 [D, k, k]  their confidences (rows [0, 1..k-1] unused)
    m    number of draft tokens to keep
    confidence_only, rerank: the ablation variants (module docstring)

    Returns a dict of arrays over the m+1 output nodes (root = node 0):
      tok, parent (output index, root -1), depth, score (fp32 V), src (gid),
      row (draft row slot d*k + j the node was expanded with, else -1),
    plus 'closure_added' (nodes the closure step had to add).
    """
    tok = np.asarray(tok)
    conf = np.asarray(conf, dtype=np.float32)
    D, k, k2 = tok.shape
    assert k == k2
    C = Candidates(root_token)

    layer = [C.add(0, tok[0, 0, r], conf[0, 0, r], 1, confidence_only) for r in range(k)]
    selections = []                      # E_1, E_2, ...: each layer's k best
    for d in range(1, D + 1):
        expanded = sorted(layer, key=C.key)[:k]
        selections.append(expanded)
        if d == D:
            break
        nxt = []
        for j, p in enumerate(expanded):
            C.row[p] = d * k + j
            for r in range(k):
                nxt.append(C.add(p, tok[d, j, r], conf[d, j, r], d + 1, confidence_only))
        layer = nxt

    n_cand = len(C) - 1
    assert 1 <= m <= n_cand, "m must not exceed the number of candidates"
    if not rerank:
        assert m <= D * k, "without rerank the tree holds at most D*k nodes"
        kept = [g for sel in selections for g in sel][:m]
    elif confidence_only:
        kept = []
        inside = {0}
        for _ in range(m):
            open_ = [g for g in range(1, len(C)) if g not in inside and C.parent[g] in inside]
            best = min(open_, key=C.key)
            kept.append(best)
            inside.add(best)
    else:
        kept = sorted(range(1, len(C)), key=C.key)[:m]

    chosen = set(kept)
    added = []
    for g in kept:
        a = C.parent[g]
        while a > 0:
            if a not in chosen:
                chosen.add(a)
                added.append(a)
            a = C.parent[a]

    if rerank and not confidence_only:
        order = [0] + sorted(chosen, key=C.key)
    else:
        order = [0] + kept           # selection order: parents come first
    index_of = {g: i for i, g in enumerate(order)}
    out = dict(
        tok=np.array([C.token[g] for g in order], dtype=np.int64),
        parent=np.array([index_of[C.parent[g]] if g else -1 for g in order], dtype=np.int64),
        depth=np.array([C.depth[g] for g in order], dtype=np.int64),
        score=np.array([C.score[g] for g in order], dtype=np.float32),
        src=np.array(order, dtype=np.int64),
        row=np.array([C.row[g] for g in order], dtype=np.int64),
        closure_added=added,
    )
    if return_candidates:
        out["candidates"] = C
    return out


def build_trees(tok, conf, m, root_tokens=None, confidence_only=False, rerank=True):
    """Batch version: tok [B, D, k, k], conf [B, D, k, k] -> stacked arrays.

    Requires the closure to add nothing (true whenever 0 <= c <= 1), so every
    sequence has exactly m+1 nodes.
    """
    B = tok.shape[0]
    outs = [build_tree(tok[b], conf[b], m,
                       -1 if root_tokens is None else root_tokens[b],
                       confidence_only=confidence_only, rerank=rerank)
            for b in range(B)]
    for o in outs:
        assert not o["closure_added"], "closure added nodes (a confidence > 1?)"
    return {key: np.stack([o[key] for o in outs])
            for key in ("tok", "parent", "depth", "score", "src", "row")}
