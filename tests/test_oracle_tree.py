"""Pins for the oracle's tree build (V_i, expansion, rerank, closure, order).

Independent checks:
  * a tree worked by hand from the definitions (tests/golden/hand_tree.json);
  * the identical-rows special case (the setting of the EAGLE-2 explainer's
    concept implementation, where every parent at a depth shares one
    candidate list): there the top-k-per-layer expansion must equal the
    global top-k of all k^d root paths of each depth, enumerated by brute
    force over the full k-ary tree;
  * a path-tuple re-statement of the expansion for general rows;
  * scores recomputed as explicit float32 products along each root path;
  * structural invariants (connected, parent first, |tree| = m+1, ...).
Mutation tests plant mistakes in the oracle and check the pins catch them.
"""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import tree as otree


def f32(x):
    return np.float32(x)


def load_hand(golden_dir):
    with open(os.path.join(golden_dir, "hand_tree.json")) as f:
        return json.load(f)


def check_hand_tree(golden_dir, build=otree.build_tree):
    h = load_hand(golden_dir)
    out = build(np.array(h["tok"]), np.array(h["conf"], dtype=np.float32), h["m"], h["root_token"])
    for key in ("tok", "parent", "depth", "src", "row"):
        assert list(out[key]) == h["expect"][key], key
    assert list(out["score"]) == h["expect"]["score"]
    assert out["closure_added"] == []


def chain_product(confs):
    v = f32(1.0)
    for c in confs:
        v = f32(np.float64(v) * np.float64(f32(c)))
    return v


def node_conf(out, tok, conf, i):
    """Confidence node i was created with, looked up from its parent's row."""
    p = out["parent"][i]
    slot = out["row"][p]
    k = tok.shape[1]
    d, j = divmod(int(slot), k)
    r = list(tok[d, j]).index(out["tok"][i])
    return conf[d, j, r]


def check_invariants(out, tok, conf, m):
    n = m + 1
    par, dep, sc = out["parent"], out["depth"], out["score"]
    assert len(par) == n and par[0] == -1 and dep[0] == 0 and sc[0] == 1.0
    for i in range(1, n):
        assert 0 <= par[i] < i
        assert dep[i] == dep[par[i]] + 1
        assert out["row"][par[i]] >= 0, "a parent must have been expanded"
    for i in range(1, n - 1):
        assert sc[i] >= sc[i + 1]
    sib = {}
    for i in range(1, n):
        sib.setdefault(int(par[i]), []).append(int(out["tok"][i]))
    for toks in sib.values():
        assert len(set(toks)) == len(toks)
    for i in range(1, n):
        confs = []
        j = i
        while j > 0:
            confs.append(node_conf(out, tok, conf, j))
            j = par[j]
        assert sc[i] == chain_product(confs[::-1])


def global_topk_expansion(row_lists, k, m):
    """Identical-rows case: row_lists[d] = list of (token, conf) shared by all
    parents at depth d.  E_d = global top-k of all depth-d root paths of the
    full k-ary tree; candidates of depth d+1 are the children of E_d; the
    result is the top-m of all candidates, as a list of token paths."""
    D = len(row_lists)

    def value(path):           # path = tuple of child ranks
        return chain_product([row_lists[d][r][1] for d, r in enumerate(path)])

    cands = [(r,) for r in range(k)]
    all_cands = list(cands)
    for d in range(1, D):
        full = list(itertools.product(range(k), repeat=d))
        best = sorted(full, key=lambda p: -float(value(p)))[:k]
        nxt = [p + (r,) for p in best for r in range(k)]
        all_cands += nxt
    top = sorted(all_cands, key=lambda p: -float(value(p)))[:m]
    return {tuple(row_lists[d][r][0] for d, r in enumerate(p)) for p in top}


def token_paths(out):
    paths = set()
    for i in range(1, len(out["parent"])):
        toks = []
        j = i
        while j > 0:
            toks.append(int(out["tok"][j]))
            j = out["parent"][j]
        paths.add(tuple(toks[::-1]))
    return paths


def identical_rows_case(rng, D, k, V):
    rows = []
    tok = np.zeros((D, k, k), dtype=np.int64)
    conf = np.zeros((D, k, k), dtype=np.float32)
    for d in range(D):
        t = rng.choice(V, size=k, replace=False)
        c = np.sort(rng.uniform(0.01, 0.9, size=k).astype(np.float32))[::-1]
        rows.append(list(zip(t.tolist(), c.tolist())))
        tok[d] = t
        conf[d] = c
    return rows, tok, conf


def check_identical_rows(build=otree.build_tree, seed=0):
    rng = np.random.default_rng(seed)
    for D, k in [(1, 3), (2, 3), (3, 3), (4, 2), (3, 4), (5, 2)]:
        rows, tok, conf = identical_rows_case(rng, D, k, 50)
        n_c = k + (D - 1) * k * k
        for m in sorted({1, min(3, n_c), n_c // 2 or 1, n_c}):
            out = build(tok, conf, m)
            assert token_paths(out) == global_topk_expansion(rows, k, m)


def path_tuple_tree(tok, conf, m):
    """General rows, restated over root paths: a candidate is the tuple of
    child ranks from the root; its parent is the tuple without its last
    element; the j-th best node of layer d (by V, then by the parent's
    creation position, then token) is expanded with row [d, j]."""
    D, k, _ = tok.shape
    info = {(): dict(V=f32(1.0), depth=0, pos=0, tok=-1)}
    order = {(): (0, 0)}

    def key(p):
        par = p[:-1]
        return (-float(info[p]["V"]), order[par], info[p]["tok"])

    layer = []
    for r in range(k):
        p = (r,)
        info[p] = dict(V=chain_product([conf[0, 0, r]]), tok=int(tok[0, 0, r]))
        order[p] = (1, r)
        layer.append(p)
    for d in range(1, D):
        exp_ = sorted(layer, key=key)[:k]
        layer = []
        for j, p in enumerate(exp_):
            for r in range(k):
                c = p + (r,)
                info[c] = dict(V=f32(np.float64(info[p]["V"]) * np.float64(conf[d, j, r])),
                               tok=int(tok[d, j, r]))
                order[c] = (d + 1, j * k + r)
                layer.append(c)
    cands = [p for p in info if p != ()]
    top = sorted(cands, key=key)[:m]
    return [tuple(info[p[:i + 1]]["tok"] for i in range(len(p))) for p in top]


def ordered_token_paths(out):
    res = []
    for i in range(1, len(out["parent"])):
        toks = []
        j = i
        while j > 0:
            toks.append(int(out["tok"][j]))
            j = out["parent"][j]
        res.append(tuple(toks[::-1]))
    return res


def random_rows(rng, D, k, V, levels=None):
    tok = np.zeros((D, k, k), dtype=np.int64)
    conf = np.zeros((D, k, k), dtype=np.float32)
    for d in range(D):
        for j in range(k):
            tok[d, j] = rng.choice(V, size=k, replace=False)
            if levels is None:
                c = rng.uniform(0.0, 1.0, size=k)
            else:       # few distinct dyadic values: exact ties in V
                c = rng.choice(levels, size=k)
            conf[d, j] = np.sort(c.astype(np.float32))[::-1]
    return tok, conf


def check_path_tuple(build=otree.build_tree, seed=1):
    rng = np.random.default_rng(seed)
    for trial in range(30):
        D = int(rng.integers(1, 5))
        k = int(rng.integers(1, 4))
        levels = None if trial % 2 else np.array([0.5, 0.25, 0.125, 0.75, 1.0])
        tok, conf = random_rows(rng, D, k, 40, levels)
        n_c = k + (D - 1) * k * k
        m = int(rng.integers(1, n_c + 1))
        out = build(tok, conf, m)
        assert ordered_token_paths(out) == path_tuple_tree(tok, conf, m)
        check_invariants(out, tok, conf, m)


def test_hand_tree(golden_dir):
    check_hand_tree(golden_dir)


def test_identical_rows_equal_global_topk_per_depth():
    check_identical_rows()


def test_general_rows_equal_path_tuple_statement():
    check_path_tuple()


def test_invariants_on_generated_workload():
    from gen import WORKLOADS, draft_logits
    from oracle import draft
    w = WORKLOADS["tiny"]
    lg = draft_logits(w).numpy()
    tok, conf, _ = draft.draft_topk(lg, w.k)
    conf32 = np.nan_to_num(conf).astype(np.float32)
    out = otree.build_tree(tok[0], conf32[0], w.m)
    check_invariants(out, tok[0], conf32[0], w.m)
    assert out["closure_added"] == []


def test_chain_and_single_depth():
    rng = np.random.default_rng(5)
    tok, conf = random_rows(rng, 4, 1, 30)          # k=1: a chain
    out = otree.build_tree(tok, conf, 3)
    assert list(out["parent"]) == [-1, 0, 1, 2]
    assert list(out["tok"][1:]) == [tok[d, 0, 0] for d in range(3)]
    tok, conf = random_rows(rng, 1, 6, 30)          # D=1: top-m of the root row
    out = otree.build_tree(tok, conf, 4)
    assert list(out["tok"][1:]) == list(tok[0, 0, :4])
    assert (out["parent"][1:] == 0).all()


def test_closure_adds_ancestors_outside_the_probability_domain():
    # With a confidence above 1 a child can outrank its parent; the closure
    # step must then add the parent (the connectivity rule).
    tok = np.array([[[5, 6], [0, 0]], [[1, 2], [3, 4]]])
    conf = np.array([[[0.5, 0.4], [0, 0]], [[0.9, 0.1], [2.0, 0.1]]], dtype=np.float32)
    out = otree.build_tree(tok, conf, 1)
    assert out["closure_added"] == [2]
    assert token_paths(out) == {(6,), (6, 3)}


def test_negative_zero_confidence_ranks_as_zero():
    """A confidence of -0 compares equal to +0 (IEEE), so the key order, the
    expansion and the kept set are those of the same rows with +0; the
    scores differ at most in the sign of zero."""
    rng = np.random.default_rng(21)
    D, k, m = 4, 4, 30
    tok = np.stack([np.stack([rng.choice(50, size=k, replace=False) for _ in range(k)]) for _ in range(D)])
    conf = (rng.integers(0, 3, size=(D, k, k)) / 4.0).astype(np.float32)   # many zeros, many ties
    neg = conf.copy()
    neg[conf == 0] = np.float32(-0.0)
    assert np.signbit(neg).any()
    for confidence_only, rerank in [(False, True), (True, True), (False, False)]:
        mm = min(m, D * k) if not rerank else m
        a = otree.build_tree(tok, conf, mm, confidence_only=confidence_only, rerank=rerank)
        b = otree.build_tree(tok, neg, mm, confidence_only=confidence_only, rerank=rerank)
        for key in ("tok", "parent", "depth", "src", "row"):
            assert (a[key] == b[key]).all(), key
        assert (a["score"] == b["score"]).all()          # -0 == +0


def test_build_trees_batch_matches_single():
    rng = np.random.default_rng(7)
    toks, confs = zip(*[random_rows(rng, 3, 3, 20) for _ in range(3)])
    tok, conf = np.stack(toks), np.stack(confs)
    bt = otree.build_trees(tok, conf, 7)
    for b in range(3):
        one = otree.build_tree(tok[b], conf[b], 7)
        for key in ("tok", "parent", "depth", "score", "src", "row"):
            assert (bt[key][b] == one[key]).all()


# --- planted mistakes -------------------------------------------------------

def _run_pins(golden_dir):
    caught = 0
    for check in (lambda: check_hand_tree(golden_dir), check_identical_rows, check_path_tuple):
        try:
            check()
        except AssertionError:
            caught += 1
    return caught


def test_pins_catch_dropped_parent_tiebreak(golden_dir, monkeypatch):
    monkeypatch.setattr(otree.Candidates, "key",
                        lambda self, g: (-float(self.score[g]), self.token[g]))
    assert _run_pins(golden_dir) >= 1


def test_pins_catch_unrounded_products(golden_dir, monkeypatch):
    monkeypatch.setattr(otree, "fl32_mul",
                        lambda a, b: np.float64(a) * np.float64(b) * (1 + 2 ** -30))
    assert _run_pins(golden_dir) >= 1


def test_pins_catch_rows_in_creation_order(golden_dir, monkeypatch):
    real = otree.build_tree

    def wrong(tok, conf, m, root_token=-1, return_candidates=False):
        # expands layer d's nodes in creation (gid) order instead of key order
        C = otree.Candidates(root_token)
        D, k, _ = tok.shape
        layer = [C.add(0, tok[0, 0, r], conf[0, 0, r], 1) for r in range(k)]
        for d in range(1, D):
            expanded = sorted(sorted(layer, key=C.key)[:k])
            nxt = []
            for j, p in enumerate(expanded):
                C.row[p] = d * k + j
                for r in range(k):
                    nxt.append(C.add(p, tok[d, j, r], conf[d, j, r], d + 1))
            layer = nxt
        kept = sorted(range(1, len(C)), key=C.key)[:m]
        order = [0] + kept
        idx = {g: i for i, g in enumerate(order)}
        return dict(tok=np.array([C.token[g] for g in order]),
                    parent=np.array([idx[C.parent[g]] if g else -1 for g in order]),
                    depth=np.array([C.depth[g] for g in order]),
                    score=np.array([C.score[g] for g in order], dtype=np.float32),
                    src=np.array(order), row=np.array([C.row[g] for g in order]),
                    closure_added=[])

    caught = 0
    for check in (lambda: check_hand_tree(golden_dir, wrong),
                  lambda: check_path_tuple(wrong)):
        try:
            check()
        except AssertionError:
            caught += 1
    assert caught >= 1
    assert real is otree.build_tree
