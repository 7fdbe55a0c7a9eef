"""Pins for the oracle's verification walks.

Independent checks:
  * hand-worked greedy and sampling walks (tests/golden/);
  * greedy = the longest root path whose every token is the argmax of its
    parent's row, found by enumerating all root paths;
  * losslessness by Monte-Carlo: over many fresh uniforms the first emitted
    token follows the target distribution after the root, and, given that a
    child x was accepted first, the next token follows the target
    distribution after x (chi-square tests);
  * special cases: a tree with only the root reduces to sampling from p_0.
A planted mistake (rejected mass not removed) must fail the Monte-Carlo pin.
"""
import json
import os

import numpy as np
import pytest
from scipy import stats

from oracle import verify as over


def test_hand_greedy(golden_dir):
    with open(os.path.join(golden_dir, "hand_tree.json")) as f:
        h = json.load(f)
    e = h["expect"]
    logits = np.zeros((4, h["V"]))
    for i, a in enumerate(h["greedy_target_argmax"]):
        logits[i, a] = 1.0
    r = over.verify_greedy(logits, e["tok"], e["parent"])
    g = h["greedy_expect"]
    assert (r.accept_len, r.path, r.tokens) == (g["accept_len"], g["path"], g["tokens"])


def test_hand_sample(golden_dir):
    with open(os.path.join(golden_dir, "hand_sample.json")) as f:
        h = json.load(f)
    logits = np.log(np.array(h["probs"]))
    r = over.verify_sample(logits, h["node_tok"], h["node_parent"], 1.0, np.array(h["u"]))
    e = h["expect"]
    assert (r.accept_len, r.path, r.tokens) == (e["accept_len"], e["path"], e["tokens"])
    assert r.ambiguous is None


def all_root_paths(parent):
    ch = over.children_of(parent)
    out = []

    def rec(p):
        out.append(p)
        for c in ch[p[-1]]:
            rec(p + [c])
    rec([0])
    return out


def random_tree_distinct_siblings(rng, n, V):
    parent = [-1]
    tok = [-1]
    used = {0: set()}
    for i in range(1, n):
        open_ = [q for q in range(i) if len(used[q]) < V]
        p = int(rng.choice(open_))
        choices = [t for t in range(V) if t not in used[p]]
        t = int(rng.choice(choices))
        used[p].add(t)
        used[i] = set()
        parent.append(p)
        tok.append(t)
    return np.array(parent), np.array(tok)


def test_greedy_is_longest_argmax_path():
    rng = np.random.default_rng(0)
    for trial in range(200):
        V = int(rng.integers(2, 6))
        n = int(rng.integers(1, 12))
        parent, tok = random_tree_distinct_siblings(rng, n, V)
        logits = np.round(rng.normal(size=(n, V)))     # ties happen
        argmax = [min(t for t in range(V) if logits[i, t] == logits[i].max()) for i in range(n)]
        good = [p for p in all_root_paths(parent)
                if all(tok[p[s + 1]] == argmax[p[s]] for s in range(len(p) - 1))]
        best = max(good, key=len)
        assert sum(len(p) == len(best) for p in good) == 1
        r = over.verify_greedy(logits, tok, parent)
        assert r.path == best
        assert r.tokens == [int(tok[i]) for i in best[1:]] + [argmax[best[-1]]]


MC_PARENT = np.array([-1, 0, 0, 0, 1, 1, 4])
MC_TOK = np.array([-1, 2, 0, 5, 1, 3, 4])


def mc_run(trials, T, seed):
    rng = np.random.default_rng(seed)
    V = 6
    logits = rng.normal(size=(7, V)) * 1.2
    logits[0, 2] += 2.0      # make the path root -> node 1 -> node 4 common
    logits[1, 1] += 2.0
    p = np.exp(logits / T)
    p /= p.sum(1, keepdims=True)
    first = np.zeros(V)
    second = np.zeros(V)
    third = np.zeros(V)
    for _ in range(trials):
        u = rng.random(size=(7, 2))
        r = over.verify_sample(logits, MC_TOK, MC_PARENT, T, u)
        first[r.tokens[0]] += 1
        if r.path[1:2] == [1]:
            second[r.tokens[1]] += 1
            if r.path[2:3] == [4]:
                third[r.tokens[2]] += 1
    return p, first, second, third


def chi2_p(obs, probs):
    probs = probs / probs.sum()
    return stats.chisquare(obs, obs.sum() * probs).pvalue


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_sampling_walk_is_lossless(T):
    p, first, second, third = mc_run(40000, T, seed=11 if T == 1.0 else 12)
    assert chi2_p(first, p[0]) > 1e-3
    assert second.sum() > 2000 and chi2_p(second, p[1]) > 1e-3
    assert third.sum() > 300 and chi2_p(third, p[4]) > 1e-3


def test_root_only_tree_samples_p0():
    rng = np.random.default_rng(3)
    logits = rng.normal(size=(1, 5))
    p = np.exp(logits[0]) / np.exp(logits[0]).sum()
    counts = np.zeros(5)
    for _ in range(20000):
        r = over.verify_sample(logits, [-1], [-1], 1.0, rng.random(size=(1, 2)))
        assert r.accept_len == 0 and len(r.tokens) == 1
        counts[r.tokens[0]] += 1
    assert chi2_p(counts, p) > 1e-3


def test_ambiguity_is_flagged_at_the_boundary():
    logits = np.log(np.array([[0.5, 0.25, 0.25], [1 / 3, 1 / 3, 1 / 3]]))
    u = np.array([[0.0, 0.0], [0.5, 0.0]])     # u * 1 == p(token 0) exactly
    r = over.verify_sample(logits, [-1, 0], [-1, 0], 1.0, u)
    assert r.ambiguous is not None and r.ambiguous[1] == "accept"


def test_bonus_on_a_boundary_lists_both_neighbours():
    # root only, p = (1/2, 1/4, 1/4): u = 1/2 puts the threshold exactly on
    # the boundary between tokens 0 and 1; the draw takes token 1 (the first
    # cumulative sum above the threshold) and either is admissible
    logits = np.log(np.array([[0.5, 0.25, 0.25]]))
    r = over.verify_sample(logits, [-1], [-1], 1.0, np.array([[0.0, 0.5]]))
    assert r.tokens == [1]
    assert r.ambiguous is not None and r.ambiguous[1] == "bonus"
    assert r.bonus_choices == (0, 1)


def test_bonus_choices_include_a_token_lighter_than_the_band():
    # token 1 carries 1e-7 of the mass, less than the band: a threshold at
    # its interval may land in token 0, 1 or 2 under rounding
    p = np.array([0.5, 1e-7, 0.5 - 1e-7])
    r = over.verify_sample(np.log(p)[None], [-1], [-1], 1.0, np.array([[0.0, 0.5 + 5e-8]]))
    assert r.tokens == [1]
    assert r.bonus_choices == (0, 1, 2)


def test_bonus_choices_skip_rejected_tokens():
    # the root's child (token 0) is rejected, so the draw is over tokens 1, 2
    # only; u = 1/2 of the residual 1/2 puts the threshold on their boundary
    logits = np.log(np.array([[0.5, 0.25, 0.25], [1 / 3, 1 / 3, 1 / 3]]))
    u = np.array([[0.0, 0.5], [0.999, 0.0]])
    r = over.verify_sample(logits, [-1, 0], [-1, 0], 1.0, u)
    assert r.accept_len == 0 and r.tokens == [2]
    assert r.bonus_choices == (1, 2)


def test_no_flag_no_choices(golden_dir):
    with open(os.path.join(golden_dir, "hand_sample.json")) as f:
        h = json.load(f)
    r = over.verify_sample(np.log(np.array(h["probs"])), h["node_tok"], h["node_parent"], 1.0, np.array(h["u"]))
    assert r.ambiguous is None and r.bonus_choices is None


def test_planted_unremoved_mass_fails_monte_carlo(monkeypatch):
    monkeypatch.setattr(over, "residual_mass", lambda Z, e, rejected: Z)
    p, first, _, _ = mc_run(20000, 1.0, seed=13)
    assert chi2_p(first, p[0]) < 1e-3


def test_batch_wrapper_pads():
    logits = np.log(np.array([[[0.7, 0.2, 0.1], [0.1, 0.8, 0.1]]]))
    acc, path, toks, _ = over.verify(logits, np.array([[-1, 0]]), np.array([[-1, 0]]),
                                     3, "greedy")
    assert acc.tolist() == [1]
    assert path.tolist() == [[0, 1, -1, -1]]
    assert toks.tolist() == [[0, 1, -1, -1]]
