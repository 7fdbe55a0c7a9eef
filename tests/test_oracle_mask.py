"""Pins for the oracle's ancestor-only attention mask.

Independent checks: the hand-worked tree's mask words, and the transitive
closure of the parent relation computed by Warshall's algorithm on random
trees (including trees of more than 64 nodes, which need several words).
"""
import json
import os

import numpy as np

from oracle import mask as omask


def warshall_ancestor_or_self(parent):
    n = len(parent)
    R = np.eye(n, dtype=bool)
    for i, p in enumerate(parent):
        if p >= 0:
            R[i, p] = True
    for k in range(n):
        R = R | (R[:, [k]] & R[[k], :])
    return R


def random_tree(rng, n):
    return np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)])


def test_hand_tree_mask(golden_dir):
    with open(os.path.join(golden_dir, "hand_tree.json")) as f:
        h = json.load(f)
    words = omask.pack_mask(omask.tree_mask(h["expect"]["parent"]))
    assert [int(w) for w in words[:, 0]] == h["expect"]["mask_words"]


def test_mask_is_transitive_closure():
    rng = np.random.default_rng(0)
    for n in (1, 2, 5, 11, 61, 64, 65, 130):
        par = random_tree(rng, n)
        M = omask.tree_mask(par)
        assert (M == warshall_ancestor_or_self(par)).all()
        assert M[:, 0].all(), "the root is an ancestor of every node"
        words = omask.pack_mask(M)
        assert words.shape == (n, (n + 63) // 64)
        assert (omask.unpack_mask(words, n) == M).all()


def test_batch_packing():
    rng = np.random.default_rng(1)
    pars = np.stack([random_tree(rng, 70) for _ in range(3)])
    words = omask.tree_masks(pars)
    for b in range(3):
        assert (omask.unpack_mask(words[b], 70) == warshall_ancestor_or_self(pars[b])).all()
