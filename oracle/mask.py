"""Oracle: the ancestor-only tree attention mask.

Follows [EAGLE-2] section "注意マスクの調整": each draft token may attend
only to its own ancestors, so tokens of different branches never see one
another.  Reading: a token also attends to itself (it is its own query
position) and the root is an ancestor of every node.

mask[i, j] is True iff j == i or j is an ancestor of i, found by walking the
parent pointers from i up to the root.  Packed form: bit (j % 64) of word
(j // 64) of row i, as uint64 words [n, ceil(n / 64)].
"""
import numpy as np


def tree_mask(parent):
    """parent int [n] (root -1) -> bool [n, n]."""
    parent = np.asarray(parent)
    n = parent.size
    M = np.zeros((n, n), dtype=bool)
    for i in range(n):
        j = i
        steps = 0
        while j != -1:
            M[i, j] = True
            j = int(parent[j])
            steps += 1
            assert steps <= n, "parent pointers contain a cycle"
    return M


def pack_mask(M):
    """bool [..., n, n] -> uint64 [..., n, ceil(n/64)]."""
    M = np.asarray(M, dtype=bool)
    n = M.shape[-1]
    W = (n + 63) // 64
    out = np.zeros(M.shape[:-1] + (W,), dtype=np.uint64)
    for j in range(n):
        bit = np.uint64(1) << np.uint64(j % 64)
        out[..., j // 64] |= np.where(M[..., j], bit, np.uint64(0))
    return out


def unpack_mask(words, n):
    """uint64 [..., W] -> bool [..., n]."""
    words = np.asarray(words, dtype=np.uint64)
    cols = []
    for j in range(n):
        cols.append(((words[..., j // 64] >> np.uint64(j % 64)) & np.uint64(1)) == 1)
    return np.stack(cols, axis=-1)


def tree_masks(parents):
    """Batch: parents [B, n] -> packed uint64 [B, n, W]."""
    return np.stack([pack_mask(tree_mask(p)) for p in np.asarray(parents)])
