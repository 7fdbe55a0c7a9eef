"""Oracle stage 3: tree-masked attention of the tree nodes over the KV prefix.

Follows [EAGLE-1] sections "用語解説" (Tree Attention) and "Tree Attention の
役割": the target model checks every branch of the draft tree in one forward
pass, each tree token attending to the sequence's prefix and, within the
tree, only to its ancestors ([EAGLE-2] section "注意マスクの調整").

Readings where the pages are silent:
  * The queries are all m+1 tree nodes, root included: the target's logits
    row i (i = 0..m) is its prediction after node i, which needs node i as a
    query.  Tree keys/values likewise cover nodes 0..m.
  * Node i (query head h, KV head g = h // (Hq / Hkv): contiguous GQA groups)
    attends to prefix positions 0..kv_len[b]-1 of head g and to tree nodes j
    with mask[i, j] set.
  * s = scale * <q, k>; out = sum_j softmax(s)_j v_j; lse = ln sum_j exp(s_j).
Inputs are widened exactly to fp64; the arithmetic is plain fp64.
"""
import numpy as np


def _keys_values(k_cache, v_cache, kv_len, k_tree, v_tree, mask, b, g, i):
    L = int(kv_len[b])
    cols = np.nonzero(mask[b, i])[0]
    K = np.concatenate([k_cache[b, g, :L], k_tree[b, g, cols]], axis=0)
    V = np.concatenate([v_cache[b, g, :L], v_tree[b, g, cols]], axis=0)
    return K, V


def attention_row(q, k_cache, v_cache, kv_len, k_tree, v_tree, mask, scale, b, i, h):
    """Output [dh] and lse of one (sequence b, node i, query head h)."""
    Hq = q.shape[2]
    Hkv = k_cache.shape[1]
    g = h // (Hq // Hkv)
    K, V = _keys_values(k_cache, v_cache, kv_len, k_tree, v_tree, mask, b, g, i)
    s = scale * (K @ np.asarray(q[b, i, h], dtype=np.float64))
    mx = s.max()
    p = np.exp(s - mx)
    l = p.sum()
    return (p @ V) / l, mx + np.log(l)


def tree_attention(q, k_cache, v_cache, kv_len, k_tree, v_tree, mask, scale):
    """All outputs.

    q [B, n, Hq, dh]; k_cache, v_cache [B, Hkv, Lmax, dh]; kv_len [B];
    k_tree, v_tree [B, Hkv, n, dh]; mask bool [B, n, n].
    Returns out fp64 [B, n, Hq, dh], lse fp64 [B, n, Hq].
    """
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    k_tree = np.asarray(k_tree, dtype=np.float64)
    v_tree = np.asarray(v_tree, dtype=np.float64)
    mask = np.asarray(mask, dtype=bool)
    B, n, Hq, dh = q.shape
    Hkv = k_cache.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, n, Hq, dh))
    lse = np.zeros((B, n, Hq))
    for b in range(B):
        L = int(kv_len[b])
        for g in range(Hkv):
            K = np.concatenate([k_cache[b, g, :L], k_tree[b, g]], axis=0)   # [L+n, dh]
            V = np.concatenate([v_cache[b, g, :L], v_tree[b, g]], axis=0)
            allowed = np.concatenate([np.ones((n, L), dtype=bool), mask[b]], axis=1)  # [n, L+n]
            for hh in range(G):
                h = g * G + hh
                s = scale * (q[b, :, h] @ K.T)                  # [n, L+n]
                s = np.where(allowed, s, -np.inf)
                mx = s.max(axis=1, keepdims=True)
                p = np.exp(s - mx)
                l = p.sum(axis=1, keepdims=True)
                out[b, :, h] = (p @ V) / l
                lse[b, :, h] = (mx + np.log(l))[:, 0]
    return out, lse
