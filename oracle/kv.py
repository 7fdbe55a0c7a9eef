"""Oracle: KV commit after verification and the paged KV layout (test
infrastructure only).

[EAGLE-1] section "検証方法" and [EAGLE-2]: after verification the accepted
draft tokens become part of the sequence, so their keys and values (computed
for the tree in the target's forward pass) join the KV cache; everything
after a rejection is discarded.  The pages name the KV cache but give no
layout; the serving systems they mention keep it in fixed-size pages
addressed through a per-sequence block table, with a slot of -1 (padding)
for tokens that are not kept.

Readings:
  * The root's K/V is already the last prefix position (it was the last
    accepted token of the previous step).  The accepted path nodes
    path[1..a] are appended, in path order, at positions kv_len .. kv_len+a-1
    of their sequence, and kv_len becomes kv_len + a.  The bonus token has no
    K/V yet (the next step's forward pass makes it).
  * slot_mapping[b, i] = the position node i occupies in its sequence's KV
    after the commit (root: kv_len - 1), or -1 for nodes not kept.
  * Paged layout: pages [num_pages, Hkv, page_size, dh]; block_table[b, p]
    is the physical page of logical page p of sequence b, so logical
    position L lives in page block_table[b, L // page_size] at row
    L % page_size.
  * Contiguous layout: cache [B, Hkv, Lmax, dh].
"""
import numpy as np


def slot_mapping(path_nodes, accept_len, kv_len, n):
    """[B, n] positions after the commit (root kv_len-1; rejected -1)."""
    B = len(accept_len)
    out = np.full((B, n), -1, dtype=np.int64)
    for b in range(B):
        out[b, 0] = kv_len[b] - 1
        for p in range(1, int(accept_len[b]) + 1):
            out[b, int(path_nodes[b, p])] = kv_len[b] + p - 1
    return out


def commit_contiguous(k_cache, v_cache, kv_len, k_tree, v_tree, path_nodes, accept_len):
    """Returns new (k_cache, v_cache, kv_len): accepted nodes appended."""
    k_cache, v_cache = k_cache.copy(), v_cache.copy()
    kv_len = np.array(kv_len, dtype=np.int64).copy()
    B = k_cache.shape[0]
    for b in range(B):
        a = int(accept_len[b])
        for p in range(1, a + 1):
            node = int(path_nodes[b, p])
            pos = kv_len[b] + p - 1
            k_cache[b, :, pos] = k_tree[b, :, node]
            v_cache[b, :, pos] = v_tree[b, :, node]
        kv_len[b] += a
    return k_cache, v_cache, kv_len


def gather_pages(pages, block_table, kv_len, Lmax):
    """Paged pool -> contiguous [B, Hkv, Lmax, dh] (positions >= kv_len zero)."""
    _, Hkv, P, dh = pages.shape
    B = block_table.shape[0]
    out = np.zeros((B, Hkv, Lmax, dh), dtype=pages.dtype)
    for b in range(B):
        for pos in range(int(kv_len[b])):
            page = int(block_table[b, pos // P])
            out[b, :, pos] = pages[page, :, pos % P]
    return out


def scatter_pages(cache, block_table, kv_len, pages):
    """Contiguous cache -> the paged pool (positions < kv_len), in place."""
    B, Hkv, _, dh = cache.shape
    P = pages.shape[2]
    for b in range(B):
        for pos in range(int(kv_len[b])):
            page = int(block_table[b, pos // P])
            pages[page, :, pos % P] = cache[b, :, pos]
    return pages


def commit_paged(k_pages, v_pages, block_table, kv_len, k_tree, v_tree, path_nodes, accept_len):
    """Returns new (k_pages, v_pages, kv_len) for the paged layout."""
    k_pages, v_pages = k_pages.copy(), v_pages.copy()
    kv_len = np.array(kv_len, dtype=np.int64).copy()
    P = k_pages.shape[2]
    for b in range(len(accept_len)):
        a = int(accept_len[b])
        for p in range(1, a + 1):
            node = int(path_nodes[b, p])
            pos = kv_len[b] + p - 1
            page = int(block_table[b, pos // P])
            k_pages[page, :, pos % P] = k_tree[b, :, node]
            v_pages[page, :, pos % P] = v_tree[b, :, node]
        kv_len[b] += a
    return k_pages, v_pages, kv_len
