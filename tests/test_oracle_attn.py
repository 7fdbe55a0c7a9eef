"""Pins for the oracle's tree attention.

Independent checks: PyTorch's scaled_dot_product_attention (a library
routine) in fp64 with an explicit boolean mask, the causal special case for
a chain tree, closed forms (equal keys give the mean of the values; a lone
key gives its value), and the GQA head mapping.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attn as oattn
from oracle import mask as omask


def random_tree(rng, n):
    return np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)])


def make(rng, B, n, Hq, Hkv, dh, Lmax, kv_len):
    q = rng.normal(size=(B, n, Hq, dh))
    kc = rng.normal(size=(B, Hkv, Lmax, dh))
    vc = rng.normal(size=(B, Hkv, Lmax, dh))
    kt = rng.normal(size=(B, Hkv, n, dh))
    vt = rng.normal(size=(B, Hkv, n, dh))
    return q, kc, vc, np.asarray(kv_len), kt, vt


def sdpa_reference(q, kc, vc, kv_len, kt, vt, mask, scale):
    B, n, Hq, dh = q.shape
    Hkv = kc.shape[1]
    G = Hq // Hkv
    out = np.zeros_like(q)
    for b in range(B):
        L = int(kv_len[b])
        for h in range(Hq):
            g = h // G
            K = torch.from_numpy(np.concatenate([kc[b, g, :L], kt[b, g]]))
            V = torch.from_numpy(np.concatenate([vc[b, g, :L], vt[b, g]]))
            allowed = torch.from_numpy(np.concatenate([np.ones((n, L), bool), mask[b]], 1))
            Q = torch.from_numpy(q[b, :, h])
            o = F.scaled_dot_product_attention(Q[None], K[None], V[None],
                                               attn_mask=allowed[None], scale=scale)
            out[b, :, h] = o[0].numpy()
    return out


def test_matches_library_attention_on_random_trees():
    rng = np.random.default_rng(0)
    B, n, Hq, Hkv, dh = 2, 9, 4, 2, 16
    q, kc, vc, kv_len, kt, vt = make(rng, B, n, Hq, Hkv, dh, 20, [20, 7])
    mask = np.stack([omask.tree_mask(random_tree(rng, n)) for _ in range(B)])
    out, lse = oattn.tree_attention(q, kc, vc, kv_len, kt, vt, mask, 0.25)
    ref = sdpa_reference(q, kc, vc, kv_len, kt, vt, mask, 0.25)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    for (b, i, h) in [(0, 0, 0), (1, 8, 3), (1, 4, 2)]:
        o1, l1 = oattn.attention_row(q, kc, vc, kv_len, kt, vt, mask, 0.25, b, i, h)
        np.testing.assert_allclose(o1, out[b, i, h], atol=1e-13)
        assert l1 == pytest.approx(lse[b, i, h], abs=1e-12)


def test_chain_tree_is_causal_attention():
    rng = np.random.default_rng(1)
    n, L, dh = 6, 10, 8
    q, kc, vc, kv_len, kt, vt = make(rng, 1, n, 2, 2, dh, L, [L])
    par = np.arange(-1, n - 1)
    mask = omask.tree_mask(par)[None]
    out, _ = oattn.tree_attention(q, kc, vc, kv_len, kt, vt, mask, dh ** -0.5)
    for h in range(2):
        K = torch.from_numpy(np.concatenate([kc[0, h], kt[0, h]]))
        V = torch.from_numpy(np.concatenate([vc[0, h], vt[0, h]]))
        Qp = torch.from_numpy(np.concatenate([np.zeros((L, dh)), q[0, :, h]]))
        ref = F.scaled_dot_product_attention(Qp[None], K[None], V[None], is_causal=True)
        np.testing.assert_allclose(out[0, :, h], ref[0, L:].numpy(), atol=1e-12)


def test_closed_forms():
    rng = np.random.default_rng(2)
    n, L, dh = 4, 5, 8
    q, kc, vc, kv_len, kt, vt = make(rng, 1, n, 1, 1, dh, L, [L])
    kc[:] = 0.3
    kt[:] = 0.3        # every key equal -> uniform weights
    par = np.array([-1, 0, 1, 0])
    mask = omask.tree_mask(par)[None]
    out, lse = oattn.tree_attention(q, kc, vc, kv_len, kt, vt, mask, 0.5)
    for i in range(n):
        cols = np.nonzero(mask[0, i])[0]
        vals = np.concatenate([vc[0, 0], vt[0, 0, cols]])
        np.testing.assert_allclose(out[0, i, 0], vals.mean(0), atol=1e-13)
        s = 0.5 * 0.3 * q[0, i, 0].sum()
        assert lse[0, i, 0] == pytest.approx(s + np.log(len(vals)), abs=1e-12)
    # empty prefix: the root sees only itself
    out, _ = oattn.tree_attention(q, kc, vc, np.array([0]), kt, vt, mask, 0.5)
    np.testing.assert_allclose(out[0, 0, 0], vt[0, 0, 0], atol=1e-15)


def test_gqa_groups_are_contiguous():
    rng = np.random.default_rng(3)
    n, L, dh = 3, 4, 8
    q, kc, vc, kv_len, kt, vt = make(rng, 1, n, 4, 2, dh, L, [L])
    mask = omask.tree_mask(np.array([-1, 0, 0]))[None]
    out, _ = oattn.tree_attention(q, kc, vc, kv_len, kt, vt, mask, 0.3)
    for h in range(4):
        g = h // 2
        o1, _ = oattn.tree_attention(q[:, :, h:h + 1], kc[:, g:g + 1], vc[:, g:g + 1],
                                     kv_len, kt[:, g:g + 1], vt[:, g:g + 1], mask, 0.3)
        np.testing.assert_allclose(out[:, :, h], o1[:, :, 0], atol=1e-14)
