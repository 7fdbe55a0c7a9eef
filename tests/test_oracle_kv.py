"""Pins for the oracle's KV commit and paged layout.

Independent checks:
  * a commit worked by hand (positions, new kv_len, slot mapping with -1 for
    the rejected node);
  * paged layout: scattering a contiguous cache into pages through a random
    block table and gathering it back is the identity;
  * the paged commit equals the contiguous commit seen through the pages.
"""
import numpy as np

from oracle import kv as okv


def test_hand_worked_commit():
    k_cache = np.zeros((1, 1, 6, 2))
    k_cache[0, 0, :3] = [[1, 1], [2, 2], [3, 3]]
    v_cache = -k_cache
    k_tree = np.array([[[[10, 10], [11, 11], [12, 12], [13, 13]]]], dtype=float)
    v_tree = -k_tree
    path = np.array([[0, 2, 3, -1]])
    acc = np.array([2])
    kc, vc, kl = okv.commit_contiguous(k_cache, v_cache, [3], k_tree, v_tree, path, acc)
    assert kl.tolist() == [5]
    assert kc[0, 0].tolist() == [[1, 1], [2, 2], [3, 3], [12, 12], [13, 13], [0, 0]]
    assert vc[0, 0, 3:5].tolist() == [[-12, -12], [-13, -13]]
    assert okv.slot_mapping(path, acc, [3], 4).tolist() == [[2, -1, 3, 4]]


def random_paged(rng, B=3, Hkv=2, dh=4, P=4, Lmax=16):
    pages_per = Lmax // P
    num_pages = B * pages_per + 3
    perm = rng.permutation(num_pages)[:B * pages_per].reshape(B, pages_per)
    kv_len = rng.integers(1, Lmax - 3, size=B)
    cache = rng.standard_normal((B, Hkv, Lmax, dh))
    for b in range(B):
        cache[b, :, kv_len[b]:] = 0
    pages = np.zeros((num_pages, Hkv, P, dh))
    return cache, perm, kv_len, pages


def test_scatter_gather_identity():
    rng = np.random.default_rng(5)
    for _ in range(10):
        cache, bt, kv_len, pages = random_paged(rng)
        okv.scatter_pages(cache, bt, kv_len, pages)
        back = okv.gather_pages(pages, bt, kv_len, cache.shape[2])
        np.testing.assert_array_equal(back, cache)


def test_paged_commit_matches_contiguous():
    rng = np.random.default_rng(6)
    for _ in range(10):
        cache, bt, kv_len, kp = random_paged(rng)
        vcache = -cache
        vp = np.zeros_like(kp)
        okv.scatter_pages(cache, bt, kv_len, kp)
        okv.scatter_pages(vcache, bt, kv_len, vp)
        B, Hkv, _, dh = cache.shape
        n = 5
        k_tree = rng.standard_normal((B, Hkv, n, dh))
        v_tree = rng.standard_normal((B, Hkv, n, dh))
        acc = rng.integers(0, 3, size=B)
        path = np.full((B, 4), -1)
        for b in range(B):
            path[b, 0] = 0
            path[b, 1:acc[b] + 1] = rng.choice(np.arange(1, n), size=acc[b], replace=False)
        kc, vc, kl = okv.commit_contiguous(cache, vcache, kv_len, k_tree, v_tree, path, acc)
        kp2, vp2, kl2 = okv.commit_paged(kp, vp, bt, kv_len, k_tree, v_tree, path, acc)
        assert (kl == kl2).all()
        np.testing.assert_array_equal(okv.gather_pages(kp2, bt, kl2, cache.shape[2]), kc)
        np.testing.assert_array_equal(okv.gather_pages(vp2, bt, kl2, cache.shape[2]), vc)
