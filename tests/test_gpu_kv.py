"""GPU parity of the paged-prefix tree attention and the KV commit.

  * eagle_tree_attn_paged: the contiguous cache is scattered into a page pool
    through a shuffled block table (oracle layout helpers); the paged kernel
    must match the oracle's attention on the contiguous cache within the bf16
    tolerance, and the contiguous kernel (same logical capacity, same launch
    plan) bit for bit.  Page sizes below, equal to and above the key tile.
  * eagle_kv_commit: random accepted paths committed on the GPU into both
    layouts equal the oracle's commit, slot mapping and new lengths.
  * Errors: an unmapped page the prefix uses, and a commit past the cache's
    capacity, set EAGLE_ERR_INVALID (nothing faults).
"""
import numpy as np
import pytest
import torch

import gen
import tree_speculative_decoding_eagle_gb300 as eg
from oracle import attn as oattn
from oracle import kv as okv
from oracle import mask as omask

pytestmark = pytest.mark.gpu


def random_tree_mask(n, B, seed):
    rng = np.random.default_rng(seed)
    masks = []
    for _ in range(B):
        par = [-1] + [int(rng.integers(max(0, i - 8), i)) for i in range(1, n)]
        masks.append(omask.tree_mask(np.array(par)))
    return np.stack(masks)


def paged_copy(cache, kv_len, page_size, rng, extra=5):
    """Scatter [B, Hkv, Lmax, dh] into a pool through a shuffled block table."""
    B, Hkv, Lmax, dh = cache.shape
    max_pages = Lmax // page_size
    num_pages = B * max_pages + extra
    table = rng.permutation(num_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    pages = np.zeros((num_pages, Hkv, page_size, dh), dtype=np.float32)
    okv.scatter_pages(cache, table, kv_len, pages)
    return pages, table


CASES = {
    "7b-p16": dict(wl="llama2-7b-b1", B=2, L=1024, L_min=700, page=16),
    "7b-p256": dict(wl="llama2-7b-b1", B=2, L=2048, L_min=1500, page=256),
    "70b-p64": dict(wl="llama2-70b-b16", B=3, L=1024, L_min=300, page=64),
    "oss-p16": dict(wl="gpt-oss-20b-b64", B=2, L=1024, L_min=900, page=16),
    "oss-p128": dict(wl="gpt-oss-20b-b64", B=2, L=2048, L_min=2048, page=128),
}


@pytest.mark.parametrize("name", list(CASES))
def test_paged_attention(name):
    c = CASES[name]
    w = gen.scaled(gen.WORKLOADS[c["wl"]], name=name, B=c["B"], L=c["L"], L_min=c["L_min"], seed=1400 + len(name))
    ai = gen.attention_inputs(w)
    kv_len = ai["kv_len"].numpy()
    rng = np.random.default_rng(1500 + len(name))
    kp, table = paged_copy(ai["k_cache"].float().numpy(), kv_len, c["page"], rng)
    vp, _ = paged_copy(ai["v_cache"].float().numpy(), kv_len, c["page"], np.random.default_rng(1500 + len(name)))
    n = w.n_nodes
    masks = random_tree_mask(n, w.B, 1600 + len(name))
    mask_gpu = torch.from_numpy(omask.pack_mask(masks).view(np.int64)).cuda()
    g = {k: v.cuda() for k, v in ai.items()}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_p, lse_p = eg.tree_attn_paged(g["q"], torch.from_numpy(kp).to(torch.bfloat16).cuda(),
                                      torch.from_numpy(vp).to(torch.bfloat16).cuda(),
                                      torch.from_numpy(table).cuda(), g["kv_len"], g["k_tree"], g["v_tree"],
                                      mask_gpu, status=status)
    out_c, lse_c = eg.tree_attn(g["q"], g["k_cache"], g["v_cache"], g["kv_len"], g["k_tree"], g["v_tree"],
                                mask_gpu)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out_p, out_c) and torch.equal(lse_p, lse_c)
    f64 = lambda t: t.double().cpu().numpy()
    q, kc, vc, kt, vt = (f64(ai[k]) for k in ("q", "k_cache", "v_cache", "k_tree", "v_tree"))
    for b in range(w.B):
        for i in (0, n // 2, n - 1):
            for h in (0, w.Hq - 1):
                o, l = oattn.attention_row(q, kc, vc, kv_len, kt, vt, masks, w.dh ** -0.5, b, i, h)
                assert np.abs(f64(out_p[b, i, h]) - o).max() <= 2e-2
                assert abs(float(lse_p[b, i, h]) - l) <= 1e-3


def test_unmapped_page_sets_status():
    w = gen.scaled(gen.WORKLOADS["llama2-7b-b1"], name="bad-page", B=1, L=512, L_min=512, seed=1700)
    ai = gen.attention_inputs(w)
    kp, table = paged_copy(ai["k_cache"].float().numpy(), ai["kv_len"].numpy(), 64, np.random.default_rng(1))
    table[0, 3] = -1                                  # a page the prefix uses
    kpg = torch.from_numpy(kp).to(torch.bfloat16).cuda()
    masks = random_tree_mask(w.n_nodes, 1, 2)
    g = {k: v.cuda() for k, v in ai.items()}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    eg.tree_attn_paged(g["q"], kpg, kpg, torch.from_numpy(table).cuda(), g["kv_len"], g["k_tree"], g["v_tree"],
                       torch.from_numpy(omask.pack_mask(masks).view(np.int64)).cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -1


def random_paths(B, n, D, rng):
    acc = rng.integers(0, D + 1, size=B)
    path = np.full((B, D + 1), -1, dtype=np.int64)
    for b in range(B):
        path[b, 0] = 0
        path[b, 1:acc[b] + 1] = rng.choice(np.arange(1, n), size=acc[b], replace=False)
    return acc, path


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_kv_commit(paged, dtype):
    rng = np.random.default_rng(1800 + paged + 2 * (dtype == "bf16"))
    B, Hkv, Lmax, dh, n, D, P = 4, 3, 256, 64, 20, 6, 16
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    kv_len = rng.integers(1, Lmax - D, size=B)
    cache_k = torch.randn((B, Hkv, Lmax, dh)).to(td)
    cache_v = torch.randn((B, Hkv, Lmax, dh)).to(td)
    for b in range(B):
        cache_k[b, :, kv_len[b]:] = 0
        cache_v[b, :, kv_len[b]:] = 0
    k_tree = torch.randn((B, Hkv, n, dh)).to(td)
    v_tree = torch.randn((B, Hkv, n, dh)).to(td)
    acc, path = random_paths(B, n, D, rng)
    kc_o, vc_o, kl_o = okv.commit_contiguous(cache_k.float().numpy(), cache_v.float().numpy(), kv_len,
                                             k_tree.float().numpy(), v_tree.float().numpy(), path, acc)
    slots_o = okv.slot_mapping(path, acc, kv_len, n)
    kl = torch.from_numpy(kv_len.astype(np.int32)).cuda()
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x).astype(np.int32)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if paged:
        pk, table = paged_copy(cache_k.float().numpy(), kv_len, P, rng)
        pv = np.zeros_like(pk)
        okv.scatter_pages(cache_v.float().numpy(), table, kv_len, pv)
        pk_g, pv_g = torch.from_numpy(pk).to(td).cuda(), torch.from_numpy(pv).to(td).cuda()
        slots = eg.kv_commit(k_tree.cuda(), v_tree.cuda(), dev(acc), dev(path), pk_g, pv_g, kl,
                             block_table=dev(table), status=status)
        got_k = okv.gather_pages(pk_g.float().cpu().numpy(), table, kl_o, Lmax)
        got_v = okv.gather_pages(pv_g.float().cpu().numpy(), table, kl_o, Lmax)
    else:
        ck, cv = cache_k.cuda(), cache_v.cuda()
        slots = eg.kv_commit(k_tree.cuda(), v_tree.cuda(), dev(acc), dev(path), ck, cv, kl, status=status)
        got_k, got_v = ck.float().cpu().numpy(), cv.float().cpu().numpy()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert (kl.cpu().numpy() == kl_o).all()
    assert (slots.cpu().numpy() == slots_o).all()
    np.testing.assert_array_equal(got_k, kc_o)
    np.testing.assert_array_equal(got_v, vc_o)


def test_kv_commit_past_capacity_sets_status():
    B, Hkv, Lmax, dh, n, D = 1, 1, 8, 64, 5, 3
    ck = torch.zeros((B, Hkv, Lmax, dh), dtype=torch.bfloat16, device="cuda")
    tree = torch.ones((B, Hkv, n, dh), dtype=torch.bfloat16, device="cuda")
    kl = torch.tensor([7], dtype=torch.int32, device="cuda")         # 7 + 2 > 8
    acc = torch.tensor([2], dtype=torch.int32, device="cuda")
    path = torch.tensor([[0, 1, 2, -1]], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    eg.kv_commit(tree, tree, acc, path, ck, ck.clone(), kl, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -1 and int(kl.item()) == 7 and float(ck.abs().sum()) == 0.0


def test_paged_attention_full_size_whole_groups():
    """70B-shaped GQA 8 at its full batch (16 sequences, 4096-token prefix,
    the unsplit two-M-tile launch), prefix in 64-token pages behind a
    shuffled block table built on the device: bit-identical to the
    contiguous kernel everywhere, and every (node, grouped head) output of
    whole (sequence, KV head) groups within the bf16 tolerance of the
    oracle."""
    from paritylib import attn_group_expected
    w = gen.WORKLOADS["llama2-70b-b16"]
    ai = gen.attention_inputs(w, device="cuda")
    B, Hkv, Lmax, dh = ai["k_cache"].shape
    P = 64
    mp = Lmax // P
    num_pages = B * mp + 16
    gcpu = torch.Generator().manual_seed(1900)
    table = torch.randperm(num_pages, generator=gcpu)[:B * mp].view(B, mp).to(torch.int32).cuda()
    idx = table.reshape(-1).long()

    def pool(cache):
        p = torch.zeros((num_pages, Hkv, P, dh), dtype=cache.dtype, device="cuda")
        p[idx] = cache.view(B, Hkv, mp, P, dh).permute(0, 2, 1, 3, 4).reshape(B * mp, Hkv, P, dh)
        return p

    kp, vp = pool(ai["k_cache"]), pool(ai["v_cache"])
    n = w.n_nodes
    masks = random_tree_mask(n, B, 1901)
    mask_gpu = torch.from_numpy(omask.pack_mask(masks).view(np.int64)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_p, lse_p = eg.tree_attn_paged(ai["q"], kp, vp, table, ai["kv_len"], ai["k_tree"], ai["v_tree"],
                                      mask_gpu, status=status)
    out_c, lse_c = eg.tree_attn(ai["q"], ai["k_cache"], ai["v_cache"], ai["kv_len"], ai["k_tree"],
                                ai["v_tree"], mask_gpu)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out_p, out_c) and torch.equal(lse_p, lse_c)
    del kp, vp
    ai_cpu = {k: v.cpu() for k, v in ai.items()}
    G = w.Hq // w.Hkv
    got = out_p.double().cpu().numpy()
    lse = lse_p.cpu().numpy()
    for (b, g) in ((0, 0), (B - 1, Hkv - 1), (9, 2)):
        o, l = attn_group_expected(ai_cpu, masks, b, g, G, dh ** -0.5)
        assert np.abs(got[b, :, g * G:(g + 1) * G] - o).max() <= 2e-2, (b, g)
        assert np.abs(lse[b, :, g * G:(g + 1) * G] - l).max() <= 1e-3, (b, g)
