"""GPU parity of the bf16 tree attention across KV-split counts.

When few (sequence, KV head, M-group) work items exist, the launch splits the
KV range S ways and the S CTAs of an item form a thread-block cluster that
merges its partial results: through the workspace when the launch is one wave
(every case here), else through distributed shared memory (the 13B-shaped
parity case).  These shapes
make the launch plan pick S = 1..8, with one and two 128-row M-tiles per CTA
and both head sizes; lengths are ragged (one sequence may have an empty
prefix, leaving whole splits empty) and every case runs twice on the same
buffers.  Sampled rows must match the oracle's attention within the bf16
tolerance, and both calls must agree bit for bit.
"""
import numpy as np
import pytest
import torch

import gen
import tree_speculative_decoding_eagle_gb300 as eg
from oracle import attn as oattn
from oracle import mask as omask

pytestmark = pytest.mark.gpu

W = gen.WORKLOADS

# (B, m, Hq, Hkv, dh, L): the launch plan's S in the comment
CASES = {
    "S1-dh128": (1, 60, 8, 8, 128, 128),     # S = 1
    "S2-dh64": (2, 39, 16, 16, 64, 256),      # S = 2
    "S3-dh128": (1, 60, 8, 8, 128, 192),      # S = 3
    "S4-dh128": (1, 60, 8, 8, 128, 256),      # S = 4
    "S5-dh64": (2, 39, 16, 16, 64, 640),      # S = 5
    "S6-dh128": (1, 60, 8, 8, 128, 384),      # S = 6
    "S7-dh128": (1, 60, 8, 8, 128, 448),      # S = 7
    "S8-dh128": (1, 60, 8, 8, 128, 512),      # S = 8
    "S6-gqa8-2mtiles": (1, 60, 64, 8, 64, 768),   # S = 6, two M-tiles per CTA
    "S8-gqa8-2mtiles": (1, 60, 64, 8, 64, 1024),  # S = 8, two M-tiles per CTA
}


def random_tree_mask(n, B, seed):
    rng = np.random.default_rng(seed)
    masks = []
    for _ in range(B):
        par = [-1] + [int(rng.integers(max(0, i - 6), i)) for i in range(1, n)]
        masks.append(omask.tree_mask(np.array(par)))
    return np.stack(masks)


@pytest.mark.parametrize("name", list(CASES))
def test_split_attention(name):
    B, m, Hq, Hkv, dh, L = CASES[name]
    w = gen.scaled(W["tiny"], name=name, B=B, m=m, Hq=Hq, Hkv=Hkv, dh=dh, L=L, L_min=L // 3,
                   dtype="bf16", seed=2100 + len(name))
    ai = gen.attention_inputs(w)
    if B > 1:
        ai["kv_len"][0] = 0          # an empty prefix: the splits of its heads are empty
    n = w.n_nodes
    masks = random_tree_mask(n, B, 2200 + len(name))
    g = {k: v.cuda() for k, v in ai.items()}
    mask_gpu = torch.from_numpy(omask.pack_mask(masks).view(np.int64)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out1, lse1 = eg.tree_attn(g["q"], g["k_cache"], g["v_cache"], g["kv_len"], g["k_tree"], g["v_tree"],
                              mask_gpu, status=status)
    out2, lse2 = eg.tree_attn(g["q"], g["k_cache"], g["v_cache"], g["kv_len"], g["k_tree"], g["v_tree"],
                              mask_gpu, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    f64 = lambda t: t.double().cpu().numpy()
    q, kc, vc, kt, vt = (f64(ai[k]) for k in ("q", "k_cache", "v_cache", "k_tree", "v_tree"))
    kv_len = ai["kv_len"].numpy()
    o_g, l_g = f64(out1), lse1.cpu().numpy()
    rng = np.random.default_rng(2300 + len(name))
    for b in range(B):
        nodes = sorted(set([0, n - 1] + list(rng.choice(n, size=min(n, 12), replace=False))))
        heads = sorted(set([0, Hq - 1] + list(rng.choice(Hq, size=min(Hq, 4), replace=False))))
        for i in nodes:
            for h in heads:
                o, l = oattn.attention_row(q, kc, vc, kv_len, kt, vt, masks, dh ** -0.5, b, int(i), int(h))
                assert np.abs(o_g[b, i, h] - o).max() <= 2e-2, (b, i, h)
                assert abs(float(l_g[b, i, h]) - l) <= 1e-3, (b, i, h)
