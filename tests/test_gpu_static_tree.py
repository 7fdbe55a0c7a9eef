"""GPU parity of the EAGLE-1 static draft tree (eagle_static_tree).

[EAGLE-2] sections "背景" and "EAGLE-1からの変更点".  The CUDA kernel gets the
oracle's draft top-k (from the oracle's stage 1) and a template, and must
reproduce the oracle's static tree bit for bit (tokens, parents, depths,
scores, rows, mask).  Invalid templates must raise EAGLE_ERR_INVALID in the
status word (the kernel validates the whole template before it indexes
anything with it).  The static tree then drives the unchanged attention and
verification kernels, compared with the oracle on the same tree.
"""
import json
import os

import numpy as np
import pytest
import torch

import gen
import tree_speculative_decoding_eagle_gb300 as eg
from oracle import attn as oattn
from oracle import draft as odraft
from oracle import mask as omask
from oracle import static_tree as ost
from oracle import verify as over

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def dev32(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).cuda()


def run_static(tok, conf, parent, rank):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = eg.static_tree(dev32(tok), torch.from_numpy(np.ascontiguousarray(conf, dtype=np.float32)).cuda(),
                         dev32(parent), dev32(rank), status=status)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}, int(status.item())


def oracle_rows(w):
    logits = gen.draft_logits(w).float().numpy()
    tok = np.zeros((w.B, w.D, w.k, w.k), dtype=np.int64)
    conf = np.zeros((w.B, w.D, w.k, w.k), dtype=np.float32)
    for b in range(w.B):
        t, c, _ = odraft.draft_topk(logits[b:b + 1], w.k)
        tok[b], conf[b] = np.where(t[0] < 0, 0, t[0]), np.nan_to_num(c[0]).astype(np.float32)
    return logits, tok, conf


def test_hand_worked_static_tree_on_gpu():
    with open(os.path.join(GOLDEN, "hand_static.json")) as f:
        h = json.load(f)
    got, st = run_static(np.array(h["tok"])[None], np.array(h["conf"], dtype=np.float32)[None],
                         h["parent"], h["rank"])
    assert st == 0
    want = ost.build_static_tree(np.array(h["tok"]), np.array(h["conf"], dtype=np.float32),
                                 h["parent"], h["rank"])
    assert list(got["tok"][0]) == h["expect"]["tok"]
    for key in ("tok", "parent", "depth", "score", "src", "row"):
        assert (got[key][0] == want[key]).all(), key


SHAPES = {
    "template-60": (gen.STATIC_SHAPE_60, dict(B=2, V=32000, D=6, k=10)),
    "narrow": (([3], [2, 1], [1, 1]), dict(B=3, V=500, D=3, k=3)),
    "deep": (([8], [4, 2, 1], [3, 1], [2], [1], [1], [1]), dict(B=2, V=2048, D=7, k=8)),
    "one-level": (([5],), dict(B=2, V=300, D=1, k=5)),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_static_tree_matches_oracle(name):
    shape, s = SHAPES[name]
    parent, rank = gen.static_template(shape)
    w = gen.scaled(gen.WORKLOADS["llama2-7b-b1"], name=name, m=len(parent) - 1, seed=900, **s)
    _, tok, conf = oracle_rows(w)
    got, st = run_static(tok, conf, parent, rank)
    assert st == 0
    want = ost.build_static_trees(tok, conf, parent, rank)
    for key in ("tok", "parent", "depth", "score", "src", "row"):
        assert (got[key] == want[key]).all(), key
    for b in range(w.B):
        assert (got["mask"][b].view(np.uint64) == omask.pack_mask(omask.tree_mask(want["parent"][b]))).all()


@pytest.mark.parametrize("parent,rank", [
    ([0, 0], [0, 0]),                              # root not -1
    ([-1, 0, 2], [0, 0, 0]),                       # parent after child
    ([-1, 0, 0], [0, 1, 1]),                       # duplicate sibling rank
    ([-1, 0], [0, 2]),                             # rank >= k
    ([-1, 0, 1, 2, 3], [0, 0, 0, 0, 0]),           # deeper than D
    ([-1, 0, 0, 1, 2, 0], [0, 0, 1, 0, 0, 1]),     # rank clash at the root
])
def test_invalid_template_sets_status(parent, rank):
    tok = np.zeros((1, 3, 2, 2), dtype=np.int64)
    conf = np.full((1, 3, 2, 2), 0.5, dtype=np.float32)
    _, st = run_static(tok, conf, parent, rank)
    assert st == -1  # EAGLE_ERR_INVALID


def test_static_tree_drives_attention_and_verify():
    parent, rank = gen.static_template(gen.STATIC_SHAPE_60)
    w = gen.scaled(gen.WORKLOADS["llama2-7b-b1"], name="static-chain", B=2, V=4096, m=len(parent) - 1,
                   Hq=8, Hkv=2, dh=128, L=300, L_min=100, modes=("greedy", "sample"), seed=901)
    logits, tok, conf = oracle_rows(w)
    got, st = run_static(tok, conf, parent, rank)
    assert st == 0
    want = ost.build_static_trees(tok, conf, parent, rank)
    # attention over the static tree's mask
    masks_bool = np.stack([omask.tree_mask(want["parent"][b]) for b in range(w.B)])
    ai = gen.attention_inputs(w)
    ai_gpu = {k: v.cuda() for k, v in ai.items()}
    mask_gpu = torch.from_numpy(got["mask"]).cuda()
    out_g, lse_g = eg.tree_attn(ai_gpu["q"], ai_gpu["k_cache"], ai_gpu["v_cache"], ai_gpu["kv_len"],
                                ai_gpu["k_tree"], ai_gpu["v_tree"], mask_gpu)
    f64 = lambda t: t.double().cpu().numpy()
    o, l = oattn.tree_attention(f64(ai["q"]), f64(ai["k_cache"]), f64(ai["v_cache"]), ai["kv_len"].numpy(),
                                f64(ai["k_tree"]), f64(ai["v_tree"]), masks_bool, w.dh ** -0.5)
    assert np.abs(f64(out_g) - o).max() <= 2e-2
    assert np.abs(lse_g.cpu().numpy() - l).max() <= 1e-3
    # verification on the static tree's nodes
    target = gen.target_logits(w, torch.from_numpy(logits).to(w.torch_dtype), want["row"])
    u = gen.uniforms(w)
    for mode in ("greedy", "sample"):
        acc, path, toks = eg.verify(target.cuda(), dev32(got["tok"]), dev32(got["parent"]), w.D, mode,
                                    w.temperature, torch.from_numpy(u).cuda() if mode == "sample" else None)
        acc, path = acc.cpu().numpy(), path.cpu().numpy()
        for b in range(w.B):
            tb = target[b].float().numpy()
            r = (over.verify_greedy(tb, want["tok"][b], want["parent"][b]) if mode == "greedy" else
                 over.verify_sample(tb, want["tok"][b], want["parent"][b], w.temperature, u[b]))
            if mode == "greedy" or r.ambiguous is None:
                assert acc[b] == r.accept_len
                assert list(path[b, :len(r.path)]) == list(r.path)
