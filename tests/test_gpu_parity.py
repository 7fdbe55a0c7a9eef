"""GPU parity: every stage of the CUDA path against the fp64 oracle.

Each case runs the full step's kernels through the C ABI on seeded inputs
and compares them with the oracle on the same inputs:
  * draft top-k tokens bit-exact, confidences and ln Z within 1e-5 relative;
  * tree (tokens, parents, depths, scores, gids, rows) and mask bit-exact
    when the CUDA tree build is given the oracle's float32 confidences;
  * the chained CUDA draft -> tree result equal to the oracle's, except
    where the oracle's scores hold a near-tie (float32 rounding of c);
  * attention within 2e-2 absolute (bf16) / 1e-4 (fp32) of fp64;
  * greedy walks bit-exact; sampling walks bit-exact up to the first
    decision the oracle flags as within rounding of its boundary.
The full-size cases use the workloads' own shapes and launch configuration;
where the oracle would take minutes it checks a sample of sequences/outputs.
"""
import numpy as np
import pytest
import torch

import gen
import tree_speculative_decoding_eagle_gb300 as eg
from oracle import draft as odraft
from oracle import mask as omask
from oracle import verify as over

from paritylib import (ATTN_TOL, LSE_TOL, Case, attn_expected, attn_group_expected, compare_draft,
                       compare_tree, compare_walk, f64, fill_trees, near_tie, oracle_tree_stage)

pytestmark = pytest.mark.gpu

W = gen.WORKLOADS
S = gen.scaled

CASES = {
    "tiny": Case(W["tiny"], [0]),
    "ragged-bf16": Case(S(W["llama2-13b-b8"], name="ragged-bf16", B=3, V=5000, D=4, k=5, m=30,
                          Hq=8, Hkv=2, dh=128, L=300, L_min=0, modes=("greedy", "sample")),
                        [0, 1, 2]),
    "wide-tree": Case(S(W["llama2-7b-b1"], name="wide-tree", B=2, V=2048, D=4, k=6, m=70, Hq=4,
                        Hkv=4, dh=64, L=64, L_min=64, modes=("greedy", "sample")), [0, 1]),
    "chain-k1": Case(S(W["tiny"], name="chain-k1", B=2, V=512, D=5, k=1, m=5, Hq=2, Hkv=1,
                       L=40, L_min=40, modes=("greedy", "sample")), [0, 1]),
    "one-level": Case(S(W["tiny"], name="one-level", B=2, V=256, D=1, k=8, m=3, Hq=2, Hkv=2,
                        dtype="bf16", modes=("greedy", "sample")), [0, 1]),
    "all-candidates": Case(S(W["tiny"], name="all-candidates", B=1, V=96, D=3, k=3, m=21,
                             modes=("greedy", "sample"), temperature=0.7), [0]),
    "llama2-7b-b1": Case(W["llama2-7b-b1"], [0]),
    "llama2-13b-b8": Case(W["llama2-13b-b8"], list(range(8)),
                          attn_samples=[(b, i, h) for b in (0, 5, 7) for i in (0, 17, 50)
                                        for h in (0, 39)]),
    # GQA 8: rows are (node, grouped head) pairs; whole groups cover every
    # 128-row M-tile of the launch, the sampled outputs other sequences
    "llama2-70b-b16": Case(W["llama2-70b-b16"], list(range(16)),
                           attn_samples=[(b, i, h) for b in (0, 9, 15) for i in (0, 23, 48)
                                         for h in (0, 7, 8, 63)],
                           attn_groups=[(0, 0), (15, 7), (6, 3)]),
    "gpt-oss-20b-b64": Case(W["gpt-oss-20b-b64"], [0, 21, 63],
                            attn_samples=[(b, i, h) for b in (0, 33, 63) for i in (0, 30, 60)
                                          for h in (0, 15, 63)],
                            attn_groups=[(0, 0), (63, 7), (33, 4)]),
}


def run_case(case):
    w = case.w
    n = w.n_nodes
    big = w.B * w.D * w.k * w.V > 50_000_000
    gdev = "cuda" if big else "cpu"
    draft = gen.draft_logits(w, device=gdev)
    draft_gpu = draft.cuda()
    seqs = case.oracle_seqs
    draft_cpu = torch.zeros((w.B, w.D, w.k, w.V), dtype=torch.float32) if big else draft.float()
    if big:
        for b in seqs:
            draft_cpu[b] = draft[b].float().cpu()
    ws = eg.Workspace()

    # ---- stage 1: draft softmax / top-k -----------------------------------
    tok_g, conf_g, stats_g = eg.draft_topk(draft_gpu, w.k, workspace=ws)
    tok_o, conf_o, stats_o, trees = oracle_tree_stage(w, draft_cpu.numpy(), seqs)
    compare_draft(w, tok_g.cpu().numpy(), conf_g.cpu().numpy(), stats_g.cpu().numpy(),
                  tok_o, conf_o, stats_o, seqs)
    # a second call on the same workspace (split tickets must have reset)
    tok_2, conf_2, _ = eg.draft_topk(draft_gpu, w.k, workspace=ws)
    for d, j in odraft.used_rows(w.D, w.k):   # other rows are never written
        assert torch.equal(tok_2[:, d, j], tok_g[:, d, j]) and torch.equal(conf_2[:, d, j], conf_g[:, d, j])

    # ---- stage 2: tree on the oracle's confidences --------------------------
    ref = seqs[0]
    tok_in = np.stack([tok_o[b] if b in trees else tok_o[ref] for b in range(w.B)])
    conf_in = np.stack([np.nan_to_num(conf_o[b] if b in trees else conf_o[ref]) for b in range(w.B)])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tg = eg.tree_build(torch.from_numpy(tok_in.astype(np.int32)).cuda(),
                       torch.from_numpy(conf_in.astype(np.float32)).cuda(), w.m, status=status)
    got = {k_: v.cpu().numpy() for k_, v in tg.items()}
    for b in range(w.B):
        want = trees[b] if b in trees else trees[ref]
        compare_tree({k_: got[k_][b] for k_ in got}, want, got["mask"][b].view(np.uint64))
    assert int(status.item()) == 0

    # ---- stage 1 -> 2 chained on the GPU ------------------------------------
    te = eg.tree_build(tok_g, conf_g, w.m)
    mism = 0
    for b in seqs:
        same = all((te[k_][b].cpu().numpy() == trees[b][k_]).all()
                   for k_ in ("tok", "parent", "depth", "src"))
        if not same:
            mism += 1
            assert near_tie(trees[b]), f"sequence {b}: trees differ without a near-tie"
    assert mism <= max(1, len(seqs) // 4)

    # ---- mask kernel on the oracle's parents --------------------------------
    nodes = fill_trees(w, trees)
    par_gpu = torch.from_numpy(nodes["parent"].astype(np.int32)).cuda()
    mk = eg.tree_mask(par_gpu).cpu().numpy().view(np.uint64)
    masks_bool = np.stack([omask.tree_mask(nodes["parent"][b]) for b in range(w.B)])
    assert (mk == omask.pack_mask(masks_bool)).all()

    # ---- stage 3: attention ---------------------------------------------------
    ai = gen.attention_inputs(w, device=gdev)
    ai_gpu = {k_: v.cuda() for k_, v in ai.items()}
    mask_gpu = torch.from_numpy(omask.pack_mask(masks_bool).view(np.int64)).cuda()
    out_g, lse_g = eg.tree_attn(ai_gpu["q"], ai_gpu["k_cache"], ai_gpu["v_cache"],
                                ai_gpu["kv_len"], ai_gpu["k_tree"], ai_gpu["v_tree"], mask_gpu,
                                workspace=ws)
    out_g, lse_g = f64(out_g), lse_g.cpu().numpy()
    tol = ATTN_TOL[w.dtype]
    ai_cpu = {k_: v.cpu() for k_, v in ai.items()}
    exp = attn_expected(case, ai_cpu, masks_bool)
    if case.attn_samples is None:
        o, l = exp
        assert np.abs(out_g - o).max() <= tol
        assert np.abs(lse_g - l).max() <= LSE_TOL
    else:
        for (b, i, h), (o, l) in exp.items():
            assert np.abs(out_g[b, i, h] - o).max() <= tol, (b, i, h)
            assert abs(lse_g[b, i, h] - l) <= LSE_TOL, (b, i, h)
    G = w.Hq // w.Hkv
    for (b, g) in case.attn_groups:
        o, l = attn_group_expected(ai_cpu, masks_bool, b, g, G, w.dh ** -0.5)
        assert np.abs(out_g[b, :, g * G:(g + 1) * G] - o).max() <= tol, (b, g)
        assert np.abs(lse_g[b, :, g * G:(g + 1) * G] - l).max() <= LSE_TOL, (b, g)
    del ai_gpu, ai

    # ---- stage 4: verification -------------------------------------------------
    target = gen.target_logits(w, draft, nodes["row"], device=gdev)
    target_gpu = target.cuda()
    u = gen.uniforms(w)
    u_gpu = torch.from_numpy(u).cuda()
    ntok_gpu = torch.from_numpy(nodes["tok"].astype(np.int32)).cuda()
    taus = {}
    for mode in w.modes:
        acc, path, toks = eg.verify(target_gpu, ntok_gpu, par_gpu, w.D, mode, w.temperature,
                                    u_gpu if mode == "sample" else None, workspace=ws)
        acc, path, toks = acc.cpu().numpy(), path.cpu().numpy(), toks.cpu().numpy()
        walks, acc_o = {}, np.zeros(w.B, dtype=np.int64)
        path_o = np.full((w.B, w.D + 1), -1)
        tok_ow = np.full((w.B, w.D + 1), -1)
        for b in seqs:
            tb = target[b].float().cpu().numpy()
            if mode == "greedy":
                r = over.verify_greedy(tb, nodes["tok"][b], nodes["parent"][b])
            else:
                r = over.verify_sample(tb, nodes["tok"][b], nodes["parent"][b], w.temperature, u[b])
            walks[b] = r
            acc_o[b] = r.accept_len
            path_o[b, :len(r.path)] = r.path
            tok_ow[b, :len(r.tokens)] = r.tokens
        # an accept test is flagged with probability about 2e-5 Z / R (R the
        # residual mass), so over a case's few hundred tests at most one is
        n_amb = compare_walk(w, mode, acc, path, toks, (acc_o, path_o, tok_ow, walks), seqs)
        assert n_amb <= 1
        taus[mode] = float(np.mean([acc_o[b] for b in seqs]))
    return taus


@pytest.mark.parametrize("name", list(CASES))
def test_parity(name):
    taus = run_case(CASES[name])
    print(name, "mean accepted length", taus)


def test_out_of_domain_confidence_sets_status():
    k, D, m = 3, 2, 4
    tok = torch.tensor([[[[0, 1, 2], [0, 0, 0], [0, 0, 0]],
                         [[3, 4, 5], [6, 7, 8], [9, 10, 11]]]], dtype=torch.int32).cuda()
    conf = torch.full((1, D, k, k), 0.3).cuda()
    conf[0, 1, 1, 0] = 1.5
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    eg.tree_build(tok, conf, m, status=status)
    assert int(status.item()) == -1


def test_empty_prefix_and_unit_mask_attention():
    w = S(W["tiny"], name="empty-prefix", B=2, L=16, L_min=0, dtype="bf16")
    ai = gen.attention_inputs(w)
    ai["kv_len"] = torch.tensor([0, 16], dtype=torch.int32)
    n = w.n_nodes
    par = np.array([-1] + [0] * (n - 1))          # a star: every node under the root
    masks = np.stack([omask.tree_mask(par)] * 2)
    g = {k_: v.cuda() for k_, v in ai.items()}
    out, lse = eg.tree_attn(g["q"], g["k_cache"], g["v_cache"], g["kv_len"], g["k_tree"],
                            g["v_tree"], torch.from_numpy(omask.pack_mask(masks).view(np.int64)).cuda())
    case = Case(w, [0, 1])
    o, l = attn_expected(case, ai, masks)
    assert np.abs(f64(out) - o).max() <= ATTN_TOL["bf16"]
    assert np.abs(lse.cpu().numpy() - l).max() <= LSE_TOL
