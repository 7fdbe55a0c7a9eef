"""GPU parity of speculative-sampling verification against the draft
distributions (eagle_verify_draft).

[EAGLE-1] section "検証方法".  The CUDA walk and the fp64 oracle walk the same
tree on the same target rows, draft rows and uniforms; accepted lengths,
paths and tokens must agree exactly up to the first decision the oracle
flags as within rounding of its boundary.  Trees: the static template with
every child token sampled from its parent's q (drafts drawn from q, as the
rule assumes), and the dynamic tree's top-k drafts.
"""
import numpy as np
import pytest
import torch

import gen
import tree_speculative_decoding_eagle_gb300 as eg
from oracle import draft as odraft
from oracle import static_tree as ost
from oracle import tree as otree
from oracle import verify_general as ovg

pytestmark = pytest.mark.gpu


def sampled_static_tree(w, draft_f64, shape, T, rng):
    """Template shape with each node's token drawn from its parent's q."""
    parent, rank = gen.static_template(shape)
    _, row = ost.template_rows(list(parent), w.k, w.D)
    n = len(parent)
    tok = np.full((w.B, n), -1, dtype=np.int64)
    node_row = np.tile(np.array(row, dtype=np.int64), (w.B, 1))
    for b in range(w.B):
        for i in range(1, n):
            d, j = divmod(row[parent[i]], w.k)
            x = draft_f64[b, d, j] / T
            q = np.exp(x - x.max())
            q /= q.sum()
            tok[b, i] = rng.choice(w.V, p=q)
    return tok, np.tile(parent.astype(np.int64), (w.B, 1)), node_row


CASES = {
    "small-f32": dict(wl="tiny", B=3, V=512, D=4, k=4, shape=([4], [2, 1], [1, 1], [1]), T=1.0, dtype="f32"),
    "small-bf16": dict(wl="tiny", B=3, V=1024, D=4, k=4, shape=([4], [3, 1], [2, 1], [1]), T=0.7, dtype="bf16"),
    "7b-template": dict(wl="llama2-7b-b1", B=2, V=32000, D=6, k=10, shape=gen.STATIC_SHAPE_60, T=1.0,
                        dtype="bf16"),
    "oss-wide": dict(wl="gpt-oss-20b-b64", B=3, V=201088, D=3, k=10, shape=([10], [3, 2, 1], [2, 1]), T=1.0,
                     dtype="bf16"),
    # vocabularies that split a sequence over 2 CTAs, and over 3 with a shorter last slice
    "cluster-2": dict(wl="tiny", B=3, V=8192, D=4, k=4, shape=([4], [3, 1], [2, 1], [1]), T=1.0, dtype="bf16"),
    "cluster-3-ragged": dict(wl="tiny", B=3, V=10000, D=4, k=4, shape=([4], [2, 2], [1, 1], [1]), T=0.8,
                             dtype="bf16"),
}


def run_and_compare(w, draft, target, tok, par, row, T, u):
    dd = torch.from_numpy
    acc, path, toks = eg.verify_draft(target.cuda(), draft.cuda(), dd(tok.astype(np.int32)).cuda(),
                                      dd(par.astype(np.int32)).cuda(), dd(row.astype(np.int32)).cuda(), w.D, T,
                                      dd(u).cuda())
    acc, path, toks = acc.cpu().numpy(), path.cpu().numpy(), toks.cpu().numpy()
    acc_o, path_o, tok_o, walks = ovg.verify_batch(target.double().numpy(), draft.double().numpy(), tok, par, row,
                                                   w.k, T, u.astype(np.float64))
    n_amb = 0
    for b in range(w.B):
        if walks[b].ambiguous is None:
            assert acc[b] == acc_o[b], (b, acc[b], acc_o[b])
            assert (path[b] == path_o[b]).all(), b
            assert (toks[b] == tok_o[b]).all(), (b, toks[b], tok_o[b])
        else:
            n_amb += 1
            pos = walks[b].ambiguous[0]
            assert (path[b, :pos + 1] == path_o[b, :pos + 1]).all(), b
    return n_amb, acc_o


@pytest.mark.parametrize("name", list(CASES))
def test_sampled_drafts_match_oracle(name):
    c = CASES[name]
    parent, _ = gen.static_template(c["shape"])
    w = gen.scaled(gen.WORKLOADS[c["wl"]], name=name, B=c["B"], V=c["V"], D=c["D"], k=c["k"],
                   m=len(parent) - 1, dtype=c["dtype"], seed=1200 + len(name))
    draft = gen.draft_logits(w)                        # [B, D, k, V] in the workload dtype
    rng = np.random.default_rng(1300 + len(name))
    tok, par, row = sampled_static_tree(w, draft.double().numpy(), c["shape"], c["T"], rng)
    target = gen.target_logits(w, draft, row)
    u = gen.uniforms(w)
    n_amb, acc_o = run_and_compare(w, draft, target, tok, par, row, c["T"], u)
    assert n_amb <= 1  # flagged walks are rare: none of these cases has one


def test_dynamic_tree_top_k_drafts():
    w = gen.scaled(gen.WORKLOADS["llama2-13b-b8"], name="dyn", B=4, V=8000, seed=1250)
    draft = gen.draft_logits(w)
    df = draft.float().numpy()
    tok = np.zeros((w.B, w.n_nodes), dtype=np.int64)
    par = np.zeros_like(tok)
    row = np.zeros_like(tok)
    for b in range(w.B):
        t, cf, _ = odraft.draft_topk(df[b:b + 1], w.k)
        tr = otree.build_tree(t[0], np.nan_to_num(cf[0]).astype(np.float32), w.m)
        tok[b], par[b], row[b] = tr["tok"], tr["parent"], tr["row"]
    target = gen.target_logits(w, draft, row)
    u = gen.uniforms(w)
    n_amb, _ = run_and_compare(w, draft, target, tok, par, row, 1.0, u)
    assert n_amb <= 1


def test_bad_draft_row_sets_status():
    w = gen.scaled(gen.WORKLOADS["tiny"], B=1, V=256, D=2, k=2, m=2, dtype="f32", seed=1260)
    draft = gen.draft_logits(w).cuda()
    target = torch.zeros((1, 3, w.V), dtype=torch.float32, device="cuda")
    tok = torch.tensor([[-1, 3, 4]], dtype=torch.int32, device="cuda")
    par = torch.tensor([[-1, 0, 0]], dtype=torch.int32, device="cuda")
    row = torch.tensor([[-1, -1, -1]], dtype=torch.int32, device="cuda")   # the root has children but no row
    u = torch.full((1, 3, 2), 0.5, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    eg.verify_draft(target, draft, tok, par, row, w.D, 1.0, u, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -1
