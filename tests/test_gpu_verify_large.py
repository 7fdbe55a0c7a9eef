"""GPU parity of the verification walk on large trees.

With m = 1000 draft nodes and V = 32000 a sequence's chunk statistics
(1001 rows x 16 chunks x 16 bytes) exceed what the walk stages in shared
memory, so the walk reads them from global memory at each step; with m = 200
they are staged.  Trees are random with bounded depth and distinct sibling
tokens, and a path through each tree is planted (the target row of each node
on it strongly favours one child's token) so walks take several steps.
Greedy walks must equal the oracle's; sampled walks must equal it wherever
the oracle flags no decision within its rounding band.
"""
import numpy as np
import pytest
import torch

import tree_speculative_decoding_eagle_gb300 as eg
from oracle import verify as over
from paritylib import check_walk

pytestmark = pytest.mark.gpu


def planted_trees(B, n, D, V, rng):
    par = np.full((B, n), -1, dtype=np.int64)
    tok = np.zeros((B, n), dtype=np.int64)
    g = torch.Generator().manual_seed(int(rng.integers(1 << 30)))
    logits = torch.randn((B, n, V), generator=g).numpy()
    for b in range(B):
        depth = np.zeros(n, dtype=np.int64)
        used = [set() for _ in range(n)]
        for i in range(1, n):
            cands = np.nonzero(depth[:i] < D)[0]
            p = int(rng.choice(cands))
            par[b, i] = p
            depth[i] = depth[p] + 1
            t = int(rng.integers(0, V))
            while t in used[p]:
                t = int(rng.integers(0, V))
            used[p].add(t)
            tok[b, i] = t
        # plant a path: from the root, favour one child's token at each node
        cur = 0
        for _ in range(D):
            kids = np.nonzero(par[b] == cur)[0]
            if kids.size == 0:
                break
            c = int(rng.choice(kids))
            logits[b, cur, tok[b, c]] = 20.0
            cur = c
    return par, tok, logits


@pytest.mark.parametrize("m", [200, 1000])
@pytest.mark.parametrize("mode", ["greedy", "sample"])
def test_verify_large_tree(m, mode):
    B, V, D, T = 2, 32000, 8, 0.8
    rng = np.random.default_rng(3000 + m + (mode == "sample"))
    n = m + 1
    par, tok, logits = planted_trees(B, n, D, V, rng)
    target = torch.from_numpy(logits).to(torch.bfloat16)
    exact = target.float().numpy()
    u = rng.random((B, n, 2)).astype(np.float32)
    acc_o, path_o, tok_o, walks = over.verify(exact, tok, par, D, mode, T, u)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, path, toks = eg.verify(target.cuda(), torch.from_numpy(tok.astype(np.int32)).cuda(),
                                torch.from_numpy(par.astype(np.int32)).cuda(), D, mode, T,
                                torch.from_numpy(u).cuda() if mode == "sample" else None, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    acc, path, toks = acc.cpu().numpy(), path.cpu().numpy(), toks.cpu().numpy()
    stopped = sum(check_walk(mode, acc[b], path[b], toks[b], acc_o[b], path_o[b], tok_o[b], walks[b])
                  for b in range(B))
    assert stopped <= 1
    assert acc_o.max() >= 1          # the planted paths make walks take steps


@pytest.mark.parametrize("where", ["root", "second"])
def test_greedy_row_without_finite_logit_sets_status(where):
    """A target row with no finite logit has no argmax.  The greedy walk stops
    at that row with bonus -1 and reports EAGLE_ERR_INVALID; the path up to
    that row is the oracle's (computed on the rows before the bad one)."""
    B, n, D, V = 1, 40, 5, 4096
    rng = np.random.default_rng(3100 + (where == "second"))
    par, tok, logits = planted_trees(B, n, D, V, rng)
    acc_o, path_o, _, _ = over.verify(logits, tok, par, D, "greedy")
    bad = 0 if where == "root" else int(path_o[0, 1])
    assert bad >= 0
    logits[0, bad, :] = -np.inf
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc, path, toks = eg.verify(torch.from_numpy(logits).to(torch.bfloat16).cuda(),
                                torch.from_numpy(tok.astype(np.int32)).cuda(),
                                torch.from_numpy(par.astype(np.int32)).cuda(), D, "greedy", status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -1
    a = 0 if where == "root" else 1
    assert int(acc[0]) == a
    assert path[0, :a + 1].tolist() == path_o[0, :a + 1].tolist()
    assert (path[0, a + 1:] == -1).all()
    assert toks[0, :a].tolist() == [int(tok[0, p]) for p in path_o[0, 1:a + 1]]
    assert (toks[0, a:] == -1).all()
