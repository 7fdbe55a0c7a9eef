"""GPU parity of the tree build on inputs that stress its ranking.

[EAGLE-2] section "動的ドラフトツリーの構築アルゴリズム": candidates are
ranked by the key (V desc, parent gid asc, token asc).  These cases make the
key's later fields decide: confidences drawn from three levels (many equal V
within and across groups, and products that round equal), rows whose
confidences are not sorted, negative zero, and the largest trees the limits
allow (k = 32; m = every candidate of a 4020-candidate expansion).  Every
output must equal the oracle's bit for bit, for each flag combination the
shape allows.  Rows with a repeated token are outside the domain: the call
must still finish with every output index in range.
"""
import zlib

import numpy as np
import pytest
import torch

import tree_speculative_decoding_eagle_gb300 as eg
from oracle import mask as omask
from oracle import tree as otree

pytestmark = pytest.mark.gpu


def flag_word(conf_only, rerank):
    return (eg.TREE_CONFIDENCE_ONLY if conf_only else 0) | (0 if rerank else eg.TREE_NO_RERANK)


def draft_rows(B, D, k, kind, rng):
    """tok int64 / conf float32 [B, D, k, k]: distinct tokens per row."""
    tok = np.zeros((B, D, k, k), dtype=np.int64)
    conf = np.zeros((B, D, k, k), dtype=np.float32)
    for b in range(B):
        for d in range(D):
            for j in range(k):
                tok[b, d, j] = rng.choice(1 << 20, size=k, replace=False)
                if kind == "levels":
                    c = rng.integers(0, 3, size=k) / 2.0
                elif kind == "levels-sorted":
                    c = np.sort(rng.integers(1, 4, size=k) / 4.0)[::-1]
                elif kind == "neg-zero":
                    c = np.where(rng.random(k) < 0.3, -0.0, rng.random(k) * 0.5)
                else:
                    c = np.sort(rng.random(k) ** 3)[::-1]
                conf[b, d, j] = np.asarray(c, dtype=np.float32)
    return tok, conf


def run_and_compare(tok, conf, m, conf_only, rerank):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = eg.tree_build(torch.from_numpy(tok.astype(np.int32)).cuda(), torch.from_numpy(conf).cuda(), m,
                        status=status, flags=flag_word(conf_only, rerank))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = {key: v.cpu().numpy() for key, v in out.items()}
    for b in range(tok.shape[0]):
        want = otree.build_tree(tok[b], conf[b], m, -1, confidence_only=conf_only, rerank=rerank)
        for key in ("tok", "parent", "depth", "src", "row"):
            assert (got[key][b] == want[key]).all(), (key, b)
        assert (got["score"][b] == want["score"]).all(), ("score", b)
        words = got["mask"][b].view(np.uint64)
        assert (words == omask.pack_mask(omask.tree_mask(want["parent"]))).all(), ("mask", b)


# (name, B, D, k, kind, m for the full method)
CASES = [
    ("levels-k6", 3, 4, 6, "levels", 100),
    ("levels-sorted-k10", 2, 6, 10, "levels-sorted", 60),
    ("neg-zero-k5", 2, 4, 5, "neg-zero", 40),
    ("levels-k1", 2, 5, 1, "levels", 5),
    ("k32-all", 1, 4, 32, "smooth", 3104),
    ("k20-D11-all", 2, 11, 20, "smooth", 4020),
]


@pytest.mark.parametrize("name,B,D,k,kind,m", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("conf_only,rerank", [(False, True), (True, True), (False, False)])
def test_tree_edge(name, B, D, k, kind, m, conf_only, rerank):
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    tok, conf = draft_rows(B, D, k, kind, rng)
    if not rerank:
        m = min(m, D * k)
    elif conf_only:
        m = min(m, 200)  # the oracle's best-first growth scans every candidate per pick
    run_and_compare(tok, conf, m, conf_only, rerank)


def test_repeated_tokens_stay_in_range():
    """Rows that repeat a token are outside the domain and not checked: the
    tree is unspecified, but the call must finish and every output index
    must stay in range."""
    rng = np.random.default_rng(7)
    tok, conf = draft_rows(2, 4, 5, "levels", rng)
    tok[:, 1:, :, 1] = tok[:, 1:, :, 0]      # every expanded row repeats its first token
    conf[:, 1:, :, 1] = conf[:, 1:, :, 0]    # with the same confidence: equal keys
    m = 40
    for conf_only, rerank in [(False, True), (True, True), (False, False)]:
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = eg.tree_build(torch.from_numpy(tok.astype(np.int32)).cuda(), torch.from_numpy(conf).cuda(),
                            min(m, 4 * 5) if not rerank else m, status=status,
                            flags=flag_word(conf_only, rerank))
        torch.cuda.synchronize()
        par = out["parent"].cpu().numpy()
        src = out["src"].cpu().numpy()
        n = par.shape[1]
        assert (par[:, 0] == -1).all()
        assert ((par[:, 1:] >= -1) & (par[:, 1:] < n)).all()
        assert ((src >= 0) & (src <= 5 + 3 * 25)).all()
