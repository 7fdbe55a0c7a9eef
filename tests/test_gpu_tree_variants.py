"""GPU parity of the tree build's ablation variants (eagle_tree_build_variant).

[EAGLE-2] section "実験結果", ablation table.  The CUDA tree build gets the
oracle's float32 confidences and token ids (from the oracle's stage 1) and
must reproduce the oracle's tree bit for bit (tokens, parents, depths,
scores, gids, rows, mask) for every combination of the two flags, on the
hand-worked golden tree, small and ragged shapes, and the full-size shapes
of the 7B (D=6) and GPT-OSS-20B (D=7) workloads.
"""
import json
import os

import numpy as np
import pytest
import torch

import gen
import tree_speculative_decoding_eagle_gb300 as eg
from oracle import draft as odraft
from oracle import mask as omask
from oracle import tree as otree

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FLAGS = [(False, True), (True, True), (False, False), (True, False)]


def flag_word(conf_only, rerank):
    return (eg.TREE_CONFIDENCE_ONLY if conf_only else 0) | (0 if rerank else eg.TREE_NO_RERANK)


def run_gpu(tok, conf, m, conf_only, rerank):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = eg.tree_build(torch.from_numpy(np.ascontiguousarray(tok, dtype=np.int32)).cuda(),
                        torch.from_numpy(np.ascontiguousarray(conf, dtype=np.float32)).cuda(), m,
                        status=status, flags=flag_word(conf_only, rerank))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return {k: v.cpu().numpy() for k, v in out.items()}


def compare(got, b, want):
    for key in ("tok", "parent", "depth", "src", "row"):
        assert (got[key][b] == want[key]).all(), key
    assert (got["score"][b] == want["score"]).all(), "score"
    words = got["mask"][b].view(np.uint64)
    assert (words == omask.pack_mask(omask.tree_mask(want["parent"]))).all(), "mask"


@pytest.mark.parametrize("conf_only,rerank", FLAGS)
def test_hand_worked_variants_on_gpu(conf_only, rerank):
    with open(os.path.join(GOLDEN, "hand_ablation.json")) as f:
        h = json.load(f)
    case = next(c for c in h["cases"] if c["confidence_only"] == conf_only and c["rerank"] == rerank)
    tok = np.array(h["tok"])[None]
    conf = np.array(h["conf"], dtype=np.float32)[None]
    got = run_gpu(tok, conf, case["m"], conf_only, rerank)
    for key in ("tok", "parent", "depth", "src", "row"):
        assert list(got[key][0]) == case[key], key


SHAPES = {
    "small": dict(B=3, V=400, D=3, k=4),
    "ragged": dict(B=2, V=777 * 8, D=4, k=5),
    "llama2-7b": dict(B=1, V=32000, D=6, k=10),
    "gpt-oss-20b": dict(B=2, V=201088, D=7, k=10),
}


@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("conf_only,rerank", FLAGS)
def test_variants_match_oracle(shape, conf_only, rerank):
    s = SHAPES[shape]
    m = 60 if s["k"] == 10 else s["k"] * s["D"] - 1
    w = gen.scaled(gen.WORKLOADS["llama2-7b-b1"], name=shape, m=m, seed=500 + len(shape), **s)
    logits = gen.draft_logits(w).float().numpy()
    tok = np.zeros((w.B, w.D, w.k, w.k), dtype=np.int64)
    conf = np.zeros((w.B, w.D, w.k, w.k), dtype=np.float32)
    for b in range(w.B):
        t, c, _ = odraft.draft_topk(logits[b:b + 1], w.k)
        tok[b], conf[b] = t[0], np.nan_to_num(c[0]).astype(np.float32)
    for d in range(w.D):                       # unused rows: any valid ids
        for j in range(w.k):
            if (d, j) not in odraft.used_rows(w.D, w.k):
                tok[:, d, j] = np.arange(w.k)
    got = run_gpu(tok, conf, m, conf_only, rerank)
    for b in range(w.B):
        want = otree.build_tree(tok[b], conf[b], m, -1, confidence_only=conf_only, rerank=rerank)
        compare(got, b, want)
