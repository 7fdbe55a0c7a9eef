"""GPU parity of the draft softmax / top-k stage on rows that stress the
selection: every token tied (a constant row), thousands tied at the top (a
two-level row), exactly k finite values (the rest -inf), a row quantised to
a handful of levels, and ordinary rows.  Tokens must equal the oracle's
(ties -> lower token id), confidences and log-sums within the parity
tolerances.

Shapes cover the three launch forms, in bf16 and fp32: 16-warp CTAs with
one segment per warp (Llama-2-7B-shaped rows for one sequence and, in two
waves, for four; k = 32 with every row split over an 8-CTA cluster; short
rows with a one-vector last segment or fewer segments than k); 4-warp ring
CTAs (rows with fewer than eight segments per warp of an 8-warp CTA:
clusters of 6 parts with k = 32, 1020 rows of 32 segments, rows with fewer
segments than warps, one-vector tails); and 8-warp ring CTAs (rows of 64
and 65 segments, with k = 10 and k = 32).
"""
import numpy as np
import pytest
import torch

import tree_speculative_decoding_eagle_gb300 as eg
from oracle import draft as odraft

from paritylib import CONF_RTOL, LOGZ_TOL

pytestmark = pytest.mark.gpu


def edge_rows(B, D, k, V, seed):
    """[B, D, k, V] float32 logits, each used row drawn from one of the kinds."""
    rng = np.random.default_rng(seed)
    x = np.empty((B, D, k, V), dtype=np.float32)
    kinds = ["constant", "two-level", "k-finite", "levels", "normal"]
    for b in range(B):
        for i, (d, j) in enumerate(odraft.used_rows(D, k)):
            kind = kinds[(i + b) % len(kinds)]
            if kind == "constant":
                row = np.full(V, -3.0, dtype=np.float32)
            elif kind == "two-level":
                row = np.where(rng.random(V) < 0.5, 1.0, 0.0).astype(np.float32)
            elif kind == "k-finite":
                row = np.full(V, -np.inf, dtype=np.float32)
                pos = rng.choice(V, size=k, replace=False)
                row[pos] = rng.normal(size=k).astype(np.float32)
            elif kind == "levels":
                row = np.floor(rng.normal(size=V) * 2.0).astype(np.float32)
            else:
                row = (4.0 * rng.normal(size=V)).astype(np.float32)
            x[b, d, j] = row
        for j in range(1, k):          # rows never read by the stage
            x[b, 0, j] = 0.0
    return x


CASES = [
    # 16-warp CTAs, one segment per warp (one wave, or several of two CTAs per SM):
    ("bf16", 1, 6, 10, 32000),
    ("bf16", 4, 6, 10, 32000),      # 408 CTAs: two waves
    ("f32", 1, 6, 10, 32000),
    ("f32", 4, 6, 10, 32000),
    ("bf16", 1, 3, 32, 4096),
    ("bf16", 1, 2, 32, 131072),     # 8-part clusters with k = 32: the part merge ranks 256 keys
    ("bf16", 16, 6, 10, 4104),      # a last segment of one 16-byte vector
    ("f32", 32, 4, 8, 1028),        # fp32 segments of 512 tokens, a one-vector tail
    # 4-warp CTAs streaming segments through the shared-memory ring:
    ("bf16", 2, 2, 4, 201088),
    ("bf16", 1, 2, 32, 201088),     # 6-part clusters with k = 32
    ("bf16", 20, 6, 10, 32000),     # 1020 rows of 32 segments: eight per warp
    ("bf16", 64, 6, 10, 4096),      # four segments per row, one per warp: the ring's look-ahead
                                    # stages are empty copy groups
    ("bf16", 24, 6, 10, 4104),      # a last segment of one 16-byte vector (lane 0 alone copies)
    ("f32", 40, 4, 8, 1028),        # fp32 segments of 512 tokens, a one-vector tail, a warp with none
    # 8-warp CTAs streaming segments through the shared-memory ring:
    ("bf16", 8, 7, 10, 65536),      # 488 rows of 64 segments
    ("bf16", 15, 2, 32, 65536),     # k = 32
    ("f32", 8, 7, 10, 32768),
    ("bf16", 8, 7, 10, 65544),      # 65 segments, the last of one vector
]


@pytest.mark.parametrize("dtype,B,D,k,V", CASES)
def test_draft_edge_rows(dtype, B, D, k, V):
    x = edge_rows(B, D, k, V, seed=B * 1000 + V + k)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    logits = torch.from_numpy(x).to(td)
    exact = logits.float().numpy()          # the values the kernel sees
    tok_o, conf_o, stats_o = odraft.draft_topk(exact, k)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):                       # twice: nothing carries over between calls
        tok, conf, stats = eg.draft_topk(logits.cuda(), k, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        tok, conf, stats = tok.cpu().numpy(), conf.cpu().numpy(), stats.cpu().numpy()
        for b in range(B):
            for d, j in odraft.used_rows(D, k):
                assert (tok[b, d, j] == tok_o[b, d, j]).all(), (b, d, j)
                np.testing.assert_allclose(conf[b, d, j], conf_o[b, d, j], rtol=CONF_RTOL, atol=1e-30)
                assert stats[b, d, j, 0] == np.float32(stats_o[b, d, j, 0])
                lz = stats_o[b, d, j, 1]
                assert abs(stats[b, d, j, 1] - lz) <= LOGZ_TOL * max(1.0, abs(lz))
