"""Checks of the seeded input generator (no method arithmetic lives there)."""
import numpy as np
import pytest
import torch
from scipy import stats

from gen import (WORKLOADS, attention_inputs, draft_logits, philox4x32_10, scaled,
                 target_logits, tree_uniforms, uint32_to_unit_float, uniforms)


def test_philox_is_injective_on_counters_and_key_sensitive():
    ctr = np.zeros((20000, 4), dtype=np.uint64)
    ctr[:, 0] = np.arange(20000)
    a = philox4x32_10(ctr, [1, 2])
    rows = {tuple(r) for r in a.tolist()}
    assert len(rows) == 20000
    b = philox4x32_10(ctr, [1, 3])
    assert (a != b).mean() > 0.99


def test_philox_words_are_uniform():
    ctr = np.zeros((50000, 4), dtype=np.uint64)
    ctr[:, 1] = np.arange(50000)
    w = philox4x32_10(ctr, [7, 0]).reshape(-1)
    counts = np.bincount((w >> np.uint32(28)).astype(np.int64), minlength=16)
    assert stats.chisquare(counts).pvalue > 1e-3
    bits = np.unpackbits(w.view(np.uint8)).mean()
    assert abs(bits - 0.5) < 2e-3


def test_unit_float_map_is_exact_and_below_one():
    u = uint32_to_unit_float(np.array([0, 255, 256, 0xFFFFFFFF], dtype=np.uint32))
    assert u.dtype == np.float32
    assert u[0] == 0 and u[1] == 0 and u[2] == 2.0 ** -24
    assert u[3] == np.float32(1 - 2.0 ** -24) and u[3] < 1


def test_tree_uniforms_shape_and_determinism():
    u = tree_uniforms(1002, 3, 5)
    assert u.shape == (3, 5, 2) and u.dtype == np.float32
    assert (u == tree_uniforms(1002, 3, 5)).all()
    assert (u != tree_uniforms(1003, 3, 5)).any()
    assert ((u >= 0) & (u < 1)).all()


def test_workload_shapes_and_determinism():
    w = WORKLOADS["tiny"]
    a = draft_logits(w)
    assert a.shape == (w.B, w.D, w.k, w.V) and a.dtype == torch.float32
    assert torch.equal(a, draft_logits(w))
    # logit = 4 z - ln(rank + 1): the spread of a row is dominated by 4 z
    assert 3.0 < float(a[0, 0, 0].std()) < 5.5
    node_row = np.full((w.B, w.n_nodes), -1)
    node_row[0, 0] = 0
    node_row[0, 3] = 5
    t = target_logits(w, a, node_row)
    assert t.shape == (w.B, w.n_nodes, w.V)
    flat = a.view(w.B, w.D * w.k, w.V)
    d0 = (t[0, 0] - flat[0, 0]).std().item()
    d3 = (t[0, 3] - flat[0, 5]).std().item()
    assert abs(d0 - w.sigma) < 0.05 and abs(d3 - w.sigma) < 0.05
    x = attention_inputs(w)
    assert x["q"].shape == (w.B, w.n_nodes, w.Hq, w.dh)
    assert x["k_cache"].shape == (w.B, w.Hkv, w.L, w.dh)
    assert x["k_tree"].shape == (w.B, w.Hkv, w.n_nodes, w.dh)
    assert uniforms(w).shape == (w.B, w.n_nodes, 2)


def test_ragged_lengths_in_range():
    w = scaled(WORKLOADS["llama2-13b-b8"], V=64, L=300, L_min=10)
    x = attention_inputs(w)
    kv = x["kv_len"].numpy()
    assert ((kv >= 10) & (kv <= 300)).all() and len(set(kv.tolist())) > 1


def test_workload_derived_sizes():
    w = WORKLOADS["llama2-7b-b1"]
    assert w.n_candidates == 510 and w.rows_used == 51 and w.n_nodes == 61
    w = WORKLOADS["gpt-oss-20b-b64"]
    assert w.n_candidates == 610 and w.rows_used == 61


def test_philox_known_answers(golden_dir):
    """The generator reproduces Philox4x32-10's published known-answer
    vectors (zero, all-ones and pi-digit counters and keys), so every round
    constant, multiplier and word permutation is as defined."""
    import os
    rows = []
    with open(os.path.join(golden_dir, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(x, 16) for x in line.split()])
    assert len(rows) == 3
    for r in rows:
        out = philox4x32_10(np.array(r[:4], dtype=np.uint64), r[4:6])
        assert out.tolist() == r[6:10], [hex(x) for x in out.tolist()]
