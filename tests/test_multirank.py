"""Several-GPU path, host side, on CPU: two gloo ranks.

A job on N GPUs splits the batch's sequences into contiguous ranges, one per
rank, and exchanges nothing on the data path; the measured time is the max
over ranks.  These tests check the split (cover every sequence once), that a
rank's range alone gives exactly the results the whole batch gives for those
sequences (the oracle, run per rank), and the max-over-ranks reduction.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import gen
from oracle import step as ostep, verify
from tree_speculative_decoding_eagle_gb300.replicas import max_over_ranks, shard


@pytest.mark.parametrize("B,world", [(1, 1), (5, 2), (2, 2), (1, 2), (7, 3), (64, 8), (0, 4)])
def test_shard_covers_batch_once(B, world):
    seen = []
    sizes = []
    for r in range(world):
        b0, b1 = shard(B, r, world)
        assert 0 <= b0 <= b1 <= B
        seen.extend(range(b0, b1))
        sizes.append(b1 - b0)
    assert seen == list(range(B))
    assert max(sizes) - min(sizes) <= 1


def test_shard_rejects_bad_requests():
    for args in [(4, 2, 2), (4, -1, 2), (4, 0, 0), (-1, 0, 1)]:
        with pytest.raises(ValueError):
            shard(*args)


def test_max_over_ranks_single_process():
    assert max_over_ranks(3.5) == 3.5


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _tiny_batch(B):
    """Whole-batch inputs: draft logits, target logits over the whole batch's
    trees, and the walk's uniforms (drawn per global sequence index)."""
    w = gen.scaled(gen.WORKLOADS["tiny"], B=B)
    draft_t = gen.draft_logits(w)
    draft = draft_t.float().numpy()
    _, _, _, t, _ = ostep.tree_stage(draft, w.k, w.m)
    target = gen.target_logits(w, draft_t, torch.from_numpy(t["row"])).float().numpy()
    u = gen.uniforms(w)
    return w, draft, target, u


def _rank_step(w, draft, target, u, b0, b1):
    """Stages 1-2, mask and the sampling walk for sequences b0..b1-1 only."""
    tok, conf, stats, t, mk = ostep.tree_stage(draft[b0:b1], w.k, w.m)
    acc, path, toks, _ = verify.verify(target[b0:b1], t["tok"], t["parent"], w.D, "sample",
                                       w.temperature, u[b0:b1])
    return tok, conf, t, mk, acc, toks


def _worker(rank, world, port, B, out_dir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, draft, target, u = _tiny_batch(B)
        b0, b1 = shard(B, rank, world)
        tok, conf, t, mk, acc, toks = _rank_step(w, draft, target, u, b0, b1)
        parts = [None] * world
        dist.all_gather_object(parts, (b0, b1, tok, conf, t["tok"], t["parent"], mk, acc, toks))
        slowest = max_over_ranks(10.0 + rank)
        if rank == 0:
            np.save(os.path.join(out_dir, "slowest.npy"), np.array([slowest]))
            import pickle
            with open(os.path.join(out_dir, "parts.pkl"), "wb") as f:
                pickle.dump(parts, f)
    finally:
        dist.destroy_process_group()


def test_two_ranks_match_whole_batch(tmp_path):
    B, world = 5, 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, B, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    import pickle
    with open(tmp_path / "parts.pkl", "rb") as f:
        parts = pickle.load(f)
    assert float(np.load(tmp_path / "slowest.npy")[0]) == 10.0 + world - 1
    w, draft, target, u = _tiny_batch(B)
    tok, conf, t, mk, acc, toks = _rank_step(w, draft, target, u, 0, B)
    covered = []
    for b0, b1, tk, cf, ntok, npar, m, a, o in parts:
        covered.extend(range(b0, b1))
        np.testing.assert_array_equal(tk, tok[b0:b1])
        np.testing.assert_array_equal(np.nan_to_num(cf), np.nan_to_num(conf[b0:b1]))
        np.testing.assert_array_equal(ntok, t["tok"][b0:b1])
        np.testing.assert_array_equal(npar, t["parent"][b0:b1])
        np.testing.assert_array_equal(m, mk[b0:b1])
        np.testing.assert_array_equal(a, acc[b0:b1])
        np.testing.assert_array_equal(o, toks[b0:b1])
    assert covered == list(range(B))
