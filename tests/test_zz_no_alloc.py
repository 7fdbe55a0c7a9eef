"""eagle_verify_noalloc: the verification stage for callers that cannot
allocate device memory for a workspace (a plugin or custom-op hook inside a
runtime that owns every device buffer, a serving loop that must not call
cudaMalloc while it runs, a process whose memory belongs to its own pool).
Its chunk records live in a fixed array inside the library instead of a
caller workspace.  It must give exactly what eagle_verify gives, call after
call, while the array keeps the previous call's records.  The file is named
so that pytest collects it last."""
import ctypes

import numpy as np
import pytest
import torch

import gen
import tree_speculative_decoding_eagle_gb300 as eg

NOALLOC_BYTES = 8 << 20


def test_requests_beyond_the_array_or_invalid_are_refused_on_the_host():
    lib = eg.load_library()
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: the argument checks come first
    one = ctypes.c_float(1.0)
    assert lib.eagle_verify_workspace_size(64, 60, 201088) <= NOALLOC_BYTES
    # 128 sequences of 61 nodes over a 201088-token vocabulary: 12.4 MB of records
    assert lib.eagle_verify_workspace_size(128, 60, 201088) > NOALLOC_BYTES
    big = [fake, eg.BF16, 201088, fake, fake, 128, 60, 6, 201088, eg.GREEDY, one, None, fake, fake, fake,
           None, None]
    assert lib.eagle_verify_noalloc(*big) == -4        # EAGLE_ERR_WORKSPACE: nothing launched
    bad = list(big)
    bad[5] = 1
    bad[0] = None                                      # no target
    assert lib.eagle_verify_noalloc(*bad) == -1
    bad = list(big)
    bad[5], bad[9], bad[11] = 1, eg.SAMPLE, None       # sampling without uniforms
    assert lib.eagle_verify_noalloc(*bad) == -1


def _library_tree(w, draft):
    tok, conf, _ = eg.draft_topk(draft, w.k)
    tree = eg.tree_build(tok, conf, w.m)
    torch.cuda.synchronize()
    return tree


def _inputs(name, seed_shift):
    w = gen.scaled(gen.WORKLOADS[name], seed=gen.WORKLOADS[name].seed + seed_shift)
    draft = gen.draft_logits(w, device="cuda")
    tree = _library_tree(w, draft)
    target = gen.target_logits(w, draft, tree["row"].cpu().numpy(), device="cuda")
    u = torch.from_numpy(gen.uniforms(w)).cuda()
    return w, tree, target, u


def _noalloc(lib, w, tree, target, mode, u, acc, path, toks, status):
    B, n, V = target.shape
    return lib.eagle_verify_noalloc(
        ctypes.c_void_p(target.data_ptr()), eg.BF16 if target.dtype == torch.bfloat16 else eg.F32,
        target.stride(1), ctypes.c_void_p(tree["tok"].data_ptr()), ctypes.c_void_p(tree["parent"].data_ptr()),
        B, n - 1, w.D, V, mode, ctypes.c_float(w.temperature),
        ctypes.c_void_p(u.data_ptr()) if mode == eg.SAMPLE else None,
        ctypes.c_void_p(acc.data_ptr()), ctypes.c_void_p(path.data_ptr()), ctypes.c_void_p(toks.data_ptr()),
        ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point_on_calls_in_a_row():
    lib = eg.load_library()
    # different shapes and modes back to back, each call after the array
    # holds the previous call's records: 13B-shaped sampling (B = 8), 7B-shaped
    # greedy, then the 13B-shaped batch again with other inputs
    calls = [("llama2-13b-b8", eg.SAMPLE, 0), ("llama2-7b-b1", eg.GREEDY, 0), ("llama2-13b-b8", eg.SAMPLE, 7)]
    for c, (name, mode, shift) in enumerate(calls):
        w, tree, target, u = _inputs(name, shift)
        ref_acc, ref_path, ref_tok = eg.verify(target, tree["tok"], tree["parent"], w.D,
                                               "greedy" if mode == eg.GREEDY else "sample", w.temperature,
                                               u if mode == eg.SAMPLE else None)
        B = w.B
        acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        path = torch.full((B, w.D + 1), -7, dtype=torch.int32, device="cuda")
        toks = torch.full((B, w.D + 1), -7, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        assert _noalloc(lib, w, tree, target, mode, u, acc, path, toks, status) == 0
        torch.cuda.synchronize()
        if c > 0:
            # after the first call (which may load the library's array) a call
            # leaves the device's free memory as it found it
            assert torch.cuda.mem_get_info()[0] == free_before, name
        assert int(status.item()) == 0
        assert torch.equal(acc, ref_acc), (name, acc.tolist(), ref_acc.tolist())
        assert torch.equal(path, ref_path), name
        assert torch.equal(toks, ref_tok), name
        assert (acc.cpu().numpy() >= 0).all()


@pytest.mark.gpu
def test_noalloc_reports_device_errors_like_the_workspace_entry_point():
    """A greedy walk over a tree whose child token is outside the vocabulary
    still returns a valid walk, and a sampling walk over such a tree reports
    EAGLE_ERR_INVALID in the status word, as eagle_verify does."""
    lib = eg.load_library()
    w, tree, target, u = _inputs("tiny", 3)
    bad = {k: v.clone() for k, v in tree.items()}
    bad["tok"][0, 1] = w.V + 5
    for mode in (eg.GREEDY, eg.SAMPLE):
        B = w.B
        want_status = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = eg.verify(target, bad["tok"], bad["parent"], w.D, "greedy" if mode == eg.GREEDY else "sample",
                        w.temperature, u if mode == eg.SAMPLE else None, status=want_status)
        acc = torch.empty(B, dtype=torch.int32, device="cuda")
        path = torch.empty((B, w.D + 1), dtype=torch.int32, device="cuda")
        toks = torch.empty((B, w.D + 1), dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _noalloc(lib, w, bad, target, mode, u, acc, path, toks, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == int(want_status.item())
        assert torch.equal(acc, ref[0]) and torch.equal(path, ref[1]) and torch.equal(toks, ref[2])
    np.testing.assert_equal(int(status.item()), -1)
