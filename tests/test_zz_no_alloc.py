"""eagle_draft_topk_noalloc: the draft stage for callers that cannot give the
library scratch memory (runtimes that hand over only input and output
buffers, or fixed device-memory budgets).  It must produce what
eagle_draft_topk produces, call after call, with no scratch at all.  This
file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

import gen
import tree_speculative_decoding_eagle_gb300 as eg
from oracle import draft as odraft

from paritylib import CONF_RTOL, LOGZ_TOL


def call_noalloc(lib, logits, k, tok, conf, stats, status):
    B, D, _, V = logits.shape
    dt = eg.BF16 if logits.dtype == torch.bfloat16 else eg.F32
    return lib.eagle_draft_topk_noalloc(ctypes.c_void_p(logits.data_ptr()), dt, B, D, k, V, logits.stride(2),
                                        ctypes.c_void_p(tok.data_ptr()), ctypes.c_void_p(conf.data_ptr()),
                                        ctypes.c_void_p(stats.data_ptr()), ctypes.c_void_p(status.data_ptr()),
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_invalid_request_is_refused_on_the_host():
    lib = eg.load_library()
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: the argument checks come first
    assert lib.eagle_draft_topk_noalloc(fake, eg.BF16, 1, 6, 0, 32000, 32000, fake, fake, None, None, None) == -1
    assert lib.eagle_draft_topk_noalloc(fake, eg.BF16, 1, 6, 10, 32000, 31999, fake, fake, None, None, None) == -1
    assert lib.eagle_draft_topk_noalloc(None, eg.BF16, 1, 6, 10, 32000, 32000, fake, fake, None, None, None) == -1


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny", "llama2-7b-b1"])
def test_noalloc_matches_workspace_entry_point_twice(name):
    lib = eg.load_library()
    w = gen.WORKLOADS[name]
    used = odraft.used_rows(w.D, w.k)
    for call in range(2):       # two calls in a row, different inputs
        wc = gen.scaled(w, seed=w.seed + 100 * call)
        logits = gen.draft_logits(wc).cuda()
        ref_tok, ref_conf, ref_stats = eg.draft_topk(logits, w.k)
        tok = torch.full_like(ref_tok, -7)
        conf = torch.full_like(ref_conf, -7.0)
        stats = torch.full_like(ref_stats, -7.0)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert call_noalloc(lib, logits, w.k, tok, conf, stats, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for d, j in used:
            assert torch.equal(tok[:, d, j], ref_tok[:, d, j]), (call, d, j)
            np.testing.assert_allclose(conf[:, d, j].cpu().numpy(), ref_conf[:, d, j].cpu().numpy(),
                                       rtol=CONF_RTOL, atol=1e-30)
            np.testing.assert_allclose(stats[:, d, j].cpu().numpy(), ref_stats[:, d, j].cpu().numpy(),
                                       rtol=LOGZ_TOL, atol=LOGZ_TOL)
