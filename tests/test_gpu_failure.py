"""Failure detection without a GPU fault: a bounded device wait that nothing
completes must give up, report EAGLE_ERR_TIMEOUT (-5) in the status word,
and leave the context usable.

eagle_selftest_wait runs the kernels' own wait helpers (the CTA-local
mbarrier wait with its suspend hint, and the polling wait for barriers that
peer CTAs of a cluster arrive on) on a barrier that can never complete, with
a 1 ms limit.  No copy, MMA or tensor memory is in flight."""
import ctypes

import numpy as np
import pytest
import torch

import tree_speculative_decoding_eagle_gb300 as eg
from oracle import mask as omask

TIMEOUT = -5


def test_selftest_arguments_are_checked_on_the_host():
    lib = eg.load_library()
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: the argument checks come first
    assert lib.eagle_selftest_wait(999, 0, fake, None, None) == -1            # limit below 1 us
    assert lib.eagle_selftest_wait(100_000_001, 0, fake, None, None) == -1    # above 100 ms
    assert lib.eagle_selftest_wait(1_000_000, 2, fake, None, None) == -1      # unknown wait
    assert lib.eagle_selftest_wait(1_000_000, 0, None, None, None) == -1      # no status word


@pytest.mark.gpu
@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_gives_up_with_timeout_status(which):
    limit = 1_000_000                       # 1 ms
    status, waited = eg.selftest_wait(limit, which)
    assert status == TIMEOUT
    assert limit <= waited < 100 * limit    # it waited the limit, then returned
    # the context is still usable: a library call and a torch op afterwards
    par = np.array([-1, 0, 0, 1, 3, 2], dtype=np.int32)
    mk = eg.tree_mask(torch.from_numpy(par[None]).cuda())
    torch.cuda.synchronize()
    assert (mk.cpu().numpy().view(np.uint64)[0] == omask.pack_mask(omask.tree_mask(par)[None])[0]).all()
    assert float(torch.ones(4, device="cuda").sum()) == 4.0


@pytest.mark.gpu
def test_repeated_timeouts_keep_the_status_protocol():
    # the status word is written only on error and keeps the first code
    for _ in range(3):
        s, _ = eg.selftest_wait(20_000, 0)
        assert s == TIMEOUT
