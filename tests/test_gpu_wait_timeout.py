"""The bounded in-kernel wait runs out as the status-word contract says.

Every wait inside the library's kernels (on an mbarrier a copy or a peer
completes) gives up after a time limit, sets SA_DEV_TIMEOUT in the caller's
status word and lets the kernel return. Here the same wait is given a short
limit and an mbarrier that receives one of its two expected arrivals, so it
must run out: the kernel returns, the status bit is set, and the context
stays usable (a decode step afterwards still matches the oracle). No fault is
involved: the wait simply stops waiting.
"""
import numpy as np
import pytest
import torch

import oracle as O
from sa_synth import config, make_workload
from gpu_util import make_decoder, dev_bits, dev_status, oracle_unit, assert_attention

pytestmark = pytest.mark.gpu

SA_DEV_TIMEOUT = 8


def test_wait_runs_out_and_the_context_stays_usable():
    import time
    from sparse_paged_kv_page_gb300 import sa_wait_selftest
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    # the phase completes: no timeout
    sa_wait_selftest(2, 2_000_000, st, res)
    torch.cuda.synchronize()
    assert int(res.item()) == 1 and int(st.item()) == 0
    # one arrival of two: the wait gives up after ~2 ms
    for arrivals in (1, 0):
        res.fill_(-1)
        t0 = time.perf_counter()
        sa_wait_selftest(arrivals, 2_000_000, st, res)
        torch.cuda.synchronize()
        assert time.perf_counter() - t0 < 5.0
        assert int(res.item()) == 0
        assert int(st.item()) & SA_DEV_TIMEOUT
    # the context is healthy: one page-level step still matches the oracle
    wl = make_workload(config(1))
    c = wl.cfg
    dec = make_decoder(wl)
    out = dec.step(dev_bits(wl.q(0), c.dtype)).float().cpu().numpy()
    r, *_ = oracle_unit(wl, 0, 0, 0, wl.q(0)[0])
    assert dec.sel_idx[0, 0, :int(dec.sel_cnt[0, 0])].cpu().tolist() == r["sel"].tolist()
    assert_attention(out[0], r["out"])
    assert dev_status(dec) == 0
