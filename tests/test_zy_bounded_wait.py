"""Failure path on the GPU without a fault: a bounded device wait that runs out.

moe_selftest_bounded_wait launches one CTA that waits on a barrier nothing ever
arrives at, through the same time-bounded wait as the pipelined kernels. The
wait gives up, the kernel records MOE_ERR_TIMEOUT in the sticky status word and
returns: the host reads the status, kernels launched while it is set do nothing,
and once it is read (and so cleared) the same context runs the layer correctly.
Collected after the other GPU tests (before the allocation-free test)."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from tests.gpu_common import TOL_BF16, cpu, rel_fro, to_dev
from token_dispatch_grouped_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_context_stays_usable():
    from token_dispatch_grouped_gb300 import binding as B
    from token_dispatch_grouped_gb300.layer import MoELayer
    torch.cuda.synchronize()
    B.moe_get_error()  # clear anything an earlier test left behind
    assert B.moe_selftest_bounded_wait(2_000_000) == B.MOE_OK  # give up after 2 ms
    assert B.moe_get_error() == B.MOE_ERR_TIMEOUT
    assert B.moe_get_error() == B.MOE_OK  # reading the word cleared it

    s = I.WORKLOADS["tiny"]
    L = MoELayer(s.T, s.d, s.E, s.K, s.h)
    ids = I.random_ids(s.T, s.E, s.K, seed=1).cuda()
    # while the word is set, a dispatch build launched after it does nothing
    assert B.moe_selftest_bounded_wait(1_000_000) == B.MOE_OK
    eti = torch.full((s.T * s.K,), -1, dtype=torch.int32, device="cuda")
    off = torch.full((s.E + 1,), -1, dtype=torch.int32, device="cuda")
    tim = torch.full((s.T * s.K,), -1, dtype=torch.int32, device="cuda")
    B.moe_build_dispatch(L.s, ids, eti, off, tim, L.ws)
    assert B.moe_get_error() == B.MOE_ERR_TIMEOUT
    assert bool((eti == -1).all()) and bool((off == -1).all()) and bool((tim == -1).all())

    # cleared: the same context runs the whole layer and matches the oracle
    inp = I.make_layer_inputs(s, seed=0)
    dv = to_dev(inp)
    r, dp, y, H, g = L.step(dv["x"], dv["Wg"], dv["W1"], dv["W3"], dv["W2"], dv["dO"])
    L.check_error()
    f = O.layer_forward(inp["x"], inp["W1"], inp["W3"], inp["W2"], cpu(r.ids), cpu(r.w))
    assert rel_fro(cpu(y), f["y"]) <= TOL_BF16
    eti_o, off_o, tim_o, _ = O.build_dispatch(cpu(r.ids), s.E)
    assert np.array_equal(cpu(dp.eti), eti_o) and np.array_equal(cpu(dp.offsets), off_o)
