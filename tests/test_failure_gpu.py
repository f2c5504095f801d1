"""The failure path on the GPU, without a fault: a bounded wait that runs out is reported.

Every kernel of the library gives up on an mbarrier wait after 2^18 polls (about one second on
GB300) and reports it through the MAMBA_ERR_TIMEOUT bit of the caller's error word.
mamba_selftest_wait_timeout waits, with the same helper and poll bound, on a barrier phase
nothing completes; this test checks that the wait ends after about a second, that the bit is
set, and that the context still runs the library's kernels correctly afterwards.
"""
import numpy as np
import pytest

import oracle
from recurrent_state_update_gb300 import binding as bd
from recurrent_state_update_gb300 import build as bld
from recurrent_state_update_gb300 import workloads as wl

from gpu_util import f64, to_dev, to_i32

pytestmark = pytest.mark.gpu

# the poll bound of the library's waits, read as time: long enough for any copy or matrix
# operation to land, short enough that a wait which never completes ends the kernel promptly
WAIT_MIN_S, WAIT_MAX_S = 0.1, 5.0


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    bld.build()
    bd.lib()
    torch.cuda.set_device(0)


def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    import torch
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    el = torch.zeros(1, dtype=torch.int64, device="cuda")
    bd.mamba_selftest_wait_timeout(err, el)
    torch.cuda.synchronize()
    assert int(err.item()) == bd.MAMBA_ERR_TIMEOUT
    waited_s = int(el.item()) * 1e-9
    print(f"the wait gave up after {waited_s:.3f} s")
    assert WAIT_MIN_S <= waited_s <= WAIT_MAX_S
    # the context still works: a conv update through the library, checked against the oracle
    shape = wl.TINY
    g = wl.rng(500, 0)
    prm = wl.layer_params(g, shape)
    st = wl.initial_states(wl.rng(500, 1), shape, 6, wl.F32, wl.F32)
    inp = wl.decode_inputs(wl.rng(500, 2), shape, prm, 3, 1, wl.F32)
    conv = to_dev(st["conv"], wl.F32)
    slot = np.array([4, -1, 1], np.int32)
    out = torch.zeros(3, 1, shape.conv_dim, device="cuda")
    bd.mamba_conv_update(bd.layer_desc(shape, state=wl.F32, act=wl.F32), conv, to_i32(slot),
                         to_dev(inp["xbc"], wl.F32), to_dev(prm["conv_w"], wl.F32), out)
    torch.cuda.synchronize()
    o_conv = st["conv"].astype(np.float64)
    for i, s in enumerate(slot):
        if s < 0:
            continue
        new_st, ref = oracle.conv_update(o_conv[s], inp["xbc"][i].astype(np.float64), prm["conv_w"].astype(np.float64))
        np.testing.assert_array_equal(f64(conv)[s], new_st)
        assert np.abs(f64(out[i]) - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())
