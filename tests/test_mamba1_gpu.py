"""GPU parity of the Mamba1 (S6) decode step and conv update against the fp64 oracle, through the
C ABI.  Tolerances as for the Mamba2 step: per (slot) tile max relative error 2e-2 for a bf16
state after one step (the oracle is fed the GPU's own previous state), 1e-5 for fp32; outputs the
same per (row) tile; the padding row and the slots no row owns are untouched.
"""
import numpy as np
import pytest

import oracle
from recurrent_state_update_gb300 import binding as bd
from recurrent_state_update_gb300 import build as bld
from recurrent_state_update_gb300 import workloads as wl

from gpu_util import f64, guarded, tile_rel_err, to_dev, to_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    bld.build()
    bd.lib()
    torch.cuda.set_device(0)


class M1:
    def __init__(self, Dn, N, S, batch, state, act, seed, pad=()):
        import torch
        self.Dn, self.N, self.state, self.act = Dn, N, state, act
        g = wl.rng(seed, 0)
        self.g = g
        self.prm = wl.mamba1_params(g, Dn, N, 4)
        self.pool0 = wl.store(0.1 * g.standard_normal((S, Dn, N)), state)
        self.slot = g.choice(S, batch, replace=False).astype(np.int32)
        for i in pad:
            self.slot[i] = -1
        self.desc = bd.mamba1_desc(Dn, N, state=state, act=act)
        self.g_pool = guarded(to_dev(self.pool0, state))  # canaries around the pool
        self.pool = self.g_pool.t
        self.dp = {k: to_dev(v, wl.F32) for k, v in self.prm.items()}
        self.batch = batch

    def step(self, inp=None, err=None):
        import torch
        inp = inp or wl.mamba1_inputs(self.g, self.prm, self.batch, self.N, self.act)
        tdt = torch.bfloat16 if self.act == wl.BF16 else torch.float32
        g_y = guarded(torch.full((self.batch, self.Dn), float("nan"), dtype=tdt, device="cuda"))
        y = g_y.t
        before = f64(self.pool)
        bd.mamba1_state_update(self.desc, self.pool, to_i32(self.slot), to_dev(inp["x"], self.act),
                               to_dev(inp["dt"], wl.F32), self.dp["A"], to_dev(inp["B"], self.act),
                               to_dev(inp["C"], self.act), y, D=self.dp["D"], dt_bias=self.dp["dt_bias"],
                               z=to_dev(inp["z"], self.act), err_word=err)
        torch.cuda.synchronize()
        self.g_pool.check("the state pool")
        g_y.check("y")
        return inp, before, f64(y)

    def oracle_row(self, inp, before, i):
        s = self.slot[i]
        up = lambda k: wl.upcast(inp[k][i:i + 1], self.act)
        P = {k: v.astype(np.float64) for k, v in self.prm.items()}
        return oracle.mamba1_update(before[s], up("x"), up("B"), up("C"), inp["dt"][i:i + 1].astype(np.float64),
                                    P["A"], D=P["D"], dt_bias=P["dt_bias"], z=up("z"))


@pytest.mark.parametrize("state,act,tol", [(wl.BF16, wl.BF16, 2e-2), (wl.F32, wl.BF16, 2e-2), (wl.F32, wl.F32, 1e-5)])
def test_mamba1_step_matches_oracle(state, act, tol):
    m = M1(64, 16, 12, 6, state, act, seed=90, pad=(2,))
    inp, before, y = m.step()
    after = f64(m.pool)
    for i, s in enumerate(m.slot):
        if s < 0:
            assert np.isnan(y[i]).all()
            continue
        h, yo = m.oracle_row(inp, before, i)
        assert tile_rel_err(after[s], h, 2) < tol
        assert tile_rel_err(y[i], yo[0], 1) < tol
    owned = set(int(s) for s in m.slot if s >= 0)
    for s in range(12):
        if s not in owned:
            np.testing.assert_array_equal(after[s], before[s])


@pytest.mark.parametrize("N", [8, 32, 64])
def test_mamba1_state_sizes(N):
    m = M1(128, N, 8, 4, wl.F32, wl.F32, seed=91 + N)
    inp, before, y = m.step()
    after = f64(m.pool)
    for i, s in enumerate(m.slot):
        h, yo = m.oracle_row(inp, before, i)
        assert tile_rel_err(after[s], h, 2) < 1e-5
        assert tile_rel_err(y[i], yo[0], 1) < 1e-5


def test_mamba1_fp32_drift_over_32_steps():
    """Both chains run independently for 32 steps (oracle in fp64)."""
    m = M1(64, 16, 6, 3, wl.F32, wl.F32, seed=95)
    ref = {int(s): wl.upcast(m.pool0[s], wl.F32) for s in m.slot}
    P = {k: v.astype(np.float64) for k, v in m.prm.items()}
    for _ in range(32):
        inp, _, _ = m.step()
        for i, s in enumerate(m.slot):
            up = lambda k: wl.upcast(inp[k][i:i + 1], wl.F32)
            ref[int(s)], _ = oracle.mamba1_update(ref[int(s)], up("x"), up("B"), up("C"),
                                                  inp["dt"][i:i + 1].astype(np.float64), P["A"], D=P["D"],
                                                  dt_bias=P["dt_bias"], z=up("z"))
    after = f64(m.pool)
    for s in m.slot:
        assert tile_rel_err(after[s], ref[int(s)], 2) < 1e-4


def test_mamba1_conv_update_matches_oracle():
    import torch
    Dn, W, S, batch = 96, 4, 7, 4
    g = wl.rng(96, 0)
    w = wl.store(g.standard_normal((Dn, W)) / 2, wl.F32)
    conv0 = wl.store(0.1 * g.standard_normal((S, Dn, W - 1)), wl.BF16)
    slot = np.array([4, -1, 0, 6], np.int32)
    x_in = wl.store(g.standard_normal((batch, 1, Dn)), wl.BF16)
    conv = to_dev(conv0, wl.BF16)
    out = torch.full((batch, 1, Dn), float("nan"), dtype=torch.bfloat16, device="cuda")
    bd.mamba1_conv_update(bd.mamba1_desc(Dn, 16, W), conv, to_i32(slot), to_dev(x_in, wl.BF16), to_dev(w, wl.F32), out)
    torch.cuda.synchronize()
    got, pool = f64(out), f64(conv)
    for i, s in enumerate(slot):
        if s < 0:
            assert np.isnan(got[i]).all()
            continue
        st, o = oracle.conv_update(wl.upcast(conv0[s], wl.BF16), wl.upcast(x_in[i], wl.BF16), w.astype(np.float64))
        assert (np.abs(got[i] - o) <= 2.0 ** -8 * np.abs(o) + 1e-5).all()
        np.testing.assert_array_equal(pool[s], st)


def test_mamba1_full_size_all_rows():
    """The benchmark's layer (d_inner 5120, d_state 16, bf16), batch 256 of 512 slots with two rows
    padded: every row checked against the oracle (a CTA walks about 17 rows, so the stage ring of
    the stream kernel wraps), padded rows' outputs untouched, slots no row owns unchanged."""
    cfg = wl.MAMBA1_DECODE
    m = M1(cfg["d_inner"], cfg["d_state"], cfg["pool"], cfg["batch"], wl.BF16, wl.BF16, seed=97, pad=(3, 200))
    inp, before, y = m.step()
    after = f64(m.pool)
    for i, s in enumerate(m.slot):
        if s < 0:
            assert np.isnan(y[i]).all()
            continue
        h, yo = m.oracle_row(inp, before, i)
        assert tile_rel_err(after[s], h, 2) < 2e-2
        assert tile_rel_err(y[i], yo[0], 1) < 2e-2
    owned = set(int(s) for s in m.slot if s >= 0)
    idle = np.array([s for s in range(cfg["pool"]) if s not in owned])
    np.testing.assert_array_equal(after[idle], before[idle])


@pytest.mark.parametrize("Dn,batch", [(320, 9), (2048, 600)])
def test_mamba1_ragged_channel_blocks(Dn, batch):
    """A partial last block of channels, and a batch long enough that each CTA walks many rows."""
    m = M1(Dn, 16, batch + 8, batch, wl.BF16, wl.BF16, seed=99 + Dn, pad=(1,))
    inp, before, y = m.step()
    after = f64(m.pool)
    for i, s in enumerate(m.slot):
        if s < 0:
            assert np.isnan(y[i]).all()
            continue
        h, yo = m.oracle_row(inp, before, i)
        assert tile_rel_err(after[s], h, 2) < 2e-2
        assert tile_rel_err(y[i], yo[0], 1) < 2e-2


def test_mamba1_bad_slot_flagged():
    import torch
    m = M1(64, 16, 6, 3, wl.BF16, wl.BF16, seed=98)
    m.slot[1] = 99
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    inp, before, y = m.step(err=err)
    assert int(err.item()) & bd.MAMBA_ERR_SLOT_RANGE
    assert np.isnan(y[1]).all()


@pytest.mark.parametrize("Dn,N,state,batch", [(64, 16, wl.BF16, 3), (5120, 16, wl.BF16, 40), (64, 64, wl.F32, 5)])
def test_mamba1_slot_below_minus_one_flagged(Dn, N, state, batch):
    """A slot id below -1 is outside the pool, not padding: flagged, its row's output and every
    slot no live row owns are left untouched (the bulk-copy stream for state rows of up to 64
    bytes, the per-channel kernel for wider ones)."""
    import torch
    m = M1(Dn, N, batch + 4, batch, state, wl.BF16, seed=99 + batch)
    m.slot[1] = -2
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    inp, before, y = m.step(err=err)
    assert int(err.item()) & bd.MAMBA_ERR_SLOT_RANGE
    assert np.isnan(y[1]).all()
    after = f64(m.pool)
    owned = set(int(s) for s in m.slot if s >= 0)
    for s in range(after.shape[0]):
        if s not in owned:
            np.testing.assert_array_equal(after[s], before[s])
