"""GPU parity of the varlen prefill conv (mamba_conv_varlen) against the fp64 oracle, through
the C ABI.

Outputs: the kernel accumulates in fp32 and rounds once to the activation dtype, so each output
must lie within 2^-8 |ref| + 1e-5 of the fp64 value (bf16; the rounding alone is 2^-9) or
1e-5 |ref| + 1e-5 (fp32).  The written conv state is a copy of inputs or of the old window:
bit-exact.
"""
import numpy as np
import pytest

import oracle
from recurrent_state_update_gb300 import binding as bd
from recurrent_state_update_gb300 import build as bld
from recurrent_state_update_gb300 import workloads as wl

from gpu_util import f64, guarded, to_dev, to_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    bld.build()
    bd.lib()
    torch.cuda.set_device(0)


def _tol(act):
    return (2.0 ** -8, 1e-5) if act == wl.BF16 else (1e-5, 1e-5)


def _check_close(got, ref, act, what):
    rel, ab = _tol(act)
    bad = np.abs(got - ref) > rel * np.abs(ref) + ab
    assert not bad.any(), f"{what}: {int(bad.sum())} outputs out of tolerance, e.g. {np.argwhere(bad)[:3]}"


class ConvProblem:
    def __init__(self, shape, lengths, seed, act, *, init_pattern=None, pad_seq=None, with_bias=True,
                 pool=True):
        import torch
        self.shape, self.act = shape, act
        g = wl.rng(seed, 0)
        self.lengths = np.asarray(lengths, np.int32)
        self.nseq = len(lengths)
        self.T = int(self.lengths.sum())
        self.cu = wl.cu_seqlens(self.lengths)
        Cd, Wc = shape.conv_dim, shape.conv_cols
        self.w = wl.layer_params(g, shape)["conv_w"]
        self.b = wl.store(g.standard_normal(Cd) / 4, wl.F32) if with_bias else None
        self.xbc = wl.prefill_xbc(g, shape, self.T, act)
        S = self.nseq + 3
        self.conv0 = wl.initial_states(wl.rng(seed, 1), shape, S, wl.F32, act)["conv"]
        self.slot = wl.rng(seed, 2).permutation(S)[:self.nseq].astype(np.int32)
        if pad_seq is not None:
            self.slot[pad_seq] = -1
        if init_pattern is None:
            init_pattern = [s % 2 for s in range(self.nseq)]
        self.init = np.asarray(init_pattern, np.uint8)
        self.desc = bd.layer_desc(shape, act=act)
        self.use_pool = pool
        tdt = torch.bfloat16 if act == wl.BF16 else torch.float32
        HP, GN = shape.nheads * shape.head_dim, shape.n_groups * shape.d_state
        nan = float("nan")
        # every written buffer sits between canary zones, checked after each call
        self.guards = {}
        if pool:
            self.guards["the conv pool"] = guarded(to_dev(self.conv0, act))
        self.guards["x"] = guarded(torch.full((self.T, HP), nan, dtype=tdt, device="cuda"))
        self.guards["B"] = guarded(torch.full((self.T, GN), nan, dtype=tdt, device="cuda"))
        self.guards["C"] = guarded(torch.full((self.T, GN), nan, dtype=tdt, device="cuda"))
        self.pool = self.guards["the conv pool"].t if pool else None
        self.x, self.B, self.C = self.guards["x"].t, self.guards["B"].t, self.guards["C"].t

    def run_gpu(self, err=None, cu=None):
        import torch
        bd.mamba_conv_varlen(self.desc, to_i32(self.cu if cu is None else cu), to_dev(self.xbc, self.act),
                             to_dev(self.w, wl.F32), self.x, self.B, self.C,
                             conv_pool=self.pool, slot_ids=to_i32(self.slot) if self.use_pool else None,
                             has_initial_state=torch.from_numpy(self.init).cuda() if self.use_pool else None,
                             conv_b=to_dev(self.b, wl.F32), err_word=err)
        torch.cuda.synchronize()
        for what, g_ in self.guards.items():
            g_.check(what)

    def got(self):
        return np.concatenate([f64(self.x), f64(self.B), f64(self.C)], axis=1)

    def run_oracle(self, channels=None):
        """Oracle outputs (T, channels) and the new windows (nseq, channels, Wc) of the sequences."""
        ch = np.arange(self.shape.conv_dim) if channels is None else np.asarray(channels)
        conv0 = wl.upcast(self.conv0, self.act)
        st = np.stack([conv0[s] if s >= 0 else np.zeros_like(conv0[0]) for s in self.slot])[:, ch]
        init = self.init.copy() if self.use_pool else np.zeros(self.nseq, np.uint8)
        init[self.slot < 0] = 0
        u = wl.upcast(self.xbc, self.act)[:, ch]
        b = None if self.b is None else wl.upcast(self.b, wl.F32)[ch]
        return oracle.conv_varlen(self.cu, u, wl.upcast(self.w, wl.F32)[ch], b, state=st, init=init)


RAGGED = [0, 1, 2, 3, 5, 63, 64, 65, 130, 0, 200, 7]
SMALL = wl.LayerShape(nheads=4, head_dim=16, d_state=32, n_groups=2, conv_kernel=4)


@pytest.mark.parametrize("act", [wl.BF16, wl.F32])
@pytest.mark.parametrize("W,num_spec", [(4, 0), (4, 2), (2, 0), (8, 1)])
def test_conv_varlen_matches_oracle(act, W, num_spec):
    shape = wl.LayerShape(nheads=4, head_dim=16, d_state=32, n_groups=2, conv_kernel=W, num_spec=num_spec)
    pr = ConvProblem(shape, RAGGED, seed=50 + W + num_spec, act=act, pad_seq=4)
    pr.run_gpu()
    new_st, out = pr.run_oracle()
    got = pr.got()
    _check_close(got, out, act, "outputs")
    pool = f64(pr.pool)
    for s, sl in enumerate(pr.slot):
        if sl >= 0:
            np.testing.assert_array_equal(pool[sl], new_st[s], err_msg=f"conv state of sequence {s}")
    # slots no sequence owns are untouched
    owned = set(int(v) for v in pr.slot if v >= 0)
    for sl in range(pool.shape[0]):
        if sl not in owned:
            np.testing.assert_array_equal(pool[sl], wl.upcast(pr.conv0[sl], act))


@pytest.mark.parametrize("act,W", [(wl.BF16, 4), (wl.F32, 4), (wl.BF16, 8), (wl.F32, 3)])
def test_conv_varlen_many_tiles_per_cta(act, W):
    """More tiles than CTAs, so every CTA cycles its shared-memory stages many times (three
    stages for W <= 6, two above); ragged lengths put sequence starts inside tiles."""
    shape = wl.LayerShape(nheads=4, head_dim=16, d_state=32, n_groups=2, conv_kernel=W, num_spec=1)
    lengths = wl.rng(70 + W, 3).integers(1, 700, size=40).tolist()
    lengths[5] = 0
    pr = ConvProblem(shape, lengths, seed=71 + W, act=act)
    pr.run_gpu()
    new_st, out = pr.run_oracle()
    _check_close(pr.got(), out, act, "outputs")
    pool = f64(pr.pool)
    for s, sl in enumerate(pr.slot):
        np.testing.assert_array_equal(pool[sl], new_st[s])


def test_conv_varlen_without_pool_starts_from_zeros():
    pr = ConvProblem(SMALL, [33, 70, 1], seed=61, act=wl.BF16, pool=False)
    pr.run_gpu()
    _, out = pr.run_oracle()
    _check_close(pr.got(), out, wl.BF16, "outputs")


def test_conv_varlen_bad_inputs_are_flagged_and_untouched():
    import torch
    pr = ConvProblem(SMALL, [40, 90, 20], seed=62, act=wl.BF16)
    pr.slot[1] = 10_000  # outside the pool
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pr.run_gpu(err)
    assert int(err.item()) & bd.MAMBA_ERR_SLOT_RANGE
    got = pr.got()
    assert np.isnan(got[40:130]).all()  # sequence 1 untouched
    assert not np.isnan(got[:40]).any() and not np.isnan(got[130:]).any()
    # non-decreasing cu_seqlens violated: nothing is written at all
    pr2 = ConvProblem(SMALL, [40, 90, 20], seed=63, act=wl.BF16)
    err.zero_()
    bad_cu = pr2.cu.copy()
    bad_cu[1], bad_cu[2] = bad_cu[2], bad_cu[1]
    pr2.run_gpu(err, cu=bad_cu)
    assert int(err.item()) & bd.MAMBA_ERR_SEQLENS
    assert np.isnan(pr2.got()).all()
    np.testing.assert_array_equal(f64(pr2.pool), wl.upcast(pr2.conv0, wl.BF16))


def test_conv_varlen_full_size_sampled_channels():
    """The Nemotron-H-8B layer on the varlen prefill lengths (8 sequences, 32768 tokens), in the
    launch configuration the benchmark times; the oracle checks 384 sampled channels (x, B and C)
    of every token, and the window of every sequence."""
    cfg = wl.CHUNKED_PREFILL
    lengths = wl.prefill_lengths(wl.rng(cfg["seed"]), cfg["nseq"], cfg["len_lo"], cfg["len_hi"], cfg["total"])
    shape = wl.NEMOTRON_H_8B
    pr = ConvProblem(shape, lengths, seed=64, act=wl.BF16, init_pattern=[1, 0, 1, 1, 0, 1, 0, 1])
    pr.run_gpu()
    g = wl.rng(64, 9)
    HP, GN = shape.nheads * shape.head_dim, shape.n_groups * shape.d_state
    ch = np.sort(np.concatenate([g.choice(HP, 128, replace=False), HP + g.choice(GN, 128, replace=False),
                                 HP + GN + g.choice(GN, 128, replace=False)]))
    new_st, out = pr.run_oracle(channels=ch)
    _check_close(pr.got()[:, ch], out, wl.BF16, "outputs")
    pool = f64(pr.pool)
    for s, sl in enumerate(pr.slot):
        np.testing.assert_array_equal(pool[sl][ch], new_st[s])


def test_prefill_conv_then_scan_matches_oracle_pipeline():
    """Prompt -> mamba_conv_varlen -> mamba_chunk_scan equals the oracle's conv followed by its
    step recurrence (the whole prefill of a Mamba2 layer before the output projection), within
    the prefill bound 2e-2 per (64-token block, head) tile of y and per (slot, head) tile of the
    state; the scan alone is also held to that bound against the oracle recurrence run on the
    GPU's own conv outputs (which may differ from the oracle's rounded conv by one bf16 ulp)."""
    import torch
    shape = wl.LayerShape(nheads=4, head_dim=64, d_state=128, n_groups=2, conv_kernel=4)
    lengths = [300, 5, 129]
    pr = ConvProblem(shape, lengths, seed=65, act=wl.BF16, init_pattern=[1, 1, 0])
    pr.run_gpu()
    g = wl.rng(65, 5)
    prm = wl.layer_params(g, shape)
    T, H, P, N, G = pr.T, shape.nheads, shape.head_dim, shape.d_state, shape.n_groups
    dt = wl.store(wl.raw_dt(g, prm["dt_bias"], (T,)), wl.F32)
    S = pr.conv0.shape[0]
    ssm0 = wl.initial_states(wl.rng(65, 6), shape, S, wl.BF16, None)["ssm"]
    ssm = to_dev(ssm0, wl.BF16)
    y = torch.zeros(T, H, P, dtype=torch.bfloat16, device="cuda")
    desc = pr.desc
    ws = torch.empty(bd.mamba_chunk_scan_workspace_bytes(desc, T, len(lengths), 256), dtype=torch.uint8,
                     device="cuda")
    dp = {k: to_dev(v, wl.F32) for k, v in prm.items()}
    bd.mamba_chunk_scan(desc, ssm, to_i32(pr.cu), to_i32(pr.slot), pr.x.view(T, H, P), to_dev(dt, wl.F32), dp["A"],
                        pr.B.view(T, G, N), pr.C.view(T, G, N), y, ws,
                        has_initial_state=torch.from_numpy(pr.init).cuda(), chunk=256, D=dp["D"],
                        dt_bias=dp["dt_bias"])
    torch.cuda.synchronize()
    # oracle: conv on the same raw inputs, its outputs rounded to bf16 as the scan receives them
    _, post = pr.run_oracle()
    post = wl.upcast(wl.store(post, wl.BF16), wl.BF16)
    HP, GN = H * P, G * N
    h0 = np.stack([wl.upcast(ssm0[s], wl.BF16) for s in pr.slot])
    h0[pr.init == 0] = 0.0
    yr, hf, _ = oracle.prefill_steps(pr.cu, post[:, :HP].reshape(T, H, P), wl.upcast(dt, wl.F32),
                                     wl.upcast(prm["A"], wl.F32), post[:, HP:HP + GN].reshape(T, G, N),
                                     post[:, HP + GN:].reshape(T, G, N), h0=h0, D=wl.upcast(prm["D"], wl.F32),
                                     dt_bias=wl.upcast(prm["dt_bias"], wl.F32))
    from gpu_util import tile_rel_err

    def y_tiles(a):  # (T, H, P) -> (64-token block, head) tiles
        a = np.concatenate([a, np.zeros(((-T) % 64, H, P))])
        return a.reshape(-1, 64, H, P).transpose(0, 2, 1, 3)

    got_y, got_h = f64(y).reshape(T, H, P), f64(ssm)
    assert tile_rel_err(y_tiles(got_y), y_tiles(yr), 2) < 2e-2
    for s, sl in enumerate(pr.slot):
        assert tile_rel_err(got_h[sl], hf[s], 2) < 2e-2
    # the scan on exactly the inputs it received
    ys, hs, _ = oracle.prefill_steps(pr.cu, f64(pr.x).reshape(T, H, P), wl.upcast(dt, wl.F32),
                                     wl.upcast(prm["A"], wl.F32), f64(pr.B).reshape(T, G, N),
                                     f64(pr.C).reshape(T, G, N), h0=h0, D=wl.upcast(prm["D"], wl.F32),
                                     dt_bias=wl.upcast(prm["dt_bias"], wl.F32))
    assert tile_rel_err(y_tiles(got_y), y_tiles(ys), 2) < 2e-2
    for s, sl in enumerate(pr.slot):
        assert tile_rel_err(got_h[sl], hs[s], 2) < 2e-2
