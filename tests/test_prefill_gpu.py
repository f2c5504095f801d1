"""GPU parity of the chunked prefill against the fp64 step-recurrence oracle, through the C ABI.

Tolerances (max relative error per tile): fp32 inputs and state 1e-4; bf16 inputs and state
2e-2 (bf16 rounding of the stored state and of the matmul operands, fp32 accumulation); an fp32
state pool with bf16 activations: states 1e-4 (fp32 arithmetic throughout), y 2^-8 (its own bf16
rounding is at most 2^-9 of the tile maximum).
Tiles: (sequence, head) for states, (64-token block, head) for y.

Besides the configs' small steps (Delta in [1e-3, 0.1]), the wide-step cases draw the step
log-uniform in [1e-3, 5] or [0.2, 5] per (token, head): with A down to -16 the per-token decay
exponent Delta*|A| reaches about 80, where a decay factor formed as a quotient of two
exponentials would overflow; the method is defined for any step, and every output and state
must be finite and within the same bounds.
"""
import numpy as np
import pytest

import oracle
from recurrent_state_update_gb300 import binding as bd
from recurrent_state_update_gb300 import build as bld
from recurrent_state_update_gb300 import workloads as wl

from gpu_util import f64, guarded, tile_rel_err, to_dev, to_i32

pytestmark = pytest.mark.gpu

SMALL = wl.LayerShape(nheads=4, head_dim=16, d_state=32, n_groups=2)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    bld.build()
    bd.lib()
    torch.cuda.set_device(0)


def _y_err(got, ref, block=64):
    """Tile error of y (T, H, P) over (64-token block, head) tiles."""
    T, H, P = ref.shape
    pad = (-T) % block
    g = np.concatenate([got, np.zeros((pad, H, P))]).reshape(-1, block, H, P).transpose(0, 2, 1, 3)
    r = np.concatenate([ref, np.zeros((pad, H, P))]).reshape(-1, block, H, P).transpose(0, 2, 1, 3)
    return tile_rel_err(g, r, 2)


class Problem:
    def __init__(self, shape, lengths, seed, act, state, has_init=None, interval=0, with_z=False, steps=None):
        import torch
        self.shape, self.act, self.state = shape, act, state
        g = wl.rng(seed, 0)
        self.prm = wl.layer_params(g, shape)
        self.lengths = np.asarray(lengths, np.int32)
        self.T = int(self.lengths.sum())
        self.cu = wl.cu_seqlens(self.lengths)
        self.inp = wl.prefill_inputs(g, shape, self.prm, self.T, act, with_z=with_z, steps=steps)
        nseq = len(lengths)
        self.nseq = nseq
        self.interval = interval
        self.max_ckpt = (int(self.lengths.max()) // interval) if interval else 0
        S = nseq * (1 + self.max_ckpt) + 3
        st = wl.initial_states(wl.rng(seed, 1), shape, S, state, None)
        self.pool0 = st["ssm"]
        ids = wl.rng(seed, 2).permutation(S).astype(np.int32)
        self.slot = ids[:nseq]
        self.ckpt = ids[nseq:nseq + nseq * self.max_ckpt].reshape(nseq, self.max_ckpt) if interval else None
        self.has = np.zeros(nseq, np.uint8) if has_init is None else np.asarray(has_init, np.uint8)
        self.desc = bd.layer_desc(shape, state=state, act=act)
        self.g_pool = guarded(to_dev(self.pool0, state))  # canaries before the first and after the last slot
        self.pool = self.g_pool.t
        dev = "cuda"
        self.d = dict(x=to_dev(self.inp["x"], act), B=to_dev(self.inp["B"], act), C=to_dev(self.inp["C"], act),
                      dt=to_dev(self.inp["dt"], wl.F32), z=to_dev(self.inp["z"], act))
        self.dp = {k: to_dev(v, wl.F32) for k, v in self.prm.items()}
        self.g_y = guarded(torch.zeros(self.T, shape.nheads, shape.head_dim, device=dev,
                                       dtype=torch.bfloat16 if act == wl.BF16 else torch.float32))
        self.y = self.g_y.t

    def run_gpu(self, err=None):
        import torch
        wsb = bd.mamba_chunk_scan_workspace_bytes(self.desc, self.T, self.nseq, 256)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        bd.mamba_chunk_scan(self.desc, self.pool, to_i32(self.cu), to_i32(self.slot), self.d["x"], self.d["dt"],
                            self.dp["A"], self.d["B"], self.d["C"], self.y, ws,
                            has_initial_state=torch.from_numpy(self.has).cuda(),
                            ckpt_slots=to_i32(self.ckpt), ckpt_interval=self.interval, chunk=256,
                            D=self.dp["D"], dt_bias=self.dp["dt_bias"], z=self.d["z"], err_word=err)
        torch.cuda.synchronize()
        self.g_pool.check("the state pool")
        self.g_y.check("y")

    def run_oracle(self, heads=None):
        """Oracle over all heads, or over the heads of whole groups listed in `heads`."""
        sh = self.shape
        up = lambda k: wl.upcast(self.inp[k], self.act)
        x, B, C = up("x"), up("B"), up("C")
        z = None if self.inp["z"] is None else up("z")
        A, D, bias = (self.prm[k].astype(np.float64) for k in ("A", "D", "dt_bias"))
        dt = self.inp["dt"].astype(np.float64)
        h0 = wl.upcast(self.pool0[self.slot], self.state) * self.has[:, None, None, None]
        G = sh.n_groups
        if heads is not None:
            hg = sh.nheads // sh.n_groups
            groups = sorted(set(h // hg for h in heads))
            hs = np.concatenate([np.arange(gg * hg, (gg + 1) * hg) for gg in groups])
            x, dt, A, D, bias, h0 = x[:, hs], dt[:, hs], A[hs], D[hs], bias[hs], h0[:, hs]
            B, C = B[:, groups], C[:, groups]
            z = None if z is None else z[:, hs]
            G = len(groups)
            self.oracle_heads = hs
        else:
            self.oracle_heads = np.arange(sh.nheads)
        return oracle.prefill_steps(self.cu, x, dt, A, B, C, h0=h0, D=D, dt_bias=bias, z=z,
                                    ckpt_interval=self.interval, max_ckpt=self.max_ckpt)

    def check(self, tol, heads=None, y_tol=None):
        y_o, hf, hc = self.run_oracle(heads)
        hs = self.oracle_heads
        pool = f64(self.pool)
        y = f64(self.y)[:, hs]
        assert np.isfinite(y).all() and np.isfinite(pool).all()
        assert _y_err(y, y_o) < (tol if y_tol is None else y_tol)
        for s in range(self.nseq):
            if self.lengths[s] == 0:  # no tokens: the slot is left as it was
                np.testing.assert_array_equal(pool[self.slot[s]], wl.upcast(self.pool0[self.slot[s]], self.state))
                continue
            assert tile_rel_err(pool[self.slot[s]][hs], hf[s], 2) < tol
            for k in range(self.max_ckpt):
                cs = self.ckpt[s, k]
                if (k + 1) * self.interval <= self.lengths[s]:
                    assert tile_rel_err(pool[cs][hs], hc[s, k], 2) < tol
                else:  # checkpoint past the sequence: slot untouched
                    np.testing.assert_array_equal(pool[cs], wl.upcast(self.pool0[cs], self.state))
        used = set(self.slot.tolist()) | (set(self.ckpt.ravel().tolist()) if self.ckpt is not None else set())
        for s in range(pool.shape[0]):
            if s not in used:
                np.testing.assert_array_equal(pool[s], wl.upcast(self.pool0[s], self.state))


def test_prefill_fp32_varlen_edges():
    """Empty, length-1, exact-chunk and partial-chunk sequences; initial states; checkpoints."""
    pr = Problem(SMALL, [300, 1, 0, 513, 256, 77, 1024], seed=1, act=wl.F32, state=wl.F32,
                 has_init=[0, 1, 1, 1, 0, 1, 0], interval=256, with_z=True)
    pr.run_gpu()
    pr.check(1e-4)


def test_prefill_tc_edges():
    """Tensor-core path: empty, length-1, 128/256-multiple and partial sequences, initial states,
    checkpoints, z gate."""
    pr = Problem(wl.NEMOTRON_H_8B, [1, 0, 128, 129, 256, 300, 1024], seed=5, act=wl.BF16, state=wl.BF16,
                 has_init=[1, 1, 0, 1, 0, 1, 1], interval=256, with_z=True)
    pr.run_gpu()
    pr.check(2e-2)


@pytest.mark.parametrize("steps", [None, wl.WIDE_STEPS])
def test_prefill_fp32_state_bf16_activations(steps):
    """An fp32 state pool with bf16 activations at the Nemotron shape: the states are computed and
    written in fp32 (held to 1e-4); y is bf16, held to its own rounding."""
    pr = Problem(wl.NEMOTRON_H_8B, [513, 1000, 129], seed=6, act=wl.BF16, state=wl.F32, has_init=[1, 0, 1],
                 interval=512, with_z=True, steps=steps)
    pr.run_gpu()
    pr.check(1e-4, y_tol=2.0 ** -8)


@pytest.mark.parametrize("steps", [wl.WIDE_STEPS, wl.LARGE_STEPS])
@pytest.mark.parametrize("H,G", [(128, 8), (24, 8)])
def test_prefill_tc_wide_steps(steps, H, G):
    """Tensor-core path with steps up to 5 (Delta*|A| up to ~80 per token) mixed with tiny ones:
    empty, length-1, partial and multi-chunk sequences, initial states, checkpoints, z gate."""
    shape = wl.LayerShape(nheads=H, head_dim=64, d_state=128, n_groups=G)
    pr = Problem(shape, [1, 0, 129, 300, 1024, 700, 2000], seed=31, act=wl.BF16, state=wl.BF16,
                 has_init=[1, 1, 0, 1, 1, 0, 1], interval=256, with_z=True, steps=steps)
    pr.run_gpu()
    pr.check(2e-2)


@pytest.mark.parametrize("act,tol", [(wl.F32, 1e-4), (wl.BF16, 2e-2)])
def test_prefill_portable_wide_steps(act, tol):
    """The portable path with wide steps (fp32 and bf16 activations and state)."""
    pr = Problem(SMALL, [300, 1, 513, 0, 1030], seed=32, act=act, state=act, has_init=[1, 0, 1, 1, 0],
                 interval=256, with_z=True, steps=wl.WIDE_STEPS)
    pr.run_gpu()
    pr.check(tol)


def test_prefill_tc_bad_seqlens_flagged_nothing_written():
    import torch
    pr = Problem(wl.NEMOTRON_H_8B, [100, 50], seed=9, act=wl.BF16, state=wl.BF16)
    pr.cu = np.array([0, 160, 150], np.int32)  # decreasing
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pr.run_gpu(err)
    assert int(err.item()) & bd.MAMBA_ERR_SEQLENS
    np.testing.assert_array_equal(f64(pr.pool), wl.upcast(pr.pool0, wl.BF16))
    assert not f64(pr.y).any()


def test_prefill_bf16_nemotron_shape():
    pr = Problem(wl.NEMOTRON_H_8B, [700, 1064, 33], seed=2, act=wl.BF16, state=wl.BF16, has_init=[1, 0, 1],
                 interval=512)
    pr.run_gpu()
    pr.check(2e-2)


def test_prefill_full_size_sampled_heads():
    """The full varlen workload (8 sequences of 512..8192 tokens summing to 32768, checkpoints
    every 1024 tokens); the oracle recomputes the heads of groups 0 and 5."""
    cfg = wl.CHUNKED_PREFILL
    lengths = wl.prefill_lengths(wl.rng(cfg["seed"]), cfg["nseq"], cfg["len_lo"], cfg["len_hi"], cfg["total"])
    pr = Problem(wl.NEMOTRON_H_8B, lengths, seed=cfg["seed"], act=wl.BF16, state=wl.BF16,
                 has_init=[1, 0, 0, 1, 0, 1, 0, 0], interval=cfg["ckpt_interval"])
    pr.run_gpu()
    hg = 16
    pr.check(2e-2, heads=list(range(0, hg)) + list(range(5 * hg, 6 * hg)))


def test_prefill_handoff_two_calls_equal_one():
    """Chunked prefill seeded from the stored state (two calls) matches one call."""
    import torch
    one = Problem(SMALL, [700], seed=3, act=wl.F32, state=wl.F32, has_init=[1])
    one.run_gpu()
    two = Problem(SMALL, [700], seed=3, act=wl.F32, state=wl.F32, has_init=[1])
    cut = 300  # not a chunk boundary
    for a, b, has in ((0, cut, 1), (cut, 700, 1)):
        sub = {k: v[a:b].contiguous() for k, v in two.d.items() if v is not None}
        y = torch.zeros(b - a, SMALL.nheads, SMALL.head_dim, device="cuda")
        wsb = bd.mamba_chunk_scan_workspace_bytes(two.desc, b - a, 1, 256)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        bd.mamba_chunk_scan(two.desc, two.pool, to_i32(np.array([0, b - a])), to_i32(two.slot), sub["x"], sub["dt"],
                            two.dp["A"], sub["B"], sub["C"], y, ws,
                            has_initial_state=torch.tensor([has], dtype=torch.uint8, device="cuda"),
                            D=two.dp["D"], dt_bias=two.dp["dt_bias"])
        two.y[a:b] = y
    torch.cuda.synchronize()
    assert _y_err(f64(two.y), f64(one.y)) < 1e-4
    assert tile_rel_err(f64(two.pool[two.slot[0]]), f64(one.pool[one.slot[0]]), 2) < 1e-4
    one.check(1e-4)


def test_prefill_bad_seqlens_flagged_nothing_written():
    import torch
    pr = Problem(SMALL, [100, 50], seed=4, act=wl.F32, state=wl.F32)
    pr.cu = np.array([0, 120, 150], np.int32)
    pr.cu[1], pr.cu[2] = 160, 150  # decreasing
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pr.run_gpu(err)
    assert int(err.item()) & bd.MAMBA_ERR_SEQLENS
    np.testing.assert_array_equal(f64(pr.pool), wl.upcast(pr.pool0, wl.F32))
    assert not f64(pr.y).any()


@pytest.mark.parametrize("H,G", [(80, 1), (24, 3), (24, 8)])
def test_prefill_tc_other_head_and_group_counts(H, G):
    """Tensor-core path at head_dim 64, d_state 128 with other head and group counts (one group
    shared by 80 heads, three groups of 8, eight groups of 3): ragged and empty sequences, initial
    states, checkpoints, z gate."""
    shape = wl.LayerShape(nheads=H, head_dim=64, d_state=128, n_groups=G)
    pr = Problem(shape, [300, 0, 1025, 128], seed=10 + H, act=wl.BF16, state=wl.BF16, has_init=[1, 1, 0, 1],
                 interval=512, with_z=True)
    pr.run_gpu()
    pr.check(2e-2)


def test_prefill_portable_bf16():
    """A shape the tensor-core path does not take (head_dim 16, d_state 32) with bf16 activations
    and state: the portable chunked path, ragged sequences, checkpoints, z gate."""
    pr = Problem(SMALL, [300, 1, 513, 64, 0], seed=12, act=wl.BF16, state=wl.BF16, has_init=[1, 0, 1, 1, 1],
                 interval=256, with_z=True)
    pr.run_gpu()
    pr.check(2e-2)
