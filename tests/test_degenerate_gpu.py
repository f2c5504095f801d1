"""GPU parity in the method's degenerate case, with the step passed raw, and with the conv bias.

* A zero step: dt = 0 with softplus off and no dt_bias makes Delta = 0, so exp(Delta A) = 1 and
  Delta x B^T = 0 and the recurrence leaves the state as it was (echobase "Mamba" notes, the
  block equations; the oracle's own pin checks the same limit).  Every launch path must leave
  the stored state bit for bit unchanged (a speculative step's scratch states equal the main
  slot's state), while y is C.h + D.x of that state and the conv windows still shift.
* Raw steps: with softplus off the step is dt + dt_bias itself ("Hybrid SSM / Mamba models and
  non-KV state", the decode call's `dt_softplus` flag); against the oracle with softplus off.
* The conv's optional bias on every decode launch path and in the standalone conv update.

Tolerances as in the other parity tests: bf16 per-tile max error 2e-2, fp32 1e-4 (prefill) and
1e-5 (Mamba1), conv windows bit-exact.
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


def _raw_steps(g, shape_):
    """Raw steps for softplus off: Delta itself, log-uniform in [1e-3, 0.5]."""
    return np.exp(g.uniform(np.log(1e-3), np.log(0.5), size=shape_)).astype(np.float32)


# (batch, ntok): the persistent stream (64 rows), the cluster split (4 rows), several tokens into
# scratch slots (8 rows, 2 tokens)
DECODE_PATHS = [(64, 1), (4, 1), (8, 2)]


@pytest.mark.parametrize("zero", [True, False], ids=["zero_step", "raw_step"])
@pytest.mark.parametrize("batch,ntok", DECODE_PATHS)
def test_decode_with_softplus_off(batch, ntok, zero):
    import torch
    shape = wl.NEMOTRON_H_8B.with_spec(ntok if ntok > 1 else 0)
    H, P = shape.nheads, shape.head_dim
    seed = 170 + batch + ntok + (0 if zero else 7)
    prm = wl.layer_params(wl.rng(seed, 0), shape)
    S = batch * (1 + (ntok if ntok > 1 else 0)) + 8
    st = wl.initial_states(wl.rng(seed, 1), shape, S, wl.BF16, wl.BF16)
    ids = wl.rng(seed, 2).permutation(S).astype(np.int32)
    slot = ids[:batch]
    scratch = ids[batch:batch + batch * ntok].reshape(batch, ntok) if ntok > 1 else None
    inp = wl.decode_inputs(wl.rng(seed, 3), shape, prm, batch, ntok, wl.BF16)
    dt = np.zeros((batch, ntok, H), np.float32) if zero else _raw_steps(wl.rng(seed, 4), (batch, ntok, H))
    g_ssm, g_conv = guarded(to_dev(st["ssm"], wl.BF16)), guarded(to_dev(st["conv"], wl.BF16))
    ssm, conv = g_ssm.t, g_conv.t
    g_y = guarded(torch.empty(batch, ntok, H * P, dtype=torch.bfloat16, device="cuda"))
    d = {k: to_dev(v, wl.F32) for k, v in prm.items()}
    bd.mamba_state_update(bd.layer_desc(shape), ssm, to_i32(slot), to_dev(inp["xbc"], wl.BF16), to_dev(dt, wl.F32),
                          d["A"], g_y.t, conv_pool=conv, conv_w=d["conv_w"],
                          scratch_slots=None if scratch is None else to_i32(scratch), D=d["D"], dt_bias=None,
                          dt_softplus=False, z=to_dev(inp["z"], wl.BF16))
    torch.cuda.synchronize()
    for g_, what in ((g_ssm, "the state pool"), (g_conv, "the conv pool"), (g_y, "y")):
        g_.check(what)
    o_ssm, o_conv = wl.upcast(st["ssm"], wl.BF16), wl.upcast(st["conv"], wl.BF16)
    y_o = oracle.decode(o_ssm, slot, wl.upcast(inp["xbc"], wl.BF16), dt.astype(np.float64),
                        prm["A"].astype(np.float64), conv_pool=o_conv, conv_w=prm["conv_w"].astype(np.float64),
                        scratch=scratch, D=prm["D"].astype(np.float64), dt_bias=None, dt_softplus=False,
                        z=wl.upcast(inp["z"], wl.BF16).reshape(batch, ntok, H, P), n_groups=shape.n_groups)
    got_y = f64(g_y.t)
    assert np.isfinite(got_y).all()
    assert tile_rel_err(got_y.reshape(batch, ntok, H, -1), y_o.reshape(batch, ntok, H, -1), 1) < 2e-2
    np.testing.assert_array_equal(f64(conv[torch.from_numpy(slot).long().cuda()]), o_conv[slot])
    targets = [slot] if scratch is None else [scratch[:, j] for j in range(ntok)]
    for tg in targets:
        got_h = ssm[torch.from_numpy(tg.copy()).long().cuda()]
        if zero:  # the state passes through unchanged, bit for bit, into every written slot
            ref = torch.from_numpy(st["ssm"][slot].view(np.int16)).cuda()
            assert torch.equal(got_h.view(torch.int16), ref)
        else:
            assert tile_rel_err(f64(got_h), o_ssm[tg], 2) < 2e-2


def _prefill(shape, lengths, act, state, dt, has, seed):
    """One mamba_chunk_scan call with softplus off and no dt_bias; returns what the checks need."""
    import torch
    g = wl.rng(seed, 0)
    prm = wl.layer_params(g, shape)
    lengths = np.asarray(lengths, np.int32)
    T, nseq = int(lengths.sum()), len(lengths)
    cu = wl.cu_seqlens(lengths)
    inp = wl.prefill_inputs(g, shape, prm, T, act, with_z=True)
    S = nseq + 2
    pool0 = wl.initial_states(wl.rng(seed, 1), shape, S, state, None)["ssm"]
    slot = wl.rng(seed, 2).permutation(S)[:nseq].astype(np.int32)
    desc = bd.layer_desc(shape, state=state, act=act)
    g_pool = guarded(to_dev(pool0, state))
    tdt = torch.bfloat16 if act == wl.BF16 else torch.float32
    g_y = guarded(torch.zeros(T, shape.nheads, shape.head_dim, dtype=tdt, device="cuda"))
    ws = torch.empty(bd.mamba_chunk_scan_workspace_bytes(desc, T, nseq, 256), dtype=torch.uint8, device="cuda")
    d = {k: to_dev(v, wl.F32) for k, v in prm.items()}
    bd.mamba_chunk_scan(desc, g_pool.t, to_i32(cu), to_i32(slot), to_dev(inp["x"], act), to_dev(dt, wl.F32),
                        d["A"], to_dev(inp["B"], act), to_dev(inp["C"], act), g_y.t, ws,
                        has_initial_state=torch.from_numpy(np.asarray(has, np.uint8)).cuda(), chunk=256, D=d["D"],
                        dt_bias=None, dt_softplus=False, z=to_dev(inp["z"], act))
    torch.cuda.synchronize()
    g_pool.check("the state pool")
    g_y.check("y")
    up = lambda k: wl.upcast(inp[k], act)
    h0 = wl.upcast(pool0[slot], state) * np.asarray(has, np.float64)[:, None, None, None]
    y_o, hf, _ = oracle.prefill_steps(cu, up("x"), dt.astype(np.float64), prm["A"].astype(np.float64), up("B"),
                                      up("C"), h0=h0, D=prm["D"].astype(np.float64), dt_bias=None, dt_softplus=False,
                                      z=up("z"))
    return dict(pool=g_pool.t, pool0=pool0, slot=slot, y=f64(g_y.t), y_o=y_o, hf=hf, T=T)


def _y_err(got, ref, block=64):
    T, H, P = ref.shape
    pad = (-T) % block
    g = np.concatenate([got, np.zeros((pad, H, P))]).reshape(-1, block, H, P).transpose(0, 2, 1, 3)
    r = np.concatenate([ref, np.zeros((pad, H, P))]).reshape(-1, block, H, P).transpose(0, 2, 1, 3)
    return tile_rel_err(g, r, 2)


# the tensor-core path (bf16, Nemotron shape) and the portable path (fp32)
PREFILL_PATHS = [(wl.NEMOTRON_H_8B, wl.BF16, wl.BF16, 2e-2), (SMALL, wl.F32, wl.F32, 1e-4)]


@pytest.mark.parametrize("zero", [True, False], ids=["zero_step", "raw_step"])
@pytest.mark.parametrize("shape,act,state,tol", PREFILL_PATHS, ids=["tensor_core", "portable"])
def test_prefill_with_softplus_off(shape, act, state, tol, zero):
    lengths, has = [300, 129, 1], [1, 1, 1]
    T = sum(lengths)
    seed = 180 + (0 if zero else 1) + (0 if act == wl.BF16 else 2)
    dt = np.zeros((T, shape.nheads), np.float32) if zero else _raw_steps(wl.rng(seed, 5), (T, shape.nheads))
    r = _prefill(shape, lengths, act, state, dt, has, seed)
    assert np.isfinite(r["y"]).all()
    assert _y_err(r["y"], r["y_o"]) < tol
    pool = r["pool"]
    for s, sl in enumerate(r["slot"]):
        if zero:  # seeded from the slot, a zero step hands the state back unchanged
            np.testing.assert_array_equal(f64(pool[int(sl)]), wl.upcast(r["pool0"][sl], state))
        else:
            assert tile_rel_err(f64(pool[int(sl)]), r["hf"][s], 2) < tol


@pytest.mark.parametrize("zero", [True, False], ids=["zero_step", "raw_step"])
def test_mamba1_with_softplus_off(zero):
    import torch
    Dn, N, S, batch, seed = 512, 16, 12, 6, 190 + int(zero)
    g = wl.rng(seed, 0)
    prm = wl.mamba1_params(g, Dn, N, 4)
    pool0 = wl.store(0.1 * g.standard_normal((S, Dn, N)), wl.BF16)
    slot = g.choice(S, batch, replace=False).astype(np.int32)
    inp = wl.mamba1_inputs(g, prm, batch, N, wl.BF16)
    dt = np.zeros((batch, Dn), np.float32) if zero else _raw_steps(wl.rng(seed, 1), (batch, Dn))
    desc = bd.mamba1_desc(Dn, N)
    g_pool = guarded(to_dev(pool0, wl.BF16))
    g_y = guarded(torch.empty(batch, Dn, dtype=torch.bfloat16, device="cuda"))
    d = {k: to_dev(v, wl.F32) for k, v in prm.items()}
    bd.mamba1_state_update(desc, g_pool.t, to_i32(slot), to_dev(inp["x"], wl.BF16), to_dev(dt, wl.F32), d["A"],
                           to_dev(inp["B"], wl.BF16), to_dev(inp["C"], wl.BF16), g_y.t, D=d["D"], dt_bias=None,
                           dt_softplus=False, z=to_dev(inp["z"], wl.BF16))
    torch.cuda.synchronize()
    g_pool.check("the state pool")
    g_y.check("y")
    after, y = f64(g_pool.t), f64(g_y.t)
    P = {k: v.astype(np.float64) for k, v in prm.items()}
    for i, s in enumerate(slot):
        up = lambda k: wl.upcast(inp[k][i:i + 1], wl.BF16)
        h, yo = oracle.mamba1_update(wl.upcast(pool0[s], wl.BF16), up("x"), up("B"), up("C"),
                                     dt[i:i + 1].astype(np.float64), P["A"], D=P["D"], dt_bias=None,
                                     dt_softplus=False, z=up("z"))
        assert tile_rel_err(y[i], yo[0], 1) < 2e-2
        if zero:
            np.testing.assert_array_equal(after[s], wl.upcast(pool0[s], wl.BF16))
        else:
            assert tile_rel_err(after[s], h, 2) < 2e-2


# (batch, ntok) as above, plus the standalone conv update (one token: the 16-byte single-token
# kernel; three tokens: the general one)
@pytest.mark.parametrize("batch,ntok", DECODE_PATHS)
def test_decode_with_conv_bias(batch, ntok):
    """The conv's optional bias (the pages' conv has one; the workloads pass none) on every decode
    launch path, against the oracle: outputs, states and the windows (bit-exact)."""
    import torch
    shape = wl.NEMOTRON_H_8B.with_spec(ntok if ntok > 1 else 0)
    H, P, Cd = shape.nheads, shape.head_dim, shape.conv_dim
    seed = 200 + batch + ntok
    g = wl.rng(seed, 0)
    prm = wl.layer_params(g, shape)
    bias = wl.store(g.standard_normal(Cd) / 4, wl.F32)
    S = batch * (1 + (ntok if ntok > 1 else 0)) + 8
    st = wl.initial_states(wl.rng(seed, 1), shape, S, wl.BF16, wl.BF16)
    ids = wl.rng(seed, 2).permutation(S).astype(np.int32)
    slot = ids[:batch]
    scratch = ids[batch:batch + batch * ntok].reshape(batch, ntok) if ntok > 1 else None
    inp = wl.decode_inputs(wl.rng(seed, 3), shape, prm, batch, ntok, wl.BF16)
    g_ssm, g_conv = guarded(to_dev(st["ssm"], wl.BF16)), guarded(to_dev(st["conv"], wl.BF16))
    ssm, conv = g_ssm.t, g_conv.t
    g_y = guarded(torch.empty(batch, ntok, H * P, dtype=torch.bfloat16, device="cuda"))
    d = {k: to_dev(v, wl.F32) for k, v in prm.items()}
    bd.mamba_state_update(bd.layer_desc(shape), ssm, to_i32(slot), to_dev(inp["xbc"], wl.BF16),
                          to_dev(inp["dt"], wl.F32), d["A"], g_y.t, conv_pool=conv, conv_w=d["conv_w"],
                          conv_b=to_dev(bias, wl.F32), scratch_slots=None if scratch is None else to_i32(scratch),
                          D=d["D"], dt_bias=d["dt_bias"], z=to_dev(inp["z"], wl.BF16))
    torch.cuda.synchronize()
    for g_, what in ((g_ssm, "the state pool"), (g_conv, "the conv pool"), (g_y, "y")):
        g_.check(what)
    o_ssm, o_conv = wl.upcast(st["ssm"], wl.BF16), wl.upcast(st["conv"], wl.BF16)
    y_o = oracle.decode(o_ssm, slot, wl.upcast(inp["xbc"], wl.BF16), inp["dt"].astype(np.float64),
                        prm["A"].astype(np.float64), conv_pool=o_conv, conv_w=prm["conv_w"].astype(np.float64),
                        conv_b=wl.upcast(bias, wl.F32), scratch=scratch, D=prm["D"].astype(np.float64),
                        dt_bias=prm["dt_bias"].astype(np.float64),
                        z=wl.upcast(inp["z"], wl.BF16).reshape(batch, ntok, H, P), n_groups=shape.n_groups)
    got_y = f64(g_y.t)
    assert tile_rel_err(got_y.reshape(batch, ntok, H, -1), y_o.reshape(batch, ntok, H, -1), 1) < 2e-2
    np.testing.assert_array_equal(f64(conv[torch.from_numpy(slot).long().cuda()]), o_conv[slot])
    for tg in ([slot] if scratch is None else [scratch[:, j] for j in range(ntok)]):
        assert tile_rel_err(f64(ssm[torch.from_numpy(tg.copy()).long().cuda()]), o_ssm[tg], 2) < 2e-2


@pytest.mark.parametrize("ntok", [1, 3])
def test_conv_update_with_bias(ntok):
    """The standalone conv update with a bias: outputs within 2^-8 of the tile maximum, windows
    bit-exact, padded rows untouched."""
    import torch
    S, batch, seed = 24, 10, 210 + ntok
    shape = wl.NEMOTRON_H_8B.with_spec(2)
    Cd = shape.conv_dim
    g = wl.rng(seed, 0)
    prm = wl.layer_params(g, shape)
    bias = wl.store(g.standard_normal(Cd) / 4, wl.F32)
    st = wl.initial_states(wl.rng(seed, 1), shape, S, wl.BF16, wl.BF16)
    slot = wl.slot_ids(wl.rng(seed, 2), S, batch, 0.2)
    inp = wl.decode_inputs(wl.rng(seed, 3), shape, prm, batch, ntok, wl.BF16)
    conv = to_dev(st["conv"], wl.BF16)
    out = torch.zeros(batch, ntok, Cd, device="cuda", dtype=torch.bfloat16)
    bd.mamba_conv_update(bd.layer_desc(shape), conv, to_i32(slot), to_dev(inp["xbc"], wl.BF16),
                         to_dev(prm["conv_w"], wl.F32), out, conv_b=to_dev(bias, wl.F32))
    torch.cuda.synchronize()
    got, o_conv = f64(conv), wl.upcast(st["conv"], wl.BF16)
    for i, s in enumerate(slot):
        if s < 0:
            assert bool((out[i] == 0).all())
            continue
        new, ref = oracle.conv_update(o_conv[s], wl.upcast(inp["xbc"], wl.BF16)[i],
                                      prm["conv_w"].astype(np.float64), wl.upcast(bias, wl.F32))
        np.testing.assert_array_equal(got[s], new)
        assert np.abs(f64(out[i]) - ref).max() <= 2 ** -8 * np.abs(ref).max() + 1e-6
    dead = np.setdiff1d(np.arange(S), slot)
    np.testing.assert_array_equal(got[dead], o_conv[dead])
