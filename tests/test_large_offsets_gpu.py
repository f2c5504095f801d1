"""GPU parity at the largest sizes the calls take: element offsets past 2^31 and the batch limit.

* The chunked prefill and the prefill conv on 270,144 tokens of the Nemotron-H-8B layer: x, z and
  y hold T x 128 x 64 elements, so every element past token 262,144 sits beyond 2^31; the oracle
  checks the heads (and channels) with the largest offsets.  Inputs this large are drawn on the
  device with a seeded generator, and the oracle reads back exactly the stored values it needs.
* The decode step at batch 65,535 (the largest the calls accept), single token and two tokens
  into scratch slots, on a small layer shape so that the pool stays small.

Tolerances as in the other parity tests: prefill y per (64-token block, head) tile and states per
(sequence, head) tile within 2e-2 (bf16); the conv outputs within 2^-8 |ref| + 1e-5 and its
windows bit-exact; decode states and outputs within 2e-2 per tile, conv windows bit-exact.
"""
import numpy as np
import pytest

import oracle
from recurrent_state_update_gb300 import binding as bd
from recurrent_state_update_gb300 import build as bld
from recurrent_state_update_gb300 import workloads as wl

from gpu_util import f64, guarded, tile_rel_err, to_dev, to_i32

pytestmark = pytest.mark.gpu

LONG = [265000, 5144]  # 270,144 tokens; the first sequence crosses 2^31 elements of x, z and y
CKPT = 65536           # checkpoints at 65,536 .. 262,144 tokens of the first sequence


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    bld.build()
    bd.lib()
    torch.cuda.set_device(0)


def _dev_normal(shape, dtype, gen, scale=1.0):
    """Seeded N(0, scale^2) values drawn on the device in slabs of rows, stored as `dtype`."""
    import torch
    t = torch.empty(shape, dtype=dtype, device="cuda")
    flat = t.view(shape[0], -1)
    for r0 in range(0, shape[0], 8192):
        blk = torch.randn(flat[r0:r0 + 8192].shape, generator=gen, device="cuda", dtype=torch.float32)
        flat[r0:r0 + 8192].copy_(blk.mul_(scale))
    return t


def _y_err(got, ref, block=64):
    T, H, P = ref.shape
    pad = (-T) % block
    g = np.concatenate([got, np.zeros((pad, H, P))]).reshape(-1, block, H, P).transpose(0, 2, 1, 3)
    r = np.concatenate([ref, np.zeros((pad, H, P))]).reshape(-1, block, H, P).transpose(0, 2, 1, 3)
    return tile_rel_err(g, r, 2)


def test_prefill_past_int32_element_offsets():
    """Tensor-core prefill of 270,144 tokens with checkpoints every 65,536: the last group's two
    highest heads against the oracle (y, both final states, the four checkpoints); every y finite;
    the slots the call does not own untouched."""
    import torch
    shape = wl.NEMOTRON_H_8B
    H, P, N, G = shape.nheads, shape.head_dim, shape.d_state, shape.n_groups
    lengths = np.asarray(LONG, np.int32)
    T, nseq = int(lengths.sum()), len(LONG)
    cu = wl.cu_seqlens(lengths)
    prm = wl.layer_params(wl.rng(150, 0), shape)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(150)
    bf = torch.bfloat16
    x = _dev_normal((T, H, P), bf, gen)
    z = _dev_normal((T, H, P), bf, gen)
    B = _dev_normal((T, G, N), bf, gen, 1.0 / np.sqrt(N))
    C = _dev_normal((T, G, N), bf, gen, 1.0 / np.sqrt(N))
    # steps log-uniform in [1e-3, 0.1] per (token, head); stored dt = softplus^-1(step) - dt_bias
    u = torch.rand((T, H), generator=gen, device="cuda", dtype=torch.float64)
    step = torch.exp(np.log(1e-3) + u * (np.log(0.1) - np.log(1e-3)))
    dt = (torch.log(torch.expm1(step)) - torch.from_numpy(prm["dt_bias"]).cuda().double()).float()
    del u, step
    max_ckpt = int(lengths.max()) // CKPT
    S = nseq + max_ckpt + 2
    g_pool = guarded(_dev_normal((S, H, P, N), bf, gen, 0.1))
    pool = g_pool.t
    pool0 = pool.clone()
    slot = np.array([3, 0], np.int32)
    ckpt = np.full((nseq, max_ckpt), -1, np.int32)
    ckpt[0] = [1, 2, 4, 5]
    has = np.array([1, 0], np.uint8)
    g_y = guarded(torch.zeros(T, H, P, dtype=bf, device="cuda"))
    y = g_y.t
    d = {k: torch.from_numpy(v).cuda() for k, v in prm.items()}
    desc = bd.layer_desc(shape)
    ws = torch.empty(bd.mamba_chunk_scan_workspace_bytes(desc, T, nseq, 256), dtype=torch.uint8, device="cuda")
    bd.mamba_chunk_scan(desc, pool, to_i32(cu), to_i32(slot), x, dt, d["A"], B, C, y, ws,
                        has_initial_state=torch.from_numpy(has).cuda(), ckpt_slots=to_i32(ckpt), ckpt_interval=CKPT,
                        chunk=256, D=d["D"], dt_bias=d["dt_bias"], z=z)
    torch.cuda.synchronize()
    g_pool.check("the state pool")
    g_y.check("y")
    assert bool(torch.isfinite(y).all())
    hs, g = [H - 2, H - 1], G - 1
    h0 = np.stack([f64(pool0[slot[0]])[hs], np.zeros((2, P, N))])
    y_o, hf, hc = oracle.prefill_steps(cu, f64(x[:, hs]), f64(dt[:, hs]), prm["A"][hs].astype(np.float64),
                                       f64(B[:, g:g + 1]), f64(C[:, g:g + 1]), h0=h0,
                                       D=prm["D"][hs].astype(np.float64), dt_bias=prm["dt_bias"][hs].astype(np.float64),
                                       z=f64(z[:, hs]), ckpt_interval=CKPT, max_ckpt=max_ckpt)
    assert _y_err(f64(y[:, hs]), y_o) < 2e-2
    for s in range(nseq):
        assert tile_rel_err(f64(pool[slot[s]])[hs], hf[s], 2) < 2e-2
    for k in range(max_ckpt):
        assert tile_rel_err(f64(pool[ckpt[0, k]])[hs], hc[0, k], 2) < 2e-2
    owned = set(slot.tolist()) | set(ckpt[0].tolist())
    for s in range(S):
        if s not in owned:
            assert torch.equal(pool[s], pool0[s])


def test_conv_varlen_past_int32_element_offsets():
    """Prefill conv of the same 270,144 tokens: the last x, B and C channels (and a few below
    them) of every token against the oracle, and both sequences' new windows bit-exact."""
    import torch
    shape = wl.NEMOTRON_H_8B
    H, P, N, G = shape.nheads, shape.head_dim, shape.d_state, shape.n_groups
    HP, GN, Cd, Wc = H * P, G * N, shape.conv_dim, shape.conv_cols
    lengths = np.asarray(LONG, np.int32)
    T, nseq = int(lengths.sum()), len(LONG)
    cu = wl.cu_seqlens(lengths)
    w = wl.layer_params(wl.rng(151, 0), shape)["conv_w"]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(151)
    bf = torch.bfloat16
    xbc = _dev_normal((T, Cd), bf, gen)
    g_pool = guarded(_dev_normal((4, Cd, Wc), bf, gen, 0.1))
    pool = g_pool.t
    pool0 = f64(pool)
    slot = np.array([2, 0], np.int32)
    init = np.array([1, 1], np.uint8)
    outs = {k: guarded(torch.zeros(T, n, dtype=bf, device="cuda")) for k, n in (("x", HP), ("B", GN), ("C", GN))}
    desc = bd.layer_desc(shape)
    bd.mamba_conv_varlen(desc, to_i32(cu), xbc, torch.from_numpy(w).cuda(), outs["x"].t, outs["B"].t, outs["C"].t,
                         conv_pool=pool, slot_ids=to_i32(slot), has_initial_state=torch.from_numpy(init).cuda())
    torch.cuda.synchronize()
    g_pool.check("the conv pool")
    for k, g_ in outs.items():
        g_.check(k)
    ch = np.array([0, HP - 9, HP - 2, HP - 1, HP + GN - 1, Cd - 2, Cd - 1])
    st = np.stack([pool0[s][ch] for s in slot])
    new_st, out = oracle.conv_varlen(cu, f64(xbc[:, torch.from_numpy(ch).cuda()]), w[ch].astype(np.float64),
                                     None, state=st, init=init)
    def column(c):
        if c < HP:
            return outs["x"].t[:, c]
        return outs["B"].t[:, c - HP] if c < HP + GN else outs["C"].t[:, c - HP - GN]
    got = f64(torch.stack([column(int(c)) for c in ch], dim=1))
    bad = np.abs(got - out) > 2.0 ** -8 * np.abs(out) + 1e-5
    assert not bad.any(), f"{int(bad.sum())} conv outputs out of tolerance, e.g. {np.argwhere(bad)[:3]}"
    pool1 = f64(pool)
    for s, sl in enumerate(slot):
        np.testing.assert_array_equal(pool1[sl][ch], new_st[s])


@pytest.mark.parametrize("ntok", [1, 2])
def test_decode_at_the_batch_limit(ntok):
    """Batch 65,535 with 10 % padded rows on a small layer (8 heads of 16 x 16, 2 groups): the
    single-token step runs the persistent stream over 131,070 (row, group) items, two tokens run
    one CTA per (row, group) into scratch slots.  256 sampled rows against the oracle; padded
    rows' outputs and every slot the call does not own untouched."""
    import torch
    batch = 65535
    shape = wl.LayerShape(nheads=8, head_dim=16, d_state=16, n_groups=2, conv_kernel=4)
    if ntok > 1:
        shape = shape.with_spec(ntok)
    H, P, N = shape.nheads, shape.head_dim, shape.d_state
    seed = 152 + ntok
    prm = wl.layer_params(wl.rng(seed, 0), shape)
    S = batch * (1 + (ntok if ntok > 1 else 0)) + 64
    st = wl.initial_states(wl.rng(seed, 1), shape, S, wl.BF16, wl.BF16)
    ids = wl.rng(seed, 2).permutation(S).astype(np.int32)
    slot = ids[:batch].copy()
    slot[wl.rng(seed, 3).choice(batch, batch // 10, replace=False)] = -1
    scratch = ids[batch:batch + batch * ntok].reshape(batch, ntok) if ntok > 1 else None
    inp = wl.decode_inputs(wl.rng(seed, 4), shape, prm, batch, ntok, wl.BF16)
    desc = bd.layer_desc(shape)
    g_ssm, g_conv = guarded(to_dev(st["ssm"], wl.BF16)), guarded(to_dev(st["conv"], wl.BF16))
    ssm, conv = g_ssm.t, g_conv.t
    ssm0, conv0 = ssm.clone(), conv.clone()
    g_y = guarded(torch.full((batch, ntok, H * P), 0x7FC1, dtype=torch.int16, device="cuda").view(torch.bfloat16))
    y = g_y.t
    d = {k: to_dev(v, wl.F32) for k, v in prm.items()}
    bd.mamba_state_update(desc, ssm, to_i32(slot), to_dev(inp["xbc"], wl.BF16), to_dev(inp["dt"], wl.F32), d["A"], y,
                          conv_pool=conv, conv_w=d["conv_w"], scratch_slots=None if scratch is None else to_i32(scratch),
                          D=d["D"], dt_bias=d["dt_bias"], z=to_dev(inp["z"], wl.BF16))
    torch.cuda.synchronize()
    for g_, what in ((g_ssm, "the state pool"), (g_conv, "the conv pool"), (g_y, "y")):
        g_.check(what)
    live = np.flatnonzero(slot >= 0)
    rows = np.sort(np.concatenate([wl.rng(seed, 5).choice(live, 250, replace=False), live[-6:]]))
    rows = np.unique(rows)
    n = len(rows)
    # the oracle on a compact pool: the sampled rows' slots (and scratch slots) only
    use = slot[rows] if scratch is None else np.concatenate([slot[rows], scratch[rows].ravel()])
    c_ssm, c_conv = wl.upcast(st["ssm"][use], wl.BF16), wl.upcast(st["conv"][use], wl.BF16)
    c_slot = np.arange(n, dtype=np.int32)
    c_scr = None if scratch is None else (n + np.arange(n * ntok, dtype=np.int32)).reshape(n, ntok)
    xbc_o, dt_o, z_o = wl.upcast(inp["xbc"], wl.BF16)[rows], inp["dt"][rows].astype(np.float64), \
        wl.upcast(inp["z"], wl.BF16)[rows]
    y_o = oracle.decode(c_ssm, c_slot, xbc_o, dt_o, prm["A"].astype(np.float64), conv_pool=c_conv,
                        conv_w=prm["conv_w"].astype(np.float64), scratch=c_scr, D=prm["D"].astype(np.float64),
                        dt_bias=prm["dt_bias"].astype(np.float64), z=z_o.reshape(n, ntok, H, P),
                        n_groups=shape.n_groups)
    got_y = f64(y[torch.from_numpy(rows).cuda()])
    assert tile_rel_err(got_y.reshape(n, ntok, H, -1), y_o.reshape(n, ntok, H, -1), 1) < 2e-2
    targets = [slot[rows]] if scratch is None else [scratch[rows, j] for j in range(ntok)]
    pos = [np.arange(n)] if scratch is None else [c_scr[:, j] for j in range(ntok)]
    for tg, ps in zip(targets, pos):
        assert tile_rel_err(f64(ssm[torch.from_numpy(tg.copy()).long().cuda()]), c_ssm[ps], 2) < 2e-2
    np.testing.assert_array_equal(f64(conv[torch.from_numpy(slot[rows]).long().cuda()]), c_conv[:n])
    pads = np.flatnonzero(slot < 0)
    assert bool((y[torch.from_numpy(pads).long().cuda()].view(torch.int16) == 0x7FC1).all())
    owned = np.zeros(S, bool)
    owned[slot[slot >= 0]] = True
    if scratch is not None:
        owned[scratch[slot >= 0].ravel()] = True
    free = torch.from_numpy(np.flatnonzero(~owned)).long().cuda()
    assert torch.equal(ssm[free], ssm0[free])
    assert torch.equal(conv[free], conv0[free])
