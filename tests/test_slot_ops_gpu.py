"""GPU parity of the prefix-cache checkpoint operations, through the C ABI.

* mamba_slot_copy: bit-exact copies (SSM and conv state), skipped rows, flagged bad ids.
* mamba_ckpt_store_int8 / mamba_ckpt_load_int8: codes and scales bit-exact against the oracle's
  fp32 quantiser, dequantised states bit-exact against the oracle's fp32 product rounded to the
  pool dtype, conv windows copied exactly.
* Dense ("all"-mode) checkpoint chains and restore: a 4000-token prompt with 1280-token blocks
  leaves states at 1280, 2560 and 3840; restoring the 3840 state into a fresh slot (exact copy,
  or through the int8 store) and replaying the last 160 tokens gives the one-pass final state
  (the page's worked example).  Tolerance 2e-2 per (slot, head) tile, the bf16 prefill bound.
"""
import numpy as np
import pytest

import oracle
from recurrent_state_update_gb300 import binding as bd
from recurrent_state_update_gb300 import build as bld
from recurrent_state_update_gb300 import workloads as wl

from gpu_util import f64, guarded, tile_rel_err, to_dev, to_i32

pytestmark = pytest.mark.gpu

SMALL = wl.LayerShape(nheads=4, head_dim=16, d_state=32, n_groups=2, conv_kernel=4, num_spec=1)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    bld.build()
    bd.lib()
    torch.cuda.set_device(0)


def _bits(t):
    """Raw bits of a CUDA tensor as a numpy integer array (bit-exact comparisons)."""
    import torch
    v = t.detach().contiguous()
    return v.view(torch.int16 if v.element_size() == 2 else torch.int32).cpu().numpy()


@pytest.mark.parametrize("state", [wl.BF16, wl.F32])
def test_slot_copy_is_bit_exact_and_skips(state):
    import torch
    shape = SMALL
    S = 12
    st = wl.initial_states(wl.rng(80), shape, S, state, wl.BF16)
    g_ssm, g_conv = guarded(to_dev(st["ssm"], state)), guarded(to_dev(st["conv"], wl.BF16))
    ssm, conv = g_ssm.t, g_conv.t
    ssm0, conv0 = _bits(ssm), _bits(conv)
    src = np.array([3, 7, -1, 5, 9, 2], np.int32)
    dst = np.array([8, 0, 4, -1, 9, 10], np.int32)  # a -1 src, a -1 dst, src == dst
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.mamba_slot_copy(bd.layer_desc(shape, state=state), ssm, to_i32(src), to_i32(dst), conv_pool=conv, err_word=err)
    torch.cuda.synchronize()
    g_ssm.check("the state pool")
    g_conv.check("the conv pool")
    assert int(err.item()) == 0
    exp_ssm, exp_conv = ssm0.copy(), conv0.copy()
    for s_, d_ in zip(src, dst):
        if s_ >= 0 and d_ >= 0:
            exp_ssm[d_], exp_conv[d_] = ssm0[s_], conv0[s_]
    np.testing.assert_array_equal(_bits(ssm), exp_ssm)
    np.testing.assert_array_equal(_bits(conv), exp_conv)
    # an id outside the pool is flagged and its row skipped; the others still copy
    err.zero_()
    bd.mamba_slot_copy(bd.layer_desc(shape, state=state), ssm, to_i32(np.array([1, 50], np.int32)),
                       to_i32(np.array([11, 6], np.int32)), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & bd.MAMBA_ERR_SLOT_RANGE
    got = _bits(ssm)
    np.testing.assert_array_equal(got[11], exp_ssm[1])
    np.testing.assert_array_equal(got[6], exp_ssm[6])


def _int8_roundtrip(shape, state, S, src, ent, seed):
    import torch
    st = wl.initial_states(wl.rng(seed), shape, S, state, wl.BF16)
    ssm, conv = to_dev(st["ssm"], state), to_dev(st["conv"], wl.BF16)
    desc = bd.layer_desc(shape, state=state)
    eb = bd.mamba_int8_entry_bytes(desc)
    nent = int(max(ent)) + 2
    g_store = guarded(torch.zeros(nent * eb, dtype=torch.uint8, device="cuda"))  # canaries around the store
    store = g_store.t
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.mamba_ckpt_store_int8(desc, ssm, to_i32(src), to_i32(ent), store, conv_pool=conv, err_word=err)
    torch.cuda.synchronize()
    g_store.check("the int8 store")
    assert int(err.item()) == 0
    return st, ssm, conv, desc, eb, store, err


def _entry_sections(store, eb, e, shape):
    H, P, N = shape.nheads, shape.head_dim, shape.d_state
    raw = store.cpu().numpy()[e * eb:(e + 1) * eb]
    a256 = lambda b: (b + 255) // 256 * 256
    q = raw[:H * P * N].view(np.int8).reshape(H, P, N)
    so = a256(H * P * N)
    sc = raw[so:so + H * N * 4].view(np.float32).reshape(H, N)
    co = so + a256(H * N * 4)
    cv = raw[co:co + shape.conv_dim * shape.conv_cols * 2].view(np.uint16).reshape(shape.conv_dim, shape.conv_cols)
    return q, sc, cv


@pytest.mark.parametrize("state", [wl.BF16, wl.F32])
def test_int8_store_and_load_match_the_oracle(state):
    import torch
    shape = SMALL
    S = 10
    src = np.array([2, 7, 5, -1], np.int32)
    ent = np.array([0, 3, 1, 2], np.int32)
    st, ssm, conv, desc, eb, store, err = _int8_roundtrip(shape, state, S, src, ent, seed=81)
    for s_, e_ in zip(src, ent):
        if s_ < 0:
            continue
        q, sc, cv = _entry_sections(store, eb, e_, shape)
        q_o, sc_o = oracle.int8_quantize(wl.upcast(st["ssm"][s_], state))
        np.testing.assert_array_equal(q, q_o)
        np.testing.assert_array_equal(sc.view(np.int32), sc_o.view(np.int32))
        np.testing.assert_array_equal(cv, st["conv"][s_])
    # entry 2 (row with src -1) was not written
    q2, sc2, _ = _entry_sections(store, eb, 2, shape)
    assert not q2.any() and not sc2.any()
    # load entries 3 and 1 into slots 0 and 9; -1 rows skipped
    before = _bits(ssm)
    bd.mamba_ckpt_load_int8(desc, ssm, to_i32(np.array([3, 1, -1], np.int32)), to_i32(np.array([0, 9, 4], np.int32)),
                            store, conv_pool=conv, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = f64(ssm)
    for e_, s_src, s_dst in ((3, 7, 0), (1, 5, 9)):
        q_o, sc_o = oracle.int8_quantize(wl.upcast(st["ssm"][s_src], state))
        back = wl.upcast(wl.store(oracle.int8_dequantize(q_o, sc_o), state), state)
        np.testing.assert_array_equal(got[s_dst], back)
        np.testing.assert_array_equal(f64(conv)[s_dst], wl.upcast(st["conv"][s_src], wl.BF16))
    untouched = [s for s in range(S) if s not in (0, 9)]
    np.testing.assert_array_equal(_bits(ssm)[untouched], before[untouched])


def test_int8_bad_ids_are_flagged():
    import torch
    shape = SMALL
    st = wl.initial_states(wl.rng(82), shape, 4, wl.BF16, wl.BF16)
    ssm = to_dev(st["ssm"], wl.BF16)
    desc = bd.layer_desc(shape)
    eb = bd.mamba_int8_entry_bytes(desc)
    store = torch.zeros(2 * eb, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bd.mamba_ckpt_store_int8(desc, ssm, to_i32(np.array([1, 9], np.int32)), to_i32(np.array([0, 1], np.int32)),
                             store, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & bd.MAMBA_ERR_SLOT_RANGE
    q1, sc1, _ = _entry_sections(store, eb, 1, shape)
    assert not q1.any() and not sc1.any()  # the bad row wrote nothing
    q0, _, _ = _entry_sections(store, eb, 0, shape)
    np.testing.assert_array_equal(q0, oracle.int8_quantize(wl.upcast(st["ssm"][1], wl.BF16))[0])


def test_int8_store_full_size():
    """Nemotron-H-8B slots (128 x 64 x 128 bf16): 32 entries, every code and scale checked."""
    import torch
    shape = wl.NEMOTRON_H_8B
    S, n = 48, 32
    g = wl.rng(83)
    ssm_np = wl.store(0.1 * g.standard_normal((S, shape.nheads, shape.head_dim, shape.d_state)), wl.BF16)
    ssm = to_dev(ssm_np, wl.BF16)
    desc = bd.layer_desc(shape)
    eb = bd.mamba_int8_entry_bytes(desc)
    store = torch.zeros(n * eb, dtype=torch.uint8, device="cuda")
    src = g.choice(S, n, replace=False).astype(np.int32)
    ent = g.permutation(n).astype(np.int32)
    bd.mamba_ckpt_store_int8(desc, ssm, to_i32(src), to_i32(ent), store)
    torch.cuda.synchronize()
    for s_, e_ in zip(src, ent):
        q, sc, _ = _entry_sections(store, eb, e_, shape)
        q_o, sc_o = oracle.int8_quantize(wl.upcast(ssm_np[s_], wl.BF16))
        np.testing.assert_array_equal(q, q_o)
        np.testing.assert_array_equal(sc, sc_o)


@pytest.mark.parametrize("via_int8", [False, True])
def test_dense_checkpoint_chain_and_restore_replay(via_int8):
    """A 4000-token prompt with 1280-token blocks ("all" mode): states at 1280, 2560, 3840; a
    second request restores the 3840 state into a fresh slot and replays only the last 160 tokens."""
    import torch
    shape = wl.NEMOTRON_H_8B
    T, block = 4000, 1280
    g = wl.rng(84, 0)
    prm = wl.layer_params(g, shape)
    inp = wl.prefill_inputs(g, shape, prm, T, wl.BF16)
    H, P, N, G = shape.nheads, shape.head_dim, shape.d_state, shape.n_groups
    S = 8
    pool = torch.zeros(S, H, P, N, dtype=torch.bfloat16, device="cuda")
    desc = bd.layer_desc(shape)
    d = {k: to_dev(inp[k], wl.BF16) for k in ("x", "B", "C")}
    dt = to_dev(inp["dt"], wl.F32)
    dp = {k: to_dev(v, wl.F32) for k, v in prm.items()}
    ckpt = np.array([[1, 2, 3]], np.int32)

    def scan(t0, t1, slot, has, ck=None, interval=0):
        L = t1 - t0
        y = torch.zeros(L, H, P, dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(bd.mamba_chunk_scan_workspace_bytes(desc, L, 1, 256), dtype=torch.uint8, device="cuda")
        bd.mamba_chunk_scan(desc, pool, to_i32(np.array([0, L])), to_i32(np.array([slot])), d["x"][t0:t1].contiguous(),
                            dt[t0:t1].contiguous(), dp["A"], d["B"][t0:t1].contiguous(), d["C"][t0:t1].contiguous(), y,
                            ws, has_initial_state=torch.tensor([has], dtype=torch.uint8, device="cuda"),
                            ckpt_slots=to_i32(ck), ckpt_interval=interval, chunk=256, D=dp["D"], dt_bias=dp["dt_bias"])
        return y

    scan(0, T, 0, 0, ckpt, block)  # request A: one pass, checkpoints into slots 1..3
    up = lambda k: wl.upcast(inp[k], wl.BF16)
    A, D, bias = (prm[k].astype(np.float64) for k in ("A", "D", "dt_bias"))
    y_o, hf, hc = oracle.prefill_steps(np.array([0, T]), up("x"), inp["dt"].astype(np.float64), A, up("B"), up("C"),
                                       D=D, dt_bias=bias, ckpt_interval=block, max_ckpt=3)
    torch.cuda.synchronize()
    got = f64(pool)
    for k in range(3):  # states after 1280, 2560 and 3840 tokens
        assert tile_rel_err(got[1 + k], hc[0, k], 2) < 2e-2
    assert tile_rel_err(got[0], hf[0], 2) < 2e-2
    # request B: restore the 3840-token state into a fresh slot (5), replay 160 tokens
    if via_int8:
        eb = bd.mamba_int8_entry_bytes(desc)
        store = torch.zeros(eb, dtype=torch.uint8, device="cuda")
        bd.mamba_ckpt_store_int8(desc, pool, to_i32(np.array([3])), to_i32(np.array([0])), store)
        bd.mamba_ckpt_load_int8(desc, pool, to_i32(np.array([0])), to_i32(np.array([5])), store)
    else:
        bd.mamba_slot_copy(desc, pool, to_i32(np.array([3])), to_i32(np.array([5])))
    yB = scan(3840, T, 5, 1)
    torch.cuda.synchronize()
    got = f64(pool)
    assert tile_rel_err(got[5], hf[0], 2) < 2e-2
    yB = f64(yB)
    yr = y_o[3840:]
    assert tile_rel_err(yB.transpose(1, 0, 2), yr.transpose(1, 0, 2), 2) < 2e-2
