"""mamba_chunk_scan_noalloc: the chunked prefill for callers that cannot allocate device memory.

Some callers cannot pass this library a workspace: an inference engine whose memory pool has
already reserved the GPU (one more cudaMalloc would fail, or would synchronise the whole device
and stall every stream), or a latency-critical path that may not call cudaMalloc / cudaFree.
For them mamba_chunk_scan_noalloc runs the same prefill out of one fixed scratch array compiled
into the library.  This test checks, through the C ABI, on two calls in a row:
  - the tensor-core path (bf16 activations and state, head_dim 64, d_state 128): outputs and
    written-back states bit for bit equal to mamba_chunk_scan with a caller workspace (the same
    deterministic kernels run), and within the prefill tests' bf16 bound of the fp64 oracle;
  - the portable path (fp32 activations and state), whose scratch holds Delta, the cumulative
    sums, C B^T and the per-chunk states: bit for bit equal to mamba_chunk_scan and within the
    fp32 bound of the oracle;
and that a problem too large for the fixed scratch is refused before anything runs.
"""
import numpy as np
import pytest

import oracle
from recurrent_state_update_gb300 import binding as bd
from recurrent_state_update_gb300 import build as bld
from recurrent_state_update_gb300 import workloads as wl

from gpu_util import f64, tile_rel_err, to_dev, to_i32

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2
FP32_TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    bld.build()
    bd.lib()
    torch.cuda.set_device(0)


def _case(seed, shape, lengths, has_init, dtype, interval):
    import torch
    g = wl.rng(seed, 0)
    prm = wl.layer_params(g, shape)
    lengths = np.asarray(lengths, np.int32)
    T = int(lengths.sum())
    inp = wl.prefill_inputs(g, shape, prm, T, dtype, with_z=True)
    nseq = len(lengths)
    max_ckpt = int(lengths.max()) // interval
    S = nseq * (1 + max_ckpt) + 2
    pool0 = wl.initial_states(wl.rng(seed, 1), shape, S, dtype, None)["ssm"]
    ids = wl.rng(seed, 2).permutation(S).astype(np.int32)
    cu = wl.cu_seqlens(lengths)
    return dict(
        shape=shape, dtype=dtype, inp=inp, prm_np=prm, pool0=pool0, cu_np=cu, slot_np=ids[:nseq],
        has_np=np.asarray(has_init, np.uint8), max_ckpt=max_ckpt, ckpt_np=ids[nseq:nseq + nseq * max_ckpt],
        desc=bd.layer_desc(shape, state=dtype, act=dtype), pool=to_dev(pool0, dtype), cu=to_i32(cu),
        slot=to_i32(ids[:nseq]), ckpt=to_i32(ids[nseq:nseq + nseq * max_ckpt].reshape(nseq, max_ckpt)),
        interval=interval, has=torch.tensor(has_init, dtype=torch.uint8, device="cuda"),
        x=to_dev(inp["x"], dtype), B=to_dev(inp["B"], dtype), C=to_dev(inp["C"], dtype),
        z=to_dev(inp["z"], dtype), dt=to_dev(inp["dt"], wl.F32),
        prm={k: to_dev(v, wl.F32) for k, v in prm.items()}, T=T, nseq=nseq)


def _run(c, pool, y, noalloc):
    import torch
    kw = dict(has_initial_state=c["has"], ckpt_slots=c["ckpt"], ckpt_interval=c["interval"], chunk=256,
              D=c["prm"]["D"], dt_bias=c["prm"]["dt_bias"], z=c["z"])
    if noalloc:
        bd.mamba_chunk_scan_noalloc(c["desc"], pool, c["cu"], c["slot"], c["x"], c["dt"], c["prm"]["A"], c["B"],
                                    c["C"], y, **kw)
    else:
        wsb = bd.mamba_chunk_scan_workspace_bytes(c["desc"], c["T"], c["nseq"], 256)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        bd.mamba_chunk_scan(c["desc"], pool, c["cu"], c["slot"], c["x"], c["dt"], c["prm"]["A"], c["B"], c["C"],
                            y, ws, **kw)
    torch.cuda.synchronize()


def _check_oracle(c, y, pool, tol):
    """y per (64-token block, head) tile, final states and checkpoints per (slot, head) tile."""
    up = lambda k: wl.upcast(c["inp"][k], c["dtype"])
    A, D, bias = (c["prm_np"][k].astype(np.float64) for k in ("A", "D", "dt_bias"))
    h0 = wl.upcast(c["pool0"][c["slot_np"]], c["dtype"]) * c["has_np"][:, None, None, None]
    y_o, hf, hc = oracle.prefill_steps(c["cu_np"], up("x"), c["inp"]["dt"].astype(np.float64), A, up("B"), up("C"),
                                       h0=h0, D=D, dt_bias=bias, z=up("z"), ckpt_interval=c["interval"],
                                       max_ckpt=c["max_ckpt"])
    T, H, P = y_o.shape
    blocks = lambda a: np.concatenate([a, np.zeros(((-T) % 64, H, P))]).reshape(-1, 64, H, P).transpose(0, 2, 1, 3)
    assert tile_rel_err(blocks(f64(y)), blocks(y_o), 2) < tol
    got = f64(pool)
    lengths = np.diff(c["cu_np"])
    ck = c["ckpt_np"].reshape(c["nseq"], c["max_ckpt"])
    for s in range(c["nseq"]):
        if lengths[s]:
            assert tile_rel_err(got[c["slot_np"][s]], hf[s], 2) < tol
        for k in range(c["max_ckpt"]):
            if (k + 1) * c["interval"] <= lengths[s]:
                assert tile_rel_err(got[ck[s, k]], hc[s, k], 2) < tol


@pytest.mark.parametrize("path", ["tensor_core", "portable"])
def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(path):
    import torch
    if path == "tensor_core":
        shape, dtype, tol, interval = wl.NEMOTRON_H_8B, wl.BF16, BF16_TOL, 512
        cases = [_case(7, shape, [300, 701, 33], [1, 0, 1], dtype, interval),
                 _case(8, shape, [1030, 5, 512], [0, 1, 1], dtype, interval)]
    else:  # fp32 activations and state take the portable path, whose scratch grows with the chunks
        shape, dtype, tol, interval = wl.NEMOTRON_H_8B, wl.F32, FP32_TOL, 256
        cases = [_case(17, shape, [300, 201, 33], [1, 0, 1], dtype, interval),
                 _case(18, shape, [530, 5], [0, 1], dtype, interval)]
    for c in cases:
        wsb = bd.mamba_chunk_scan_workspace_bytes(c["desc"], c["T"], c["nseq"], 256)
        assert wsb <= bd.mamba_chunk_scan_static_scratch_bytes()
        if path == "portable":
            assert wsb > 1 << 20  # the fixed scratch really carries the per-chunk data
    for c in cases:  # two calls in a row on the shared fixed scratch
        ref_pool, got_pool = c["pool"].clone(), c["pool"].clone()
        y_ref = torch.zeros_like(c["x"])
        y_got = torch.full_like(c["x"], 7.0)
        _run(c, ref_pool, y_ref, noalloc=False)
        _run(c, got_pool, y_got, noalloc=True)
        assert torch.equal(y_got, y_ref)
        assert torch.equal(got_pool, ref_pool)
        _check_oracle(c, y_got, got_pool, tol)


def test_noalloc_refuses_a_problem_larger_than_its_scratch():
    import torch
    # fp32 activations take the portable path, whose scratch grows with the number of chunks
    desc = bd.layer_desc(wl.NEMOTRON_H_8B, state=wl.F32, act=wl.F32)
    limit = bd.mamba_chunk_scan_static_scratch_bytes()
    T = 8192  # 32 chunks of per-chunk fp32 states: more than the fixed scratch holds
    assert bd.mamba_chunk_scan_workspace_bytes(desc, T, 1, 256) > limit
    one = torch.zeros(1, dtype=torch.int32, device="cuda")
    f = torch.zeros(1, dtype=torch.float32, device="cuda")  # placeholders: the call is refused before any launch
    pool = torch.zeros(1, 128, 64, 128, dtype=torch.float32, device="cuda")
    x = torch.zeros(T, 128, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(bd.MambaError) as e:
        bd.mamba_chunk_scan_noalloc(desc, pool, to_i32(np.array([0, T])), one, x, f, f, f, f, x)
    assert e.value.status == bd.MAMBA_ENOSPACE
