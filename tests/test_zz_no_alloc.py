"""mamba_chunk_scan_noalloc: the chunked prefill for callers that cannot allocate device memory.

Some callers cannot pass this library a workspace: an inference engine whose memory pool has
already reserved the GPU (one more cudaMalloc would fail, or would synchronise the whole device
and stall every stream), or a latency-critical path that may not call cudaMalloc / cudaFree.
For them mamba_chunk_scan_noalloc runs the same prefill out of one fixed scratch array compiled
into the library.  This test checks, through the C ABI, that two calls in a row give the same
outputs and written-back states as mamba_chunk_scan with a caller-provided workspace, within
the bf16 tolerance the prefill tests use, and that a problem too large for the fixed scratch is
refused before anything runs.
"""
import numpy as np
import pytest

from recurrent_state_update_gb300 import binding as bd
from recurrent_state_update_gb300 import build as bld
from recurrent_state_update_gb300 import workloads as wl

from gpu_util import f64, tile_rel_err, to_dev, to_i32

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    bld.build()
    bd.lib()
    torch.cuda.set_device(0)


def _case(seed, lengths, has_init):
    import torch
    shape = wl.NEMOTRON_H_8B
    g = wl.rng(seed, 0)
    prm = wl.layer_params(g, shape)
    lengths = np.asarray(lengths, np.int32)
    T = int(lengths.sum())
    inp = wl.prefill_inputs(g, shape, prm, T, wl.BF16, with_z=True)
    nseq = len(lengths)
    interval = 512
    max_ckpt = int(lengths.max()) // interval
    S = nseq * (1 + max_ckpt) + 2
    pool = to_dev(wl.initial_states(wl.rng(seed, 1), shape, S, wl.BF16, None)["ssm"], wl.BF16)
    ids = wl.rng(seed, 2).permutation(S).astype(np.int32)
    return dict(
        desc=bd.layer_desc(shape), pool=pool, cu=to_i32(wl.cu_seqlens(lengths)), slot=to_i32(ids[:nseq]),
        ckpt=to_i32(ids[nseq:nseq + nseq * max_ckpt].reshape(nseq, max_ckpt)), interval=interval,
        has=torch.tensor(has_init, dtype=torch.uint8, device="cuda"),
        x=to_dev(inp["x"], wl.BF16), B=to_dev(inp["B"], wl.BF16), C=to_dev(inp["C"], wl.BF16),
        z=to_dev(inp["z"], wl.BF16), dt=to_dev(inp["dt"], wl.F32),
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


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    import torch
    cases = [_case(7, [300, 701, 33], [1, 0, 1]), _case(8, [1030, 5, 512], [0, 1, 1])]
    for c in cases:  # two calls in a row on the shared fixed scratch
        ref_pool, got_pool = c["pool"].clone(), c["pool"].clone()
        y_ref = torch.zeros_like(c["x"])
        y_got = torch.full_like(c["x"], 7.0)
        _run(c, ref_pool, y_ref, noalloc=False)
        _run(c, got_pool, y_got, noalloc=True)
        T, H, P = c["x"].shape
        blocks = lambda t: np.concatenate([f64(t), np.zeros(((-T) % 64, H, P))]).reshape(-1, 64, H, P)
        assert tile_rel_err(blocks(y_got).transpose(0, 2, 1, 3), blocks(y_ref).transpose(0, 2, 1, 3), 2) < BF16_TOL
        assert tile_rel_err(f64(got_pool), f64(ref_pool), 2) < BF16_TOL


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
