"""The decode calls replayed from a CUDA graph equal the same calls launched eagerly, byte for byte.

The calls allocate nothing and never synchronise the host, so a serving loop can capture them.
Two copies of the same pools run the same three steps, one eagerly and one from a graph captured
once and replayed: the persistent stream (batch 256), the cluster split (batch 4) and a
speculative step into scratch slots (batch 128, 4 tokens).  Pools and outputs are compared byte
for byte after the replay.
"""
import numpy as np
import pytest

from recurrent_state_update_gb300 import binding as bd
from recurrent_state_update_gb300 import build as bld
from recurrent_state_update_gb300 import workloads as wl

from gpu_util import to_dev, to_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    bld.build()
    bd.lib()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("batch,ntok", [(256, 1), (4, 1), (128, 4)])
def test_decode_graph_replay_equals_eager(batch, ntok):
    import torch
    shape = wl.NEMOTRON_H_8B.with_spec(ntok if ntok > 1 else 0)
    H, P = shape.nheads, shape.head_dim
    seed = 240 + batch + ntok
    prm = wl.layer_params(wl.rng(seed, 0), shape)
    d = {k: to_dev(v, wl.F32) for k, v in prm.items()}
    S = batch * (1 + (ntok if ntok > 1 else 0)) + 8
    st = wl.initial_states(wl.rng(seed, 1), shape, S, wl.BF16, wl.BF16)
    ids = wl.rng(seed, 2).permutation(S).astype(np.int32)
    slot = to_i32(ids[:batch])
    scratch = to_i32(ids[batch:batch * (1 + ntok)].reshape(batch, ntok)) if ntok > 1 else None
    steps = [wl.decode_inputs(wl.rng(seed, 3, k), shape, prm, batch, ntok, wl.BF16) for k in range(3)]
    inputs = [dict(xbc=to_dev(i["xbc"], wl.BF16), dt=to_dev(i["dt"], wl.F32), z=to_dev(i["z"], wl.BF16)) for i in steps]
    desc = bd.layer_desc(shape)

    def make():
        return (to_dev(st["ssm"], wl.BF16), to_dev(st["conv"], wl.BF16),
                [torch.empty(batch, ntok, H * P, dtype=torch.bfloat16, device="cuda") for _ in range(3)])

    def run(ssm, conv, ys):
        for k in range(3):
            bd.mamba_state_update(desc, ssm, slot, inputs[k]["xbc"], inputs[k]["dt"], d["A"], ys[k], conv_pool=conv,
                                  conv_w=d["conv_w"], scratch_slots=scratch, D=d["D"], dt_bias=d["dt_bias"],
                                  z=inputs[k]["z"])

    ssm_e, conv_e, ys_e = make()
    run(ssm_e, conv_e, ys_e)
    torch.cuda.synchronize()

    ssm_g, conv_g, ys_g = make()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            run(ssm_g, conv_g, ys_g)
    torch.cuda.synchronize()
    # capturing runs nothing: the pools are still the initial ones until the replay
    assert torch.equal(ssm_g, to_dev(st["ssm"], wl.BF16))
    graph.replay()
    torch.cuda.synchronize()
    for a, b, what in ((ssm_e, ssm_g, "state pool"), (conv_e, conv_g, "conv pool")):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), what
    for k in range(3):
        assert torch.equal(ys_e[k].view(torch.int16), ys_g[k].view(torch.int16)), f"y of step {k}"
