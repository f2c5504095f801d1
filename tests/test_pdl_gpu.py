"""Programmatic dependent launch changes no result.

Every kernel of the library is launched with the programmatic stream-serialization attribute
and waits (griddepcontrol.wait) before it touches global memory, so results must equal those of
plain launches bit for bit.  MAMBA_PDL=0 turns the attribute off; it is read once per process,
so the same seeded work runs in two child processes, one per setting: three single-token decode
steps through the persistent stream, a speculative step into scratch slots, a tensor-core
prefill and a prefill conv, each back to back on one stream.  Every output and pool is compared
byte for byte.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import sys
    import numpy as np
    import torch
    sys.path.insert(0, {root!r})
    sys.path.insert(0, {tests!r})
    from recurrent_state_update_gb300 import binding as bd, build as bld, workloads as wl
    from gpu_util import to_dev, to_i32
    bld.build()
    torch.cuda.set_device(0)
    out = {{}}
    shape = wl.NEMOTRON_H_8B
    H, P = shape.nheads, shape.head_dim
    prm = wl.layer_params(wl.rng(230, 0), shape)
    d = {{k: to_dev(v, wl.F32) for k, v in prm.items()}}
    # decode: 3 single-token steps, batch 64 (persistent stream), then a 4-token speculative step
    batch, S = 64, 64 * 5 + 8
    st = wl.initial_states(wl.rng(230, 1), shape.with_spec(4), S, wl.BF16, wl.BF16)
    ssm = to_dev(st["ssm"], wl.BF16)
    ids = wl.rng(230, 2).permutation(S).astype(np.int32)
    slot, scratch = ids[:batch], ids[batch:batch * 5].reshape(batch, 4)
    conv1 = to_dev(wl.initial_states(wl.rng(230, 3), shape, S, wl.BF16, wl.BF16)["conv"], wl.BF16)
    ys = []
    for step in range(3):
        inp = wl.decode_inputs(wl.rng(230, 4, step), shape, prm, batch, 1, wl.BF16)
        y = torch.empty(batch, 1, H * P, dtype=torch.bfloat16, device="cuda")
        bd.mamba_state_update(bd.layer_desc(shape), ssm, to_i32(slot), to_dev(inp["xbc"], wl.BF16),
                              to_dev(inp["dt"], wl.F32), d["A"], y, conv_pool=conv1, conv_w=d["conv_w"], D=d["D"],
                              dt_bias=d["dt_bias"], z=to_dev(inp["z"], wl.BF16))
        ys.append(y)
    spec = shape.with_spec(4)
    conv4 = to_dev(st["conv"], wl.BF16)
    inp = wl.decode_inputs(wl.rng(230, 5), spec, prm, batch, 4, wl.BF16)
    y4 = torch.empty(batch, 4, H * P, dtype=torch.bfloat16, device="cuda")
    bd.mamba_state_update(bd.layer_desc(spec), ssm, to_i32(slot), to_dev(inp["xbc"], wl.BF16),
                          to_dev(inp["dt"], wl.F32), d["A"], y4, conv_pool=conv4, conv_w=d["conv_w"],
                          scratch_slots=to_i32(scratch), D=d["D"], dt_bias=d["dt_bias"], z=to_dev(inp["z"], wl.BF16))
    # prefill conv, then the tensor-core scan on its outputs
    lens = np.array([700, 129, 1064], np.int32)
    T = int(lens.sum())
    cu = to_i32(wl.cu_seqlens(lens))
    xbc = to_dev(wl.prefill_xbc(wl.rng(230, 6), shape, T, wl.BF16), wl.BF16)
    cpool = to_dev(wl.initial_states(wl.rng(230, 7), shape, 6, wl.BF16, wl.BF16)["conv"], wl.BF16)
    x = torch.empty(T, H * P, dtype=torch.bfloat16, device="cuda")
    B = torch.empty(T, shape.n_groups * shape.d_state, dtype=torch.bfloat16, device="cuda")
    C = torch.empty_like(B)
    pslot = to_i32(np.array([4, 1, 2], np.int32))
    has = torch.tensor([1, 0, 1], dtype=torch.uint8, device="cuda")
    bd.mamba_conv_varlen(bd.layer_desc(shape), cu, xbc, d["conv_w"], x, B, C, conv_pool=cpool, slot_ids=pslot,
                         has_initial_state=has)
    pin = wl.prefill_inputs(wl.rng(230, 8), shape, prm, T, wl.BF16, with_z=True)
    pool = to_dev(wl.initial_states(wl.rng(230, 9), shape, 6, wl.BF16, None)["ssm"], wl.BF16)
    yp = torch.empty(T, H, P, dtype=torch.bfloat16, device="cuda")
    desc = bd.layer_desc(shape)
    ws = torch.empty(bd.mamba_chunk_scan_workspace_bytes(desc, T, 3, 256), dtype=torch.uint8, device="cuda")
    bd.mamba_chunk_scan(desc, pool, cu, pslot, x.view(T, H, P), to_dev(pin["dt"], wl.F32), d["A"],
                        B.view(T, shape.n_groups, shape.d_state), C.view(T, shape.n_groups, shape.d_state), yp, ws,
                        has_initial_state=has, chunk=256, D=d["D"], dt_bias=d["dt_bias"],
                        z=to_dev(pin["z"], wl.BF16))
    torch.cuda.synchronize()
    tensors = dict(ssm=ssm, conv1=conv1, conv4=conv4, y4=y4, x=x, B=B, C=C, cpool=cpool, pool=pool, yp=yp)
    for k, t in enumerate(ys):
        tensors["y%d" % k] = t
    np.savez({path!r}, **{{k: v.view(torch.int16).cpu().numpy() for k, v in tensors.items()}})
""")


def test_results_identical_with_and_without_dependent_launch(tmp_path):
    outs = {}
    for pdl in ("1", "0"):
        path = str(tmp_path / f"pdl{pdl}.npz")
        code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), path=path)
        env = dict(os.environ, MAMBA_PDL=pdl)
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=600)
        assert r.returncode == 0, r.stderr[-3000:]
        outs[pdl] = np.load(path)
    assert sorted(outs["1"].files) == sorted(outs["0"].files)
    for k in outs["1"].files:
        np.testing.assert_array_equal(outs["1"][k], outs["0"][k], err_msg=k)
