"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

* the library builds, loads and exports every function include/mamba_state.h declares;
* the size helpers reproduce the state sizes printed on the pages (tests/golden/state_bytes.txt);
* host-checkable argument errors return the documented status before anything is launched.
"""
import ctypes
import os
import re

import pytest

from recurrent_state_update_gb300 import binding as bd
from recurrent_state_update_gb300 import build as bld
from recurrent_state_update_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mamba_state.h")


@pytest.fixture(scope="module")
def lib():
    bld.build()
    return bd.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(mamba_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("mamba_conv_update", "mamba_state_update", "mamba_chunk_scan", "mamba_spec_commit",
              "mamba_chunk_scan_workspace_bytes", "mamba_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), n
        assert n in bd.SIGNATURES, f"binding lacks {n}"


def _golden():
    out = {}
    for line in open(os.path.join(ROOT, "tests", "golden", "state_bytes.txt")):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = (s.strip() for s in line.split("=", 1))
            out[k] = float(v)
    return out


def test_state_sizes_match_the_pages(lib):
    g = _golden()
    f32_ssm = bd.layer_desc(wl.NEMOTRON_H_8B, state=wl.F32, act=wl.BF16)
    bf16_ssm = bd.layer_desc(wl.NEMOTRON_H_8B, state=wl.BF16, act=wl.BF16)
    assert bd.mamba_conv_dim(f32_ssm) == 10240
    ssm32 = bd.mamba_ssm_state_bytes(f32_ssm)
    ssm16 = bd.mamba_ssm_state_bytes(bf16_ssm)
    conv = bd.mamba_conv_state_bytes(f32_ssm)
    assert ssm16 == wl.NEMOTRON_H_8B.nheads * wl.NEMOTRON_H_8B.head_dim * wl.NEMOTRON_H_8B.d_state * 2
    # the page's 97.4 MiB: 24 layers of fp32 SSM + bf16 conv state
    assert 24 * (ssm32 + conv) == g["seq_state_bytes_24_layers_f32_ssm_bf16_conv"]
    assert round((ssm32 + conv) / 2 ** 20, 2) == g["layer_state_mib_f32_ssm_bf16_conv"]
    assert round(100 * conv / (ssm32 + conv), 1) == g["conv_share_percent"]
    assert int(24 * (ssm32 + conv) / (128 * 1024)) == g["crossover_tokens_vs_128KiB_per_token_f32"]
    assert int(24 * (ssm16 + conv) / (128 * 1024)) == g["crossover_tokens_vs_128KiB_per_token_bf16"]
    # the other page's 96 MiB: 48 layers of bf16 SSM state
    assert 48 * ssm16 == g["seq_ssm_bytes_48_layers_bf16"]
    assert 48 * ssm16 / 2 ** 20 == g["seq_ssm_mib_48_layers_bf16"]
    assert 48 * ssm16 / g["kv_bytes_per_token"] == g["crossover_tokens_48_layers"]
    # speculative columns widen the conv state only
    spec = bd.layer_desc(wl.NEMOTRON_H_8B.with_spec(4), state=wl.BF16, act=wl.BF16)
    assert bd.mamba_conv_state_bytes(spec) == 10240 * 7 * 2
    assert bd.mamba_ssm_state_bytes(spec) == ssm16


def test_supported_shapes(lib):
    assert bd.mamba_decode_supported(bd.layer_desc(wl.NEMOTRON_H_8B)) == bd.MAMBA_OK
    assert bd.mamba_decode_supported(bd.layer_desc(wl.TINY, state=wl.F32, act=wl.F32)) == bd.MAMBA_OK
    odd = wl.LayerShape(nheads=4, head_dim=24, d_state=40, n_groups=1)
    assert bd.mamba_decode_supported(bd.layer_desc(odd)) == bd.MAMBA_EUNSUPPORTED
    bad = wl.LayerShape(nheads=6, head_dim=64, d_state=128, n_groups=4)  # 6 % 4 != 0
    assert bd.mamba_decode_supported(bd.layer_desc(bad)) == bd.MAMBA_EINVAL
    assert bd.mamba_conv_dim(bd.layer_desc(bad)) == -1
    mixed = bd.layer_desc(wl.NEMOTRON_H_8B, conv=wl.F32)  # conv dtype != act dtype
    assert bd.mamba_decode_supported(mixed) == bd.MAMBA_EUNSUPPORTED


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert bd.status_string(code).startswith("MAMBA_")
    assert "unknown" in bd.status_string(7)


def test_workspace_bytes(lib):
    d = bd.layer_desc(wl.NEMOTRON_H_8B)
    # tensor-core layer (bf16, head_dim 64, d_state 128): only the sequence order is kept
    assert 0 < bd.mamba_chunk_scan_workspace_bytes(d, 32768, 8, 256) <= 4096
    # portable layer (fp32 activations): at least the per-chunk fp32 states of every chunk
    d32 = bd.layer_desc(wl.NEMOTRON_H_8B, state=wl.F32, act=wl.F32)
    ws = bd.mamba_chunk_scan_workspace_bytes(d32, 32768, 8, 256)
    assert ws >= (32768 // 256 + 8) * 128 * 64 * 128 * 4
    assert bd.mamba_chunk_scan_workspace_bytes(d, -1, 8, 256) == 0


# --------------------------------------------------------------------------------------------
# host-side validation: every call below returns before any CUDA call is made
# --------------------------------------------------------------------------------------------

FAKE = 0x10000  # a 16-byte aligned non-null value; never dereferenced because validation fails first


def _state_update(lib, desc, **over):
    args = dict(ssm=FAKE, ssm_stride=128 * 64 * 128, num_slots=8, conv=None, conv_stride=0, conv_w=None,
                conv_b=None, slot=FAKE, scratch=None, batch=4, ntok=1, xbc=FAKE, dt=FAKE, A=FAKE, D=None,
                dt_bias=None, softplus=1, z=None, y=FAKE)
    args.update(over)
    return lib.mamba_state_update(ctypes.byref(desc), args["ssm"], args["ssm_stride"], args["num_slots"],
                                  args["conv"], args["conv_stride"], args["conv_w"], args["conv_b"], args["slot"],
                                  args["scratch"], args["batch"], args["ntok"], args["xbc"], args["dt"], args["A"],
                                  args["D"], args["dt_bias"], args["softplus"], args["z"], args["y"], None, None)


def test_state_update_host_errors(lib):
    d = bd.layer_desc(wl.NEMOTRON_H_8B)
    assert _state_update(lib, d, batch=0) == bd.MAMBA_OK  # nothing to do, nothing launched
    assert _state_update(lib, d, ssm=None) == bd.MAMBA_EINVAL
    assert _state_update(lib, d, slot=None) == bd.MAMBA_EINVAL
    assert _state_update(lib, d, A=None) == bd.MAMBA_EINVAL
    assert _state_update(lib, d, batch=-1) == bd.MAMBA_EINVAL
    assert _state_update(lib, d, ntok=0) == bd.MAMBA_EINVAL
    assert _state_update(lib, d, ntok=9) == bd.MAMBA_EINVAL
    assert _state_update(lib, d, ssm_stride=100) == bd.MAMBA_EINVAL
    assert _state_update(lib, d, num_slots=0) == bd.MAMBA_EINVAL
    assert _state_update(lib, d, conv=FAKE, conv_stride=10240 * 3) == bd.MAMBA_EINVAL  # conv_w missing
    assert _state_update(lib, d, ssm=FAKE + 8) == bd.MAMBA_EALIGN
    assert _state_update(lib, d, ssm_stride=128 * 64 * 128 + 4) == bd.MAMBA_EALIGN
    assert _state_update(lib, d, y=FAKE + 1) == bd.MAMBA_EALIGN
    odd = bd.layer_desc(wl.LayerShape(nheads=4, head_dim=24, d_state=40, n_groups=1))
    assert _state_update(lib, odd, ssm_stride=4 * 24 * 40) == bd.MAMBA_EUNSUPPORTED
    bad = bd.LayerDesc(128, 64, 128, 8, 4, 0, 1, 1, 1, 7)  # dt dtype code 7
    assert _state_update(lib, bad) == bd.MAMBA_EINVAL
    assert _state_update(lib, bd.LayerDesc(128, 64, 128, 8, 9, 0, 1, 1, 1, 0)) == bd.MAMBA_EINVAL  # W > 8


def test_conv_and_commit_host_errors(lib):
    d = bd.layer_desc(wl.NEMOTRON_H_8B)
    r = lib.mamba_conv_update(ctypes.byref(d), None, 10240 * 3, 8, FAKE, 4, 1, FAKE, FAKE, None, FAKE, None, None)
    assert r == bd.MAMBA_EINVAL
    r = lib.mamba_conv_update(ctypes.byref(d), FAKE, 10, 8, FAKE, 4, 1, FAKE, FAKE, None, FAKE, None, None)
    assert r == bd.MAMBA_EINVAL
    r = lib.mamba_conv_update(ctypes.byref(d), FAKE, 10240 * 3, 8, FAKE, 0, 1, FAKE, FAKE, None, FAKE, None, None)
    assert r == bd.MAMBA_OK
    # commit: ntok beyond num_spec cannot re-seat the conv window
    r = lib.mamba_spec_commit(ctypes.byref(d), FAKE, 128 * 64 * 128, 8, FAKE, 10240 * 3, FAKE, FAKE, FAKE, 4, 4,
                              None, None)
    assert r == bd.MAMBA_EINVAL
    r = lib.mamba_spec_commit(ctypes.byref(d), None, 128 * 64 * 128, 8, None, 0, FAKE, FAKE, FAKE, 4, 4, None, None)
    assert r == bd.MAMBA_EINVAL


def test_chunk_scan_host_errors(lib):
    d = bd.layer_desc(wl.NEMOTRON_H_8B)
    need = bd.mamba_chunk_scan_workspace_bytes(d, 1000, 2, 256)

    def call(**over):
        a = dict(ssm=FAKE, stride=128 * 64 * 128, ns=8, cu=FAKE, nseq=2, T=1000, slot=FAKE, hi=None, ck=None, mc=0,
                 ci=0, chunk=256, x=FAKE, dt=FAKE, A=FAKE, B=FAKE, C=FAKE, ws=FAKE, wsb=need)
        a.update(over)
        return lib.mamba_chunk_scan(ctypes.byref(d), a["ssm"], a["stride"], a["ns"], a["cu"], a["nseq"], a["T"],
                                    a["slot"], a["hi"], a["ck"], a["mc"], a["ci"], a["chunk"], a["x"], a["dt"],
                                    a["A"], a["B"], a["C"], None, None, 1, None, FAKE, a["ws"], a["wsb"], None, None)

    assert call(nseq=0) == bd.MAMBA_OK
    assert call(ssm=None) == bd.MAMBA_EINVAL
    assert call(ws=None) == bd.MAMBA_EINVAL
    assert call(wsb=need - 1) == bd.MAMBA_ENOSPACE
    assert call(chunk=100) == bd.MAMBA_EUNSUPPORTED  # neither a tensor-core nor a portable chunk
    assert call(ck=FAKE, mc=4, ci=1000) == bd.MAMBA_EINVAL  # interval not a multiple of the chunk
    assert call(ws=FAKE + 4) == bd.MAMBA_EALIGN


def test_conv_varlen_host_errors(lib):
    d = bd.layer_desc(wl.NEMOTRON_H_8B)

    def call(**over):
        a = dict(pool=FAKE, stride=10240 * 3, ns=8, cu=FAKE, nseq=2, T=100, slot=FAKE, xbc=FAKE, w=FAKE,
                 x=FAKE, B=FAKE, C=FAKE, dd=d)
        a.update(over)
        return lib.mamba_conv_varlen(ctypes.byref(a["dd"]), a["pool"], a["stride"], a["ns"], a["cu"], a["nseq"],
                                     a["T"], a["slot"], None, a["xbc"], a["w"], None, a["x"], a["B"], a["C"],
                                     None, None)

    assert call(nseq=0, T=0) == bd.MAMBA_OK
    assert call(nseq=0, T=5) == bd.MAMBA_EINVAL
    assert call(cu=None) == bd.MAMBA_EINVAL
    assert call(w=None) == bd.MAMBA_EINVAL
    assert call(B=None) == bd.MAMBA_EINVAL
    assert call(slot=None) == bd.MAMBA_EINVAL  # a conv pool needs slot ids
    assert call(stride=10) == bd.MAMBA_EINVAL
    assert call(x=FAKE + 2) == bd.MAMBA_EALIGN
    assert call(xbc=FAKE + 8) == bd.MAMBA_EALIGN
    odd = bd.layer_desc(wl.LayerShape(nheads=3, head_dim=2, d_state=8, n_groups=1, conv_kernel=4))
    assert call(dd=odd, stride=(6 + 16) * 3) == bd.MAMBA_EUNSUPPORTED  # x block of 6 bf16 is not 16 bytes


def test_checkpoint_ops_host_errors(lib):
    d = bd.layer_desc(wl.NEMOTRON_H_8B)
    st = 128 * 64 * 128
    r = lib.mamba_slot_copy(ctypes.byref(d), None, st, 8, None, 0, FAKE, FAKE, 4, None, None)
    assert r == bd.MAMBA_EINVAL
    r = lib.mamba_slot_copy(ctypes.byref(d), FAKE, st, 8, None, 0, FAKE, FAKE, 0, None, None)
    assert r == bd.MAMBA_OK  # nothing to copy
    r = lib.mamba_slot_copy(ctypes.byref(d), FAKE + 8, st, 8, None, 0, FAKE, FAKE, 4, None, None)
    assert r == bd.MAMBA_EALIGN
    r = lib.mamba_slot_copy(ctypes.byref(d), FAKE, st - 1, 8, None, 0, FAKE, FAKE, 4, None, None)
    assert r == bd.MAMBA_EINVAL
    eb = lib.mamba_int8_entry_bytes(ctypes.byref(d))
    # codes (1 MiB) + scales (64 KiB) + conv window (60 KiB), each on a 256-byte boundary
    assert eb == 128 * 64 * 128 + 128 * 128 * 4 + 10240 * 3 * 2
    for fn in (lib.mamba_ckpt_store_int8, lib.mamba_ckpt_load_int8):
        assert fn(ctypes.byref(d), FAKE, st, None, 0, 8, FAKE, FAKE, 4, None, 4, None, None) == bd.MAMBA_EINVAL
        assert fn(ctypes.byref(d), FAKE, st, None, 0, 8, FAKE, FAKE, 4, FAKE + 4, 4, None, None) == bd.MAMBA_EALIGN
        assert fn(ctypes.byref(d), FAKE, st, None, 0, 8, FAKE, FAKE, 0, FAKE, 4, None, None) == bd.MAMBA_OK
    odd = bd.layer_desc(wl.LayerShape(nheads=2, head_dim=4, d_state=12, n_groups=1, conv_kernel=4))
    assert lib.mamba_ckpt_store_int8(ctypes.byref(odd), FAKE, 96, None, 0, 8, FAKE, FAKE, 4, FAKE, 4, None,
                                     None) == bd.MAMBA_EUNSUPPORTED


def test_mamba1_host_errors(lib):
    d = bd.mamba1_desc(5120, 16)
    st = 5120 * 16

    def call(dd=d, pool=FAKE, stride=st, A=FAKE, x=FAKE):
        return lib.mamba1_state_update(ctypes.byref(dd), pool, stride, 8, FAKE, 4, x, FAKE, A, FAKE, FAKE, None,
                                       None, 1, None, FAKE, None, None)

    assert call(pool=None) == bd.MAMBA_EINVAL
    assert call(A=None) == bd.MAMBA_EINVAL
    assert call(stride=st - 1) == bd.MAMBA_EINVAL
    assert call(pool=FAKE + 2) == bd.MAMBA_EALIGN
    assert call(x=FAKE + 1) == bd.MAMBA_EALIGN
    assert call(dd=bd.mamba1_desc(5120, 12)) == bd.MAMBA_EUNSUPPORTED
    assert call(dd=bd.mamba1_desc(5121, 16)) == bd.MAMBA_EINVAL
    r = lib.mamba1_conv_update(ctypes.byref(d), None, 5120 * 3, 8, FAKE, 4, 1, FAKE, FAKE, None, FAKE, None, None)
    assert r == bd.MAMBA_EINVAL


def test_check_slot_ids(lib):
    """Host-side slot-id check: range, padding, distinct ids across rows and scratch slots."""
    import numpy as np
    ok = np.array([3, -1, 0, 7], np.int32)
    assert bd.mamba_check_slot_ids(ok, 8) == (bd.MAMBA_OK, -1)
    assert bd.mamba_check_slot_ids(np.array([3, 8], np.int32), 8) == (bd.MAMBA_EINVAL, 1)      # outside the pool
    assert bd.mamba_check_slot_ids(np.array([3, -2], np.int32), 8) == (bd.MAMBA_EINVAL, 1)     # below -1
    assert bd.mamba_check_slot_ids(np.array([5, -1, 5], np.int32), 8) == (bd.MAMBA_EINVAL, 2)  # used twice
    assert bd.mamba_check_slot_ids(np.array([-1, -1], np.int32), 8) == (bd.MAMBA_OK, -1)       # padding repeats
    assert bd.mamba_check_slot_ids(np.zeros(0, np.int32), 8) == (bd.MAMBA_OK, -1)
    # scratch slots: (batch, ntok); entry (i, j) is reported as batch + i*ntok + j
    rows = np.array([0, 1, -1], np.int32)
    scratch = np.array([[2, 3], [4, -1], [0, 1]], np.int32)  # the padding row's entries are ignored
    assert bd.mamba_check_slot_ids(rows, 8, scratch) == (bd.MAMBA_OK, -1)
    scratch[1, 1] = 2  # row 1 token 1 reuses row 0's scratch slot
    assert bd.mamba_check_slot_ids(rows, 8, scratch) == (bd.MAMBA_EINVAL, 3 + 1 * 2 + 1)
    scratch[1, 1] = 1  # a scratch slot equal to a live row's own slot
    assert bd.mamba_check_slot_ids(rows, 8, scratch) == (bd.MAMBA_EINVAL, 3 + 1 * 2 + 1)
    # invalid arguments
    bad = ctypes.c_int64(0)
    assert lib.mamba_check_slot_ids(None, 2, None, 0, 8, ctypes.byref(bad)) == bd.MAMBA_EINVAL and bad.value == -1
    assert lib.mamba_check_slot_ids(ok.ctypes.data, 4, None, 0, 0, None) == bd.MAMBA_EINVAL


def test_selftest_wait_timeout_needs_an_error_word(lib):
    assert lib.mamba_selftest_wait_timeout(None, None, None) == bd.MAMBA_EINVAL


def test_binding_rejects_tensors_of_the_wrong_dtype():
    """The binding checks each tensor's dtype against the layer descriptor before it passes a
    pointer (checked here with host tensors: the check comes before any device access)."""
    import torch
    shape = wl.TINY
    desc = bd.layer_desc(shape)  # bf16 state and activations, fp32 dt
    bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
    ok = dict(ssm_pool=torch.zeros(2, 4, 16, 16, dtype=bf), slot_ids=torch.zeros(1, dtype=i32),
              xbc=torch.zeros(1, 1, shape.conv_dim, dtype=bf), dt=torch.zeros(1, 1, 4, dtype=f32),
              A=torch.zeros(4, dtype=f32), y=torch.zeros(1, 1, 64, dtype=bf))
    for name, bad in (("ssm_pool", torch.zeros(2, 4, 16, 16, dtype=f32)), ("slot_ids", torch.zeros(1, dtype=torch.int64)),
                      ("xbc", torch.zeros(1, 1, shape.conv_dim, dtype=f32)), ("dt", torch.zeros(1, 1, 4, dtype=bf)),
                      ("y", torch.zeros(1, 1, 64, dtype=f32))):
        args = dict(ok, **{name: bad})
        with pytest.raises(ValueError, match=f"mamba_state_update: {name} must be"):
            bd.mamba_state_update(desc, args["ssm_pool"], args["slot_ids"], args["xbc"], args["dt"], args["A"],
                                  args["y"])
    with pytest.raises(ValueError, match="mamba_chunk_scan: has_initial_state must be"):
        bd.mamba_chunk_scan(desc, ok["ssm_pool"], torch.zeros(2, dtype=i32), ok["slot_ids"],
                            torch.zeros(1, 4, 16, dtype=bf), torch.zeros(1, 4, dtype=f32), ok["A"],
                            torch.zeros(1, 1, 16, dtype=bf), torch.zeros(1, 1, 16, dtype=bf),
                            torch.zeros(1, 4, 16, dtype=bf), None, has_initial_state=torch.zeros(1, dtype=torch.bool))


def test_zero_size_calls_launch_nothing(lib):
    """A call with no rows (or no sequences) returns MAMBA_OK before touching any pointer or the
    device: the Mamba1 step and conv, the speculative commit and the allocation-free prefill
    (the other entry points' zero-size calls are checked with their argument errors above)."""
    d = bd.layer_desc(wl.NEMOTRON_H_8B)
    d1 = bd.mamba1_desc(5120, 16)
    assert lib.mamba1_state_update(ctypes.byref(d1), None, 5120 * 16, 8, None, 0, None, None, None, None, None,
                                   None, None, 1, None, None, None, None) == bd.MAMBA_OK
    assert lib.mamba1_conv_update(ctypes.byref(d1), None, 5120 * 3, 8, None, 0, 1, None, None, None, None, None,
                                  None) == bd.MAMBA_OK
    assert lib.mamba_spec_commit(ctypes.byref(d), None, 128 * 64 * 128, 8, None, 0, None, None, None, 0, 4, None,
                                 None) == bd.MAMBA_OK
    assert lib.mamba_chunk_scan_noalloc(ctypes.byref(d), None, 128 * 64 * 128, 8, None, 0, 0, None, None, None, 0,
                                        0, 256, None, None, None, None, None, None, None, 1, None, None, None,
                                        None) == bd.MAMBA_OK
    # negative sizes are argument errors, not empty calls
    assert lib.mamba1_state_update(ctypes.byref(d1), None, 5120 * 16, 8, None, -1, None, None, None, None, None,
                                   None, None, 1, None, None, None, None) == bd.MAMBA_EINVAL
    assert lib.mamba_chunk_scan_noalloc(ctypes.byref(d), None, 128 * 64 * 128, 8, None, -1, 0, None, None, None, 0,
                                        0, 256, None, None, None, None, None, None, None, 1, None, None, None,
                                        None) == bd.MAMBA_EINVAL
