"""Thin ctypes binding of libmamba_state.so (argument marshalling only).

Every function here has the name of the C entry point it calls, takes torch CUDA tensors (or
None for nullable arguments), passes their device pointers and sizes, and raises
:class:`MambaError` on a non-zero status.  All arithmetic happens in the CUDA kernels; there is
no CPU path.  Loading fails loudly when the library has not been built.

Layouts are the ones the C header documents (include/mamba_state.h); tensors must be
contiguous except the pools, whose slot stride is taken from ``stride(0)``.  Each tensor's
dtype is checked against the layer descriptor before its pointer is passed (ValueError), since
the C ABI sees only addresses.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import workloads as wl

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmamba_state.so")

MAMBA_OK, MAMBA_EINVAL, MAMBA_EUNSUPPORTED, MAMBA_ECUDA, MAMBA_EALIGN, MAMBA_ENOSPACE = 0, -1, -2, -3, -4, -5
MAMBA_F32, MAMBA_BF16 = 0, 1
MAMBA_ERR_SLOT_RANGE, MAMBA_ERR_ACCEPT_RANGE, MAMBA_ERR_SEQLENS, MAMBA_ERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8


class MambaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


class LayerDesc(ctypes.Structure):
    """Mirror of ``mamba_layer_desc``."""

    _fields_ = [(n, ctypes.c_int32) for n in ("nheads", "head_dim", "d_state", "n_groups", "conv_kernel",
                                              "num_spec", "state_dtype", "conv_dtype", "act_dtype",
                                              "dt_dtype")]


class Mamba1Desc(ctypes.Structure):
    """Mirror of ``mamba1_layer_desc``."""

    _fields_ = [(n, ctypes.c_int32) for n in ("d_inner", "d_state", "conv_kernel", "num_spec", "state_dtype",
                                              "conv_dtype", "act_dtype", "dt_dtype")]


def mamba1_desc(d_inner: int, d_state: int, conv_kernel: int = 4, num_spec: int = 0, state: str = wl.BF16,
                act: str = wl.BF16, dt: str = wl.F32) -> Mamba1Desc:
    code = wl.DTYPE_CODE
    return Mamba1Desc(d_inner, d_state, conv_kernel, num_spec, code[state], code[act], code[act], code[dt])


def layer_desc(shape: "wl.LayerShape", state: str = wl.BF16, act: str = wl.BF16, dt: str = wl.F32,
               conv: str | None = None) -> LayerDesc:
    code = wl.DTYPE_CODE
    return LayerDesc(shape.nheads, shape.head_dim, shape.d_state, shape.n_groups, shape.conv_kernel,
                     shape.num_spec, code[state], code[conv or act], code[act], code[dt])


_lock = threading.Lock()
_lib = None
_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_dp = ctypes.POINTER(LayerDesc)
_d1 = ctypes.POINTER(Mamba1Desc)

# (name, restype, argtypes) of every exported entry point
SIGNATURES = {
    "mamba_conv_dim": (_i32, [_dp]),
    "mamba_ssm_state_bytes": (_i64, [_dp]),
    "mamba_conv_state_bytes": (_i64, [_dp]),
    "mamba_decode_supported": (ctypes.c_int, [_dp]),
    "mamba_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "mamba_conv_update": (ctypes.c_int, [_dp, _vp, _i64, _i64, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "mamba_state_update": (ctypes.c_int, [_dp, _vp, _i64, _i64, _vp, _i64, _vp, _vp, _vp, _vp, _i32, _i32, _vp,
                                          _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp]),
    "mamba_spec_commit": (ctypes.c_int, [_dp, _vp, _i64, _i64, _vp, _i64, _vp, _vp, _vp, _i32, _i32, _vp, _vp]),
    "mamba_conv_varlen": (ctypes.c_int, [_dp, _vp, _i64, _i64, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                         _vp, _vp, _vp]),
    "mamba1_conv_update": (ctypes.c_int, [_d1, _vp, _i64, _i64, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "mamba1_state_update": (ctypes.c_int, [_d1, _vp, _i64, _i64, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                           _vp, _vp, _vp, _vp]),
    "mamba_slot_copy": (ctypes.c_int, [_dp, _vp, _i64, _i64, _vp, _i64, _vp, _vp, _i32, _vp, _vp]),
    "mamba_int8_entry_bytes": (_sz, [_dp]),
    "mamba_ckpt_store_int8": (ctypes.c_int, [_dp, _vp, _i64, _vp, _i64, _i64, _vp, _vp, _i32, _vp, _i64, _vp, _vp]),
    "mamba_ckpt_load_int8": (ctypes.c_int, [_dp, _vp, _i64, _vp, _i64, _i64, _vp, _vp, _i32, _vp, _i64, _vp, _vp]),
    "mamba_chunk_scan_workspace_bytes": (_sz, [_dp, _i32, _i32, _i32]),
    "mamba_chunk_scan": (ctypes.c_int, [_dp, _vp, _i64, _i64, _vp, _i32, _i32, _vp, _vp, _vp, _i32, _i32, _i32,
                                        _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _sz, _vp, _vp]),
    "mamba_chunk_scan_noalloc": (ctypes.c_int, [_dp, _vp, _i64, _i64, _vp, _i32, _i32, _vp, _vp, _vp, _i32, _i32,
                                                _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp]),
    "mamba_chunk_scan_static_scratch_bytes": (_sz, []),
    "mamba_check_slot_ids": (ctypes.c_int, [_vp, _i32, _vp, _i32, _i64, ctypes.POINTER(_i64)]),
    "mamba_selftest_wait_timeout": (ctypes.c_int, [_vp, _vp, _vp]),
}


def lib():
    """The loaded library; raises if it was not built (there is no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with recurrent_state_update_gb300.build.build()")
            h = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(h, name)
                f.restype = res
                f.argtypes = args
            _lib = h
        return _lib


def status_string(status: int) -> str:
    return lib().mamba_status_string(int(status)).decode()


def _check(rc: int, what: str):
    if rc != MAMBA_OK:
        raise MambaError(rc, what)


def _ptr(t):
    """Device pointer of a CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return t.data_ptr()


def _cptr(t):
    if t is not None and not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return _ptr(t)


def _code_dtype(code):
    import torch
    return torch.bfloat16 if code == MAMBA_BF16 else torch.float32


def _expect(what, **tensors):
    """Raises ValueError when a tensor's dtype is not the one the call reads it as.  Each keyword
    is (tensor or None, the torch dtype the library expects)."""
    for name, (t, want) in tensors.items():
        if t is not None and t.dtype != want:
            raise ValueError(f"{what}: {name} must be {want}, got {t.dtype}")


def _layer_dtypes(desc):
    """(state, conv, activations, dt, fp32, int32, uint8) torch dtypes of a Mamba2 or Mamba1 desc."""
    import torch
    return (_code_dtype(desc.state_dtype), _code_dtype(desc.conv_dtype), _code_dtype(desc.act_dtype),
            _code_dtype(desc.dt_dtype), torch.float32, torch.int32, torch.uint8)


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


# ------------------------------------------------------------------------------------------
# sizes
# ------------------------------------------------------------------------------------------

def mamba_conv_dim(desc: LayerDesc) -> int:
    return lib().mamba_conv_dim(ctypes.byref(desc))


def mamba_ssm_state_bytes(desc: LayerDesc) -> int:
    return lib().mamba_ssm_state_bytes(ctypes.byref(desc))


def mamba_conv_state_bytes(desc: LayerDesc) -> int:
    return lib().mamba_conv_state_bytes(ctypes.byref(desc))


def mamba_decode_supported(desc: LayerDesc) -> int:
    return lib().mamba_decode_supported(ctypes.byref(desc))


def mamba_selftest_wait_timeout(err_word, elapsed_ns=None, stream=None):
    """Diagnostic: one bounded wait that runs out (err_word: device int32; elapsed_ns: device int64)."""
    _check(lib().mamba_selftest_wait_timeout(_ptr(err_word), _ptr(elapsed_ns), _stream(stream)),
           "mamba_selftest_wait_timeout")


def mamba_check_slot_ids(slot_ids, num_slots: int, scratch_slots=None) -> tuple[int, int]:
    """Host-side check of one call's slot ids (numpy int32 arrays: (batch,) and (batch, ntok)).
    Returns (status, index of the first offending entry or -1)."""
    import numpy as np
    ids = np.ascontiguousarray(slot_ids, dtype=np.int32)
    sc = None if scratch_slots is None else np.ascontiguousarray(scratch_slots, dtype=np.int32)
    ntok = 0 if sc is None else (sc.shape[1] if sc.ndim == 2 else 1)
    bad = _i64(-1)
    rc = lib().mamba_check_slot_ids(ids.ctypes.data if ids.size else None, int(ids.shape[0]),
                                    None if sc is None else sc.ctypes.data, int(ntok), int(num_slots),
                                    ctypes.byref(bad))
    return rc, int(bad.value)


def mamba_chunk_scan_workspace_bytes(desc: LayerDesc, total_tokens: int, nseq: int, chunk: int) -> int:
    return lib().mamba_chunk_scan_workspace_bytes(ctypes.byref(desc), total_tokens, nseq, chunk)


# ------------------------------------------------------------------------------------------
# decode
# ------------------------------------------------------------------------------------------

def mamba_conv_update(desc: LayerDesc, conv_pool, slot_ids, xbc_in, conv_w, xbc_out, *, conv_b=None,
                      err_word=None, stream=None):
    """Causal conv1d + SiLU over (batch, ntok, conv_dim) inputs, conv state updated in place."""
    _, cv, act, _, f32, i32, _ = _layer_dtypes(desc)
    _expect("mamba_conv_update", conv_pool=(conv_pool, cv), slot_ids=(slot_ids, i32), xbc_in=(xbc_in, act),
            conv_w=(conv_w, f32), xbc_out=(xbc_out, act), conv_b=(conv_b, f32), err_word=(err_word, i32))
    batch, ntok = int(slot_ids.shape[0]), int(xbc_in.shape[1])
    rc = lib().mamba_conv_update(ctypes.byref(desc), _ptr(conv_pool), conv_pool.stride(0), conv_pool.shape[0],
                                 _cptr(slot_ids), batch, ntok, _cptr(xbc_in), _cptr(conv_w), _cptr(conv_b),
                                 _cptr(xbc_out), _ptr(err_word), _stream(stream))
    _check(rc, "mamba_conv_update")


def mamba_state_update(desc: LayerDesc, ssm_pool, slot_ids, xbc, dt, A, y, *, conv_pool=None, conv_w=None,
                       conv_b=None, scratch_slots=None, D=None, dt_bias=None, dt_softplus=True, z=None,
                       err_word=None, stream=None):
    """The batched decode step (conv fused when ``conv_pool`` is given), in place on the pools."""
    st, cv, act, dtt, f32, i32, _ = _layer_dtypes(desc)
    _expect("mamba_state_update", ssm_pool=(ssm_pool, st), slot_ids=(slot_ids, i32), xbc=(xbc, act), dt=(dt, dtt),
            A=(A, f32), y=(y, act), conv_pool=(conv_pool, cv), conv_w=(conv_w, f32), conv_b=(conv_b, f32),
            scratch_slots=(scratch_slots, i32), D=(D, f32), dt_bias=(dt_bias, f32), z=(z, act),
            err_word=(err_word, i32))
    batch, ntok = int(slot_ids.shape[0]), int(xbc.shape[1])
    conv_stride = conv_pool.stride(0) if conv_pool is not None else 0
    rc = lib().mamba_state_update(ctypes.byref(desc), _ptr(ssm_pool), ssm_pool.stride(0), ssm_pool.shape[0],
                                  _ptr(conv_pool), conv_stride, _cptr(conv_w), _cptr(conv_b), _cptr(slot_ids),
                                  _cptr(scratch_slots), batch, ntok, _cptr(xbc), _cptr(dt), _cptr(A), _cptr(D),
                                  _cptr(dt_bias), int(bool(dt_softplus)), _cptr(z), _cptr(y), _ptr(err_word),
                                  _stream(stream))
    _check(rc, "mamba_state_update")


def mamba_spec_commit(desc: LayerDesc, ssm_pool, slot_ids, scratch_slots, accept_len, *, conv_pool=None,
                      err_word=None, stream=None):
    """Keep accept_len[i] of the speculative tokens: copy the scratch state, re-seat the conv window."""
    st, cv, _, _, _, i32, _ = _layer_dtypes(desc)
    _expect("mamba_spec_commit", ssm_pool=(ssm_pool, st), slot_ids=(slot_ids, i32), scratch_slots=(scratch_slots, i32),
            accept_len=(accept_len, i32), conv_pool=(conv_pool, cv), err_word=(err_word, i32))
    batch, ntok = int(scratch_slots.shape[0]), int(scratch_slots.shape[1])
    conv_stride = conv_pool.stride(0) if conv_pool is not None else 0
    rc = lib().mamba_spec_commit(ctypes.byref(desc), _ptr(ssm_pool), ssm_pool.stride(0), ssm_pool.shape[0],
                                 _ptr(conv_pool), conv_stride, _cptr(slot_ids), _cptr(scratch_slots),
                                 _cptr(accept_len), batch, ntok, _ptr(err_word), _stream(stream))
    _check(rc, "mamba_spec_commit")


# ------------------------------------------------------------------------------------------
# Mamba1 (S6) layers
# ------------------------------------------------------------------------------------------

def mamba1_conv_update(desc: Mamba1Desc, conv_pool, slot_ids, x_in, conv_w, x_out, *, conv_b=None, err_word=None,
                       stream=None):
    """Causal conv1d + SiLU of a Mamba1 layer over (batch, ntok, d_inner) inputs, conv state in place."""
    _, cv, act, _, f32, i32, _ = _layer_dtypes(desc)
    _expect("mamba1_conv_update", conv_pool=(conv_pool, cv), slot_ids=(slot_ids, i32), x_in=(x_in, act),
            conv_w=(conv_w, f32), x_out=(x_out, act), conv_b=(conv_b, f32), err_word=(err_word, i32))
    batch, ntok = int(slot_ids.shape[0]), int(x_in.shape[1])
    rc = lib().mamba1_conv_update(ctypes.byref(desc), _ptr(conv_pool), conv_pool.stride(0), conv_pool.shape[0],
                                  _cptr(slot_ids), batch, ntok, _cptr(x_in), _cptr(conv_w), _cptr(conv_b),
                                  _cptr(x_out), _ptr(err_word), _stream(stream))
    _check(rc, "mamba1_conv_update")


def mamba1_state_update(desc: Mamba1Desc, ssm_pool, slot_ids, x, dt, A, B, C, y, *, D=None, dt_bias=None,
                        dt_softplus=True, z=None, err_word=None, stream=None):
    """The batched single-token Mamba1 decode step, in place on the (slots, d_inner, d_state) pool."""
    st, _, act, dtt, f32, i32, _ = _layer_dtypes(desc)
    _expect("mamba1_state_update", ssm_pool=(ssm_pool, st), slot_ids=(slot_ids, i32), x=(x, act), dt=(dt, dtt),
            A=(A, f32), B=(B, act), C=(C, act), y=(y, act), D=(D, f32), dt_bias=(dt_bias, f32), z=(z, act),
            err_word=(err_word, i32))
    batch = int(slot_ids.shape[0])
    rc = lib().mamba1_state_update(ctypes.byref(desc), _ptr(ssm_pool), ssm_pool.stride(0), ssm_pool.shape[0],
                                   _cptr(slot_ids), batch, _cptr(x), _cptr(dt), _cptr(A), _cptr(B), _cptr(C), _cptr(D),
                                   _cptr(dt_bias), int(bool(dt_softplus)), _cptr(z), _cptr(y), _ptr(err_word),
                                   _stream(stream))
    _check(rc, "mamba1_state_update")


# ------------------------------------------------------------------------------------------
# prefix-cache checkpoints
# ------------------------------------------------------------------------------------------

def mamba_slot_copy(desc: LayerDesc, ssm_pool, src_slots, dst_slots, *, conv_pool=None, err_word=None, stream=None):
    """Copy whole slot states src_slots[i] -> dst_slots[i] (checkpoint restore, copy-on-write)."""
    st, cv, _, _, _, i32, _ = _layer_dtypes(desc)
    _expect("mamba_slot_copy", ssm_pool=(ssm_pool, st), src_slots=(src_slots, i32), dst_slots=(dst_slots, i32),
            conv_pool=(conv_pool, cv), err_word=(err_word, i32))
    n = int(src_slots.shape[0])
    conv_stride = conv_pool.stride(0) if conv_pool is not None else 0
    rc = lib().mamba_slot_copy(ctypes.byref(desc), _ptr(ssm_pool), ssm_pool.stride(0), ssm_pool.shape[0],
                               _ptr(conv_pool), conv_stride, _cptr(src_slots), _cptr(dst_slots), n, _ptr(err_word),
                               _stream(stream))
    _check(rc, "mamba_slot_copy")


def mamba_int8_entry_bytes(desc: LayerDesc) -> int:
    return lib().mamba_int8_entry_bytes(ctypes.byref(desc))


def mamba_ckpt_store_int8(desc: LayerDesc, ssm_pool, src_slots, dst_entries, store, *, conv_pool=None,
                          err_word=None, stream=None):
    """Quantise slots into int8 store entries (per-(head, d_state channel) symmetric scales)."""
    st, cv, _, _, _, i32, _ = _layer_dtypes(desc)
    _expect("mamba_ckpt_store_int8", ssm_pool=(ssm_pool, st), src_slots=(src_slots, i32),
            dst_entries=(dst_entries, i32), conv_pool=(conv_pool, cv), err_word=(err_word, i32))
    n = int(src_slots.shape[0])
    eb = mamba_int8_entry_bytes(desc)
    conv_stride = conv_pool.stride(0) if conv_pool is not None else 0
    rc = lib().mamba_ckpt_store_int8(ctypes.byref(desc), _ptr(ssm_pool), ssm_pool.stride(0), _ptr(conv_pool),
                                     conv_stride, ssm_pool.shape[0], _cptr(src_slots), _cptr(dst_entries), n,
                                     _ptr(store), (store.numel() * store.element_size()) // eb, _ptr(err_word),
                                     _stream(stream))
    _check(rc, "mamba_ckpt_store_int8")


def mamba_ckpt_load_int8(desc: LayerDesc, ssm_pool, src_entries, dst_slots, store, *, conv_pool=None,
                         err_word=None, stream=None):
    """Dequantise int8 store entries into slots."""
    st, cv, _, _, _, i32, _ = _layer_dtypes(desc)
    _expect("mamba_ckpt_load_int8", ssm_pool=(ssm_pool, st), src_entries=(src_entries, i32),
            dst_slots=(dst_slots, i32), conv_pool=(conv_pool, cv), err_word=(err_word, i32))
    n = int(src_entries.shape[0])
    eb = mamba_int8_entry_bytes(desc)
    conv_stride = conv_pool.stride(0) if conv_pool is not None else 0
    rc = lib().mamba_ckpt_load_int8(ctypes.byref(desc), _ptr(ssm_pool), ssm_pool.stride(0), _ptr(conv_pool),
                                    conv_stride, ssm_pool.shape[0], _cptr(src_entries), _cptr(dst_slots), n,
                                    _ptr(store), (store.numel() * store.element_size()) // eb, _ptr(err_word),
                                    _stream(stream))
    _check(rc, "mamba_ckpt_load_int8")


# ------------------------------------------------------------------------------------------
# prefill
# ------------------------------------------------------------------------------------------

def mamba_conv_varlen(desc: LayerDesc, cu_seqlens, xbc, conv_w, x_out, B_out, C_out, *, conv_pool=None,
                      slot_ids=None, has_initial_state=None, conv_b=None, err_word=None, stream=None):
    """Varlen causal conv1d + SiLU of a prefill batch into x | B | C, continuing each sequence
    from its conv state and writing the state back (when ``conv_pool`` is given)."""
    _, cv, act, _, f32, i32, u8 = _layer_dtypes(desc)
    _expect("mamba_conv_varlen", cu_seqlens=(cu_seqlens, i32), xbc=(xbc, act), conv_w=(conv_w, f32), x_out=(x_out, act),
            B_out=(B_out, act), C_out=(C_out, act), conv_pool=(conv_pool, cv), slot_ids=(slot_ids, i32),
            has_initial_state=(has_initial_state, u8), conv_b=(conv_b, f32), err_word=(err_word, i32))
    nseq = int(cu_seqlens.shape[0]) - 1
    total = int(xbc.shape[0])
    conv_stride = conv_pool.stride(0) if conv_pool is not None else 0
    num_slots = conv_pool.shape[0] if conv_pool is not None else 0
    rc = lib().mamba_conv_varlen(ctypes.byref(desc), _ptr(conv_pool), conv_stride, num_slots, _cptr(cu_seqlens),
                                 nseq, total, _cptr(slot_ids), _cptr(has_initial_state), _cptr(xbc), _cptr(conv_w),
                                 _cptr(conv_b), _cptr(x_out), _cptr(B_out), _cptr(C_out), _ptr(err_word),
                                 _stream(stream))
    _check(rc, "mamba_conv_varlen")


def mamba_chunk_scan(desc: LayerDesc, ssm_pool, cu_seqlens, slot_ids, x, dt, A, B, C, y, workspace, *,
                     has_initial_state=None, ckpt_slots=None, ckpt_interval=0, chunk=256, D=None, dt_bias=None,
                     dt_softplus=True, z=None, err_word=None, stream=None):
    """Varlen chunked prefill (SSD form); final states and checkpoints written into the pool."""
    st, _, act, dtt, f32, i32, u8 = _layer_dtypes(desc)
    _expect("mamba_chunk_scan", ssm_pool=(ssm_pool, st), cu_seqlens=(cu_seqlens, i32), slot_ids=(slot_ids, i32), x=(x, act),
            dt=(dt, dtt), A=(A, f32), B=(B, act), C=(C, act), y=(y, act), has_initial_state=(has_initial_state, u8),
            ckpt_slots=(ckpt_slots, i32), D=(D, f32), dt_bias=(dt_bias, f32), z=(z, act), err_word=(err_word, i32))
    nseq = int(cu_seqlens.shape[0]) - 1
    total = int(x.shape[0])
    max_ckpt = int(ckpt_slots.shape[1]) if ckpt_slots is not None else 0
    rc = lib().mamba_chunk_scan(ctypes.byref(desc), _ptr(ssm_pool), ssm_pool.stride(0), ssm_pool.shape[0],
                                _cptr(cu_seqlens), nseq, total, _cptr(slot_ids), _cptr(has_initial_state),
                                _cptr(ckpt_slots), max_ckpt, int(ckpt_interval), int(chunk), _cptr(x), _cptr(dt),
                                _cptr(A), _cptr(B), _cptr(C), _cptr(D), _cptr(dt_bias), int(bool(dt_softplus)),
                                _cptr(z), _cptr(y), _ptr(workspace),
                                0 if workspace is None else workspace.numel() * workspace.element_size(),
                                _ptr(err_word), _stream(stream))
    _check(rc, "mamba_chunk_scan")


def mamba_chunk_scan_static_scratch_bytes() -> int:
    return lib().mamba_chunk_scan_static_scratch_bytes()


def mamba_chunk_scan_noalloc(desc: LayerDesc, ssm_pool, cu_seqlens, slot_ids, x, dt, A, B, C, y, *,
                             has_initial_state=None, ckpt_slots=None, ckpt_interval=0, chunk=256, D=None,
                             dt_bias=None, dt_softplus=True, z=None, err_word=None, stream=None):
    """mamba_chunk_scan for callers that cannot allocate: the library's fixed scratch is used
    instead of a caller workspace (see the C header for its size limit and sharing rules)."""
    st, _, act, dtt, f32, i32, u8 = _layer_dtypes(desc)
    _expect("mamba_chunk_scan_noalloc", ssm_pool=(ssm_pool, st), cu_seqlens=(cu_seqlens, i32), slot_ids=(slot_ids, i32), x=(x, act),
            dt=(dt, dtt), A=(A, f32), B=(B, act), C=(C, act), y=(y, act), has_initial_state=(has_initial_state, u8),
            ckpt_slots=(ckpt_slots, i32), D=(D, f32), dt_bias=(dt_bias, f32), z=(z, act), err_word=(err_word, i32))
    nseq = int(cu_seqlens.shape[0]) - 1
    total = int(x.shape[0])
    max_ckpt = int(ckpt_slots.shape[1]) if ckpt_slots is not None else 0
    rc = lib().mamba_chunk_scan_noalloc(ctypes.byref(desc), _ptr(ssm_pool), ssm_pool.stride(0), ssm_pool.shape[0],
                                        _cptr(cu_seqlens), nseq, total, _cptr(slot_ids), _cptr(has_initial_state),
                                        _cptr(ckpt_slots), max_ckpt, int(ckpt_interval), int(chunk), _cptr(x),
                                        _cptr(dt), _cptr(A), _cptr(B), _cptr(C), _cptr(D), _cptr(dt_bias),
                                        int(bool(dt_softplus)), _cptr(z), _cptr(y), _ptr(err_word), _stream(stream))
    _check(rc, "mamba_chunk_scan_noalloc")
