"""fp64 CPU oracle for the Mamba2 recurrent-state update -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The product path (the CUDA library and its binding) never does, and
shares no code with it.

The arithmetic lives in ``mamba_oracle.c`` (plain C, double precision, one loop per sum);
this module compiles it with gcc, loads it with ctypes and marshals numpy float64 arrays.
Each wrapper names the passage of the pages the C function follows:

* "Hybrid SSM / Mamba models and non-KV state" (mlinterviewnotes.com): state shapes,
  slot pool with a padding slot, the decode call with D / z / dt_bias / dt_softplus /
  state_batch_indices, prefill chunks seeded from the stored state, align-mode checkpoints, the
  affine-composition snippet.
* echobase "Mamba" notes: x = SiLU(Conv1d(x')), h_t = exp(Delta_t A) h_{t-1} + Delta_t B_t x_t,
  y_t = C_t h_t (+ D x_t), y_hat = y * SiLU(z), and the SSD form Y = (M (.) L) X.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mamba_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmamba_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libmamba_oracle.so`` (plain gcc, no ISA flags)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra",
           "-Wno-unused-parameter", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i32, i64 = ctypes.c_int, ctypes.c_int64
        lib.oracle_conv_update.argtypes = [i32, i32, i32, i32, _dp, _dp, _dp, _dp, _dp]
        lib.oracle_conv_update.restype = None
        lib.oracle_ssm_update.argtypes = [i32, i32, i32, i32, i32, _dp, _dp, _dp, _dp, _dp, _dp,
                                          _dp, _dp, _dp, i32, _dp, _dp]
        lib.oracle_ssm_update.restype = None
        lib.oracle_decode.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, _dp, i64, _dp, i64,
                                      _dp, _dp, _ip, _ip, _dp, _dp, _dp, _dp, _dp, i32, _dp, _dp, i32]
        lib.oracle_decode.restype = i32
        lib.oracle_spec_commit.argtypes = [i64, i32, i32, i32, i32, _dp, i64, _dp, i64, _ip, _ip, _ip]
        lib.oracle_spec_commit.restype = i32
        lib.oracle_mamba1_update.argtypes = [i32, i32, i32, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, i32, _dp, _dp]
        lib.oracle_mamba1_update.restype = None
        _i8 = ctypes.POINTER(ctypes.c_int8)
        _fp = ctypes.POINTER(ctypes.c_float)
        lib.oracle_int8_quantize.argtypes = [i32, i32, i32, _dp, _i8, _fp]
        lib.oracle_int8_quantize.restype = None
        lib.oracle_int8_dequantize.argtypes = [i32, i32, i32, _i8, _fp, _dp]
        lib.oracle_int8_dequantize.restype = None
        lib.oracle_conv_varlen.argtypes = [i32, i32, i32, i32, _ip, ctypes.POINTER(ctypes.c_uint8), _dp,
                                           _dp, _dp, _dp, _dp]
        lib.oracle_conv_varlen.restype = i32
        lib.oracle_prefill_steps.argtypes = [i32, i32, i32, i32, i32, _ip, _dp, _dp, _dp, _dp, _dp,
                                             _dp, _dp, _dp, i32, _dp, _dp, _dp, i32, i32, _dp, i32]
        lib.oracle_prefill_steps.restype = i32
        lib.oracle_prefill_materialised.argtypes = [i32, i32, i32, i32, i32, _dp, _dp, _dp, _dp,
                                                    _dp, _dp, _dp, _dp, i32, _dp, _dp, _dp]
        lib.oracle_prefill_materialised.restype = i32
        lib.oracle_prefill_chunked.argtypes = [i32, i32, i32, i32, i32, i32, _dp, _dp, _dp, _dp,
                                               _dp, _dp, _dp, _dp, i32, _dp, _dp, _dp]
        lib.oracle_prefill_chunked.restype = i32
        _lib = lib
        return lib


def _f64(a):
    """Contiguous float64 copy-or-view of ``a`` (None stays None)."""
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return None if a is None else a.ctypes.data_as(_dp)


def _pi(a):
    return None if a is None else a.ctypes.data_as(_ip)


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# --------------------------------------------------------------------------------------
# decode
# --------------------------------------------------------------------------------------

def conv_update(state, u, w, b=None):
    """Causal depthwise conv1d + SiLU over ``u`` (ntok x Cd) for one request.

    ``state`` is Cd x Wc (oldest column first) and is returned shifted by ntok with the new
    inputs appended.  Follows x = SiLU(Conv1d(x')) (echobase "Mamba" notes) and the conv
    state as a FIFO holding the most recent W-1 inputs ("Hybrid SSM / Mamba models and non-KV
    state", the two-objects list).  Returns (new_state, out).
    """
    lib = _load()
    st = _f64(state).copy()
    u = _f64(u)
    w = _f64(w)
    b = _f64(b)
    Cd, Wc = st.shape
    W = w.shape[1]
    ntok = u.shape[0]
    out = np.empty((ntok, Cd), np.float64)
    lib.oracle_conv_update(Cd, Wc, W, ntok, _p(st), _p(u), _p(w), _p(b), _p(out))
    return st, out


def ssm_update(h, x, B, C, dt, A, D=None, dt_bias=None, dt_softplus=True, z=None, record=False):
    """Selective state update of one request over ntok tokens (echobase "Mamba" notes).

    h: H x P x N.  x, z: ntok x H x P.  B, C: ntok x G x N.  dt: ntok x H.
    Returns (h_new, y) or (h_new, y, h_after_each_token) when ``record``.
    """
    lib = _load()
    h = _f64(h).copy()
    H, P, N = h.shape
    x = _f64(x)
    ntok = x.shape[0]
    B = _f64(B)
    G = B.shape[1]
    y = np.empty((ntok, H, P), np.float64)
    h_tok = np.empty((ntok, H, P, N), np.float64) if record else None
    lib.oracle_ssm_update(H, P, N, G, ntok, _p(h), _p(h_tok), _p(x), _p(B), _p(_f64(C)),
                          _p(_f64(dt)), _p(_f64(A)), _p(_f64(D)), _p(_f64(dt_bias)),
                          int(bool(dt_softplus)), _p(_f64(z)), _p(y))
    return (h, y, h_tok) if record else (h, y)


def mamba1_update(h, x, B, C, dt, A, D=None, dt_bias=None, dt_softplus=True, z=None):
    """Mamba1 (S6) state update of one request over ntok tokens (echobase "Mamba" notes, with a
    per-channel step and a D x N matrix A; the (D, N) Mamba1 state of "Hybrid SSM / Mamba models
    and non-KV state").  h: D x N.  x, dt, z: ntok x D.  B, C: ntok x N.  A: D x N.
    Returns (h_new, y) with y ntok x D."""
    lib = _load()
    h = _f64(h).copy()
    Dn, N = h.shape
    x = _f64(x)
    ntok = x.shape[0]
    y = np.empty((ntok, Dn), np.float64)
    lib.oracle_mamba1_update(Dn, N, ntok, _p(h), _p(x), _p(_f64(dt)), _p(_f64(A)), _p(_f64(B)), _p(_f64(C)),
                             _p(_f64(D)), _p(_f64(dt_bias)), int(bool(dt_softplus)), _p(_f64(z)), _p(y))
    return h, y


def decode(ssm_pool, slot, xbc, dt, A, *, conv_pool=None, conv_w=None, conv_b=None, scratch=None,
           D=None, dt_bias=None, dt_softplus=True, z=None, n_groups=1, y=None, nthreads=None):
    """Batched decode over a slot pool, in place on ``ssm_pool`` / ``conv_pool`` (fp64).

    ssm_pool: S x H x P x N.  conv_pool: S x Cd x Wc or None (then ``xbc`` is post-conv).
    slot: batch (int, -1 = padding).  scratch: batch x ntok or None.
    xbc: batch x ntok x Cd.  dt: batch x ntok x H.  z: batch x ntok x H x P or None.
    Returns y (batch x ntok x H x P); rows with slot -1 keep the values of ``y`` passed in
    (NaN when None), since the padding row's output is not written.
    """
    lib = _load()
    assert ssm_pool.dtype == np.float64 and ssm_pool.flags.c_contiguous
    S, H, P, N = ssm_pool.shape
    G = int(n_groups)
    xbc = _f64(xbc)
    batch, ntok, Cd = xbc.shape
    assert Cd == H * P + 2 * G * N
    if y is None:
        y = np.full((batch, ntok, H, P), np.nan)
    else:
        y = _f64(y).copy()
    W = Wc = 0
    conv_stride = 0
    if conv_pool is not None:
        assert conv_pool.dtype == np.float64 and conv_pool.flags.c_contiguous
        Wc = conv_pool.shape[2]
        W = np.asarray(conv_w).shape[1]
        conv_stride = Cd * Wc
    rc = lib.oracle_decode(H, P, N, G, W, Wc, ntok, batch, _p(ssm_pool), H * P * N,
                           _p(conv_pool), conv_stride, _p(_f64(conv_w)), _p(_f64(conv_b)),
                           _pi(_i32(slot)), _pi(_i32(scratch)), _p(xbc), _p(_f64(dt)), _p(_f64(A)),
                           _p(_f64(D)), _p(_f64(dt_bias)), int(bool(dt_softplus)), _p(_f64(z)), _p(y),
                           nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_decode failed: {rc}")
    return y


def spec_commit(ssm_pool, slot, scratch, accept, *, conv_pool=None):
    """Speculative commit (accept a of ntok drafts), in place on the fp64 pools."""
    lib = _load()
    S = ssm_pool.shape[0]
    elems = int(np.prod(ssm_pool.shape[1:]))
    scratch = _i32(scratch)
    batch, ntok = scratch.shape
    Cd = Wc = 0
    if conv_pool is not None:
        Cd, Wc = conv_pool.shape[1], conv_pool.shape[2]
    rc = lib.oracle_spec_commit(elems, Cd, Wc, ntok, batch, _p(ssm_pool), elems, _p(conv_pool),
                                Cd * Wc, _pi(_i32(slot)), _pi(scratch), _pi(_i32(accept)))
    if rc != 0:
        raise RuntimeError(f"oracle_spec_commit failed: {rc}")


# --------------------------------------------------------------------------------------
# prefill
# --------------------------------------------------------------------------------------

def int8_quantize(state):
    """Per-(head, k-channel) symmetric int8 quantisation of a temporal state H x P x N (the
    k-channel is the d_state index n).  Follows the int8 checkpoint store of "Hybrid SSM / Mamba
    models and non-KV state" (quantised once on store); computed in float32, the precision the
    codes are decided in.  Returns (q int8 H x P x N, scale float32 H x N)."""
    lib = _load()
    st = _f64(state)
    H, P, N = st.shape
    q = np.zeros((H, P, N), np.int8)
    sc = np.zeros((H, N), np.float32)
    lib.oracle_int8_quantize(H, P, N, _p(st), q.ctypes.data_as(ctypes.POINTER(ctypes.c_int8)),
                             sc.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    return q, sc


def int8_dequantize(q, scale):
    """state' = q * scale (float32 product), as float64 values (dequantised once on a hit)."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.int8)
    sc = np.ascontiguousarray(scale, dtype=np.float32)
    H, P, N = q.shape
    out = np.empty((H, P, N), np.float64)
    lib.oracle_int8_dequantize(H, P, N, q.ctypes.data_as(ctypes.POINTER(ctypes.c_int8)),
                               sc.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), _p(out))
    return out


def conv_varlen(cu_seqlens, u, w, b=None, *, state=None, init=None):
    """Varlen causal conv1d + SiLU of a prefill batch, with the conv state carried in and out.

    Follows x = SiLU(Conv1d(x')) (echobase "Mamba" notes) applied to whole prompts, with the
    conv state as the window of the most recent inputs that a later chunk continues from
    ("Hybrid SSM / Mamba models and non-KV state": the conv state object and the chunked-prefill
    hand-off).  u: T x Cd raw inputs; w: Cd x W; state: nseq x Cd x Wc (oldest first) or None
    (zeros, Wc = W-1); init: nseq flags (None = no sequence starts from its state).
    Returns (new_state, out) with out T x Cd.
    """
    lib = _load()
    u = _f64(u)
    T, Cd = u.shape
    w = _f64(w)
    W = w.shape[1]
    cu = _i32(cu_seqlens)
    nseq = cu.shape[0] - 1
    if state is None:
        st = np.zeros((nseq, Cd, W - 1), np.float64)
    else:
        st = _f64(state).copy()
    Wc = st.shape[2]
    flags = None if init is None else np.ascontiguousarray(init, dtype=np.uint8)
    out = np.full((T, Cd), np.nan)
    rc = lib.oracle_conv_varlen(Cd, Wc, W, nseq, _pi(cu),
                                None if flags is None else flags.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
                                _p(st), _p(u), _p(w), _p(_f64(b)), _p(out))
    if rc != 0:
        raise RuntimeError(f"oracle_conv_varlen failed: {rc}")
    return st, out


def prefill_steps(cu_seqlens, x, dt, A, B, C, *, h0=None, D=None, dt_bias=None, dt_softplus=True,
                  z=None, ckpt_interval=0, max_ckpt=0, nthreads=None):
    """Varlen prefill by the step recurrence.  Returns (y, h_final, h_ckpt or None).

    x, z: T x H x P; dt: T x H; B, C: T x G x N; h0: nseq x H x P x N or None.
    h_ckpt[s, k-1] is the state after the first k*ckpt_interval tokens of sequence s
    (NaN where the sequence is shorter).
    """
    lib = _load()
    x = _f64(x)
    T, H, P = x.shape
    B = _f64(B)
    G, N = B.shape[1], B.shape[2]
    cu = _i32(cu_seqlens)
    nseq = cu.shape[0] - 1
    y = np.empty((T, H, P), np.float64)
    hf = np.empty((nseq, H, P, N), np.float64)
    hc = np.full((nseq, max_ckpt, H, P, N), np.nan) if (ckpt_interval > 0 and max_ckpt > 0) else None
    rc = lib.oracle_prefill_steps(H, P, N, G, nseq, _pi(cu), _p(_f64(h0)), _p(x), _p(_f64(dt)),
                                  _p(_f64(A)), _p(B), _p(_f64(C)), _p(_f64(D)), _p(_f64(dt_bias)),
                                  int(bool(dt_softplus)), _p(_f64(z)), _p(y), _p(hf),
                                  int(ckpt_interval), int(max_ckpt), _p(hc),
                                  nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_prefill_steps failed: {rc}")
    return y, hf, hc


def prefill_materialised(x, dt, A, B, C, *, h0=None, D=None, dt_bias=None, dt_softplus=True, z=None):
    """One sequence by the materialised SSD form Y = (M (.) L) X.  Returns (y, h_final)."""
    lib = _load()
    x = _f64(x)
    T, H, P = x.shape
    B = _f64(B)
    G, N = B.shape[1], B.shape[2]
    y = np.empty((T, H, P), np.float64)
    hf = np.empty((H, P, N), np.float64)
    rc = lib.oracle_prefill_materialised(H, P, N, G, T, _p(_f64(h0)), _p(x), _p(_f64(dt)),
                                         _p(_f64(A)), _p(B), _p(_f64(C)), _p(_f64(D)),
                                         _p(_f64(dt_bias)), int(bool(dt_softplus)), _p(_f64(z)),
                                         _p(y), _p(hf))
    if rc != 0:
        raise RuntimeError(f"oracle_prefill_materialised failed: {rc}")
    return y, hf


def prefill_chunked(x, dt, A, B, C, *, chunk, h0=None, D=None, dt_bias=None, dt_softplus=True, z=None):
    """One sequence by the chunked SSD decomposition (fp64).  Returns (y, h_final)."""
    lib = _load()
    x = _f64(x)
    T, H, P = x.shape
    B = _f64(B)
    G, N = B.shape[1], B.shape[2]
    y = np.empty((T, H, P), np.float64)
    hf = np.empty((H, P, N), np.float64)
    rc = lib.oracle_prefill_chunked(H, P, N, G, T, int(chunk), _p(_f64(h0)), _p(x), _p(_f64(dt)),
                                    _p(_f64(A)), _p(B), _p(_f64(C)), _p(_f64(D)), _p(_f64(dt_bias)),
                                    int(bool(dt_softplus)), _p(_f64(z)), _p(y), _p(hf))
    if rc != 0:
        raise RuntimeError(f"oracle_prefill_chunked failed: {rc}")
    return y, hf
