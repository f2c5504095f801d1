"""Seeded synthetic inputs for the Mamba2 recurrent-state update.

This module holds only input recipes (shapes, distributions, seeds, storage rounding).  It
contains none of the method's arithmetic and is shared by the tests, the benchmark and the
oracle checks, so that every side sees the same stored values.

Shapes follow the Nemotron-H-8B Mamba2 mixer given in "Hybrid SSM / Mamba models and non-KV
state" (mlinterviewnotes.com), section on vLLM's state shapes: 128 heads x head_dim 64,
d_state 128, 8 groups, conv kernel 4, conv_dim = d_inner + 2*g*d_state = 10240.

Value distributions (the workload recipe):
  x, z ~ N(0, 1);  B, C ~ N(0, 1)/sqrt(N);  A_h = -exp(U(ln 1, ln 16));  D_h ~ N(0, 1);
  conv taps ~ N(0, 1)/2;  initial SSM and conv states ~ N(0, 0.1^2);
  dt_bias_h = softplus^-1(u_h) with u_h log-uniform in [0.005, 0.02];  raw dt ~ N(0, 1)
  redrawn until dt + dt_bias lies in [softplus^-1(1e-3), softplus^-1(0.1)], i.e. the step
  size stays in [1e-3, 0.1].
Values are drawn in float64 and rounded once to the storage type (bf16 round-to-nearest-even
or fp32); both the GPU and the oracle receive exactly those stored values.

Wide-step inputs (parity cases beyond the configs' small steps; the method is defined for any
step Delta > 0 and any A < 0): the step itself is drawn log-uniform in [lo, hi] per (token, head)
and raw dt = softplus^-1(step) - dt_bias, so that with A down to -16 the per-token decay exponent
Delta*|A| spans about 1e-3 .. 80 (WIDE_STEPS), or lies only in the large range (LARGE_STEPS).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

F32 = "f32"
BF16 = "bf16"
DTYPE_CODE = {F32: 0, BF16: 1}
DTYPE_BYTES = {F32: 4, BF16: 2}


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """One Mamba2 layer: heads, head_dim, d_state, groups, conv kernel, speculative columns."""

    nheads: int
    head_dim: int
    d_state: int
    n_groups: int
    conv_kernel: int = 4
    num_spec: int = 0

    @property
    def conv_dim(self) -> int:
        return self.nheads * self.head_dim + 2 * self.n_groups * self.d_state

    @property
    def conv_cols(self) -> int:
        return self.conv_kernel - 1 + self.num_spec

    def with_spec(self, num_spec: int) -> "LayerShape":
        return dataclasses.replace(self, num_spec=num_spec)


# Nemotron-H-8B mixer shape (TP = 1).
NEMOTRON_H_8B = LayerShape(nheads=128, head_dim=64, d_state=128, n_groups=8, conv_kernel=4)
# Tiny decode shape: 4 heads x 16 x 16, one group, conv kernel 4 (conv_dim 96).
TINY = LayerShape(nheads=4, head_dim=16, d_state=16, n_groups=1, conv_kernel=4)

# Workloads, by what they are.
TINY_DECODE = dict(name="tiny decode, 4 x 16 x 16 fp32 state, batch 4 of 8 slots, 32 steps",
                   shape=TINY, layers=1, batch=4, pool=8, steps=32, state=F32, act=F32, seed=0)
NEMOTRON_DECODE = dict(name="Nemotron-H-8B decode, 48 layers, batch 256 of 512 slots, bf16 state",
                       shape=NEMOTRON_H_8B, layers=48, batch=256, pool=512, steps=1, state=BF16,
                       act=BF16, seed=1)
PADDING_SWEEP = dict(name="batch/padding sweep at the Nemotron-H-8B shape, 10% padded, 16 steps",
                     shape=NEMOTRON_H_8B, batches=(1, 8, 64, 256, 1024), pool=1536, pad_frac=0.1,
                     steps=16, state=BF16, act=BF16, seed=2)
CHUNKED_PREFILL = dict(name="varlen chunked prefill, 8 sequences of 512..8192 summing to 32768",
                       shape=NEMOTRON_H_8B, nseq=8, len_lo=512, len_hi=8192, total=32768,
                       chunk=256, ckpt_interval=1024, state=BF16, act=BF16, seed=3)
SPEC_DECODE = dict(name="speculative decode, batch 128, 4 draft tokens, 4 scratch slots each",
                   shape=NEMOTRON_H_8B.with_spec(4), batch=128, ntok=4, state=BF16, act=BF16, seed=4)


MAMBA1_DECODE = dict(name="Mamba1 (S6) decode, Mamba-2.8B-like layers (d_inner 5120, d_state 16, W 4), 64 layers, "
                          "batch 256 of 512 slots, bf16 state",
                     d_inner=5120, d_state=16, conv_kernel=4, layers=64, batch=256, pool=512, seed=6)


def rng(*key: int) -> np.random.Generator:
    """PCG64 stream for a (config seed, layer, step, ...) key."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


# --------------------------------------------------------------------------------------
# storage rounding (numpy has no bf16: bf16 values are carried as their uint16 bit patterns)
# --------------------------------------------------------------------------------------

def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 bits."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        rounded = np.where(nan, np.uint16(0x7FC0), rounded)
    return rounded


def bf16_bits_to_f32(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def store(a, dtype: str) -> np.ndarray:
    """Round float64 values to the storage dtype: float32 array, or uint16 bf16 bits."""
    if dtype == F32:
        return np.ascontiguousarray(a, dtype=np.float32)
    if dtype == BF16:
        return f32_to_bf16_bits(np.asarray(a, dtype=np.float64).astype(np.float32))
    raise ValueError(dtype)


def upcast(stored: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of stored data (inverse view of :func:`store`)."""
    if dtype == F32:
        return np.asarray(stored, dtype=np.float32).astype(np.float64)
    if dtype == BF16:
        return bf16_bits_to_f32(stored).astype(np.float64)
    raise ValueError(dtype)


# --------------------------------------------------------------------------------------
# per-layer parameters and per-step inputs
# --------------------------------------------------------------------------------------

DELTA_LO, DELTA_HI = 1e-3, 0.1
WIDE_STEPS = (1e-3, 5.0)   # tiny and large steps mixed
LARGE_STEPS = (0.2, 5.0)   # large steps only


def _inv_softplus(u):
    return np.log(np.expm1(u))


def layer_params(g: np.random.Generator, shape: LayerShape) -> dict:
    """A, D, dt_bias (per head) and conv taps (conv_dim x W), all float32."""
    H = shape.nheads
    A = -np.exp(g.uniform(math.log(1.0), math.log(16.0), size=H))
    D = g.standard_normal(H)
    u = np.exp(g.uniform(math.log(0.005), math.log(0.02), size=H))
    dt_bias = _inv_softplus(u)
    conv_w = g.standard_normal((shape.conv_dim, shape.conv_kernel)) / 2.0
    return dict(A=store(A, F32), D=store(D, F32), dt_bias=store(dt_bias, F32),
                conv_w=store(conv_w, F32))


def raw_dt(g: np.random.Generator, dt_bias: np.ndarray, lead: tuple) -> np.ndarray:
    """Raw dt ~ N(0, 1) per (lead..., head), redrawn until dt + dt_bias keeps the step in range."""
    lo = _inv_softplus(DELTA_LO) - dt_bias.astype(np.float64)
    hi = _inv_softplus(DELTA_HI) - dt_bias.astype(np.float64)
    out = g.standard_normal(lead + dt_bias.shape)
    bad = (out < lo) | (out > hi)
    while bad.any():
        out[bad] = g.standard_normal(int(bad.sum()))
        bad = (out < lo) | (out > hi)
    return out


def wide_dt(g: np.random.Generator, dt_bias: np.ndarray, lead: tuple, steps: tuple) -> np.ndarray:
    """Raw dt per (lead..., head) whose step softplus(dt + dt_bias) is log-uniform in steps = (lo, hi)."""
    lo, hi = steps
    u = np.exp(g.uniform(math.log(lo), math.log(hi), size=lead + dt_bias.shape))
    return _inv_softplus(u) - dt_bias.astype(np.float64)


def step_dt(g: np.random.Generator, dt_bias: np.ndarray, lead: tuple, steps) -> np.ndarray:
    """The configs' raw dt (steps None) or wide-step raw dt (steps = (lo, hi))."""
    return raw_dt(g, dt_bias, lead) if steps is None else wide_dt(g, dt_bias, lead, steps)


def xbc_values(g: np.random.Generator, shape: LayerShape, lead: tuple) -> np.ndarray:
    """Raw xBC rows (lead..., conv_dim): x channels N(0,1), B and C channels N(0,1)/sqrt(N)."""
    HP = shape.nheads * shape.head_dim
    v = g.standard_normal(lead + (shape.conv_dim,))
    v[..., HP:] /= math.sqrt(shape.d_state)
    return v


def decode_inputs(g: np.random.Generator, shape: LayerShape, params: dict, batch: int, ntok: int,
                  act: str, with_z: bool = True, steps=None) -> dict:
    """One decode step's inputs: xbc (batch, ntok, conv_dim), dt fp32 (batch, ntok, H), z."""
    xbc = store(xbc_values(g, shape, (batch, ntok)), act)
    dt = store(step_dt(g, params["dt_bias"], (batch, ntok), steps), F32)
    z = store(g.standard_normal((batch, ntok, shape.nheads * shape.head_dim)), act) if with_z else None
    return dict(xbc=xbc, dt=dt, z=z)


def initial_states(g: np.random.Generator, shape: LayerShape, nslots: int, state: str,
                   conv: str | None) -> dict:
    """Slot pools filled with N(0, 0.1^2): ssm (S, H, P, N) and conv (S, conv_dim, Wc)."""
    ssm = store(0.1 * g.standard_normal((nslots, shape.nheads, shape.head_dim, shape.d_state)), state)
    out = dict(ssm=ssm)
    if conv is not None:
        out["conv"] = store(0.1 * g.standard_normal((nslots, shape.conv_dim, shape.conv_cols)), conv)
    return out


def slot_ids(g: np.random.Generator, pool: int, batch: int, pad_frac: float = 0.0) -> np.ndarray:
    """Random distinct slot ids; round(pad_frac * batch) rows (random positions) set to -1."""
    ids = g.choice(pool, size=batch, replace=False).astype(np.int32)
    npad = int(round(pad_frac * batch))
    if npad:
        ids[g.choice(batch, size=npad, replace=False)] = -1
    return ids


def prefill_lengths(g: np.random.Generator, nseq: int, lo: int, hi: int, total: int) -> np.ndarray:
    """nseq integer lengths in [lo, hi] summing to ``total`` (draw nseq-1, the last closes the sum)."""
    for _ in range(100000):
        head = g.integers(lo, hi + 1, size=nseq - 1)
        last = total - int(head.sum())
        if lo <= last <= hi:
            return np.concatenate([head, [last]]).astype(np.int32)
    raise RuntimeError("could not draw lengths")


def cu_seqlens(lengths) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(lengths, dtype=np.int64))]).astype(np.int32)


def prefill_inputs(g: np.random.Generator, shape: LayerShape, params: dict, T: int, act: str,
                   dt_dtype: str = F32, with_z: bool = False, steps=None) -> dict:
    """Post-conv prefill inputs: x (T, H, P), B, C (T, G, N), dt (T, H), z (T, H, P) optional."""
    H, P, N, G = shape.nheads, shape.head_dim, shape.d_state, shape.n_groups
    x = store(g.standard_normal((T, H, P)), act)
    B = store(g.standard_normal((T, G, N)) / math.sqrt(N), act)
    C = store(g.standard_normal((T, G, N)) / math.sqrt(N), act)
    dt = store(step_dt(g, params["dt_bias"], (T,), steps), dt_dtype)
    z = store(g.standard_normal((T, H, P)), act) if with_z else None
    return dict(x=x, B=B, C=C, dt=dt, z=z)


def prefill_xbc(g: np.random.Generator, shape: LayerShape, T: int, act: str) -> np.ndarray:
    """Raw (pre-conv) prefill rows xBC (T, conv_dim), distributed like the decode inputs."""
    return store(xbc_values(g, shape, (T,)), act)


def mamba1_params(g: np.random.Generator, d_inner: int, d_state: int, conv_kernel: int) -> dict:
    """Mamba1 layer parameters: A (D, N) = -exp(U(ln 1, ln 16)), D, dt_bias (per channel), conv taps."""
    A = -np.exp(g.uniform(math.log(1.0), math.log(16.0), size=(d_inner, d_state)))
    D = g.standard_normal(d_inner)
    u = np.exp(g.uniform(math.log(0.005), math.log(0.02), size=d_inner))
    conv_w = g.standard_normal((d_inner, conv_kernel)) / 2.0
    return dict(A=store(A, F32), D=store(D, F32), dt_bias=store(_inv_softplus(u), F32), conv_w=store(conv_w, F32))


def mamba1_inputs(g: np.random.Generator, params: dict, batch: int, d_state: int, act: str) -> dict:
    """One Mamba1 decode step: x (conv output) and z N(0,1), B, C N(0,1)/sqrt(N), raw dt fp32."""
    Dn = params["D"].shape[0]
    x = store(g.standard_normal((batch, Dn)), act)
    B = store(g.standard_normal((batch, d_state)) / math.sqrt(d_state), act)
    C = store(g.standard_normal((batch, d_state)) / math.sqrt(d_state), act)
    dt = store(raw_dt(g, params["dt_bias"], (batch,)), F32)
    z = store(g.standard_normal((batch, Dn)), act)
    return dict(x=x, B=B, C=C, dt=dt, z=z)


def accept_lengths(g: np.random.Generator, batch: int, ntok: int) -> np.ndarray:
    """Accepted draft counts, uniform in 0..ntok."""
    return g.integers(0, ntok + 1, size=batch).astype(np.int32)
