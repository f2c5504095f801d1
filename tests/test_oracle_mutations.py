"""Planted mistakes in a copy of the fp64 oracle must each fail a pin (CPU only).

The pins in test_oracle_pins.py are only worth something if a plausible slip in the oracle's
arithmetic breaks one of them.  Each case below copies the oracle's C source into a scratch
directory, changes one expression the way a hurried reader of the pages might (a dropped term,
a wrong sign or index, a swapped operand, an off-by-one bound), rebuilds the copy and runs the
whole pin suite against it in a separate process.  The pin suite must fail.  The unchanged copy
must pass, so a failure means the planted mistake was caught, not that the harness is broken.

Nothing here touches the repository's own oracle build or the CUDA library.
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (what the mistake is, text in mamba_oracle.c, what it becomes); the first occurrence changes
MUTATIONS = [
    # decode step (echobase "Mamba" notes, block equations; selective_state_update's D and z)
    ("skip term D x dropped", "double yv = acc + (D ? D[hh] * xv : 0.0);", "double yv = acc;"),
    ("decay sign flipped", "const double a = exp(delta * A[hh]);", "const double a = exp(-delta * A[hh]);"),
    ("C used in place of B in the input term", "hrow[n] = a * hrow[n] + delta * Bj[n] * xv;",
     "hrow[n] = a * hrow[n] + delta * Cj[n] * xv;"),
    ("readout from the decayed old state", "acc += Ct[n] * h[(int64_t)p * N + n];",
     "acc += Ct[n] * h[(int64_t)p * N + n] * a;"),
    ("dt_bias dropped", "double s = dt + (dt_bias ? dt_bias[head] : 0.0);", "double s = dt;"),
    ("heads mapped to groups round-robin", "const int g = hh / (c->H / c->G);", "const int g = hh % c->G;"),
    ("gate z without SiLU", "if (z) yv *= silu(z[xi]);", "if (z) yv *= z[xi];"),
    ("softplus replaced by exp below zero", "s > 0.0 ? s + log1p(exp(-s)) : log1p(exp(s))",
     "s > 0.0 ? s + log1p(exp(-s)) : exp(s)"),
    ("sigmoid of the negative branch inverted", "return e / (1.0 + e);", "return 1.0 / (1.0 + e);"),
    # the slot pool: scratch slots of a speculative step and the commit
    ("every scratch slot gets the last token's state",
     "memcpy(c->ssm_pool + (int64_t)d * c->ssm_stride, h_tok + (int64_t)j * HPN,",
     "memcpy(c->ssm_pool + (int64_t)d * c->ssm_stride, h_tok + (int64_t)(c->ntok - 1) * HPN,"),
    ("commit copies the state one token early",
     "ssm_pool + (int64_t)scratch[(int64_t)i * ntok + (a - 1)] * ssm_stride,",
     "ssm_pool + (int64_t)scratch[(int64_t)i * ntok + (a > 1 ? a - 2 : 0)] * ssm_stride,"),
    ("commit moves the conv window by the accepted count", "const int shift = ntok - a;", "const int shift = a;"),
    # causal conv1d over the conv state (the conv-state FIFO of the most recent inputs)
    ("conv bias dropped", "double v = b ? b[c] : 0.0;", "double v = 0.0;"),
    ("conv state keeps the output instead of the input", "st[Wc - 1] = u[(int64_t)j * Cd + c];",
     "st[Wc - 1] = out[(int64_t)j * Cd + c];"),
    ("conv taps reversed", "v += w[(int64_t)c * W + k] * st[Wc - (W - 1) + k];",
     "v += w[(int64_t)c * W + (W - 2 - k)] * st[Wc - (W - 1) + k];"),
    ("conv window shifted by one too few",
     "for (int k = Wc - 1; k >= 0; --k) st[k] = (k - shift >= 0) ? st[k - shift] : 0.0;",
     "for (int k = Wc - 1; k >= 0; --k) st[k] = (k - shift + 1 >= 0 && k - shift + 1 < Wc) ? st[k - shift + 1] : 0.0;"),
    # SSD forms (Y = (M (.) L) X, its chunked decomposition and the chunk-state hand-off)
    ("decay product starts one token early", "for (int k = j + 1; k <= i; ++k) prod *= Abar[k];",
     "for (int k = j; k <= i; ++k) prod *= Abar[k];"),
    ("off-diagonal term measured from the chunk's first token", "acc += exp(cum[i]) * ch;",
     "acc += exp(cum[i] - cum[0]) * ch;"),
    ("diagonal of the masked block dropped", "for (int j = 0; j <= i; ++j) {", "for (int j = 0; j < i; ++j) {"),
    ("chunk state passed on without its decay", "for (int64_t e = 0; e < PN; ++e) h[e] = exp(cum_end) * h[e] + S[e];",
     "for (int64_t e = 0; e < PN; ++e) h[e] = h[e] + S[e];"),
    ("checkpoint taken one token late",
     "if (c->h_ckpt && c->ckpt_interval > 0 && done % c->ckpt_interval == 0) {",
     "if (c->h_ckpt && c->ckpt_interval > 0 && (done + 1) % c->ckpt_interval == 0) {"),
    # int8 checkpoint quantiser (per-(head, k-channel) symmetric)
    ("column maximum taken over the wrong axis",
     "const float v = fabsf((float)state[((int64_t)h * P + p) * N + n]);",
     "const float v = fabsf((float)state[((int64_t)h * P + (n % P)) * N + p % N]);"),
    ("codes truncated instead of rounded", "r = rintf((float)state[i] * rs);", "r = truncf((float)state[i] * rs);"),
    ("scale on a 128-step grid", "const float sc = amax / 127.0f;", "const float sc = amax / 128.0f;"),
    ("dequantised with the neighbouring channel's scale",
     "out[i] = (double)((float)q[i] * scale[(int64_t)h * N + n]);",
     "out[i] = (double)((float)q[i] * scale[(int64_t)h * N + (n + 1) % N]);"),
    # varlen prefill conv
    ("stored window used without an initial state", "for (int i = 0; i < Wc; ++i) stream[i] = has ? st[i] : 0.0;",
     "for (int i = 0; i < Wc; ++i) stream[i] = st[i];"),
    ("prefill conv window off by one",
     "for (int k = 0; k < W; ++k) v += w[(int64_t)c * W + k] * stream[Wc + q - (W - 1) + k];",
     "for (int k = 0; k < W; ++k) v += w[(int64_t)c * W + k] * stream[Wc + q - W + k];"),
    ("written-back window one input short", "for (int i = 0; i < Wc; ++i) st[i] = stream[L + i];",
     "for (int i = 0; i < Wc; ++i) st[i] = stream[L + i - (L > 0)];"),
    # Mamba1 (S6) step
    ("Mamba1 step shared by all channels",
     "const double delta = make_delta(dt[(int64_t)j * D + d], dt_bias, d, dt_softplus);",
     "const double delta = make_delta(dt[(int64_t)j * D + d], dt_bias, 0, dt_softplus);"),
    ("Mamba1 readout through B", "acc += Cm[(int64_t)j * N + n] * hrow[n];", "acc += Bm[(int64_t)j * N + n] * hrow[n];"),
    ("Mamba1 skip with one channel's D", "double yv = acc + (Dskip ? Dskip[d] * xv : 0.0);",
     "double yv = acc + (Dskip ? Dskip[0] * xv : 0.0);"),
]


def _copy_tree(dst):
    """The oracle, the pins and the input recipes (nothing of the CUDA library)."""
    os.makedirs(os.path.join(dst, "oracle"))
    for f in ("__init__.py", "mamba_oracle.c"):
        shutil.copy(os.path.join(ROOT, "oracle", f), os.path.join(dst, "oracle", f))
    os.makedirs(os.path.join(dst, "recurrent_state_update_gb300"))
    for f in ("__init__.py", "workloads.py"):
        shutil.copy(os.path.join(ROOT, "recurrent_state_update_gb300", f),
                    os.path.join(dst, "recurrent_state_update_gb300", f))
    os.makedirs(os.path.join(dst, "tests"))
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))


def _run_pins(dst):
    # the copy's own directory on the path; no conftest (it only registers the GPU marker and
    # would import torch in every one of these processes)
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1", PYTHONPATH=dst)
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-x", "-q", "-p", "no:cacheprovider",
                        "--noconftest"], cwd=dst, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout + r.stderr


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    """Pin-suite exit code and output for the unchanged copy and every planted mistake, run side
    by side in separate processes (each copy builds its own oracle library)."""
    cases = [("unchanged", None, None)] + MUTATIONS

    # the copies' directories are made here, one at a time (making numbered directories from
    # several threads at once races)
    dirs = [str(tmp_path_factory.mktemp("oracle_copy")) for _ in cases]

    def run(job):
        (what, old, new), dst = job
        _copy_tree(dst)
        if old is not None:
            src = os.path.join(dst, "oracle", "mamba_oracle.c")
            text = open(src).read()
            if old not in text:
                return None, f"the oracle no longer contains the expression this case changes: {old}"
            with open(src, "w") as f:
                f.write(text.replace(old, new, 1))
        return _run_pins(dst)

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        return dict(zip((c[0] for c in cases), ex.map(run, zip(cases, dirs))))


def test_unchanged_copy_passes_the_pins(outcomes):
    rc, out = outcomes["unchanged"]
    assert rc == 0, out[-2000:]


@pytest.mark.parametrize("what", [m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(outcomes, what):
    rc, out = outcomes[what]
    assert rc is not None, out
    # exit code 1: the suite ran and a pin failed (a build or collection error would be 2 or more);
    # a negative code: the changed oracle crashed inside a pin (an index now runs past a buffer)
    assert (rc == 1 and " failed" in out) or rc < 0, f"{what}: no pin failed\n{out[-2000:]}"
