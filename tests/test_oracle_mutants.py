"""The oracle's pins catch plausible mistakes (CPU only).

Each case copies the oracle package into a scratch directory, plants one
mistake in the copy's C source (a flipped sign, a dropped term, a wrong index, a
swapped operand, a broken state hand-off), and runs the pin file
tests/test_oracle_pins.py against that copy in a child process.  The pins must
fail for every planted mistake; the unmodified copy must pass, which shows the
child really loads the copy.  The repository's own oracle is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, original text, planted text); each original occurs exactly once in mamba_oracle.c
MUTANTS = [
    # Mamba-1 scan
    ("A sign", "A[n] = -exp(p->A_log[c * N + n]);", "A[n] = exp(p->A_log[c * N + n]);"),
    ("A_log ignores the channel", "A[n] = -exp(p->A_log[c * N + n]);", "A[n] = -exp(p->A_log[n]);"),
    ("decay without delta", "h[n] = exp(delta * A[n]) * h[n]", "h[n] = exp(A[n]) * h[n]"),
    ("input without delta", "+ delta * p->Bm[bc + n] * ut;", "+ p->Bm[bc + n] * ut;"),
    ("B read out instead of C", "yt += p->Cm[bc + n] * h[n];", "yt += p->Bm[bc + n] * h[n];"),
    ("D term dropped", "yt += Dc * ut;", "yt += 0.0 * Dc * ut;"),
    ("dt_bias dropped", "oracle_softplus(p->dt[idx] + bias);", "oracle_softplus(p->dt[idx]);"),
    ("gate without SiLU", "yt *= oracle_silu(p->z[idx]);", "yt *= p->z[idx];"),
    ("softplus without log1p", "+ log1p(exp(-a));", "+ log(exp(-a));"),
    ("SiLU sign", "return x / (1.0 + exp(-x));", "return x / (1.0 + exp(x));"),
    ("ssm step slab ignores batch", "double* slab = ssm_state + layer * B * Di * N;",
     "double* slab = ssm_state + layer * Di * N;"),
    # Mamba-1 conv
    ("conv taps reversed", "pre += p->w[c * K + k] * win[k];", "pre += p->w[c * K + (K - 1 - k)] * win[k];"),
    ("conv shift one slot short", "for (long k = 0; k + 1 < K; ++k) win[k] = win[k + 1];",
     "for (long k = 0; k + 2 < K; ++k) win[k] = win[k + 1];"),
    ("conv bias dropped", "double bias = p->bias ? p->bias[c] : 0.0;", "double bias = 0.0;"),
    ("conv state stored reversed", "p->state_out[(b * p->Di + c) * K + k] = win[k];",
     "p->state_out[(b * p->Di + c) * K + k] = win[K - 1 - k];"),
    ("conv step slab ignores batch", "double* slab = conv_state + layer * B * Di * K;",
     "double* slab = conv_state + layer * Di * K;"),
    # Mamba-3 SISO step
    ("m3 k and k_prev swapped", "be * kp * vp + g * k[bh * N + n] * xp;", "be * k[bh * N + n] * vp + g * kp * xp;"),
    ("m3 x in place of v_prev", "be * kp * vp + g", "be * kp * xp + g"),
    ("m3 read out with k", "acc += q[bh * N + n] * hrow[n];", "acc += k[bh * N + n] * hrow[n];"),
    ("m3 D term dropped", "y[bh * P + p] = acc + (D ? D[hd] : 0.0) * xp;", "y[bh * P + p] = acc;"),
    ("m3 k state takes q", "ks[bh * N + n] = k[bh * N + n];", "ks[bh * N + n] = q[bh * N + n];"),
    ("m3 v state not handed on", "vs[bh * P + p] = x[bh * P + p];", "vs[bh * P + p] = vs[bh * P + p];"),
    ("m3 alpha per head", "const double a = alpha[bh],", "const double a = alpha[hd],"),
    ("m3 k state slab ignores batch", "double* ks = k_state + layer * B * H * N;",
     "double* ks = k_state + layer * H * N;"),
    # Mamba-3 step inputs (angle state, rotation, trapezoid weights)
    ("m3 rotation by the old angle", "const double t = th[bh * n_angles + i];",
     "const double t = th[bh * n_angles + i] - d * angles[b * n_angles + i];"),
    ("m3 rotation sin sign", "k[e] = c * k_in[e] - s * k_in[o];", "k[e] = c * k_in[e] + s * k_in[o];"),
    ("m3 rotation pairs in halves", "const long e = bh * N + 2 * i, o = e + 1;",
     "const long e = bh * N + i, o = e + N / 2;"),
    ("m3 q not rotated", "q[e] = c * q_in[e] - s * q_in[o];\n                q[o] = s * q_in[e] + c * q_in[o];",
     "q[e] = q_in[e];\n                q[o] = q_in[o];"),
    ("m3 angle increment without dt", "th[bh * n_angles + i] += d * angles[b * n_angles + i];",
     "th[bh * n_angles + i] += angles[b * n_angles + i];"),
    ("m3 angles of batch row 0", "+= d * angles[b * n_angles + i];", "+= d * angles[i];"),
    ("m3 angle state slab ignores batch", "angle_state + layer * B * H * n_angles",
     "angle_state + layer * H * n_angles"),
    ("m3 beta without alpha", "beta[bh] = (1.0 - lam[bh]) * d * a;", "beta[bh] = (1.0 - lam[bh]) * d;"),
    ("m3 gamma decayed", "gamma[bh] = lam[bh] * d;", "gamma[bh] = lam[bh] * d * a;"),
    ("m3 trapezoid weights swapped", "gamma[bh] = lam[bh] * d;", "gamma[bh] = (1.0 - lam[bh]) * d;"),
    ("m3 alpha without dt", "const double a = exp(d * A[bh]);", "const double a = exp(A[bh]);"),
]


def _copy_oracle(dst):
    os.makedirs(os.path.join(dst, "oracle"))
    for f in ("__init__.py", "mamba_oracle.c", "mamba_oracle.h"):
        shutil.copy(os.path.join(ROOT, "oracle", f), os.path.join(dst, "oracle", f))
    return os.path.join(dst, "oracle", "mamba_oracle.c")


def _run_pins(workdir):
    """Run the pin file with `workdir`'s oracle first on the import path."""
    env = dict(os.environ, PYTHONPATH=os.pathsep.join([workdir, ROOT]), PYTHONDONTWRITEBYTECODE="1")
    probe = "import oracle, sys; sys.stdout.write(oracle.__file__)"
    where = subprocess.run([sys.executable, "-c", probe], cwd=workdir, env=env, capture_output=True, text=True)
    assert where.returncode == 0, where.stderr
    assert os.path.realpath(where.stdout).startswith(os.path.realpath(workdir)), where.stdout
    return subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider",
                           "--rootdir", workdir], cwd=workdir, env=env, capture_output=True, text=True,
                          timeout=300)


def test_unmodified_copy_passes_the_pins(tmp_path):
    _copy_oracle(str(tmp_path))
    r = _run_pins(str(tmp_path))
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(tmp_path, name, old, new):
    src = _copy_oracle(str(tmp_path))
    text = open(src).read()
    assert text.count(old) == 1, f"{name}: the original text must occur exactly once"
    with open(src, "w") as f:
        f.write(text.replace(old, new))
    r = _run_pins(str(tmp_path))
    assert r.returncode == 1 and " failed" in r.stdout, f"{name} survived the pins:\n{r.stdout[-1500:]}"
