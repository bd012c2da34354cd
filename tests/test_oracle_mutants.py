"""Plants plausible mistakes in a copy of the oracle's C source (on the CPU) and
checks that the pin suite catches every one of them.  The oracle itself is not
modified: each mutant is compiled from a patched temporary copy."""
import os
import subprocess

import numpy as np

import pytest

import oracle_pins
from oracle import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")

# (label, text in kda_oracle.c, replacement)
MUTANTS = [
    ("decay dropped", "S[(size_t)i * Dv + j] *= a;", "S[(size_t)i * Dv + j] *= 1.0;"),
    ("decay sign", "double a = exp(g[i]);", "double a = exp(-g[i]);"),
    ("retrieval error sign", "u[j] = v[j] - r;", "u[j] = v[j] + r;"),
    ("rank-1 update sign", "S[(size_t)i * Dv + j] += bk * u[j];", "S[(size_t)i * Dv + j] -= bk * u[j];"),
    ("beta dropped", "double bk = beta * kh[i];", "double bk = kh[i];"),
    ("output reads key", "r += S[(size_t)i * Dv + j] * qh[i];\n            o[j] = r;",
     "r += S[(size_t)i * Dv + j] * kh[i];\n            o[j] = r;"),
    ("retrieval on transposed state", "for (int i = 0; i < Dk; ++i) r += S[(size_t)i * Dv + j] * kh[i];\n        u[j]",
     "for (int i = 0; i < Dk; ++i) r += S[(size_t)j * Dv + i] * kh[i];\n        u[j]"),
    ("no normalisation", "double inv = 1.0 / sqrt(ss + KDA_ORACLE_EPS);", "double inv = 1.0;"),
    ("wrong eps", "#define KDA_ORACLE_EPS 1e-6", "#define KDA_ORACLE_EPS 1e-3"),
    ("first checkpoint skipped", "int64_t done = t - t0 + 1;\n                if (ckpt_stride > 0 && ckpts && done % ckpt_stride == 0) {",
     "int64_t done = t - t0 + 1;\n                if (ckpt_stride > 0 && ckpts && done % ckpt_stride == 0 && done > ckpt_stride) {"),
    ("initial state ignored", "if (init_state) memcpy(S, init_state + ((size_t)n * H + h) * SS, sizeof(double) * SS);\n            else memset(S, 0, sizeof(double) * SS);\n            int64_t t0 = cu_seqlens[n], t1",
     "memset(S, 0, sizeof(double) * SS);\n            int64_t t0 = cu_seqlens[n], t1"),
    ("chunked: Gram of decayed keys uses the wrong decay", "kk += Kg[(size_t)r * Dk + d] * Kd[(size_t)i * Dk + d];",
     "kk += Kg[(size_t)r * Dk + d] * Kg[(size_t)i * Dk + d];"),
    ("chunked: UT transform sign", "x -= Lm[(size_t)r * C + i] * Tm[(size_t)i * C + j];",
     "x += Lm[(size_t)r * C + i] * Tm[(size_t)i * C + j];"),
    ("chunked: causal matrix excludes diagonal", "Mc[(size_t)r * C + i] = (i <= r) ? qk : 0.0;",
     "Mc[(size_t)r * C + i] = (i < r) ? qk : 0.0;"),
    ("chunked: end-decay exponent sign", "exp(b[(size_t)(L - 1) * Dk + d] - b[(size_t)r * Dk + d]);",
     "exp(b[(size_t)r * Dk + d] - b[(size_t)(L - 1) * Dk + d]);"),
    ("chunked: state decay dropped", "double s = gl * S[(size_t)d * Dv + e];", "double s = S[(size_t)d * Dv + e];"),
    ("chunked: pseudo-value sign", "W[(size_t)r * Dv + e] = Uv[(size_t)r * Dv + e] - s;",
     "W[(size_t)r * Dv + e] = Uv[(size_t)r * Dv + e] + s;"),
    ("chunked: beta dropped in Wk", "s += Tm[(size_t)r * C + i] * beta[(size_t)(t0 + c0 + i) * H + h] * Kg[(size_t)i * Dk + d];",
     "s += Tm[(size_t)r * C + i] * Kg[(size_t)i * Dk + d];"),
    ("gdn: decay only on the old state", "S[ij] = al * (S[ij] - b * kh[i] * ktS[j]) + b * kh[i] * vv[j];",
     "S[ij] = al * S[ij] - b * kh[i] * ktS[j] + b * kh[i] * vv[j];"),
]


@pytest.mark.parametrize("label,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, label, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for '{label}' not unique/found"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", str(mut), "-o", str(so), "-lm"],
                   check=True)
    lib = oracle.load(str(so))
    res = oracle_pins.run_all(lib=lib)
    failed = [n for n, (_, _, ok) in res.items() if not ok]
    assert failed, f"mutant '{label}' passed every pin"


# Mistakes planted in the float64 prologue / epilogue functions (Python),
# each caught by at least one pin.
def _conv_reversed_taps(x, w, cu_seqlens=None, silu=False, history=None):
    return _orig_conv(x, np.asarray(w)[::-1].copy(), cu_seqlens, silu, history)


def _conv_crosses_sequences(x, w, cu_seqlens=None, silu=False, history=None):
    return _orig_conv(x, w, None, silu, None if history is None else history[:1])


def _conv_skips_current_token(x, w, cu_seqlens=None, silu=False, history=None):
    w = np.asarray(w, np.float64)
    shifted = np.concatenate([np.zeros_like(w[:1]), w[:-1]], 0)
    return _orig_conv(x, shifted, cu_seqlens, silu, history)


def _conv_wrong_activation(x, w, cu_seqlens=None, silu=False, history=None):
    y = _orig_conv(x, w, cu_seqlens, False, history)
    return y / (1.0 + np.exp(y)) if silu else y


def _conv_ignores_history(x, w, cu_seqlens=None, silu=False, history=None):
    return _orig_conv(x, w, cu_seqlens, silu, None)


def _tail_off_by_one(x, W, cu_seqlens=None, history=None):
    t = _orig_tail(x, W, cu_seqlens, history)
    return np.concatenate([t[:, :1], t[:, :-1]], 1)


def _gate_wrong_sign(o, z):
    return _orig_gate(o, -np.asarray(z, np.float64))


_orig_conv = oracle.short_conv
_orig_gate = oracle.output_gate
_orig_tail = oracle.conv_tail

PY_MUTANTS = [("conv taps reversed", "short_conv", _conv_reversed_taps),
              ("conv crosses sequence starts", "short_conv", _conv_crosses_sequences),
              ("conv skips the current token", "short_conv", _conv_skips_current_token),
              ("activation sigmoid(-x)", "short_conv", _conv_wrong_activation),
              ("gate sigmoid(-z)", "output_gate", _gate_wrong_sign),
              ("convolution history ignored", "short_conv", _conv_ignores_history),
              ("convolution state shifted by a row", "conv_tail", _tail_off_by_one)]


@pytest.mark.parametrize("label,name,fn", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_python_mutant_is_caught(monkeypatch, label, name, fn):
    monkeypatch.setattr(oracle, name, fn)
    res = oracle_pins.run_all()
    failed = [n for n, (_, _, ok) in res.items() if not ok]
    assert failed, f"mutant '{label}' passed every pin"
