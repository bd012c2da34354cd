"""Float64 CPU oracle for the Kimi Delta Attention core recurrence (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline / reference leg may import this module; the library under
``linear_attention_serving_k1_gb300`` never does.  It shares no code with the
CUDA path.  The arithmetic lives in ``kda_oracle.c`` (plain C, float64,
OpenMP over sequence x head); this file only compiles it with gcc and
marshals numpy arrays.

Sources: the page "Kimi K3 reconstructs long-context inference efficiency
through KDA, cross-depth attention, and latent expert routing", sections
"Methodology notes" (DeltaNet and Delta Rule; Kimi Delta Attention; FlashKDA)
and "Key data" (decode cost); the zsxq post on SemiAnalysis' Kimi K3 analysis,
sections "一、Kimi Delta Attention（KDA）" and "五、KV缓存效率与服务性能".

Parity status: every function here is pinned by tests/test_oracle_pins.py
(closed forms, invariants, special cases and an independent chunked
formulation); tests/test_oracle_mutants.py plants mistakes in a copy of the C
source and checks that the pins catch each one.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle with gcc into a shared object (rebuilt if stale)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    lib.oracle_prefill.restype = ctypes.c_int
    lib.oracle_prefill.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _i64p, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, _dp, _dp, ctypes.c_int, _dp,
                                   ctypes.c_int64]
    lib.oracle_prefill_chunked.restype = ctypes.c_int
    lib.oracle_prefill_chunked.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _i64p, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           _dp, _dp, ctypes.c_int, _dp, ctypes.c_int64]
    lib.oracle_decode.restype = None
    lib.oracle_decode.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_int]
    lib.oracle_gdn_prefill.restype = None
    lib.oracle_gdn_prefill.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _i64p, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, _dp, _dp]
    lib.oracle_ckpt_count.restype = ctypes.c_int64
    lib.oracle_ckpt_count.argtypes = [_i64p, ctypes.c_int, ctypes.c_int]
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    return lib


def load(path: str | None = None):
    """Load (compiling if needed) the oracle library.  ``path`` loads another build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(compile_oracle()))
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor -> numpy without importing torch here
        x = x.detach().cpu()
        if str(x.dtype) in ("torch.bfloat16", "torch.float16"):
            x = x.float()
        x = x.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def _cu(cu_seqlens, T):
    if cu_seqlens is None:
        return np.array([0, T], dtype=np.int64)
    if hasattr(cu_seqlens, "detach"):
        cu_seqlens = cu_seqlens.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))


def prefill(q, k, v, g, beta, init_state=None, cu_seqlens=None, ckpt_stride=0, lib=None,
            chunk=None):
    """Token-by-token (or, with ``chunk``, chunked) float64 prefill.

    q, k, g: [T, H, Dk]; v: [T, H, Dv]; beta: [T, H]; init_state: [N, H, Dk, Dv]
    or None (zeros); cu_seqlens: [N + 1] or None (one sequence of length T).
    Returns (out [T, H, Dv], final_state [N, H, Dk, Dv], ckpts [n_ckpt, H, Dk, Dv]).
    """
    lib = lib or load()
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    T, H, Dk = q.shape
    Dv = v.shape[2]
    cu = _cu(cu_seqlens, T)
    N = cu.shape[0] - 1
    s0 = _f64(init_state)
    out = np.zeros((T, H, Dv), np.float64)
    fin = np.zeros((N, H, Dk, Dv), np.float64)
    nck = int(lib.oracle_ckpt_count(cu.ctypes.data_as(_i64p), N, int(ckpt_stride)))
    ck = np.zeros((max(nck, 1), H, Dk, Dv), np.float64)
    if chunk is None:
        rc = lib.oracle_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(s0),
                                cu.ctypes.data_as(_i64p), N, H, Dk, Dv, _ptr(out), _ptr(fin),
                                int(ckpt_stride), _ptr(ck), nck)
    else:
        rc = lib.oracle_prefill_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(s0),
                                        cu.ctypes.data_as(_i64p), N, H, Dk, Dv, int(chunk),
                                        _ptr(out), _ptr(fin), int(ckpt_stride), _ptr(ck), nck)
    if rc != 0:
        raise ValueError(f"oracle prefill failed with code {rc}")
    return out, fin, ck[:nck]


def prefill_heads(q, k, v, g, beta, init_state=None, cu_seqlens=None, ckpt_stride=0, heads=None):
    """Prefill restricted to a subset of heads (heads are independent chains).

    Returns the same triple as ``prefill`` with the head axis reduced to ``heads``.
    """
    if heads is None:
        return prefill(q, k, v, g, beta, init_state, cu_seqlens, ckpt_stride)
    idx = list(heads)

    def sel(x, axis):
        if x is None:
            return None
        x = _f64(x)
        return np.ascontiguousarray(np.take(x, idx, axis=axis))

    return prefill(sel(q, 1), sel(k, 1), sel(v, 1), sel(g, 1), sel(beta, 1),
                   sel(init_state, 1), cu_seqlens, ckpt_stride)


def decode(q, k, v, g, beta, state, lib=None):
    """One decode step.  q, k, g: [N, H, Dk]; v: [N, H, Dv]; beta: [N, H];
    state: [N, H, Dk, Dv].  Returns (out [N, H, Dv], new_state) without
    modifying the argument."""
    lib = lib or load()
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    N, H, Dk = q.shape
    Dv = v.shape[2]
    st = np.array(_f64(state), dtype=np.float64, copy=True)
    out = np.zeros((N, H, Dv), np.float64)
    lib.oracle_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(st), _ptr(out),
                      N, H, Dk, Dv)
    return out, st


def gdn_prefill(q, k, v, a, beta, init_state=None, cu_seqlens=None, lib=None):
    """Scalar-gate Gated DeltaNet prefill; a: [T, H] log-decay."""
    lib = lib or load()
    q, k, v, a, beta = (_f64(x) for x in (q, k, v, a, beta))
    T, H, Dk = q.shape
    Dv = v.shape[2]
    cu = _cu(cu_seqlens, T)
    N = cu.shape[0] - 1
    s0 = _f64(init_state)
    out = np.zeros((T, H, Dv), np.float64)
    fin = np.zeros((N, H, Dk, Dv), np.float64)
    lib.oracle_gdn_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(a), _ptr(beta), _ptr(s0),
                           cu.ctypes.data_as(_i64p), N, H, Dk, Dv, _ptr(out), _ptr(fin))
    return out, fin


def short_conv(x, w, cu_seqlens=None, silu=False, history=None):
    """Causal depthwise short convolution along time, inside each sequence.

    x: [T, H, D]; w: [W, H, D] taps; cu_seqlens: [N + 1] token offsets (None:
    one sequence).  For token t of a sequence starting at s:
        y[t] = sum_{i < W} w[i] * x[t - (W - 1) + i]
    with x[tau] for tau < s taken from ``history`` [N, W - 1, H, D] (the W - 1
    rows before the sequence, oldest first; None: zeros), so nothing crosses
    into another sequence (tap W - 1 multiplies the current token), then
    y * sigmoid(y) when ``silu``.  float64 throughout.

    Source: "Kimi K3 reconstructs long-context inference efficiency through
    KDA, cross-depth attention, and latent expert routing", section
    "Methodology notes", item "Memory control: Kimi Delta Attention" (KDA
    combines a short convolution with the L2-normalised q/k and an output
    forget gate); width, causality and activation are readings, the pages
    give none.
    """
    x = _f64(x)
    w = _f64(w)
    T = x.shape[0]
    W = w.shape[0]
    cu = _cu(cu_seqlens, T)
    y = np.zeros_like(x)
    hist = None if history is None else _f64(history)
    for n in range(cu.shape[0] - 1):
        s, e = int(cu[n]), int(cu[n + 1])
        for t in range(s, e):
            for i in range(W):
                tau = t - (W - 1) + i
                if tau >= s:
                    y[t] += w[i] * x[tau]
                elif hist is not None:
                    y[t] += w[i] * hist[n, (W - 1) + (tau - s)]
    if silu:
        y = y / (1.0 + np.exp(-y))
    return y


def conv_tail(x, W, cu_seqlens=None, history=None):
    """The convolution state after each sequence: its last W - 1 input rows
    (oldest first) [N, W - 1, H, D], reaching into ``history`` (or zeros) when
    the sequence is shorter."""
    x = _f64(x)
    T, H, D = x.shape
    cu = _cu(cu_seqlens, T)
    N = cu.shape[0] - 1
    hist = np.zeros((N, W - 1, H, D)) if history is None else _f64(history)
    out = np.zeros((N, W - 1, H, D))
    for n in range(N):
        s, e = int(cu[n]), int(cu[n + 1])
        seq = np.concatenate([hist[n], x[s:e]], 0)
        out[n] = seq[seq.shape[0] - (W - 1):]
    return out


def output_gate(o, z):
    """The output forget gate read as an elementwise sigmoid gate:
    out = o * sigmoid(z) (same shapes; float64).  Source: the page named in
    ``short_conv``, same item; the gate's form is a reading."""
    o = _f64(o)
    z = _f64(z)
    return o / (1.0 + np.exp(-z))


def prefill_fused(q, k, v, g, beta, init_state=None, cu_seqlens=None, ckpt_stride=0, conv_w=None,
                  silu=False, gate=None, conv_state=None, return_conv_state=False, lib=None):
    """The prefill with the steps around the recurrence: q, k, v pass through
    ``short_conv`` (taps conv_w [3, W, H, D] for q, k, v; None: none; history
    ``conv_state`` [N, 3, W - 1, H, D] or None for zeros) before the
    recurrence, and its output through ``output_gate`` (gate [T, H, Dv];
    None: none).  Returns (out, final_state, ckpts) like ``prefill``, and with
    ``return_conv_state`` also the convolution state after each sequence
    ([N, 3, W - 1, H, D], ``conv_tail``) as a fourth element."""
    tails = None
    if conv_w is not None:
        conv_w = _f64(conv_w)
        W = conv_w.shape[1]
        hist = [None] * 3 if conv_state is None else [_f64(conv_state)[:, t] for t in range(3)]
        tails = np.stack([conv_tail(x, W, cu_seqlens, hist[t]) for t, x in enumerate((q, k, v))], 1)
        q = short_conv(q, conv_w[0], cu_seqlens, silu, hist[0])
        k = short_conv(k, conv_w[1], cu_seqlens, silu, hist[1])
        v = short_conv(v, conv_w[2], cu_seqlens, silu, hist[2])
    o, f, ck = prefill(q, k, v, g, beta, init_state, cu_seqlens, ckpt_stride, lib=lib)
    if gate is not None:
        o = output_gate(o, gate)
    if return_conv_state:
        return o, f, ck, tails
    return o, f, ck


def decode_fused(q, k, v, g, beta, state, conv_w=None, silu=False, gate=None, conv_state=None, lib=None):
    """One decode step with the steps around the recurrence: each sequence's
    new q, k, v ([N, H, D]) are convolved with its history ``conv_state``
    [N, 3, W - 1, H, D] (None: zeros), the step runs as ``decode`` and the
    output is gated.  Returns (out, new_state, new_conv_state or None)."""
    new_cs = None
    if conv_w is not None:
        conv_w = _f64(conv_w)
        W = conv_w.shape[1]
        N, H, D = q.shape
        cs = np.zeros((N, 3, W - 1, H, D)) if conv_state is None else _f64(conv_state)
        xs = []
        for t, x in enumerate((q, k, v)):
            x = _f64(x)
            rows = np.concatenate([cs[:, t], x[:, None]], 1)          # [N, W, H, D], oldest first
            y = np.einsum("nwhd,whd->nhd", rows, conv_w[t])
            xs.append(y / (1.0 + np.exp(-y)) if silu else y)
        new_cs = np.stack([np.concatenate([cs[:, t], _f64(x)[:, None]], 1)[:, 1:]
                           for t, x in enumerate((q, k, v))], 1)
        q, k, v = xs
    o, st = decode(q, k, v, g, beta, state, lib=lib)
    if gate is not None:
        o = output_gate(o, gate)
    return o, st, new_cs


def num_threads(lib=None) -> int:
    lib = lib or load()
    return int(lib.oracle_num_threads())
