"""Pins for the float64 oracle: facts fixed by the KDA pages and by mathematics.

Each pin runs the oracle (optionally a given build of it, ``lib``) on small
seeded inputs and returns the largest violation it finds (0 = exact).  None of
them re-types the recurrence: they use closed forms of special cases, an
independent arrangement (Gated DeltaNet), an independent algorithm (the
chunked UT-transform form), a finite-difference gradient of the retrieval
loss, and structural invariants (continuation, resume, linearity, column and
sequence independence, non-expansion).

Sources: "Kimi K3 reconstructs long-context inference efficiency through KDA,
cross-depth attention, and latent expert routing", section "Methodology
notes" (the Delta Rule minimises the L2 value-retrieval error; KDA's forgetting
factor is a diagonal matrix; q and k are L2-normalised; FlashKDA unrolls the
recurrence by blocks) and section "Key data" (linear prefill, constant decode);
the zsxq post on SemiAnalysis' Kimi K3 analysis, section
"一、Kimi Delta Attention（KDA）" (GDN's scalar forget gate alpha; the UT
transform) and section "五、KV缓存效率与服务性能" (state snapshots every 32K
tokens and at prompt boundaries).
"""
from __future__ import annotations

import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
from oracle import oracle  # noqa: E402

EPS = 1e-6  # the reading of the L2-norm epsilon (the pages give none)


def _rng(seed):
    return np.random.default_rng(seed)


def _inputs(rng, T, H, Dk, Dv, g_scale=1.0, beta=None):
    q = rng.standard_normal((T, H, Dk))
    k = rng.standard_normal((T, H, Dk))
    v = rng.standard_normal((T, H, Dv))
    g = -np.exp(rng.uniform(-5, -1, (T, H, Dk))) * g_scale
    b = 1 / (1 + np.exp(-rng.standard_normal((T, H)))) if beta is None else beta
    return q, k, v, g, b


def _unit(x):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + EPS)


def pin_beta0_g0_identity(lib=None, seed=1):
    """beta = 0, g = 0: S never changes and o_t = S0^T qhat_t."""
    rng = _rng(seed)
    T, H, Dk, Dv = 9, 2, 5, 7
    q, k, v, g, b = _inputs(rng, T, H, Dk, Dv)
    g[:] = 0
    b = np.zeros((T, H))
    s0 = rng.standard_normal((1, H, Dk, Dv))
    o, f, _ = oracle.prefill(q, k, v, g, b, s0, lib=lib)
    want = np.einsum("hkv,thk->thv", s0[0], _unit(q))
    return max(np.abs(f - s0).max(), np.abs(o - want).max())


def pin_beta0_decay_closed_form(lib=None, seed=2):
    """beta = 0: S_t = Diag(exp sum_{s<=t} g_s) S0, applied to the key rows."""
    rng = _rng(seed)
    T, H, Dk, Dv = 11, 2, 6, 9
    q, k, v, g, _ = _inputs(rng, T, H, Dk, Dv)
    b = np.zeros((T, H))
    s0 = rng.standard_normal((1, H, Dk, Dv))
    o, f, _ = oracle.prefill(q, k, v, g, b, s0, lib=lib)
    cg = np.cumsum(g, axis=0)                       # [T, H, Dk]
    St = np.exp(cg)[..., None] * s0[0][None]        # [T, H, Dk, Dv]
    want_o = np.einsum("thkv,thk->thv", St, _unit(q))
    return max(np.abs(f[0] - St[-1]).max(), np.abs(o - want_o).max())


def pin_retrieval_exact(lib=None, seed=3):
    """Delta rule: with beta * |khat|^2 = 1 the updated state retrieves v_t
    exactly from k_t, whatever the decay: S_t^T khat_t = v_t."""
    rng = _rng(seed)
    T, H, Dk, Dv = 12, 2, 8, 5
    q, k, v, g, _ = _inputs(rng, T, H, Dk, Dv)
    k *= rng.uniform(0.5, 3.0, (T, H, 1))
    nk = (k * k).sum(-1)
    b = (nk + EPS) / nk                               # beta * |khat|^2 == 1
    s0 = rng.standard_normal((1, H, Dk, Dv))
    _, _, ck = oracle.prefill(q, k, v, g, b, s0, ckpt_stride=1, lib=lib)
    if ck.shape[0] != T:
        return np.inf
    got = np.einsum("thkv,thk->thv", ck, _unit(k))
    return np.abs(got - v).max()


def pin_orthogonal_complement_untouched(lib=None, seed=4):
    """The update only moves the state along khat: for x orthogonal to khat_t,
    x^T S_t = x^T Diag(alpha_t) S_{t-1}."""
    rng = _rng(seed)
    T, H, D = 10, 2, 6
    q, k, v, g, b = _inputs(rng, T, H, D, D)
    s0 = rng.standard_normal((1, H, D, D))
    _, _, ck = oracle.prefill(q, k, v, g, b, s0, ckpt_stride=1, lib=lib)
    if ck.shape[0] != T:
        return np.inf
    prev = np.concatenate([s0, ck[:-1]], 0)          # S_{t-1}
    worst = 0.0
    for t in range(T):
        for h in range(H):
            kh = k[t, h] / np.linalg.norm(k[t, h])
            x = rng.standard_normal(D)
            x -= (x @ kh) * kh                         # x orthogonal to k
            lhs = x @ ck[t, h]
            rhs = x @ (np.exp(g[t, h])[:, None] * prev[t, h])
            worst = max(worst, np.abs(lhs - rhs).max())
    return worst


def pin_replacement_memory(lib=None, seed=5):
    """g = 0, beta*|khat|^2 = 1, k_t = e_{t mod Dk}: row i of S is erased and
    replaced by v_t / |khat| for the last token whose key was e_i (khat =
    e_i / sqrt(1 + eps)); untouched rows keep S0."""
    rng = _rng(seed)
    T, H, Dk, Dv = 7, 1, 4, 3
    q, _, v, _, _ = _inputs(rng, T, H, Dk, Dv)
    k = np.zeros((T, H, Dk))
    for t in range(T):
        k[t, 0, t % Dk] = 1.0
    g = np.zeros((T, H, Dk))
    b = np.full((T, H), 1.0 + EPS)
    s0 = rng.standard_normal((1, H, Dk, Dv))
    _, f, _ = oracle.prefill(q, k, v, g, b, s0, lib=lib)
    want = s0[0, 0].copy()
    for t in range(T):
        want[int(np.argmax(k[t, 0]))] = v[t, 0] * np.sqrt(1.0 + EPS)
    return np.abs(f[0, 0] - want).max()


def pin_output_reads_updated_state(lib=None, seed=6):
    """T = 1 from a zero state: o_1 = beta (khat . qhat) v_1 (the output reads
    the state after the update, with no extra scale)."""
    rng = _rng(seed)
    H, Dk, Dv = 3, 5, 4
    q, k, v, g, b = _inputs(rng, 1, H, Dk, Dv)
    o, _, _ = oracle.prefill(q, k, v, g, b, None, lib=lib)
    want = (b[0] * (_unit(k[0]) * _unit(q[0])).sum(-1))[:, None] * v[0]
    return np.abs(o[0] - want).max()


def pin_delta_is_gradient_step(lib=None, seed=7):
    """One token from S0: S_1 = S' - beta * grad_S 0.5 |S^T khat - v|^2 at
    S' = Diag(alpha) S0, the gradient taken by central finite differences."""
    rng = _rng(seed)
    Dk, Dv = 3, 2
    q, k, v, g, b = _inputs(rng, 1, 1, Dk, Dv)
    s0 = rng.standard_normal((1, 1, Dk, Dv))
    _, f, _ = oracle.prefill(q, k, v, g, b, s0, lib=lib)
    Sp = np.exp(g[0, 0])[:, None] * s0[0, 0]
    kh = _unit(k[0, 0])

    def loss(S):
        r = S.T @ kh - v[0, 0]
        return 0.5 * float(r @ r)

    grad = np.zeros_like(Sp)
    hstep = 1e-5
    for i in range(Dk):
        for j in range(Dv):
            e = np.zeros_like(Sp)
            e[i, j] = hstep
            grad[i, j] = (loss(Sp + e) - loss(Sp - e)) / (2 * hstep)
    want = Sp - b[0, 0] * grad
    return np.abs(f[0, 0] - want).max()


def pin_gated_deltanet(lib=None, seed=8):
    """g constant over channels reduces KDA to Gated DeltaNet (scalar alpha),
    computed by an independent arrangement alpha (I - beta k k^T) S + beta k v^T."""
    rng = _rng(seed)
    T, H, D = 40, 2, 8
    q, k, v, _, b = _inputs(rng, T, H, D, D)
    a = -np.exp(rng.uniform(-5, -1, (T, H)))
    g = np.repeat(a[..., None], D, axis=-1)
    s0 = rng.standard_normal((1, H, D, D))
    o1, f1, _ = oracle.prefill(q, k, v, g, b, s0, lib=lib)
    o2, f2 = oracle.gdn_prefill(q, k, v, a, b, s0, lib=lib)
    return max(np.abs(o1 - o2).max(), np.abs(f1 - f2).max())


def pin_chunked_equals_recurrence(lib=None, seed=9):
    """The UT-transform chunked form equals the token recurrence (ragged
    lengths, partial last chunks, C in {1, 4, 16, 64}, checkpoints)."""
    rng = _rng(seed)
    lens = [1, 63, 64, 65, 130]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, D = int(cu[-1]), 2, 16
    q, k, v, g, b = _inputs(rng, T, H, D, D)
    s0 = rng.standard_normal((len(lens), H, D, D)) * 0.1
    o, f, ck = oracle.prefill(q, k, v, g, b, s0, cu, ckpt_stride=64, lib=lib)
    worst = 0.0
    for C in (1, 4, 16, 64):
        o2, f2, ck2 = oracle.prefill(q, k, v, g, b, s0, cu, ckpt_stride=64, lib=lib, chunk=C)
        if ck2.shape != ck.shape:
            return np.inf
        worst = max(worst, np.abs(o - o2).max(), np.abs(f - f2).max(), np.abs(ck - ck2).max())
    return worst


def pin_decode_continues_prefill(lib=None, seed=10):
    """prefill over t tokens, then one decode step on token t+1, equals prefill
    over t+1 tokens (output of that token and final state)."""
    rng = _rng(seed)
    T, H, D = 25, 3, 8
    q, k, v, g, b = _inputs(rng, T, H, D, D)
    s0 = rng.standard_normal((1, H, D, D)) * 0.1
    o, f, _ = oracle.prefill(q, k, v, g, b, s0, lib=lib)
    _, fp, _ = oracle.prefill(q[:-1], k[:-1], v[:-1], g[:-1], b[:-1], s0, lib=lib)
    od, sd = oracle.decode(q[-1:], k[-1:], v[-1:], g[-1:], b[-1:], fp, lib=lib)
    return max(np.abs(od[0] - o[-1]).max(), np.abs(sd - f).max())


def pin_linearity(lib=None, seed=11):
    """For fixed q, k, g, beta the map (S0, V) -> (O, S_T) is linear."""
    rng = _rng(seed)
    T, H, D = 30, 2, 6
    q, k, v1, g, b = _inputs(rng, T, H, D, D)
    v2 = rng.standard_normal(v1.shape)
    s0 = rng.standard_normal((1, H, D, D))
    oa, fa, _ = oracle.prefill(q, k, v1, g, b, s0, lib=lib)
    ob, fb, _ = oracle.prefill(q, k, v2, g, b, None, lib=lib)
    oc, fc, _ = oracle.prefill(q, k, 2.0 * v1 + 3.0 * v2, g, b, 2.0 * s0, lib=lib)
    return max(np.abs(2 * oa + 3 * ob - oc).max(), np.abs(2 * fa + 3 * fb - fc).max())


def pin_value_columns_independent(lib=None, seed=12):
    """Value columns evolve independently: running on a block of v's columns
    (and the matching state columns) reproduces those columns."""
    rng = _rng(seed)
    T, H, Dk, Dv = 20, 2, 6, 8
    q, k, v, g, b = _inputs(rng, T, H, Dk, Dv)
    s0 = rng.standard_normal((1, H, Dk, Dv))
    o, f, _ = oracle.prefill(q, k, v, g, b, s0, lib=lib)
    o2, f2, _ = oracle.prefill(q, k, v[..., 2:5], g, b, s0[..., 2:5], lib=lib)
    return max(np.abs(o[..., 2:5] - o2).max(), np.abs(f[..., 2:5] - f2).max())


def pin_sequences_independent(lib=None, seed=13):
    """Packed sequences restart from their own initial state: a packed run equals
    running each sequence alone; an empty sequence returns its initial state."""
    rng = _rng(seed)
    lens = [5, 0, 17, 1]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, D = int(cu[-1]), 2, 5
    q, k, v, g, b = _inputs(rng, T, H, D, D)
    s0 = rng.standard_normal((len(lens), H, D, D))
    o, f, _ = oracle.prefill(q, k, v, g, b, s0, cu, lib=lib)
    worst = 0.0
    for n, L in enumerate(lens):
        a, z = cu[n], cu[n + 1]
        if L == 0:
            worst = max(worst, np.abs(f[n] - s0[n]).max())
            continue
        on, fn, _ = oracle.prefill(q[a:z], k[a:z], v[a:z], g[a:z], b[a:z], s0[n:n + 1], lib=lib)
        worst = max(worst, np.abs(o[a:z] - on).max(), np.abs(f[n] - fn[0]).max())
    return worst


def pin_checkpoint_resume(lib=None, seed=14):
    """Snapshot j of sequence n is the state after its first j*stride tokens
    (ordered by sequence, then j); resuming from a snapshot reproduces the rest."""
    rng = _rng(seed)
    lens = [40, 9, 33]
    stride = 8
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, D = int(cu[-1]), 2, 4
    q, k, v, g, b = _inputs(rng, T, H, D, D)
    s0 = rng.standard_normal((len(lens), H, D, D))
    o, f, ck = oracle.prefill(q, k, v, g, b, s0, cu, ckpt_stride=stride, lib=lib)
    want_n = sum(L // stride for L in lens)
    if ck.shape[0] != want_n:
        return np.inf
    worst, slot = 0.0, 0
    for n, L in enumerate(lens):
        a = cu[n]
        for j in range(1, L // stride + 1):
            z = a + j * stride
            _, fj, _ = oracle.prefill(q[a:z], k[a:z], v[a:z], g[a:z], b[a:z], s0[n:n + 1], lib=lib)
            worst = max(worst, np.abs(ck[slot] - fj[0]).max())
            z2 = cu[n + 1]
            orr, fr, _ = oracle.prefill(q[z:z2], k[z:z2], v[z:z2], g[z:z2], b[z:z2],
                                        ck[slot:slot + 1], lib=lib)
            if z2 > z:
                worst = max(worst, np.abs(orr - o[z:z2]).max())
            worst = max(worst, np.abs(fr[0] - f[n]).max())
            slot += 1
    return worst


def pin_non_expansive(lib=None, seed=15):
    """With v = 0, beta in [0, 2] and g <= 0 each step is a product of
    contractions: |S_t|_F never increases.  Returns the largest increase."""
    rng = _rng(seed)
    T, H, D = 50, 2, 6
    q, k, _, g, _ = _inputs(rng, T, H, D, D)
    v = np.zeros((T, H, D))
    b = rng.uniform(0, 2, (T, H))
    s0 = rng.standard_normal((1, H, D, D))
    _, _, ck = oracle.prefill(q, k, v, g, b, s0, ckpt_stride=1, lib=lib)
    if ck.shape[0] != T:
        return np.inf
    norms = np.concatenate([np.linalg.norm(s0, axis=(2, 3)), np.linalg.norm(ck, axis=(2, 3))], 0)
    inc = np.diff(norms, axis=0).max()
    # a decay that does nothing (alpha=1) would not shrink: demand strict shrink overall
    shrink = norms[-1] / norms[0]
    return max(0.0, inc) + (np.inf if np.any(shrink > 0.999) else 0.0)


def pin_qk_scale_invariance(lib=None, seed=16):
    """q and k enter only through their directions (L2 normalisation): scaling
    them by positive factors leaves outputs and states unchanged (up to eps)."""
    rng = _rng(seed)
    T, H, D = 15, 2, 6
    q, k, v, g, b = _inputs(rng, T, H, D, D)
    s0 = rng.standard_normal((1, H, D, D))
    o, f, _ = oracle.prefill(q, k, v, g, b, s0, lib=lib)
    o2, f2, _ = oracle.prefill(q * 7.0, k * 0.25, v, g, b, s0, lib=lib)
    return max(np.abs(o - o2).max(), np.abs(f - f2).max())


def pin_decode_heads_match_prefill_T1(lib=None, seed=17):
    """Decode over N sequences x H heads equals a one-token prefill of each."""
    rng = _rng(seed)
    N, H, D = 3, 2, 5
    q, k, v, g, b = _inputs(rng, N, H, D, D)
    st = rng.standard_normal((N, H, D, D))
    od, sd = oracle.decode(q, k, v, g, b, st, lib=lib)
    worst = 0.0
    for n in range(N):
        o, f, _ = oracle.prefill(q[n:n + 1], k[n:n + 1], v[n:n + 1], g[n:n + 1], b[n:n + 1],
                                 st[n:n + 1], lib=lib)
        worst = max(worst, np.abs(od[n] - o[0]).max(), np.abs(sd[n] - f[0]).max())
    return worst


# ---------------------------------------------------------------- prologue / epilogue
# The short convolution and the output gate (page "Kimi K3 reconstructs ...",
# section "Methodology notes", item "Memory control: Kimi Delta Attention").
def pin_conv_identity_tap(lib=None, seed=18):
    """Taps (0, .., 0, 1) without activation pass the inputs through unchanged,
    and the fused prefill then equals the plain one exactly."""
    rng = _rng(seed)
    T, H, D = 23, 2, 6
    q, k, v, g, b = _inputs(rng, T, H, D, D)
    cu = np.array([0, 9, 9, 23])
    w = np.zeros((3, 4, H, D))
    w[:, 3] = 1.0
    worst = np.abs(oracle.short_conv(q, w[0], cu) - q).max()
    o1, f1, _ = oracle.prefill_fused(q, k, v, g, b, None, cu, conv_w=w, lib=lib)
    o2, f2, _ = oracle.prefill(q, k, v, g, b, None, cu, lib=lib)
    return max(worst, np.abs(o1 - o2).max(), np.abs(f1 - f2).max())


def pin_conv_matches_library(lib=None, seed=19):
    """Per sequence and channel, the causal convolution is numpy's full
    convolution with the reversed taps, cut to the sequence length."""
    rng = _rng(seed)
    T, H, D, W = 30, 2, 3, 4
    x = rng.standard_normal((T, H, D))
    w = rng.standard_normal((W, H, D))
    cu = np.array([0, 2, 17, 30])
    y = oracle.short_conv(x, w, cu)
    worst = 0.0
    for n in range(3):
        s, e = cu[n], cu[n + 1]
        for h in range(H):
            for d in range(D):
                ref = np.convolve(x[s:e, h, d], w[::-1, h, d], mode="full")[: e - s]
                worst = max(worst, np.abs(y[s:e, h, d] - ref).max())
    return worst


def pin_conv_stays_in_sequence(lib=None, seed=20):
    """An impulse at the last token of one sequence leaves the next sequence
    at zero, and one at a sequence's first token touches nothing before it."""
    rng = _rng(seed)
    T, H, D, W = 12, 1, 2, 4
    w = rng.standard_normal((W, H, D))
    cu = np.array([0, 5, 12])
    worst = 0.0
    for pos, zero in ((4, slice(5, 12)), (5, slice(0, 5))):
        x = np.zeros((T, H, D))
        x[pos] = 1.0
        y = oracle.short_conv(x, w, cu)
        worst = max(worst, np.abs(y[zero]).max())
        # and inside its own sequence the impulse response is the taps, newest first
        s_end = 5 if pos < 5 else 12
        for j in range(min(W, s_end - pos)):
            worst = max(worst, np.abs(y[pos + j] - w[W - 1 - j]).max())
    return worst


def pin_conv_history_continues(lib=None, seed=23):
    """A sequence convolved in two parts, the second seeded with the first's
    last W - 1 inputs, gives the whole sequence's convolution; and the fused
    prefill of the parts (state and convolution state handed on) reproduces
    the fused prefill of the whole."""
    rng = _rng(seed)
    T, H, D, W, cut = 19, 2, 4, 4, 7
    q, k, v, g, b = _inputs(rng, T, H, D, D)
    w = rng.standard_normal((3, W, H, D))
    worst = 0.0
    whole = oracle.short_conv(q, w[0])
    tail = oracle.conv_tail(q[:cut], W)
    second = oracle.short_conv(q[cut:], w[0], history=tail)
    worst = max(worst, np.abs(whole[cut:] - second).max())
    o, f, _, cs = oracle.prefill_fused(q, k, v, g, b, conv_w=w, silu=True, return_conv_state=True, lib=lib)
    o1, f1, _, cs1 = oracle.prefill_fused(q[:cut], k[:cut], v[:cut], g[:cut], b[:cut], conv_w=w, silu=True,
                                          return_conv_state=True, lib=lib)
    o2, f2, _, cs2 = oracle.prefill_fused(q[cut:], k[cut:], v[cut:], g[cut:], b[cut:], f1, conv_w=w, silu=True,
                                          conv_state=cs1, return_conv_state=True, lib=lib)
    worst = max(worst, np.abs(o[cut:] - o2).max(), np.abs(f - f2).max(), np.abs(cs - cs2).max())
    # the convolution state is the raw input rows themselves
    worst = max(worst, np.abs(cs[0, 0] - q[T - (W - 1):]).max(), np.abs(cs[0, 2] - v[T - (W - 1):]).max())
    return worst


def pin_decode_fused_continues_prefill(lib=None, seed=24):
    """prefill_fused over t tokens, then decode_fused on token t + 1 with the
    handed-on state and convolution state, equals prefill_fused over t + 1
    tokens (its last output, final state and convolution state)."""
    rng = _rng(seed)
    T, H, D, W = 11, 2, 5, 3
    q, k, v, g, b = _inputs(rng, T, H, D, D)
    w = rng.standard_normal((3, W, H, D))
    z = rng.standard_normal((T, H, D))
    s0 = rng.standard_normal((1, H, D, D)) * 0.1
    o, f, _, cs = oracle.prefill_fused(q, k, v, g, b, s0, conv_w=w, gate=z, return_conv_state=True, lib=lib)
    _, fp, _, csp = oracle.prefill_fused(q[:-1], k[:-1], v[:-1], g[:-1], b[:-1], s0, conv_w=w, gate=z[:-1],
                                         return_conv_state=True, lib=lib)
    od, sd, csd = oracle.decode_fused(q[-1:], k[-1:], v[-1:], g[-1:], b[-1:], fp, conv_w=w, gate=z[-1:],
                                      conv_state=csp, lib=lib)
    return max(np.abs(od[0] - o[-1]).max(), np.abs(sd - f).max(), np.abs(csd - cs).max())


def pin_silu_closed_form(lib=None, seed=21):
    """With pass-through taps, the activation is x sigmoid(x): 0 at 0,
    (3/4) ln 3 at ln 3 and -(1/4) ln 3 at -ln 3 (sigmoid(ln 3) = 3/4)."""
    l3 = np.log(3.0)
    x = np.array([0.0, l3, -l3]).reshape(3, 1, 1)
    w = np.ones((1, 1, 1))
    y = oracle.short_conv(x, w, None, silu=True).ravel()
    return np.abs(y - np.array([0.0, 0.75 * l3, -0.25 * l3])).max()


def pin_output_gate_values(lib=None, seed=22):
    """sigmoid(0) = 1/2, sigmoid(+-ln 3) = 3/4, 1/4 and sigmoid(60) = 1 to
    double precision: the gate halves, scales by 3/4 and 1/4, or passes o."""
    rng = _rng(seed)
    o = rng.standard_normal((4, 2, 3))
    l3 = np.log(3.0)
    z = np.broadcast_to(np.array([0.0, l3, -l3, 60.0]).reshape(4, 1, 1), o.shape)
    want = o * np.array([0.5, 0.75, 0.25, 1.0]).reshape(4, 1, 1)
    return np.abs(oracle.output_gate(o, z) - want).max()


# name -> (pin, bar).  Bars: 1e-12 where the identity is exact in float64
# arithmetic up to rounding; looser where a finite difference or eps enters.
PINS = {
    "beta0_g0_identity": (pin_beta0_g0_identity, 1e-12),
    "beta0_decay_closed_form": (pin_beta0_decay_closed_form, 1e-12),
    "retrieval_exact": (pin_retrieval_exact, 1e-11),
    "orthogonal_complement_untouched": (pin_orthogonal_complement_untouched, 1e-11),
    "replacement_memory": (pin_replacement_memory, 1e-12),
    "output_reads_updated_state": (pin_output_reads_updated_state, 1e-12),
    "delta_is_gradient_step": (pin_delta_is_gradient_step, 1e-8),
    "gated_deltanet": (pin_gated_deltanet, 1e-11),
    "chunked_equals_recurrence": (pin_chunked_equals_recurrence, 1e-10),
    "decode_continues_prefill": (pin_decode_continues_prefill, 1e-12),
    "linearity": (pin_linearity, 1e-10),
    "value_columns_independent": (pin_value_columns_independent, 1e-12),
    "sequences_independent": (pin_sequences_independent, 1e-12),
    "checkpoint_resume": (pin_checkpoint_resume, 1e-12),
    "non_expansive": (pin_non_expansive, 1e-12),
    "qk_scale_invariance": (pin_qk_scale_invariance, 1e-4),
    "decode_heads_match_prefill_T1": (pin_decode_heads_match_prefill_T1, 1e-12),
    "conv_identity_tap": (pin_conv_identity_tap, 0.0),
    "conv_matches_library": (pin_conv_matches_library, 1e-12),
    "conv_stays_in_sequence": (pin_conv_stays_in_sequence, 0.0),
    "silu_closed_form": (pin_silu_closed_form, 1e-15),
    "conv_history_continues": (pin_conv_history_continues, 1e-12),
    "decode_fused_continues_prefill": (pin_decode_fused_continues_prefill, 1e-12),
    "output_gate_values": (pin_output_gate_values, 1e-15),
}


def run_all(lib=None):
    """{name: (violation, bar, ok)} for every pin."""
    res = {}
    for name, (fn, bar) in PINS.items():
        try:
            val = float(fn(lib=lib))
        except Exception:  # a broken build may raise; that counts as caught
            val = np.inf
        res[name] = (val, bar, bool(val <= bar))
    return res
