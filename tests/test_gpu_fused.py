"""kda_prefill_fused: the short convolution of q, k, v before the recurrence
and the sigmoid output gate after it, fused into the prefill kernels, against
the float64 oracle's own convolution, recurrence and gate on the same seeded
inputs (bars as for kda_prefill: max|o - o_ref| / rms(o_ref) <= 2e-2 on bf16
outputs, <= 1e-4 on fp32 outputs, relative Frobenius error of states and
checkpoints <= 1e-2)."""
import numpy as np
import pytest
import torch

from kda_parity import (TOL_OUT_BF16, TOL_OUT_FP32, TOL_STATE, bf16_half_ulp, gpu_inputs, out_err, state_err,
                        to_np)
from linear_attention_serving_k1_gb300 import kda, workloads
from oracle import oracle

pytestmark = pytest.mark.gpu

LENS = [1, 3, 63, 64, 65, 130, 200]


def _fused_inputs(dtype, D, W, seed):
    w = workloads.custom_prefill(H=2, D=D, lens=LENS, dtype=dtype, init="randn", ckpt_stride=64, seed=seed,
                                 varlen=True)
    inp = workloads.make_prefill(w)
    gen = torch.Generator().manual_seed(seed + 1)
    taps = torch.rand(3, W, 2, D, generator=gen) * 2.0 - 1.0
    z = torch.randn(w.total_tokens, 2, D, generator=gen).to(inp["q"].dtype)
    return w, inp, taps, z


@pytest.mark.parametrize("dtype,D,seg", [("bf16", 128, 0), ("bf16", 128, 2), ("fp32", 64, 0)])
@pytest.mark.parametrize("W,silu,use_gate", [(4, False, True), (4, True, True), (2, True, False), (3, False, False)])
def test_fused_matches_oracle(dtype, D, seg, W, silu, use_gate):
    w, inp, taps, z = _fused_inputs(dtype, D, W, seed=71 + W)
    d = gpu_inputs(inp)
    cap = kda.num_checkpoints(w.lens, 64)
    o, f, ck = kda.prefill_fused(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                                 conv_w=taps.cuda(), conv_silu=silu, gate=z.cuda() if use_gate else None,
                                 ckpt_stride=64, ckpt_capacity=cap, segment_chunks=seg)
    torch.cuda.synchronize()
    o_r, f_r, ck_r = oracle.prefill_fused(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["init_state"],
                                          inp["cu_host"].numpy(), 64, conv_w=taps.double().numpy(), silu=silu,
                                          gate=z if use_gate else None)
    tol = TOL_OUT_FP32 if dtype == "fp32" else TOL_OUT_BF16
    assert torch.isfinite(o.float()).all()
    eo = out_err(to_np(o), o_r)
    assert eo <= tol, f"output error {eo:.3e}"
    assert state_err(to_np(f), f_r) <= TOL_STATE
    assert state_err(to_np(ck[:cap]), ck_r) <= TOL_STATE


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 64)])
def test_pass_through_taps_equal_plain_prefill(dtype, D):
    """Taps (0, 0, 0, 1) without activation or gate reproduce kda_prefill: bit
    for bit on the fp32 path; on the tensor-core path the convolved rows pass
    through f16, which keeps every bf16 input except those below f16's normal
    range (about 6e-5), so the results agree to well inside the bars."""
    w, inp, taps, _ = _fused_inputs(dtype, D, 4, seed=81)
    taps.zero_()
    taps[:, 3] = 1.0
    d = gpu_inputs(inp)
    o1, f1, _ = kda.prefill_fused(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                                  conv_w=taps.cuda())
    o2, f2, _ = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"])
    torch.cuda.synchronize()
    if dtype == "fp32":
        assert torch.equal(o1, o2)
        assert torch.equal(f1, f2)
    else:
        assert out_err(to_np(o1), to_np(o2)) <= 2e-3
        assert state_err(to_np(f1), to_np(f2)) <= 1e-3


def test_gate_alone_scales_the_plain_output():
    """Without taps the fused call is kda_prefill followed by o * sigmoid(z)."""
    w, inp, _, z = _fused_inputs("bf16", 128, 4, seed=91)
    d = gpu_inputs(inp)
    o1, f1, _ = kda.prefill_fused(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                                  gate=z.cuda())
    o2, f2, _ = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"])
    torch.cuda.synchronize()
    assert torch.equal(f1, f2)
    # o1 rounds o * sigmoid(z) once; o2 * sigmoid(z) carries o2's own rounding:
    # they differ by at most a few bf16 half-units of the gated value
    want = oracle.output_gate(to_np(o2), z)
    diff = np.abs(to_np(o1) - want)
    assert (diff <= 4 * bf16_half_ulp(want) + 1e-30).all()


def _split(inp, cuts):
    """The packed inputs cut into (first cuts[n] tokens of each sequence, the rest)."""
    cu = inp["cu_host"].tolist()
    first, rest = [], []
    for n in range(len(cu) - 1):
        first += list(range(cu[n], cu[n] + cuts[n]))
        rest += list(range(cu[n] + cuts[n], cu[n + 1]))
    f_idx, r_idx = torch.tensor(first, dtype=torch.long), torch.tensor(rest, dtype=torch.long)
    lens = [cu[n + 1] - cu[n] for n in range(len(cu) - 1)]
    cu1 = torch.tensor([0] + list(np.cumsum(cuts)), dtype=torch.int32)
    cu2 = torch.tensor([0] + list(np.cumsum([L - c for L, c in zip(lens, cuts)])), dtype=torch.int32)
    pick = lambda idx: {n: inp[n][idx].contiguous() for n in ("q", "k", "v", "g", "beta")}
    return pick(f_idx), pick(r_idx), cu1, cu2, f_idx, r_idx


@pytest.mark.parametrize("dtype,D,W", [("bf16", 128, 4), ("bf16", 128, 3), ("fp32", 64, 4)])
def test_resume_with_convolution_state(dtype, D, W):
    """A packed batch prefilled in two parts, the second seeded with the first's
    final states and convolution state, gives the single call's results; the
    convolution state handed on is the raw rows themselves."""
    w, inp, taps, z = _fused_inputs(dtype, D, W, seed=101)
    d = gpu_inputs(inp)
    N, H = w.num_seqs, 2
    cs_whole = torch.empty(N, 3, W - 1, H, D, dtype=d["q"].dtype, device="cuda")
    o, f, _ = kda.prefill_fused(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                                conv_w=taps.cuda(), conv_silu=True, gate=z.cuda(), conv_state_out=cs_whole)
    cuts = [min(L, c) for L, c in zip(w.lens, [0, 2, 40, 64, 1, 77, 130])]
    p1, p2, cu1, cu2, i1, i2 = _split(inp, cuts)
    cs = torch.empty_like(cs_whole)
    _, f1, _ = kda.prefill_fused(*(p1[n].cuda() for n in ("q", "k", "v", "g", "beta")), d["init_state"],
                                 cu1.cuda(), conv_w=taps.cuda(), conv_silu=True, gate=z[i1].contiguous().cuda(),
                                 conv_state_out=cs)
    o2, f2, _ = kda.prefill_fused(*(p2[n].cuda() for n in ("q", "k", "v", "g", "beta")), f1, cu2.cuda(),
                                  conv_w=taps.cuda(), conv_silu=True, gate=z[i2].contiguous().cuda(),
                                  conv_state_in=cs, conv_state_out=cs)   # updated in place
    torch.cuda.synchronize()
    # each run against the oracle's single call over the whole sequences (two
    # GPU runs chunk the second part differently, so they are compared through it)
    o_r, f_r, _, cs_r = oracle.prefill_fused(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                             inp["init_state"], inp["cu_host"].numpy(), 0,
                                             conv_w=taps.double().numpy(), silu=True, gate=z,
                                             return_conv_state=True)
    tol = TOL_OUT_FP32 if dtype == "fp32" else TOL_OUT_BF16
    assert out_err(to_np(o), o_r) <= tol
    assert out_err(to_np(o2), o_r[i2.numpy()]) <= tol
    assert state_err(to_np(f2), f_r) <= TOL_STATE
    assert state_err(to_np(f), f_r) <= TOL_STATE
    # the convolution state handed on is the raw rows: exact, whichever way it was reached
    assert torch.equal(cs, cs_whole)
    assert np.array_equal(to_np(cs_whole), cs_r)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 64)])
def test_decode_fused_continues_prefill_fused(dtype, D):
    """prefill_fused over all but the last token of each sequence, then
    decode_fused on the last tokens with the handed-on states and convolution
    state, equals the oracle's fused prefill over the whole sequences."""
    W = 4
    lens = [5, 70, 130]
    w = workloads.custom_prefill(H=2, D=D, lens=lens, dtype=dtype, init="randn", seed=111, varlen=True)
    inp = workloads.make_prefill(w)
    gen = torch.Generator().manual_seed(112)
    taps = torch.rand(3, W, 2, D, generator=gen) * 2.0 - 1.0
    z = torch.randn(w.total_tokens, 2, D, generator=gen).to(inp["q"].dtype)
    p1, p2, cu1, _, i1, i2 = _split(inp, [L - 1 for L in lens])
    d = gpu_inputs(inp)
    cs = torch.empty(3, 3, W - 1, 2, D, dtype=d["q"].dtype, device="cuda")
    _, st, _ = kda.prefill_fused(*(p1[n].cuda() for n in ("q", "k", "v", "g", "beta")), d["init_state"],
                                 cu1.cuda(), conv_w=taps.cuda(), gate=z[i1].contiguous().cuda(), conv_state_out=cs)
    od = kda.decode_fused(*(p2[n].cuda() for n in ("q", "k", "v", "g", "beta")), st, conv_w=taps.cuda(),
                          conv_state=cs, gate=z[i2].contiguous().cuda())
    torch.cuda.synchronize()
    o_r, f_r, _, cs_r = oracle.prefill_fused(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                             inp["init_state"], inp["cu_host"].numpy(), 0,
                                             conv_w=taps.double().numpy(), gate=z, return_conv_state=True)
    tol = TOL_OUT_FP32 if dtype == "fp32" else TOL_OUT_BF16
    assert out_err(to_np(od), o_r[i2.numpy()]) <= tol
    assert state_err(to_np(st), f_r) <= TOL_STATE
    assert np.array_equal(to_np(cs), cs_r)   # advanced by the decoded tokens' raw rows
