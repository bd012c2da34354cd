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
