"""Scalar-gate prefill (one log-decay per token and head, the Gated DeltaNet
form): the float64 oracle's scalar-gate recurrence pins it, and the library
must give exactly what its per-channel form gives with the gate repeated over
the key channels."""
import numpy as np
import pytest
import torch

from kda_parity import TOL_OUT_BF16, TOL_OUT_FP32, TOL_STATE, gpu_inputs, out_err, state_err, to_np
from linear_attention_serving_k1_gb300 import kda, workloads
from oracle import oracle

pytestmark = pytest.mark.gpu


def _inputs(dtype, D, lens, seed):
    w = workloads.custom_prefill(H=3, D=D, lens=lens, dtype=dtype, init="randn", seed=seed, varlen=True)
    inp = workloads.make_prefill(w)
    d = gpu_inputs(inp)
    a = inp["g"][:, :, 0].contiguous()          # one log-decay per token and head
    return w, inp, d, a


def _prefill(d, gate, **kw):
    o, f, _ = kda.prefill(d["q"], d["k"], d["v"], gate, d["beta"], d["init_state"], d["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    return o, f


@pytest.mark.parametrize("dtype,D,tol", [("bf16", 128, TOL_OUT_BF16), ("fp32", 64, TOL_OUT_FP32),
                                         ("fp32", 128, TOL_OUT_FP32)])
def test_scalar_gate_matches_oracle(dtype, D, tol):
    w, inp, d, a = _inputs(dtype, D, [1, 63, 64, 65, 200, 0, 130], seed=41)
    o, f = _prefill(d, a.to(d["g"].device))
    o_r, f_r = oracle.gdn_prefill(inp["q"], inp["k"], inp["v"], a, inp["beta"], inp["init_state"],
                                  inp["cu_host"].numpy())
    assert out_err(to_np(o), o_r) <= tol
    assert state_err(to_np(f), f_r) <= TOL_STATE


@pytest.mark.parametrize("segment_chunks", [0, 2])
def test_scalar_gate_equals_repeated_per_channel_gate(segment_chunks):
    w, inp, d, a = _inputs("bf16", 128, [64, 320, 17], seed=42)
    a_dev = a.to(d["g"].device)
    o1, f1 = _prefill(d, a_dev, segment_chunks=segment_chunks)
    rep = a_dev[:, :, None].expand(-1, -1, 128).contiguous()
    o2, f2 = _prefill(d, rep, segment_chunks=segment_chunks)
    assert torch.equal(o1, o2)
    assert torch.equal(f1, f2)
