"""Shared helpers of the GPU parity tests: run the CUDA path and the oracle on
the same seeded inputs and compute the error metrics the tolerances use."""
from __future__ import annotations

import numpy as np
import torch

from linear_attention_serving_k1_gb300 import kda, workloads
from oracle import oracle

# Tolerances: max|o - o_ref| / rms(o_ref) and relative Frobenius error of states.
TOL_OUT_FP32 = 1e-4
TOL_OUT_BF16 = 2e-2
TOL_STATE = 1e-2


def bf16_half_ulp(x) -> np.ndarray:
    """Largest error of rounding the exact value x to bf16 (8 significant bits):
    half the bf16 spacing 2^(e-7) of the binade [2^e, 2^(e+1)) holding |x|."""
    ax = np.maximum(np.abs(np.asarray(x, np.float64)), np.finfo(np.float32).tiny)
    e = np.floor(np.log2(ax))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def out_err(o_gpu, o_ref, bf16_output=None) -> float:
    """max |o - o_ref| / rms(o_ref).

    For bf16 outputs (detected from the values when bf16_output is None) the
    half-ulp that rounding the exact result to bf16 costs by itself is not
    counted: |o - o_ref| is reduced by bf16_half_ulp(o_ref) before the max.
    Outputs here are heavy-tailed (max/rms ~ 10-20), so that rounding alone can
    reach 2e-2 * rms; the bar is meant for the arithmetic."""
    o_gpu = np.asarray(o_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    if o_ref.size == 0:
        return 0.0
    rms = np.sqrt(np.mean(o_ref * o_ref))
    diff = np.abs(o_gpu - o_ref)
    if bf16_output is None:
        bf16_output = bool(np.all(o_gpu.astype(np.float32).view(np.uint32) & 0xFFFF == 0))
    if bf16_output:
        diff = np.maximum(diff - bf16_half_ulp(o_ref), 0.0)
    return float(diff.max() / max(rms, 1e-30))


def out_err_raw(o_gpu, o_ref) -> float:
    """max |o - o_ref| / rms(o_ref) with nothing discounted."""
    return out_err(o_gpu, o_ref, bf16_output=False)


def state_err(s_gpu, s_ref) -> float:
    s_gpu = np.asarray(s_gpu, np.float64)
    s_ref = np.asarray(s_ref, np.float64)
    if s_ref.size == 0:
        return 0.0
    return float(np.linalg.norm(s_gpu - s_ref) / max(np.linalg.norm(s_ref), 1e-30))


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def gpu_inputs(inp, device="cuda"):
    out = {}
    for key in ("q", "k", "v", "g", "beta", "init_state", "cu_seqlens"):
        x = inp[key]
        out[key] = None if x is None else x.to(device).contiguous()
    return out


def run_gpu_prefill(inp, ckpt_stride=0, device="cuda"):
    w = inp["workload"]
    d = gpu_inputs(inp, device)
    cap = kda.num_checkpoints(w.lens, ckpt_stride)
    o, f, ck = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                           num_seqs=w.num_seqs, ckpt_stride=ckpt_stride,
                           ckpt_capacity=cap if ckpt_stride else None)
    torch.cuda.synchronize()
    return o, f, (ck[:cap] if ck is not None else None)


def run_oracle_prefill(inp, ckpt_stride=0, heads=None):
    w = inp["workload"]
    cu = inp["cu_host"].numpy()
    return oracle.prefill_heads(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["init_state"],
                                cu, ckpt_stride, heads=heads)
