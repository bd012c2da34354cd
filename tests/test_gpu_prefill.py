"""GPU parity of kda_prefill against the float64 oracle (same seeded inputs).

Bars: max|o - o_ref| / rms(o_ref) <= 1e-4 on fp32 inputs, <= 2e-2 on bf16
inputs; relative Frobenius error of final states and checkpoints <= 1e-2.
The bf16 / head-dim-128 cases run the tensor-core path, the others the fp32
CUDA-core path."""
import numpy as np
import pytest
import torch

from kda_parity import (TOL_OUT_BF16, TOL_OUT_FP32, TOL_STATE, gpu_inputs, out_err, run_gpu_prefill,
                        run_oracle_prefill, state_err, to_np)
from linear_attention_serving_k1_gb300 import kda, workloads
from oracle import oracle

pytestmark = pytest.mark.gpu


def _tol(dtype):
    return TOL_OUT_FP32 if dtype == "fp32" else TOL_OUT_BF16


def _check(inp, ckpt_stride=0, heads=None, report=None):
    w = inp["workload"]
    o, f, ck = run_gpu_prefill(inp, ckpt_stride=ckpt_stride)
    o_r, f_r, ck_r = run_oracle_prefill(inp, ckpt_stride=ckpt_stride, heads=heads)
    if heads is not None:
        o, f = o[:, heads], f[:, heads]
        ck = ck[:, heads] if ck is not None else None
    eo, ef = out_err(to_np(o), o_r), state_err(to_np(f), f_r)
    ec = state_err(to_np(ck), ck_r) if ckpt_stride else 0.0
    if report is not None:
        report.update(out=eo, state=ef, ckpt=ec)
    assert eo <= _tol(w.dtype), f"output error {eo:.3e}"
    assert ef <= TOL_STATE, f"final-state error {ef:.3e}"
    if ckpt_stride:
        assert ck.shape[0] == ck_r.shape[0]
        assert ec <= TOL_STATE, f"checkpoint error {ec:.3e}"
    return eo, ef, ec


def test_workload1_oracle_scale_fp32():
    """B=1, H=2, T=256, D=64, all fp32, zero initial state."""
    w = workloads.workload(1)
    eo, ef, _ = _check(workloads.make_prefill(w))
    assert ef <= 1e-4


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 64), ("fp32", 128), ("bf16", 64)])
def test_ragged_tails_and_checkpoints(dtype, D):
    w = workloads.custom_prefill(H=3, D=D, lens=[1, 63, 64, 65, 127, 130, 256], dtype=dtype,
                                 init="randn", ckpt_stride=64, seed=21)
    _check(workloads.make_prefill(w), ckpt_stride=64)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 64)])
def test_empty_sequences_in_pack(dtype, D):
    w = workloads.custom_prefill(H=2, D=D, lens=[0, 70, 0, 0, 5, 0], dtype=dtype, init="randn",
                                 seed=4, varlen=True)
    inp = workloads.make_prefill(w)
    _check(inp)
    _, f, _ = run_gpu_prefill(inp)
    s0 = inp["init_state"].numpy()
    for n in (0, 2, 3, 5):   # empty sequences return their initial state unchanged
        assert np.array_equal(to_np(f[n]), s0[n].astype(np.float64))


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 64)])
def test_zero_initial_state_is_null(dtype, D):
    w = workloads.custom_prefill(H=2, D=D, lens=[200], dtype=dtype, init="zeros", seed=5)
    _check(workloads.make_prefill(w))


def test_equal_length_batch_without_cu_seqlens():
    w = workloads.custom_prefill(H=4, D=128, lens=[192, 192, 192], dtype="bf16", init="randn",
                                 seed=6, varlen=False)
    inp = workloads.make_prefill(w)
    assert inp["cu_seqlens"] is None
    _check(inp)


def test_final_state_may_alias_initial_state():
    w = workloads.custom_prefill(H=2, D=128, lens=[100, 300], dtype="bf16", init="randn", seed=8)
    inp = workloads.make_prefill(w)
    d = gpu_inputs(inp)
    s = d["init_state"].clone()
    kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], s, d["cu_seqlens"], final_state=s)
    torch.cuda.synchronize()
    _, f_r, _ = run_oracle_prefill(inp)
    assert state_err(to_np(s), f_r) <= TOL_STATE


def test_no_tokens():
    """T = 0: nothing to compute; final state = initial state."""
    w = workloads.custom_prefill(H=2, D=128, lens=[0, 0], dtype="bf16", init="randn", seed=9, varlen=True)
    inp = workloads.make_prefill(w)
    d = gpu_inputs(inp)
    o, f, _ = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"])
    torch.cuda.synchronize()
    assert o.shape[0] == 0
    assert torch.equal(f, d["init_state"])


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 64)])
def test_beta0_g0_keeps_state(dtype, D):
    """beta = 0 and g = 0: S unchanged and o_t = S0^T qhat_t (GPU side of the pin)."""
    w = workloads.custom_prefill(H=2, D=D, lens=[150], dtype=dtype, init="randn", seed=10)
    inp = workloads.make_prefill(w)
    inp["g"] = torch.zeros_like(inp["g"])
    inp["beta"] = torch.zeros_like(inp["beta"])
    inp["init_state"] = inp["init_state"] * 100.0
    d = gpu_inputs(inp)
    o, f, _ = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], None)
    torch.cuda.synchronize()
    assert state_err(to_np(f), to_np(d["init_state"])) <= (1e-6 if dtype == "fp32" else 1e-2)
    qf = inp["q"].double()
    qh = qf / torch.sqrt((qf * qf).sum(-1, keepdim=True) + 1e-6)
    want = torch.einsum("hkv,thk->thv", inp["init_state"][0].double(), qh).numpy()
    assert out_err(to_np(o), want) <= _tol(dtype)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 64)])
def test_prefill_then_decode_continues(dtype, D):
    """prefill(t tokens) then decode(token t+1) == prefill(t+1 tokens), all on the GPU."""
    w = workloads.custom_prefill(H=2, D=D, lens=[131], dtype=dtype, init="randn", seed=12)
    inp = workloads.make_prefill(w)
    d = gpu_inputs(inp)
    o_all, f_all, _ = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], None)
    _, f_pre, _ = kda.prefill(*(d[n][:-1].contiguous() for n in ("q", "k", "v", "g", "beta")),
                              d["init_state"], None)
    st = f_pre.clone()
    od = kda.decode(*(d[n][-1:].contiguous() for n in ("q", "k", "v", "g", "beta")), st)
    torch.cuda.synchronize()
    assert out_err(to_np(od[0]), to_np(o_all[-1])) <= _tol(dtype)
    assert state_err(to_np(st), to_np(f_all)) <= TOL_STATE


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 64)])
def test_resume_from_checkpoint(dtype, D):
    """prefill(T) == prefill(T - stride, init = snapshot after stride tokens)."""
    stride = 128
    w = workloads.custom_prefill(H=2, D=D, lens=[448], dtype=dtype, init="randn", ckpt_stride=stride, seed=13)
    inp = workloads.make_prefill(w)
    d = gpu_inputs(inp)
    o, f, ck = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], None,
                           ckpt_stride=stride, ckpt_capacity=3)
    o2, f2, _ = kda.prefill(*(d[n][stride:].contiguous() for n in ("q", "k", "v", "g", "beta")),
                            ck[0:1].contiguous(), None)
    torch.cuda.synchronize()
    assert out_err(to_np(o2), to_np(o[stride:])) <= _tol(dtype)
    assert state_err(to_np(f2), to_np(f)) <= TOL_STATE
    _, f256, _ = kda.prefill(*(d[n][:256].contiguous() for n in ("q", "k", "v", "g", "beta")),
                             d["init_state"], None)
    torch.cuda.synchronize()
    assert state_err(to_np(ck[1]), to_np(f256[0])) <= TOL_STATE


def test_checkpoint_overflow_is_reported():
    """More snapshots due than slots: the extra ones are dropped and the device
    status word reports KDA_ERR_CKPT_OVERFLOW; outputs are unaffected."""
    w = workloads.custom_prefill(H=2, D=128, lens=[256, 192], dtype="bf16", init="randn", ckpt_stride=64, seed=14)
    inp = workloads.make_prefill(w)
    d = gpu_inputs(inp)
    desc = kda.make_desc(448, 2, 128, 2, kda.DTYPE_BF16, 64, 64, 3)
    ws = kda.alloc_workspace(desc, "cuda")
    ck = torch.zeros(3, 2, 128, 128, device="cuda")
    o, f, _ = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                          ckpt_stride=64, ckpts=ck, ckpt_capacity=3, workspace=ws)
    assert kda.prefill_status(ws) == kda.STATUS_CODES["KDA_ERR_CKPT_OVERFLOW"]
    assert kda.prefill_status(ws) == 0          # reading clears it
    o_r, f_r, ck_r = run_oracle_prefill(inp, ckpt_stride=64)
    assert out_err(to_np(o), o_r) <= TOL_OUT_BF16
    assert state_err(to_np(ck), ck_r[:3]) <= TOL_STATE


def test_malformed_cu_seqlens_is_reported():
    w = workloads.custom_prefill(H=2, D=128, lens=[64, 64], dtype="bf16", init="randn", seed=15)
    inp = workloads.make_prefill(w)
    d = gpu_inputs(inp)
    bad = torch.tensor([0, 100, 64], dtype=torch.int32, device="cuda")   # decreasing
    desc = kda.make_desc(128, 2, 128, 2, kda.DTYPE_BF16)
    ws = kda.alloc_workspace(desc, "cuda")
    kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], bad, workspace=ws)
    assert kda.prefill_status(ws) == kda.STATUS_CODES["KDA_ERR_INVALID_ARG"]


def test_workload2_full():
    """B=1, H=32, T=8192, D=128, bf16, random initial state: every output and state."""
    rep = {}
    _check(workloads.make_prefill(workloads.workload(2)), report=rep)
    print("workload 2 errors", rep)


def test_workload4_sampled_heads_with_checkpoints():
    """B=1, H=32, T=131072 with snapshots every 32768 tokens; the GPU runs all
    heads, the oracle recomputes heads 0 and 31 (heads are independent)."""
    w = workloads.workload(4)
    rep = {}
    _check(workloads.make_prefill(w), ckpt_stride=w.ckpt_stride, heads=[0, 31], report=rep)
    print("workload 4 errors", rep)


def test_workload5_varlen_sampled_heads():
    """16 packed sequences with lengths U[1024, 32768]; heads 0 and 17 recomputed."""
    rep = {}
    _check(workloads.make_prefill(workloads.workload(5)), heads=[0, 17], report=rep)
    print("workload 5 errors", rep)
