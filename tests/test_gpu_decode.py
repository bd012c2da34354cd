"""GPU parity of kda_decode against the float64 oracle."""
import numpy as np
import pytest
import torch

from kda_parity import TOL_OUT_BF16, TOL_OUT_FP32, TOL_STATE, out_err, state_err, to_np
from linear_attention_serving_k1_gb300 import kda, workloads
from oracle import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_decode_steps(D, dtype):
    w = workloads.DecodeWorkload("t", N=5, H=3, D=D, steps=4, dtype=dtype, seed=11)
    st = workloads.make_decode_state(w)
    st_gpu = st.cuda()
    ref = st.numpy().astype(np.float64)
    for s in range(w.steps):
        x = workloads.make_decode_step(w, s)
        o = kda.decode(*(x[n].cuda() for n in ("q", "k", "v", "g", "beta")), st_gpu)
        o_ref, ref = oracle.decode(x["q"], x["k"], x["v"], x["g"], x["beta"], ref)
        torch.cuda.synchronize()
        tol = TOL_OUT_FP32 if dtype == "fp32" else TOL_OUT_BF16
        assert out_err(to_np(o), o_ref) <= tol
        assert state_err(to_np(st_gpu), ref) <= (1e-5 if dtype == "fp32" else TOL_STATE)


def test_decode_beta0_g0_keeps_state():
    w = workloads.DecodeWorkload("t", N=4, H=2, D=128, steps=1, dtype="bf16", seed=2)
    st = workloads.make_decode_state(w).cuda()
    s0 = st.clone()
    x = workloads.make_decode_step(w, 0)
    x["g"].zero_()
    x["beta"].zero_()
    o = kda.decode(*(x[n].cuda() for n in ("q", "k", "v", "g", "beta")), st)
    torch.cuda.synchronize()
    assert torch.equal(st, s0)
    qf = x["q"].double()
    qh = qf / torch.sqrt((qf * qf).sum(-1, keepdim=True) + 1e-6)
    want = torch.einsum("nhkv,nhk->nhv", s0.cpu().double(), qh).numpy()
    assert out_err(to_np(o), want) <= TOL_OUT_BF16


def test_workload3_64_steps_sampled():
    """256 sequences x 32 heads, D=128, 64 consecutive in-place steps; the
    oracle follows sequences {0, 97, 255} x heads {0, 31} through all steps."""
    w = workloads.workload(3)
    st = workloads.make_decode_state(w)
    st_gpu = st.cuda()
    ns, hs = [0, 97, 255], [0, 31]
    ref = st[ns][:, hs].numpy().astype(np.float64)
    worst_o = worst_s = 0.0
    for s in range(w.steps):
        x = workloads.make_decode_step(w, s)
        o = kda.decode(*(x[n].cuda() for n in ("q", "k", "v", "g", "beta")), st_gpu)
        sel = {n: x[n][ns][:, hs] for n in ("q", "k", "v", "g", "beta")}
        o_ref, ref = oracle.decode(sel["q"], sel["k"], sel["v"], sel["g"], sel["beta"], ref)
        torch.cuda.synchronize()
        worst_o = max(worst_o, out_err(to_np(o[ns][:, hs]), o_ref))
    worst_s = state_err(to_np(st_gpu[ns][:, hs]), ref)
    print(f"workload 3: output {worst_o:.3e} state {worst_s:.3e}")
    assert worst_o <= TOL_OUT_BF16
    assert worst_s <= TOL_STATE
