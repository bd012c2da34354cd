"""First GPU parity checks: decode and prefill on small seeded cases."""
import numpy as np
import pytest
import torch

from kda_parity import (TOL_OUT_BF16, TOL_OUT_FP32, TOL_STATE, out_err, run_gpu_prefill,
                        run_oracle_prefill, state_err, to_np)
from linear_attention_serving_k1_gb300 import kda, workloads
from oracle import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_decode_small(D, dtype):
    w = workloads.DecodeWorkload("t", N=5, H=3, D=D, steps=3, dtype=dtype, seed=11)
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


@pytest.mark.parametrize("dtype,D", [("fp32", 64), ("bf16", 128), ("fp32", 128), ("bf16", 64)])
def test_prefill_small_ragged(dtype, D):
    w = workloads.custom_prefill(H=2, D=D, lens=[1, 63, 64, 65, 130], dtype=dtype, init="randn",
                                 ckpt_stride=64, seed=21)
    inp = workloads.make_prefill(w)
    o, f, ck = run_gpu_prefill(inp, ckpt_stride=64)
    o_r, f_r, ck_r = run_oracle_prefill(inp, ckpt_stride=64)
    tol = TOL_OUT_FP32 if dtype == "fp32" else TOL_OUT_BF16
    assert out_err(to_np(o), o_r) <= tol
    assert state_err(to_np(f), f_r) <= TOL_STATE
    assert ck.shape[0] == ck_r.shape[0] == 4
    assert state_err(to_np(ck), ck_r) <= TOL_STATE
