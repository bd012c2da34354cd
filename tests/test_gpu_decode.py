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


@pytest.mark.parametrize("D,dtype", [(128, torch.bfloat16), (64, torch.float32)])
def test_paged_decode_matches_gathered_states(D, dtype):
    """Decode over a state pool through slot ids: the same bits as decoding the
    gathered states; padding rows (slot -1) output zeros; other slots untouched."""
    gen = torch.Generator(device="cpu").manual_seed(77)
    N, H, P = 5, 4, 7
    slots = torch.tensor([3, 0, -1, 6, 2], dtype=torch.int32)
    pool = (0.05 * torch.randn(P, H, D, D, generator=gen)).cuda()
    q = torch.randn(N, H, D, generator=gen).to(dtype).cuda()
    k = torch.randn(N, H, D, generator=gen).to(dtype).cuda()
    v = torch.randn(N, H, D, generator=gen).to(dtype).cuda()
    g = (-torch.exp(torch.empty(N, H, D).uniform_(-5, -1, generator=gen))).cuda()
    beta = torch.sigmoid(torch.randn(N, H, generator=gen)).cuda()
    valid = [i for i in range(N) if slots[i] >= 0]
    gathered = pool[slots[valid].long()].clone()
    out_ref = kda.decode(q[valid].contiguous(), k[valid].contiguous(), v[valid].contiguous(),
                         g[valid].contiguous(), beta[valid].contiguous(), gathered)
    pool2 = pool.clone()
    out = kda.decode_paged(q, k, v, g, beta, pool2, slots.cuda())
    torch.cuda.synchronize()
    assert torch.equal(out[valid], out_ref)
    assert torch.count_nonzero(out[2]) == 0
    for j, i in enumerate(valid):
        assert torch.equal(pool2[slots[i]], gathered[j])
    for s in (1, 4, 5):
        assert torch.equal(pool2[s], pool[s])
