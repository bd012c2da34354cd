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


@pytest.mark.parametrize("D,dtype,tol", [(128, torch.bfloat16, TOL_OUT_BF16), (64, torch.float32, TOL_OUT_FP32)])
def test_multi_token_decode_against_oracle(D, dtype, tol):
    """m tokens per sequence in one call: every output follows the token
    recurrence from the given state, and each state is written after its own
    commit length (0 = untouched, m = all)."""
    gen = torch.Generator(device="cpu").manual_seed(78)
    N, m, H = 4, 5, 3
    s0 = 0.05 * torch.randn(N, H, D, D, generator=gen, dtype=torch.float64)
    q = torch.randn(N, m, H, D, generator=gen).to(dtype)
    k = torch.randn(N, m, H, D, generator=gen).to(dtype)
    v = torch.randn(N, m, H, D, generator=gen).to(dtype)
    g = -torch.exp(torch.empty(N, m, H, D).uniform_(-5, -1, generator=gen))
    beta = torch.sigmoid(torch.randn(N, m, H, generator=gen))
    commit = torch.tensor([0, 2, 5, 1], dtype=torch.int32)
    st = s0.float().cuda()
    out = kda.decode_multi(q.cuda(), k.cuda(), v.cuda(), g.cuda(), beta.cuda(), st, commit.cuda())
    torch.cuda.synchronize()
    flat = lambda x: x.reshape(N * m, *x.shape[2:])
    cu = np.arange(N + 1, dtype=np.int64) * m
    o_r, _, _ = oracle.prefill(flat(q), flat(k), flat(v), flat(g), flat(beta), s0, cu)
    assert out_err(to_np(out).reshape(N * m, H, D), o_r) <= tol
    for n in range(N):
        c = int(commit[n])
        if c == 0:
            assert torch.equal(st[n].cpu(), s0[n].float())   # untouched
            continue
        _, f_r, _ = oracle.prefill(q[n, :c], k[n, :c], v[n, :c], g[n, :c], beta[n, :c], s0[n:n + 1], None)
        assert state_err(to_np(st[n]), f_r[0]) <= TOL_STATE


def test_single_token_multi_decode_is_decode():
    gen = torch.Generator(device="cpu").manual_seed(79)
    N, H, D = 3, 4, 128
    st = (0.05 * torch.randn(N, H, D, D, generator=gen)).cuda()
    q, k, v = (torch.randn(N, H, D, generator=gen).to(torch.bfloat16).cuda() for _ in range(3))
    g = (-torch.exp(torch.empty(N, H, D).uniform_(-5, -1, generator=gen))).cuda()
    beta = torch.sigmoid(torch.randn(N, H, generator=gen)).cuda()
    st1, st2 = st.clone(), st.clone()
    o1 = kda.decode(q, k, v, g, beta, st1)
    o2 = kda.decode_multi(q[:, None], k[:, None], v[:, None], g[:, None], beta[:, None], st2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2[:, 0])
    assert torch.equal(st1, st2)
