"""GPU parity beyond the benchmark recipe: un-normalised q/k, strong decay, a
state of wide dynamic range, the bounded-wait unwind, prefill over a state
pool and repeated decode slots.

Every case runs the CUDA path through the C ABI and compares it with the
float64 oracle on the same seeded inputs (bars: max|o - o_ref| / rms(o_ref)
<= 2e-2 on bf16 outputs, <= 1e-4 on fp32 outputs; relative Frobenius error
of final states and checkpoints <= 1e-2)."""
import numpy as np
import pytest
import torch

from kda_parity import (TOL_OUT_BF16, TOL_OUT_FP32, TOL_STATE, gpu_inputs, out_err, run_oracle_prefill,
                        state_err, to_np)
from linear_attention_serving_k1_gb300 import kda, workloads
from oracle import oracle

pytestmark = pytest.mark.gpu

LENS = [1, 63, 64, 65, 130]

# (dtype, D, segment_chunks, scalar_gate): the tensor-core path with one
# segment and with the segmented two-stream plan, the fp32 CUDA-core path, and
# the scalar-gate forms of both
PATHS = [("bf16", 128, 0, False), ("bf16", 128, 2, False), ("fp32", 64, 0, False),
         ("bf16", 128, 0, True), ("fp32", 64, 0, True)]


def _scalar_gate(inp):
    out = dict(inp)
    out["g"] = inp["g"][:, :, 0].contiguous()
    return out


def _run(inp, ckpt_stride=0, segment_chunks=0, wait_limit=0, workspace=None):
    w = inp["workload"]
    d = gpu_inputs(inp)
    cap = kda.num_checkpoints(w.lens, ckpt_stride)
    o, f, ck = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                           num_seqs=w.num_seqs, ckpt_stride=ckpt_stride,
                           ckpt_capacity=cap if ckpt_stride else None, segment_chunks=segment_chunks,
                           wait_limit=wait_limit, workspace=workspace)
    torch.cuda.synchronize()
    return o, f, (ck[:cap] if ck is not None else None)


def _oracle(inp, ckpt_stride=0):
    if inp["g"].dim() == 2:   # scalar gate: the oracle's own scalar-gate recurrence
        cu = inp["cu_host"].numpy()
        o, f = oracle.gdn_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["init_state"], cu)
        return o, f, None
    return run_oracle_prefill(inp, ckpt_stride=ckpt_stride)


def _check(inp, dtype, ckpt_stride=0, segment_chunks=0):
    o, f, ck = _run(inp, ckpt_stride, segment_chunks)
    o_r, f_r, ck_r = _oracle(inp, ckpt_stride)
    tol = TOL_OUT_FP32 if dtype == "fp32" else TOL_OUT_BF16
    assert torch.isfinite(o.float()).all() and torch.isfinite(f).all()
    eo, ef = out_err(to_np(o), o_r), state_err(to_np(f), f_r)
    assert eo <= tol, f"output error {eo:.3e}"
    assert ef <= TOL_STATE, f"final-state error {ef:.3e}"
    if ck_r is not None and ckpt_stride:
        ec = state_err(to_np(ck), ck_r)
        assert ec <= TOL_STATE, f"checkpoint error {ec:.3e}"
    return eo, ef


@pytest.mark.parametrize("dtype,D,seg,sg", PATHS)
def test_unnormalised_qk(dtype, D, seg, sg):
    """q and k rows scaled by independent factors in [0.05, 40]: the library's
    own L2 normalisation (folded into scalars on the tensor-core path) must
    give the oracle's result, which normalises the raw rows."""
    w = workloads.custom_prefill(H=3, D=D, lens=LENS, dtype=dtype, init="randn", ckpt_stride=64, seed=41,
                                 varlen=True)
    inp = workloads.scale_qk_rows(workloads.make_prefill(w), 0.05, 40.0, seed=42)
    qn = inp["q"].float().norm(dim=-1)
    assert qn.min() < 0.2 and qn.max() > 10   # the rows really are far from unit length
    if sg:
        inp = _scalar_gate(inp)
    _check(inp, dtype, ckpt_stride=0 if sg else 64, segment_chunks=seg)


@pytest.mark.parametrize("dtype,D,seg,sg", PATHS)
def test_strong_decay_matches_oracle(dtype, D, seg, sg):
    """g in [-3, -1] per token and channel: one chunk decays by about e^-128,
    beyond the range of a single e^(+-b) factor; the decays are referred to
    the middle of each channel's range, so the result still matches."""
    w = workloads.custom_prefill(H=2, D=D, lens=LENS + [300], dtype=dtype, init="randn", ckpt_stride=64,
                                 seed=43, varlen=True)
    inp = workloads.strong_decay_gates(workloads.make_prefill(w), 1.0, 3.0, seed=44)
    if sg:
        inp = _scalar_gate(inp)
    _check(inp, dtype, ckpt_stride=0 if sg else 64, segment_chunks=seg)
    # and the status word stays clean
    d = gpu_inputs(inp)
    T, H = d["q"].shape[0], d["q"].shape[1]
    desc = kda.make_desc(T, H, D, w.num_seqs, kda.DTYPE_BF16 if dtype == "bf16" else kda.DTYPE_FP32,
                         segment_chunks=seg, scalar_gate=sg)
    ws = kda.alloc_workspace(desc, "cuda")
    kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                segment_chunks=seg, workspace=ws)
    assert kda.prefill_status(ws) == 0


@pytest.mark.parametrize("dtype,D,seg", [("bf16", 128, 0), ("bf16", 128, 2), ("fp32", 64, 0)])
def test_small_beta_wide_state_range(dtype, D, seg):
    """beta in [1e-3, 1e-2] and half of the key channels decaying by 1-3
    nepers per token over a 1,000-token sequence: the state rows of those
    channels stay near beta |k| |v| (about 1e-4, at the edge of the f16 normal
    range the tensor-core operands have) while the other rows grow over the
    sequence, so the state spans several orders of magnitude.  Outputs, final
    states and checkpoints still meet the bars."""
    w = workloads.custom_prefill(H=2, D=D, lens=[1000, 130], dtype=dtype, init="randn", ckpt_stride=256,
                                 seed=47, varlen=True)
    inp = workloads.make_prefill(w)
    gen = torch.Generator().manual_seed(48)
    inp["beta"] = 1e-3 + 9e-3 * torch.rand(inp["beta"].shape, generator=gen)
    strong = workloads.strong_decay_gates(inp, 1.0, 3.0, seed=49)["g"]
    inp["g"] = torch.cat([strong[..., : D // 2], inp["g"][..., D // 2:]], dim=-1).contiguous()
    inp["init_state"] = inp["init_state"] * 1e-3
    _check(inp, dtype, ckpt_stride=256, segment_chunks=seg)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 64)])
def test_decay_beyond_range_is_reported(dtype, D):
    """g = -4 everywhere: a chunk decays by e^-256, beyond the stated range.
    The call reports KDA_ERR_UNSUPPORTED and every output stays finite."""
    w = workloads.custom_prefill(H=2, D=D, lens=[200], dtype=dtype, init="randn", seed=45)
    inp = workloads.make_prefill(w)
    inp["g"] = torch.full_like(inp["g"], -4.0)
    d = gpu_inputs(inp)
    desc = kda.make_desc(200, 2, D, 1, kda.DTYPE_BF16 if dtype == "bf16" else kda.DTYPE_FP32)
    ws = kda.alloc_workspace(desc, "cuda")
    o, f, _ = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], None, workspace=ws)
    assert kda.prefill_status(ws) == kda.STATUS_CODES["KDA_ERR_UNSUPPORTED"]
    assert torch.isfinite(o.float()).all() and torch.isfinite(f).all()


@pytest.mark.parametrize("which,value", [("k", 1.0e5), ("q", -2.0e5), ("v", 7.0e4), ("k", 5.0e4)])
def test_f16_operand_range_is_reported(which, value):
    """The tensor-core path holds q, k and v in f16 operands before
    normalisation: with the debug build, one element beyond the f16 range
    (65504), or a q or k row whose norm reaches it (5e4 in two channels), is
    reported as KDA_ERR_UNSUPPORTED (the release build leaves the check out). One element of 6e4 instead reports nothing: q and k
    then match the oracle (they are normalised); v gives finite outputs (a
    state holding entries near 3e4 beside entries near 1 is beyond what the
    f16 state operand's 11 bits keep within the output bar)."""
    w = workloads.custom_prefill(H=2, D=128, lens=[150], dtype="bf16", init="randn", seed=46)
    inp = workloads.make_prefill(w)
    desc = kda.make_desc(150, 2, 128, 1, kda.DTYPE_BF16)
    ws = kda.alloc_workspace(desc, "cuda")
    big = {n: inp[n].clone() for n in ("q", "k", "v")}
    big[which][97, 1, 5] = value
    if value < 6.5e4:
        big[which][97, 1, 6] = value
    d = gpu_inputs(inp)
    with kda.using_library(kda.load_debug_library()):
        kda.prefill(*(big[n].cuda() for n in ("q", "k", "v")), d["g"], d["beta"], d["init_state"], None,
                    workspace=ws)
        assert kda.prefill_status(ws) == kda.STATUS_CODES["KDA_ERR_UNSUPPORTED"]
    # in range (one element at 6e4 leaves the row norm below the bound): no report
    big[which][97, 1, 5] = 6.0e4 if which != "q" else -6.0e4
    big[which][97, 1, 6] = inp[which][97, 1, 6]
    with kda.using_library(kda.load_debug_library()):
        o, f, _ = kda.prefill(*(big[n].cuda() for n in ("q", "k", "v")), d["g"], d["beta"], d["init_state"], None,
                              workspace=ws)
        assert kda.prefill_status(ws) == kda.KDA_OK
    if which == "v":
        assert torch.isfinite(o.float()).all() and torch.isfinite(f).all()
        return
    o_r, f_r, _ = oracle.prefill(big["q"], big["k"], big["v"], inp["g"], inp["beta"], inp["init_state"], None)
    assert out_err(to_np(o), o_r) <= TOL_OUT_BF16
    assert state_err(to_np(f), f_r) <= TOL_STATE


@pytest.mark.parametrize("seg", [0, 2])
def test_bounded_wait_gives_up_cleanly(seg):
    """With a wait limit of one poll, the tensor-core kernels' waits give up:
    each CTA drains its own copies and MMAs, frees its TMEM, records
    KDA_ERR_TIMEOUT and returns.  The next call on the same context, with the
    default limit, matches the oracle."""
    w = workloads.custom_prefill(H=4, D=128, lens=[700, 130], dtype="bf16", init="randn", seed=46, varlen=True)
    inp = workloads.make_prefill(w)
    d = gpu_inputs(inp)
    desc = kda.make_desc(830, 4, 128, 2, kda.DTYPE_BF16, segment_chunks=seg, wait_limit=1)
    ws = kda.alloc_workspace(desc, "cuda")
    kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                segment_chunks=seg, wait_limit=1, workspace=ws)
    assert kda.prefill_status(ws) == kda.STATUS_CODES["KDA_ERR_TIMEOUT"]
    o, f, _ = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                          segment_chunks=seg, workspace=ws)
    assert kda.prefill_status(ws) == 0
    o_r, f_r, _ = run_oracle_prefill(inp)
    assert out_err(to_np(o), o_r) <= TOL_OUT_BF16
    assert state_err(to_np(f), f_r) <= TOL_STATE


@pytest.mark.parametrize("dtype,D,seg", [("bf16", 128, 0), ("bf16", 128, 2), ("fp32", 64, 0)])
def test_pooled_prefill_equals_gather_prefill_scatter(dtype, D, seg):
    """kda_prefill_pooled reads initial states from pool slots and writes final
    states and snapshots to pool slots: bit-identical to gathering the states,
    a dense kda_prefill, and scattering the results."""
    w = workloads.custom_prefill(H=2, D=D, lens=[130, 0, 200], dtype=dtype, init="randn", ckpt_stride=64,
                                 seed=47, varlen=True)
    inp = workloads.make_prefill(w)
    d = gpu_inputs(inp)
    P = 9
    gen = torch.Generator().manual_seed(48)
    pool = (torch.randn(P, 2, D, D, generator=gen) * 0.01).cuda()
    init_slots = torch.tensor([5, -1, 2], dtype=torch.int32, device="cuda")    # -1: start from zeros
    final_slots = torch.tensor([5, 0, 3], dtype=torch.int32, device="cuda")    # 5: ends where it began
    n_ck = kda.num_checkpoints(w.lens, 64)                                       # 2 + 0 + 3
    ckpt_slots = torch.tensor([4, 6, 7, 8, 1][:n_ck], dtype=torch.int32, device="cuda")
    # dense reference: gather, prefill, scatter
    s0 = torch.stack([pool[5], torch.zeros_like(pool[0]), pool[2]])
    o_ref, f_ref, ck_ref = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], s0.contiguous(),
                                       d["cu_seqlens"], ckpt_stride=64, ckpt_capacity=n_ck, segment_chunks=seg)
    want = pool.clone()
    for n, sl in enumerate([5, 0, 3]):
        want[sl] = f_ref[n]
    for j, sl in enumerate(ckpt_slots.tolist()):
        want[sl] = ck_ref[j]
    o = kda.prefill_pooled(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, init_slots, final_slots,
                           d["cu_seqlens"], ckpt_stride=64, ckpt_slots=ckpt_slots, segment_chunks=seg)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref)
    assert torch.equal(pool, want)
    # and against the oracle
    o_r, f_r, ck_r = run_oracle_prefill(dict(inp, init_state=s0.cpu()), ckpt_stride=64)
    tol = TOL_OUT_FP32 if dtype == "fp32" else TOL_OUT_BF16
    assert out_err(to_np(o), o_r) <= tol
    assert state_err(to_np(pool[[5, 0, 3]]), f_r) <= TOL_STATE
    assert state_err(to_np(pool[ckpt_slots.long()]), ck_r) <= TOL_STATE


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 64)])
def test_pooled_prefill_then_paged_decode_continues(dtype, D):
    """A prompt prefilled into pool slots, then one decode step on those slots,
    equals the oracle's prefill over the prompt plus that token."""
    lens = [100, 37]
    w = workloads.custom_prefill(H=2, D=D, lens=[L + 1 for L in lens], dtype=dtype, init="randn", seed=49,
                                 varlen=True)
    inp = workloads.make_prefill(w)
    o_r, f_r, _ = run_oracle_prefill(inp)
    cu = inp["cu_host"].tolist()
    pre = {n: torch.cat([inp[n][cu[i]:cu[i + 1] - 1] for i in range(2)]) for n in ("q", "k", "v", "g", "beta")}
    last = {n: torch.stack([inp[n][cu[i + 1] - 1] for i in range(2)]) for n in ("q", "k", "v", "g", "beta")}
    cu_pre = torch.tensor([0, lens[0], lens[0] + lens[1]], dtype=torch.int32, device="cuda")
    pool = torch.zeros(4, 2, D, D, device="cuda")
    pool[1] = inp["init_state"][0].cuda()
    pool[3] = inp["init_state"][1].cuda()
    slots = torch.tensor([1, 3], dtype=torch.int32, device="cuda")
    kda.prefill_pooled(*(pre[n].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")), pool, slots, slots,
                       cu_pre)
    od = kda.decode_paged(*(last[n].cuda().contiguous() for n in ("q", "k", "v", "g", "beta")), pool, slots)
    torch.cuda.synchronize()
    tol = TOL_OUT_FP32 if dtype == "fp32" else TOL_OUT_BF16
    want_o = np.stack([o_r[cu[i + 1] - 1] for i in range(2)])
    assert out_err(to_np(od), want_o) <= tol
    assert state_err(to_np(pool[[1, 3]]), f_r) <= TOL_STATE


def test_repeated_decode_slot_is_reported():
    """Two sequences naming the same pool slot set the caller's status word;
    distinct slots leave it at zero."""
    N, H, D = 4, 2, 128
    dw = workloads.DecodeWorkload("dup", N=N, H=H, D=D, steps=1, dtype="bf16", seed=50)
    x = {k_: t.cuda() for k_, t in workloads.make_decode_step(dw, 0).items()}
    pool = torch.zeros(6, H, D, D, device="cuda")
    for slots, want in (([0, 2, 4, 5], 0), ([0, 2, 0, 5], kda.STATUS_CODES["KDA_ERR_INVALID_ARG"]),
                        ([7, 2, 7, 5], 0)):   # 7 is outside the pool: padding rows, never a repeat
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        sl = torch.tensor(slots, dtype=torch.int32, device="cuda")
        kda.decode_paged(x["q"], x["k"], x["v"], x["g"], x["beta"], pool, sl, status=status)
        xm = {n: t[:, None].contiguous() for n, t in x.items()}
        status2 = torch.zeros(1, dtype=torch.int32, device="cuda")
        kda.decode_multi(xm["q"], xm["k"], xm["v"], xm["g"], xm["beta"], pool, slot_ids=sl, status=status2)
        torch.cuda.synchronize()
        assert int(status.item()) == want, slots
        assert int(status2.item()) == want, slots
