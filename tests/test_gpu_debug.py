"""The bounds-checking debug build (libkda_debug.so, the kernels compiled with
KDA_DEBUG): on valid calls it gives the release build's results bit for bit
and reports nothing; when its checks take the token buffers to be shorter than
the call says (KDA_DEBUG_CLIP_TOKENS, the memory behind them still there), it
skips the accesses past the declared end, returns KDA_ERR_BOUNDS with the
index and the extent, and the next call on the same context is clean."""
import pytest
import torch

from kda_parity import gpu_inputs
from linear_attention_serving_k1_gb300 import kda, workloads

pytestmark = pytest.mark.gpu

LENS = [1, 63, 64, 65, 130, 200]
BOUNDS = kda.STATUS_CODES["KDA_ERR_BOUNDS"]


@pytest.fixture(scope="module")
def dbg():
    return kda.load_debug_library()


def _prefill_inputs(dtype, D, lens, seed, H=2):
    w = workloads.custom_prefill(H=H, D=D, lens=lens, dtype=dtype, init="randn", ckpt_stride=64, seed=seed,
                                 varlen=True)
    return w, gpu_inputs(workloads.make_prefill(w))


def _both(dbg, fn):
    """fn() with the release library, then with the debug build."""
    a = fn()
    with kda.using_library(dbg):
        b = fn()
    torch.cuda.synchronize()
    return a, b


def _equal(a, b):
    if isinstance(a, (tuple, list)):
        return all(_equal(x, y) for x, y in zip(a, b))
    return (a is None and b is None) or torch.equal(a, b)


@pytest.mark.parametrize("dtype,D,seg,rctas", [("bf16", 128, 0, 0), ("bf16", 128, 2, 0), ("bf16", 128, 2, 3),
                                               ("fp32", 64, 0, 0)])
def test_prefill_bit_identical_to_release(dbg, dtype, D, seg, rctas):
    w, d = _prefill_inputs(dtype, D, LENS, seed=201)
    cap = kda.num_checkpoints(w.lens, 64)
    fn = lambda: kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                             ckpt_stride=64, ckpt_capacity=cap, segment_chunks=seg, recurrence_ctas=rctas)
    a, b = _both(dbg, fn)
    assert _equal(a, b)


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp32", 64)])
def test_fused_and_pooled_prefill_bit_identical_to_release(dbg, dtype, D):
    w, d = _prefill_inputs(dtype, D, LENS, seed=202)
    gen = torch.Generator().manual_seed(203)
    taps = (torch.rand(3, 4, 2, D, generator=gen) * 2.0 - 1.0).cuda()
    z = torch.randn(w.total_tokens, 2, D, generator=gen).to(d["q"].dtype).cuda()
    N = w.num_seqs
    cs = torch.empty(N, 3, 3, 2, D, dtype=d["q"].dtype, device="cuda")
    fused = lambda: kda.prefill_fused(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                                      conv_w=taps, conv_silu=True, gate=z, conv_state_out=cs) + (cs.clone(),)
    a, b = _both(dbg, fused)
    assert _equal(a, b)
    # the pool: initial states in slots 2N-1 .. N, finals in slots 0 .. N-1, one padding entry
    P = 2 * N
    pool0 = 0.05 * torch.randn(P, 2, D, D, generator=gen)
    init_slots = torch.arange(2 * N - 1, N - 1, -1, dtype=torch.int32)
    init_slots[1] = -1
    final_slots = torch.arange(N, dtype=torch.int32)

    def pooled():
        pool = pool0.cuda()
        out = kda.prefill_pooled(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, init_slots.cuda(),
                                 final_slots.cuda(), d["cu_seqlens"])
        return out, pool

    a, b = _both(dbg, pooled)
    assert _equal(a, b)


@pytest.mark.parametrize("D,dtype", [(128, torch.bfloat16), (64, torch.float32)])
def test_decode_bit_identical_to_release(dbg, D, dtype):
    gen = torch.Generator().manual_seed(204)
    N, m, H, P = 5, 3, 2, 7
    mk = lambda *s: torch.randn(*s, generator=gen).to(dtype).cuda()
    q, k, v = mk(N, m, H, D), mk(N, m, H, D), mk(N, m, H, D)
    g = (-torch.exp(torch.empty(N, m, H, D).uniform_(-5, -1, generator=gen))).cuda()
    beta = torch.sigmoid(torch.randn(N, m, H, generator=gen)).cuda()
    s0 = (0.05 * torch.randn(P, H, D, D, generator=gen)).cuda()
    slots = torch.tensor([3, 0, -1, 6, 2], dtype=torch.int32).cuda()
    commit = torch.tensor([0, 2, 3, 1, 3], dtype=torch.int32).cuda()
    taps = (torch.rand(3, 4, H, D, generator=gen) * 2.0 - 1.0).cuda()
    z = mk(N, H, D)
    t0 = lambda x: x[:, 0].contiguous()

    def run():
        st1, st2, st3, st4 = s0[:N].clone(), s0.clone(), s0.clone(), s0[:N].clone()
        cs = torch.zeros(N, 3, 3, H, D, dtype=dtype, device="cuda")
        o1 = kda.decode(t0(q), t0(k), t0(v), t0(g), t0(beta), st1)
        o2 = kda.decode_paged(t0(q), t0(k), t0(v), t0(g), t0(beta), st2, slots)
        o3 = kda.decode_multi(q, k, v, g, beta, st3, commit, slot_ids=slots)
        o4 = kda.decode_fused(t0(q), t0(k), t0(v), t0(g), t0(beta), st4, conv_w=taps, conv_state=cs, gate=z)
        return o1, o2, o3, o4, st1, st2, st3, st4, cs

    a, b = _both(dbg, run)
    assert _equal(a, b)


def _nan_like(t):
    return torch.full_like(t, float("nan"))


@pytest.mark.parametrize("dtype,D,seg", [("bf16", 128, 0), ("bf16", 128, 1), ("fp32", 64, 0)])
def test_clipped_token_rows_are_reported_and_skipped(dbg, monkeypatch, dtype, D, seg):
    """The checks take q, k, v, g, beta and out to end one row early: the
    call reports that row, leaves its output unwritten (the NaN it held), and
    the sequences before it come out as in the release build."""
    w, d = _prefill_inputs(dtype, D, [70, 125], seed=205)
    T = w.total_tokens
    ref, _, _ = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                            segment_chunks=seg)
    out = _nan_like(ref)
    monkeypatch.setenv("KDA_DEBUG_CLIP_TOKENS", "1")
    with kda.using_library(dbg):
        with pytest.raises(kda.KDAError) as ei:
            kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"], out=out,
                        segment_chunks=seg)
    torch.cuda.synchronize()
    assert ei.value.code == BOUNDS
    assert f"token row index {T - 1} outside [0, {T - 1})" in str(ei.value)
    assert torch.isnan(out[T - 1].float()).all()
    assert torch.equal(out[:70], ref[:70])
    # the same context, the variable gone: a clean call, as the release build
    monkeypatch.delenv("KDA_DEBUG_CLIP_TOKENS")
    with kda.using_library(dbg):
        again, _, _ = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                                  segment_chunks=seg)
    torch.cuda.synchronize()
    assert torch.equal(again, ref)


@pytest.mark.parametrize("D,dtype", [(128, torch.bfloat16), (64, torch.float32)])
def test_clipped_decode_rows_are_reported_and_skipped(dbg, monkeypatch, D, dtype):
    """Decode with the last sequence's row past the declared end: its output
    and its state are left as they were; the other sequences step as in the
    release build."""
    gen = torch.Generator().manual_seed(206)
    N, H = 4, 2
    mk = lambda *s: torch.randn(*s, generator=gen).to(dtype).cuda()
    q, k, v = mk(N, H, D), mk(N, H, D), mk(N, H, D)
    g = (-torch.exp(torch.empty(N, H, D).uniform_(-5, -1, generator=gen))).cuda()
    beta = torch.sigmoid(torch.randn(N, H, generator=gen)).cuda()
    s0 = (0.05 * torch.randn(N, H, D, D, generator=gen)).cuda()
    st_ref = s0.clone()
    ref = kda.decode(q, k, v, g, beta, st_ref)
    st = s0.clone()
    out = _nan_like(ref)
    monkeypatch.setenv("KDA_DEBUG_CLIP_TOKENS", "1")
    with kda.using_library(dbg):
        with pytest.raises(kda.KDAError) as ei:
            kda.decode(q, k, v, g, beta, st, out=out)
    torch.cuda.synchronize()
    assert ei.value.code == BOUNDS
    assert f"token row index {N - 1} outside [0, {N - 1})" in str(ei.value)
    assert torch.isnan(out[N - 1].float()).all()
    assert torch.equal(st[N - 1], s0[N - 1])
    assert torch.equal(out[:N - 1], ref[:N - 1])
    assert torch.equal(st[:N - 1], st_ref[:N - 1])
    monkeypatch.delenv("KDA_DEBUG_CLIP_TOKENS")
    st2 = s0.clone()
    with kda.using_library(dbg):
        again = kda.decode(q, k, v, g, beta, st2)
    torch.cuda.synchronize()
    assert torch.equal(again, ref) and torch.equal(st2, st_ref)
