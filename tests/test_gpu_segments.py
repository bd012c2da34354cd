"""Segmented tensor-core prefill: the preparation of segment s + 1 overlaps the
recurrence over segment s, records pass through a two-slot ring and the state
through an fp32 carry.  The segment length is a tuning knob only, so every
choice must give bit-identical outputs, states and checkpoints; one choice is
also checked against the float64 oracle."""
import pytest
import torch

from kda_parity import TOL_OUT_BF16, TOL_STATE, gpu_inputs, out_err, run_oracle_prefill, state_err, to_np
from linear_attention_serving_k1_gb300 import kda, workloads

pytestmark = pytest.mark.gpu

LENS = [1, 63, 64, 65, 127, 130, 256, 700, 0, 129]


def _run(d, w, ckpt_stride=0, **kw):
    cap = kda.num_checkpoints(w.lens, ckpt_stride)
    o, f, ck = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                           num_seqs=w.num_seqs, ckpt_stride=ckpt_stride,
                           ckpt_capacity=cap if ckpt_stride else None, **kw)
    torch.cuda.synchronize()
    return o, f, (ck[:cap] if ck is not None else None)


def test_segment_length_does_not_change_results():
    w = workloads.custom_prefill(H=3, D=128, lens=LENS, dtype="bf16", init="randn", ckpt_stride=64,
                                 seed=31, varlen=True)
    inp = workloads.make_prefill(w)
    d = gpu_inputs(inp)
    o0, f0, c0 = _run(d, w, ckpt_stride=64)
    for G in (1, 2, 3, 5, 11):
        o, f, c = _run(d, w, ckpt_stride=64, segment_chunks=G)
        assert torch.equal(o, o0), f"outputs differ at segment_chunks={G}"
        assert torch.equal(f, f0), f"final states differ at segment_chunks={G}"
        assert torch.equal(c, c0), f"checkpoints differ at segment_chunks={G}"
    o_r, f_r, c_r = run_oracle_prefill(inp, ckpt_stride=64)
    assert out_err(to_np(o), o_r) <= TOL_OUT_BF16
    assert state_err(to_np(f), f_r) <= TOL_STATE
    assert state_err(to_np(c), c_r) <= TOL_STATE


def test_max_seq_len_bound_is_enforced():
    """A sequence longer than max_seq_len is reported; a sufficient bound is fine."""
    w = workloads.custom_prefill(H=2, D=128, lens=[64, 300], dtype="bf16", init="randn", seed=32, varlen=True)
    inp = workloads.make_prefill(w)
    d = gpu_inputs(inp)
    T = sum(w.lens)
    for bound, expect in ((128, "KDA_ERR_INVALID_ARG"), (300, None), (320, None)):
        desc = kda.make_desc(T, 2, 128, 2, kda.DTYPE_BF16, max_seq_len=bound, segment_chunks=1)
        ws = kda.alloc_workspace(desc, "cuda")
        o, f, _ = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                              workspace=ws, max_seq_len=bound, segment_chunks=1)
        st = kda.prefill_status(ws)
        if expect is None:
            assert st == 0
            o_r, f_r, _ = run_oracle_prefill(inp)
            assert out_err(to_np(o), o_r) <= TOL_OUT_BF16
            assert state_err(to_np(f), f_r) <= TOL_STATE
        else:
            assert st == kda.STATUS_CODES[expect]


def test_segmented_final_state_may_alias_initial_state():
    w = workloads.custom_prefill(H=2, D=128, lens=[200, 0, 333], dtype="bf16", init="randn", seed=33,
                                 varlen=True)
    inp = workloads.make_prefill(w)
    d = gpu_inputs(inp)
    _, f_ref, _ = _run(d, w, segment_chunks=2)
    s = d["init_state"].clone()
    kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], s, d["cu_seqlens"], final_state=s,
                segment_chunks=2)
    torch.cuda.synchronize()
    assert torch.equal(s, f_ref)


def test_segmented_prefill_in_cuda_graph():
    """The two-stream fork/join is legal inside a stream capture and the graph
    replays the same results."""
    w = workloads.custom_prefill(H=4, D=128, lens=[640], dtype="bf16", init="randn", seed=34)
    inp = workloads.make_prefill(w)
    d = gpu_inputs(inp)
    o_ref, f_ref, _ = _run(d, w, segment_chunks=3)
    T = 640
    desc = kda.make_desc(T, 4, 128, 1, kda.DTYPE_BF16, segment_chunks=3)
    ws = kda.alloc_workspace(desc, "cuda")
    out = torch.empty_like(d["q"])
    fin = torch.empty_like(d["init_state"])
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], None)
    kw = dict(out=out, final_state=fin, workspace=ws, segment_chunks=3)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        kda.prefill(*args, stream=s, **kw)          # warm-up (creates the side stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        kda.prefill(*args, stream=s, **kw)
    out.zero_()
    fin.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, o_ref)
    assert torch.equal(fin, f_ref)


def test_many_chains_persistent_recurrence():
    """More chains (sequences x heads) than the one-CTA-per-chain plan takes:
    with segments, the recurrence runs on a small grid whose CTAs take chains
    one after another (barrier phases and ring positions carried across
    chains).  Every segment length gives the same bytes as one segment, and
    the oracle agrees."""
    lens = [1, 700, 0, 64, 65, 300, 130, 1000]
    w = workloads.custom_prefill(H=16, D=128, lens=lens, dtype="bf16", init="randn", ckpt_stride=64,
                                 seed=35, varlen=True)
    inp = workloads.make_prefill(w)
    d = gpu_inputs(inp)
    assert w.num_seqs * w.H > 96
    o0, f0, c0 = _run(d, w, ckpt_stride=64, segment_chunks=1 << 20)
    for G in (1, 2, 3, 5):
        o, f, c = _run(d, w, ckpt_stride=64, segment_chunks=G, max_seq_len=max(lens))
        assert torch.equal(o, o0), f"outputs differ at segment_chunks={G}"
        assert torch.equal(f, f0), f"final states differ at segment_chunks={G}"
        assert torch.equal(c, c0), f"checkpoints differ at segment_chunks={G}"
    o_r, f_r, c_r = run_oracle_prefill(inp, ckpt_stride=64)
    assert out_err(to_np(o0), o_r) <= TOL_OUT_BF16
    assert state_err(to_np(f0), f_r) <= TOL_STATE
    assert state_err(to_np(c0), c_r) <= TOL_STATE
