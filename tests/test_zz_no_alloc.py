"""kda_prefill_noalloc: the prefill for callers that cannot allocate device
memory (its scratch is an array built into the library).  Checked through the
C ABI against kda_prefill, which takes a caller workspace, on two calls in a
row (the array keeps the first call's contents).

Collected last on purpose (file name), so that a run stopping at the first
failure has run every other test first.  It must pass alone in a fresh
process as well as after the other tests."""
import ctypes

import pytest
import torch

from kda_parity import TOL_OUT_BF16, TOL_OUT_FP32, TOL_STATE, gpu_inputs, out_err, state_err, to_np
from linear_attention_serving_k1_gb300 import kda, workloads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,D,lens,stride", [
    ("bf16", 128, [100, 200], 64),     # tensor-core path
    ("fp32", 64, [65, 130, 1], 64),    # CUDA-core path
])
def test_noalloc_matches_workspace_prefill_twice(dtype, D, lens, stride):
    tol = TOL_OUT_FP32 if dtype == "fp32" else TOL_OUT_BF16
    for seed in (31, 32):   # two calls in a row, different inputs
        w = workloads.custom_prefill(H=3, D=D, lens=lens, dtype=dtype, init="randn", ckpt_stride=stride,
                                     seed=seed, varlen=True)
        d = gpu_inputs(workloads.make_prefill(w))
        cap = kda.num_checkpoints(w.lens, stride)
        o_ref, f_ref, ck_ref = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                                           d["cu_seqlens"], ckpt_stride=stride, ckpt_capacity=cap)
        o, f, ck = kda.prefill_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                                       d["cu_seqlens"], ckpt_stride=stride, ckpt_capacity=cap)
        torch.cuda.synchronize()
        assert out_err(to_np(o), to_np(o_ref)) <= tol
        assert state_err(to_np(f), to_np(f_ref)) <= TOL_STATE
        assert state_err(to_np(ck), to_np(ck_ref)) <= TOL_STATE


@pytest.mark.parametrize("segment_chunks", [1, 2])
def test_noalloc_segmented_is_bit_identical(segment_chunks):
    """With an explicit segment length the call runs the segmented plan: the
    two-slot record ring and the fp32 carry between segments then live in the
    built-in array too.  Two calls in a row, compared bit for bit with
    kda_prefill at the same segment length."""
    for seed in (33, 34):
        w = workloads.custom_prefill(H=3, D=128, lens=[300, 0, 129, 64], dtype="bf16", init="randn",
                                     ckpt_stride=64, seed=seed, varlen=True)
        d = gpu_inputs(workloads.make_prefill(w))
        cap = kda.num_checkpoints(w.lens, 64)
        desc = kda.make_desc(w.total_tokens, 3, 128, w.num_seqs, kda.DTYPE_BF16, 64, 64, cap,
                             segment_chunks=segment_chunks)
        assert kda.workspace_size(desc) <= kda.NOALLOC_SCRATCH_BYTES
        assert kda.launch_count(desc) > 3   # more than one segment
        o_ref, f_ref, ck_ref = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                                           d["cu_seqlens"], ckpt_stride=64, ckpt_capacity=cap,
                                           segment_chunks=segment_chunks)
        o, f, ck = kda.prefill_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                                       d["cu_seqlens"], ckpt_stride=64, ckpt_capacity=cap,
                                       segment_chunks=segment_chunks)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref)
        assert torch.equal(f, f_ref)
        assert torch.equal(ck, ck_ref)


def test_noalloc_takes_shorter_segments_when_the_automatic_plan_does_not_fit():
    """One sequence of 2,048 tokens at 32 heads: the automatic plan (one
    segment, every record) needs about 96 MB, more than the built-in array,
    while segments of 5 chunks fit; the call takes the longest segments that
    fit and matches kda_prefill bit for bit (results do not depend on the
    segment length)."""
    w = workloads.custom_prefill(H=32, D=128, lens=[2048], dtype="bf16", init="randn", ckpt_stride=512, seed=35,
                                 varlen=True)
    d = gpu_inputs(workloads.make_prefill(w))
    cap = kda.num_checkpoints(w.lens, 512)
    desc = kda.make_desc(2048, 32, 128, 1, kda.DTYPE_BF16, 64, 512, cap)
    assert kda.workspace_size(desc) > kda.NOALLOC_SCRATCH_BYTES
    fit = kda.make_desc(2048, 32, 128, 1, kda.DTYPE_BF16, 64, 512, cap, segment_chunks=5)
    assert kda.workspace_size(fit) <= kda.NOALLOC_SCRATCH_BYTES
    o_ref, f_ref, ck_ref = kda.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"],
                                       d["cu_seqlens"], ckpt_stride=512, ckpt_capacity=cap)
    o, f, ck = kda.prefill_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d["init_state"], d["cu_seqlens"],
                                   ckpt_stride=512, ckpt_capacity=cap)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref)
    assert torch.equal(f, f_ref)
    assert torch.equal(ck, ck_ref)


def test_noalloc_rejects_calls_beyond_its_scratch():
    """About 1M tokens of one sequence at 32 heads fit no plan: every segment
    length is raised to at least 65 chunks (256 segments at most), and two ring
    slots of 65 chunks of 32 heads already need about 377 MB."""
    lib = kda.load_library()
    T = 1 << 20   # about 1M tokens x 32 heads needs far more than the built-in array
    desc = kda.make_desc(T, 32, 128, 1, kda.DTYPE_BF16)
    assert kda.workspace_size(desc) > kda.NOALLOC_SCRATCH_BYTES
    p = ctypes.c_void_p(4096)
    rc = lib.kda_prefill_noalloc(p, p, p, p, p, None, None, ctypes.c_void_p(8192), None, None,
                                 ctypes.byref(desc), None)
    assert rc == kda.STATUS_CODES["KDA_ERR_UNSUPPORTED"]
    assert b"scratch" in lib.kda_last_error()
