"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function include/kda.h declares, and rejects invalid calls on the host
before touching the device (no compute call is made here)."""
import ctypes
import os
import re

import pytest

from linear_attention_serving_k1_gb300 import build, kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    try:
        build.nvcc()
    except RuntimeError:
        pytest.skip("no CUDA toolkit to build the library")
    build.build()
    return kda.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(kda.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_debug_build_exports_the_same_abi(lib):
    """The bounds-checking debug build is built beside the library and exports
    the same functions (its checks run on the GPU: tests/test_gpu_debug.py)."""
    dbg = kda.load_debug_library()
    assert os.path.exists(build.debug_library_path())
    for n in declared_functions():
        assert hasattr(dbg, n), n
    assert dbg.kda_version() == lib.kda_version()
    assert kda.STATUS_CODES["KDA_ERR_BOUNDS"] == -7


def test_version(lib):
    assert lib.kda_version() >= 100


def _desc(**kw):
    raw_gate = kw.pop("raw_scalar_gate", None)
    d = dict(T=256, H=2, D=64, num_seqs=1, dtype_code=kda.DTYPE_FP32, chunk=64, ckpt_stride=0,
             ckpt_capacity=0)
    d.update(kw)
    desc = kda.make_desc(**d)
    if raw_gate is not None:   # a value the binding would not produce
        desc.scalar_gate = raw_gate
    return desc


def test_workspace_size(lib):
    n = lib.kda_prefill_workspace_size(ctypes.byref(_desc()))
    assert n > 0 and n % 256 == 0
    bigger = lib.kda_prefill_workspace_size(ctypes.byref(_desc(T=1024)))
    assert bigger > n


INVALID_DESCS = [
    (dict(D=96), -2), (dict(chunk=32), -2), (dict(num_seqs=0), -1), (dict(T=-1), -1),
    (dict(H=0), -1), (dict(dtype_code=7), -1), (dict(ckpt_stride=100), -1),
    (dict(max_seq_len=-1), -1), (dict(segment_chunks=-2), -1), (dict(raw_scalar_gate=2), -1),
]


@pytest.mark.parametrize("build_kind", ["release", "debug"])
@pytest.mark.parametrize("kw,code", INVALID_DESCS)
def test_invalid_desc(lib, build_kind, kw, code):
    """Refused on the host before anything is launched, the same way by the
    library and by its debug build."""
    if build_kind == "debug":
        lib = kda.load_debug_library()
    d = _desc(**kw)
    assert lib.kda_prefill_workspace_size(ctypes.byref(d)) == 0
    rc = lib.kda_prefill(*([ctypes.c_void_p(16)] * 7), ctypes.c_void_p(16), None, None,
                         ctypes.byref(d), ctypes.c_void_p(256), ctypes.c_size_t(1 << 30), None)
    assert rc == code
    assert lib.kda_last_error()


def test_segmented_workspace_is_bounded(lib):
    """The tensor-core path keeps a two-slot ring of records instead of every
    chunk's: for a long single sequence (131072 tokens, 32 heads) the automatic
    plan needs a fraction of the one-segment workspace, and a max_seq_len bound
    shrinks a many-sequence batch's need the same way."""
    long = dict(T=131072, H=32, D=128, dtype_code=kda.DTYPE_BF16)
    auto = lib.kda_prefill_workspace_size(ctypes.byref(_desc(**long)))
    whole = lib.kda_prefill_workspace_size(ctypes.byref(_desc(segment_chunks=1 << 20, **long)))
    record_bytes = 90624
    assert whole >= 2048 * 32 * record_bytes
    assert 0 < auto < whole // 4
    # explicit segment lengths: ring of 2 x G x H records plus a 64 KB state per
    # head, G raised to 2048 / 256 chunks (at most 256 segments)
    for G in (1, 4, 16):
        Ge = max(G, 2048 // 256)
        n = lib.kda_prefill_workspace_size(ctypes.byref(_desc(segment_chunks=G, **long)))
        assert n >= 2 * Ge * 32 * record_bytes + 32 * 128 * 128 * 4
        assert n < 2 * Ge * 32 * record_bytes + 32 * 128 * 128 * 4 + 8192


def test_workspace_grows_with_segment_length(lib):
    """kda_prefill_noalloc's fallback searches for the longest segments that
    fit its array by bisection: below a sequence's chunk count the workspace
    must not shrink as segment_chunks grows. Checked over batch shapes of the
    tensor-core path, with and without a max_seq_len bound."""
    for T, N, H, L in ((2048, 1, 32, 0), (8192, 4, 8, 0), (70000, 16, 4, 8192), (131072, 1, 2, 0)):
        maxc = -(-(L or T) // 64)
        prev = 0
        for G in sorted({1, 2, 3, 5, 8, 13, 21, 34, 55, 89, 144, 233, maxc // 2, maxc - 1}):
            if not 1 <= G < maxc:
                continue
            d = _desc(T=T, num_seqs=N, H=H, D=128, dtype_code=kda.DTYPE_BF16, max_seq_len=L, segment_chunks=G)
            n = lib.kda_prefill_workspace_size(ctypes.byref(d))
            assert n > 0 and n >= prev, (T, N, H, G, n, prev)
            prev = n
            assert lib.kda_prefill_launch_count(ctypes.byref(d)) <= 1 + 2 * 256


def test_launch_count(lib):
    """Three launches without segments (table, K1, K2); 1 + 2 x segments with."""
    assert lib.kda_prefill_launch_count(ctypes.byref(_desc())) == 3
    long = dict(T=131072, H=32, D=128, dtype_code=kda.DTYPE_BF16)
    assert lib.kda_prefill_launch_count(ctypes.byref(_desc(segment_chunks=1 << 20, **long))) == 3
    assert lib.kda_prefill_launch_count(ctypes.byref(_desc(segment_chunks=512, **long))) == 1 + 2 * 4
    assert lib.kda_prefill_launch_count(ctypes.byref(_desc(segment_chunks=500, **long))) == 1 + 2 * 5
    assert lib.kda_prefill_launch_count(ctypes.byref(_desc(H=0))) == -1
    # automatic plan: segments of whole K1 waves, 4 on all SMs first, a 2-wave
    # tail: workload 2 (8192 tokens x 32 heads) -> 38, 45, 30, 15 chunks;
    # workload 4 (131072 tokens) -> 21 segments
    assert lib.kda_prefill_launch_count(ctypes.byref(_desc(T=8192, H=32, D=128, dtype_code=kda.DTYPE_BF16))) == 1 + 2 * 4
    assert lib.kda_prefill_launch_count(ctypes.byref(_desc(**long))) == 1 + 2 * 21


def test_prefill_rejects_before_launch(lib):
    d = _desc()
    ws = lib.kda_prefill_workspace_size(ctypes.byref(d))
    p = ctypes.c_void_p(4096)
    # NULL q
    assert lib.kda_prefill(None, p, p, p, p, None, None, ctypes.c_void_p(8192), None, None,
                           ctypes.byref(d), ctypes.c_void_p(1 << 20), ws, None) == -1
    # workspace too small / misaligned / missing
    assert lib.kda_prefill(p, p, p, p, p, None, None, ctypes.c_void_p(8192), None, None,
                           ctypes.byref(d), ctypes.c_void_p(1 << 20), ws - 1, None) == -5
    assert lib.kda_prefill(p, p, p, p, p, None, None, ctypes.c_void_p(8192), None, None,
                           ctypes.byref(d), ctypes.c_void_p((1 << 20) + 8), ws, None) == -5
    assert lib.kda_prefill(p, p, p, p, p, None, None, ctypes.c_void_p(8192), None, None,
                           ctypes.byref(d), None, ws, None) == -5
    # out aliasing q
    assert lib.kda_prefill(p, ctypes.c_void_p(8192), p, p, p, None, None, p, None, None,
                           ctypes.byref(d), ctypes.c_void_p(1 << 20), ws, None) == -1
    # equal-length batch that does not divide
    d2 = _desc(T=255, num_seqs=2)
    ws2 = lib.kda_prefill_workspace_size(ctypes.byref(d2))
    assert lib.kda_prefill(p, p, p, p, p, None, None, ctypes.c_void_p(8192), None, None,
                           ctypes.byref(d2), ctypes.c_void_p(1 << 20), ws2, None) == -1
    # checkpoints requested with capacity but no buffer
    d3 = _desc(ckpt_stride=64, ckpt_capacity=4)
    ws3 = lib.kda_prefill_workspace_size(ctypes.byref(d3))
    assert lib.kda_prefill(p, p, p, p, p, None, None, ctypes.c_void_p(8192), None, None,
                           ctypes.byref(d3), ctypes.c_void_p(1 << 20), ws3, None) == -1


def test_decode_rejects_before_launch(lib):
    p = ctypes.c_void_p(4096)
    o = ctypes.c_void_p(8192)
    assert lib.kda_decode(p, p, p, p, p, p, o, 2, 2, 64, 128, 0, None) == -2    # Dk != Dv
    assert lib.kda_decode(p, p, p, p, p, p, o, 2, 2, 96, 96, 0, None) == -2     # head dim
    assert lib.kda_decode(p, p, p, p, p, p, o, -1, 2, 64, 64, 0, None) == -1    # N < 0
    assert lib.kda_decode(None, p, p, p, p, p, o, 2, 2, 64, 64, 0, None) == -1  # NULL q
    assert lib.kda_decode(p, p, p, p, p, ctypes.c_void_p(4100), o, 2, 2, 64, 64, 0, None) == -1  # misaligned state
    assert lib.kda_decode(p, p, p, p, p, p, p, 2, 2, 64, 64, 0, None) == -1     # out aliases q
    assert lib.kda_decode(p, p, p, p, p, p, o, 2, 2, 64, 64, 5, None) == -1     # dtype
    assert lib.kda_decode(p, p, p, p, p, p, o, 0, 2, 64, 64, 0, None) == 0      # empty: nothing to do


def test_decode_paged_rejects_before_launch(lib):
    p = ctypes.c_void_p(4096)
    args = [p] * 6
    # NULL slot ids with rows to decode
    assert lib.kda_decode_paged(*args, ctypes.c_int64(8), None, ctypes.c_void_p(8192), 2, 2, 128, 128,
                                kda.DTYPE_BF16, None, None) == -1
    # negative pool size
    assert lib.kda_decode_paged(*args, ctypes.c_int64(-1), p, ctypes.c_void_p(8192), 2, 2, 128, 128,
                                kda.DTYPE_BF16, None, None) == -1
    # unsupported head dim
    assert lib.kda_decode_paged(*args, ctypes.c_int64(8), p, ctypes.c_void_p(8192), 2, 2, 96, 96,
                                kda.DTYPE_BF16, None, None) == -2
    # nothing to do
    assert lib.kda_decode_paged(*args, ctypes.c_int64(8), None, ctypes.c_void_p(8192), 0, 2, 128, 128,
                                kda.DTYPE_BF16, None, None) == 0


def test_fused_and_pooled_reject_before_launch(lib):
    p = ctypes.c_void_p(4096)
    d = _desc(T=128, H=2, D=128, dtype_code=kda.DTYPE_BF16)
    ws = lib.kda_prefill_workspace_size(ctypes.byref(d))
    o = ctypes.c_void_p(8192)
    # taps given without a width
    assert lib.kda_prefill_fused(p, p, p, p, p, None, None, o, None, None, p, None, None, None, ctypes.byref(d),
                                 ctypes.c_void_p(1 << 20), ws, None) == kda.STATUS_CODES["KDA_ERR_INVALID_ARG"]
    # a convolution state without taps
    assert lib.kda_prefill_fused(p, p, p, p, p, None, None, o, None, None, None, p, None, None, ctypes.byref(d),
                                 ctypes.c_void_p(1 << 20), ws, None) == kda.STATUS_CODES["KDA_ERR_INVALID_ARG"]
    # fused decode: width out of range, state without taps
    assert lib.kda_decode_fused(p, p, p, p, p, p, None, p, None, o, 2, 2, 128, 128, kda.DTYPE_BF16, 5, 0,
                                None) == kda.STATUS_CODES["KDA_ERR_UNSUPPORTED"]
    assert lib.kda_decode_fused(p, p, p, p, p, p, p, None, None, o, 2, 2, 128, 128, kda.DTYPE_BF16, 0, 0,
                                None) == kda.STATUS_CODES["KDA_ERR_INVALID_ARG"]
    # width beyond the supported four taps
    d5 = _desc(T=128, H=2, D=128, dtype_code=kda.DTYPE_BF16, conv_width=5)
    assert lib.kda_prefill_workspace_size(ctypes.byref(d5)) == 0
    # the gate may not alias the output
    assert lib.kda_prefill_fused(p, p, p, p, p, None, None, o, None, None, None, None, None, o, ctypes.byref(d),
                                 ctypes.c_void_p(1 << 20), ws, None) == kda.STATUS_CODES["KDA_ERR_INVALID_ARG"]
    # pooled: slot tables without a pool; checkpoints without their slot table
    assert lib.kda_prefill_pooled(p, p, p, p, p, None, o, None, ctypes.c_int64(4), p, None, None,
                                  ctypes.byref(d), ctypes.c_void_p(1 << 20), ws, None) == -1
    dc = _desc(T=128, H=2, D=128, dtype_code=kda.DTYPE_BF16, ckpt_stride=64, ckpt_capacity=2)
    wsc = lib.kda_prefill_workspace_size(ctypes.byref(dc))
    assert lib.kda_prefill_pooled(p, p, p, p, p, None, o, p, ctypes.c_int64(4), None, None, None,
                                  ctypes.byref(dc), ctypes.c_void_p(1 << 20), wsc, None) == -1
