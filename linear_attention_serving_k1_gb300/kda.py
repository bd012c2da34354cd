"""Thin Python binding of the C ABI in include/kda.h (argument marshalling only).

Every step of the computation runs in the CUDA kernels of ``_build/libkda.so``
(or, inside ``using_library(load_debug_library())``, of its bounds-checking
debug build); PyTorch only provides device memory and the current stream.
There is no CPU fallback: if the library is missing or no GPU is present,
calls raise.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional

import torch

from . import build as _build

KDA_OK = 0
STATUS_NAMES = {0: "KDA_OK", -1: "KDA_ERR_INVALID_ARG", -2: "KDA_ERR_UNSUPPORTED", -3: "KDA_ERR_CUDA",
                -4: "KDA_ERR_CKPT_OVERFLOW", -5: "KDA_ERR_WORKSPACE", -6: "KDA_ERR_TIMEOUT",
                -7: "KDA_ERR_BOUNDS"}
STATUS_CODES = {v: k for k, v in STATUS_NAMES.items()}
DTYPE_BF16, DTYPE_FP32 = 0, 1

# Every symbol include/kda.h declares.
EXPORTS = ("kda_prefill_workspace_size", "kda_prefill_launch_count", "kda_prefill", "kda_prefill_status",
           "kda_prefill_pooled", "kda_prefill_fused", "kda_decode", "kda_decode_fused", "kda_decode_paged",
           "kda_decode_multi", "kda_prefill_noalloc", "kda_last_error", "kda_version")

# Size of the library's built-in scratch array used by kda_prefill_noalloc.
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


class KDAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class PrefillDesc(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int64),
                ("num_heads", ctypes.c_int32), ("head_dim_k", ctypes.c_int32),
                ("head_dim_v", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("chunk", ctypes.c_int32), ("ckpt_stride", ctypes.c_int32),
                ("ckpt_capacity", ctypes.c_int64), ("max_seq_len", ctypes.c_int64),
                ("segment_chunks", ctypes.c_int32), ("scalar_gate", ctypes.c_int32),
                ("recurrence_ctas", ctypes.c_int32), ("conv_width", ctypes.c_int32),
                ("conv_silu", ctypes.c_int32), ("wait_limit", ctypes.c_uint32)]


_lib = None
_vp = ctypes.c_void_p


def default_library_path() -> str:
    """libkda.so, or its bounds-checking debug build when the environment
    variable KDA_LIBRARY is "debug" (every call of the binding then runs with
    the index checks, and one that fails raises KDAError KDA_ERR_BOUNDS)."""
    if os.environ.get("KDA_LIBRARY", "") == "debug":
        return _build.debug_library_path()
    return _build.library_path()


def load_library(path: Optional[str] = None):
    """Load the library (default_library_path() unless `path` is given; raises
    if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or default_library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with linear_attention_serving_k1_gb300.build.build()")
    lib = ctypes.CDLL(path)
    lib.kda_prefill_workspace_size.restype = ctypes.c_size_t
    lib.kda_prefill_workspace_size.argtypes = [ctypes.POINTER(PrefillDesc)]
    lib.kda_prefill_launch_count.restype = ctypes.c_int32
    lib.kda_prefill_launch_count.argtypes = [ctypes.POINTER(PrefillDesc)]
    lib.kda_prefill.restype = ctypes.c_int
    lib.kda_prefill.argtypes = [_vp] * 10 + [ctypes.POINTER(PrefillDesc), _vp, ctypes.c_size_t, _vp]
    lib.kda_prefill_status.restype = ctypes.c_int
    lib.kda_prefill_status.argtypes = [_vp, _vp]
    lib.kda_decode.restype = ctypes.c_int
    lib.kda_decode.argtypes = [_vp] * 7 + [ctypes.c_int32] * 5 + [_vp]
    lib.kda_prefill_fused.restype = ctypes.c_int
    lib.kda_prefill_fused.argtypes = [_vp] * 14 + [ctypes.POINTER(PrefillDesc), _vp, ctypes.c_size_t, _vp]
    lib.kda_decode_fused.restype = ctypes.c_int
    lib.kda_decode_fused.argtypes = [_vp] * 10 + [ctypes.c_int32] * 7 + [_vp]
    lib.kda_prefill_pooled.restype = ctypes.c_int
    lib.kda_prefill_pooled.argtypes = [_vp] * 8 + [ctypes.c_int64, _vp, _vp, _vp, ctypes.POINTER(PrefillDesc),
                                                   _vp, ctypes.c_size_t, _vp]
    lib.kda_decode_paged.restype = ctypes.c_int
    lib.kda_decode_paged.argtypes = [_vp] * 6 + [ctypes.c_int64, _vp, _vp] + [ctypes.c_int32] * 5 + [_vp, _vp]
    lib.kda_decode_multi.restype = ctypes.c_int
    lib.kda_decode_multi.argtypes = ([_vp] * 6 + [ctypes.c_int64, _vp, _vp, _vp] + [ctypes.c_int32] * 6 +
                                     [_vp, _vp])
    lib.kda_prefill_noalloc.restype = ctypes.c_int
    lib.kda_prefill_noalloc.argtypes = [_vp] * 10 + [ctypes.POINTER(PrefillDesc), _vp]
    lib.kda_last_error.restype = ctypes.c_char_p
    lib.kda_last_error.argtypes = []
    lib.kda_version.restype = ctypes.c_int32
    lib.kda_version.argtypes = []
    if path == default_library_path():
        _lib = lib
    return lib


def load_debug_library():
    """Load the debug build libkda_debug.so (same ABI; every data-dependent
    global index checked, failures returned as KDA_ERR_BOUNDS)."""
    return load_library(_build.debug_library_path())


@contextlib.contextmanager
def using_library(lib):
    """Route this module's calls to `lib` (for example the debug build) inside
    the block."""
    global _lib
    prev = load_library()
    _lib = lib
    try:
        yield lib
    finally:
        _lib = prev


def _check(code: int):
    if code != KDA_OK:
        raise KDAError(code, load_library().kda_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to the KDA library must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the KDA library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_FP32
    raise ValueError(f"q/k/v must be bf16 or fp32, got {t.dtype}")


def make_desc(T: int, H: int, D: int, num_seqs: int, dtype_code: int, chunk: int = 64,
              ckpt_stride: int = 0, ckpt_capacity: int = 0, max_seq_len: int = 0,
              segment_chunks: int = 0, scalar_gate: bool = False, wait_limit: int = 0,
              recurrence_ctas: int = 0, conv_width: int = 0, conv_silu: bool = False) -> PrefillDesc:
    return PrefillDesc(num_seqs, T, H, D, D, dtype_code, chunk, ckpt_stride, ckpt_capacity,
                       max_seq_len, segment_chunks, int(bool(scalar_gate)), recurrence_ctas, conv_width,
                       int(bool(conv_silu)), wait_limit)


def workspace_size(desc: PrefillDesc) -> int:
    n = load_library().kda_prefill_workspace_size(ctypes.byref(desc))
    if n == 0:
        raise KDAError(-1, load_library().kda_last_error().decode())
    return int(n)


def launch_count(desc: PrefillDesc) -> int:
    """Kernel launches one ``kda_prefill`` call with ``desc`` enqueues."""
    n = load_library().kda_prefill_launch_count(ctypes.byref(desc))
    if n < 0:
        raise KDAError(-1, load_library().kda_last_error().decode())
    return int(n)


def alloc_workspace(desc: PrefillDesc, device) -> torch.Tensor:
    return torch.empty(workspace_size(desc), dtype=torch.uint8, device=device)


def num_checkpoints(lens, ckpt_stride: int) -> int:
    return 0 if ckpt_stride <= 0 else int(sum(int(L) // ckpt_stride for L in lens))


def prefill(q, k, v, g, beta, init_state=None, cu_seqlens=None, *, num_seqs: Optional[int] = None,
            chunk: int = 64, ckpt_stride: int = 0, ckpts=None, ckpt_capacity: Optional[int] = None,
            out=None, final_state=None, workspace=None, stream=None, want_final: bool = True,
            max_seq_len: int = 0, segment_chunks: int = 0, wait_limit: int = 0, recurrence_ctas: int = 0):
    """Chunked KDA prefill through ``kda_prefill``.

    q, k: [T, H, D]; v: [T, H, D]; g: [T, H, D] (a decay per key channel) or
    [T, H] (one per head: the scalar-gate form); beta: [T, H]; init_state: [N, H, D, D] fp32 or
    None; cu_seqlens: [N + 1] int32 on the device, or None with ``num_seqs``
    equal-length sequences (default 1).  ``max_seq_len`` (0 = unknown) bounds
    every sequence's length; ``segment_chunks`` (0 = automatic) sets the
    overlap granularity of the tensor-core path.  Returns (out, final_state, ckpts).
    """
    T, H, D = q.shape
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else (num_seqs or 1)
    dev = q.device
    if out is None:
        out = torch.empty(T, H, v.shape[2], dtype=q.dtype, device=dev)
    if final_state is None and want_final:
        final_state = torch.empty(N, H, D, v.shape[2], dtype=torch.float32, device=dev)
    if ckpt_stride > 0 and ckpts is None:
        cap = ckpt_capacity if ckpt_capacity is not None else max(1, (T // ckpt_stride) + N)
        ckpts = torch.zeros(cap, H, D, v.shape[2], dtype=torch.float32, device=dev)
    cap = ckpt_capacity if ckpt_capacity is not None else (ckpts.shape[0] if ckpts is not None else 0)
    desc = make_desc(T, H, D, N, _dtype_code(q), chunk, ckpt_stride, cap, max_seq_len, segment_chunks,
                     scalar_gate=g.dim() == 2, wait_limit=wait_limit, recurrence_ctas=recurrence_ctas)
    if workspace is None:
        workspace = alloc_workspace(desc, dev)
    code = load_library().kda_prefill(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state), _ptr(cu_seqlens),
        _ptr(out), _ptr(final_state), _ptr(ckpts), ctypes.byref(desc), _ptr(workspace),
        ctypes.c_size_t(workspace.numel()), _stream(stream))
    _check(code)
    return out, final_state, ckpts


def prefill_noalloc(q, k, v, g, beta, init_state=None, cu_seqlens=None, *, num_seqs: Optional[int] = None,
                    chunk: int = 64, ckpt_stride: int = 0, ckpts=None, ckpt_capacity: Optional[int] = None,
                    out=None, final_state=None, stream=None, max_seq_len: int = 0,
                    segment_chunks: int = 0):
    """``kda_prefill_noalloc``: the same prefill with the library's built-in
    scratch array instead of a workspace, for callers that cannot allocate
    device memory.  Calls on one device share that array: do not let them
    overlap on the GPU.  Returns (out, final_state, ckpts)."""
    T, H, D = q.shape
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else (num_seqs or 1)
    dev = q.device
    if out is None:
        out = torch.empty(T, H, v.shape[2], dtype=q.dtype, device=dev)
    if final_state is None:
        final_state = torch.empty(N, H, D, v.shape[2], dtype=torch.float32, device=dev)
    if ckpt_stride > 0 and ckpts is None:
        cap = ckpt_capacity if ckpt_capacity is not None else max(1, (T // ckpt_stride) + N)
        ckpts = torch.zeros(cap, H, D, v.shape[2], dtype=torch.float32, device=dev)
    cap = ckpt_capacity if ckpt_capacity is not None else (ckpts.shape[0] if ckpts is not None else 0)
    desc = make_desc(T, H, D, N, _dtype_code(q), chunk, ckpt_stride, cap, max_seq_len, segment_chunks,
                     scalar_gate=g.dim() == 2)
    code = load_library().kda_prefill_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state), _ptr(cu_seqlens),
        _ptr(out), _ptr(final_state), _ptr(ckpts), ctypes.byref(desc), _stream(stream))
    _check(code)
    return out, final_state, ckpts


def prefill_fused(q, k, v, g, beta, init_state=None, cu_seqlens=None, *, conv_w=None, conv_silu: bool = False,
                  gate=None, conv_state_in=None, conv_state_out=None, num_seqs: Optional[int] = None,
                  chunk: int = 64, ckpt_stride: int = 0, ckpts=None, ckpt_capacity: Optional[int] = None, out=None,
                  final_state=None, workspace=None, stream=None, max_seq_len: int = 0, segment_chunks: int = 0):
    """``kda_prefill_fused``: the prefill with the short convolution of q, k, v
    (taps ``conv_w`` [3, W, H, D] fp32, W <= 4, optional SiLU; history
    ``conv_state_in`` [N, 3, W - 1, H, D] or None for zeros; the state after
    each sequence written to ``conv_state_out`` when given) before the
    recurrence and the output gate ``out = o * sigmoid(gate)`` (``gate``
    [T, H, Dv], the dtype of q) after it.  Returns (out, final_state, ckpts)."""
    T, H, D = q.shape
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else (num_seqs or 1)
    dev = q.device
    if out is None:
        out = torch.empty(T, H, v.shape[2], dtype=q.dtype, device=dev)
    if final_state is None:
        final_state = torch.empty(N, H, D, v.shape[2], dtype=torch.float32, device=dev)
    if ckpt_stride > 0 and ckpts is None:
        cap = ckpt_capacity if ckpt_capacity is not None else max(1, (T // ckpt_stride) + N)
        ckpts = torch.zeros(cap, H, D, v.shape[2], dtype=torch.float32, device=dev)
    cap = ckpt_capacity if ckpt_capacity is not None else (ckpts.shape[0] if ckpts is not None else 0)
    W = int(conv_w.shape[1]) if conv_w is not None else 0
    desc = make_desc(T, H, D, N, _dtype_code(q), chunk, ckpt_stride, cap, max_seq_len, segment_chunks,
                     scalar_gate=g.dim() == 2, conv_width=W, conv_silu=conv_silu)
    if workspace is None:
        workspace = alloc_workspace(desc, dev)
    code = load_library().kda_prefill_fused(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state), _ptr(cu_seqlens), _ptr(out),
        _ptr(final_state), _ptr(ckpts), _ptr(conv_w), _ptr(conv_state_in), _ptr(conv_state_out), _ptr(gate),
        ctypes.byref(desc), _ptr(workspace),
        ctypes.c_size_t(workspace.numel()), _stream(stream))
    _check(code)
    return out, final_state, ckpts


def prefill_pooled(q, k, v, g, beta, state_pool, init_slots=None, final_slots=None, cu_seqlens=None, *,
                   num_seqs: Optional[int] = None, chunk: int = 64, ckpt_stride: int = 0, ckpt_slots=None,
                   out=None, workspace=None, stream=None, max_seq_len: int = 0, segment_chunks: int = 0):
    """Chunked prefill through ``kda_prefill_pooled``: sequence n starts from
    slot ``init_slots[n]`` of ``state_pool`` [P, H, D, D] and its final state
    goes to slot ``final_slots[n]``; snapshot j goes to slot ``ckpt_slots[j]``
    (int32 tables on the device; None = none of that kind; an id outside
    [0, P) is skipped).  Returns out."""
    T, H, D = q.shape
    N = (cu_seqlens.numel() - 1) if cu_seqlens is not None else (num_seqs or 1)
    dev = q.device
    if out is None:
        out = torch.empty(T, H, v.shape[2], dtype=q.dtype, device=dev)
    cap = ckpt_slots.numel() if (ckpt_stride > 0 and ckpt_slots is not None) else 0
    desc = make_desc(T, H, D, N, _dtype_code(q), chunk, ckpt_stride, cap, max_seq_len, segment_chunks,
                     scalar_gate=g.dim() == 2)
    if workspace is None:
        workspace = alloc_workspace(desc, dev)
    code = load_library().kda_prefill_pooled(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), _ptr(out), _ptr(state_pool),
        ctypes.c_int64(state_pool.shape[0]), _ptr(init_slots), _ptr(final_slots),
        _ptr(ckpt_slots) if cap else None, ctypes.byref(desc), _ptr(workspace),
        ctypes.c_size_t(workspace.numel()), _stream(stream))
    _check(code)
    return out


def prefill_status(workspace: torch.Tensor, stream=None) -> int:
    """Device-side status of the last prefill on ``workspace`` (synchronises)."""
    return int(load_library().kda_prefill_status(_ptr(workspace), _stream(stream)))


def decode(q, k, v, g, beta, state, out=None, stream=None):
    """One decode step through ``kda_decode``; ``state`` [N, H, D, D] is updated in place."""
    N, H, D = q.shape
    if out is None:
        out = torch.empty(N, H, v.shape[2], dtype=q.dtype, device=q.device)
    code = load_library().kda_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state),
                                     _ptr(out), N, H, D, v.shape[2], _dtype_code(q), _stream(stream))
    _check(code)
    return out


def decode_fused(q, k, v, g, beta, state, *, conv_w=None, conv_silu: bool = False, conv_state=None, gate=None,
                 out=None, stream=None):
    """One decode step through ``kda_decode_fused``: q, k, v [N, H, D]
    convolved with the history ``conv_state`` [N, 3, W - 1, H, D] (advanced in
    place; None: zeros), the step on ``state`` [N, H, D, D] (in place), the
    output gated by ``gate`` [N, H, D] (None: none)."""
    N, H, D = q.shape
    if out is None:
        out = torch.empty(N, H, v.shape[2], dtype=q.dtype, device=q.device)
    W = int(conv_w.shape[1]) if conv_w is not None else 0
    code = load_library().kda_decode_fused(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(conv_state), _ptr(conv_w), _ptr(gate),
        _ptr(out), N, H, D, v.shape[2], _dtype_code(q), W, int(bool(conv_silu)), _stream(stream))
    _check(code)
    return out


def decode_paged(q, k, v, g, beta, state_pool, slot_ids, out=None, stream=None, status=None):
    """One decode step through ``kda_decode_paged``: sequence n reads and
    updates slot ``slot_ids[n]`` of ``state_pool`` [P, H, D, D] (int32 ids on
    the device; an id outside [0, P) marks a padding row with a zero output).
    ``status`` (an int32 device tensor holding 0, or None) is set to
    KDA_ERR_INVALID_ARG when two sequences name the same slot."""
    N, H, D = q.shape
    if out is None:
        out = torch.empty(N, H, v.shape[2], dtype=q.dtype, device=q.device)
    code = load_library().kda_decode_paged(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_pool),
        ctypes.c_int64(state_pool.shape[0]), _ptr(slot_ids), _ptr(out), N, H, D, v.shape[2],
        _dtype_code(q), _ptr(status), _stream(stream))
    _check(code)
    return out


def decode_multi(q, k, v, g, beta, state, commit_len=None, slot_ids=None, out=None, stream=None,
                 status=None):
    """m tokens per sequence through ``kda_decode_multi``: q, k, g [N, m, H, D],
    v [N, m, H, D], beta [N, m, H]; ``state`` dense [N, H, D, D] or, with
    ``slot_ids``, a pool [P, H, D, D]; ``commit_len`` int32 [N] on the device
    (None: all m tokens) sets after how many tokens each state is written."""
    N, m, H, D = q.shape
    if out is None:
        out = torch.empty(N, m, H, v.shape[3], dtype=q.dtype, device=q.device)
    pool = state.shape[0] if slot_ids is not None else 0
    code = load_library().kda_decode_multi(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), ctypes.c_int64(pool),
        _ptr(slot_ids), _ptr(commit_len), _ptr(out), N, m, H, D, v.shape[3], _dtype_code(q), _ptr(status),
        _stream(stream))
    _check(code)
    return out
