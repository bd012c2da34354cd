"""Seeded synthetic inputs for the KDA workloads.

This module holds only random-number recipes: no step of the method's
arithmetic lives here, so both the CUDA path (through the tests and the
benchmark) and the float64 oracle read the very same values from it.

Recipe (the five workloads the KDA pages' complexity figures are quoted for;
the pages publish no dataset, so these synthetic draws stand in):
  * q, k, v ~ N(0, 1) per element; q and k are then divided by their L2 norm
    per (token, head) in fp32; the bf16 workloads cast q, k, v to bf16 once.
  * g = -exp(a), a ~ U(-5, -1), per token, head and key channel (fp32), so
    g lies in [-0.368, -0.0067] (alpha = exp g in (0.69, 0.993)).
  * beta = sigmoid(z), z ~ N(0, 1), per token and head (fp32).
  * initial states ~ N(0, sigma^2) with sigma = 0.01, fp32, or zeros.
  * varlen: sequence lengths ~ U_int[1024, 32768] from their own seed.
Workload i uses seed 1000 + i.  Decode step s draws from seed
(base_seed * 1_000_003 + s).
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import torch


@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    H: int
    D: int
    lens: tuple            # per-sequence lengths
    dtype: str             # "bf16" or "fp32": dtype of q, k, v and out
    init: str              # "zeros" or "randn"
    chunk: int = 64
    ckpt_stride: int = 0
    seed: int = 0
    varlen: bool = False   # packed with cu_seqlens (else equal-length batch)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lens))

    @property
    def num_seqs(self) -> int:
        return len(self.lens)


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    N: int
    H: int
    D: int
    steps: int
    dtype: str
    seed: int = 0


def varlen_lengths(n: int, lo: int, hi: int, seed: int) -> tuple:
    g = torch.Generator(device="cpu").manual_seed(seed)
    return tuple(int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g).tolist())


def workload(i: int):
    """The five named workloads (1-based index)."""
    if i == 1:
        return PrefillWorkload("prefill B1 H2 T256 D64 fp32", H=2, D=64, lens=(256,), dtype="fp32",
                               init="zeros", seed=1001)
    if i == 2:
        return PrefillWorkload("prefill B1 H32 T8192 D128 bf16", H=32, D=128, lens=(8192,),
                               dtype="bf16", init="randn", seed=1002)
    if i == 3:
        return DecodeWorkload("decode N256 H32 D128 bf16 x64 steps", N=256, H=32, D=128, steps=64,
                              dtype="bf16", seed=1003)
    if i == 4:
        return PrefillWorkload("long prefill B1 H32 T131072 D128 bf16 ckpt32768", H=32, D=128,
                               lens=(131072,), dtype="bf16", init="randn", ckpt_stride=32768,
                               seed=1004)
    if i == 5:
        return PrefillWorkload("varlen prefill 16 seqs U[1024,32768] H32 D128 bf16", H=32, D=128,
                               lens=varlen_lengths(16, 1024, 32768, 1005), dtype="bf16",
                               init="randn", seed=1005, varlen=True)
    raise ValueError(f"no workload {i}")


def custom_prefill(H: int, D: int, lens: Sequence[int], dtype: str = "bf16", init: str = "randn",
                   ckpt_stride: int = 0, seed: int = 7, varlen: Optional[bool] = None,
                   name: str = "custom") -> PrefillWorkload:
    lens = tuple(int(x) for x in lens)
    if varlen is None:
        varlen = len(set(lens)) > 1
    return PrefillWorkload(name, H=H, D=D, lens=lens, dtype=dtype, init=init,
                           ckpt_stride=ckpt_stride, seed=seed, varlen=varlen)


def _torch_dtype(name: str):
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True)


def _draw_token_inputs(gen, T: int, H: int, D: int, dtype: str, device):
    f32 = torch.float32
    q = _unit_rows(torch.randn(T, H, D, generator=gen, device=device, dtype=f32))
    k = _unit_rows(torch.randn(T, H, D, generator=gen, device=device, dtype=f32))
    v = torch.randn(T, H, D, generator=gen, device=device, dtype=f32)
    a = torch.rand(T, H, D, generator=gen, device=device, dtype=f32) * 4.0 - 5.0
    g = -torch.exp(a)
    beta = torch.sigmoid(torch.randn(T, H, generator=gen, device=device, dtype=f32))
    td = _torch_dtype(dtype)
    return q.to(td), k.to(td), v.to(td), g.contiguous(), beta.contiguous()


def make_prefill(w: PrefillWorkload, device="cpu") -> dict:
    """Inputs of a prefill workload as torch tensors on ``device``.

    Keys: q, k, v ([T, H, D], bf16/fp32), g ([T, H, D] fp32), beta ([T, H] fp32),
    init_state ([N, H, D, D] fp32 or None), cu_seqlens ([N+1] int32, or None
    for an equal-length batch), plus the workload itself.
    """
    gen = torch.Generator(device=device).manual_seed(w.seed)
    T, H, D = w.total_tokens, w.H, w.D
    q, k, v, g, beta = _draw_token_inputs(gen, T, H, D, w.dtype, device)
    s0 = None
    if w.init == "randn":
        s0 = torch.randn(w.num_seqs, H, D, D, generator=gen, device=device,
                         dtype=torch.float32) * 0.01
    cu = torch.zeros(w.num_seqs + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(w.lens, dtype=torch.int64), 0).to(torch.int32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, init_state=s0,
                cu_seqlens=cu.to(device) if w.varlen else None, cu_host=cu, workload=w)


def scale_qk_rows(inp: dict, lo: float = 0.05, hi: float = 40.0, seed: int = 0) -> dict:
    """The same inputs with every (token, head) row of q and k multiplied by its
    own factor, log-uniform in [lo, hi] (drawn in fp32, the product cast back
    to the inputs' dtype once), so that q and k reach the library un-normalised.
    Returns a new dict; the other entries are shared."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    q, k = inp["q"], inp["k"]
    T, H = q.shape[0], q.shape[1]
    out = dict(inp)
    for name, x in (("q", q), ("k", k)):
        u = torch.rand(T, H, 1, generator=gen, dtype=torch.float32)
        f = torch.exp(torch.log(torch.tensor(lo)) + u * (torch.log(torch.tensor(hi)) - torch.log(torch.tensor(lo))))
        out[name] = (x.float().cpu() * f).to(x.dtype).to(x.device)
    return out


def strong_decay_gates(inp: dict, lo: float = 1.0, hi: float = 3.0, seed: int = 0) -> dict:
    """The same inputs with g replaced by -U(lo, hi) per element (fp32): a decay
    of 1 to 3 nepers per token and channel, so that one chunk of 64 tokens
    decays by about e^-128.  Returns a new dict; the other entries are shared."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    g = inp["g"]
    out = dict(inp)
    out["g"] = (-(lo + (hi - lo) * torch.rand(g.shape, generator=gen, dtype=torch.float32))).to(g.device)
    return out


def make_decode_state(w: DecodeWorkload, device="cpu") -> torch.Tensor:
    gen = torch.Generator(device=device).manual_seed(w.seed)
    return torch.randn(w.N, w.H, w.D, w.D, generator=gen, device=device,
                       dtype=torch.float32) * 0.01


def make_decode_step(w: DecodeWorkload, step: int, device="cpu") -> dict:
    """Token inputs of decode step ``step``: q, k, v [N, H, D], g [N, H, D], beta [N, H]."""
    gen = torch.Generator(device=device).manual_seed(w.seed * 1_000_003 + step)
    q, k, v, g, beta = _draw_token_inputs(gen, w.N, w.H, w.D, w.dtype, device)
    return dict(q=q, k=k, v=v, g=g, beta=beta)
