"""Seeded synthetic inputs for the GLA forward pass.

This module only draws random numbers in the shapes and distributions of the benchmark workloads; it holds
none of the method's arithmetic and imports neither the CUDA binding nor the oracle, so both sides (and the
benchmark) can take their inputs from here.

Recipe (per workload): a CPU ``torch.Generator`` seeded with ``seed``; for varlen workloads the sequence
lengths are drawn first (uniform integers in [lo, hi]); then q, k ~ N(0,1) [B,T,H,K], v ~ N(0,1)
[B,T,H,V], g = logsigmoid(N(0,1)) / 16 [B,T,H,K] (drawn and transformed in fp32, then cast), and, when the
workload has an initial state, h0 = 0.1 * N(0,1) fp32 [N,H,K,V].  q, k, v, g are cast to the input dtype.
scale = K ** -0.5.

WY-representation workload (gated delta rule, ``make_wy_inputs``): the same generator and length draw,
then k = N(0,1) / sqrt(K) [B,T,H,K] (rows of about unit norm, as the rule's normalised keys),
v ~ N(0,1) [B,T,HV,V], beta = sigmoid(N(0,1)) [B,T,HV], A [B,T,HV,BT] unit lower-triangular per chunk (1 on
the chunk's diagonal, 0.1 * N(0,1) below it, 0 above; chunks start at each sequence's first row), and the
log2-domain gate g = -4 * U(0,1) fp32 [B,T,HV] (a factor 2^g in [1/16, 1]).  k, v, beta, A are cast to the
input dtype.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch
import torch.nn.functional as F


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "f32" | "bf16" | "f16"
    B: int
    T: int                # per-sequence length (dense) or packed total (varlen, filled in)
    H: int
    K: int
    V: int
    chunk: int = 64
    h0: bool = False
    ht: bool = True
    varlen: tuple = ()    # (n_seqs, lo, hi) for varlen packing, empty for dense
    seed: int = 0
    note: str = field(default="", compare=False)


# The five benchmark workloads, named by what they are.
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", "f32", B=1, T=256, H=2, K=64, V=64, seed=1000,
                         note="fp32 B=1 H=2 T=256 K=V=64, no h0, stores ht"),
    "b4_t2k_h8": Workload("b4_t2k_h8", "bf16", B=4, T=2048, H=8, K=128, V=128, h0=True, seed=1001,
                          note="bf16 B=4 H=8 T=2048 K=V=128 with h0, stores ht"),
    "b8_t4k_h16_v256": Workload("b8_t4k_h16_v256", "bf16", B=8, T=4096, H=16, K=128, V=256, seed=1002,
                                note="bf16 B=8 H=16 T=4096 K=128 V=256, stores ht"),
    "varlen16_h16": Workload("varlen16_h16", "bf16", B=1, T=0, H=16, K=128, V=128, h0=True,
                             varlen=(16, 128, 8192), seed=1003,
                             note="bf16 varlen, 16 sequences with lengths uniform in [128, 8192], H=16 "
                                  "K=V=128, per-sequence h0, stores ht"),
    "long_t64k_h32": Workload("long_t64k_h32", "bf16", B=1, T=65536, H=32, K=128, V=128, seed=1004,
                              note="bf16 B=1 H=32 T=65536 K=V=128, stores ht"),
}

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    h0: torch.Tensor | None
    cu_seqlens: torch.Tensor | None   # int32 [N+1] (CPU)
    scale: float
    B: int
    T: int
    H: int
    K: int
    V: int
    N: int
    chunk: int
    dtype: str


def make_inputs(dtype="bf16", B=1, T=64, H=1, K=64, V=64, h0=False, lengths=None, varlen=None,
                seed=0, chunk=64) -> Inputs:
    """Draw one input set on the CPU.

    Dense: ``B`` sequences of ``T`` rows.  Varlen: pass explicit ``lengths`` (list of ints), or
    ``varlen=(n, lo, hi)`` to draw n lengths uniformly in [lo, hi] from the same generator; B is then 1 and
    T is the packed total.
    """
    gen = torch.Generator().manual_seed(int(seed))
    cu = None
    if varlen:
        n, lo, hi = varlen
        lengths = torch.randint(lo, hi + 1, (n,), generator=gen).tolist()
    if lengths is not None:
        lengths = [int(x) for x in lengths]
        B, T = 1, sum(lengths)
        cu = torch.tensor([0] + lengths, dtype=torch.int64).cumsum(0).to(torch.int32)
    N = B if cu is None else cu.numel() - 1
    tdt = TORCH_DTYPE[dtype]
    q = torch.randn(B, T, H, K, generator=gen).to(tdt)
    k = torch.randn(B, T, H, K, generator=gen).to(tdt)
    v = torch.randn(B, T, H, V, generator=gen).to(tdt)
    g = (F.logsigmoid(torch.randn(B, T, H, K, generator=gen)) / 16).to(tdt)
    h = (0.1 * torch.randn(N, H, K, V, generator=gen)) if h0 else None
    return Inputs(q, k, v, g, h, cu, K ** -0.5, B, T, H, K, V, N, chunk, dtype)


@dataclass
class WyInputs:
    k: torch.Tensor
    v: torch.Tensor
    beta: torch.Tensor
    A: torch.Tensor
    g: torch.Tensor | None
    cu_seqlens: torch.Tensor | None   # int32 [N+1] (CPU)
    B: int
    T: int
    H: int
    HV: int
    K: int
    V: int
    BT: int
    N: int
    dtype: str


def make_wy_inputs(dtype="bf16", B=1, T=64, H=1, HV=1, K=64, V=64, BT=64, gate=True, lengths=None, varlen=None,
                   seed=0) -> WyInputs:
    """Draw one WY-representation input set on the CPU (dense, or varlen as in ``make_inputs``)."""
    gen = torch.Generator().manual_seed(int(seed))
    cu = None
    if varlen:
        n, lo, hi = varlen
        lengths = torch.randint(lo, hi + 1, (n,), generator=gen).tolist()
    if lengths is not None:
        lengths = [int(x) for x in lengths]
        B, T = 1, sum(lengths)
        cu = torch.tensor([0] + lengths, dtype=torch.int64).cumsum(0).to(torch.int32)
    N = B if cu is None else cu.numel() - 1
    tdt = TORCH_DTYPE[dtype]
    k = (torch.randn(B, T, H, K, generator=gen) / K ** 0.5).to(tdt)
    v = torch.randn(B, T, HV, V, generator=gen).to(tdt)
    beta = torch.sigmoid(torch.randn(B, T, HV, generator=gen)).to(tdt)
    # position of every row inside its chunk (chunks start at each sequence's first row)
    if cu is None:
        pos = (torch.arange(T) % BT).repeat(B)
    else:
        starts = torch.repeat_interleave(cu[:-1].long(), torch.tensor(lengths))
        pos = (torch.arange(T) - starts) % BT
    col = torch.arange(BT)
    A = 0.1 * torch.randn(B * T, HV, BT, generator=gen)
    A = torch.where(col[None, None, :] < pos[:, None, None], A, torch.zeros(()))
    A = torch.where(col[None, None, :] == pos[:, None, None], torch.ones(()), A)
    A = A.reshape(B, T, HV, BT).to(tdt)
    g = (-4.0 * torch.rand(B, T, HV, generator=gen)) if gate else None
    return WyInputs(k, v, beta, A, g, cu, B, T, H, HV, K, V, BT, N, dtype)


def wy_workload_inputs(name: str, BT: int = 64) -> WyInputs:
    """The WY workload with the shapes of forward workload ``name`` (HV = H key and value heads)."""
    w = WORKLOADS[name]
    return make_wy_inputs(w.dtype, B=w.B, T=w.T, H=w.H, HV=w.H, K=w.K, V=w.V, BT=BT, varlen=w.varlen or None,
                          seed=w.seed + 50)


def workload_inputs(name: str) -> Inputs:
    w = WORKLOADS[name]
    return make_inputs(w.dtype, B=w.B, T=w.T, H=w.H, K=w.K, V=w.V, h0=w.h0,
                       varlen=w.varlen or None, seed=w.seed, chunk=w.chunk)


def stored_numpy(x: torch.Tensor):
    """A CPU tensor as the numpy array of its stored words: float32 and float16 as they are, bf16 as uint16
    bit patterns."""
    x = x.detach().contiguous().cpu()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view("uint16")
    if x.dtype in (torch.float32, torch.float16):
        return x.numpy()
    raise TypeError(f"unsupported dtype {x.dtype}")
