"""Seeded synthetic inputs for the KDA workloads.

This module only draws random tensors with the shapes and value
distributions of the workloads described for Kimi Delta Attention (Kimi K3
technical report, section 2.1.1, Eq. 1, 2 and 5). It contains none of the
method's arithmetic: no gate, no decay, no recurrence. Both the CUDA path
and the CPU oracle take their inputs from here, so neither depends on the
other.

Recipe (identical for every workload, only sizes differ):
  * q, k ~ N(0, 1), then L2-normalised per (token, head) in fp32 and cast to
    the I/O dtype.  Eq. 2 normalises q and k upstream of the recurrence, so
    the path receives unit vectors.
  * v ~ N(0, 1).
  * beta = sigmoid(N(0, 1)) per (token, head): Eq. 2 produces beta with a
    sigmoid upstream, so the path receives values in (0, 1).
  * z ~ N(0, z_std^2) per (token, head, channel): the decay logit before the
    per-head bias.
  * dt_bias b ~ U(-b_range, b_range) per (head, channel), fp32.
  * A_log ~ N(0, alog_std^2) per head, fp32.
  * initial state S0 ~ N(0, s0_std^2) fp32 per (sequence, head), or absent.
  * variable lengths ~ U{len_lo .. len_hi} per sequence.

Every tensor is produced in fp32 first and then cast with round-to-nearest-
even, so that the exact values given to the GPU are known; the oracle reads
those values upcast to fp64.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shapes and value distributions of one synthetic KDA workload."""

    name: str
    H: int
    d: int
    dtype: str  # "f32" | "bf16"
    n_seq: int = 1
    seq_len: Optional[int] = None  # fixed length (None => varlen)
    len_lo: int = 0
    len_hi: int = 0
    chunk: int = 64
    z_std: float = 1.0
    b_range: float = 0.0
    alog_std: float = 0.0
    s0_std: float = 0.0  # 0 => zero initial state (passed as NULL)
    decode_steps: int = 0  # > 0 => decode workload (one token per sequence per step)


# The five workloads of the KDA hot path (sizes from the task configuration).
TINY_F32 = Workload("kda_tiny_f32_T256_H2_d64", H=2, d=64, dtype="f32", n_seq=1, seq_len=256,
                    z_std=2.0, b_range=0.0, alog_std=0.0, s0_std=0.0)
PREFILL_4K = Workload("kda_prefill_bf16_T4096_H32_d128", H=32, d=128, dtype="bf16", n_seq=1,
                      seq_len=4096, z_std=1.5, b_range=1.0, alog_std=0.25, s0_std=0.0)
VARLEN_32 = Workload("kda_varlen_bf16_N32_len512-8192_H32_d128", H=32, d=128, dtype="bf16",
                     n_seq=32, seq_len=None, len_lo=512, len_hi=8192, z_std=1.5, b_range=1.0,
                     alog_std=0.25, s0_std=0.02)
LONG_1M = Workload("kda_prefill_bf16_T1048576_H32_d128", H=32, d=128, dtype="bf16", n_seq=1,
                   seq_len=1 << 20, z_std=1.5, b_range=1.0, alog_std=0.25, s0_std=0.0)
DECODE_256 = Workload("kda_decode_bf16_N256_H32_d128_512steps", H=32, d=128, dtype="bf16",
                      n_seq=256, seq_len=1, z_std=1.5, b_range=1.0, alog_std=0.25, s0_std=0.02,
                      decode_steps=512)

WORKLOADS = [TINY_F32, PREFILL_4K, VARLEN_32, LONG_1M, DECODE_256]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def seq_lengths(w: Workload, seed: int) -> list[int]:
    """Per-sequence lengths (fixed, or uniform in [len_lo, len_hi])."""
    if w.seq_len is not None:
        return [int(w.seq_len)] * w.n_seq
    g = _gen(seed + 7919, "cpu")
    lens = torch.randint(w.len_lo, w.len_hi + 1, (w.n_seq,), generator=g)
    return [int(x) for x in lens]


def cu_seqlens_of(lengths) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    # L2 normalisation of the last axis in fp32 (input recipe, Eq. 2 upstream of the path).
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def make_tokens(T: int, H: int, d_k: int, d_v: int, dtype: str, seed: int, *,
                z_std: float, device="cpu", gen: Optional[torch.Generator] = None):
    """Per-token inputs q, k, v, z [T, H, d], beta [T, H] in the I/O dtype.

    Draw order is fixed: q, k, v, beta, z.
    """
    dt = _DTYPES[dtype]
    g = gen if gen is not None else _gen(seed, device)
    f32 = torch.float32
    q = _unit_rows(torch.randn((T, H, d_k), generator=g, device=device, dtype=f32)).to(dt)
    k = _unit_rows(torch.randn((T, H, d_k), generator=g, device=device, dtype=f32)).to(dt)
    v = torch.randn((T, H, d_v), generator=g, device=device, dtype=f32).to(dt)
    beta = torch.sigmoid(torch.randn((T, H), generator=g, device=device, dtype=f32)).to(dt)
    z = (torch.randn((T, H, d_k), generator=g, device=device, dtype=f32) * z_std).to(dt)
    return q, k, v, beta, z


def make_output_gate_inputs(T: int, H: int, d_v: int, dtype: str, seed: int, device="cpu"):
    """Inputs of the output epilogue (Eq. 6 without projections): the gate pre-activation
    g = W_g x ~ N(0, 1) [T, H, d_v] in the I/O dtype, and the per-head RMSNorm weight
    w = 1 + 0.1 N(0, 1) [H, d_v] fp32.  Draw order: g, w."""
    gen = _gen(seed, device)
    g = torch.randn((T, H, d_v), generator=gen, device=device, dtype=torch.float32).to(_DTYPES[dtype])
    w = 1.0 + 0.1 * torch.randn((H, d_v), generator=gen, device=device, dtype=torch.float32)
    return g, w


def make_head_params(H: int, d_k: int, seed: int, *, b_range: float, alog_std: float):
    """dt_bias [H, d_k] fp32 and A_log [H] fp32 (CPU)."""
    g = _gen(seed + 104729, "cpu")
    if b_range > 0:
        b = (torch.rand((H, d_k), generator=g, dtype=torch.float32) * 2.0 - 1.0) * b_range
    else:
        b = torch.zeros((H, d_k), dtype=torch.float32)
    if alog_std > 0:
        a = torch.randn((H,), generator=g, dtype=torch.float32) * alog_std
    else:
        a = torch.zeros((H,), dtype=torch.float32)
    return b, a


def make_state(N: int, H: int, d_k: int, d_v: int, std: float, seed: int, device="cpu"):
    """Initial state [N, H, d_k, d_v] fp32 ~ N(0, std^2)."""
    g = _gen(seed + 1299709, device)
    return torch.randn((N, H, d_k, d_v), generator=g, device=device, dtype=torch.float32) * std


def make_prefill(w: Workload, seed: int, device="cpu", *, T_override: Optional[int] = None):
    """All inputs of a prefill workload as a dict of tensors.

    ``T_override`` shortens a fixed-length workload (same distributions), for
    oracle-sized parity cases and bounded CPU samples.
    """
    if w.seq_len is not None:
        T1 = int(T_override) if T_override is not None else int(w.seq_len)
        lengths = [T1] * w.n_seq
    else:
        lengths = seq_lengths(w, seed)
    T = sum(lengths)
    q, k, v, beta, z = make_tokens(T, w.H, w.d, w.d, w.dtype, seed, z_std=w.z_std, device=device)
    b, a = make_head_params(w.H, w.d, seed, b_range=w.b_range, alog_std=w.alog_std)
    s0 = make_state(len(lengths), w.H, w.d, w.d, w.s0_std, seed, device) if w.s0_std > 0 else None
    return dict(q=q, k=k, v=v, beta=beta, z=z, dt_bias=b.to(device), A_log=a.to(device),
                initial_state=s0, lengths=lengths, cu_seqlens=cu_seqlens_of(lengths).to(device),
                g_min=-5.0, scale=1.0, chunk=w.chunk)


def make_prefill_shard(w: Workload, seed: int, rank: int, world: int, device="cpu"):
    """Rank `rank`'s share of a global varlen batch of world * w.n_seq sequences: the sequences
    [rank * n, (rank + 1) * n), n = w.n_seq, as one batch (the inputs of make_prefill, plus `seq_ids`).
    Every sequence is drawn from its own generators (seeded by the global seed and its index: its
    length, tokens and initial state), so a sequence is the same whatever the number of ranks; the
    head parameters are the global seed's."""
    n = w.n_seq
    ids = list(range(rank * n, (rank + 1) * n))
    lengths, parts, states = [], [], []
    for i in ids:
        si = seed * 1000003 + 7 * i + 1
        if w.seq_len is not None:
            L = int(w.seq_len)
        else:
            L = int(torch.randint(w.len_lo, w.len_hi + 1, (1,), generator=_gen(si + 7919, "cpu")))
        lengths.append(L)
        parts.append(make_tokens(L, w.H, w.d, w.d, w.dtype, si, z_std=w.z_std, device=device))
        if w.s0_std > 0:
            states.append(make_state(1, w.H, w.d, w.d, w.s0_std, si, device))
    q, k, v, beta, z = (torch.cat([p_[j] for p_ in parts], 0) for j in range(5))
    b, a = make_head_params(w.H, w.d, seed, b_range=w.b_range, alog_std=w.alog_std)
    s0 = torch.cat(states, 0) if states else None
    return dict(q=q, k=k, v=v, beta=beta, z=z, dt_bias=b.to(device), A_log=a.to(device),
                initial_state=s0, lengths=lengths, cu_seqlens=cu_seqlens_of(lengths).to(device),
                g_min=-5.0, scale=1.0, chunk=w.chunk, seq_ids=ids)


def make_decode(w: Workload, seed: int, device="cpu", *, n_seq: Optional[int] = None,
                steps: Optional[int] = None):
    """Decode workload: per-step tokens [steps, N, H, d] and the state [N, H, d, d]."""
    N = int(n_seq) if n_seq is not None else w.n_seq
    S = int(steps) if steps is not None else w.decode_steps
    q, k, v, beta, z = make_tokens(S * N, w.H, w.d, w.d, w.dtype, seed, z_std=w.z_std, device=device)
    shp = (S, N, w.H)
    b, a = make_head_params(w.H, w.d, seed, b_range=w.b_range, alog_std=w.alog_std)
    s0 = make_state(N, w.H, w.d, w.d, w.s0_std, seed, device)
    return dict(q=q.view(*shp, w.d), k=k.view(*shp, w.d), v=v.view(*shp, w.d),
                beta=beta.view(*shp), z=z.view(*shp, w.d), dt_bias=b.to(device),
                A_log=a.to(device), state=s0, g_min=-5.0, scale=1.0)
