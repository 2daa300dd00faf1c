"""Seeded synthetic inputs for the Mamba2 recurrent path.

This module only draws random tensors; it holds none of the method's
arithmetic and is shared by the tests, the benchmark and the smoke check (the
oracle and the CUDA path each receive its tensors as inputs).

Every draw uses ``torch.Generator('cpu').manual_seed(seed)`` in a fixed order:
(lengths, when the row count depends on them), xBC, z, dt, conv weight, conv
bias, A_log, dt_bias, D, then slots, fresh flags and pool contents.

Distributions (the five named workloads):
  xBC, z, dt ~ N(0, 1) at the activation dtype; conv weight ~ N(0, 0.5^2);
  conv bias ~ N(0, 0.1^2); A_log = log U[1, 16]; dt_bias = inverse softplus of
  U[1e-3, 0.1]; D ~ N(1, 0.1^2); norm weight = 1; eps = 1e-5; resumed SSM
  states ~ N(0, 0.1^2) fp32; resumed conv histories ~ N(0, 1) at the
  activation dtype. Slots a batch does not name hold a NaN sentinel, and so do
  the slots of fresh sequences (a dirty slot that must never be read).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

SENTINEL_F32 = 0x7FC0DEAD  # quiet-NaN payload for unused fp32 SSM slots
SENTINEL_BF16 = 0x7FDE  # quiet NaN for unused bf16 conv slots
SENTINEL_F32_ACT = 0x7FC0BEEF  # quiet NaN for unused fp32 conv slots


@dataclass(frozen=True)
class Dims:
    heads: int
    headdim: int
    d_state: int
    ngroups: int
    conv_kernel: int

    @property
    def d_inner(self) -> int:
        return self.heads * self.headdim

    @property
    def conv_dim(self) -> int:
        return self.d_inner + 2 * self.ngroups * self.d_state

    def tuple4(self):
        return (self.heads, self.headdim, self.d_state, self.ngroups)


@dataclass
class Params:
    conv_w: torch.Tensor  # [conv_dim, K] f32
    conv_b: torch.Tensor  # [conv_dim] f32
    A_log: torch.Tensor  # [H] f32
    dt_bias: torch.Tensor  # [H] f32
    D: torch.Tensor  # [H] f32
    norm_w: torch.Tensor  # [d_inner] f32
    norm_groups: int
    eps: float


@dataclass
class Batch:
    cu_seqlens: List[int]
    slots: List[int]
    fresh: List[int]

    @property
    def num_seqs(self) -> int:
        return len(self.slots)

    @property
    def rows(self) -> int:
        return self.cu_seqlens[-1] if self.cu_seqlens else 0

    def lengths(self) -> List[int]:
        return [b - a for a, b in zip(self.cu_seqlens[:-1], self.cu_seqlens[1:])]


@dataclass
class Workload:
    name: str
    dims: Dims
    act: torch.dtype
    params: Params
    batch: Batch
    xBC: torch.Tensor  # [rows, conv_dim] act
    z: torch.Tensor  # [rows, d_inner] act
    dt: torch.Tensor  # [rows, H] act
    conv_state: torch.Tensor  # [slots, K-1, conv_dim] act
    ssm_state: torch.Tensor  # [slots, H, P, N] f32
    # decode tokens: [steps, n, ...] (empty when the workload has none)
    dec_xBC: Optional[torch.Tensor] = None
    dec_z: Optional[torch.Tensor] = None
    dec_dt: Optional[torch.Tensor] = None
    extra: dict = field(default_factory=dict)


def _normal(g, shape, std=1.0, mean=0.0, dtype=torch.float32):
    t = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(dtype)


def _uniform(g, shape, lo, hi):
    return torch.rand(shape, generator=g, dtype=torch.float32) * (hi - lo) + lo


def draw_tokens(g, rows: int, dims: Dims, act: torch.dtype):
    xBC = _normal(g, (rows, dims.conv_dim), dtype=act)
    z = _normal(g, (rows, dims.d_inner), dtype=act)
    dt = _normal(g, (rows, dims.heads), dtype=act)
    return xBC, z, dt


def draw_params(g, dims: Dims, norm_groups: int, eps: float = 1e-5) -> Params:
    conv_w = _normal(g, (dims.conv_dim, dims.conv_kernel), std=0.5)
    conv_b = _normal(g, (dims.conv_dim,), std=0.1)
    A_log = torch.log(_uniform(g, (dims.heads,), 1.0, 16.0))
    y = _uniform(g, (dims.heads,), 1e-3, 0.1).double()
    dt_bias = (y + torch.log(-torch.expm1(-y))).float()  # inverse softplus of y
    D = _normal(g, (dims.heads,), std=0.1, mean=1.0)
    norm_w = torch.ones(dims.d_inner, dtype=torch.float32)
    return Params(conv_w, conv_b, A_log, dt_bias, D, norm_w, norm_groups, eps)


def empty_pools(num_slots: int, dims: Dims, act: torch.dtype):
    """Pools filled with the NaN sentinel."""
    hist = dims.conv_kernel - 1
    conv = torch.empty((num_slots, hist, dims.conv_dim), dtype=act)
    if act == torch.bfloat16:
        conv.view(torch.int16).fill_(SENTINEL_BF16)
    else:
        conv.view(torch.int32).fill_(SENTINEL_F32_ACT)
    ssm = torch.empty((num_slots, dims.heads, dims.headdim, dims.d_state), dtype=torch.float32)
    ssm.view(torch.int32).fill_(SENTINEL_F32)
    return conv, ssm


def fill_resumed_slots(g, conv, ssm, slots, fresh, act):
    """Random histories and states for the resuming sequences' slots."""
    for s, f in zip(slots, fresh):
        if f:
            continue
        conv[s] = _normal(g, conv.shape[1:], dtype=act)
        ssm[s] = _normal(g, ssm.shape[1:], std=0.1)


def make_prefill(name, seed, dims: Dims, lengths, act, num_slots, fresh, slots=None,
                 norm_groups=1, eps=1e-5) -> Workload:
    """A packed varlen prefill batch with the standard distributions.

    ``seed`` is an int or an already-advanced ``torch.Generator``.
    """
    g = seed if isinstance(seed, torch.Generator) else torch.Generator("cpu").manual_seed(seed)
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    xBC, z, dt = draw_tokens(g, cu[-1], dims, act)
    params = draw_params(g, dims, norm_groups, eps)
    if slots is None:
        slots = torch.randperm(num_slots, generator=g)[: len(lengths)].tolist()
    conv, ssm = empty_pools(num_slots, dims, act)
    fill_resumed_slots(g, conv, ssm, slots, fresh, act)
    batch = Batch(cu, list(slots), [int(bool(f)) for f in fresh])
    return Workload(name, dims, act, params, batch, xBC, z, dt, conv, ssm)


def draw_proj(g, dims: Dims, d_model: int, act=torch.bfloat16):
    """Random-init projection weights of the layer: w_in [d_inner + conv_dim + heads, d_model]
    ~ N(0, 1/d_model), w_out [d_model, d_inner] ~ N(0, 1/d_inner) (unit-variance outputs)."""
    d_in_proj = dims.d_inner + dims.conv_dim + dims.heads
    w_in = _normal(g, (d_in_proj, d_model), std=d_model ** -0.5, dtype=act)
    w_out = _normal(g, (d_model, dims.d_inner), std=dims.d_inner ** -0.5, dtype=act)
    return w_in, w_out


def padded_batch(seed: int, lengths, seqlen: int, sides, dims: Dims, act, num_slots: int = 0,
                 norm_groups: int = 1):
    """A padded batch [batch, seqlen, ...] (standard distributions at every position,
    padding included, so the padding's values are arbitrary) with its attention mask:
    row b holds lengths[b] tokens, at the end of the row when sides[b] == "left"
    (left padding) and at its start when "right". Returns (xBC, z, dt, mask, params,
    conv pool, ssm pool, slots); the pools hold the NaN sentinel."""
    g = torch.Generator("cpu").manual_seed(seed)
    batch = len(lengths)
    xBC, z, dt = draw_tokens(g, batch * seqlen, dims, act)
    params = draw_params(g, dims, norm_groups)
    mask = torch.zeros((batch, seqlen), dtype=torch.uint8)
    for b, (L, side) in enumerate(zip(lengths, sides)):
        if side == "left":
            mask[b, seqlen - L:] = 1
        else:
            mask[b, :L] = 1
    num_slots = max(num_slots, batch)
    slots = torch.randperm(num_slots, generator=g)[:batch].tolist()
    conv, ssm = empty_pools(num_slots, dims, act)
    return (xBC.view(batch, seqlen, -1), z.view(batch, seqlen, -1), dt.view(batch, seqlen, -1), mask, params,
            conv, ssm, slots)


# --------------------------------------------------------------------------
# the five named workloads
# --------------------------------------------------------------------------

DIMS_TINY = Dims(heads=4, headdim=16, d_state=16, ngroups=2, conv_kernel=4)
DIMS_130M = Dims(heads=24, headdim=64, d_state=128, ngroups=1, conv_kernel=4)
DIMS_48H = Dims(heads=48, headdim=64, d_state=128, ngroups=1, conv_kernel=4)


def tiny(seed: int = 0) -> Workload:
    """1 fresh sequence of 64 tokens, 4 heads x 16, d_state 16, 2 groups, fp32."""
    return make_prefill("tiny: 1x64 tok, 4 heads x 16, d_state 16, 2 groups, fp32", seed,
                        DIMS_TINY, [64], torch.float32, 1, [1], slots=[0], norm_groups=2)


def prefill_130m(seed: int = 1, tokens: int = 2048) -> Workload:
    """mamba2-130m-shaped layer: 1 fresh sequence, 24 heads x 64, d_state 128, bf16."""
    return make_prefill(f"prefill 1x{tokens} tok, 24 heads x 64, d_state 128, bf16", seed,
                        DIMS_130M, [tokens], torch.bfloat16, 1, [1], slots=[0])


def varlen_130m(seed: int = 2, num_seqs: int = 8, lo: int = 100, hi: int = 4000,
                num_slots: int = 64) -> Workload:
    """8 packed sequences, lengths U[100, 4000], half fresh, 64-slot pool."""
    g = torch.Generator("cpu").manual_seed(seed)
    lengths = torch.randint(lo, hi + 1, (num_seqs,), generator=g).tolist()
    fresh_idx = set(torch.randperm(num_seqs, generator=g)[: num_seqs // 2].tolist())
    fresh = [1 if i in fresh_idx else 0 for i in range(num_seqs)]
    return make_prefill(f"varlen prefill {num_seqs} seqs ({sum(lengths)} tok), 24 heads x 64, bf16",
                        g, DIMS_130M, lengths, torch.bfloat16, num_slots, fresh)


def decode_batch(seed: int = 3, num_seqs: int = 256, steps: int = 128, num_slots: int = 512,
                 dims: Dims = DIMS_48H) -> Workload:
    """256 sequences x 1 token per step against a 512-slot pool, none fresh."""
    g = torch.Generator("cpu").manual_seed(seed)
    act = torch.bfloat16
    xBC, z, dt = draw_tokens(g, steps * num_seqs, dims, act)
    params = draw_params(g, dims, 1)
    slots = torch.randperm(num_slots, generator=g)[:num_seqs].tolist()
    fresh = [0] * num_seqs
    conv, ssm = empty_pools(num_slots, dims, act)
    fill_resumed_slots(g, conv, ssm, slots, fresh, act)
    batch = Batch(list(range(num_seqs + 1)), slots, fresh)
    w = Workload(f"decode {num_seqs} seqs x {steps} steps, {dims.heads} heads x 64, bf16", dims, act,
                 params, batch, xBC[:0], z[:0], dt[:0], conv, ssm)
    w.dec_xBC = xBC.view(steps, num_seqs, -1)
    w.dec_z = z.view(steps, num_seqs, -1)
    w.dec_dt = dt.view(steps, num_seqs, -1)
    return w


def long_prefill(seed: int = 4, tokens: int = 65536, decode_steps: int = 64,
                 dims: Dims = DIMS_48H) -> Workload:
    """1 fresh sequence of 65536 tokens, 48 heads x 64, then 64 decode tokens."""
    g = torch.Generator("cpu").manual_seed(seed)
    act = torch.bfloat16
    xBC, z, dt = draw_tokens(g, tokens, dims, act)
    params = draw_params(g, dims, 1)
    dxBC, dz, ddt = draw_tokens(g, decode_steps, dims, act)
    conv, ssm = empty_pools(1, dims, act)
    batch = Batch([0, tokens], [0], [1])
    w = Workload(f"long prefill 1x{tokens} tok + {decode_steps} decode, {dims.heads} heads x 64, bf16",
                 dims, act, params, batch, xBC, z, dt, conv, ssm)
    w.dec_xBC = dxBC.view(decode_steps, 1, -1)
    w.dec_z = dz.view(decode_steps, 1, -1)
    w.dec_dt = ddt.view(decode_steps, 1, -1)
    return w


def named(i: int, **kw) -> Workload:
    return [tiny, prefill_130m, varlen_130m, decode_batch, long_prefill][i](**kw)


# --------------------------------------------------------------------------
# Mamba-3 SISO forward (page "Mamba-3 SISO Long-Ragged Multi-Chunk Joint States
# Full VJP"): its frozen shapes are GQA 1 -> 32, Q/K width 128, V width 64,
# rotary-angle width 32, three to five packed sequences of ragged lengths
# spanning 3 to 15 chunks of 64 tokens (never a multiple of 64). The page gives
# no value distributions; these follow the Mamba2 workloads' (activations
# N(0, 1); dt from dt_bias = inverse-softplus U[1e-3, 0.1]; decay rate
# A = U[1, 16] per head; D ~ N(1, 0.1^2)), with biases N(0, 0.1^2).
# --------------------------------------------------------------------------

@dataclass
class Mamba3Batch:
    name: str
    heads: int
    headdim: int
    d_state: int
    rot_dim: int
    cu_seqlens: List[int]
    q: torch.Tensor       # [T, N] bf16
    k: torch.Tensor       # [T, N] bf16
    v: torch.Tensor       # [T, H, P] bf16
    adt: torch.Tensor     # [T, H] f32
    dt: torch.Tensor      # [T, H] f32
    trap: torch.Tensor    # [T, H] bf16
    q_bias: torch.Tensor  # [H, N] f32
    k_bias: torch.Tensor  # [H, N] f32
    angles: torch.Tensor  # [T, R] bf16
    d: torch.Tensor       # [H] f32
    z: torch.Tensor       # [T, H, P] bf16

    @property
    def rows(self) -> int:
        return self.cu_seqlens[-1]

    def tensors(self):
        return (self.q, self.k, self.v, self.adt, self.dt, self.trap, self.q_bias, self.k_bias, self.angles,
                self.d, self.z)


def mamba3_batch(seed: int = 5, lengths=None, heads: int = 32, headdim: int = 64, d_state: int = 128,
                 rot_dim: int = 32, chunk: int = 64) -> Mamba3Batch:
    """Three to five packed sequences, each 3 to 15 chunks long and not a multiple of the chunk
    (drawn when `lengths` is None)."""
    g = torch.Generator("cpu").manual_seed(seed)
    if lengths is None:
        n = int(torch.randint(3, 6, (1,), generator=g))
        lengths = []
        for _ in range(n):
            L = int(torch.randint(2 * chunk + 1, 15 * chunk, (1,), generator=g))
            lengths.append(L + 1 if L % chunk == 0 else L)
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    T, H, P, N, R = cu[-1], heads, headdim, d_state, rot_dim
    bf = torch.bfloat16
    q = _normal(g, (T, N), dtype=bf)
    k = _normal(g, (T, N), dtype=bf)
    v = _normal(g, (T, H, P), dtype=bf)
    z = _normal(g, (T, H, P), dtype=bf)
    y = _uniform(g, (H,), 1e-3, 0.1).double()
    dt_bias = y + torch.log(-torch.expm1(-y))
    dt = torch.nn.functional.softplus(_normal(g, (T, H)).double() + dt_bias).float()
    A = _uniform(g, (H,), 1.0, 16.0)
    adt = (-A * dt).float()
    trap = _normal(g, (T, H), dtype=bf)
    q_bias = _normal(g, (H, N), std=0.1)
    k_bias = _normal(g, (H, N), std=0.1)
    angles = _normal(g, (T, R), dtype=bf)
    d = _normal(g, (H,), std=0.1, mean=1.0)
    return Mamba3Batch(f"mamba3 siso {len(lengths)} seqs ({T} tok), {H} heads x {P}, N {N}, R {R}", H, P, N, R, cu,
                       q, k, v, adt, dt, trap, q_bias, k_bias, angles, d, z)
