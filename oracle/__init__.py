"""Plain CPU oracle for the Mamba2 recurrent path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA product path never calls it and
shares no code with it (``mamba2_ref.c`` has its own validation, rounding and
arithmetic).

The C source follows gllm PR #85 "feat(backend): Mamba2 ops, with CPU
reference implementations", sections "Ops" and "CPU reference": each op is the
token-at-a-time definition in double with the SSM state rounded to fp32 after
every token. This module marshals torch CPU tensors into the C library
(built on demand with gcc) and turns status codes into exceptions; the
padded-batch index maps at its end (spans, gather, scatter) are written out in
plain Python.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading
from pathlib import Path

import torch

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "mamba2_ref.c"
_HDR = _HERE / "mamba2_ref.h"
_SRC3 = _HERE / "mamba3_ref.c"
_HDR3 = _HERE / "mamba3_ref.h"
_LIB = _HERE / "libmamba2_ref.so"

F32, BF16 = 0, 1
OK, ERR_INVALID_ARGUMENT, ERR_SLOT_OUT_OF_RANGE, ERR_SLOT_SHARED, ERR_RUNS_DONT_COVER_ROWS = range(5)
STATUS_NAMES = {
    OK: "OK",
    ERR_INVALID_ARGUMENT: "INVALID_ARGUMENT",
    ERR_SLOT_OUT_OF_RANGE: "SLOT_OUT_OF_RANGE",
    ERR_SLOT_SHARED: "SLOT_SHARED",
    ERR_RUNS_DONT_COVER_ROWS: "RUNS_DONT_COVER_ROWS",
}

_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    """A non-OK status from the oracle; ``.status`` holds the code."""

    def __init__(self, status: int, op: str):
        super().__init__(f"oracle {op}: {STATUS_NAMES.get(status, status)}")
        self.status = status


def build(force: bool = False) -> Path:
    """Compile ``libmamba2_ref.so`` with gcc (OpenMP, no FP contraction)."""
    newest = max(f.stat().st_mtime for f in (_SRC, _HDR, _SRC3, _HDR3))
    if not force and _LIB.exists() and _LIB.stat().st_mtime >= newest:
        return _LIB
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=str(_HERE))
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", str(_SRC), str(_SRC3), "-o", tmp, "-lm"]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, _LIB)
    except subprocess.CalledProcessError as e:  # pragma: no cover
        os.unlink(tmp)
        raise RuntimeError(f"oracle build failed:\n{e.stderr}") from e
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(str(build()))
            i32, p, f32 = ctypes.c_int32, ctypes.c_void_p, ctypes.c_float
            lib.mamba2_ref_validate_batch.argtypes = [i32, p, p, i32, i32]
            lib.mamba2_ref_causal_conv1d.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32, i32, p, p, p, p]
            lib.mamba2_ref_ssd_scan.argtypes = [p, p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, i32, p, p, p, p]
            lib.mamba2_ref_gated_rmsnorm.argtypes = [p, p, p, p, i32, i32, i32, f32, i32, p]
            lib.mamba2_ref_decode_step.argtypes = [p, p, p, p, p, p, p, p, p, p, i32, f32, p, p,
                                                  i32, i32, i32, i32, i32, i32, i32, i32, p, p, p]
            lib.mamba2_ref_state_bytes_per_layer.argtypes = [i32] * 6
            lib.mamba2_ref_state_bytes_per_layer.restype = ctypes.c_int64
            lib.mamba2_ref_num_threads.restype = ctypes.c_int
            lib.mamba3_ref_siso_forward.argtypes = [p] * 16 + [i32, p, i32, i32, i32, i32, p]
            lib.mamba2_ref_set_num_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------

def _act_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"activation dtype {t.dtype} not supported")


def _ptr(t):
    if t is None:
        return None
    assert t.device.type == "cpu" and t.is_contiguous(), "oracle wants contiguous CPU tensors"
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else ctypes.c_void_p(0)


def _i32(seq) -> torch.Tensor:
    return torch.as_tensor(seq, dtype=torch.int32).contiguous()


def _u8(seq) -> torch.Tensor:
    return torch.as_tensor(seq, dtype=torch.uint8).contiguous()


def _check(status: int, op: str):
    if status != OK:
        raise OracleError(status, op)


def num_threads() -> int:
    return int(_load().mamba2_ref_num_threads())


def set_num_threads(n: int) -> None:
    _load().mamba2_ref_set_num_threads(int(n))


# --------------------------------------------------------------------------
# ops
# --------------------------------------------------------------------------

def validate_batch(cu_seqlens, slots, num_slots: int, rows: int) -> int:
    """Status of a RecurrentBatch (range, then shared, then coverage)."""
    slots_t = _i32(slots)
    cu = _i32(cu_seqlens)
    n = slots_t.numel()
    return int(_load().mamba2_ref_validate_batch(n, _ptr(cu), _ptr(slots_t), num_slots, rows))


def causal_conv1d(x, weight, bias, conv_state, cu_seqlens, slots, fresh):
    """Depthwise causal conv + SiLU per run; ``conv_state`` updated in place.

    Returns ``(dst, dst_f64)``: the act-typed output and its unrounded values.
    """
    rows, conv_dim = x.shape
    kernel = weight.shape[1]
    dst = torch.empty_like(x)
    dst64 = torch.empty(x.shape, dtype=torch.float64)
    cu, sl, fr = _i32(cu_seqlens), _i32(slots), _u8(fresh)
    st = _load().mamba2_ref_causal_conv1d(
        _ptr(dst), _ptr(x), _ptr(weight), _ptr(bias), _ptr(conv_state),
        conv_state.shape[0], rows, conv_dim, kernel, _act_code(x), sl.numel(),
        _ptr(cu), _ptr(sl), _ptr(fr), _ptr(dst64))
    _check(st, "causal_conv1d")
    return dst, dst64


def ssd_scan(xbc, dt, A_log, dt_bias, D, ssm_state, dims, cu_seqlens, slots, fresh):
    """Token-at-a-time selective scan; ``ssm_state`` updated in place.

    ``dims`` = (heads, headdim, d_state, ngroups). Returns ``(y, y_f64)``.
    """
    H, P, N, G = dims
    rows = xbc.shape[0]
    dst = torch.empty((rows, H * P), dtype=xbc.dtype)
    dst64 = torch.empty((rows, H * P), dtype=torch.float64)
    cu, sl, fr = _i32(cu_seqlens), _i32(slots), _u8(fresh)
    st = _load().mamba2_ref_ssd_scan(
        _ptr(dst), _ptr(xbc), _ptr(dt), _ptr(A_log), _ptr(dt_bias), _ptr(D), _ptr(ssm_state),
        ssm_state.shape[0], rows, H, P, N, G, _act_code(xbc), sl.numel(),
        _ptr(cu), _ptr(sl), _ptr(fr), _ptr(dst64))
    _check(st, "ssd_scan")
    return dst, dst64


def gated_rmsnorm(x, z, weight, groups: int, eps: float):
    """rmsnorm(x * silu(z)) * weight per group. Returns ``(out, out_f64)``."""
    rows, dim = x.shape
    dst = torch.empty_like(x)
    dst64 = torch.empty(x.shape, dtype=torch.float64)
    st = _load().mamba2_ref_gated_rmsnorm(
        _ptr(dst), _ptr(x), _ptr(z), _ptr(weight), rows, dim, groups, float(eps),
        _act_code(x), _ptr(dst64))
    _check(st, "gated_rmsnorm")
    return dst, dst64


def decode_step(xBC, z, dt, conv_w, conv_b, A_log, dt_bias, D, norm_w, norm_groups, eps,
                conv_state, ssm_state, dims, slots, fresh):
    """One token per sequence through conv -> scan -> norm; states in place.

    Returns ``(dst, dst_f64)``: the act-typed output and the norm's unrounded values.
    """
    H, P, N, G = dims
    n = xBC.shape[0]
    dst = torch.empty((n, H * P), dtype=xBC.dtype)
    dst64 = torch.empty((n, H * P), dtype=torch.float64)
    sl, fr = _i32(slots), _u8(fresh)
    st = _load().mamba2_ref_decode_step(
        _ptr(dst), _ptr(xBC), _ptr(z), _ptr(dt), _ptr(conv_w), _ptr(conv_b), _ptr(A_log),
        _ptr(dt_bias), _ptr(D), _ptr(norm_w), norm_groups, float(eps), _ptr(conv_state),
        _ptr(ssm_state), ssm_state.shape[0], H, P, N, G, conv_w.shape[1], _act_code(xBC),
        sl.numel(), _ptr(sl), _ptr(fr), _ptr(dst64))
    _check(st, "decode_step")
    return dst, dst64


def mamba3_siso_forward(q, k, v, adt, dt, trap, q_bias, k_bias, angles, d, z, cu_seqlens):
    """Mamba-3 SISO forward (page "Mamba-3 SISO Long-Ragged Multi-Chunk Joint States Full
    VJP", forward steps 1-7), fp64. q, k [T, N] bf16; v, z [T, H, P] bf16; adt, dt [T, H]
    f32; trap [T, H] bf16; q_bias, k_bias [H, N] f32; angles [T, R] bf16; d [H] f32.

    Returns ``(out, final_angle, final_ssm, final_k, final_v, out_f64)``.
    """
    T, N = q.shape
    H, P = v.shape[1], v.shape[2]
    R = angles.shape[1]
    S = len(cu_seqlens) - 1
    out = torch.empty((T, H, P), dtype=torch.bfloat16)
    out64 = torch.empty((T, H, P), dtype=torch.float64)
    fa = torch.empty((S, H, R), dtype=torch.bfloat16)
    fs = torch.empty((S, H, P, N), dtype=torch.float32)
    fk = torch.empty((S, H, N), dtype=torch.float32)
    fv = torch.empty((S, H, P), dtype=torch.bfloat16)
    cu = _i32(cu_seqlens)
    st = _load().mamba3_ref_siso_forward(
        _ptr(out), _ptr(fa), _ptr(fs), _ptr(fk), _ptr(fv), _ptr(q), _ptr(k), _ptr(v), _ptr(adt), _ptr(dt),
        _ptr(trap), _ptr(q_bias), _ptr(k_bias), _ptr(angles), _ptr(d), _ptr(z), S, _ptr(cu), H, P, N, R,
        _ptr(out64))
    _check(st, "mamba3_siso_forward")
    return out, fa, fs, fk, fv, out64


def state_bytes_per_layer(heads, headdim, d_state, ngroups, conv_kernel, conv_act=BF16) -> int:
    return int(_load().mamba2_ref_state_bytes_per_layer(heads, headdim, d_state, ngroups,
                                                        conv_kernel, conv_act))


# --------------------------------------------------------------------------
# Padded batches (page "Granite Mamba2 Inference Optimization": the layer's
# forward takes an attention mask and serves variable-length padded batches).
# Reading: a padding position is not a token of any sequence, and a row's
# tokens are one contiguous span. Plain index work, written out in Python.
# --------------------------------------------------------------------------

def padded_spans(mask):
    """(status, cu_seqlens, first) of a [batch, seqlen] mask: row b's tokens are the
    positions with mask != 0, which must be one run [first, first + len); an empty
    row has first 0. A row with two runs gives ERR_INVALID_ARGUMENT."""
    cu, first = [0], []
    for row in mask.tolist():
        pos = [t for t, m in enumerate(row) if m != 0]
        if pos and pos != list(range(pos[0], pos[0] + len(pos))):
            return ERR_INVALID_ARGUMENT, None, None
        first.append(pos[0] if pos else 0)
        cu.append(cu[-1] + len(pos))
    return OK, cu, first


def pack_rows(src, cu_seqlens, first):
    """Packed [cu[-1], ...] rows: row cu[b] + k is padded row (b, first[b] + k)."""
    out = []
    for b in range(len(first)):
        for k in range(cu_seqlens[b + 1] - cu_seqlens[b]):
            out.append(src[b, first[b] + k])
    return torch.stack(out) if out else src.new_zeros((0,) + tuple(src.shape[2:]))


def unpack_rows(src, cu_seqlens, first, seqlen):
    """Padded [batch, seqlen, ...]: each sequence's packed rows at its span, zeros elsewhere."""
    batch = len(first)
    out = src.new_zeros((batch, seqlen) + tuple(src.shape[1:]))
    for b in range(batch):
        for k in range(cu_seqlens[b + 1] - cu_seqlens[b]):
            out[b, first[b] + k] = src[cu_seqlens[b] + k]
    return out


# --------------------------------------------------------------------------
# The projections around the path (gllm PR #85, "Ops": the model splits in_proj
# into z, xBC and dt). A library matmul in double, then the column split.
# --------------------------------------------------------------------------

def in_proj(hidden, w_in, dims):
    """(z, xBC, dt) in double: hidden [rows, d_model] . w_in^T, w_in [d_in_proj, d_model]
    (output features x input features), columns split d_inner | conv_dim | heads."""
    H, P, N, G = dims
    d_inner, conv_dim = H * P, H * P + 2 * G * N
    assert w_in.shape[0] == d_inner + conv_dim + H
    y = hidden.double() @ w_in.double().t()
    return y[:, :d_inner], y[:, d_inner:d_inner + conv_dim], y[:, d_inner + conv_dim:]


def out_proj(x, w_out):
    """x [rows, d_inner] . w_out^T in double, w_out [d_model, d_inner]."""
    return x.double() @ w_out.double().t()
