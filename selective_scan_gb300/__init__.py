"""Python binding of libmamba2, the GB300 (sm_103a) Mamba2 recurrent hot path.

Argument marshalling only: every step runs in the CUDA kernels behind the C ABI
declared in ``include/mamba2.h``. Tensors are torch CUDA tensors (device memory
and streams come from PyTorch); batch metadata (``cu_seqlens``, ``slots``,
``fresh``) are host sequences. There is no fallback: importing the package
without the built library raises.

Entry points (same names as the C ABI without the ``mamba2_`` prefix):
``causal_conv1d``, ``ssd_scan`` (+ ``ssd_scan_workspace_bytes``),
``gated_rmsnorm``, ``decode_step``, ``decode_step_device``, ``prefill_host`` (+
``prefill_host_workspace_bytes``), ``padded_spans``, ``pack_rows``, ``unpack_rows``,
``in_proj``, ``out_proj``, ``state_bytes_per_layer``; and the Mamba-3 SISO forward
``mamba3_siso_varlen_forward`` (C name unchanged). ``selective_scan_gb300.padded`` holds the padded-batch
layer view built on them (attention mask in, HF-style cache out).
"""
from __future__ import annotations

import ctypes
from pathlib import Path
from typing import Optional, Sequence

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "libmamba2.so"

F32, BF16 = 0, 1
(OK, ERR_INVALID_ARGUMENT, ERR_SLOT_OUT_OF_RANGE, ERR_SLOT_SHARED, ERR_RUNS_DONT_COVER_ROWS,
 ERR_NOT_IMPLEMENTED, ERR_CUDA, ERR_WORKSPACE_TOO_SMALL) = range(8)
MAX_SEQS = 1024


class Mamba2Error(RuntimeError):
    """A non-OK status from libmamba2; ``.status`` holds the code."""

    def __init__(self, status: int, op: str, detail: str = ""):
        msg = f"{op}: {_lib().mamba2_status_string(status).decode()}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)
        self.status = status


class RecurrentBatch(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32),
                ("cu_seqlens", ctypes.POINTER(ctypes.c_int32)),
                ("slots", ctypes.POINTER(ctypes.c_int32)),
                ("fresh", ctypes.POINTER(ctypes.c_uint8))]


class Dims(ctypes.Structure):
    _fields_ = [("heads", ctypes.c_int32), ("headdim", ctypes.c_int32), ("d_state", ctypes.c_int32),
                ("ngroups", ctypes.c_int32), ("conv_kernel", ctypes.c_int32)]


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        if not LIB_PATH.exists():
            raise ImportError(f"{LIB_PATH} is not built; run selective_scan_gb300/build.py (nvcc, sm_103a)")
        lib = ctypes.CDLL(str(LIB_PATH))
        p, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
        rb, dims = ctypes.POINTER(RecurrentBatch), ctypes.POINTER(Dims)
        lib.mamba2_causal_conv1d.argtypes = [p, p, p, p, p, i32, i32, i32, i32, ctypes.c_int, rb, p]
        lib.mamba2_ssd_scan_workspace_bytes.argtypes = [dims, i32, rb]
        lib.mamba2_ssd_scan_workspace_bytes.restype = sz
        lib.mamba2_ssd_scan.argtypes = [p, p, p, p, p, p, p, i32, i32, dims, ctypes.c_int, rb, p, sz, p]
        lib.mamba2_gated_rmsnorm.argtypes = [p, p, p, p, i32, i32, i32, f32, ctypes.c_int, p]
        lib.mamba2_decode_step.argtypes = [p, p, p, p, p, p, p, p, p, p, i32, f32, p, p, i32, dims,
                                           ctypes.c_int, rb, p]
        lib.mamba2_decode_step_device.argtypes = [p, p, p, p, p, p, p, p, p, p, i32, f32, p, p, i32, dims,
                                                  ctypes.c_int, p, p, p, i32, p, p]
        lib.mamba2_in_proj.argtypes = [p, p, p, p, p, i32, i32, dims, ctypes.c_int, p]
        lib.mamba2_out_proj.argtypes = [p, p, p, i32, i32, i32, ctypes.c_int, p]
        lib.mamba2_padded_spans.argtypes = [p, i32, i32, p, p]
        lib.mamba2_pack_rows.argtypes = [p, p, i32, i32, i32, p, p, p]
        lib.mamba2_unpack_rows.argtypes = [p, p, i32, i32, i32, p, p, p]
        lib.mamba2_state_bytes_per_layer.argtypes = [dims, ctypes.c_int]
        lib.mamba2_state_bytes_per_layer.restype = ctypes.c_int64
        lib.mamba2_status_string.argtypes = [ctypes.c_int]
        lib.mamba2_status_string.restype = ctypes.c_char_p
        lib.mamba2_last_cuda_error.restype = ctypes.c_char_p
        lib.mamba2_device_timeouts.restype = ctypes.c_uint
        lib.mamba2_selftest_bounded_wait.argtypes = [p, p]
        lib.mamba2_selftest_bounded_wait.restype = ctypes.c_int
        lib.mamba2_prefill_host_workspace_bytes.argtypes = [dims, ctypes.c_int, rb, i32]
        lib.mamba2_prefill_host_workspace_bytes.restype = sz
        lib.mamba2_prefill_host.argtypes = [p, p, p, p, p, p, p, p, p, p, i32, f32, p, p, i32, dims, ctypes.c_int,
                                            rb, i32, p, sz, p]
        lib.mamba3_siso_varlen_forward.argtypes = [p] * 16 + [p, i32, i32, i32, i32, i32, i32, p]
        for name in ("mamba2_causal_conv1d", "mamba2_ssd_scan", "mamba2_gated_rmsnorm", "mamba2_decode_step",
                     "mamba2_decode_step_device", "mamba2_prefill_host", "mamba2_padded_spans", "mamba2_pack_rows",
                     "mamba2_unpack_rows", "mamba2_in_proj", "mamba2_out_proj", "mamba3_siso_varlen_forward"):
            getattr(lib, name).restype = ctypes.c_int
        _LIB = lib
    return _LIB


def library():
    """The loaded ctypes library (raises ImportError if it is not built)."""
    return _lib()


# --------------------------------------------------------------------------
# marshalling
# --------------------------------------------------------------------------

def _dt(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported activation dtype {t.dtype}")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Batch:
    """A RecurrentBatch marshalled once (host arrays kept alive); pass it as
    ``batch=`` to reuse it across calls instead of cu_seqlens/slots/fresh."""

    def __init__(self, cu_seqlens: Optional[Sequence[int]], slots: Sequence[int], fresh: Sequence[int]):
        n = len(slots)
        self.slots = (ctypes.c_int32 * max(n, 1))(*[int(s) for s in slots])
        self.fresh = (ctypes.c_uint8 * max(n, 1))(*[1 if f else 0 for f in fresh])
        self.cu = None
        if cu_seqlens is not None:
            self.cu = (ctypes.c_int32 * (len(cu_seqlens)))(*[int(c) for c in cu_seqlens])
        self.rb = RecurrentBatch(
            n, ctypes.cast(self.cu, ctypes.POINTER(ctypes.c_int32)) if self.cu is not None else None,
            ctypes.cast(self.slots, ctypes.POINTER(ctypes.c_int32)),
            ctypes.cast(self.fresh, ctypes.POINTER(ctypes.c_uint8)))

    def ref(self):
        return ctypes.byref(self.rb)


_Batch = Batch


def _batch(cu_seqlens, slots, fresh, batch):
    return batch if batch is not None else Batch(cu_seqlens, slots, fresh)


def _dims(d) -> Dims:
    if isinstance(d, Dims):
        return d
    return Dims(int(d.heads), int(d.headdim), int(d.d_state), int(d.ngroups), int(d.conv_kernel))


def _check(st: int, op: str):
    if st != OK:
        detail = _lib().mamba2_last_cuda_error().decode() if st == ERR_CUDA else ""
        raise Mamba2Error(st, op, detail)


# --------------------------------------------------------------------------
# entry points
# --------------------------------------------------------------------------

def causal_conv1d(dst, x, weight, bias, conv_state, cu_seqlens=None, slots=None, fresh=None, stream=None,
                  check=True, batch=None) -> int:
    """``mamba2_causal_conv1d``: dst = silu(depthwise causal conv) per run; conv_state updated."""
    rows, conv_dim = x.shape
    b = _batch(cu_seqlens, slots, fresh, batch)
    st = _lib().mamba2_causal_conv1d(_ptr(dst), _ptr(x), _ptr(weight), _ptr(bias), _ptr(conv_state),
                                     conv_state.shape[0], rows, conv_dim, weight.shape[1], _dt(x), b.ref(),
                                     _stream(stream))
    if check:
        _check(st, "mamba2_causal_conv1d")
    return st


def ssd_scan_workspace_bytes(dims, rows, cu_seqlens=None, slots=None, fresh=None, batch=None) -> int:
    """``mamba2_ssd_scan_workspace_bytes`` for this batch on the current device."""
    b = _batch(cu_seqlens, slots, fresh, batch)
    d = _dims(dims)
    return int(_lib().mamba2_ssd_scan_workspace_bytes(ctypes.byref(d), int(rows), b.ref()))


def ssd_scan(dst, xbc, dt, A_log, dt_bias, D, ssm_state, dims, cu_seqlens=None, slots=None, fresh=None,
             workspace=None, stream=None, check=True, batch=None) -> int:
    """``mamba2_ssd_scan``: chunked selective scan; ssm_state updated at the slots.

    ``workspace`` is a device tensor of at least ``ssd_scan_workspace_bytes`` bytes
    (allocated here with torch when None and needed).
    """
    import torch
    rows = xbc.shape[0]
    d = _dims(dims)
    b = _batch(cu_seqlens, slots, fresh, batch)
    if workspace is None:
        need = int(_lib().mamba2_ssd_scan_workspace_bytes(ctypes.byref(d), rows, b.ref()))
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=xbc.device)
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = _lib().mamba2_ssd_scan(_ptr(dst), _ptr(xbc), _ptr(dt), _ptr(A_log), _ptr(dt_bias), _ptr(D),
                                _ptr(ssm_state), ssm_state.shape[0], rows, ctypes.byref(d), _dt(xbc), b.ref(),
                                ws_ptr, ws_bytes, _stream(stream))
    if check:
        _check(st, "mamba2_ssd_scan")
    return st


def gated_rmsnorm(dst, x, z, weight, groups, eps, stream=None, check=True) -> int:
    """``mamba2_gated_rmsnorm``: dst = rmsnorm(x * silu(z)) * weight per group."""
    rows, dim = x.shape
    st = _lib().mamba2_gated_rmsnorm(_ptr(dst), _ptr(x), _ptr(z), _ptr(weight), rows, dim, int(groups),
                                     float(eps), _dt(x), _stream(stream))
    if check:
        _check(st, "mamba2_gated_rmsnorm")
    return st


def decode_step(dst, xBC, z, dt, conv_w, conv_b, A_log, dt_bias, D, norm_w, norm_groups, eps,
                conv_state, ssm_state, dims, slots=None, fresh=None, cu_seqlens=None, stream=None, check=True,
                batch=None) -> int:
    """``mamba2_decode_step``: fused conv -> scan -> gated norm for one token per sequence."""
    d = _dims(dims)
    b = _batch(cu_seqlens, slots, fresh, batch)
    st = _lib().mamba2_decode_step(_ptr(dst), _ptr(xBC), _ptr(z), _ptr(dt), _ptr(conv_w), _ptr(conv_b),
                                   _ptr(A_log), _ptr(dt_bias), _ptr(D), _ptr(norm_w), int(norm_groups),
                                   float(eps), _ptr(conv_state), _ptr(ssm_state), ssm_state.shape[0],
                                   ctypes.byref(d), _dt(xBC), b.ref(), _stream(stream))
    if check:
        _check(st, "mamba2_decode_step")
    return st


def decode_step_device(dst, xBC, z, dt, conv_w, conv_b, A_log, dt_bias, D, norm_w, norm_groups, eps,
                       conv_state, ssm_state, dims, slots_dev, fresh_dev, num_seqs_dev, status_dev,
                       stream=None, check=True) -> int:
    """``mamba2_decode_step_device``: the fused decode step with its batch in device memory.

    ``slots_dev`` (int32), ``fresh_dev`` (uint8) are device tensors of the capacity
    (their length); ``num_seqs_dev`` and ``status_dev`` are one-element int32 device
    tensors. The batch is checked on the device: ``status_dev`` holds the outcome once
    the stream has passed the call. The return value covers the host checks only.
    """
    d = _dims(dims)
    st = _lib().mamba2_decode_step_device(_ptr(dst), _ptr(xBC), _ptr(z), _ptr(dt), _ptr(conv_w), _ptr(conv_b),
                                          _ptr(A_log), _ptr(dt_bias), _ptr(D), _ptr(norm_w), int(norm_groups),
                                          float(eps), _ptr(conv_state), _ptr(ssm_state), ssm_state.shape[0],
                                          ctypes.byref(d), _dt(xBC), _ptr(slots_dev), _ptr(fresh_dev),
                                          _ptr(num_seqs_dev), int(slots_dev.shape[0]), _ptr(status_dev),
                                          _stream(stream))
    if check:
        _check(st, "mamba2_decode_step_device")
    return st


def in_proj(z, xBC, dt, hidden, w_in, dims, stream=None, check=True) -> int:
    """``mamba2_in_proj``: hidden . w_in^T split into z, xBC, dt (tcgen05 GEMM, bf16)."""
    d = _dims(dims)
    st = _lib().mamba2_in_proj(_ptr(z), _ptr(xBC), _ptr(dt), _ptr(hidden), _ptr(w_in), hidden.shape[0],
                               hidden.shape[1], ctypes.byref(d), _dt(hidden), _stream(stream))
    if check:
        _check(st, "mamba2_in_proj")
    return st


def out_proj(out, x, w_out, stream=None, check=True) -> int:
    """``mamba2_out_proj``: out = x . w_out^T (tcgen05 GEMM, bf16)."""
    st = _lib().mamba2_out_proj(_ptr(out), _ptr(x), _ptr(w_out), x.shape[0], x.shape[1], w_out.shape[0], _dt(x),
                                _stream(stream))
    if check:
        _check(st, "mamba2_out_proj")
    return st


def padded_spans(mask):
    """``mamba2_padded_spans``: (cu_seqlens, first) lists of a [batch, seqlen] host mask
    (nonzero = token); raises Mamba2Error when a row's tokens are not one span."""
    import torch
    m = mask.to(torch.uint8).contiguous()
    batch, seqlen = int(m.shape[0]), int(m.shape[1])
    cu = (ctypes.c_int32 * (batch + 1))()
    first = (ctypes.c_int32 * max(batch, 1))()
    st = _lib().mamba2_padded_spans(m.data_ptr() if m.numel() else None, batch, seqlen, cu, first)
    _check(st, "mamba2_padded_spans")
    return list(cu), list(first)[:batch]


def _pack(fn, name, dst, src, batch, seqlen, width_bytes, cu_seqlens, first, stream, check):
    cu = (ctypes.c_int32 * (len(cu_seqlens)))(*[int(v) for v in cu_seqlens])
    fi = (ctypes.c_int32 * max(len(first), 1))(*[int(v) for v in first])
    st = fn(_ptr(dst), _ptr(src), int(batch), int(seqlen), int(width_bytes), cu, fi, _stream(stream))
    if check:
        _check(st, name)
    return st


def pack_rows(dst, src, cu_seqlens, first, stream=None, check=True) -> int:
    """``mamba2_pack_rows``: padded ``src`` [batch, seqlen, ...] -> packed ``dst`` [rows, ...]."""
    width = src[0, 0].numel() * src.element_size() if src.numel() else dst.shape[-1] * dst.element_size()
    return _pack(_lib().mamba2_pack_rows, "mamba2_pack_rows", dst, src, src.shape[0], src.shape[1], width,
                 cu_seqlens, first, stream, check)


def unpack_rows(dst, src, cu_seqlens, first, stream=None, check=True) -> int:
    """``mamba2_unpack_rows``: packed ``src`` [rows, ...] -> padded ``dst`` [batch, seqlen, ...], zeros at padding."""
    width = dst[0, 0].numel() * dst.element_size() if dst.numel() else src.shape[-1] * src.element_size()
    return _pack(_lib().mamba2_unpack_rows, "mamba2_unpack_rows", dst, src, dst.shape[0], dst.shape[1], width,
                 cu_seqlens, first, stream, check)


def prefill_host_workspace_bytes(dims, act: int, piece_rows: int, cu_seqlens=None, slots=None, fresh=None,
                                 batch=None) -> int:
    """``mamba2_prefill_host_workspace_bytes`` for this batch and piece size."""
    b = _batch(cu_seqlens, slots, fresh, batch)
    d = _dims(dims)
    return int(_lib().mamba2_prefill_host_workspace_bytes(ctypes.byref(d), int(act), b.ref(), int(piece_rows)))


def prefill_host(out_host, xBC_host, z_host, dt_host, conv_w, conv_b, A_log, dt_bias, D, norm_w, norm_groups, eps,
                 conv_state, ssm_state, dims, cu_seqlens=None, slots=None, fresh=None, piece_rows=8192,
                 workspace=None, stream=None, check=True, batch=None) -> int:
    """``mamba2_prefill_host``: conv -> scan -> gated norm from host tensors, streamed in pieces.

    ``out_host``, ``xBC_host``, ``z_host``, ``dt_host`` are CPU tensors (pinned for
    overlap); the weights and pools are device tensors. ``workspace`` is a device
    tensor of at least ``prefill_host_workspace_bytes`` bytes (allocated here with
    torch when None). Asynchronous: synchronise the stream before reading ``out_host``.
    """
    import torch
    d = _dims(dims)
    b = _batch(cu_seqlens, slots, fresh, batch)
    act = _dt(xBC_host)
    if workspace is None:
        need = int(_lib().mamba2_prefill_host_workspace_bytes(ctypes.byref(d), act, b.ref(), int(piece_rows)))
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=ssm_state.device)
    st = _lib().mamba2_prefill_host(_ptr(out_host), _ptr(xBC_host), _ptr(z_host), _ptr(dt_host), _ptr(conv_w),
                                    _ptr(conv_b), _ptr(A_log), _ptr(dt_bias), _ptr(D), _ptr(norm_w), int(norm_groups),
                                    float(eps), _ptr(conv_state), _ptr(ssm_state), ssm_state.shape[0], ctypes.byref(d),
                                    act, b.ref(), int(piece_rows), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream))
    if check:
        _check(st, "mamba2_prefill_host")
    return st


def mamba3_siso_varlen_forward(out, final_angle, final_ssm, final_k, final_v, q, k, v, adt, dt, trap, q_bias,
                               k_bias, angles, d, z, cu_seqlens, stream=None, check=True) -> int:
    """``mamba3_siso_varlen_forward`` (include/mamba3.h): the Mamba-3 SISO forward over a
    packed batch. q, k [rows, d_state]; v, z, out [rows, heads, headdim]; adt, dt, trap
    [rows, heads]; angles [rows, rot_dim]; biases [heads, d_state]; d [heads]; the final
    states [num_seqs, heads, ...]; cu_seqlens a host sequence."""
    cu = list(cu_seqlens)
    n = len(cu) - 1
    rows, heads, headdim = v.shape
    arr = (ctypes.c_int32 * max(1, len(cu)))(*cu)
    st = _lib().mamba3_siso_varlen_forward(
        _ptr(out), _ptr(final_angle), _ptr(final_ssm), _ptr(final_k), _ptr(final_v), _ptr(q), _ptr(k), _ptr(v),
        _ptr(adt), _ptr(dt), _ptr(trap), _ptr(q_bias), _ptr(k_bias), _ptr(angles), _ptr(d), _ptr(z), arr, n,
        int(rows), int(heads), int(headdim), int(q.shape[1]), int(angles.shape[1]), _stream(stream))
    if check:
        _check(st, "mamba3_siso_varlen_forward")
    return st


def state_bytes_per_layer(dims, conv_dtype: int = BF16) -> int:
    """``mamba2_state_bytes_per_layer``: fp32 SSM state + conv history per sequence per layer."""
    d = _dims(dims)
    return int(_lib().mamba2_state_bytes_per_layer(ctypes.byref(d), int(conv_dtype)))


def status_string(status: int) -> str:
    return _lib().mamba2_status_string(int(status)).decode()
