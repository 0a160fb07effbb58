"""Python binding of libssu, the GB300 (sm_103a) selective state update.

Argument marshalling only: tensors are checked for shape, their pointers and
strides are packed into the C structs of ``include/ssu.h``, and the C entry
point launches the CUDA kernel on the current torch stream.  Every step of the
update runs in the CUDA kernels; there is no CPU or PyTorch fallback.  When
``libssu.so`` is not built, every call raises.

Entry points (same names as the C ABI):
  ssu_update_onetoken  one decode token per sequence
  ssu_replay_update    one decode token per sequence, state kept as a
                       checkpoint plus a buffer of recent inputs
  ssu_replay_verify    speculative decoding on that form: T drafts per
                       sequence appended and verified, nothing committed
  ssu_update_packed    packed variable-length / MTP rows (cu_seqlens) or the
                       dense [batch, steps, heads, dim] form
  ssu_shadow_refresh   the low-precision read copy of checkpoints
  ssu_ssd_prefill      packed variable-length SSD prefill (and
                       ssd_combined_fwd_varlen, the MATE-shaped call)
  ssu_ssd_prefill_static  the same on the library's own device scratch
  ssu_batch_copy       batched state copies with memmove semantics
  ssu_prewarm          load a configuration's kernel before graph capture
and ``selective_state_update``, the MATE/FlashInfer-shaped call (MATE
documentation, page "Mamba / SSU", API reference) that picks one of the two
update entry points from the call shape.
"""
from __future__ import annotations

import ctypes
import functools
import os
from typing import Optional

import torch

__all__ = ["ssu_update_onetoken", "ssu_selftest_timeout", "ssu_update_packed", "ssu_replay_update", "ssu_replay_verify", "ssu_shadow_refresh",
           "ssu_ssd_prefill", "ssu_ssd_prefill_static", "ssd_combined_fwd_varlen",
           "ssu_batch_copy", "copy_table",
           "slot_copies", "ssu_prewarm",
           "selective_state_update",
           "SLOTS_STRIDED", "SLOTS_PER_ROW", "DEV_BAD_SLOT", "DEV_BAD_ENTRY", "DEV_BAD_SEQLEN", "DEV_TIMEOUT",
           "library_path", "lib"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libssu.so")

# ssu.h constants
OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA = 0, 1, 2, 3
SLOTS_STRIDED, SLOTS_PER_ROW = 0, 1
DEV_BAD_SLOT, DEV_BAD_ENTRY, DEV_BAD_SEQLEN, DEV_TIMEOUT, DEV_BAD_COUNT, DEV_BAD_COPY = 0x1, 0x2, 0x4, 0x8, 0x10, 0x20
UNSUP_RAND_SEED, UNSUP_STATE_SCALE, UNSUP_INTERMEDIATE, UNSUP_CACHE_STEPS, UNSUP_ALGORITHM = (
    0x01, 0x02, 0x04, 0x08, 0x10)
_DTYPE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
_ITYPE = {torch.int32: 0, torch.int64: 1}


class SlotTable(ctypes.Structure):
    _fields_ = [("entries", ctypes.c_void_p), ("type", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("s0", ctypes.c_int64), ("s1", ctypes.c_int64), ("extent", ctypes.c_int64)]


_I64x3 = ctypes.c_int64 * 3


class Args(ctypes.Structure):
    _fields_ = [
        ("slots", ctypes.c_int64), ("heads", ctypes.c_int64), ("dim", ctypes.c_int64),
        ("dstate", ctypes.c_int64), ("groups", ctypes.c_int64),
        ("state_dtype", ctypes.c_int32), ("io_dtype", ctypes.c_int32), ("dt_dtype", ctypes.c_int32),
        ("dt_softplus", ctypes.c_int32), ("disable_state_update", ctypes.c_int32),
        ("reserved0", ctypes.c_int32), ("pad_slot_id", ctypes.c_int64),
        ("state", ctypes.c_void_p), ("x", ctypes.c_void_p), ("dt", ctypes.c_void_p),
        ("B", ctypes.c_void_p), ("C", ctypes.c_void_p), ("z", ctypes.c_void_p),
        ("A", ctypes.c_void_p), ("D", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("y", ctypes.c_void_p),
        ("x_stride", _I64x3), ("dt_stride", _I64x3), ("B_stride", _I64x3), ("C_stride", _I64x3),
        ("z_stride", _I64x3), ("y_stride", _I64x3),
        ("d_status", ctypes.c_void_p), ("unsupported", ctypes.c_uint32),
    ]


class ReplayBuffers(ctypes.Structure):
    _fields_ = [("len", ctypes.c_int64), ("x", ctypes.c_void_p), ("dt", ctypes.c_void_p),
                ("B", ctypes.c_void_p), ("count_in", ctypes.c_void_p), ("count_out", ctypes.c_void_p),
                ("shadow_format", ctypes.c_int32), ("reserved0", ctypes.c_int32), ("shadow", ctypes.c_void_p),
                ("shadow_scale", ctypes.c_void_p)]


class SsdArgs(ctypes.Structure):
    _fields_ = [
        ("tokens", ctypes.c_int64), ("heads", ctypes.c_int64), ("dim", ctypes.c_int64), ("dstate", ctypes.c_int64),
        ("groups", ctypes.c_int64), ("nseq", ctypes.c_int64), ("nchunks", ctypes.c_int64),
        ("chunk_size", ctypes.c_int64),
        ("io_dtype", ctypes.c_int32), ("dt_dtype", ctypes.c_int32), ("state_dtype", ctypes.c_int32),
        ("meta_type", ctypes.c_int32), ("dt_softplus", ctypes.c_int32), ("return_intermediate", ctypes.c_int32),
        ("dt_min", ctypes.c_float), ("dt_max", ctypes.c_float),
        ("x", ctypes.c_void_p), ("dt", ctypes.c_void_p), ("B", ctypes.c_void_p), ("C", ctypes.c_void_p),
        ("z", ctypes.c_void_p), ("A", ctypes.c_void_p), ("D", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("cu_chunk_seqlens", ctypes.c_void_p), ("seq_idx", ctypes.c_void_p),
        ("last_chunk_indices", ctypes.c_void_p), ("initial_states", ctypes.c_void_p),
        ("y", ctypes.c_void_p), ("states", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_uint64), ("d_status", ctypes.c_void_p),
    ]


# formats of the read copy (SSU_SHADOW_*)
SHADOW_NONE, SHADOW_F16, SHADOW_E4M3, SHADOW_NVFP4 = 0, 1, 2, 3


def nvfp4_scale_words(dstate: int) -> int:
    """Floats of one row's NVFP4 scale record (SSU_NVFP4_SCALE_WORDS): the
    fp32 row scale, then the dstate / 16 E4M3 block codes as bytes, padded to
    a multiple of 16 bytes."""
    return (4 + dstate // 16 + 15) // 16 * 4


def _shadow_format(shadow: Optional[torch.Tensor], state: torch.Tensor) -> int:
    """The read copy's format from its tensor: float16 values (F16); one uint8
    / float8_e4m3fn code per state element (E4M3); uint8 bytes of two E2M1
    codes, or float4_e2m1fn_x2, with half the state's last dimension (NVFP4)."""
    if shadow is None:
        return SHADOW_NONE
    if shadow.dtype == torch.float16:
        return SHADOW_F16
    fp4 = getattr(torch, "float4_e2m1fn_x2", None)
    half = tuple(shadow.shape) == (*state.shape[:-1], state.shape[-1] // 2)
    if (shadow.dtype == torch.uint8 and half) or (fp4 is not None and shadow.dtype == fp4):
        return SHADOW_NVFP4
    if shadow.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        return SHADOW_E4M3
    raise ValueError("a read copy is float16 (fp16 values), uint8 / float8_e4m3fn (E4M3 codes) or uint8 / "
                     "float4_e2m1fn_x2 with half the last dimension (NVFP4 code pairs)")


def _check_copy_scales(fmt: int, shadow_scale: Optional[torch.Tensor], state: torch.Tensor) -> None:
    if fmt == SHADOW_E4M3:
        _need(shadow_scale is not None and shadow_scale.dtype == torch.float32 and shadow_scale.is_cuda
              and shadow_scale.is_contiguous() and tuple(shadow_scale.shape) == tuple(state.shape[:-1]),
              "an E4M3 read copy needs contiguous fp32 row scales shaped like the state without dstate")
    elif fmt == SHADOW_NVFP4:
        want = (*state.shape[:-1], nvfp4_scale_words(state.shape[-1]))
        _need(shadow_scale is not None and shadow_scale.dtype == torch.float32 and shadow_scale.is_cuda
              and shadow_scale.is_contiguous() and tuple(shadow_scale.shape) == want,
              f"an NVFP4 read copy needs contiguous fp32 scale records of shape {want}")


_lib = None


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded libssu (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"libssu.so is not built ({_LIB_PATH} is missing); build it with "
                "`python -m selective_state_update_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(_LIB_PATH)
        p_args, p_tab = ctypes.POINTER(Args), ctypes.POINTER(SlotTable)
        L.ssu_update_onetoken.argtypes = [p_args, ctypes.c_int64, p_tab, p_tab, ctypes.c_void_p]
        L.ssu_update_onetoken.restype = ctypes.c_int
        L.ssu_selftest_timeout.argtypes = [p_args, ctypes.c_int64, p_tab, p_tab, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_void_p]
        L.ssu_selftest_timeout.restype = ctypes.c_int
        L.ssu_update_packed.argtypes = [p_args, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                        ctypes.c_int64, ctypes.c_void_p, ctypes.c_int32, p_tab, p_tab,
                                        ctypes.c_void_p]
        L.ssu_update_packed.restype = ctypes.c_int
        L.ssu_replay_update.argtypes = [p_args, ctypes.c_int64, p_tab, ctypes.POINTER(ReplayBuffers),
                                        ctypes.c_void_p]
        L.ssu_replay_update.restype = ctypes.c_int
        L.ssu_replay_verify.argtypes = [p_args, ctypes.c_int64, ctypes.c_int64, p_tab, ctypes.POINTER(ReplayBuffers),
                                        ctypes.c_void_p]
        L.ssu_replay_verify.restype = ctypes.c_int
        L.ssu_batch_copy.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p,
                                     ctypes.c_void_p]
        L.ssu_batch_copy.restype = ctypes.c_int
        L.ssu_ssd_workspace_size.argtypes = [ctypes.c_int64] * 6 + [ctypes.POINTER(ctypes.c_uint64)]
        L.ssu_ssd_workspace_size.restype = ctypes.c_int
        L.ssu_ssd_prefill.argtypes = [ctypes.POINTER(SsdArgs), ctypes.c_void_p]
        L.ssu_ssd_prefill.restype = ctypes.c_int
        L.ssu_ssd_prefill_static.argtypes = [ctypes.POINTER(SsdArgs), ctypes.c_void_p]
        L.ssu_ssd_prefill_static.restype = ctypes.c_int
        L.ssu_shadow_refresh.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.ssu_shadow_refresh.restype = ctypes.c_int
        L.ssu_prewarm.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                  ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int32]
        L.ssu_prewarm.restype = ctypes.c_int
        L.ssu_last_error.argtypes = []
        L.ssu_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _raise(rc: int):
    msg = lib().ssu_last_error().decode(errors="replace")
    if rc == ERR_INVALID:
        raise ValueError(msg)
    if rc == ERR_UNSUPPORTED:
        raise NotImplementedError(msg)
    raise RuntimeError(f"libssu: {msg}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _strides3(t: Optional[torch.Tensor]):
    return _I64x3(*(t.stride() if t is not None else (0, 0, 0)))


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _table(t: Optional[torch.Tensor], mode: int) -> Optional[SlotTable]:
    if t is None:
        return None
    _need(t.dtype in _ITYPE, "slot tables must be int32 or int64")
    _need(t.is_cuda, "slot tables must be CUDA tensors")
    if t.dim() == 1:
        s0 = s1 = t.stride(0)
        extent = (t.shape[0] - 1) * t.stride(0) + 1 if t.shape[0] > 0 else 0
    elif t.dim() == 2:
        s0, s1 = t.stride(0), t.stride(1)
        extent = ((t.shape[0] - 1) * s0 + (t.shape[1] - 1) * s1 + 1) if t.numel() > 0 else 0
    else:
        raise ValueError("slot tables are [n] or [sequences, steps]")
    return SlotTable(t.data_ptr(), _ITYPE[t.dtype], mode, s0, s1, extent)


def _args(state, x, dt, A, B, C, D, z, dt_bias, dt_softplus, pad_slot_id, out, disable_state_update,
          status, unsupported) -> Args:
    _need(state.dim() == 4, "state must be [slots, heads, dim, dstate]")
    slots, heads, dim, dstate = state.shape
    _need(state.is_contiguous(), "state must be contiguous")
    _need(state.dtype in _DTYPE and x.dtype in _DTYPE and dt.dtype in _DTYPE, "unsupported dtype")
    rows = x.shape[0]
    _need(x.dim() == 3 and tuple(x.shape[1:]) == (heads, dim), "x must be [rows, heads, dim]")
    _need(dt.dim() == 3 and tuple(dt.shape) == (rows, heads, dim), "dt must be [rows, heads, dim]")
    _need(B.dim() == 3 and B.shape[0] == rows and B.shape[2] == dstate, "B must be [rows, groups, dstate]")
    groups = B.shape[1]
    _need(tuple(C.shape) == tuple(B.shape), "C must have the shape of B")
    _need(B.dtype == x.dtype and C.dtype == x.dtype, "B and C must have the dtype of x")
    _need(tuple(out.shape) == (rows, heads, dim) and out.dtype == x.dtype, "out must be [rows, heads, dim] in x's dtype")
    if z is not None:
        _need(tuple(z.shape) == (rows, heads, dim) and z.dtype == x.dtype, "z must be [rows, heads, dim] in x's dtype")
    for name, t in (("A", A), ("D", D), ("dt_bias", dt_bias)):
        if t is not None:
            _need(t.dtype == torch.float32 and t.numel() == heads and t.is_contiguous(),
                  f"{name} must be a contiguous fp32 [heads] tensor")
    tensors = [state, x, dt, A, B, C, D, z, dt_bias, out, status]
    _need(all(t is None or t.is_cuda for t in tensors), "all tensors must be CUDA tensors")
    if status is not None:
        _need(status.dtype == torch.int32 and status.numel() >= 1, "status must be an int32 CUDA tensor")
    return Args(
        slots=slots, heads=heads, dim=dim, dstate=dstate, groups=groups,
        state_dtype=_DTYPE[state.dtype], io_dtype=_DTYPE[x.dtype], dt_dtype=_DTYPE[dt.dtype],
        dt_softplus=int(bool(dt_softplus)), disable_state_update=int(bool(disable_state_update)),
        reserved0=0, pad_slot_id=int(pad_slot_id),
        state=state.data_ptr(), x=x.data_ptr(), dt=dt.data_ptr(), B=B.data_ptr(), C=C.data_ptr(),
        z=_ptr(z), A=A.data_ptr(), D=_ptr(D), dt_bias=_ptr(dt_bias), y=out.data_ptr(),
        x_stride=_strides3(x), dt_stride=_strides3(dt), B_stride=_strides3(B), C_stride=_strides3(C),
        z_stride=_strides3(z), y_stride=_strides3(out), d_status=_ptr(status), unsupported=unsupported)


def _dt3(dt: torch.Tensor, x: torch.Tensor) -> torch.Tensor:
    """A per-head step [rows, heads] is passed as a [rows, heads, dim] view
    with stride 0 over dim (MATE prewarm: dt_dim = 1)."""
    if dt.dim() == x.dim() - 1:
        return dt.unsqueeze(-1).expand(*dt.shape, x.shape[-1])
    return dt


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


def _on_device_of_first(fn):
    """Run a wrapper with the device of its first tensor argument current, so
    that the launch, the default stream and the library's per-device set-up
    all belong to the device the operands live on."""
    @functools.wraps(fn)
    def wrapper(*args, **kwargs):
        t = args[0] if args else next(iter(kwargs.values()), None)
        if isinstance(t, torch.Tensor) and t.is_cuda and t.device.index != torch.cuda.current_device():
            with torch.cuda.device(t.device):
                return fn(*args, **kwargs)
        return fn(*args, **kwargs)
    return wrapper


@_on_device_of_first
def ssu_update_onetoken(state, x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=False,
                        state_batch_indices=None, dst_state_batch_indices=None, pad_slot_id=-1,
                        out=None, disable_state_update=False, status=None, stream=None,
                        unsupported: int = 0) -> torch.Tensor:
    """One decode token per sequence: x, dt, z are [batch, heads, dim] (dt may
    be [batch, heads]), B and C [batch, groups, dstate].  The state is updated
    in place; returns y ([batch, heads, dim], x's dtype)."""
    dt = _dt3(dt, x)
    if out is None:
        out = torch.empty_like(x)
    a = _args(state, x, dt, A, B, C, D, z, dt_bias, dt_softplus, pad_slot_id, out,
              disable_state_update, status, unsupported)
    rt = _table(state_batch_indices, SLOTS_STRIDED)
    wt = _table(dst_state_batch_indices, SLOTS_STRIDED)
    rc = lib().ssu_update_onetoken(ctypes.byref(a), x.shape[0], None if rt is None else ctypes.byref(rt),
                                   None if wt is None else ctypes.byref(wt), _stream(stream))
    if rc != OK:
        _raise(rc)
    return out


@_on_device_of_first
def ssu_selftest_timeout(state, x, dt, A, B, C, withhold_unit: int, wait_cycles: int, D=None, z=None,
                         dt_bias=None, dt_softplus=False, state_batch_indices=None, dst_state_batch_indices=None,
                         pad_slot_id=-1, out=None, status=None, stream=None) -> torch.Tensor:
    """Test of the kernels' exit path (``ssu_selftest_timeout`` in
    ``include/ssu.h``): the one-token update with unit ``withhold_unit``
    never staged and every wait limited to ``wait_cycles`` SM cycles; the
    device status gets DEV_TIMEOUT.  Returns y (partly unwritten)."""
    dt = _dt3(dt, x)
    if out is None:
        out = torch.empty_like(x)
    a = _args(state, x, dt, A, B, C, D, z, dt_bias, dt_softplus, pad_slot_id, out, False, status, 0)
    rt = _table(state_batch_indices, SLOTS_STRIDED)
    wt = _table(dst_state_batch_indices, SLOTS_STRIDED)
    rc = lib().ssu_selftest_timeout(ctypes.byref(a), x.shape[0], None if rt is None else ctypes.byref(rt),
                                    None if wt is None else ctypes.byref(wt), int(withhold_unit), int(wait_cycles),
                                    _stream(stream))
    if rc != OK:
        _raise(rc)
    return out


@_on_device_of_first
def ssu_update_packed(state, x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=False,
                      state_batch_indices=None, dst_state_batch_indices=None, pad_slot_id=-1,
                      out=None, disable_state_update=False, cu_seqlens=None, num_accepted_tokens=None,
                      slot_mode: int = SLOTS_STRIDED, status=None, stream=None,
                      unsupported: int = 0) -> torch.Tensor:
    """Packed rows: x is [rows, heads, dim] with ``cu_seqlens`` ([nseq+1]), or
    the dense [nseq, steps, heads, dim] form without it (dt, z, B, C, out
    shaped alike).  ``slot_mode`` selects the table addressing
    (SLOTS_STRIDED: entry b*s0 + t*s1; SLOTS_PER_ROW: cu_seqlens[b] + t)."""
    steps = 0
    dense_shape = None
    if x.dim() == 4:
        _need(cu_seqlens is None, "the dense [batch, steps, heads, dim] form takes no cu_seqlens")
        nseq, steps = x.shape[0], x.shape[1]
        dense_shape = x.shape
        flat = lambda t: None if t is None else t.reshape(nseq * steps, *t.shape[2:])
        x, z, B, C = flat(x), flat(z), flat(B), flat(C)
        dt = flat(dt)
        if out is not None:
            _need(tuple(out.shape) == tuple(dense_shape), "out must have the shape of x")
            out_flat = out.view(nseq * steps, *out.shape[2:])
        else:
            out_flat = None
    else:
        _need(cu_seqlens is not None, "packed [rows, heads, dim] rows need cu_seqlens")
        nseq = cu_seqlens.numel() - 1
        out_flat = out
    dt = _dt3(dt, x)
    if out_flat is None:
        out_flat = torch.empty_like(x)
    meta_type = 0
    for t in (cu_seqlens, num_accepted_tokens):
        if t is not None:
            _need(t.dtype in _ITYPE and t.is_cuda and t.is_contiguous(),
                  "cu_seqlens / num_accepted_tokens must be contiguous int32/int64 CUDA tensors")
    if cu_seqlens is not None and num_accepted_tokens is not None:
        _need(cu_seqlens.dtype == num_accepted_tokens.dtype,
              "cu_seqlens and num_accepted_tokens must share one dtype")
    meta = cu_seqlens if cu_seqlens is not None else num_accepted_tokens
    if meta is not None:
        meta_type = _ITYPE[meta.dtype]
    if num_accepted_tokens is not None:
        _need(num_accepted_tokens.numel() >= nseq, "num_accepted_tokens needs one entry per sequence")
    a = _args(state, x, dt, A, B, C, D, z, dt_bias, dt_softplus, pad_slot_id, out_flat,
              disable_state_update, status, unsupported)
    rt = _table(state_batch_indices, slot_mode)
    wt = _table(dst_state_batch_indices, slot_mode)
    rc = lib().ssu_update_packed(ctypes.byref(a), nseq, x.shape[0], _ptr(cu_seqlens), steps,
                                 _ptr(num_accepted_tokens), meta_type,
                                 None if rt is None else ctypes.byref(rt),
                                 None if wt is None else ctypes.byref(wt), _stream(stream))
    if rc != OK:
        _raise(rc)
    if dense_shape is not None:
        return out if out is not None else out_flat.view(dense_shape)
    return out_flat


@_on_device_of_first
def ssu_replay_update(state, x, dt, A, B, C, x_buf, dt_buf, B_buf, count_in, count_out=None, D=None, z=None,
                      dt_bias=None, dt_softplus=False, state_batch_indices=None, pad_slot_id=-1, out=None,
                      status=None, stream=None, shadow=None, shadow_scale=None):
    """One decode token per sequence on the checkpoint + buffer form of the
    state (article "ReplaySSM: Cache SSM Inputs, Not State", section 核心做法).

    ``state`` holds the checkpoints ``[slots, heads, dim, dstate]``; the buffers
    are ``x_buf`` ``[slots, L, heads, dim]`` (x's dtype), ``dt_buf`` (same
    shape, fp32 processed steps) and ``B_buf`` ``[slots, L, groups, dstate]``;
    ``count_in`` ``[batch]`` int32 gives the entries buffered per sequence.
    Returns ``(y, count_out)``; pass ``count_out`` as the next call's
    ``count_in``."""
    dt = _dt3(dt, x)
    if out is None:
        out = torch.empty_like(x)
    batch = x.shape[0]
    if count_out is None:
        count_out = torch.empty_like(count_in)
    slots, heads, dim, dstate = state.shape
    _need(x_buf.dim() == 4 and x_buf.shape[0] == slots and tuple(x_buf.shape[2:]) == (heads, dim),
          "x_buf must be [slots, L, heads, dim]")
    L = x_buf.shape[1]
    _need(x_buf.dtype == x.dtype and x_buf.is_contiguous(), "x_buf must be contiguous in x's dtype")
    _need(tuple(dt_buf.shape) == tuple(x_buf.shape) and dt_buf.dtype == torch.float32 and dt_buf.is_contiguous(),
          "dt_buf must be a contiguous fp32 tensor shaped like x_buf")
    _need(B_buf.dim() == 4 and tuple(B_buf.shape) == (slots, L, B.shape[1], dstate) and B_buf.dtype == x.dtype
          and B_buf.is_contiguous(), "B_buf must be [slots, L, groups, dstate], contiguous, in x's dtype")
    for t in (count_in, count_out):
        _need(t.dtype == torch.int32 and t.is_cuda and t.is_contiguous() and t.numel() >= batch,
              "counts must be contiguous int32 CUDA tensors with one entry per sequence")
    _need(all(t.is_cuda for t in (x_buf, dt_buf, B_buf)), "buffers must be CUDA tensors")
    a = _args(state, x, dt, A, B, C, D, z, dt_bias, dt_softplus, pad_slot_id, out, False, status, 0)
    rt = _table(state_batch_indices, SLOTS_STRIDED)
    fmt = _shadow_format(shadow, state)
    if fmt != SHADOW_NONE:
        shape = (*state.shape[:-1], state.shape[-1] // 2) if fmt == SHADOW_NVFP4 else tuple(state.shape)
        _need(shadow.is_cuda and shadow.is_contiguous() and tuple(shadow.shape) == shape,
              "the read copy must be a contiguous CUDA tensor shaped like the checkpoints")
        _check_copy_scales(fmt, shadow_scale, state)
    rb = ReplayBuffers(L, x_buf.data_ptr(), dt_buf.data_ptr(), B_buf.data_ptr(), count_in.data_ptr(),
                       count_out.data_ptr(), fmt, 0, _ptr(shadow),
                       _ptr(shadow_scale) if fmt in (SHADOW_E4M3, SHADOW_NVFP4) else None)
    rc = lib().ssu_replay_update(ctypes.byref(a), batch, None if rt is None else ctypes.byref(rt),
                                 ctypes.byref(rb), _stream(stream))
    if rc != OK:
        _raise(rc)
    return out, count_out


@_on_device_of_first
def ssu_replay_verify(state, x, dt, A, B, C, x_buf, dt_buf, B_buf, count_in, count_out=None, D=None, z=None,
                      dt_bias=None, dt_softplus=False, state_batch_indices=None, pad_slot_id=-1, out=None,
                      status=None, stream=None):
    """Speculative decoding on the checkpoint + buffer form (article "ReplaySSM",
    section 投机解码回滚): x ``[batch, T, heads, dim]``, dt the same (or
    ``[batch, T, heads]``), B, C ``[batch, T, groups, dstate]``, z like x; the
    checkpoints and buffers as for :func:`ssu_replay_update`.  The drafts are
    appended after the ``count_in`` committed entries and verified; returns
    ``(y [batch, T, heads, dim], count_out)`` with count_out the committed
    entries (the flush, when it fires, leaves 0).  Accepting the first ``a``
    drafts of sequence b is ``count[b] = count_out[b] + a``."""
    _need(x.dim() == 4 and B.dim() == 4, "x must be [batch, T, heads, dim], B [batch, T, groups, dstate]")
    batch, T = x.shape[0], x.shape[1]
    if dt.dim() == 3:
        dt = dt.unsqueeze(-1).expand(*dt.shape, x.shape[-1])
    if out is None:
        out = torch.empty_like(x)
    if count_out is None:
        count_out = torch.empty_like(count_in)
    slots, heads, dim, dstate = state.shape
    for name, t in (("x", x), ("out", out)) + ((("z", z),) if z is not None else ()):
        _need(t.is_contiguous(), f"{name} must be contiguous")
    _need(B.is_contiguous() and C.is_contiguous(), "B and C must be contiguous")
    _need(x_buf.dim() == 4 and x_buf.shape[0] == slots and tuple(x_buf.shape[2:]) == (heads, dim),
          "x_buf must be [slots, L, heads, dim]")
    L = x_buf.shape[1]
    _need(x_buf.dtype == x.dtype and x_buf.is_contiguous(), "x_buf must be contiguous in x's dtype")
    _need(tuple(dt_buf.shape) == tuple(x_buf.shape) and dt_buf.dtype == torch.float32 and dt_buf.is_contiguous(),
          "dt_buf must be a contiguous fp32 tensor shaped like x_buf")
    _need(B_buf.dim() == 4 and tuple(B_buf.shape) == (slots, L, B.shape[2], dstate) and B_buf.dtype == x.dtype
          and B_buf.is_contiguous(), "B_buf must be [slots, L, groups, dstate], contiguous, in x's dtype")
    for t in (count_in, count_out):
        _need(t.dtype == torch.int32 and t.is_cuda and t.is_contiguous() and t.numel() >= batch,
              "counts must be contiguous int32 CUDA tensors with one entry per sequence")
    _need(all(t.is_cuda for t in (x_buf, dt_buf, B_buf)), "buffers must be CUDA tensors")
    rows = batch * T
    flat = lambda t: None if t is None else t.reshape(rows, *t.shape[2:])
    a = _args(state, flat(x), flat(dt), A, flat(B), flat(C), D, flat(z), dt_bias, dt_softplus, pad_slot_id,
              flat(out), False, status, 0)
    rt = _table(state_batch_indices, SLOTS_STRIDED)
    rb = ReplayBuffers(L, x_buf.data_ptr(), dt_buf.data_ptr(), B_buf.data_ptr(), count_in.data_ptr(),
                       count_out.data_ptr(), SHADOW_NONE, 0, None, None)
    rc = lib().ssu_replay_verify(ctypes.byref(a), batch, T, None if rt is None else ctypes.byref(rt),
                                 ctypes.byref(rb), _stream(stream))
    if rc != OK:
        _raise(rc)
    return out, count_out


_SSD_WORKSPACE = {}


def _ssd_workspace(device, nbytes: int, stream) -> torch.Tensor:
    """A workspace per (device, stream) that only grows (the "cached
    workspace" of the MATE page): a steady-state call allocates nothing, and
    calls on different streams never share one.  It is allocated on the
    stream the call runs on, so the caching allocator hands a replaced one
    out again only after that stream's work on it."""
    handle = _stream(stream)
    key = (str(device), handle)
    ws = _SSD_WORKSPACE.get(key)
    if ws is None or ws.numel() < nbytes:
        if stream is None:  # the call runs on the current stream
            ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        else:
            s = stream if isinstance(stream, torch.cuda.Stream) else torch.cuda.ExternalStream(handle, device=device)
            with torch.cuda.stream(s):
                ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _SSD_WORKSPACE[key] = ws
    return ws


@_on_device_of_first
def ssu_ssd_prefill(x, dt, A, B, C, chunk_size: int, cu_chunk_seqlens, seq_idx, last_chunk_indices=None,
                    out=None, D=None, z=None, dt_bias=None, dt_softplus=False, dt_limit=(0.0, float("inf")),
                    initial_states=None, return_intermediate_states=False, state_dtype=None, nseq=None,
                    status=None, stream=None):
    """Packed variable-length SSD prefill (see ``include/ssu.h``).  x ``[tokens,
    heads, dim]`` bf16, dt ``[tokens, heads]``, B, C ``[tokens, groups,
    dstate]`` bf16.  Returns (y, states)."""
    _need(x.dim() == 3 and dt.dim() == 2 and B.dim() == 3 and C.shape == B.shape, "x, dt, B, C shapes")
    tokens, heads, dim = x.shape
    groups, dstate = B.shape[1], B.shape[2]
    _need(dt.shape == (tokens, heads) and B.shape[0] == tokens, "dt must be [tokens, heads], B [tokens, ...]")
    for t in (x, dt, B, C, z, out, initial_states):
        _need(t is None or (t.is_cuda and t.is_contiguous()), "tensors must be contiguous CUDA tensors")
    meta = cu_chunk_seqlens.dtype
    _need(meta in _ITYPE and seq_idx.dtype == meta and (last_chunk_indices is None or last_chunk_indices.dtype == meta),
          "cu_chunk_seqlens, seq_idx and last_chunk_indices share one integer dtype")
    nchunks = seq_idx.numel()
    if nseq is None:
        nseq = last_chunk_indices.numel() if last_chunk_indices is not None else initial_states.shape[0]
    sdt = state_dtype or (initial_states.dtype if initial_states is not None else C.dtype)
    out = out if out is not None else torch.empty_like(x)
    states = torch.empty(((nchunks if return_intermediate_states else nseq), heads, dim, dstate), dtype=sdt,
                         device=x.device)
    if initial_states is not None and initial_states.dtype != sdt:
        initial_states = initial_states.to(sdt)
    nbytes = ctypes.c_uint64(0)
    rc = lib().ssu_ssd_workspace_size(nchunks, heads, groups, dim, dstate, chunk_size, ctypes.byref(nbytes))
    if rc != OK:
        _raise(rc)
    ws = _ssd_workspace(x.device, nbytes.value, stream)
    hi = float(dt_limit[1])
    a = SsdArgs(tokens=tokens, heads=heads, dim=dim, dstate=dstate, groups=groups, nseq=nseq, nchunks=nchunks,
                chunk_size=chunk_size, io_dtype=_DTYPE.get(x.dtype, -1), dt_dtype=_DTYPE[dt.dtype],
                state_dtype=_DTYPE[sdt], meta_type=_ITYPE[meta], dt_softplus=int(bool(dt_softplus)),
                return_intermediate=int(bool(return_intermediate_states)), dt_min=float(dt_limit[0]),
                dt_max=min(hi, 3.4028234663852886e38),
                x=x.data_ptr(), dt=dt.data_ptr(), B=B.data_ptr(), C=C.data_ptr(), z=_ptr(z), A=A.data_ptr(),
                D=_ptr(D), dt_bias=_ptr(dt_bias), cu_chunk_seqlens=cu_chunk_seqlens.data_ptr(),
                seq_idx=seq_idx.data_ptr(), last_chunk_indices=_ptr(last_chunk_indices),
                initial_states=_ptr(initial_states), y=out.data_ptr(), states=states.data_ptr(),
                workspace=ws.data_ptr(), workspace_bytes=ws.numel(), d_status=_ptr(status))
    rc = lib().ssu_ssd_prefill(ctypes.byref(a), _stream(stream))
    if rc != OK:
        _raise(rc)
    return out, states


SSD_STATIC_SCRATCH_BYTES = 64 << 20  # SSU_SSD_STATIC_SCRATCH_BYTES


@_on_device_of_first
def ssu_ssd_prefill_static(x, dt, A, B, C, chunk_size: int, cu_chunk_seqlens, seq_idx, last_chunk_indices=None,
                           out=None, D=None, z=None, dt_bias=None, dt_softplus=False, dt_limit=(0.0, float("inf")),
                           initial_states=None, return_intermediate_states=False, state_dtype=None, nseq=None,
                           status=None, stream=None):
    """ssu_ssd_prefill on the library's own scratch (``ssu_ssd_prefill_static``
    in ``include/ssu.h``): no workspace is allocated; the call's workspace must
    fit SSD_STATIC_SCRATCH_BYTES, and calls must not overlap in time.
    Returns (y, states)."""
    _need(x.dim() == 3 and dt.dim() == 2 and B.dim() == 3 and C.shape == B.shape, "x, dt, B, C shapes")
    tokens, heads, dim = x.shape
    groups, dstate = B.shape[1], B.shape[2]
    _need(dt.shape == (tokens, heads) and B.shape[0] == tokens, "dt must be [tokens, heads], B [tokens, ...]")
    for t in (x, dt, B, C, z, out, initial_states):
        _need(t is None or (t.is_cuda and t.is_contiguous()), "tensors must be contiguous CUDA tensors")
    meta = cu_chunk_seqlens.dtype
    _need(meta in _ITYPE and seq_idx.dtype == meta and (last_chunk_indices is None or last_chunk_indices.dtype == meta),
          "cu_chunk_seqlens, seq_idx and last_chunk_indices share one integer dtype")
    nchunks = seq_idx.numel()
    if nseq is None:
        nseq = last_chunk_indices.numel() if last_chunk_indices is not None else initial_states.shape[0]
    sdt = state_dtype or (initial_states.dtype if initial_states is not None else C.dtype)
    out = out if out is not None else torch.empty_like(x)
    states = torch.empty(((nchunks if return_intermediate_states else nseq), heads, dim, dstate), dtype=sdt,
                         device=x.device)
    if initial_states is not None and initial_states.dtype != sdt:
        initial_states = initial_states.to(sdt)
    hi = float(dt_limit[1])
    a = SsdArgs(tokens=tokens, heads=heads, dim=dim, dstate=dstate, groups=groups, nseq=nseq, nchunks=nchunks,
                chunk_size=chunk_size, io_dtype=_DTYPE.get(x.dtype, -1), dt_dtype=_DTYPE[dt.dtype],
                state_dtype=_DTYPE[sdt], meta_type=_ITYPE[meta], dt_softplus=int(bool(dt_softplus)),
                return_intermediate=int(bool(return_intermediate_states)), dt_min=float(dt_limit[0]),
                dt_max=min(hi, 3.4028234663852886e38),
                x=x.data_ptr(), dt=dt.data_ptr(), B=B.data_ptr(), C=C.data_ptr(), z=_ptr(z), A=A.data_ptr(),
                D=_ptr(D), dt_bias=_ptr(dt_bias), cu_chunk_seqlens=cu_chunk_seqlens.data_ptr(),
                seq_idx=seq_idx.data_ptr(), last_chunk_indices=_ptr(last_chunk_indices),
                initial_states=_ptr(initial_states), y=out.data_ptr(), states=states.data_ptr(),
                workspace=None, workspace_bytes=0, d_status=_ptr(status))
    rc = lib().ssu_ssd_prefill_static(ctypes.byref(a), _stream(stream))
    if rc != OK:
        _raise(rc)
    return out, states


@_on_device_of_first
def ssd_combined_fwd_varlen(x, dt, A, B, C, chunk_size, cu_seqlens, cu_chunk_seqlens, last_chunk_indices, seq_idx,
                            out=None, D=None, z=None, dt_bias=None, dt_softplus=False, dt_limit=(0.0, float("inf")),
                            initial_states=None, return_intermediate_states=False, state_dtype=None,
                            checkpoint_token_indices=None, checkpoint_state_slots=None, checkpoint_states=None):
    """The MATE-shaped prefill call (MATE "Mamba / SSU", API reference of
    ssd_combined_fwd_varlen): y into ``out`` (allocated when None), returns
    the state buffer.  The checkpoint_* arguments are not implemented and
    raise."""
    if any(v is not None for v in (checkpoint_token_indices, checkpoint_state_slots, checkpoint_states)):
        raise NotImplementedError("checkpoint_* (replay checkpoints during prefill) is not implemented")
    _, states = ssu_ssd_prefill(x, dt, A, B, C, chunk_size, cu_chunk_seqlens, seq_idx, last_chunk_indices, out=out,
                                D=D, z=z, dt_bias=dt_bias, dt_softplus=dt_softplus, dt_limit=dt_limit,
                                initial_states=initial_states, return_intermediate_states=return_intermediate_states,
                                state_dtype=state_dtype, nseq=cu_seqlens.numel() - 1)
    return states


@_on_device_of_first
def ssu_shadow_refresh(state: torch.Tensor, shadow: torch.Tensor, shadow_scale: Optional[torch.Tensor] = None,
                       stream=None) -> None:
    """The low-precision read copy of a contiguous state tensor ``[..., dstate]``
    into ``shadow``: float16 values; uint8 / float8_e4m3fn E4M3 codes with fp32
    ``shadow_scale`` of shape ``state.shape[:-1]``; or NVFP4 -- uint8 code
    pairs of shape ``[..., dstate / 2]`` with fp32 scale records of shape
    ``[..., nvfp4_scale_words(dstate)]``."""
    fmt = _shadow_format(shadow, state)
    _need(fmt != SHADOW_NONE, "shadow must be given")
    shape = (*state.shape[:-1], state.shape[-1] // 2) if fmt == SHADOW_NVFP4 else tuple(state.shape)
    _need(state.is_cuda and state.is_contiguous() and shadow.is_cuda and shadow.is_contiguous()
          and tuple(shadow.shape) == shape, "state and shadow must be contiguous CUDA tensors of matching shapes")
    _check_copy_scales(fmt, shadow_scale, state)
    dstate = state.shape[-1]
    rc = lib().ssu_shadow_refresh(state.data_ptr(), _DTYPE[state.dtype], state.numel() // dstate, dstate, fmt,
                                  shadow.data_ptr(), _ptr(shadow_scale) if fmt != SHADOW_F16 else None,
                                  _stream(stream))
    if rc != OK:
        _raise(rc)


@_on_device_of_first
def ssu_batch_copy(copies: torch.Tensor, max_bytes: int, status: Optional[torch.Tensor] = None,
                   stream=None) -> None:
    """Batched copies with memmove semantics (see ``include/ssu.h``).

    ``copies`` is a contiguous int64 CUDA tensor ``[n, 3]`` of (source
    address, destination address, bytes), e.g. from ``copy_table`` or
    ``slot_copies``; ``max_bytes`` bounds every copy's length."""
    _need(copies.dtype == torch.int64 and copies.dim() == 2 and copies.shape[1] == 3 and copies.is_contiguous(),
          "copies must be a contiguous int64 [n, 3] tensor")
    _need(copies.is_cuda or copies.numel() == 0, "copies must be a CUDA tensor")
    _need(max_bytes >= 0, "max_bytes must not be negative")
    if status is not None:
        _need(status.dtype == torch.int32 and status.is_cuda, "status must be an int32 CUDA tensor")
    rc = lib().ssu_batch_copy(copies.data_ptr() if copies.numel() else None, copies.shape[0], max_bytes,
                              _ptr(status), _stream(stream))
    if rc != OK:
        _raise(rc)


def copy_table(entries, device) -> torch.Tensor:
    """Descriptors ``[n, 3]`` from (source address, destination address,
    bytes) triples."""
    return torch.tensor(list(entries), dtype=torch.int64).reshape(-1, 3).to(device)


def slot_copies(pool: torch.Tensor, src_slots: torch.Tensor, dst_slots: torch.Tensor) -> torch.Tensor:
    """Descriptors copying whole slots of a contiguous pool ``[slots, ...]``:
    slot src_slots[i] to slot dst_slots[i] (addresses computed on the device,
    no host round trip)."""
    _need(pool.is_contiguous(), "pool must be contiguous")
    _need(src_slots.shape == dst_slots.shape and src_slots.dim() == 1, "slot lists must be 1-D and equal in length")
    slot_bytes = pool[0].numel() * pool.element_size()
    base = pool.data_ptr()
    s = src_slots.to(device=pool.device, dtype=torch.int64) * slot_bytes + base
    d = dst_slots.to(device=pool.device, dtype=torch.int64) * slot_bytes + base
    return torch.stack([s, d, torch.full_like(s, slot_bytes)], dim=1).contiguous()


def ssu_prewarm(*, state_dtype: torch.dtype, io_dtype: torch.dtype, heads: int, dim: int,
                dstate: int, groups: int, dt_dtype: torch.dtype = torch.float32,
                packed: bool = False) -> None:
    """Load the kernel of one configuration on the current device, outside
    any graph capture (MATE "Mamba / SSU", Graph capture)."""
    rc = lib().ssu_prewarm(_DTYPE[state_dtype], _DTYPE[io_dtype], _DTYPE[dt_dtype], heads, dim,
                           dstate, groups, int(bool(packed)))
    if rc != OK:
        _raise(rc)


@_on_device_of_first
def selective_state_update(state, x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=False,
                           state_batch_indices=None, pad_slot_id=-1, state_scale=None, out=None,
                           disable_state_update=False, intermediate_states_buffer=None,
                           intermediate_state_indices=None, intermediate_state_scales=None,
                           rand_seed=None, philox_rounds=10, cache_steps=0, algorithm="auto",
                           dst_state_batch_indices=None, cu_seqlens=None, num_accepted_tokens=None,
                           backend="auto", slot_mode: int = SLOTS_STRIDED, status=None):
    """The MATE / FlashInfer-shaped entry (argument order and defaults of the
    MATE "Mamba / SSU" API reference).  The call shape picks the kernel: a 4-D
    x, cu_seqlens or num_accepted_tokens go to the packed kernel, anything
    else to the one-token kernel.  Arguments without implemented semantics
    raise NotImplementedError."""
    unsup = 0
    if rand_seed is not None:
        unsup |= UNSUP_RAND_SEED
    if state_scale is not None:
        unsup |= UNSUP_STATE_SCALE
    if (intermediate_states_buffer is not None or intermediate_state_indices is not None
            or intermediate_state_scales is not None):
        unsup |= UNSUP_INTERMEDIATE
    if cache_steps != 0:
        unsup |= UNSUP_CACHE_STEPS
    if algorithm != "auto" or backend != "auto":
        unsup |= UNSUP_ALGORITHM
    common = dict(D=D, z=z, dt_bias=dt_bias, dt_softplus=dt_softplus,
                  state_batch_indices=state_batch_indices,
                  dst_state_batch_indices=dst_state_batch_indices, pad_slot_id=pad_slot_id, out=out,
                  disable_state_update=disable_state_update, status=status, unsupported=unsup)
    if x.dim() == 4 or cu_seqlens is not None or num_accepted_tokens is not None:
        if x.dim() == 3 and cu_seqlens is None:
            # num_accepted_tokens alone on [batch, heads, dim]: one token per sequence
            cu_seqlens = torch.arange(0, x.shape[0] + 1, device=x.device,
                                      dtype=num_accepted_tokens.dtype)
        return ssu_update_packed(state, x, dt, A, B, C, cu_seqlens=cu_seqlens,
                                 num_accepted_tokens=num_accepted_tokens, slot_mode=slot_mode, **common)
    return ssu_update_onetoken(state, x, dt, A, B, C, **common)
