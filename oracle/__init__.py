"""Double-precision CPU oracle for the Mamba-2 selective state update.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never calls it, and it shares no code with the CUDA library.

The arithmetic lives in ``ssu_oracle.c`` (plain C, double precision); this
module compiles it with gcc and marshals torch CPU tensors into it.  The
semantics it follows are those of the "Mamba / SSU" page of the MATE
documentation ("SSU at a glance" and the API reference) and of the recurrence
written out in the article "ReplaySSM: Cache SSM Inputs, Not State"
(section 三个瓶颈); ``ssu_oracle.c`` gives the passage for each step.

Functions with no pin by the pages: the head -> group map (contiguous blocks,
``g = h // (heads // groups)``) is a convention; parity for it is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssu_oracle.c")
_HDR = os.path.join(_HERE, "ssu_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libssu_oracle.so")

F32, F16, BF16, F64 = 0, 1, 2, 3
OK, INVALID, ALIASING = 0, 1, 2
SLOTS_STRIDED, SLOTS_PER_ROW = 0, 1
TOUCH_READ, TOUCH_WRITTEN = 1, 2

_DTYPE_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16, torch.float64: F64}

from .memcopy import batch_copy  # noqa: E402  (batched copies with memmove semantics)


class OracleError(RuntimeError):
    """The oracle rejected its inputs (``code`` is INVALID or ALIASING)."""

    def __init__(self, code: int, msg: str):
        super().__init__(f"oracle rejected the inputs ({'aliasing' if code == ALIASING else 'invalid'}): {msg}")
        self.code = code


def build(force: bool = False) -> str:
    """Compile ``ssu_oracle.c`` into ``oracle/_build/libssu_oracle.so``."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = force or not os.path.exists(_LIB_PATH) or max(
        os.path.getmtime(_SRC), os.path.getmtime(_HDR)) > os.path.getmtime(_LIB_PATH)
    if stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-Wall", "-Wextra",
                        "-fno-fast-math", _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Table(ctypes.Structure):
    _fields_ = [("entries", ctypes.c_void_p), ("s0", ctypes.c_int64), ("s1", ctypes.c_int64),
                ("extent", ctypes.c_int64), ("mode", ctypes.c_int32)]


class _Problem(ctypes.Structure):
    _fields_ = [
        ("slots", ctypes.c_int64), ("heads", ctypes.c_int64), ("dim", ctypes.c_int64),
        ("dstate", ctypes.c_int64), ("groups", ctypes.c_int64),
        ("state_dtype", ctypes.c_int32), ("io_dtype", ctypes.c_int32), ("dt_dtype", ctypes.c_int32),
        ("dt_per_head", ctypes.c_int32),
        ("state_in", ctypes.c_void_p), ("state_out", ctypes.c_void_p),
        ("x", ctypes.c_void_p), ("dt", ctypes.c_void_p), ("B", ctypes.c_void_p),
        ("C", ctypes.c_void_p), ("z", ctypes.c_void_p),
        ("A", ctypes.c_void_p), ("D", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("y", ctypes.c_void_p), ("y_exact", ctypes.c_void_p),
        ("dt_softplus", ctypes.c_int32), ("disable_state_update", ctypes.c_int32),
        ("pad_slot_id", ctypes.c_int64),
        ("nseq", ctypes.c_int64), ("rows", ctypes.c_int64),
        ("cu_seqlens", ctypes.c_void_p), ("num_accepted", ctypes.c_void_p),
        ("read", _Table), ("dst", _Table),
        ("slot_touched", ctypes.c_void_p),
    ]


class _ReplayProblem(ctypes.Structure):
    _fields_ = [
        ("slots", ctypes.c_int64), ("heads", ctypes.c_int64), ("dim", ctypes.c_int64),
        ("dstate", ctypes.c_int64), ("groups", ctypes.c_int64),
        ("state_dtype", ctypes.c_int32), ("io_dtype", ctypes.c_int32), ("dt_dtype", ctypes.c_int32),
        ("dt_per_head", ctypes.c_int32),
        ("ckpt_in", ctypes.c_void_p), ("ckpt_out", ctypes.c_void_p),
        ("x", ctypes.c_void_p), ("dt", ctypes.c_void_p), ("B", ctypes.c_void_p),
        ("C", ctypes.c_void_p), ("z", ctypes.c_void_p),
        ("A", ctypes.c_void_p), ("D", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("y", ctypes.c_void_p), ("y_exact", ctypes.c_void_p),
        ("dt_softplus", ctypes.c_int32), ("pad_slot_id", ctypes.c_int64), ("batch", ctypes.c_int64),
        ("slot_of", ctypes.c_void_p), ("len", ctypes.c_int64),
        ("xbuf", ctypes.c_void_p), ("dtbuf", ctypes.c_void_p), ("Bbuf", ctypes.c_void_p),
        ("count_in", ctypes.c_void_p), ("count_out", ctypes.c_void_p),
        ("shadow_format", ctypes.c_int32), ("shadow", ctypes.c_void_p), ("shadow_scale", ctypes.c_void_p),
    ]


class _VerifyProblem(ctypes.Structure):
    _fields_ = [
        ("slots", ctypes.c_int64), ("heads", ctypes.c_int64), ("dim", ctypes.c_int64),
        ("dstate", ctypes.c_int64), ("groups", ctypes.c_int64),
        ("state_dtype", ctypes.c_int32), ("io_dtype", ctypes.c_int32), ("dt_dtype", ctypes.c_int32),
        ("dt_per_head", ctypes.c_int32),
        ("ckpt_in", ctypes.c_void_p), ("ckpt_out", ctypes.c_void_p),
        ("x", ctypes.c_void_p), ("dt", ctypes.c_void_p), ("B", ctypes.c_void_p),
        ("C", ctypes.c_void_p), ("z", ctypes.c_void_p),
        ("A", ctypes.c_void_p), ("D", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("y", ctypes.c_void_p), ("y_exact", ctypes.c_void_p),
        ("dt_softplus", ctypes.c_int32), ("pad_slot_id", ctypes.c_int64), ("batch", ctypes.c_int64),
        ("ntok", ctypes.c_int64), ("slot_of", ctypes.c_void_p), ("len", ctypes.c_int64),
        ("xbuf", ctypes.c_void_p), ("dtbuf", ctypes.c_void_p), ("Bbuf", ctypes.c_void_p),
        ("count_in", ctypes.c_void_p), ("count_out", ctypes.c_void_p),
    ]


class _SsdProblem(ctypes.Structure):
    _fields_ = [
        ("tokens", ctypes.c_int64), ("heads", ctypes.c_int64), ("dim", ctypes.c_int64),
        ("dstate", ctypes.c_int64), ("groups", ctypes.c_int64), ("nchunks", ctypes.c_int64),
        ("nseq", ctypes.c_int64),
        ("io_dtype", ctypes.c_int32), ("dt_dtype", ctypes.c_int32), ("state_dtype", ctypes.c_int32),
        ("x", ctypes.c_void_p), ("dt", ctypes.c_void_p), ("B", ctypes.c_void_p), ("C", ctypes.c_void_p),
        ("z", ctypes.c_void_p), ("A", ctypes.c_void_p), ("D", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("dt_softplus", ctypes.c_int32), ("dt_lo", ctypes.c_double), ("dt_hi", ctypes.c_double),
        ("cu_chunk", ctypes.c_void_p), ("seq_idx", ctypes.c_void_p), ("initial_states", ctypes.c_void_p),
        ("y", ctypes.c_void_p), ("y_exact", ctypes.c_void_p), ("states", ctypes.c_void_p),
    ]


# Formats of the low-precision read copy (ssu_oracle.h, ORC_SHADOW_*).
SHADOW_NONE, SHADOW_F16, SHADOW_E4M3, SHADOW_NVFP4 = 0, 1, 2, 3


def nvfp4_scale_words(dstate: int) -> int:
    """Floats of one row's NVFP4 scale record (ssu_oracle.h): the fp32 row
    scale, then the dstate / 16 E4M3 block-scale codes as bytes, padded to a
    multiple of 16 bytes."""
    return (4 + dstate // 16 + 15) // 16 * 4

_lib = None


def load_library(path: str):
    """Load a compiled oracle from ``path`` and declare its C signatures."""
    lib = ctypes.CDLL(path)
    lib.orc_ssu_run.argtypes = [ctypes.POINTER(_Problem), ctypes.c_char_p, ctypes.c_int]
    lib.orc_ssu_run.restype = ctypes.c_int
    lib.orc_replay_run.argtypes = [ctypes.POINTER(_ReplayProblem), ctypes.c_char_p, ctypes.c_int]
    lib.orc_replay_run.restype = ctypes.c_int
    lib.orc_replay_verify_run.argtypes = [ctypes.POINTER(_VerifyProblem), ctypes.c_char_p, ctypes.c_int]
    lib.orc_replay_verify_run.restype = ctypes.c_int
    lib.orc_softplus.argtypes = [ctypes.c_double]
    lib.orc_softplus.restype = ctypes.c_double
    lib.orc_silu.argtypes = [ctypes.c_double]
    lib.orc_silu.restype = ctypes.c_double
    lib.orc_decode.argtypes = [ctypes.c_uint32, ctypes.c_int]
    lib.orc_decode.restype = ctypes.c_double
    lib.orc_encode.argtypes = [ctypes.c_double, ctypes.c_int]
    lib.orc_encode.restype = ctypes.c_uint32
    lib.orc_ssd_run.argtypes = [ctypes.POINTER(_SsdProblem), ctypes.c_char_p, ctypes.c_int]
    lib.orc_ssd_run.restype = ctypes.c_int
    lib.orc_shadow_refresh.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    lib.orc_shadow_refresh.restype = ctypes.c_int
    lib.orc_e4m3_encode.argtypes = [ctypes.c_double]
    lib.orc_e4m3_encode.restype = ctypes.c_uint8
    lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_decode.restype = ctypes.c_double
    lib.orc_e2m1_encode.argtypes = [ctypes.c_double]
    lib.orc_e2m1_encode.restype = ctypes.c_uint8
    lib.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e2m1_decode.restype = ctypes.c_double
    lib.orc_nvfp4_scale_words.argtypes = [ctypes.c_int64]
    lib.orc_nvfp4_scale_words.restype = ctypes.c_int64
    return lib


def compile_source(src_path: str, out_path: str) -> str:
    """Compile an oracle source file (the tests use this to build deliberately
    broken copies and check that the pins catch them)."""
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fno-fast-math",
                    "-I", _HERE, src_path, "-o", out_path, "-lm"], check=True)
    return out_path


def _load():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def softplus(v: float, lib=None) -> float:
    return (lib or _load()).orc_softplus(float(v))


def silu(z: float, lib=None) -> float:
    return (lib or _load()).orc_silu(float(z))


def decode(bits: int, dtype: torch.dtype, lib=None) -> float:
    return (lib or _load()).orc_decode(int(bits), _DTYPE_CODE[dtype])


def encode(v: float, dtype: torch.dtype, lib=None) -> int:
    return int((lib or _load()).orc_encode(float(v), _DTYPE_CODE[dtype]))


@dataclass
class Table:
    """A slot table as the oracle reads it: ``entries`` flat, addressed by
    ``b*s0 + step*s1`` (STRIDED) or ``cu_seqlens[b] + step`` (PER_ROW)."""
    entries: torch.Tensor
    s0: int = 1
    s1: int = 0
    mode: int = SLOTS_STRIDED

    @staticmethod
    def of(t: Optional[torch.Tensor], mode: int = SLOTS_STRIDED) -> Optional["Table"]:
        """Stride view of a 1-D ``[n]`` table (as ``[n, 1]``) or a 2-D table."""
        if t is None:
            return None
        if t.dim() == 1:
            return Table(t, t.stride(0), t.stride(0), mode)
        return Table(t, t.stride(0), t.stride(1), mode)


def _cpu(t: Optional[torch.Tensor]) -> Optional[torch.Tensor]:
    return None if t is None else t.detach().to("cpu").contiguous()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


@dataclass
class Result:
    state: torch.Tensor        # pool after the call, state dtype
    y: torch.Tensor            # [rows, heads, dim] io dtype
    y_exact: torch.Tensor      # [rows, heads, dim] float64 before rounding
    touched: torch.Tensor      # [slots] uint8, OR of TOUCH_READ / TOUCH_WRITTEN


def ssu(state: torch.Tensor, x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor,
        B: torch.Tensor, C: torch.Tensor, D: Optional[torch.Tensor] = None,
        z: Optional[torch.Tensor] = None, dt_bias: Optional[torch.Tensor] = None,
        dt_softplus: bool = False, read: Optional[Table] = None, dst: Optional[Table] = None,
        pad_slot_id: int = -1, disable_state_update: bool = False,
        cu_seqlens: Optional[torch.Tensor] = None, num_accepted: Optional[torch.Tensor] = None,
        state_out: Optional[torch.Tensor] = None, lib=None) -> Result:
    """Run the oracle.  Tensors may live anywhere; they are copied to the host.

    Shapes: state ``[slots, heads, dim, dstate]``; x, z ``[rows, heads, dim]``;
    dt ``[rows, heads, dim]`` or ``[rows, heads]`` (per-head step);
    B, C ``[rows, groups, dstate]``; A, D, dt_bias ``[heads]`` fp32.
    With ``cu_seqlens`` None every row is its own one-token sequence.
    ``state_out`` (host, contiguous, same shape and dtype as ``state``) may be
    given to avoid a copy of a large pool; it must already hold ``state``.
    """
    lib = lib or _load()
    s_in = _cpu(state)
    slots, heads, dim, dstate = s_in.shape
    rows = x.shape[0]
    groups = B.shape[1]
    if state_out is None:
        state_out = s_in.clone()
    xs, dts, Bs, Cs, zs = _cpu(x), _cpu(dt), _cpu(B), _cpu(C), _cpu(z)
    As = _cpu(A).to(torch.float32)
    Ds = None if D is None else _cpu(D).to(torch.float32)
    bs = None if dt_bias is None else _cpu(dt_bias).to(torch.float32)
    y = torch.empty((rows, heads, dim), dtype=x.dtype)
    y_exact = torch.empty((rows, heads, dim), dtype=torch.float64)
    touched = torch.zeros(slots, dtype=torch.uint8)
    cu = None if cu_seqlens is None else _cpu(cu_seqlens).to(torch.int64)
    acc = None if num_accepted is None else _cpu(num_accepted).to(torch.int64)
    nseq = rows if cu is None else cu.numel() - 1

    keep = []

    def table(tb: Optional[Table]) -> _Table:
        if tb is None:
            return _Table(None, 0, 0, 0, SLOTS_STRIDED)
        e = _cpu(tb.entries).reshape(-1).to(torch.int64)
        keep.append(e)
        return _Table(e.data_ptr(), tb.s0, tb.s1, e.numel(), tb.mode)

    pr = _Problem(
        slots=slots, heads=heads, dim=dim, dstate=dstate, groups=groups,
        state_dtype=_DTYPE_CODE[s_in.dtype], io_dtype=_DTYPE_CODE[xs.dtype],
        dt_dtype=_DTYPE_CODE[dts.dtype], dt_per_head=int(dts.dim() == 2),
        state_in=s_in.data_ptr(), state_out=state_out.data_ptr(),
        x=xs.data_ptr(), dt=dts.data_ptr(), B=Bs.data_ptr(), C=Cs.data_ptr(), z=_ptr(zs),
        A=As.data_ptr(), D=_ptr(Ds), dt_bias=_ptr(bs),
        y=y.data_ptr(), y_exact=y_exact.data_ptr(),
        dt_softplus=int(bool(dt_softplus)), disable_state_update=int(bool(disable_state_update)),
        pad_slot_id=int(pad_slot_id), nseq=nseq, rows=rows,
        cu_seqlens=_ptr(cu), num_accepted=_ptr(acc),
        read=table(read), dst=table(dst), slot_touched=touched.data_ptr(),
    )
    for t, name in ((xs, "x"), (zs, "z")):
        if t is not None and t.dtype != xs.dtype:
            raise ValueError(f"{name} must have the io dtype")
    if Bs.dtype != xs.dtype or Cs.dtype != xs.dtype:
        raise ValueError("B and C must have the io dtype")
    err = ctypes.create_string_buffer(512)
    rc = lib.orc_ssu_run(ctypes.byref(pr), err, 512)
    if rc != OK:
        raise OracleError(rc, err.value.decode())
    return Result(state=state_out, y=y, y_exact=y_exact, touched=touched)


@dataclass
class ReplayResult:
    ckpt: torch.Tensor         # checkpoints after the call
    y: torch.Tensor            # [batch, heads, dim] io dtype
    y_exact: torch.Tensor      # float64 before rounding
    xbuf: torch.Tensor         # buffers after the call
    dtbuf: torch.Tensor
    Bbuf: torch.Tensor
    count: torch.Tensor        # [batch] int64 entries buffered after the call
    shadow: Optional[torch.Tensor] = None        # read copy after the call
    shadow_scale: Optional[torch.Tensor] = None


def replay(ckpt: torch.Tensor, x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
           C: torch.Tensor, xbuf: torch.Tensor, dtbuf: torch.Tensor, Bbuf: torch.Tensor,
           count: torch.Tensor, D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
           dt_bias: Optional[torch.Tensor] = None, dt_softplus: bool = False,
           slot_of: Optional[torch.Tensor] = None, pad_slot_id: int = -1, shadow: Optional[torch.Tensor] = None,
           shadow_scale: Optional[torch.Tensor] = None, shadow_format: int = SHADOW_NONE, lib=None) -> ReplayResult:
    """One ReplaySSM decode step (one token per sequence) on the host.

    ckpt ``[slots, heads, dim, dstate]``; xbuf ``[slots, L, heads, dim]`` (x's dtype);
    dtbuf ``[slots, L, heads, dim]`` fp32; Bbuf ``[slots, L, groups, dstate]`` (x's dtype);
    count ``[batch]`` entries buffered per sequence.  With a read copy
    (``shadow_format`` SHADOW_F16: ``shadow`` fp16 codes as int16/float16,
    SHADOW_E4M3: uint8 codes and ``shadow_scale [slots, heads, dim]`` fp32,
    SHADOW_NVFP4: uint8 ``[slots, heads, dim, dstate / 2]`` code pairs and
    ``shadow_scale [slots, heads, dim, nvfp4_scale_words(dstate)]`` fp32 records),
    steps that do not fold read it instead of the checkpoint and a fold
    rewrites it.  Inputs are not modified."""
    lib = lib or _load()
    c_in = _cpu(ckpt)
    slots, heads, dim, dstate = c_in.shape
    batch = x.shape[0]
    groups = B.shape[1]
    L = xbuf.shape[1]
    c_out = c_in.clone()
    xs, dts, Bs, Cs, zs = _cpu(x), _cpu(dt), _cpu(B), _cpu(C), _cpu(z)
    As = _cpu(A).to(torch.float32)
    Ds = None if D is None else _cpu(D).to(torch.float32)
    bs = None if dt_bias is None else _cpu(dt_bias).to(torch.float32)
    xb, db, Bb = _cpu(xbuf).clone(), _cpu(dtbuf).to(torch.float32).clone(), _cpu(Bbuf).clone()
    cin = _cpu(count).to(torch.int64)
    cout = torch.zeros(batch, dtype=torch.int64)
    so = None if slot_of is None else _cpu(slot_of).to(torch.int64)
    y = torch.empty((batch, heads, dim), dtype=x.dtype)
    y_exact = torch.empty((batch, heads, dim), dtype=torch.float64)
    if Bs.dtype != xs.dtype or Cs.dtype != xs.dtype or xb.dtype != xs.dtype or Bb.dtype != xs.dtype:
        raise ValueError("B, C and the x / B buffers must have the io dtype")
    pr = _ReplayProblem(
        slots=slots, heads=heads, dim=dim, dstate=dstate, groups=groups,
        state_dtype=_DTYPE_CODE[c_in.dtype], io_dtype=_DTYPE_CODE[xs.dtype], dt_dtype=_DTYPE_CODE[dts.dtype],
        dt_per_head=int(dts.dim() == 2), ckpt_in=c_in.data_ptr(), ckpt_out=c_out.data_ptr(),
        x=xs.data_ptr(), dt=dts.data_ptr(), B=Bs.data_ptr(), C=Cs.data_ptr(), z=_ptr(zs),
        A=As.data_ptr(), D=_ptr(Ds), dt_bias=_ptr(bs), y=y.data_ptr(), y_exact=y_exact.data_ptr(),
        dt_softplus=int(bool(dt_softplus)), pad_slot_id=int(pad_slot_id), batch=batch,
        slot_of=_ptr(so), len=L, xbuf=xb.data_ptr(), dtbuf=db.data_ptr(), Bbuf=Bb.data_ptr(),
        count_in=cin.data_ptr(), count_out=cout.data_ptr())
    sh = sc = None
    if shadow_format != SHADOW_NONE:
        sh = _cpu(shadow).clone()
        sc = None if shadow_scale is None else _cpu(shadow_scale).to(torch.float32).clone()
        pr.shadow_format, pr.shadow, pr.shadow_scale = shadow_format, sh.data_ptr(), _ptr(sc)
    err = ctypes.create_string_buffer(512)
    rc = lib.orc_replay_run(ctypes.byref(pr), err, 512)
    if rc != OK:
        raise OracleError(rc, err.value.decode())
    return ReplayResult(ckpt=c_out, y=y, y_exact=y_exact, xbuf=xb, dtbuf=db, Bbuf=Bb, count=cout, shadow=sh,
                        shadow_scale=sc)


def replay_verify(ckpt: torch.Tensor, x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                  C: torch.Tensor, xbuf: torch.Tensor, dtbuf: torch.Tensor, Bbuf: torch.Tensor, count: torch.Tensor,
                  D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
                  dt_bias: Optional[torch.Tensor] = None, dt_softplus: bool = False,
                  slot_of: Optional[torch.Tensor] = None, pad_slot_id: int = -1, lib=None) -> ReplayResult:
    """Speculative decoding on the checkpoint + buffer form (article
    "ReplaySSM", section 投机解码回滚) on the host: x ``[batch, T, heads, dim]``,
    dt ``[batch, T, heads, dim]`` (or ``[batch, T, heads]``), B, C ``[batch, T,
    groups, dstate]``; the other arguments as for :func:`replay`.  Returns the
    drafts' outputs ``[batch, T, heads, dim]``, the checkpoints and buffers
    after the call and the committed count (the drafts are appended but not
    committed).  Inputs are not modified."""
    lib = lib or _load()
    c_in = _cpu(ckpt)
    slots, heads, dim, dstate = c_in.shape
    batch, T = x.shape[0], x.shape[1]
    groups = B.shape[2]
    L = xbuf.shape[1]
    c_out = c_in.clone()
    xs, dts, Bs, Cs, zs = _cpu(x), _cpu(dt), _cpu(B), _cpu(C), _cpu(z)
    As = _cpu(A).to(torch.float32)
    Ds = None if D is None else _cpu(D).to(torch.float32)
    bs = None if dt_bias is None else _cpu(dt_bias).to(torch.float32)
    xb, db, Bb = _cpu(xbuf).clone(), _cpu(dtbuf).to(torch.float32).clone(), _cpu(Bbuf).clone()
    cin = _cpu(count).to(torch.int64)
    cout = torch.zeros(batch, dtype=torch.int64)
    so = None if slot_of is None else _cpu(slot_of).to(torch.int64)
    y = torch.empty((batch, T, heads, dim), dtype=x.dtype)
    y_exact = torch.empty((batch, T, heads, dim), dtype=torch.float64)
    if Bs.dtype != xs.dtype or Cs.dtype != xs.dtype or xb.dtype != xs.dtype or Bb.dtype != xs.dtype:
        raise ValueError("B, C and the x / B buffers must have the io dtype")
    pr = _VerifyProblem(
        slots=slots, heads=heads, dim=dim, dstate=dstate, groups=groups,
        state_dtype=_DTYPE_CODE[c_in.dtype], io_dtype=_DTYPE_CODE[xs.dtype], dt_dtype=_DTYPE_CODE[dts.dtype],
        dt_per_head=int(dts.dim() == 3), ckpt_in=c_in.data_ptr(), ckpt_out=c_out.data_ptr(),
        x=xs.data_ptr(), dt=dts.data_ptr(), B=Bs.data_ptr(), C=Cs.data_ptr(), z=_ptr(zs),
        A=As.data_ptr(), D=_ptr(Ds), dt_bias=_ptr(bs), y=y.data_ptr(), y_exact=y_exact.data_ptr(),
        dt_softplus=int(bool(dt_softplus)), pad_slot_id=int(pad_slot_id), batch=batch, ntok=T,
        slot_of=_ptr(so), len=L, xbuf=xb.data_ptr(), dtbuf=db.data_ptr(), Bbuf=Bb.data_ptr(),
        count_in=cin.data_ptr(), count_out=cout.data_ptr())
    err = ctypes.create_string_buffer(512)
    rc = lib.orc_replay_verify_run(ctypes.byref(pr), err, 512)
    if rc != OK:
        raise OracleError(rc, err.value.decode())
    return ReplayResult(ckpt=c_out, y=y, y_exact=y_exact, xbuf=xb, dtbuf=db, Bbuf=Bb, count=cout)


def shadow_refresh(state: torch.Tensor, shadow_format: int, lib=None):
    """The read copy of a state pool ``[..., dstate]``: (codes, row scales)
    -- fp16 codes as float16 and no scales for SHADOW_F16, uint8 E4M3 codes
    and fp32 scales of shape ``state.shape[:-1]`` for SHADOW_E4M3, uint8 code
    pairs ``[..., dstate / 2]`` and fp32 scale records ``[...,
    nvfp4_scale_words(dstate)]`` for SHADOW_NVFP4."""
    lib = lib or _load()
    st = _cpu(state).contiguous()
    dstate = st.shape[-1]
    rows = st.numel() // dstate
    if shadow_format == SHADOW_F16:
        codes, scale = torch.empty(st.shape, dtype=torch.float16), None
    elif shadow_format == SHADOW_E4M3:
        codes, scale = torch.empty(st.shape, dtype=torch.uint8), torch.empty(st.shape[:-1], dtype=torch.float32)
    elif shadow_format == SHADOW_NVFP4:
        codes = torch.empty((*st.shape[:-1], dstate // 2), dtype=torch.uint8)
        scale = torch.zeros((*st.shape[:-1], nvfp4_scale_words(dstate)), dtype=torch.float32)
    else:
        raise ValueError("unknown read-copy format")
    rc = lib.orc_shadow_refresh(st.data_ptr(), _DTYPE_CODE[st.dtype], rows, dstate, shadow_format, codes.data_ptr(),
                                _ptr(scale))
    if rc != OK:
        raise OracleError(rc, "shadow refresh failed")
    return codes, scale


@dataclass
class SsdResult:
    y: torch.Tensor            # [tokens, heads, dim] io dtype
    y_exact: torch.Tensor      # float64 before rounding
    states: torch.Tensor       # [nchunks, heads, dim, dstate]: the state at the end of each chunk


def ssd(x: torch.Tensor, dt: torch.Tensor, A: torch.Tensor, B: torch.Tensor, C: torch.Tensor,
        cu_chunk_seqlens: torch.Tensor, seq_idx: torch.Tensor, nseq: int, D: Optional[torch.Tensor] = None,
        z: Optional[torch.Tensor] = None, dt_bias: Optional[torch.Tensor] = None, dt_softplus: bool = False,
        dt_limit=(0.0, float("inf")), initial_states: Optional[torch.Tensor] = None,
        state_dtype: Optional[torch.dtype] = None, lib=None) -> SsdResult:
    """Packed variable-length SSD prefill on the host (MATE "Mamba / SSU",
    SSD packed prefill): x ``[tokens, heads, dim]``, dt ``[tokens, heads]``,
    B, C ``[tokens, groups, dstate]``; chunk c covers tokens
    ``[cu_chunk_seqlens[c], cu_chunk_seqlens[c+1])`` and belongs to sequence
    ``seq_idx[c]``.  Returns y and the state at the end of every chunk, in
    ``state_dtype`` (default: initial_states' dtype, else C's)."""
    lib = lib or _load()
    xs, dts, Bs, Cs, zs = _cpu(x), _cpu(dt), _cpu(B), _cpu(C), _cpu(z)
    tokens, heads, dim = xs.shape
    groups, dstate = Bs.shape[1], Bs.shape[2]
    cu = _cpu(cu_chunk_seqlens).to(torch.int64).contiguous()
    si = _cpu(seq_idx).to(torch.int64).contiguous()
    nchunks = si.numel()
    init = None if initial_states is None else _cpu(initial_states).contiguous()
    sdt = state_dtype or (init.dtype if init is not None else Cs.dtype)
    As = _cpu(A).to(torch.float32)
    Ds = None if D is None else _cpu(D).to(torch.float32)
    bs = None if dt_bias is None else _cpu(dt_bias).to(torch.float32)
    y = torch.empty((tokens, heads, dim), dtype=xs.dtype)
    y_exact = torch.empty((tokens, heads, dim), dtype=torch.float64)
    states = torch.empty((nchunks, heads, dim, dstate), dtype=sdt)
    if init is not None and init.dtype != sdt:
        init = init.to(sdt)
    pr = _SsdProblem(
        tokens=tokens, heads=heads, dim=dim, dstate=dstate, groups=groups, nchunks=nchunks, nseq=nseq,
        io_dtype=_DTYPE_CODE[xs.dtype], dt_dtype=_DTYPE_CODE[dts.dtype], state_dtype=_DTYPE_CODE[sdt],
        x=xs.data_ptr(), dt=dts.data_ptr(), B=Bs.data_ptr(), C=Cs.data_ptr(), z=_ptr(zs), A=As.data_ptr(),
        D=_ptr(Ds), dt_bias=_ptr(bs), dt_softplus=int(bool(dt_softplus)), dt_lo=float(dt_limit[0]),
        dt_hi=float(dt_limit[1]), cu_chunk=cu.data_ptr(), seq_idx=si.data_ptr(), initial_states=_ptr(init),
        y=y.data_ptr(), y_exact=y_exact.data_ptr(), states=states.data_ptr())
    err = ctypes.create_string_buffer(512)
    rc = lib.orc_ssd_run(ctypes.byref(pr), err, 512)
    if rc != OK:
        raise OracleError(rc, err.value.decode())
    return SsdResult(y=y, y_exact=y_exact, states=states)
