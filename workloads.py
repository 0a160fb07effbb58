"""Seeded synthetic inputs for the selective state update.

This module only draws random numbers and lays out tables; it holds none of
the update's arithmetic.  The oracle, the CUDA tests and the benchmark all take
their inputs from here.

The five named workloads follow the shapes, dtypes and value distributions of
the decode workloads this library is measured on:

  tiny_onetoken   batch 2, heads 8, dim 8, dstate 128, groups 2; fp16 zero
                  state; no slot tables (the minimal example of the MATE
                  "Mamba / SSU" page).
  b256_fp32       batch 256 one-token decode, heads 128, dim 64, dstate 128,
                  groups 8, fp32 pool of 512 slots, random distinct read and
                  destination slots with 5% pad (pad id 0), softplus with bias.
  b1024_bf16      batch 1024 one-token decode, bf16 pool of 1024 slots,
                  identity tables, pad id -1.
  mtp_64x7_fp32   64 sequences x 7 speculative rows (448 rows), fp32 pool of
                  1024 slots, 2-D read table arange(448).view(64, 7),
                  destination table read + 448, num_accepted U{1..7}.
  varlen_fp16     128 sequences with lengths U{0..8}, heads 64, groups 1,
                  fp16 pool of 2048 slots, one flat [rows] read table (no
                  destination table), 3% pad (pad id -1), read per packed row.

Two more exercise the neighbouring rows: replay_b256_fp32 (the checkpoint +
buffer form on the b256 shapes) and copy_slots_b256_fp32 (whole-slot state
copies in the b256 pool).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import torch

SLOTS_STRIDED = 0   # entry = b*s0 + t*s1 (a flat table is addressed as [n, 1])
SLOTS_PER_ROW = 1   # entry = cu_seqlens[b] + t (one entry per packed row)


@dataclass
class Workload:
    name: str
    kind: str                                  # "onetoken" or "packed"
    state: torch.Tensor                        # [slots, heads, dim, dstate]
    x: torch.Tensor                            # [rows, heads, dim]
    dt: torch.Tensor                           # [rows, heads, dim] or [rows, heads]
    A: torch.Tensor                            # [heads] fp32
    B: torch.Tensor                            # [rows, groups, dstate]
    C: torch.Tensor                            # [rows, groups, dstate]
    D: Optional[torch.Tensor] = None           # [heads] fp32
    z: Optional[torch.Tensor] = None           # [rows, heads, dim]
    dt_bias: Optional[torch.Tensor] = None     # [heads] fp32
    dt_softplus: bool = False
    read: Optional[torch.Tensor] = None        # slot table (int32)
    dst: Optional[torch.Tensor] = None         # slot table (int32)
    slot_mode: int = SLOTS_STRIDED
    pad_slot_id: int = -1
    disable_state_update: bool = False
    cu_seqlens: Optional[torch.Tensor] = None  # [nseq + 1] int32
    num_accepted: Optional[torch.Tensor] = None  # [nseq] int32
    dense_steps: int = 0                       # >0: dense [nseq, steps, ...] form, no cu_seqlens
    # checkpoint + buffer form (kind "replay"): state holds the checkpoints
    xbuf: Optional[torch.Tensor] = None        # [slots, L, heads, dim] io dtype
    dtbuf: Optional[torch.Tensor] = None       # [slots, L, heads, dim] fp32 processed steps
    Bbuf: Optional[torch.Tensor] = None        # [slots, L, groups, dstate] io dtype
    count: Optional[torch.Tensor] = None       # [batch] int32 buffered entries per sequence
    shadow: Optional[torch.Tensor] = None      # read copy of the checkpoints (fp16, uint8 E4M3 codes, or
                                               # uint8 NVFP4 code pairs [..., dstate / 2])
    shadow_scale: Optional[torch.Tensor] = None  # fp32 E4M3 row scales [slots, heads, dim] or NVFP4 scale records
    meta: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return self.x.shape[0]

    @property
    def nseq(self) -> int:
        if self.kind in ("onetoken", "replay", "verify"):
            return self.rows
        if self.cu_seqlens is not None:
            return self.cu_seqlens.numel() - 1
        return self.rows // self.dense_steps

    def to(self, device) -> "Workload":
        moved = {}
        for k, v in self.__dict__.items():
            moved[k] = v.to(device) if isinstance(v, torch.Tensor) else v
        return replace(self, **moved)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, g, device, mean=0.0, std=1.0, dtype=torch.float32):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return (t * std + mean).to(dtype)


def _uniform(shape, g, device, lo=0.0, hi=1.0):
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


def _decode_inputs(g, device, rows, heads, dim, dstate, groups, io_dtype):
    """x, z, B, C ~ N(0,1) in the io dtype; dt ~ N(0,1) fp32;
    dt_bias ~ N(-3, 0.5); A = -exp(U(0, 2.8)); D ~ N(0, 1)."""
    x = _normal((rows, heads, dim), g, device, dtype=io_dtype)
    z = _normal((rows, heads, dim), g, device, dtype=io_dtype)
    dt = _normal((rows, heads, dim), g, device)
    dt_bias = _normal((heads,), g, device, mean=-3.0, std=0.5)
    A = -torch.exp(_uniform((heads,), g, device, 0.0, 2.8))
    D = _normal((heads,), g, device)
    B = _normal((rows, groups, dstate), g, device, dtype=io_dtype)
    C = _normal((rows, groups, dstate), g, device, dtype=io_dtype)
    return dict(x=x, z=z, dt=dt, dt_bias=dt_bias, A=A, D=D, B=B, C=C)


def _pool(g, device, slots, heads, dim, dstate, dtype, std=0.1):
    return _normal((slots, heads, dim, dstate), g, device, std=std, dtype=dtype)


def tiny_onetoken(device="cpu", seed=1001) -> Workload:
    g = _gen(seed, device)
    batch, heads, dim, dstate, groups = 2, 8, 8, 128, 2
    state = torch.zeros((batch, heads, dim, dstate), dtype=torch.float16, device=device)
    x = _normal((batch, heads, dim), g, device, dtype=torch.bfloat16)
    dt = _uniform((batch, heads, dim), g, device, 0.0, 0.1)
    A = -_uniform((heads,), g, device)
    B = _normal((batch, groups, dstate), g, device, dtype=torch.bfloat16)
    C = _normal((batch, groups, dstate), g, device, dtype=torch.bfloat16)
    return Workload("tiny_onetoken", "onetoken", state, x, dt, A, B, C)


def _distinct_tables_with_pad(g, batch, slots, pad, n_pad, device):
    """Read and destination tables of ``batch`` entries each: exactly ``n_pad``
    entries of each table (at random positions) are the pad id, and the other
    entries are distinct slots, disjoint between the two tables, never the pad
    slot (2 * (batch - n_pad) <= slots - 1 keeps this feasible)."""
    candidates = torch.tensor([s for s in range(slots) if s != pad], dtype=torch.int64)
    need = 2 * (batch - n_pad)
    if need > candidates.numel():
        raise ValueError(f"{need} distinct slots needed, {candidates.numel()} available")
    perm = candidates[torch.randperm(candidates.numel(), generator=g)][:need]
    tables = []
    for k in range(2):
        t = torch.full((batch,), pad, dtype=torch.int64)
        keep = torch.ones(batch, dtype=torch.bool)
        keep[torch.randperm(batch, generator=g)[:n_pad]] = False
        t[keep] = perm[k * (batch - n_pad):(k + 1) * (batch - n_pad)]
        tables.append(t.to(torch.int32).to(device))
    return tables[0], tables[1]


def b256_fp32(device="cpu", seed=1002, in_place=False, batch=256) -> Workload:
    """``batch`` other than 256 gives the same workload at another size (pool
    of 2 * batch slots); profiling uses it for captures that must stay small."""
    heads, dim, dstate, groups, pad = 128, 64, 128, 8, 0
    slots = 2 * batch
    g = _gen(seed, device)
    inp = _decode_inputs(g, device, batch, heads, dim, dstate, groups, torch.bfloat16)
    state = _pool(g, device, slots, heads, dim, dstate, torch.float32)
    gh = _gen(seed + 7, "cpu")
    read, dst = _distinct_tables_with_pad(gh, batch, slots, pad, max(1, round(0.05 * batch)), device)
    if in_place:
        dst = read.clone()
    return Workload("b256_fp32" + ("_inplace" if in_place else ""), "onetoken", state,
                    dt_softplus=True, read=read, dst=dst, pad_slot_id=pad, **inp)


def b1024_bf16(device="cpu", seed=1003) -> Workload:
    heads, dim, dstate, groups, slots, batch = 128, 64, 128, 8, 1024, 1024
    g = _gen(seed, device)
    inp = _decode_inputs(g, device, batch, heads, dim, dstate, groups, torch.bfloat16)
    state = _pool(g, device, slots, heads, dim, dstate, torch.bfloat16)
    ident = torch.arange(batch, dtype=torch.int32, device=device)
    return Workload("b1024_bf16", "onetoken", state, dt_softplus=True, read=ident,
                    dst=ident.clone(), pad_slot_id=-1, **inp)


def mtp_64x7_fp32(device="cpu", seed=1004, batch=64) -> Workload:
    """``batch`` other than 64 gives the same workload with another number of
    sequences (pool of 16 * batch slots); profiling uses it for small captures."""
    heads, dim, dstate, groups, steps = 128, 64, 128, 8, 7
    nseq, slots = batch, 16 * batch
    rows = nseq * steps
    g = _gen(seed, device)
    inp = _decode_inputs(g, device, rows, heads, dim, dstate, groups, torch.bfloat16)
    state = _pool(g, device, slots, heads, dim, dstate, torch.float32)
    gh = _gen(seed + 7, "cpu")
    read = torch.arange(rows, dtype=torch.int32, device=device).view(nseq, steps)
    dst = (read + rows).contiguous()
    cu = torch.arange(0, rows + 1, steps, dtype=torch.int32, device=device)
    acc = torch.randint(1, steps + 1, (nseq,), generator=gh, dtype=torch.int64).to(torch.int32).to(device)
    return Workload("mtp_64x7_fp32", "packed", state, dt_softplus=True, read=read, dst=dst,
                    pad_slot_id=-1, cu_seqlens=cu, num_accepted=acc, **inp)


def varlen_fp16(device="cpu", seed=1005, disable_state_update=False,
                slot_mode=SLOTS_PER_ROW) -> Workload:
    heads, dim, dstate, groups, slots, nseq = 64, 64, 128, 1, 2048, 128
    gh = _gen(seed + 7, "cpu")
    lens = torch.randint(0, 9, (nseq,), generator=gh, dtype=torch.int64)
    lens[int(torch.randint(0, nseq, (1,), generator=gh))] = 0   # at least one empty sequence
    rows = int(lens.sum())
    cu = torch.zeros(nseq + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lens, 0)
    acc = torch.ones(nseq, dtype=torch.int64)
    for b in range(nseq):
        if lens[b] > 0:
            acc[b] = int(torch.randint(1, int(lens[b]) + 1, (1,), generator=gh))
    read = torch.randperm(slots, generator=gh)[:rows].clone()
    n_pad = round(0.03 * rows)
    read[torch.randperm(rows, generator=gh)[:n_pad]] = -1
    g = _gen(seed, device)
    inp = _decode_inputs(g, device, rows, heads, dim, dstate, groups, torch.bfloat16)
    state = _pool(g, device, slots, heads, dim, dstate, torch.float16)
    name = "varlen_fp16" + ("_disable" if disable_state_update else "")
    if slot_mode == SLOTS_STRIDED:
        name += "_strided"
    return Workload(name, "packed", state, dt_softplus=True,
                    read=read.to(torch.int32).to(device), dst=None, slot_mode=slot_mode,
                    pad_slot_id=-1, disable_state_update=disable_state_update,
                    cu_seqlens=cu.to(torch.int32).to(device),
                    num_accepted=acc.to(torch.int32).to(device), meta={"lengths": lens.tolist()}, **inp)


def _replay_buffers(g, device, slots, L, heads, dim, dstate, groups, io_dtype):
    """A history of buffered steps: x, B ~ N(0,1) in the io dtype; processed
    steps dt' ~ U(0.001, 0.2) in fp32."""
    xbuf = _normal((slots, L, heads, dim), g, device, dtype=io_dtype)
    dtbuf = _uniform((slots, L, heads, dim), g, device, 0.001, 0.2)
    Bbuf = _normal((slots, L, groups, dstate), g, device, dtype=io_dtype)
    return xbuf, dtbuf, Bbuf


def replay_b256_fp32(device="cpu", seed=1006, batch=256, buffer_len=16) -> Workload:
    """Batch-256 decode on the checkpoint + buffer form: the b256_fp32 shapes
    and distributions, one slot table (read = write), a buffer of
    ``buffer_len`` entries per slot, sequence b holding b % L entries so that
    every step folds 1/L of the sequences."""
    heads, dim, dstate, groups, pad = 128, 64, 128, 8, 0
    slots = 2 * batch
    g = _gen(seed, device)
    inp = _decode_inputs(g, device, batch, heads, dim, dstate, groups, torch.bfloat16)
    state = _pool(g, device, slots, heads, dim, dstate, torch.float32)
    xbuf, dtbuf, Bbuf = _replay_buffers(g, device, slots, buffer_len, heads, dim, dstate, groups, torch.bfloat16)
    gh = _gen(seed + 7, "cpu")
    read, _ = _distinct_tables_with_pad(gh, batch, slots, pad, max(1, round(0.05 * batch)), device)
    count = (torch.arange(batch, dtype=torch.int32) % buffer_len).to(device)
    return Workload("replay_b256_fp32", "replay", state, dt_softplus=True, read=read, pad_slot_id=pad,
                    xbuf=xbuf, dtbuf=dtbuf, Bbuf=Bbuf, count=count, meta={"buffer_len": buffer_len}, **inp)


def replay_e4m3_b256_fp32(device="cpu", seed=1008, batch=256, buffer_len=16) -> Workload:
    """replay_b256_fp32 with an E4M3 read copy of the checkpoints (codes and
    row scales allocated here, filled by the caller with the copy of the
    checkpoints: the copy's arithmetic is not this module's)."""
    w = replay_b256_fp32(device=device, seed=seed, batch=batch, buffer_len=buffer_len)
    w.name = "replay_e4m3_b256_fp32"
    w.shadow = torch.zeros(w.state.shape, dtype=torch.uint8, device=device)
    w.shadow_scale = torch.ones(w.state.shape[:-1], dtype=torch.float32, device=device)
    w.meta["shadow_format"] = "e4m3"
    return w


def replay_nvfp4_b256_fp32(device="cpu", seed=1012, batch=256, buffer_len=16) -> Workload:
    """replay_b256_fp32 with an NVFP4 read copy of the checkpoints (E2M1 code
    pairs [slots, heads, dim, dstate / 2] and per-row scale records of
    (4 + dstate / 16 + 15) // 16 * 4 floats, allocated here, filled by the
    caller with the copy of the checkpoints)."""
    w = replay_b256_fp32(device=device, seed=seed, batch=batch, buffer_len=buffer_len)
    w.name = "replay_nvfp4_b256_fp32"
    n = w.state.shape[-1]
    w.shadow = torch.zeros((*w.state.shape[:-1], n // 2), dtype=torch.uint8, device=device)
    w.shadow_scale = torch.zeros((*w.state.shape[:-1], (4 + n // 16 + 15) // 16 * 4), dtype=torch.float32,
                                 device=device)
    w.meta["shadow_format"] = "nvfp4"
    return w


def replay_f16copy_b256_fp32(device="cpu", seed=1009, batch=256, buffer_len=16) -> Workload:
    """replay_b256_fp32 with an fp16 read copy of the checkpoints (allocated
    here, filled by the caller)."""
    w = replay_b256_fp32(device=device, seed=seed, batch=batch, buffer_len=buffer_len)
    w.name = "replay_f16copy_b256_fp32"
    w.shadow = torch.zeros(w.state.shape, dtype=torch.float16, device=device)
    w.meta["shadow_format"] = "f16"
    return w


def verify_b256_t4_fp32(device="cpu", seed=1011, batch=256, buffer_len=16, ntok=4) -> Workload:
    """Speculative decoding on the checkpoint + buffer form at batch 256: the
    b256_fp32 shapes and distributions (fp32 checkpoints, 512 slots, 13 pad
    entries), a buffer of 16 entries, 4 drafts per sequence; sequence b holds
    b % 9 committed entries, so the flush (c + 2T >= L, i.e. c = 8) fires for
    1/9 of the sequences."""
    heads, dim, dstate, groups, pad = 128, 64, 128, 8, 0
    slots = 2 * batch
    g = _gen(seed, device)
    inp = _decode_inputs(g, device, batch * ntok, heads, dim, dstate, groups, torch.bfloat16)
    for k in ("x", "z", "dt", "B", "C"):
        inp[k] = inp[k].view(batch, ntok, *inp[k].shape[1:])
    state = _pool(g, device, slots, heads, dim, dstate, torch.float32)
    xbuf, dtbuf, Bbuf = _replay_buffers(g, device, slots, buffer_len, heads, dim, dstate, groups, torch.bfloat16)
    gh = _gen(seed + 7, "cpu")
    read, _ = _distinct_tables_with_pad(gh, batch, slots, pad, max(1, round(0.05 * batch)), device)
    count = (torch.arange(batch, dtype=torch.int32) % (buffer_len - 2 * ntok + 1)).to(device)
    return Workload("verify_b256_t4_fp32", "verify", state, dt_softplus=True, read=read, pad_slot_id=pad,
                    xbuf=xbuf, dtbuf=dtbuf, Bbuf=Bbuf, count=count, meta={"buffer_len": buffer_len, "ntok": ntok},
                    **inp)


def replay_problem(seed: int, *, slots: int = 16, heads: int = 4, dim: int = 8, dstate: int = 16,
                   groups: int = 2, nseq: int = 4, buffer_len: int = 4, state_dtype=torch.float32,
                   io_dtype=torch.bfloat16, with_D: bool = True, with_z: bool = True, with_bias: bool = True,
                   dt_softplus: bool = True, pad_slot_id: int = -1, pad_frac: float = 0.2,
                   tables: bool = True, device="cpu") -> Workload:
    """A small seeded problem on the checkpoint + buffer form: distinct slots
    (some pad), counts U{0..L-1}, random buffered histories."""
    gh = _gen(seed, "cpu")
    read = None
    if tables:
        usable = torch.tensor([s for s in range(slots) if s != pad_slot_id], dtype=torch.int64)
        if nseq > usable.numel():
            raise ValueError("not enough slots")
        read = usable[torch.randperm(usable.numel(), generator=gh)[:nseq]].clone()
        n_pad = int(round(pad_frac * nseq))
        if n_pad:
            read[torch.randperm(nseq, generator=gh)[:n_pad]] = pad_slot_id
        read = read.to(torch.int32)
    count = torch.randint(0, buffer_len, (nseq,), generator=gh, dtype=torch.int64).to(torch.int32)
    g = _gen(seed + 1, "cpu")
    x = _normal((nseq, heads, dim), g, "cpu", dtype=io_dtype)
    z = _normal((nseq, heads, dim), g, "cpu", dtype=io_dtype) if with_z else None
    dt = _normal((nseq, heads, dim), g, "cpu") if dt_softplus else _uniform((nseq, heads, dim), g, "cpu", 0.0, 0.2)
    dt_bias = _step_bias(g, heads, dt_softplus) if with_bias else None
    A = -torch.exp(_uniform((heads,), g, "cpu", 0.0, 2.8))
    D = _normal((heads,), g, "cpu") if with_D else None
    B = _normal((nseq, groups, dstate), g, "cpu", dtype=io_dtype)
    C = _normal((nseq, groups, dstate), g, "cpu", dtype=io_dtype)
    state = _pool(g, "cpu", slots, heads, dim, dstate, state_dtype, std=0.5)
    xbuf, dtbuf, Bbuf = _replay_buffers(g, "cpu", slots, buffer_len, heads, dim, dstate, groups, io_dtype)
    w = Workload(f"replay_{seed}", "replay", state, x, dt, A, B, C, D=D, z=z, dt_bias=dt_bias,
                 dt_softplus=dt_softplus, read=read, pad_slot_id=pad_slot_id, xbuf=xbuf, dtbuf=dtbuf, Bbuf=Bbuf,
                 count=count, meta={"buffer_len": buffer_len})
    return w.to(device)


def verify_problem(seed: int, *, ntok: int = 2, buffer_len: int = 8, **kw) -> Workload:
    """A small seeded problem for speculative decoding on the checkpoint +
    buffer form: replay_problem's pool, buffers and counts (U{0..L-1}) with
    ``ntok`` draft tokens per sequence -- x, z, dt ``[nseq, T, heads, dim]``,
    B, C ``[nseq, T, groups, dstate]`` -- drawn as the one-token inputs."""
    device = kw.pop("device", "cpu")
    w = replay_problem(seed, buffer_len=buffer_len, **kw)
    nseq, heads, dim = w.x.shape
    groups, dstate = w.B.shape[1], w.B.shape[2]
    g = _gen(seed + 7, "cpu")
    io = w.x.dtype
    x = _normal((nseq, ntok, heads, dim), g, "cpu", dtype=io)
    z = _normal((nseq, ntok, heads, dim), g, "cpu", dtype=io) if w.z is not None else None
    dt = (_normal((nseq, ntok, heads, dim), g, "cpu") if w.dt_softplus
          else _uniform((nseq, ntok, heads, dim), g, "cpu", 0.0, 0.2))
    B = _normal((nseq, ntok, groups, dstate), g, "cpu", dtype=io)
    C = _normal((nseq, ntok, groups, dstate), g, "cpu", dtype=io)
    w = replace(w, name=f"verify_{seed}", kind="verify", x=x, z=z, dt=dt, B=B, C=C,
                meta=dict(w.meta, ntok=ntok))
    return w.to(device)


@dataclass
class CopyWorkload:
    """Whole-slot copies inside one state pool: slot src[i] to slot dst[i]."""
    name: str
    state: torch.Tensor                        # [slots, heads, dim, dstate]
    src: torch.Tensor                          # [n] int64 slots
    dst: torch.Tensor                          # [n] int64 slots, disjoint from src
    kind: str = "copy"
    meta: dict = field(default_factory=dict)

    @property
    def nseq(self) -> int:
        return self.src.numel()

    def to(self, device) -> "CopyWorkload":
        return replace(self, state=self.state.to(device), src=self.src.to(device), dst=self.dst.to(device))


def copy_slots_b256_fp32(device="cpu", seed=1007, batch=256) -> CopyWorkload:
    """``batch`` whole-slot copies of 4 MiB (heads 128, dim 64, dstate 128,
    fp32) between random distinct slots of a pool of 2 * batch slots, sources
    and destinations disjoint (the slot moves of speculative decoding)."""
    slots = 2 * batch
    g = _gen(seed, device)
    state = _pool(g, device, slots, 128, 64, 128, torch.float32)
    perm = torch.randperm(slots, generator=_gen(seed + 1, "cpu"))
    return CopyWorkload("copy_slots_b256_fp32", state, perm[:batch].to(device), perm[batch:].to(device))




def _step_bias(g, heads, softplus):
    """dt_bias for the small problems: N(-1, 0.5) before a softplus; without
    one U(0, 0.1), so that dt' = dt + bias stays >= 0 (A < 0 and dt' >= 0 keep
    the recurrence decaying, 0 < exp(A dt') <= 1)."""
    if softplus:
        return _normal((heads,), g, "cpu", mean=-1.0, std=0.5)
    return _uniform((heads,), g, "cpu", 0.0, 0.1)


def random_problem(seed: int, *, kind: str = "onetoken", slots: int = 16, heads: int = 4,
                   dim: int = 8, dstate: int = 16, groups: int = 2, nseq: int = 3,
                   max_len: int = 3, state_dtype=torch.float32, io_dtype=torch.bfloat16,
                   dt_dtype=torch.float32, per_head_dt: bool = False, with_D: bool = True,
                   with_z: bool = True, with_bias: bool = True, dt_softplus: bool = True,
                   tables: str = "distinct", pad_slot_id: int = -1, pad_frac: float = 0.2,
                   slot_mode: int = SLOTS_STRIDED, with_accepted: bool = True,
                   allow_empty: bool = True, disable_state_update: bool = False,
                   state_std: float = 0.5, dense: bool = False, min_len: int = 0,
                   device="cpu") -> Workload:
    """A small seeded problem for parity sweeps.

    ``tables``: "none" (sequence b uses slot b), "read" (read table only),
    "distinct" (read and destination tables of distinct, disjoint slots),
    "inplace" (destination table equal to the read table).
    For ``kind="packed"`` the read/destination tables are 2-D ``[nseq, max_len]``
    in STRIDED mode, or flat ``[rows]`` in PER_ROW mode; ``dense`` makes every
    sequence ``max_len`` long and drops cu_seqlens (the dense 4-D form);
    ``min_len`` raises the shortest length of the others.
    """
    gh = _gen(seed, "cpu")
    if kind == "onetoken":
        lens = torch.ones(nseq, dtype=torch.int64)
    elif dense:
        lens = torch.full((nseq,), max_len, dtype=torch.int64)
    else:
        lens = torch.randint(max(min_len, 0 if allow_empty else 1), max_len + 1, (nseq,), generator=gh)
    rows = int(lens.sum())
    cu = torch.zeros(nseq + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lens, 0)
    per_seq = 1 if kind == "onetoken" else max_len
    # entries needed by each table
    if kind == "onetoken" or slot_mode == SLOTS_PER_ROW:
        n_entries = rows if kind == "packed" else nseq
    else:
        n_entries = nseq * per_seq
    need = n_entries * (2 if tables == "distinct" else 1)
    usable = torch.tensor([s for s in range(slots) if s != pad_slot_id], dtype=torch.int64)
    if tables != "none" and need > usable.numel():
        raise ValueError(f"need {need} distinct slots, have {usable.numel()}")
    perm = usable[torch.randperm(usable.numel(), generator=gh)]
    read = dst = None
    if tables != "none":
        read = perm[:n_entries].clone()
        if tables == "distinct":
            dst = perm[n_entries:2 * n_entries].clone()
        n_pad = int(round(pad_frac * n_entries))
        for t in (read, dst):
            if t is not None and n_pad > 0:
                t[torch.randperm(n_entries, generator=gh)[:n_pad]] = pad_slot_id
        if tables == "inplace":
            dst = read.clone()
        if kind == "packed" and slot_mode == SLOTS_STRIDED:
            read = read.view(nseq, per_seq)
            dst = None if dst is None else dst.view(nseq, per_seq)
        read = read.to(torch.int32)
        dst = None if dst is None else dst.to(torch.int32)
    acc = None
    if kind == "packed" and with_accepted:
        acc = torch.ones(nseq, dtype=torch.int64)
        for b in range(nseq):
            if lens[b] > 0:
                acc[b] = int(torch.randint(1, int(lens[b]) + 1, (1,), generator=gh))
        acc = acc.to(torch.int32)
    g = _gen(seed + 1, "cpu")
    x = _normal((rows, heads, dim), g, "cpu", dtype=io_dtype)
    z = _normal((rows, heads, dim), g, "cpu", dtype=io_dtype) if with_z else None
    dt_shape = (rows, heads) if per_head_dt else (rows, heads, dim)
    dt = (_normal(dt_shape, g, "cpu") if dt_softplus else _uniform(dt_shape, g, "cpu", 0.0, 0.2)).to(dt_dtype)
    dt_bias = _step_bias(g, heads, dt_softplus) if with_bias else None
    A = -torch.exp(_uniform((heads,), g, "cpu", 0.0, 2.8))
    D = _normal((heads,), g, "cpu") if with_D else None
    B = _normal((rows, groups, dstate), g, "cpu", dtype=io_dtype)
    C = _normal((rows, groups, dstate), g, "cpu", dtype=io_dtype)
    state = _pool(g, "cpu", slots, heads, dim, dstate, state_dtype, std=state_std)
    w = Workload(f"random_{kind}_{seed}", kind, state, x, dt, A, B, C, D=D, z=z, dt_bias=dt_bias,
                 dt_softplus=dt_softplus, read=read, dst=dst, slot_mode=slot_mode,
                 pad_slot_id=pad_slot_id, disable_state_update=disable_state_update,
                 cu_seqlens=None if (kind == "onetoken" or dense) else cu.to(torch.int32),
                 num_accepted=acc, dense_steps=max_len if dense else 0,
                 meta={"lengths": lens.tolist()})
    return w.to(device)


# ---------------------------------------------------------------------------
# Packed variable-length SSD prefill.
# ---------------------------------------------------------------------------
@dataclass
class SsdWorkload:
    name: str
    x: torch.Tensor                      # [tokens, heads, dim] io dtype
    dt: torch.Tensor                     # [tokens, heads] fp32
    A: torch.Tensor                      # [heads] fp32
    B: torch.Tensor                      # [tokens, groups, dstate]
    C: torch.Tensor                      # [tokens, groups, dstate]
    cu_seqlens: torch.Tensor             # [nseq + 1] int32
    cu_chunk_seqlens: torch.Tensor       # [nchunks + 1] int32
    seq_idx: torch.Tensor                # [nchunks] int32
    last_chunk_indices: torch.Tensor     # [nseq] int32
    chunk_size: int
    D: Optional[torch.Tensor] = None
    z: Optional[torch.Tensor] = None
    dt_bias: Optional[torch.Tensor] = None
    dt_softplus: bool = True
    dt_limit: tuple = (0.0, float("inf"))
    initial_states: Optional[torch.Tensor] = None   # [nseq, heads, dim, dstate]
    state_dtype: torch.dtype = torch.float32
    kind: str = "ssd"
    meta: dict = field(default_factory=dict)

    @property
    def nseq(self) -> int:
        return self.cu_seqlens.numel() - 1

    @property
    def tokens(self) -> int:
        return self.x.shape[0]

    def to(self, device) -> "SsdWorkload":
        moved = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in self.__dict__.items()}
        return replace(self, **moved)


def ssd_chunks(lengths, chunk_size):
    """Chunking of packed sequences as vLLM's Mamba-2 prefill lays it out:
    each sequence cut into chunks of ``chunk_size`` tokens from its first
    token, the last one partial; no chunk spans two sequences.  Returns
    (cu_seqlens, cu_chunk_seqlens, seq_idx, last_chunk_indices), int32."""
    cu, cu_chunk, seq_idx, last = [0], [0], [], []
    for b, n in enumerate(lengths):
        if n < 1:
            raise ValueError("every prefill sequence has at least one token")
        start = cu[-1]
        for k in range((n + chunk_size - 1) // chunk_size):
            cu_chunk.append(start + min((k + 1) * chunk_size, n))
            seq_idx.append(b)
        last.append(len(seq_idx) - 1)
        cu.append(start + n)
    t = lambda v: torch.tensor(v, dtype=torch.int32)
    return t(cu), t(cu_chunk), t(seq_idx), t(last)


def ssd_problem(seed: int, lengths, *, heads=4, dim=8, dstate=16, groups=2, chunk_size=16,
                io_dtype=torch.bfloat16, state_dtype=torch.float32, with_init=True, with_D=True, with_z=True,
                with_bias=True, dt_softplus=True, dt_limit=(0.0, float("inf")), device="cpu",
                name=None) -> SsdWorkload:
    """A seeded SSD prefill problem: x, z, B, C ~ N(0,1) in the io dtype; dt ~
    N(0,1) fp32 per (token, head); dt_bias as the decode workloads; A =
    -exp(U(0, 2.8)); D ~ N(0,1); initial states N(0, 0.1)."""
    cu, cu_chunk, seq_idx, last = ssd_chunks(list(lengths), chunk_size)
    tokens = int(cu[-1])
    g = _gen(seed, "cpu")
    x = _normal((tokens, heads, dim), g, "cpu", dtype=io_dtype)
    z = _normal((tokens, heads, dim), g, "cpu", dtype=io_dtype) if with_z else None
    dt = _normal((tokens, heads), g, "cpu") if dt_softplus else _uniform((tokens, heads), g, "cpu", 0.0, 0.1)
    dt_bias = _step_bias(g, heads, dt_softplus) if with_bias else None
    A = -torch.exp(_uniform((heads,), g, "cpu", 0.0, 2.8))
    D = _normal((heads,), g, "cpu") if with_D else None
    B = _normal((tokens, groups, dstate), g, "cpu", dtype=io_dtype)
    C = _normal((tokens, groups, dstate), g, "cpu", dtype=io_dtype)
    init = _normal((len(lengths), heads, dim, dstate), g, "cpu", std=0.1, dtype=state_dtype) if with_init else None
    w = SsdWorkload(name or f"ssd_{seed}", x, dt, A, B, C, cu, cu_chunk, seq_idx, last, chunk_size, D=D, z=z,
                    dt_bias=dt_bias, dt_softplus=dt_softplus, dt_limit=dt_limit, initial_states=init,
                    state_dtype=state_dtype)
    return w.to(device)


def ssd_prefill_16k_bf16(device="cpu", seed=1010, batch=8) -> SsdWorkload:
    """Mamba-2 prefill on the decode workloads' layer shape (heads 128, dim 64,
    dstate 128, groups 8), chunk 256, bf16 x/z/B/C, fp32 dt with bias and
    softplus, fp32 initial and returned states; ``batch`` sequences with
    lengths U{1024..3072} (about 2048 tokens each, ragged last chunks)."""
    gl = _gen(seed + 3, "cpu")
    lengths = torch.randint(1024, 3073, (batch,), generator=gl).tolist()
    return ssd_problem(seed, lengths, heads=128, dim=64, dstate=128, groups=8, chunk_size=256, device=device,
                       name="ssd_prefill_16k_bf16")


NAMED = {
    "tiny_onetoken": tiny_onetoken,
    "b256_fp32": b256_fp32,
    "b1024_bf16": b1024_bf16,
    "mtp_64x7_fp32": mtp_64x7_fp32,
    "varlen_fp16": varlen_fp16,
    "varlen_fp16_disable": lambda device="cpu", seed=1005: varlen_fp16(device, seed, disable_state_update=True),
    "replay_b256_fp32": replay_b256_fp32,
    "replay_e4m3_b256_fp32": replay_e4m3_b256_fp32,
    "replay_nvfp4_b256_fp32": replay_nvfp4_b256_fp32,
    "replay_f16copy_b256_fp32": replay_f16copy_b256_fp32,
    "copy_slots_b256_fp32": copy_slots_b256_fp32,
    "verify_b256_t4_fp32": verify_b256_t4_fp32,
    "ssd_prefill_16k_bf16": ssd_prefill_16k_bf16,
}
