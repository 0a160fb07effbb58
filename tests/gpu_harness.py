"""Helpers for the GPU tests: run a workload through libssu's C ABI (via the
Python binding), cut sampled sub-problems out of full-size workloads for the
oracle, and compare results."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import replace

import numpy as np
import torch

import workloads
from ssu_testlib import assert_state_close, assert_y_close, run_oracle

DEV = "cuda"


def run_gpu(w: workloads.Workload, status: torch.Tensor = None, y_fill=None):
    """Run `w` (already on the GPU) in place; returns y."""
    import selective_state_update_gb300 as ssu
    out = torch.empty_like(w.x)
    if y_fill is not None:
        out.fill_(y_fill)
    common = dict(D=w.D, z=w.z, dt_bias=w.dt_bias, dt_softplus=w.dt_softplus,
                  state_batch_indices=w.read, dst_state_batch_indices=w.dst,
                  pad_slot_id=w.pad_slot_id, disable_state_update=w.disable_state_update, status=status)
    if w.kind == "onetoken":
        return ssu.ssu_update_onetoken(w.state, w.x, w.dt, w.A, w.B, w.C, out=out, **common)
    if w.dense_steps:
        n, s = w.nseq, w.dense_steps
        d4 = lambda t: None if t is None else t.view(n, s, *t.shape[1:])
        y = ssu.ssu_update_packed(w.state, d4(w.x), d4(w.dt), w.A, d4(w.B), d4(w.C),
                                  num_accepted_tokens=w.num_accepted, slot_mode=w.slot_mode,
                                  out=d4(out), **{**common, "z": d4(w.z)})
        return y.view(w.rows, *y.shape[2:])
    return ssu.ssu_update_packed(w.state, w.x, w.dt, w.A, w.B, w.C, cu_seqlens=w.cu_seqlens,
                                 num_accepted_tokens=w.num_accepted, slot_mode=w.slot_mode,
                                 out=out, **common)


def full_check(w_cpu: workloads.Workload, status_expected: int = 0):
    """Run the whole workload on the GPU and on the oracle and compare every
    output: y within the output tolerance, written slots within the state
    tolerance, every other slot bit-identical."""
    ref = run_oracle(w_cpu)
    w = w_cpu.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = run_gpu(w, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == status_expected
    assert_y_close(y, ref.y_exact)
    got = w.state.cpu()
    written = (ref.touched & 2).bool()
    assert torch.equal(got[~written], w_cpu.state[~written]), "a slot that is not written changed"
    if written.any():
        assert_state_close(got[written], ref.state[written])
    return ref, y, got


def _seq_rows(w):
    lens = w.meta.get("lengths")
    if lens is None:
        if w.kind == "onetoken":
            lens = [1] * w.nseq
        elif w.cu_seqlens is not None:
            cu = w.cu_seqlens.cpu().tolist()
            lens = [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
        else:
            lens = [w.dense_steps] * w.nseq
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return lens, cu


def subproblem(w: workloads.Workload, seqs):
    """Cut sequences `seqs` out of workload `w` (CPU tensors) into a small
    problem with its own compact pool.  Returns (sub, rows, slot_map) where
    rows are the original row indices in the order of the sub-problem's rows
    and slot_map maps original slot -> sub slot."""
    seqs = list(seqs)
    lens, cu = _seq_rows(w)
    rows = [r for b in seqs for r in range(cu[b], cu[b + 1])]
    sub_lens = [lens[b] for b in seqs]
    pad = w.pad_slot_id
    mode = w.slot_mode

    def table_rows(t):
        if t is None:
            return None
        if w.kind == "onetoken":
            return t.reshape(-1)[seqs]
        if mode == workloads.SLOTS_PER_ROW:
            return t.reshape(-1)[rows]
        return t[seqs]

    rd, wr = table_rows(w.read), table_rows(w.dst)
    if rd is None:
        # no table: sequence b reads and writes slot b at every step
        if w.kind == "onetoken":
            rd = torch.tensor(seqs, dtype=torch.int32)
        else:
            width = max(max(sub_lens), 1)
            rd = torch.tensor(seqs, dtype=torch.int32).view(-1, 1).repeat(1, width)
            mode = workloads.SLOTS_STRIDED
    used = sorted({int(v) for t in (rd, wr) if t is not None for v in t.reshape(-1).tolist()} - {pad})
    order = ([pad] if 0 <= pad < w.state.shape[0] else []) + used
    slot_map = {s: i for i, s in enumerate(order)}
    sub_pad = slot_map.get(pad, pad)

    def remap(t):
        if t is None:
            return None
        return torch.tensor([sub_pad if v == pad else slot_map[v] for v in t.reshape(-1).tolist()],
                            dtype=t.dtype).view(t.shape)

    state = w.state[order] if order else w.state[:1]
    sel = lambda t: None if t is None else t[rows]
    sub_cu = None
    if w.kind == "packed":
        sub_cu = torch.tensor(np.concatenate([[0], np.cumsum(sub_lens)]), dtype=torch.int32)
    sub = replace(w, state=state, x=sel(w.x), dt=sel(w.dt), B=sel(w.B), C=sel(w.C), z=sel(w.z),
                  read=remap(rd), dst=remap(wr), pad_slot_id=sub_pad, slot_mode=mode,
                  meta={"lengths": sub_lens}, cu_seqlens=sub_cu,
                  num_accepted=None if w.num_accepted is None else w.num_accepted[seqs],
                  dense_steps=0)
    return sub, rows, slot_map


def sampled_check(w_cpu: workloads.Workload, seqs, y_gpu: torch.Tensor, state_gpu: torch.Tensor):
    """Compare the GPU's results of a full-size run on the sampled sequences
    with the oracle run on just those sequences."""
    sub, rows, slot_map = subproblem(w_cpu, seqs)
    ref = run_oracle(sub)
    assert_y_close(y_gpu[rows].cpu(), ref.y_exact, what="y (sampled)")
    inv = {v: k for k, v in slot_map.items()}
    written = [i for i in range(sub.state.shape[0]) if ref.touched[i] & 2]
    if written:
        got = state_gpu[[inv[i] for i in written]].cpu()
        assert_state_close(got, ref.state[written], what="state (sampled)")
    return ref


def written_slots(w: workloads.Workload):
    """Slots a call may write (non-pad destinations of non-empty rows), from
    the tables alone; used for the "nothing else changes" property."""
    if w.disable_state_update:
        return set()
    lens, cu = _seq_rows(w)
    pad = w.pad_slot_id
    out = set()
    wt = w.dst if w.dst is not None else w.read
    for b, L in enumerate(lens):
        for t in range(L):
            if wt is None:
                s = b
            elif w.kind == "onetoken":
                s = int(wt.reshape(-1)[b])
            elif w.slot_mode == workloads.SLOTS_PER_ROW:
                s = int(wt.reshape(-1)[cu[b] + t])
            elif wt.dim() == 1:
                s = int(wt[b + t])
            else:
                s = int(wt[b, t])
            if s != pad:
                out.add(s)
    return out


def assert_untouched(before: torch.Tensor, after: torch.Tensor, written):
    """Every slot outside `written` is bit-identical (compared on the device)."""
    mask = torch.ones(before.shape[0], dtype=torch.bool, device=before.device)
    if written:
        mask[torch.tensor(sorted(written), device=before.device)] = False
    assert torch.equal(before[mask], after[mask]), "a slot that is not written changed"


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def complete_check(w_cpu: workloads.Workload, y_gpu: torch.Tensor, state_gpu: torch.Tensor, per_chunk: int = 16):
    """Compare EVERY sequence of a full-size run with the oracle, element by
    element: the sequences are cut into independent sub-problems of
    `per_chunk` sequences (each with its own compact pool; the workloads give
    every sequence its own slots), the oracle runs them on all host threads
    (its C entry point runs without the GIL), and each sub-problem's y rows
    and written slots are held to the output and state tolerances.  Returns
    the number of sequences compared."""
    y_all = y_gpu.cpu()
    pool = state_gpu.cpu()
    nseq = w_cpu.nseq
    chunks = [list(range(i, min(i + per_chunk, nseq))) for i in range(0, nseq, per_chunk)]

    def one(seqs):
        sub, rows, slot_map = subproblem(w_cpu, seqs)
        ref = run_oracle(sub)
        if rows:
            assert_y_close(y_all[rows], ref.y_exact, what=f"y (sequences {seqs[0]}..{seqs[-1]})")
        inv = {v: k for k, v in slot_map.items()}
        written = [i for i in range(sub.state.shape[0]) if ref.touched[i] & 2]
        if written:
            assert_state_close(pool[[inv[i] for i in written]], ref.state[written],
                               what=f"state (sequences {seqs[0]}..{seqs[-1]})")
        return len(seqs)

    with ThreadPoolExecutor(max(1, min(host_threads(), len(chunks)))) as ex:
        done = sum(ex.map(one, chunks))
    assert done == nseq
    return done
