"""Benchmark of libssu's selective state update on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one call of the update over one batch of the workload (every step
of the update runs in one kernel launch).  Without --workload the five decode
configurations are timed one after another in the same run: the batch-256
one-token decode with an fp32 pool is the headline line, and every
configuration (the tiny one-token case, batch 256 fp32, batch 1024 bf16, MTP
packed 64 x 7 fp32, variable-length packed fp16 and its disable_state_update
run) gets its own entry under "configs".  Inputs are resident in HBM when a
timed region starts; the state moved per step is far larger than L2 (except
for the tiny case, which is launch-bound), so no flush is needed between
steps.  Prints ONE JSON line.

--impl reference times the CPU oracle (the plain double-precision definition)
on the host cores, on bounded samples of the same workload.

--record-traffic CSV reads an ncu CSV (dram__bytes_read.sum and
dram__bytes_write.sum per launch) of a --workload run and records the DRAM
bytes per call of that workload's kernels, with the hash of their sources, in
profiles/traffic.json; the bench line reports it as roofline.traffic while the
sources are unchanged.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "SSU state-updates/s and achieved HBM GB/s (% of GB300 peak) at batch 256"
UNIT = "state-updates/s"
FALLBACK_HBM_GBS = 6800.0

DESCRIPTIONS = {
    "b256_fp32": "one-token decode, batch 256, heads 128, dim 64, dstate 128, groups 8, fp32 state "
                 "pool of 512 slots, random distinct read/destination slots with 5% pad (id 0), "
                 "bf16 x/z/B/C, fp32 dt with bias and softplus, D",
    "b1024_bf16": "one-token decode, batch 1024, heads 128, dim 64, dstate 128, groups 8, bf16 state "
                  "pool of 1024 slots, identity tables",
    "mtp_64x7_fp32": "MTP packed decode, 64 sequences x 7 rows, heads 128, dim 64, dstate 128, groups 8, "
                     "fp32 pool of 1024 slots, 2-D read table, destination table read+448, "
                     "num_accepted U{1..7}",
    "varlen_fp16": "variable-length packed decode, 128 sequences of length U{0..8}, heads 64, dim 64, "
                   "dstate 128, groups 1, fp16 pool of 2048 slots, flat per-row read table, 3% pad",
    "varlen_fp16_disable": "varlen_fp16 with disable_state_update=True on identical inputs (seeds read, "
                           "nothing written)",
    "tiny_onetoken": "one-token decode, batch 2, heads 8, dim 8, dstate 128, groups 2, fp16 zero state",
    "replay_b256_fp32": "one-token decode on the checkpoint + buffer form (ReplaySSM), batch 256, heads 128, "
                        "dim 64, dstate 128, groups 8, fp32 checkpoints (512 slots), buffer length 16, "
                        "sequence b starting with b % 16 buffered entries (1/16 of the sequences fold per step)",
    "replay_e4m3_b256_fp32": "replay_b256_fp32 with an E4M3 read copy of the checkpoints (one fp32 scale per "
                             "state row): steps that do not fold read the copy, folds rewrite it",
    "replay_nvfp4_b256_fp32": "replay_b256_fp32 with an NVFP4 read copy of the checkpoints (E2M1 codes, an E4M3 "
                              "scale per 16 elements, an fp32 scale per state row): steps that do not fold read "
                              "the copy, folds rewrite it",
    "replay_f16copy_b256_fp32": "replay_b256_fp32 with an fp16 read copy of the checkpoints: steps that do not "
                                "fold read the copy, folds rewrite it",
    "copy_slots_b256_fp32": "256 whole-slot state copies of 4 MiB (heads 128, dim 64, dstate 128, fp32) between "
                            "random disjoint slot sets of a 512-slot pool; steps alternate the direction",
    "verify_b256_t4_fp32": "speculative decoding on the checkpoint + buffer form (ReplaySSM), batch 256, 4 drafts "
                           "per sequence, heads 128, dim 64, dstate 128, groups 8, fp32 checkpoints (512 slots, 13 "
                           "pad entries), buffer length 16, sequence b holding (b + step) % 9 committed entries (the "
                           "flush c + 2T >= L fires for 1/9 of the sequences each step)",
    "ssd_prefill_16k_bf16": "packed variable-length SSD prefill, 8 sequences of U{1024..3072} tokens (14269 in "
                            "all), heads 128, dim 64, dstate 128, groups 8, chunk 256, bf16 x/z/B/C/y, fp32 dt "
                            "with bias and softplus, D, fp32 initial and final states",
}
COPY_METRIC = "whole-slot state copies/s and achieved HBM GB/s (read + write)"
COPY_UNIT = "copies/s"
SSD_METRIC = "SSD prefill tokens/s and achieved HBM GB/s (inputs and outputs once)"
VERIFY_METRIC = "verified draft tokens/s and achieved HBM GB/s"
VERIFY_UNIT = "draft-tokens/s"
SSD_UNIT = "tokens/s"
KERNEL_SOURCES = {"onetoken": ["ssu_onetoken.cu", "ssu_device.cuh", "ssu_internal.h"],
                  "packed": ["ssu_packed.cu", "ssu_packed_long.cu", "ssu_device.cuh", "ssu_internal.h"],
                  "replay": ["ssu_replay.cuh", "ssu_replay_bf16.cu", "ssu_device.cuh", "ssu_internal.h"],
                  "copy": ["ssu_copy.cu", "ssu_device.cuh", "ssu_internal.h"],
                  "verify": ["ssu_verify.cu", "ssu_verify.h", "ssu_device.cuh", "ssu_internal.h"],
                  "ssd": ["ssu_ssd.cu", "ssu_ssd_tc.cu", "ssu_ssd_params.h", "ssu_device.cuh", "ssu_internal.h"]}


# --------------------------------------------------------------------------
# Accounting (host side, from the tables).
# --------------------------------------------------------------------------
def _lengths(w):
    if w.kind in ("onetoken", "replay"):
        return [1] * w.nseq
    if w.cu_seqlens is not None:
        cu = w.cu_seqlens.cpu().tolist()
        return [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
    return [w.dense_steps] * w.nseq


def _entry_slot(table, w, b, t, cu):
    if table is None:
        return b
    flat = table.reshape(-1)
    if w.kind == "onetoken":
        return int(flat[b])
    if w.slot_mode == workloads.SLOTS_PER_ROW:
        return int(flat[cu[b] + t])
    if table.dim() == 1:
        return int(flat[b + t])
    return int(table[b, t])


def replay_bytes(w) -> dict:
    """Bytes one call on the checkpoint + buffer form must move: every non-pad
    sequence reads its checkpoint and its c buffered entries (x, dt' per head
    row, B per group); a folding sequence writes the checkpoint back, any
    other appends one entry; plus the small operands and the counts."""
    H, P, N = w.state.shape[1:]
    G = w.B.shape[1]
    sb = H * P * N * w.state.element_size()
    # a read copy: what a step that does not fold reads instead of the
    # checkpoint, and what a fold writes besides it
    cb = sb if w.shadow is None else (w.shadow[0].numel() * w.shadow.element_size()
                                      + (0 if w.shadow_scale is None else w.shadow_scale[0].numel() * 4))
    io = w.x.element_size()
    entry = H * P * (io + 4) + G * N * io
    L = w.xbuf.shape[1]
    counts = w.count.cpu().tolist()
    slots = w.read.cpu().tolist() if w.read is not None else list(range(w.nseq))
    rd = wr = folds = 0
    for b, c in enumerate(counts):
        if slots[b] == w.pad_slot_id:
            continue
        rd += (sb if c + 1 == L else cb) + c * entry
        if c + 1 == L:
            wr += sb + (cb if w.shadow is not None else 0)
            folds += 1
        else:
            wr += entry
    small = sum(t.numel() * t.element_size() for t in (w.x, w.dt, w.B, w.C, w.z, w.A, w.D, w.dt_bias, w.read)
                if t is not None)
    small += w.x.numel() * w.x.element_size() + 2 * w.count.numel() * 4
    return {"state_read": rd, "state_write": wr, "small": small, "total": rd + wr + small, "folds": folds,
            "state_bytes_per_unit": sb}


def algorithmic_bytes(w) -> dict:
    """Bytes one call must move: each non-pad seed read once, each non-pad
    destination written once per token, plus every small operand once."""
    if w.kind == "replay":
        return replay_bytes(w)
    H, P, N = w.state.shape[1:]
    sb = H * P * N * w.state.element_size()
    lens = _lengths(w)
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    read_tab = None if w.read is None else w.read.cpu()
    dst_tab = None if w.dst is None else w.dst.cpu()
    acc = None if w.num_accepted is None else w.num_accepted.cpu().tolist()
    seeds = writes = 0
    for b, L in enumerate(lens):
        if L == 0:
            continue
        t_seed = max(acc[b] - 1, 0) if (acc is not None and w.kind == "packed") else 0
        if _entry_slot(read_tab, w, b, t_seed, cu) != w.pad_slot_id:
            seeds += 1
        if w.disable_state_update:
            continue
        wt = dst_tab if dst_tab is not None else read_tab
        for t in range(L):
            if _entry_slot(wt, w, b, t, cu) != w.pad_slot_id:
                writes += 1
    small = 0
    for t in (w.x, w.dt, w.B, w.C, w.z, w.A, w.D, w.dt_bias, w.read, w.dst, w.cu_seqlens,
              w.num_accepted):
        if t is not None:
            small += t.numel() * t.element_size()
    small += w.x.numel() * w.x.element_size()     # y
    return {"state_read": seeds * sb, "state_write": writes * sb, "small": small,
            "total": (seeds + writes) * sb + small, "seeds": seeds, "writes": writes,
            "state_bytes_per_unit": sb}


def kernel_hash(kind: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "selective_state_update_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_NAMES = {"onetoken": ["ssu_onetoken_kernel"], "packed": ["ssu_packed_kernel", "ssu_packed_long_kernel"], "replay": ["ssu_replay_kernel"],
                "copy": ["ssu_copy_kernel"], "verify": ["ssu_verify_fold_kernel", "ssu_verify_kernel"],
                "ssd": ["ssd_chunk_state_kernel", "ssd_state_pass_kernel", "ssd_scan_tc_kernel"]}


def profiled_traffic(kind: str, workload: str, batch=None):
    """DRAM bytes per call recorded in profiles/traffic.json from an ncu
    capture (--record-traffic), if that capture was taken of the kernel
    sources as they are now; None otherwise, and None for a run at another
    batch (--batch): the records are of the workloads at their own sizes."""
    if batch is not None:
        return None
    try:
        with open(TRAFFIC_JSON) as f:
            rec = json.load(f).get(f"{kind}/{workload}")
    except (OSError, ValueError):
        return None
    if not rec or rec.get("kernel_source_sha256_16") != kernel_hash(kind):
        return None
    return int(rec["bytes_per_call"])


_NCU_SCALE = {"byte": 1, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "kibyte": 1024, "mibyte": 1024 ** 2,
              "gibyte": 1024 ** 3}


def traffic_from_ncu_csv(path: str, kind: str) -> dict:
    """Per kernel of `kind`: the launches in an ncu --csv log and the median
    DRAM bytes (read + write) per launch; the call's bytes are the sum over
    the kind's kernels (each launches once per call)."""
    import csv
    per = {}
    with open(path, newline="") as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for row in csv.DictReader(lines):
        name = row.get("Kernel Name", "")
        base = next((k for k in KERNEL_NAMES[kind] if re.search(rf"\b{k}\b", name)), None)
        metric = row.get("Metric Name", "")
        if base is None or metric not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        v = float(row["Metric Value"].replace(",", "")) * _NCU_SCALE[row.get("Metric Unit", "byte").lower()]
        per.setdefault(base, {}).setdefault(row["ID"], 0.0)
        per[base][row["ID"]] += v
    if not per:
        raise SystemExit(f"no launch of {KERNEL_NAMES[kind]} with DRAM byte counters in {path}")
    out = {k: {"launches": len(v), "median_bytes": statistics.median(v.values())} for k, v in per.items()}
    return {"kernels": out, "bytes_per_call": int(sum(k["median_bytes"] for k in out.values()))}


def record_traffic(csv_path: str, workload: str, command: str) -> dict:
    kind = workload_kind(workload)
    rec = traffic_from_ncu_csv(csv_path, kind)
    rec.update({"kernel_source_sha256_16": kernel_hash(kind), "command": command,
                "recorded": time.strftime("%Y-%m-%d")})
    try:
        with open(TRAFFIC_JSON) as f:
            allrec = json.load(f)
    except (OSError, ValueError):
        allrec = {}
    allrec[f"{kind}/{workload}"] = rec
    with open(TRAFFIC_JSON, "w") as f:
        json.dump(allrec, f, indent=1, sort_keys=True)
        f.write("\n")
    return rec


LONG_ROWS_PER_SEQ = 6  # the library's packed kernel for long sequences takes rows >= 6 * nseq


def kernel_name(w) -> str:
    if w.kind == "packed" and w.rows >= LONG_ROWS_PER_SEQ * w.nseq:
        return "ssu_packed_long_kernel"
    return f"ssu_{w.kind}_kernel"


def workload_kind(workload: str) -> str:
    if workload.startswith("copy_"):
        return "copy"
    if workload.startswith("ssd_"):
        return "ssd"
    if workload.startswith("verify_"):
        return "verify"
    if workload.startswith("replay_"):
        return "replay"
    return "onetoken" if workload in ("tiny_onetoken", "b256_fp32", "b1024_bf16") else "packed"


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# --------------------------------------------------------------------------
# Several GPUs: independent replicas (each rank owns its own pool and batch;
# sequences never cross ranks, so there is no data exchange).  Timing takes
# the slowest rank; throughput counts the work of all ranks.
# --------------------------------------------------------------------------
def max_over_ranks(value: float, device) -> float:
    """Largest `value` over the ranks of the default process group (the value
    itself without one)."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank: int, world: int, steps: int, slowest_ms: float) -> float:
    """Whole-job throughput: the units every rank processed over the time of
    the slowest rank."""
    return units_per_rank * world * steps / (slowest_ms * 1e-3)


# --------------------------------------------------------------------------
# Clocks sampled while the timed region runs.
# --------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, device: torch.device):
        # nvidia-smi numbers GPUs physically; name ours by its UUID.
        try:
            u = str(torch.cuda.get_device_properties(device).uuid)
            self.dev = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            self.dev = str(device.index or 0)
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------
# Our arm.
# --------------------------------------------------------------------------
def _call(ssu, w, out, stream=None):
    common = dict(D=w.D, z=w.z, dt_bias=w.dt_bias, dt_softplus=w.dt_softplus,
                  state_batch_indices=w.read, dst_state_batch_indices=w.dst,
                  pad_slot_id=w.pad_slot_id, disable_state_update=w.disable_state_update, out=out,
                  stream=stream)
    if w.kind == "onetoken":
        return ssu.ssu_update_onetoken(w.state, w.x, w.dt, w.A, w.B, w.C, **common)
    if w.kind == "replay":
        # steady decode: this step's counts are the last step's output
        spare = w.meta.setdefault("count_spare", torch.empty_like(w.count))
        y, cnt = ssu.ssu_replay_update(w.state, w.x, w.dt, w.A, w.B, w.C, w.xbuf, w.dtbuf, w.Bbuf, w.count,
                                       count_out=spare, D=w.D, z=w.z, dt_bias=w.dt_bias,
                                       dt_softplus=w.dt_softplus, state_batch_indices=w.read,
                                       pad_slot_id=w.pad_slot_id, out=out, stream=stream, shadow=w.shadow,
                                       shadow_scale=w.shadow_scale)
        w.meta["count_spare"], w.count = w.count, cnt
        return y
    return ssu.ssu_update_packed(w.state, w.x, w.dt, w.A, w.B, w.C, cu_seqlens=w.cu_seqlens,
                                 num_accepted_tokens=w.num_accepted, slot_mode=w.slot_mode, **common)


def _per_step_inputs(w):
    return [t for t in (w.x, w.dt, w.z, w.B, w.C, w.read, w.dst, w.cu_seqlens, w.num_accepted)
            if t is not None]


DECODE_SUITE = ["b256_fp32", "tiny_onetoken", "b1024_bf16", "mtp_64x7_fp32", "varlen_fp16", "varlen_fp16_disable"]


def time_decode(workload, args, rank, world, device) -> dict:
    """Time one decode workload: `args.warmup` untimed calls, then
    `args.steps` timed calls bracketed by a barrier and a synchronize, with
    CUDA events on the launching stream around each call and around the whole
    region, clocks sampled meanwhile; then the end-to-end rate through the
    public call with the step's inputs copied from pinned host memory and y
    copied back inside the timed region."""
    import selective_state_update_gb300 as ssu
    w = make_workload(workload, args.batch, device, seed_offset=97 * rank)
    torch.cuda.synchronize()
    acct = algorithmic_bytes(w)
    tokens = w.rows
    ssu.ssu_prewarm(state_dtype=w.state.dtype, io_dtype=w.x.dtype, heads=w.state.shape[1],
                    dim=w.state.shape[2], dstate=w.state.shape[3], groups=w.B.shape[1],
                    packed=w.kind == "packed")
    stream = torch.cuda.current_stream()
    out = torch.empty_like(w.x)
    for _ in range(args.warmup):
        _call(ssu, w, out)
    torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    whole0, whole1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(device) as clocks:
        whole0.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            _call(ssu, w, out)
            ev[i][1].record(stream)
        whole1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = whole0.elapsed_time(whole1)
    launch_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    total_ms = max_over_ranks(total_ms, device)

    # End to end through the public call: per step, pinned host -> device
    # copies of the step's inputs, the update, and y back to pinned host.
    host_in = [t.cpu().pin_memory() for t in _per_step_inputs(w)]
    dev_in = _per_step_inputs(w)
    host_y = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_y.numel() * host_y.element_size()
    e2e_steps = max(3, min(args.steps, 400))
    for _ in range(2):
        for h, d in zip(host_in, dev_in):
            d.copy_(h, non_blocking=True)
        _call(ssu, w, out)
        host_y.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        for h, d in zip(host_in, dev_in):
            d.copy_(h, non_blocking=True)
        _call(ssu, w, out)
        host_y.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, device)

    peak, peak_src = hbm_peak()
    achieved = acct["total"] / (launch_ms * 1e-3) / 1e9
    kind = w.kind
    moved = acct["state_read"] + acct["state_write"]
    rec = {
        "value": aggregate_rate(tokens, world, args.steps, total_ms),
        "unit": UNIT,
        "ms_per_step": total_ms / args.steps,
        "config": {"workload": f"{workload}: {DESCRIPTIONS[workload]}"
                               + (f" (batch {args.batch})" if args.batch else ""),
                   "sequences_per_gpu": w.nseq, "rows_per_gpu": tokens,
                   "state_dtype": str(w.state.dtype).replace("torch.", ""),
                   "io_dtype": str(w.x.dtype).replace("torch.", ""),
                   "parallelism": f"{world} independent replicas (one pool and batch per GPU)",
                   "l2": ("no flush: inputs larger than L2 (%.2f GB of state moved per step)" % (moved / 1e9))
                         if moved > 200e6 else
                         "no flush: launch-bound case (%.1f KB of state per step, L2-resident)" % (moved / 1e3)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_src} copy bandwidth",
                     "traffic": profiled_traffic(kind, workload, args.batch),
                     "algorithmic_bytes_per_launch": acct["total"],
                     "kernel": kernel_name(w), "launch_ms": launch_ms},
        "e2e": {"value": aggregate_rate(tokens, world, e2e_steps, e2e_s * 1e3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
    }
    del w, out, host_in, dev_in, host_y
    torch.cuda.empty_cache()
    return rec


def run_ours(args, rank, world, device):
    from selective_state_update_gb300 import build as ssu_build
    import selective_state_update_gb300 as ssu
    ssu_build.build()
    ssu.lib()
    suite = [args.workload] if args.workload else DECODE_SUITE
    recs = {name: time_decode(name, args, rank, world, device) for name in suite}
    head = recs[suite[0]]
    result = {
        "metric": METRIC,
        "value": head["value"],
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": head["config"],
        "roofline": head["roofline"],
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
    }
    if len(suite) > 1:
        result["configs"] = {
            name: {"workload": r["config"]["workload"], "value": r["value"], "unit": r["unit"],
                   "ms_per_step": r["ms_per_step"], "launch_ms": r["roofline"]["launch_ms"],
                   "algorithmic_bytes_per_launch": r["roofline"]["algorithmic_bytes_per_launch"],
                   "achieved_gbs": r["roofline"]["achieved"], "roofline_frac": r["roofline"]["frac"],
                   "traffic": r["roofline"]["traffic"], "kernel": r["roofline"]["kernel"],
                   "e2e": r["e2e"], "gpu_launches": r["gpu_launches"], "clocks": r["clocks"], "l2": r["config"]["l2"]}
            for name, r in recs.items()}
        result["gpu_launches_all_configs"] = sum(r["gpu_launches"] for r in recs.values())
    return result


def run_copy(args, rank, world, device):
    """The slot-copy workload: one step = one ssu_batch_copy call moving every
    copy of the batch (even steps source -> destination, odd steps back)."""
    from selective_state_update_gb300 import build as ssu_build
    import selective_state_update_gb300 as ssu
    ssu_build.build()
    ssu.lib()
    w = make_workload(args.workload, args.batch, device, seed_offset=97 * rank)
    slot_bytes = w.state[0].numel() * w.state.element_size()
    tables = [ssu.slot_copies(w.state, w.src, w.dst), ssu.slot_copies(w.state, w.dst, w.src)]
    status = torch.zeros(1, dtype=torch.int32, device=device)
    call = lambda i: ssu.ssu_batch_copy(tables[i % 2], slot_bytes, status=status)
    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    whole0, whole1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(device) as clocks:
        whole0.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            call(i)
            ev[i][1].record(stream)
        whole1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(whole0.elapsed_time(whole1), device)
    launch_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    if int(status.item()) != 0:
        raise SystemExit(f"ssu_batch_copy reported status {int(status.item())}")
    # End to end: the step's descriptor table from pinned host memory, the
    # copies, the status word back to pinned host memory.
    host_tabs = [t.cpu().pin_memory() for t in tables]
    host_status = torch.empty(1, dtype=torch.int32, pin_memory=True)
    h2d = host_tabs[0].numel() * 8
    e2e_steps = max(3, min(args.steps, 400))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        tables[i % 2].copy_(host_tabs[i % 2], non_blocking=True)
        call(i)
        host_status.copy_(status, non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, device)
    n = w.nseq
    algo = 2 * n * slot_bytes + 2 * n * 24
    peak, peak_src = hbm_peak()
    achieved = algo / (launch_ms * 1e-3) / 1e9
    return {
        "metric": COPY_METRIC, "value": aggregate_rate(n, world, args.steps, total_ms), "unit": COPY_UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}"
                               + (f" (batch {args.batch})" if args.batch else ""),
                   "copies_per_gpu": n, "bytes_per_copy": slot_bytes,
                   "parallelism": f"{world} independent replicas (one pool per GPU)",
                   "l2": "no flush: %.2f GB moved per step" % (algo / 1e9)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_src} copy bandwidth", "traffic": profiled_traffic("copy", args.workload, args.batch),
                     "algorithmic_bytes_per_launch": algo, "kernel": "ssu_copy_kernel", "launch_ms": launch_ms},
        "e2e": {"value": aggregate_rate(n, world, e2e_steps, e2e_s * 1e3), "unit": COPY_UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4},
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
    }


def copy_oracle_rate(w_cpu, budget_s: float):
    """The copy oracle on samples of the slot-copy workload: each sample a
    few whole-slot copies applied to a compact buffer of their slots."""
    import numpy as np
    import oracle
    nbytes = w_cpu.state[0].numel() * w_cpu.state.element_size()
    done, spent, samples, idx, per = 0, 0.0, 0, 0, 4
    n = w_cpu.nseq
    while spent < budget_s:
        ids = [(idx + i) % n for i in range(per)]
        idx += per
        # compact buffer: the sampled source slots, then room for their destinations
        srcs = w_cpu.state[w_cpu.src[ids]].contiguous().view(-1).view(torch.uint8).numpy()
        buf = np.concatenate([srcs, np.zeros_like(srcs)])
        copies = [(i * nbytes, (per + i) * nbytes, nbytes) for i in range(per)]
        t0 = time.perf_counter()
        oracle.batch_copy(buf, copies)
        spent += time.perf_counter() - t0
        done += per
        samples += 1
    return done / spent, f"{done} copies of {nbytes} bytes in {samples} samples"


def verify_bytes(w, count) -> dict:
    """Bytes one verification call must move: per non-pad sequence the
    checkpoint once, its c committed entries, the drafts' inputs, outputs and
    appended entries, and on a flush the checkpoint written once; pad
    sequences only their drafts' inputs and outputs."""
    batch, T, H, P = w.x.shape
    G, N = w.B.shape[2], w.B.shape[3]
    io = w.x.element_size()
    sb = H * P * N * w.state.element_size()
    entry = H * P * (io + 4) + G * N * io               # x, dt' and B of one buffered step
    draft_in = H * P * (io * (2 if w.z is not None else 1) + w.dt.element_size()) + 2 * G * N * io
    draft_out = H * P * io
    L = w.xbuf.shape[1]
    total = 0
    for b in range(batch):
        total += T * (draft_in + draft_out) + 4 + 4 + 4  # drafts, y, table entry and counts
        if int(w.read[b]) == w.pad_slot_id:
            continue
        c = int(count[b])
        total += sb + c * entry + T * entry
        if c + 2 * T >= L:
            total += sb
    return {"total": total, "state_bytes_per_unit": sb}


def run_verify(args, rank, world, device):
    """The verification workload: one step = one ssu_replay_verify call over
    the batch (its fold and verify launches); the committed counts cycle
    through (b + step) % 9, arrays prepared before the timed region."""
    from selective_state_update_gb300 import build as ssu_build
    import selective_state_update_gb300 as ssu
    ssu_build.build()
    ssu.lib()
    w = make_workload(args.workload, args.batch, device, seed_offset=97 * rank)
    batch, T = w.x.shape[0], w.x.shape[1]
    period = w.xbuf.shape[1] - 2 * T + 1
    counts = [((torch.arange(batch, device=device) + k) % period).to(torch.int32) for k in range(period)]
    count_out = torch.empty(batch, dtype=torch.int32, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    out = torch.empty_like(w.x)

    def call(i):
        return ssu.ssu_replay_verify(w.state, w.x, w.dt, w.A, w.B, w.C, w.xbuf, w.dtbuf, w.Bbuf, counts[i % period],
                                     count_out=count_out, D=w.D, z=w.z, dt_bias=w.dt_bias, dt_softplus=w.dt_softplus,
                                     state_batch_indices=w.read, pad_slot_id=w.pad_slot_id, out=out, status=status)
    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    whole0, whole1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(device) as clocks:
        whole0.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            call(i)
            ev[i][1].record(stream)
        whole1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(whole0.elapsed_time(whole1), device)
    call_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    if int(status.item()) != 0:
        raise SystemExit(f"ssu_replay_verify reported status {int(status.item())}")
    acct = [verify_bytes(w, counts[k].cpu()) for k in range(period)]
    algo = statistics.mean(a["total"] for a in acct)
    # End to end: the drafts' inputs and the counts from pinned host memory,
    # the call, y back to pinned host memory.
    dev_in = [t for t in (w.x, w.dt, w.z, w.B, w.C) if t is not None]
    host_in = [t.cpu().pin_memory() for t in dev_in]
    host_counts = [c.cpu().pin_memory() for c in counts]
    host_y = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host_in) + batch * 4
    d2h = host_y.numel() * host_y.element_size()
    e2e_steps = max(3, min(args.steps, 400))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        for hsrc, d in zip(host_in, dev_in):
            d.copy_(hsrc, non_blocking=True)
        counts[i % period].copy_(host_counts[i % period], non_blocking=True)
        call(i)
        host_y.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, device)
    peak, peak_src = hbm_peak()
    achieved = algo / (call_ms * 1e-3) / 1e9
    units = batch * T
    return {
        "metric": VERIFY_METRIC, "value": aggregate_rate(units, world, args.steps, total_ms), "unit": VERIFY_UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}"
                               + (f" (batch {args.batch})" if args.batch else ""),
                   "sequences_per_gpu": batch, "drafts_per_sequence": T,
                   "parallelism": f"{world} independent replicas (one pool and batch per GPU)",
                   "l2": "no flush: %.2f GB of checkpoints read per step" % (algo / 1e9)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_src} copy bandwidth", "traffic": profiled_traffic("verify", args.workload, args.batch),
                     "algorithmic_bytes_per_launch": algo,
                     "kernel": "verify call (ssu_verify_fold_kernel + ssu_verify_kernel)", "launch_ms": call_ms},
        "e2e": {"value": aggregate_rate(units, world, e2e_steps, e2e_s * 1e3), "unit": VERIFY_UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": (1 if w.state.shape[2] <= 64 else 2) * args.steps,  # the fold runs in the verify launch up to dim 64
        "clocks": clocks.summary(),
    }


def verify_oracle_rate(w_cpu, budget_s: float):
    """The oracle's verification on samples of the workload: a few sequences
    at a time (with their committed entries), all heads."""
    import oracle
    oracle.build()
    batch, T = w_cpu.x.shape[0], w_cpu.x.shape[1]
    done, spent, idx, per = 0, 0.0, 0, 2
    while spent < budget_s:
        seqs = [(idx + i) % batch for i in range(per)]
        idx += per
        sel = torch.tensor(seqs)
        slots = w_cpu.read[sel].long()
        keep = slots != w_cpu.pad_slot_id
        used = slots[keep]
        order = torch.cat([used, torch.tensor([s for s in range(w_cpu.state.shape[0]) if s not in set(used.tolist())][:1])])
        remap = {int(s): i for i, s in enumerate(order.tolist())}
        slot_of = torch.tensor([remap.get(int(s), -1) if k else -1 for s, k in zip(slots, keep)])
        t0 = time.perf_counter()
        oracle.replay_verify(w_cpu.state[order], w_cpu.x[sel], w_cpu.dt[sel], w_cpu.A, w_cpu.B[sel], w_cpu.C[sel],
                             w_cpu.xbuf[order], w_cpu.dtbuf[order], w_cpu.Bbuf[order], w_cpu.count[sel], D=w_cpu.D,
                             z=None if w_cpu.z is None else w_cpu.z[sel], dt_bias=w_cpu.dt_bias,
                             dt_softplus=w_cpu.dt_softplus, slot_of=slot_of, pad_slot_id=-1)
        spent += time.perf_counter() - t0
        done += per * T
    return done / spent, f"{done} draft tokens in samples of {per} sequences"


def ssd_accounting(w) -> dict:
    """Bytes the prefill must move at least (every input read once, y and the
    returned states written once) and the tensor-core work of the chunked
    evaluation, per call."""
    T, H, P = w.x.shape
    G, N = w.B.shape[1], w.B.shape[2]
    io = w.x.element_size()
    sb = H * P * N * torch.finfo(w.state_dtype).bits // 8
    nseq = w.nseq
    meta = (w.cu_chunk_seqlens.numel() + w.seq_idx.numel() + w.last_chunk_indices.numel()) * 4
    inputs = (T * H * P * io * (2 if w.z is not None else 1) + T * H * w.dt.element_size() + 2 * T * G * N * io
              + (nseq * sb if w.initial_states is not None else 0) + meta)
    outputs = T * H * P * io + nseq * sb
    nchunks = w.seq_idx.numel()
    ch = nchunks * H
    # chunk states, then the scan's C . S_in^T and the causal C . B^T and
    # W . X products, counted on 16 x 16 tiles up to the diagonal
    lens = (w.cu_chunk_seqlens[1:] - w.cu_chunk_seqlens[:-1]).tolist()
    causal = sum(sum((t // 16 + 1) * 16 for t in range(0, L, 16)) * 16 for L in lens)  # (t, s) pairs, 16-row tiles
    flops = H * (2 * T * P * N + 2 * T * N * P + 2 * causal * N + 2 * causal * P)
    # the chunk states cross the workspace four times (written, read and
    # replaced by the entering states, read by the scan); C . B^T stays in
    # the scan's tensor memory
    return {"inputs": inputs, "outputs": outputs, "total": inputs + outputs, "flops": flops,
            "workspace": 4 * ch * P * N * 4, "tokens": T}


def run_ssd(args, rank, world, device):
    """The SSD prefill workload: one step = one ssu_ssd_prefill call over the
    packed batch (three kernel launches)."""
    from selective_state_update_gb300 import build as ssu_build
    import selective_state_update_gb300 as ssu
    ssu_build.build()
    ssu.lib()
    w = make_workload(args.workload, args.batch, device, seed_offset=97 * rank)
    acct = ssd_accounting(w)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    out = torch.empty_like(w.x)

    def call():
        return ssu.ssu_ssd_prefill(w.x, w.dt, w.A, w.B, w.C, w.chunk_size, w.cu_chunk_seqlens, w.seq_idx,
                                   w.last_chunk_indices, out=out, D=w.D, z=w.z, dt_bias=w.dt_bias,
                                   dt_softplus=w.dt_softplus, dt_limit=w.dt_limit,
                                   initial_states=w.initial_states, state_dtype=w.state_dtype, nseq=w.nseq,
                                   status=status)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    whole0, whole1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(device) as clocks:
        whole0.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            call()
            ev[i][1].record(stream)
        whole1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(whole0.elapsed_time(whole1), device)
    call_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    if int(status.item()) != 0:
        raise SystemExit(f"ssu_ssd_prefill reported status {int(status.item())}")
    # End to end: the step's inputs from pinned host memory, the prefill, y
    # and the returned states back to pinned host memory.
    dev_in = [t for t in (w.x, w.dt, w.z, w.B, w.C, w.initial_states, w.cu_chunk_seqlens, w.seq_idx,
                          w.last_chunk_indices) if t is not None]
    host_in = [t.cpu().pin_memory() for t in dev_in]
    host_y = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    _, st = call()
    host_s = torch.empty(st.shape, dtype=st.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_y.numel() * host_y.element_size() + host_s.numel() * host_s.element_size()
    e2e_steps = max(3, min(args.steps, 50))
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        for h, d in zip(host_in, dev_in):
            d.copy_(h, non_blocking=True)
        _, st = call()
        host_y.copy_(out, non_blocking=True)
        host_s.copy_(st, non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, device)
    peak, peak_src = hbm_peak()
    achieved = acct["total"] / (call_ms * 1e-3) / 1e9
    return {
        "metric": SSD_METRIC, "value": aggregate_rate(acct["tokens"], world, args.steps, total_ms),
        "unit": SSD_UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS[args.workload]}"
                               + (f" (batch {args.batch})" if args.batch else ""),
                   "tokens_per_gpu": acct["tokens"], "chunks": int(w.seq_idx.numel()),
                   "parallelism": f"{world} independent replicas (one packed batch per GPU)",
                   "l2": "no flush: %.2f GB of inputs and outputs per step" % (acct["total"] / 1e9),
                   "tensor_flops_per_call": acct["flops"],
                   "workspace_bytes_moved_per_call": acct["workspace"]},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_src} copy bandwidth", "traffic": profiled_traffic("ssd", args.workload, args.batch),
                     "algorithmic_bytes_per_launch": acct["total"],
                     "kernel": "ssd prefill call (ssd_chunk_state + ssd_state_pass + ssd_scan_tc)",
                     "launch_ms": call_ms},
        "e2e": {"value": aggregate_rate(acct["tokens"], world, e2e_steps, e2e_s * 1e3), "unit": SSD_UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks.summary(),
    }


def ssd_oracle_rate(w_cpu, budget_s: float, heads_per_sample: int = 16):
    """The oracle's packed SSD on samples of the prefill workload: each sample
    one whole sequence on one block of `heads_per_sample` heads (whole
    groups), sequences and head blocks in turn; a token counts as
    heads_per_sample / heads of a token."""
    import oracle
    oracle.build()
    H, G = w_cpu.x.shape[1], w_cpu.B.shape[1]
    hs = max(heads_per_sample, H // G)
    gs = hs // (H // G)
    cu = w_cpu.cu_seqlens.tolist()
    cuc = w_cpu.cu_chunk_seqlens.tolist()
    si = w_cpu.seq_idx.tolist()
    done, spent, samples = 0.0, 0.0, 0
    while spent < budget_s:
        b = samples % w_cpu.nseq
        h0 = (samples // w_cpu.nseq * hs) % H
        g0 = h0 // (H // G)
        lo, hi = cu[b], cu[b + 1]
        chunks = [c for c in range(len(si)) if si[c] == b]
        sub_cu = torch.tensor([cuc[c] - lo for c in chunks] + [cuc[chunks[-1] + 1] - lo], dtype=torch.int32)
        hsl, gsl = slice(h0, h0 + hs), slice(g0, g0 + gs)
        sub = lambda t, sl: None if t is None else t[lo:hi, sl].contiguous()
        t0 = time.perf_counter()
        oracle.ssd(sub(w_cpu.x, hsl), sub(w_cpu.dt, hsl), w_cpu.A[hsl], sub(w_cpu.B, gsl), sub(w_cpu.C, gsl),
                   sub_cu, torch.zeros(len(chunks), dtype=torch.int32), 1,
                   D=None if w_cpu.D is None else w_cpu.D[hsl], z=sub(w_cpu.z, hsl),
                   dt_bias=None if w_cpu.dt_bias is None else w_cpu.dt_bias[hsl], dt_softplus=w_cpu.dt_softplus,
                   dt_limit=w_cpu.dt_limit,
                   initial_states=None if w_cpu.initial_states is None else
                   w_cpu.initial_states[b:b + 1, hsl].contiguous(),
                   state_dtype=w_cpu.state_dtype)
        spent += time.perf_counter() - t0
        done += (hi - lo) * hs / H
        samples += 1
    return done / spent, (f"{samples} samples of one whole sequence on {hs} of {H} heads "
                          f"({done:.0f} token-equivalents)")


# --------------------------------------------------------------------------
# The oracle on the host cores.
# --------------------------------------------------------------------------
def _sample_problem(w, seqs):
    """The sequences `seqs` of workload `w` (CPU tensors) with a compact pool."""
    from dataclasses import replace
    lens = _lengths(w)
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    rows = [r for b in seqs for r in range(cu[b], cu[b + 1])]
    sub_lens = [lens[b] for b in seqs]
    pad = w.pad_slot_id

    def rows_of(t):
        if t is None:
            return None
        if w.kind in ("onetoken", "replay"):
            return t.reshape(-1)[seqs]
        if w.slot_mode == workloads.SLOTS_PER_ROW:
            return t.reshape(-1)[rows]
        return t[seqs]

    rd, wr = rows_of(w.read), rows_of(w.dst)
    used = sorted({int(v) for t in (rd, wr) if t is not None for v in t.reshape(-1).tolist()} - {pad})
    order = ([pad] if 0 <= pad < w.state.shape[0] else []) + used
    m = {s: i for i, s in enumerate(order)}
    new_pad = m.get(pad, pad)
    remap = lambda t: None if t is None else torch.tensor(
        [new_pad if v == pad else m[v] for v in t.reshape(-1).tolist()], dtype=t.dtype).view(t.shape)
    sel = lambda t: None if t is None else t[rows]
    sub_cu = torch.tensor([sum(sub_lens[:i]) for i in range(len(sub_lens) + 1)], dtype=torch.int32)
    if w.kind == "replay":
        sub = replace(w, state=w.state[order], x=sel(w.x), dt=sel(w.dt), B=sel(w.B), C=sel(w.C), z=sel(w.z),
                      read=remap(rd), pad_slot_id=new_pad, xbuf=w.xbuf[order], dtbuf=w.dtbuf[order],
                      Bbuf=w.Bbuf[order], count=w.count[seqs], meta=dict(w.meta))
        if w.shadow is not None:
            import oracle
            sub.shadow, sub.shadow_scale = oracle.shadow_refresh(sub.state, _oracle_shadow_format(w))
        return sub
    return replace(w, state=w.state[order], x=sel(w.x), dt=sel(w.dt), B=sel(w.B), C=sel(w.C), z=sel(w.z),
                   read=remap(rd), dst=remap(wr), pad_slot_id=new_pad,
                   cu_seqlens=sub_cu if w.kind == "packed" else None,
                   num_accepted=None if w.num_accepted is None else w.num_accepted[seqs], dense_steps=0)


def _oracle_shadow_format(w):
    import oracle
    if w.shadow is None:
        return oracle.SHADOW_NONE
    return {"f16": oracle.SHADOW_F16, "e4m3": oracle.SHADOW_E4M3,
            "nvfp4": oracle.SHADOW_NVFP4}[w.meta["shadow_format"]]


def _oracle_call(sub):
    import oracle
    if sub.kind == "replay":
        return oracle.replay(sub.state, sub.x, sub.dt, sub.A, sub.B, sub.C, sub.xbuf, sub.dtbuf, sub.Bbuf, sub.count,
                             D=sub.D, z=sub.z, dt_bias=sub.dt_bias, dt_softplus=sub.dt_softplus,
                             slot_of=sub.read, pad_slot_id=sub.pad_slot_id, shadow=sub.shadow,
                             shadow_scale=sub.shadow_scale, shadow_format=_oracle_shadow_format(sub))
    mode = oracle.SLOTS_PER_ROW if sub.slot_mode == workloads.SLOTS_PER_ROW else oracle.SLOTS_STRIDED
    return oracle.ssu(sub.state, sub.x, sub.dt, sub.A, sub.B, sub.C, D=sub.D, z=sub.z, dt_bias=sub.dt_bias,
                      dt_softplus=sub.dt_softplus, read=oracle.Table.of(sub.read, mode),
                      dst=oracle.Table.of(sub.dst, mode), pad_slot_id=sub.pad_slot_id,
                      disable_state_update=sub.disable_state_update, cu_seqlens=sub.cu_seqlens,
                      num_accepted=sub.num_accepted if sub.kind == "packed" else None)


SEEDS = {"tiny_onetoken": 1001, "b256_fp32": 1002, "b1024_bf16": 1003, "mtp_64x7_fp32": 1004,
         "varlen_fp16": 1005, "varlen_fp16_disable": 1005, "replay_b256_fp32": 1006, "copy_slots_b256_fp32": 1007, "replay_e4m3_b256_fp32": 1008, "replay_nvfp4_b256_fp32": 1012,
         "replay_f16copy_b256_fp32": 1009, "ssd_prefill_16k_bf16": 1010, "verify_b256_t4_fp32": 1011}


def make_workload(workload, batch, device, seed_offset=0):
    gen = workloads.NAMED[workload]
    kw = {}
    if batch is not None:
        if workload not in ("b256_fp32", "mtp_64x7_fp32", "replay_b256_fp32", "replay_e4m3_b256_fp32",
                            "replay_nvfp4_b256_fp32",
                            "replay_f16copy_b256_fp32", "copy_slots_b256_fp32", "ssd_prefill_16k_bf16",
                            "verify_b256_t4_fp32"):
            raise SystemExit(f"--batch does not apply to the {workload} workload")
        kw["batch"] = batch
    w = gen(device=device, seed=SEEDS[workload] + seed_offset, **kw)
    if getattr(w, "shadow", None) is not None and str(device) != "cpu":
        # the read copy of the checkpoints, built by the library
        import selective_state_update_gb300 as ssu
        ssu.ssu_shadow_refresh(w.state, w.shadow, w.shadow_scale)
    return w


def _cpu_workload(args):
    return make_workload(args.workload or DECODE_SUITE[0], args.batch, "cpu")


def oracle_rate(w_cpu, budget_s: float):
    """Time the oracle on samples of `w_cpu` for about `budget_s` seconds;
    returns (sequence-token updates per second, description)."""
    import oracle
    oracle.build()
    nseq = w_cpu.nseq
    lens = _lengths(w_cpu)
    done_tokens, spent, nsamples, idx = 0, 0.0, 0, 0
    per = 1
    while spent < budget_s:
        seqs = [(idx + i) % nseq for i in range(per)]
        idx += per
        sub = _sample_problem(w_cpu, seqs)
        t0 = time.perf_counter()
        _oracle_call(sub)
        dt = time.perf_counter() - t0
        spent += dt
        done_tokens += sum(lens[b] for b in seqs)
        nsamples += 1
        if dt < 0.5 and per < nseq:
            per = min(nseq, per * 2)
    return done_tokens / spent, f"{done_tokens} sequence-tokens in {nsamples} samples of consecutive sequences"


def host_threads() -> int:
    """The host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_rate_threaded(w_cpu, budget_s: float, threads: int):
    """The oracle, unchanged, on `threads` host threads at once (its C call
    runs without the GIL): one-sequence samples, cycled until about
    `budget_s` seconds of wall time have passed; returns (sequence-token
    updates per second over the wall time, description)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    oracle.build()
    lens = _lengths(w_cpu)
    order = [b for b in range(w_cpu.nseq) if lens[b] > 0][:2 * threads]
    subs = [(_sample_problem(w_cpu, [b]), lens[b]) for b in order]
    if not subs:
        return 0.0, "no non-empty sequence to sample"
    stop = time.perf_counter() + budget_s

    def worker(i):
        done, k = 0, i
        while time.perf_counter() < stop:
            sub, n = subs[k % len(subs)]
            _oracle_call(sub)
            done += n
            k += threads
        return done

    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        total = sum(ex.map(worker, range(threads)))
    el = time.perf_counter() - t0
    return total / el, f"{total} sequence-tokens on {threads} threads, cycling {len(subs)} one-sequence samples"


def run_reference(args):
    wl = args.workload or DECODE_SUITE[0]
    w_cpu = _cpu_workload(args)
    import oracle
    oracle.build()
    if getattr(w_cpu, "kind", "") == "verify":
        budget = min(150.0, 5.0 + 1.0 * (args.steps + args.warmup))
        value, sample = verify_oracle_rate(w_cpu, budget)
        return {
            "impl": "reference", "metric": VERIFY_METRIC, "value": value, "unit": VERIFY_UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * w_cpu.x.shape[0] * w_cpu.x.shape[1] / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{wl}: {DESCRIPTIONS[wl]}"},
            "cpu_baseline": {"value": value, "unit": VERIFY_UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": VERIFY_UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
    if getattr(w_cpu, "kind", "") == "ssd":
        budget = min(150.0, 5.0 + 1.0 * (args.steps + args.warmup))
        value, sample = ssd_oracle_rate(w_cpu, budget)
        return {
            "impl": "reference", "metric": SSD_METRIC, "value": value, "unit": SSD_UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * ssd_accounting(w_cpu)["tokens"] / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{wl}: {DESCRIPTIONS[wl]}"},
            "cpu_baseline": {"value": value, "unit": SSD_UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": SSD_UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
    if getattr(w_cpu, "kind", "") == "copy":
        budget = min(150.0, 1.0 + 0.05 * (args.steps + args.warmup))
        value, sample = copy_oracle_rate(w_cpu, budget)
        return {
            "impl": "reference", "metric": COPY_METRIC, "value": value, "unit": COPY_UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": {"workload": f"{wl}: {DESCRIPTIONS[wl]}"},
            "cpu_baseline": {"value": value, "unit": COPY_UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": COPY_UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
    lens = _lengths(w_cpu)
    # one step = the oracle on one sequence; size the run to end within minutes
    steps_total = args.steps + args.warmup
    seq_per_step = 1
    for i in range(args.warmup):
        _oracle_call(_sample_problem(w_cpu, [i % w_cpu.nseq]))
    t0 = time.perf_counter()
    tokens = 0
    budget = 150.0
    done_steps = 0
    for i in range(args.steps):
        b = (i * 37) % w_cpu.nseq
        _oracle_call(_sample_problem(w_cpu, [b]))
        tokens += lens[b]
        done_steps += 1
        if time.perf_counter() - t0 > budget:
            break
    el = time.perf_counter() - t0
    value = tokens / el
    sample = (f"{done_steps} steps of one sequence each ({tokens} sequence-tokens) of the workload; "
              f"{steps_total} requested")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": done_steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / max(done_steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{wl}: {DESCRIPTIONS[wl]}"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(workloads.NAMED), default=None,
                    help="time one workload (default: the five decode configurations, batch 256 fp32 as headline)")
    ap.add_argument("--batch", type=int, default=None,
                    help="b256_fp32 / mtp_64x7_fp32 with another number of sequences (profiling captures)")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--record-traffic", metavar="CSV", default=None,
                    help="record the DRAM bytes per call of --workload's kernels from an ncu CSV into "
                         "profiles/traffic.json (no GPU needed)")
    ap.add_argument("--record-command", default="", help="the command the ncu CSV was captured with")
    args = ap.parse_args()
    if args.record_traffic:
        if not args.workload:
            ap.error("--record-traffic needs --workload")
        print(json.dumps(record_traffic(args.record_traffic, args.workload, args.record_command)))
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    # The oracle baseline runs before the first GPU call (no fork after CUDA init).
    cpu = None
    wl = args.workload or DECODE_SUITE[0]
    is_copy = wl.startswith("copy_")
    is_ssd = wl.startswith("ssd_")
    is_verify = wl.startswith("verify_")
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        w_cpu = _cpu_workload(args)
        if is_verify:
            rate, desc = verify_oracle_rate(w_cpu, args.cpu_baseline_seconds)
            cpu = {"value": rate, "unit": VERIFY_UNIT, "cores": 1, "kind": "oracle",
                   "sample": f"{desc} of {wl} (single-threaded plain C, double precision)"}
        elif is_ssd:
            rate, desc = ssd_oracle_rate(w_cpu, args.cpu_baseline_seconds)
            cpu = {"value": rate, "unit": SSD_UNIT, "cores": 1, "kind": "oracle",
                   "sample": f"{desc} of {wl} (single-threaded plain C, double precision)"}
        elif is_copy:
            rate, desc = copy_oracle_rate(w_cpu, args.cpu_baseline_seconds)
            cpu = {"value": rate, "unit": COPY_UNIT, "cores": 1, "kind": "oracle",
                   "sample": f"{desc} of {wl} (numpy, one thread)"}
        else:
            rate, desc = oracle_rate(w_cpu, args.cpu_baseline_seconds)
            cpu = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
                   "sample": f"{desc} of {wl} (single-threaded plain C, double precision)"}
            threads = host_threads()
            if threads > 1:
                # all host cores, the single-core figure kept beside it; should the
                # threaded run fail, the single-core figure stands and says why
                try:
                    trate, tdesc = oracle_rate_threaded(w_cpu, args.cpu_baseline_seconds, threads)
                    cpu = {"value": trate, "unit": UNIT, "cores": threads, "kind": "oracle",
                           "sample": f"{tdesc} of {wl} (plain C, double precision)",
                           "single_core": {"value": rate, "sample": cpu["sample"]}}
                except Exception as e:  # noqa: BLE001 -- a baseline, not the measurement
                    cpu["sample"] += f"; the {threads}-thread run failed: {type(e).__name__}: {e}"
        del w_cpu

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (libssu has no CPU path)")
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    device = torch.device("cuda", local_rank if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(device)
    run = run_verify if is_verify else (run_ssd if is_ssd else (run_copy if is_copy else run_ours))
    res = run(args, rank, world, device)
    res["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
