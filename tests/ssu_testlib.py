"""Shared test helpers: run the oracle on a workload, decode tensors to float64,
compare with the tolerances the library promises."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

# Tolerances (GPU vs oracle).
#  fp32 state: |d| <= 1e-5 |ref| + 1e-6
#  fp16/bf16 state: one unit in the last place of the state dtype, plus the
#  fp32 tolerance (the recurrence itself runs in fp32)
#  outputs y (bf16/fp16): |d| <= 1e-2 |ref| + 1e-2
STATE_F32_RTOL, STATE_F32_ATOL = 1e-5, 1e-6
Y_RTOL, Y_ATOL = 1e-2, 1e-2


def oracle_tables(w: workloads.Workload):
    mode = oracle.SLOTS_PER_ROW if w.slot_mode == workloads.SLOTS_PER_ROW else oracle.SLOTS_STRIDED
    return oracle.Table.of(w.read, mode), oracle.Table.of(w.dst, mode)


def oracle_cu(w: workloads.Workload):
    if w.kind == "onetoken":
        return None
    if w.cu_seqlens is not None:
        return w.cu_seqlens
    return torch.arange(0, w.rows + 1, w.dense_steps, dtype=torch.int64)


def run_oracle(w: workloads.Workload, state_out=None, **over) -> oracle.Result:
    read, dst = oracle_tables(w)
    kw = dict(D=w.D, z=w.z, dt_bias=w.dt_bias, dt_softplus=w.dt_softplus, read=read, dst=dst,
              pad_slot_id=w.pad_slot_id, disable_state_update=w.disable_state_update,
              cu_seqlens=oracle_cu(w), num_accepted=w.num_accepted if w.kind == "packed" else None,
              state_out=state_out)
    kw.update(over)
    return oracle.ssu(w.state, w.x, w.dt, w.A, w.B, w.C, **kw)


def f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a float tensor (fp16/bf16/fp32 are exact in double)."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def ulp_of(v: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Spacing of the floating-point format at |v| (for fp16/bf16/fp32)."""
    fi = torch.finfo(dtype)
    frac = {torch.float16: 10, torch.bfloat16: 7, torch.float32: 23}[dtype]
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, fi.tiny)))
    e = np.maximum(e, np.log2(fi.tiny))
    return np.ldexp(1.0, (e - frac).astype(np.int64))


def assert_state_close(got: torch.Tensor, ref: torch.Tensor, what: str = "state"):
    """fp32: 1e-5 relative + 1e-6 absolute.  fp16/bf16: one ulp of the state
    dtype at the value's magnitude, on top of the fp32 tolerance: the
    recurrence is carried in fp32, so where cancellation makes a value tiny
    its own ulp is finer than fp32 arithmetic on O(1) operands resolves."""
    assert got.dtype == ref.dtype and got.shape == ref.shape
    g, r = f64(got), f64(ref)
    d = np.abs(g - r)
    if got.dtype == torch.float32:
        bad = d > STATE_F32_RTOL * np.abs(r) + STATE_F32_ATOL
    else:
        ulp = ulp_of(np.maximum(np.abs(g), np.abs(r)), got.dtype)
        bad = d > ulp * (1 + 1e-12) + STATE_F32_RTOL * np.abs(r) + STATE_F32_ATOL
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"first at {tuple(i)}: got {g[tuple(i)]!r} ref {r[tuple(i)]!r}")


def assert_y_close(got: torch.Tensor, ref_exact: torch.Tensor, what: str = "y"):
    g, r = f64(got), ref_exact.detach().to("cpu").numpy()
    d = np.abs(g - r)
    bad = d > Y_RTOL * np.abs(r) + Y_ATOL
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; first at "
                             f"{tuple(i)}: got {g[tuple(i)]!r} ref {r[tuple(i)]!r}")


def assert_e4m3_codes_close(got: torch.Tensor, want: torch.Tensor, values: torch.Tensor, what: str = "E4M3 codes"):
    """E4M3 read-copy codes (uint8, rows along the last axis) against the
    oracle's, which round v * 448 / amax, formed in double, to the nearest
    grid value.  The kernels form that quotient in fp32 (the factor 448 / amax
    and the product each rounded, together within 2^-22 relative of the exact
    quotient), so where the exact quotient lies within 2^-20 of the midpoint
    between two neighbouring grid values a code may sit one step away on the
    other side; everywhere else the codes must be equal."""
    got, want = got.cpu().view(torch.uint8), want.cpu().view(torch.uint8)
    assert got.shape == want.shape == values.shape
    diff = got != want
    if not diff.any():
        return
    vd = values.detach().cpu().to(torch.float64)
    amax = vd.abs().amax(dim=-1, keepdim=True)
    q = (vd * 448.0 / torch.where(amax > 0, amax, torch.ones_like(amax)))[diff]
    g, w = got[diff].to(torch.int64), want[diff].to(torch.int64)
    gm, wm = g & 0x7F, w & 0x7F
    grid = torch.arange(0, 128, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    mid = (grid[gm] + grid[wm]) / 2
    near = (q.abs() - mid).abs() <= 2.0 ** -20 * q.abs()
    ok = ((gm - wm).abs() == 1) & ((g & 0x80) == (w & 0x80)) & near
    if not ok.all():
        i = int(torch.nonzero(~ok)[0])
        raise AssertionError(f"{what}: {int((~ok).sum())} of {int(diff.sum())} differing codes are not one step "
                             f"apart at a tie; first: got {int(g[i]):#x} want {int(w[i]):#x} for v*448/amax = "
                             f"{float(q[i])!r}")
