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


_E2M1 = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _near_tie(q: torch.Tensor, a: torch.Tensor, b: torch.Tensor) -> torch.Tensor:
    """|q| within 2^-20 (relative) of the midpoint between grid values a, b."""
    mid = (a + b) / 2
    return (q.abs() - mid).abs() <= 2.0 ** -20 * q.abs()


def assert_nvfp4_close(got_codes: torch.Tensor, got_rec: torch.Tensor, values: torch.Tensor, what: str = "NVFP4"):
    """An NVFP4 read copy (code pairs [..., n/2], scale records) against the
    exact definition applied to `values` (rows along the last axis): the row
    scale amax / (6 * 448) in fp32 bit for bit; each block's E4M3 code the
    nearest to (block amax) / (6 s), or one step away where that quotient lies
    within 2^-20 of a midpoint (the kernels form it in fp32); each element's
    E2M1 code the nearest to v / (block scale * s) with the block scale the
    copy holds, or one step away at such a near-tie."""
    n = values.shape[-1]
    vd = values.detach().cpu().to(torch.float64).reshape(-1, n)
    rows = vd.shape[0]
    codes = got_codes.detach().cpu().view(torch.uint8).reshape(rows, n // 2)
    rec = got_rec.detach().cpu().reshape(rows, -1)
    amax = vd.abs().amax(dim=1)
    want_s = torch.where(amax > 0, amax / 2688.0, torch.ones_like(amax)).to(torch.float32)
    s = rec[:, 0]
    if not torch.equal(s, want_s):
        i = int(torch.nonzero(s != want_s)[0])
        raise AssertionError(f"{what}: row scale {float(s[i])!r}, want {float(want_s[i])!r}")
    sd = s.to(torch.float64)
    bcode = rec.view(torch.uint8)[:, 4:4 + n // 16].contiguous()
    bmax = vd.abs().view(rows, n // 16, 16).amax(dim=2)
    qb = bmax / (6.0 * sd[:, None])
    e4 = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    want_b = (qb.reshape(-1, 1) - e4.view(1, -1)).abs().argmin(dim=1).view(rows, n // 16)
    gb = bcode.to(torch.int64) & 0x7F
    if (gb > 126).any():
        raise AssertionError(f"{what}: a block code is E4M3 NaN")
    bad = (gb != want_b) & ~(((gb - want_b).abs() == 1) & _near_tie(qb, e4[gb], e4[want_b]))
    exact_tie = ((qb.reshape(-1, 1) - e4.view(1, -1)).abs() == (qb.reshape(-1, 1) - e4[want_b].reshape(-1, 1)).abs())
    bad &= ~(exact_tie.sum(dim=1).view(rows, n // 16) > 1)  # an exact tie: either neighbour, checked below
    if bad.any() or (bcode & 0x80).any():
        i = torch.nonzero(bad)[0].tolist() if bad.any() else [0, 0]
        raise AssertionError(f"{what}: block code {int(gb[i[0], i[1]])} at {i}, nearest {int(want_b[i[0], i[1]])}")
    bs = e4[gb].repeat_interleave(16, dim=1)
    den = bs * sd[:, None]
    q = torch.where(den > 0, vd / torch.where(den > 0, den, 1.0), torch.zeros_like(vd))
    grid = torch.tensor(_E2M1, dtype=torch.float64)
    c = torch.stack([codes & 15, codes >> 4], dim=-1).reshape(rows, n).to(torch.int64)
    mag = c & 7
    dist = (q.abs().clamp(max=6.0).unsqueeze(-1) - grid.view(1, 1, -1)).abs()
    best = dist.min(dim=-1).values
    ok_mag = (dist.gather(-1, mag.unsqueeze(-1)).squeeze(-1) == best)
    near = torch.zeros_like(ok_mag)
    for k in range(7):
        near |= ((mag == k) | (mag == k + 1)) & _near_tie(q, grid[k], grid[k + 1])
    sign_ok = (q == 0) | (((c >> 3) & 1).to(torch.bool) == torch.signbit(q)) | (mag == 0)
    bad = ~((ok_mag | near) & sign_ok)
    if bad.any():
        r, e = torch.nonzero(bad)[0].tolist()
        raise AssertionError(f"{what}: {int(bad.sum())} element codes off; first row {r} element {e}: code "
                             f"{int(c[r, e])} for v / (block scale * s) = {float(q[r, e])!r}")
