"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes a loaded oracle library (``lib``) and raises on a
mismatch, so the same pins run against the real oracle (test_oracle_pins.py)
and against deliberately broken copies of it (test_oracle_mutations.py).

What pins what:
  * closed forms of special cases (dt = 0, zero state, A = 0, x = 0, basis
    vectors for B and C), evaluated here with numpy from the decoded inputs;
  * the unrolled form of the recurrence given in the article "ReplaySSM:
    Cache SSM Inputs, Not State" (section 核心做法):
        S_h = gamma_{1:h} S_0 + sum_j gamma_{j+1:h} dt'_j x_j B_j,
    gamma_{i:h} = prod_{m=i..h} exp(A dt'_m), against the oracle's
    token-by-token loop;
  * worked examples computed by hand (values in the comments);
  * the slot effects of the call forms printed on the MATE "Mamba / SSU"
    page (tests/golden/page_examples.json);
  * invariants the page states: pad slots are never written,
    disable_state_update leaves the pool unchanged, flat and 2-D tables
    name the same entries for one sequence, empty sequences are skipped;
  * format conversions against fixed encodings and numpy / torch casts.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle
import workloads
from ssu_testlib import f64, run_oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
LN2 = math.log(2.0)


def _close(a, b, rtol=1e-12, atol=1e-12, what=""):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    if a.shape != b.shape or not np.all(np.abs(a - b) <= rtol * np.abs(b) + atol):
        d = np.max(np.abs(a - b)) if a.shape == b.shape else "shape"
        raise AssertionError(f"{what}: max abs diff {d}")


def _dt_eff(w: workloads.Workload) -> np.ndarray:
    """Processed step dt' as numpy float64 [rows, heads, dim]."""
    d = f64(w.dt)
    if d.ndim == 2:
        d = np.repeat(d[:, :, None], w.x.shape[2], axis=2)
    if w.dt_bias is not None:
        d = d + f64(w.dt_bias)[None, :, None]
    if w.dt_softplus:
        d = np.logaddexp(0.0, d)          # log(1 + e^d), numpy's routine
    return d


def _silu_np(z):
    return z * (1.0 / (1.0 + np.exp(-z)))


def _problem(seed, **kw):
    base = dict(slots=24, heads=4, dim=3, dstate=8, groups=2, nseq=3, max_len=3,
                state_dtype=torch.float64, io_dtype=torch.bfloat16, tables="distinct")
    base.update(kw)
    return workloads.random_problem(seed, **base)


# --------------------------------------------------------------------------
# Format conversions (used for every stored value).
# --------------------------------------------------------------------------
def pin_conversions(lib):
    enc, dec = oracle.encode, oracle.decode
    f16, bf16 = torch.float16, torch.bfloat16
    fixed = [
        (1.0, f16, 0x3C00), (-2.0, f16, 0xC000), (65504.0, f16, 0x7BFF),
        (2.0 ** -24, f16, 0x0001), (1 + 2.0 ** -11, f16, 0x3C00), (1 + 3 * 2.0 ** -11, f16, 0x3C02),
        (65520.0, f16, 0x7C00), (2.0 ** -25, f16, 0x0000), (3 * 2.0 ** -26, f16, 0x0001),
        (1.0, bf16, 0x3F80), (-0.5, bf16, 0xBF00), (1 + 2.0 ** -8, bf16, 0x3F80),
        (1 + 3 * 2.0 ** -8, bf16, 0x3F82), (2.0 ** -133, bf16, 0x0001),
    ]
    for v, dt, bits in fixed:
        got = enc(v, dt, lib=lib)
        if got != bits:
            raise AssertionError(f"encode({v!r}, {dt}) = {got:#06x}, expected {bits:#06x}")
    for bits, dt, v in [(0x3C00, f16, 1.0), (0x0001, f16, 2.0 ** -24), (0x7BFF, f16, 65504.0),
                        (0x3F80, bf16, 1.0), (0xC0A0, bf16, -5.0), (0x8001, f16, -(2.0 ** -24))]:
        if dec(bits, dt, lib=lib) != v:
            raise AssertionError(f"decode({bits:#06x}, {dt}) != {v}")
    rng = np.random.default_rng(7)
    vals = rng.standard_normal(4000) * np.exp(rng.uniform(-12, 10, 4000))
    ref16 = vals.astype(np.float16).view(np.uint16)          # numpy's direct double -> half
    for v, r in zip(vals, ref16):
        if enc(v, f16, lib=lib) != int(r):
            raise AssertionError(f"fp16 encode({v!r}) disagrees with numpy")
    vals32 = vals.astype(np.float32)                         # exact in double
    refbf = torch.from_numpy(vals32).to(bf16).view(torch.int16).numpy().view(np.uint16)
    for v, r in zip(vals32, refbf):
        if enc(float(v), bf16, lib=lib) != int(r):
            raise AssertionError(f"bf16 encode({v!r}) disagrees with torch")
    for v in vals[:500]:
        if oracle.decode(enc(v, torch.float32, lib=lib), torch.float32, lib=lib) != float(np.float32(v)):
            raise AssertionError("fp32 round trip")


# --------------------------------------------------------------------------
# Scalar functions.
# --------------------------------------------------------------------------
def pin_scalar_functions(lib):
    sp, si = (lambda v: oracle.softplus(v, lib=lib)), (lambda v: oracle.silu(v, lib=lib))
    _close(sp(0.0), LN2, what="softplus(0) = ln 2")
    for v in np.linspace(-30, 30, 121):
        _close(sp(v) - sp(-v), v, atol=1e-12, what="softplus(v) - softplus(-v) = v")
        _close(si(v) - si(-v), v, atol=1e-12, what="silu(v) - silu(-v) = v")
        _close(si(v) + si(-v), v * math.tanh(v / 2), atol=1e-12, what="silu(v) + silu(-v)")
    _close(sp(-40.0), math.exp(-40.0), rtol=1e-12, atol=0, what="softplus(-40) = e^-40")
    _close(sp(40.0), 40.0, rtol=1e-15, atol=0, what="softplus(40) = 40")
    _close(si(0.0), 0.0, what="silu(0) = 0")


# --------------------------------------------------------------------------
# Hand-worked examples (heads 1, dim 1, dstate 2, groups 1, fp64 state).
# --------------------------------------------------------------------------
def _hand(lib, *, S0, A, dt, x, B, C, D=None, z=None, bias=None, softplus=False, cu=None, acc=None):
    rows = len(x)
    st = torch.tensor(S0, dtype=torch.float64).view(1, 1, 1, 2)
    xs = torch.tensor(x, dtype=torch.float32).view(rows, 1, 1)
    dts = torch.tensor(dt, dtype=torch.float32).view(rows, 1, 1)
    Bs = torch.tensor(B, dtype=torch.float32).view(rows, 1, 2)
    Cs = torch.tensor(C, dtype=torch.float32).view(rows, 1, 2)
    zs = None if z is None else torch.tensor(z, dtype=torch.float32).view(rows, 1, 1)
    t = lambda v: None if v is None else torch.tensor([v], dtype=torch.float32)
    tab = torch.zeros(rows, dtype=torch.int64)
    read = oracle.Table(tab, 0, 0, oracle.SLOTS_STRIDED)
    r = oracle.ssu(st, xs, dts, t(A), Bs, Cs, D=t(D), z=zs, dt_bias=t(bias), dt_softplus=softplus,
                   read=read, cu_seqlens=None if cu is None else torch.tensor(cu),
                   num_accepted=None if acc is None else torch.tensor(acc), lib=lib)
    return r.y_exact.view(-1).numpy(), r.state.view(-1).numpy()


def pin_hand_worked(lib):
    # 1) A = 0 so dA = 1; dt' = 0.5; S0 = [1, 2], x = 2, B = [1, .5], C = [1, 1], D = .5
    #    S1 = [1 + .5*2*1, 2 + .5*2*.5] = [2, 2.5];  y = 2 + 2.5 + .5*2 = 5.5
    y, s = _hand(lib, S0=[1, 2], A=0.0, dt=[0.5], x=[2.0], B=[[1, .5]], C=[[1, 1]], D=0.5)
    _close(y, [5.5], what="hand 1 y")
    _close(s, [2.0, 2.5], what="hand 1 state")
    # 2) same with z = 2: y = 5.5 * 2 / (1 + e^-2)
    y, _ = _hand(lib, S0=[1, 2], A=0.0, dt=[0.5], x=[2.0], B=[[1, .5]], C=[[1, 1]], D=0.5, z=[2.0])
    _close(y, [5.5 * 2.0 / (1.0 + math.exp(-2.0))], what="hand 2 y (silu gate)")
    # 3) softplus on, dt + bias = 0 -> dt' = ln 2; A = -1 -> dA = 1/2.
    #    S0 = [4, -2], x = 1, B = [1, 1], C = [1, -1]:
    #    S1 = [2 + ln2, -1 + ln2]; y = S1[0] - S1[1] = 3.
    y, s = _hand(lib, S0=[4, -2], A=-1.0, dt=[0.75], bias=-0.75, x=[1.0], B=[[1, 1]], C=[[1, -1]],
                 softplus=True)
    _close(y, [3.0], what="hand 3 y")
    _close(s, [2 + LN2, -1 + LN2], what="hand 3 state")
    # 4) two tokens of one sequence, dt' = ln 2 each (dt = 0, softplus), A = -1, D = 0.5.
    #    token 1: x = 2, B = [1, 0], C = [0, 1] -> S1 = [.5 + 2 ln2, 1], y1 = 1 + .5*2 = 2
    #    token 2: x = -1, B = [0, 1], C = [1, 0] -> S2 = [.25 + ln2, .5 - ln2],
    #             y2 = .25 + ln2 - .5 = ln2 - .25
    #    both tokens publish to slot 0 (no destination table, read table [0, 0]);
    #    the last one wins.
    y, s = _hand(lib, S0=[1, 2], A=-1.0, dt=[0.0, 0.0], x=[2.0, -1.0], B=[[1, 0], [0, 1]],
                 C=[[0, 1], [1, 0]], D=0.5, softplus=True, cu=[0, 2])
    _close(y, [2.0, LN2 - 0.25], what="hand 4 y")
    _close(s, [0.25 + LN2, 0.5 - LN2], what="hand 4 state")


# --------------------------------------------------------------------------
# Closed forms on random data.
# --------------------------------------------------------------------------
def _seed_state(w, res_touched=None):
    """Seed state per sequence as numpy [nseq, heads, dim, dstate] (zeros for pad/no seed)."""
    st = f64(w.state)
    out = np.zeros((w.nseq,) + st.shape[1:])
    lens = w.meta["lengths"]
    cu = np.concatenate([[0], np.cumsum(lens)])
    for b in range(w.nseq):
        if lens[b] == 0:
            continue
        t = 0
        if w.kind == "packed" and w.num_accepted is not None:
            t = max(int(w.num_accepted[b]) - 1, 0)
        if w.read is None:
            s = b
        elif w.slot_mode == workloads.SLOTS_PER_ROW:
            s = int(w.read.reshape(-1)[cu[b] + t])
        elif w.read.dim() == 1:
            s = int(w.read[b + t])
        else:
            s = int(w.read[b, t])
        if s != w.pad_slot_id:
            out[b] = st[s]
    return out


def _groups_of(w):
    H, G = w.x.shape[1], w.B.shape[1]
    return np.arange(H) // (H // G)


def pin_dt_zero(lib):
    """dt' = 0 (dt = 0, no bias, softplus off): dA = 1 and no input term, so the
    published state is bit-identical to the seed and y = S.C + D x (x silu(z))."""
    for sd in (torch.float64, torch.float32, torch.float16, torch.bfloat16):
        w = _problem(11, state_dtype=sd, dt_softplus=False, with_bias=False, kind="onetoken",
                     tables="distinct", pad_frac=0.0)
        w.dt.zero_()
        r = run_oracle(w, lib=lib)
        g = _groups_of(w)
        Cn, xn, zn = f64(w.C), f64(w.x), f64(w.z)
        S = _seed_state(w)
        y = np.einsum("bhpn,bhn->bhp", S, Cn[:, g, :]) + f64(w.D)[None, :, None] * xn
        y = y * _silu_np(zn)
        _close(r.y_exact.numpy(), y, rtol=1e-12, atol=1e-12, what=f"dt=0 y ({sd})")
        for b in range(w.nseq):
            s_in, s_out = int(w.read[b]), int(w.dst[b])
            if not torch.equal(r.state[s_out], w.state[s_in]):
                raise AssertionError(f"dt=0 must leave the state bit-unchanged ({sd})")


def pin_zero_state(lib):
    """Zero seed (pad read): after one token S = dt' x B, so
    y = dt' (B.C) x + D x, then times silu(z)."""
    w = _problem(12, kind="onetoken", tables="distinct", pad_frac=0.0)
    w.read[:] = w.pad_slot_id
    r = run_oracle(w, lib=lib)
    g = _groups_of(w)
    d, xn = _dt_eff(w), f64(w.x)
    BC = np.einsum("bhn,bhn->bh", f64(w.B)[:, g, :], f64(w.C)[:, g, :])
    y = (d * BC[:, :, None] * xn + f64(w.D)[None, :, None] * xn) * _silu_np(f64(w.z))
    _close(r.y_exact.numpy(), y, rtol=1e-11, atol=1e-12, what="zero-state y")
    for b in range(w.nseq):
        S = d[b][:, :, None] * xn[b][:, :, None] * f64(w.B)[b, g][:, None, :]
        _close(f64(r.state[int(w.dst[b])]), S, rtol=1e-12, atol=1e-14, what="zero-state state")


def pin_A_zero(lib):
    """A = 0: dA = 1, S' = S + dt' x B."""
    w = _problem(13, kind="onetoken", tables="inplace", pad_frac=0.0)
    w.A.zero_()
    r = run_oracle(w, lib=lib)
    g = _groups_of(w)
    S = _seed_state(w)
    d, xn, Bn = _dt_eff(w), f64(w.x), f64(w.B)
    for b in range(w.nseq):
        ref = S[b] + (d[b] * xn[b])[:, :, None] * Bn[b, g][:, None, :]
        _close(f64(r.state[int(w.dst[b])]), ref, rtol=1e-12, atol=1e-14, what="A=0 state")


def pin_decay_only(lib):
    """x = 0 over several tokens: S_T = exp(A * sum_t dt'_t) S_0 and
    y_t = S_t . C_t (the D x term vanishes)."""
    w = _problem(14, kind="packed", tables="distinct", pad_frac=0.0, max_len=4, allow_empty=False,
                 with_z=False, nseq=3)
    w.x.zero_()
    r = run_oracle(w, lib=lib)
    A, d, g = f64(w.A), _dt_eff(w), _groups_of(w)
    S0 = _seed_state(w)
    cu = np.concatenate([[0], np.cumsum(w.meta["lengths"])])
    for b in range(w.nseq):
        acc_d = np.zeros(d.shape[1:])
        for t, row in enumerate(range(cu[b], cu[b + 1])):
            acc_d = acc_d + d[row]
            St = np.exp(A[:, None] * acc_d)[:, :, None] * S0[b]
            yt = np.einsum("hpn,hn->hp", St, f64(w.C)[row, g])
            _close(r.y_exact[row].numpy(), yt, rtol=1e-11, atol=1e-13, what="decay-only y")
        last = int(w.dst[b, w.meta["lengths"][b] - 1])
        _close(f64(r.state[last]), St, rtol=1e-11, atol=1e-14, what="decay-only state")


def pin_unrolled(lib):
    """Multi-token recurrence against its unrolled form (ReplaySSM, 核心做法):
    S_h = gamma_{1:h} S_0 + sum_{j<=h} gamma_{j+1:h} dt'_j x_j B_j,  with
    gamma_{i:h} = prod_{m=i..h} exp(A dt'_m); y_h = S_h . C_h + D x_h, gated."""
    for sd in (torch.float64,):
        w = _problem(15, kind="packed", tables="distinct", pad_frac=0.0, max_len=5, nseq=3,
                     allow_empty=False, state_dtype=sd, heads=4, groups=2, dim=3, dstate=8,
                     slots=40)
        r = run_oracle(w, lib=lib)
        A, d, g = f64(w.A), _dt_eff(w), _groups_of(w)
        xn, Bn, Cn, Dn, zn = f64(w.x), f64(w.B), f64(w.C), f64(w.D), f64(w.z)
        S0 = _seed_state(w)
        cu = np.concatenate([[0], np.cumsum(w.meta["lengths"])])
        for b in range(w.nseq):
            rows = list(range(cu[b], cu[b + 1]))
            alpha = [np.exp(A[:, None] * d[r_]) for r_ in rows]      # [heads, dim] each
            for hidx in range(len(rows)):
                gam = np.ones_like(alpha[0])
                for m in range(0, hidx + 1):
                    gam = gam * alpha[m]
                S = gam[:, :, None] * S0[b]
                for j in range(hidx + 1):
                    gj = np.ones_like(alpha[0])
                    for m in range(j + 1, hidx + 1):
                        gj = gj * alpha[m]
                    rj = rows[j]
                    S = S + (gj * d[rj] * xn[rj])[:, :, None] * Bn[rj, g][:, None, :]
                rh = rows[hidx]
                y = np.einsum("hpn,hn->hp", S, Cn[rh, g]) + Dn[:, None] * xn[rh]
                y = y * _silu_np(zn[rh])
                _close(r.y_exact[rh].numpy(), y, rtol=1e-11, atol=1e-12, what="unrolled y")
                _close(f64(r.state[int(w.dst[b, hidx])]), S, rtol=1e-11, atol=1e-13,
                       what="unrolled state")


def pin_basis_vectors(lib):
    """B = e_j and C = e_k with j != k: only column j receives the input, and
    y reads column k of the updated state."""
    w = _problem(16, kind="onetoken", tables="distinct", pad_frac=0.0, with_z=False, groups=1)
    j, k = 2, 5
    w.B.zero_()
    w.C.zero_()
    w.B[:, :, j] = 1
    w.C[:, :, k] = 1
    r = run_oracle(w, lib=lib)
    A, d, xn = f64(w.A), _dt_eff(w), f64(w.x)
    S0 = _seed_state(w)
    for b in range(w.nseq):
        dA = np.exp(A[:, None] * d[b])
        ref = dA[:, :, None] * S0[b]
        ref[:, :, j] += d[b] * xn[b]
        _close(f64(r.state[int(w.dst[b])]), ref, rtol=1e-12, atol=1e-14, what="basis state")
        _close(r.y_exact[b].numpy(), ref[:, :, k] + f64(w.D)[:, None] * xn[b], what="basis y")


def pin_group_map(lib):
    """Convention (not fixed by the pages): head h uses group h // (heads/groups).
    With B, C non-zero only in group 1 of 2, heads 2 and 3 of 4 get the input
    term, heads 0 and 1 only decay."""
    w = _problem(17, kind="onetoken", tables="distinct", pad_frac=0.0, heads=4, groups=2,
                 with_z=False, with_D=False)
    w.B[:, 0, :] = 0
    w.C[:, 0, :] = 0
    r = run_oracle(w, lib=lib)
    A, d = f64(w.A), _dt_eff(w)
    S0 = _seed_state(w)
    for b in range(w.nseq):
        out = f64(r.state[int(w.dst[b])])
        dA = np.exp(A[:, None] * d[b])
        _close(out[:2], dA[:2, :, None] * S0[b][:2], what="group 0 heads only decay")
        if np.allclose(out[2:], dA[2:, :, None] * S0[b][2:]):
            raise AssertionError("group 1 heads received no input")
        _close(r.y_exact[b, :2].numpy(), np.zeros((2, w.x.shape[2])), what="group 0 y")


# --------------------------------------------------------------------------
# Slot semantics.
# --------------------------------------------------------------------------
def _golden():
    with open(os.path.join(GOLDEN, "page_examples.json")) as f:
        return json.load(f)


def _page_problem(ex, heads=2, dim=2, dstate=4, groups=1, seed=21):
    rows = ex.get("rows") or (ex["batch"] * ex.get("steps", 1))
    g = torch.Generator().manual_seed(seed)
    state = (torch.randn((ex["slots"], heads, dim, dstate), generator=g, dtype=torch.float64) * 0.5)
    x = torch.randn((rows, heads, dim), generator=g).to(torch.bfloat16)
    dt = torch.rand((rows, heads, dim), generator=g) * 0.2
    A = -torch.rand(heads, generator=g)
    B = torch.randn((rows, groups, dstate), generator=g).to(torch.bfloat16)
    C = torch.randn((rows, groups, dstate), generator=g).to(torch.bfloat16)
    return state, x, dt, A, B, C


def _touched(res, bit):
    return sorted(int(i) for i in torch.nonzero(res.touched & bit).view(-1))


def pin_page_examples(lib):
    gold = _golden()
    # minimal one-token example
    ex = gold["minimal_onetoken"]
    state, x, dt, A, B, C = _page_problem(ex)
    tab = torch.tensor(ex["read"])
    res = oracle.ssu(state, x, dt, A, B, C, read=oracle.Table.of(tab), dst=oracle.Table.of(tab),
                     pad_slot_id=ex["pad_slot_id"], lib=lib)
    if _touched(res, oracle.TOUCH_READ) != ex["expect_seed_slots"]:
        raise AssertionError("minimal example: seed slots")
    if _touched(res, oracle.TOUCH_WRITTEN) != ex["expect_written_slots"]:
        raise AssertionError("minimal example: written slots")
    for s in ex["expect_untouched_slots"]:
        if not torch.equal(res.state[s], state[s]):
            raise AssertionError("minimal example: untouched slot changed")
    # 2-D MTP example
    ex = gold["mtp_2d"]
    state, x, dt, A, B, C = _page_problem(ex)
    read, dst = torch.tensor(ex["read"]), torch.tensor(ex["dst"])
    res = oracle.ssu(state, x, dt, A, B, C, read=oracle.Table.of(read), dst=oracle.Table.of(dst),
                     pad_slot_id=ex["pad_slot_id"], cu_seqlens=torch.tensor(ex["cu_seqlens"]),
                     num_accepted=torch.tensor(ex["num_accepted"]), lib=lib)
    if _touched(res, oracle.TOUCH_READ) != ex["expect_seed_slots"]:
        raise AssertionError(f"MTP example: seed slots {_touched(res, oracle.TOUCH_READ)}")
    if _touched(res, oracle.TOUCH_WRITTEN) != ex["expect_written_slots"]:
        raise AssertionError("MTP example: written slots")
    for s in range(14):
        if not torch.equal(res.state[s], state[s]):
            raise AssertionError("MTP example: a read-side slot changed")
    # flat table, one sequence; also the same call with the table as [1, rows]
    ex = gold["flat_one_sequence"]
    state, x, dt, A, B, C = _page_problem(ex)
    tab = torch.tensor(ex["read"])
    common = dict(pad_slot_id=ex["pad_slot_id"], cu_seqlens=torch.tensor(ex["cu_seqlens"]),
                  num_accepted=torch.tensor(ex["num_accepted"]), lib=lib)
    flat = oracle.ssu(state, x, dt, A, B, C, read=oracle.Table.of(tab), dst=oracle.Table.of(tab), **common)
    two_d = oracle.ssu(state, x, dt, A, B, C, read=oracle.Table.of(tab.view(1, -1)),
                       dst=oracle.Table.of(tab.view(1, -1)), **common)
    per_row = oracle.ssu(state, x, dt, A, B, C, read=oracle.Table.of(tab, oracle.SLOTS_PER_ROW),
                         dst=oracle.Table.of(tab, oracle.SLOTS_PER_ROW), **common)
    if _touched(flat, oracle.TOUCH_READ) != []:
        raise AssertionError("flat example: the seed is the pad slot and must not count as read")
    if _touched(flat, oracle.TOUCH_WRITTEN) != ex["expect_written_slots"]:
        raise AssertionError("flat example: written slots")
    if not torch.equal(flat.state[0], state[0]):
        raise AssertionError("flat example: pad slot 0 was written")
    for other in (two_d, per_row):
        if not (torch.equal(other.state, flat.state) and torch.equal(other.y_exact, flat.y_exact)):
            raise AssertionError("flat, 2-D and per-row tables must name the same entries")
    # the seed is the pad: token 0 starts from zero, so y_0 = dt'_0 x_0 (B_0 . C_0)
    bc = float(np.dot(f64(B)[0, 0], f64(C)[0, 0]))
    _close(flat.y_exact[0].numpy(), f64(dt)[0] * f64(x)[0] * bc, rtol=1e-12, atol=1e-15,
           what="flat example: zero seed")


def pin_pad_never_written(lib):
    """pad_slot_id = 0, a real slot full of data: it must stay byte-identical,
    and a pad read must equal a read of an all-zero slot."""
    w = _problem(31, kind="packed", tables="distinct", pad_slot_id=0, pad_frac=0.3,
                 slot_mode=workloads.SLOTS_STRIDED, nseq=4, max_len=3, slots=40)
    r = run_oracle(w, lib=lib)
    if not torch.equal(r.state[0], w.state[0]):
        raise AssertionError("pad slot was written")
    zeroed = w.state.clone()
    zeroed[0] = 0
    r2 = run_oracle(workloads.replace(w, state=zeroed), lib=lib)
    if not torch.equal(r2.y_exact, r.y_exact):
        raise AssertionError("a pad read is not a zero state")


def pin_disable_and_untouched(lib):
    """disable_state_update leaves the pool bit-identical and changes no y;
    slots that are not written keep their bytes."""
    w = _problem(32, kind="packed", tables="distinct", nseq=4, max_len=3, slots=40,
                 state_dtype=torch.bfloat16)
    r = run_oracle(w, lib=lib)
    written = set(_touched(r, oracle.TOUCH_WRITTEN))
    for s in range(w.state.shape[0]):
        if s not in written and not torch.equal(r.state[s], w.state[s]):
            raise AssertionError(f"untouched slot {s} changed")
    rd = run_oracle(workloads.replace(w, disable_state_update=True), lib=lib)
    if not torch.equal(rd.state, w.state):
        raise AssertionError("disable_state_update changed the pool")
    if not torch.equal(rd.y_exact, r.y_exact):
        raise AssertionError("disable_state_update changed y")


def pin_table_forms(lib):
    """No table == identity table; no destination table == destination equal to
    the read table; one-token == packed with every length 1."""
    w = _problem(33, kind="onetoken", tables="none", nseq=5, slots=5)
    ident = torch.arange(5, dtype=torch.int32)
    a = run_oracle(w, lib=lib)
    b = run_oracle(workloads.replace(w, read=ident, dst=ident.clone()), lib=lib)
    if not (torch.equal(a.state, b.state) and torch.equal(a.y_exact, b.y_exact)):
        raise AssertionError("no table != identity table")
    w = _problem(34, kind="packed", tables="read", nseq=3, max_len=3, slots=20)
    a = run_oracle(w, lib=lib)
    b = run_oracle(workloads.replace(w, dst=w.read.clone()), lib=lib)
    if not (torch.equal(a.state, b.state) and torch.equal(a.y_exact, b.y_exact)):
        raise AssertionError("absent destination table != destination = read table")
    w = _problem(35, kind="onetoken", tables="distinct", nseq=4, slots=20)
    a = run_oracle(w, lib=lib)
    cu = torch.arange(0, 5, dtype=torch.int32)
    b = run_oracle(workloads.replace(w, kind="packed", cu_seqlens=cu, read=w.read.view(4, 1),
                                     dst=w.dst.view(4, 1), meta={"lengths": [1] * 4}), lib=lib)
    if not (torch.equal(a.state, b.state) and torch.equal(a.y_exact, b.y_exact)):
        raise AssertionError("one-token != packed with lengths 1")


def pin_seed_position(lib):
    """The read slot is table[b, max(num_accepted - 1, 0)].  Slot s holds the
    constant s + 1, dt' = 0 and x = 0, so y = (s + 1) * sum(C) names s."""
    nseq, steps, slots = 4, 4, 16
    state = torch.arange(1, slots + 1, dtype=torch.float64).view(slots, 1, 1, 1).repeat(1, 1, 1, 2)
    read = torch.arange(nseq * steps).view(nseq, steps)
    rows = nseq * steps
    x = torch.zeros((rows, 1, 1))
    dt = torch.zeros((rows, 1, 1))
    B = torch.zeros((rows, 1, 2))
    C = torch.ones((rows, 1, 2))
    for acc, t_seed in (([0, 1, 2, 4], [0, 0, 1, 3]), ([3, 3, 1, 2], [2, 2, 0, 1])):
        res = oracle.ssu(state, x, dt, torch.zeros(1), B, C, read=oracle.Table.of(read),
                         dst=oracle.Table.of(read + 0), cu_seqlens=torch.arange(0, rows + 1, steps),
                         num_accepted=torch.tensor(acc), lib=lib)
        for b in range(nseq):
            expect = 2.0 * (read[b, t_seed[b]] + 1)
            if res.y_exact[b * steps, 0, 0] != expect:
                raise AssertionError(f"seed of sequence {b} with num_accepted {acc[b]}")


def pin_seed_position_per_row(lib):
    """PER_ROW addressing: sequence b's step t uses flat entry cu_seqlens[b] + t.
    Lengths [2, 0, 3, 1] give cu_seqlens [0, 2, 2, 5, 6]; with num_accepted
    [2, 1, 1, 1] the seeds are entries 1, -, 2, 5 (worked by hand)."""
    slots, rows = 12, 6
    state = torch.arange(1, slots + 1, dtype=torch.float64).view(slots, 1, 1, 1).repeat(1, 1, 1, 2)
    tab = torch.tensor([7, 3, 9, 4, 10, 2])           # entry -> slot
    cu = torch.tensor([0, 2, 2, 5, 6])
    x, dt, B = torch.zeros((rows, 1, 1)), torch.zeros((rows, 1, 1)), torch.zeros((rows, 1, 2))
    C = torch.ones((rows, 1, 2))
    res = oracle.ssu(state, x, dt, torch.zeros(1), B, C,
                     read=oracle.Table.of(tab, oracle.SLOTS_PER_ROW), cu_seqlens=cu,
                     num_accepted=torch.tensor([2, 1, 1, 1]), lib=lib)
    for row, seed_entry in ((0, 1), (2, 2), (5, 5)):
        if res.y_exact[row, 0, 0] != 2.0 * (int(tab[seed_entry]) + 1):
            raise AssertionError(f"per-row seed of the sequence starting at row {row}")
    if _touched(res, oracle.TOUCH_WRITTEN) != sorted(tab.tolist()):
        raise AssertionError("per-row: every row publishes to its own entry")
    # num_accepted past a sequence's length would seed from the next
    # sequence's entry (sequence 0: entry 2 belongs to sequence 2): refused
    for acc in ([3, 1, 1, 1], [2, 1, 4, 1], [2, 1, 1, 2]):
        try:
            oracle.ssu(state, x, dt, torch.zeros(1), B, C, read=oracle.Table.of(tab, oracle.SLOTS_PER_ROW),
                       cu_seqlens=cu, num_accepted=torch.tensor(acc), lib=lib)
        except oracle.OracleError as e:
            if e.code != oracle.INVALID:
                raise
        else:
            raise AssertionError(f"per-row seed past the sequence accepted (num_accepted {acc})")


def pin_per_head_dt(lib):
    """A per-head step dt [rows, heads] is the full [rows, heads, dim] step with
    each head's value repeated over dim."""
    w = _problem(39, kind="packed", tables="distinct", nseq=3, max_len=3, slots=40, per_head_dt=True)
    full = w.dt[:, :, None].expand(-1, -1, w.x.shape[2]).contiguous()
    a = run_oracle(w, lib=lib)
    b = run_oracle(workloads.replace(w, dt=full), lib=lib)
    if not (torch.equal(a.state, b.state) and torch.equal(a.y_exact, b.y_exact)):
        raise AssertionError("per-head dt differs from the broadcast full dt")
    if torch.equal(w.dt[:, 0], w.dt[:, 1]):
        raise AssertionError("test needs distinct per-head steps")


def pin_aliasing_refused(lib):
    """Cross-sequence aliasing has no deterministic answer and is refused;
    a sequence reading its own later destination is fine."""
    w = _problem(36, kind="packed", tables="distinct", pad_frac=0.0, nseq=3, max_len=2,
                 allow_empty=False, slots=20)
    bad = w.dst.clone()
    bad[1, 0] = bad[0, 0]
    try:
        run_oracle(workloads.replace(w, dst=bad), lib=lib)
        raise AssertionError("write-write collision accepted")
    except oracle.OracleError as e:
        if e.code != oracle.ALIASING:
            raise
    bad = w.dst.clone()
    t0 = max(int(w.num_accepted[0]) - 1, 0)
    bad[1, 0] = w.read[0, t0]
    try:
        run_oracle(workloads.replace(w, dst=bad), lib=lib)
        raise AssertionError("overwritten seed accepted")
    except oracle.OracleError as e:
        if e.code != oracle.ALIASING:
            raise
    # the same tables are fine when nothing is written
    run_oracle(workloads.replace(w, dst=bad, disable_state_update=True), lib=lib)
    ok = w.dst.clone()
    ok[0, 0] = w.read[0, t0]      # sequence 0 overwrites its own seed
    run_oracle(workloads.replace(w, dst=ok), lib=lib)


def pin_empty_sequences(lib):
    """Empty sequences are skipped: nothing read, nothing written."""
    w = _problem(37, kind="packed", tables="distinct", pad_frac=0.0, nseq=6, max_len=2, slots=40)
    lens = w.meta["lengths"]
    assert 0 in lens
    r = run_oracle(w, lib=lib)
    for b, L in enumerate(lens):
        if L == 0:
            for s in w.dst[b].tolist() + w.read[b].tolist():
                if r.touched[s] != 0:
                    raise AssertionError("an empty sequence touched a slot")


def pin_bounded_decay(lib):
    """A < 0 and dt' >= 0 give 0 < dA <= 1, so |S'| <= |S| + |dt' x B|."""
    w = _problem(38, kind="onetoken", tables="distinct", pad_frac=0.0)
    r = run_oracle(w, lib=lib)
    g = _groups_of(w)
    S0, d, xn, Bn = _seed_state(w), _dt_eff(w), f64(w.x), f64(w.B)
    for b in range(w.nseq):
        bound = np.abs(S0[b]) + np.abs((d[b] * xn[b])[:, :, None] * Bn[b, g][:, None, :])
        if np.any(np.abs(f64(r.state[int(w.dst[b])])) > bound * (1 + 1e-12) + 1e-300):
            raise AssertionError("decay bound violated")


# --------------------------------------------------------------------------
# ReplaySSM decode step (article "ReplaySSM: Cache SSM Inputs, Not State",
# section 核心做法): checkpoint + buffer of the inputs since the last fold.
# --------------------------------------------------------------------------
def _replay_scenario(seed, L, counts, heads=4, dim=3, dstate=8, groups=2, io=torch.bfloat16,
                     state_dtype=torch.float64, with_z=True, pad_last=False):
    """Sequences b with counts[b] buffered steps each, built from explicit
    token histories; returns the replay inputs and, per sequence, the plain
    token-by-token history to compare with."""
    g = torch.Generator().manual_seed(seed)
    nseq = len(counts)
    slots = 2 * nseq + 3
    slot_of = torch.randperm(slots, generator=g)[:nseq]
    if pad_last:
        slot_of[-1] = -1
    ckpt = (torch.randn((slots, heads, dim, dstate), generator=g, dtype=torch.float64) * 0.5).to(state_dtype)
    xbuf = torch.randn((slots, L, heads, dim), generator=g).to(io)
    dtbuf = torch.rand((slots, L, heads, dim), generator=g) * 0.3
    Bbuf = torch.randn((slots, L, groups, dstate), generator=g).to(io)
    x = torch.randn((nseq, heads, dim), generator=g).to(io)
    dt = torch.rand((nseq, heads, dim), generator=g) * 0.3
    B = torch.randn((nseq, groups, dstate), generator=g).to(io)
    C = torch.randn((nseq, groups, dstate), generator=g).to(io)
    z = torch.randn((nseq, heads, dim), generator=g).to(io) if with_z else None
    A = -torch.exp(torch.rand(heads, generator=g) * 2.0)
    D = torch.randn(heads, generator=g)
    count = torch.tensor(counts, dtype=torch.int64)
    return dict(ckpt=ckpt, x=x, dt=dt, A=A, B=B, C=C, xbuf=xbuf, dtbuf=dtbuf, Bbuf=Bbuf, count=count,
                D=D, z=z, slot_of=slot_of)


def _plain_history(sc, b, lib):
    """The same sequence run token by token by the plain update: buffered
    entries first (their processed steps as dt, softplus off), then the
    current token; all tokens publish to the sequence's slot."""
    s = int(sc["slot_of"][b])
    c = int(sc["count"][b])
    xs = torch.cat([sc["xbuf"][s, :c], sc["x"][b:b + 1]])
    dts = torch.cat([sc["dtbuf"][s, :c], sc["dt"][b:b + 1]])
    Bs = torch.cat([sc["Bbuf"][s, :c], sc["B"][b:b + 1]])
    Cs = torch.cat([sc["C"][b:b + 1].expand(c, -1, -1), sc["C"][b:b + 1]])
    zs = None if sc["z"] is None else torch.cat([sc["z"][b:b + 1].expand(c, -1, -1), sc["z"][b:b + 1]])
    tab = torch.full((1, c + 1), s, dtype=torch.int64)
    return oracle.ssu(sc["ckpt"], xs, dts, sc["A"], Bs, Cs, D=sc["D"], z=zs, read=oracle.Table.of(tab),
                      cu_seqlens=torch.tensor([0, c + 1]), lib=lib)


def _run_replay(sc, lib, **kw):
    return oracle.replay(sc["ckpt"], sc["x"], sc["dt"], sc["A"], sc["B"], sc["C"], sc["xbuf"], sc["dtbuf"],
                         sc["Bbuf"], sc["count"], D=sc["D"], z=sc["z"], slot_of=sc["slot_of"], lib=lib, **kw)


def pin_replay_lossless(lib):
    """The method is lossless: y from checkpoint + buffer equals the plain
    recurrence run over the buffered steps and the current one, and a fold
    leaves in the checkpoint the state the plain recurrence reaches."""
    L = 5
    counts = [0, 1, 2, 3, 4, 4, 2]
    sc = _replay_scenario(41, L, counts)
    r = _run_replay(sc, lib)
    for b, c in enumerate(counts):
        h = _plain_history(sc, b, lib)
        _close(r.y_exact[b].numpy(), h.y_exact[c].numpy(), rtol=1e-11, atol=1e-12, what=f"replay y (c={c})")
        s = int(sc["slot_of"][b])
        if c + 1 == L:
            _close(f64(r.ckpt[s]), f64(h.state[s]), rtol=1e-11, atol=1e-13, what="folded checkpoint")
            if int(r.count[b]) != 0:
                raise AssertionError("a fold must empty the buffer")
        else:
            if not torch.equal(r.ckpt[s], sc["ckpt"][s]):
                raise AssertionError("a step that does not fold must not write the checkpoint")
            if int(r.count[b]) != c + 1:
                raise AssertionError("a step that does not fold buffers one more entry")


def pin_replay_buffer_entries(lib):
    """A step that does not fold appends the current token as entry c: x and
    B with their bits, the processed step dt' (softplus(dt + bias)) in fp32;
    older entries and other slots are untouched."""
    L = 4
    counts = [0, 2, 1]
    sc = _replay_scenario(42, L, counts)
    bias = torch.full((sc["x"].shape[1],), -0.5)
    r = _run_replay(sc, lib, dt_bias=bias, dt_softplus=True)
    groups = sc["B"].shape[1]
    for b, c in enumerate(counts):
        s = int(sc["slot_of"][b])
        if not torch.equal(r.xbuf[s, c], sc["x"][b]):
            raise AssertionError("appended x")
        if not torch.equal(r.Bbuf[s, c], sc["B"][b]):
            raise AssertionError("appended B")
        d = np.logaddexp(0.0, f64(sc["dt"][b]) + f64(bias)[:, None])
        _close(r.dtbuf[s, c].double().numpy(), d, rtol=1e-7, atol=1e-9, what="appended processed step")
        if not (torch.equal(r.xbuf[s, :c], sc["xbuf"][s, :c]) and torch.equal(r.dtbuf[s, :c], sc["dtbuf"][s, :c])):
            raise AssertionError("older entries changed")
        assert groups == r.Bbuf.shape[2]
    used = set(int(v) for v in sc["slot_of"])
    for s in range(sc["ckpt"].shape[0]):
        if s not in used and not (torch.equal(r.xbuf[s], sc["xbuf"][s]) and torch.equal(r.ckpt[s], sc["ckpt"][s])):
            raise AssertionError("a slot no sequence uses changed")


def pin_replay_buffer_len_one(lib):
    """L = 1: the buffer is always empty, every step folds, and the step is
    the plain update (the article's bit-for-bit anchor)."""
    sc = _replay_scenario(43, 1, [0, 0, 0], state_dtype=torch.float32)
    bias = torch.full((sc["x"].shape[1],), -1.0)
    r = _run_replay(sc, lib, dt_bias=bias, dt_softplus=True)
    plain = oracle.ssu(sc["ckpt"], sc["x"], sc["dt"], sc["A"], sc["B"], sc["C"], D=sc["D"], z=sc["z"],
                       dt_bias=bias, dt_softplus=True, read=oracle.Table.of(sc["slot_of"]), lib=lib)
    if not (torch.equal(r.y_exact, plain.y_exact) and torch.equal(r.ckpt, plain.state)):
        raise AssertionError("L = 1 differs from the plain update")
    if torch.any(r.count != 0):
        raise AssertionError("L = 1 leaves entries in the buffer")


def pin_replay_pad_and_aliasing(lib):
    """A pad slot has no history: y is the zero-state closed form and nothing
    is written; two sequences on one slot are refused."""
    sc = _replay_scenario(44, 3, [1, 2], with_z=False, pad_last=True)
    r = _run_replay(sc, lib)
    b = 1
    gi = np.arange(sc["x"].shape[1]) // (sc["x"].shape[1] // sc["B"].shape[1])
    d, xn = f64(sc["dt"][b]), f64(sc["x"][b])
    bc = np.einsum("hn,hn->h", f64(sc["B"][b])[gi], f64(sc["C"][b])[gi])
    _close(r.y_exact[b].numpy(), d * bc[:, None] * xn + f64(sc["D"])[:, None] * xn, what="pad replay y")
    if not torch.equal(r.ckpt, sc["ckpt"]) or int(r.count[b]) != 0:
        raise AssertionError("pad bookkeeping: nothing is written and no entry is kept")
    sc2 = _replay_scenario(45, 3, [1, 1])
    sc2["slot_of"][1] = sc2["slot_of"][0]
    try:
        _run_replay(sc2, lib)
        raise AssertionError("two sequences on one slot accepted")
    except oracle.OracleError as e:
        if e.code != oracle.ALIASING:
            raise


def pin_e4m3_codes(lib):
    """OCP FP8 E4M3 as the read copy stores it: every finite code decodes and
    re-encodes to itself; random values (normal, subnormal, ties) encode as
    torch's float8_e4m3fn cast does; past 448 the encoder clamps to +-448;
    NaN keeps the NaN code."""
    for code in range(256):
        v = lib.orc_e4m3_decode(code)
        if (code & 0x7f) == 0x7f:
            if not np.isnan(v):
                raise AssertionError("E4M3 NaN code")
            continue
        if lib.orc_e4m3_encode(v) != code and not (v == 0.0 and code == 0x80 and lib.orc_e4m3_encode(v) == 0):
            if not (code == 0x80 and lib.orc_e4m3_encode(-0.0) == 0x80):
                raise AssertionError(f"E4M3 code {code:#x} does not round-trip")
    g = torch.Generator().manual_seed(61)
    vals = torch.cat([(torch.rand(4000, generator=g) - 0.5) * 900, (torch.rand(2000, generator=g) - 0.5) * 0.03,
                      torch.tensor([2.0 ** -10, 3 * 2.0 ** -10, 1.0625, 1.1875, 17.0, 456.0, -464.0])])
    want = vals.to(torch.float8_e4m3fn).view(torch.uint8)
    got = torch.tensor([lib.orc_e4m3_encode(float(v)) for v in vals], dtype=torch.uint8)
    if not torch.equal(got, want):
        raise AssertionError(f"E4M3 encoding differs from torch on {int((got != want).sum())} values")
    for v, c in ((470.0, 0x7e), (-1e30, 0xfe), (float("inf"), 0x7e), (float("nan"), 0x7f)):
        if lib.orc_e4m3_encode(v) != c:
            raise AssertionError(f"E4M3 of {v}")


def _e4m3_nearest(q: torch.Tensor) -> torch.Tensor:
    """E4M3 codes of float64 values `q` (|q| <= 448) found by brute force: the
    non-negative finite grid is enumerated by torch's float8_e4m3fn decoding
    of codes 0..126, the nearest grid value to |q| is taken, an exact tie goes
    to the even code, and the sign bit is that of q."""
    grid = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    a = q.abs().reshape(-1, 1)
    d = (a - grid.view(1, -1)).abs()
    best = d.min(dim=1, keepdim=True).values
    cand = d == best
    odd = (torch.arange(127) % 2 == 1).view(1, -1)
    pick_even = cand & ~odd
    idx = torch.where(pick_even.any(dim=1), pick_even.to(torch.int64).argmax(dim=1),
                      cand.to(torch.int64).argmax(dim=1))
    sign = torch.signbit(q.reshape(-1)).to(torch.int64) * 0x80
    return (idx | sign).to(torch.uint8).view(q.shape)


def pin_shadow_refresh(lib):
    """The read copy of a pool: fp16 codes are torch's round-to-nearest-even
    cast.  E4M3: the row's largest magnitude amax maps to 448; every code is
    the nearest E4M3 grid value to v * 448 / amax (exact ties to the even
    code), found by brute force over the grid; the row scale is amax / 448
    rounded to fp32; an all-zero row gets scale 1 and zero codes; rows of
    exact midpoints between grid values round to the even neighbour."""
    g = torch.Generator().manual_seed(62)
    st = torch.randn((3, 2, 4, 32), generator=g) * torch.rand((3, 2, 4, 1), generator=g) * 5
    st[1, 0, 2] = 0.0
    # a row whose amax is 448, so that v * 448 / amax = v exactly: midpoints
    # between neighbouring grid values (normal and subnormal), each a tie
    ties = torch.tensor([448.0, 1.0625, 1.1875, -1.0625, 2.0 ** -10, 3 * 2.0 ** -10, 5 * 2.0 ** -10, 17.0,
                         19.0, 208.0, 432.0, -0.0, 0.0, 2.0 ** -7 + 2.0 ** -11, 0.5, -0.5625])
    st[2, 1, 3] = torch.cat([ties, torch.zeros(32 - ties.numel())])
    h, none = oracle.shadow_refresh(st, oracle.SHADOW_F16, lib=lib)
    if none is not None or not torch.equal(h, st.half()):
        raise AssertionError("fp16 read copy")
    codes, scale = oracle.shadow_refresh(st, oracle.SHADOW_E4M3, lib=lib)
    sd = st.to(torch.float64)
    amax = sd.abs().amax(dim=-1)
    want_scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).to(torch.float32)
    q = torch.where(amax[..., None] > 0, sd * 448.0 / torch.where(amax > 0, amax, 1.0)[..., None], sd)
    want_codes = _e4m3_nearest(q)
    if not torch.equal(scale, want_scale):
        raise AssertionError("E4M3 row scales")
    if not torch.equal(codes, want_codes):
        raise AssertionError(f"E4M3 read copy: {int((codes != want_codes).sum())} codes differ")
    tie_codes = codes[2, 1, 3, :ties.numel()].tolist()
    if tie_codes[1] != 0x38 or tie_codes[2] != 0x3a or tie_codes[4] != 0 or tie_codes[5] != 2:
        raise AssertionError(f"E4M3 ties: {tie_codes[:6]}")
    if float(scale[1, 0, 2]) != 1.0 or int(codes[1, 0, 2].abs().sum()) != 0:
        raise AssertionError("zero row")
    bf = st.to(torch.bfloat16)  # a 16-bit pool: the copy is of the stored values
    c16, s16 = oracle.shadow_refresh(bf, oracle.SHADOW_E4M3, lib=lib)
    c32, s32 = oracle.shadow_refresh(bf.float(), oracle.SHADOW_E4M3, lib=lib)
    if not (torch.equal(c16, c32) and torch.equal(s16, s32)):
        raise AssertionError("bf16 pool read copy")


# E2M1 magnitudes by code (OCP Microscaling formats, FP4 E2M1: bias 1, one
# fraction bit, exponent field 0 the subnormal 0.5), written out from the
# format's definition.
_E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _e2m1_nearest(q: torch.Tensor) -> torch.Tensor:
    """E2M1 codes of float64 values `q` by brute force: the nearest of the
    eight magnitudes to |q| (|q| past 6 takes 6), an exact tie to the even
    code, the sign in bit 3."""
    grid = torch.tensor(_E2M1_GRID, dtype=torch.float64)
    a = q.abs().reshape(-1, 1).clamp(max=6.0)
    d = (a - grid.view(1, -1)).abs()
    cand = d == d.min(dim=1, keepdim=True).values
    even = cand & (torch.arange(8) % 2 == 0).view(1, -1)
    idx = torch.where(even.any(dim=1), even.to(torch.int64).argmax(dim=1), cand.to(torch.int64).argmax(dim=1))
    sign = torch.signbit(q.reshape(-1)).to(torch.int64) * 8
    return (idx | sign).to(torch.uint8).view(q.shape)


def pin_e2m1_codes(lib):
    """FP4 E2M1 as the NVFP4 read copy stores it: the sixteen codes decode to
    the format's magnitudes with the sign in bit 3; random values, every
    midpoint between neighbours (a tie: to the even code) and values past 6
    (saturated) encode as the brute-force nearest grid value."""
    for code in range(16):
        want = _E2M1_GRID[code & 7] * (-1.0 if code & 8 else 1.0)
        got = lib.orc_e2m1_decode(code)
        if got != want or (code == 8 and not np.signbit(got)):
            raise AssertionError(f"E2M1 code {code} decodes to {got}, not {want}")
    g = torch.Generator().manual_seed(64)
    mids = [(a + b) / 2 for a, b in zip(_E2M1_GRID, _E2M1_GRID[1:])]
    vals = torch.cat([(torch.rand(3000, generator=g) - 0.5) * 16, torch.tensor(mids, dtype=torch.float32),
                      -torch.tensor(mids, dtype=torch.float32), torch.tensor([6.5, 7.0, 1e9, -9.0, 0.0, -0.0])])
    vals = vals.to(torch.float64)
    want = _e2m1_nearest(vals)
    got = torch.tensor([lib.orc_e2m1_encode(float(v)) for v in vals], dtype=torch.uint8)
    if not torch.equal(got, want):
        i = int(torch.nonzero(got != want)[0])
        raise AssertionError(f"E2M1 of {float(vals[i])}: {int(got[i])}, nearest {int(want[i])}")
    if [lib.orc_e2m1_encode(m) for m in mids] != [0, 2, 2, 4, 4, 6, 6]:
        raise AssertionError("E2M1 ties")


def _nvfp4_expected(st: torch.Tensor):
    """The NVFP4 read copy of `st` built by brute force: s = amax / (6 * 448)
    rounded to fp32 (1 for an all-zero row); per block of 16 the E4M3 code
    nearest (block amax) / (6 s); per element the E2M1 code nearest
    v / (block scale * s) (zero where the block scale is zero)."""
    sd = st.to(torch.float64).reshape(-1, st.shape[-1])
    rows, n = sd.shape
    amax = sd.abs().amax(dim=1)
    s = torch.where(amax > 0, amax / (6.0 * 448.0), torch.ones_like(amax)).to(torch.float32).to(torch.float64)
    bmax = sd.abs().view(rows, n // 16, 16).amax(dim=2)
    bcode = _e4m3_nearest(bmax / (6.0 * s[:, None]))
    bsv = bcode.view(torch.float8_e4m3fn).to(torch.float64)
    den = (bsv * s[:, None]).repeat_interleave(16, dim=1)
    q = torch.where(den > 0, sd / torch.where(den > 0, den, 1.0), torch.zeros_like(sd))
    codes = _e2m1_nearest(q)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).view(*st.shape[:-1], n // 2)
    return packed, s.to(torch.float32).view(st.shape[:-1]), bcode.view(*st.shape[:-1], n // 16)


def _nvfp4_dequant(codes: torch.Tensor, rec: torch.Tensor) -> torch.Tensor:
    n = codes.shape[-1] * 2
    grid = torch.tensor([_E2M1_GRID[c & 7] * (-1.0 if c & 8 else 1.0) for c in range(16)], dtype=torch.float64)
    v = torch.stack([grid[(codes & 15).long()], grid[(codes >> 4).long()]], dim=-1).reshape(*codes.shape[:-1], n)
    bsv = rec.view(torch.uint8)[..., 4:4 + n // 16].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
    return v * bsv.repeat_interleave(16, dim=-1) * rec[..., :1].to(torch.float64)


def _nvfp4_error_bound(st: torch.Tensor, rec: torch.Tensor) -> torch.Tensor:
    """Per element, the most the NVFP4 copy may be off: half the largest E2M1
    step (1) times block scale times s, or, where the block scale rounded
    below (block amax) / (6 s) so that its largest values saturate at 6,
    6 s times that shortfall."""
    n = st.shape[-1]
    sd = st.to(torch.float64)
    s = rec[..., :1].to(torch.float64)
    bs = rec.view(torch.uint8)[..., 4:4 + n // 16].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
    bmax = sd.abs().view(*st.shape[:-1], n // 16, 16).amax(dim=-1)
    per_block = s * torch.maximum(bs, 6.0 * (bmax / (6.0 * s) - bs).clamp(min=0.0))
    return per_block.repeat_interleave(16, dim=-1)


def pin_nvfp4_refresh(lib):
    """The NVFP4 read copy of a pool, against a brute-force construction: the
    row scale is amax / (6 * 448) in fp32, each block of 16 keeps the nearest
    E4M3 code of its amax / (6 s), each element the nearest E2M1 code of
    v / (block scale * s), two codes a byte (the even element low); an
    all-zero row keeps scale 1 and zero codes; a row already on the grid
    (codes times block scales times a power-of-two s) round-trips exactly;
    every element lies within its block's largest half-step (block scale * s)
    of its value, or within the shortfall of a block scale that rounded down;
    a bf16 pool is copied as its stored values."""
    g = torch.Generator().manual_seed(65)
    st = torch.randn((3, 2, 4, 64), generator=g) * torch.rand((3, 2, 4, 1), generator=g) * 5
    st[1, 0, 2] = 0.0
    st[2, 1, 1, 16:32] = 1e-9 * torch.randn(16, generator=g)  # a block far below the row's largest
    codes, rec = oracle.shadow_refresh(st, oracle.SHADOW_NVFP4, lib=lib)
    if codes.shape != (3, 2, 4, 32) or rec.shape != (3, 2, 4, oracle.nvfp4_scale_words(64)):
        raise AssertionError(f"NVFP4 shapes {tuple(codes.shape)} {tuple(rec.shape)}")
    wc, ws, wb = _nvfp4_expected(st)
    if not torch.equal(rec[..., 0], ws):
        raise AssertionError("NVFP4 row scales")
    if not torch.equal(rec.view(torch.uint8)[..., 4:8], wb):
        raise AssertionError("NVFP4 block scales")
    if not torch.equal(codes, wc):
        raise AssertionError(f"NVFP4 codes: {int((codes != wc).sum())} bytes differ")
    if float(rec[1, 0, 2, 0]) != 1.0 or int(codes[1, 0, 2].sum()) != 0:
        raise AssertionError("NVFP4 zero row")
    dq = _nvfp4_dequant(codes, rec)
    if not torch.all((dq - st.to(torch.float64)).abs() <= _nvfp4_error_bound(st, rec) * (1 + 1e-12)):
        raise AssertionError("NVFP4 element error above its block's bound")
    # a row on the grid: E2M1 magnitudes times E4M3 block scales times s = 2^-7,
    # each block holding one 6 so that its amax / (6 s) is its scale
    grid_row = torch.tensor([_E2M1_GRID[(3 * i) % 8] * (-1.0 if i % 5 == 0 else 1.0) for i in range(64)])
    grid_row[0::16] = 6.0
    bscale = torch.tensor([448.0, 1.0, 0.25, 20.0]).repeat_interleave(16)
    exact = (grid_row * bscale * 2.0 ** -7).view(1, 64)
    c1, r1 = oracle.shadow_refresh(exact, oracle.SHADOW_NVFP4, lib=lib)
    if not torch.equal(_nvfp4_dequant(c1, r1), exact.to(torch.float64)):
        raise AssertionError("a row on the NVFP4 grid must round-trip")
    bf = st.to(torch.bfloat16)
    c16, s16 = oracle.shadow_refresh(bf, oracle.SHADOW_NVFP4, lib=lib)
    c32, s32 = oracle.shadow_refresh(bf.float(), oracle.SHADOW_NVFP4, lib=lib)
    if not (torch.equal(c16, c32) and torch.equal(s16, s32)):
        raise AssertionError("bf16 pool NVFP4 read copy")


def pin_replay_nvfp4_read_copy(lib):
    """Steps that do not fold read the NVFP4 copy: a checkpoint on the copy's
    grid gives exactly the checkpoint's y; a general one moves y by no more
    than the copy's rounding (per element the bound of pin_nvfp4_refresh) and
    does move it; a fold rewrites the copy from the new checkpoint, other
    steps leave it."""
    L = 4
    counts = [0, 1, 2, 3, 3, 2]
    sc = _replay_scenario(46, L, counts, dstate=32, state_dtype=torch.float32)
    ck = sc["ckpt"]
    codes, rec = oracle.shadow_refresh(ck, oracle.SHADOW_NVFP4, lib=lib)
    # a checkpoint on the NVFP4 grid: each block's first element +6, the row
    # scale a power of two (the block holding the row's largest keeps the
    # scale 448), so that the values are exact in fp32 and their copy is the
    # same codes and scales
    cg = codes.clone()
    cg[..., 0::8] = (cg[..., 0::8] & 0xF0) | 7
    rg = rec.clone()
    rg[..., 0] = torch.exp2(torch.round(torch.log2(rec[..., 0])))
    grid = _nvfp4_dequant(cg, rg).to(torch.float32)
    c2, r2 = oracle.shadow_refresh(grid, oracle.SHADOW_NVFP4, lib=lib)
    if not (torch.equal(c2, cg) and torch.equal(r2.view(torch.int32), rg.view(torch.int32))):
        raise AssertionError("the NVFP4 copy of values on its grid must be those codes and scales")
    sg = dict(sc, ckpt=grid)
    plain = _run_replay(sg, lib)
    r = _run_replay(sg, lib, shadow=cg, shadow_scale=rg, shadow_format=oracle.SHADOW_NVFP4)
    if not torch.equal(r.y_exact, plain.y_exact):
        raise AssertionError("an exact NVFP4 read copy must give the checkpoint's y")
    plain = _run_replay(sc, lib)
    r = _run_replay(sc, lib, shadow=codes, shadow_scale=rec, shadow_format=oracle.SHADOW_NVFP4)
    half = _nvfp4_error_bound(ck, rec)
    moved = False
    for b, c in enumerate(counts):
        s = int(sc["slot_of"][b])
        if c + 1 == L:
            cs, ss = oracle.shadow_refresh(r.ckpt[s], oracle.SHADOW_NVFP4, lib=lib)
            if not (torch.equal(r.shadow[s], cs) and torch.equal(r.shadow_scale[s], ss)):
                raise AssertionError("a fold must rewrite the NVFP4 copy from the new checkpoint")
            continue
        if not (torch.equal(r.shadow[s], codes[s]) and torch.equal(r.shadow_scale[s], rec[s])):
            raise AssertionError("a step that does not fold must not write the NVFP4 copy")
        Cb = sc["C"][b].double()
        hpg = ck.shape[1] // Cb.shape[0]
        dy = (plain.y_exact[b] - r.y_exact[b]).abs()
        for h in range(ck.shape[1]):
            err = half[s, h] @ Cb[h // hpg].abs()
            zz = sc["z"][b, h].double()
            gate = (zz / (1 + torch.exp(-zz))).abs()
            if not torch.all(dy[h] <= gate * err * (1 + 1e-9) + 1e-12):
                raise AssertionError("NVFP4 read-copy error above its bound")
        moved |= float(dy.max()) > 0
    if not moved:
        raise AssertionError("the readout did not use the NVFP4 copy")


def _e4m3_dequant(codes, scale):
    return codes.view(torch.float8_e4m3fn).to(torch.float64) * scale.to(torch.float64)[..., None]


def pin_replay_read_copy(lib):
    """Steps that do not fold read the copy: with a checkpoint already on the
    copy's grid (E4M3 codes times a row scale, or fp16 values) y is exactly
    the y read from the checkpoint; with a general checkpoint y moves by no
    more than the copy's rounding (half an E4M3 ulp, relative 2^-4, or the
    subnormal quantum 2^-10 scale, per element), and does move.  A fold
    writes the checkpoint and the copy of it; other steps leave the copy."""
    L = 4
    counts = [0, 1, 2, 3, 3, 2]
    sc = _replay_scenario(44, L, counts, state_dtype=torch.float32)
    ck = sc["ckpt"]
    # a checkpoint on the E4M3 grid: codes times a power-of-two row scale,
    # each row holding one 448 (so amax / 448 is that scale): its copy is exact
    codes0, scale0 = oracle.shadow_refresh(ck, oracle.SHADOW_E4M3, lib=lib)
    codes0[..., 0] = 0x7e
    pow2 = torch.exp2(torch.round(torch.log2(scale0)))
    grid = _e4m3_dequant(codes0, pow2).to(torch.float32)
    sg = dict(sc, ckpt=grid)
    cg, sgs = oracle.shadow_refresh(grid, oracle.SHADOW_E4M3, lib=lib)
    plain = _run_replay(sg, lib)
    r = _run_replay(sg, lib, shadow=cg, shadow_scale=sgs, shadow_format=oracle.SHADOW_E4M3)
    if not torch.equal(r.y_exact, plain.y_exact):
        raise AssertionError("an exact read copy must give the checkpoint's y")
    h16 = ck.half().float()
    sh = dict(sc, ckpt=h16)
    p16 = _run_replay(sh, lib)
    r16 = _run_replay(sh, lib, shadow=h16.half(), shadow_format=oracle.SHADOW_F16)
    if not torch.equal(r16.y_exact, p16.y_exact):
        raise AssertionError("an exact fp16 read copy must give the checkpoint's y")
    # general checkpoint: bounded, nonzero change of the readout y
    codes, scale = oracle.shadow_refresh(ck, oracle.SHADOW_E4M3, lib=lib)
    plain = _run_replay(sc, lib)
    r = _run_replay(sc, lib, shadow=codes, shadow_scale=scale, shadow_format=oracle.SHADOW_E4M3)
    moved = False
    for b, c in enumerate(counts):
        s = int(sc["slot_of"][b])
        if c + 1 == L:
            if not torch.equal(r.y_exact[b], plain.y_exact[b]):
                raise AssertionError("a folding step reads the checkpoint, not the copy")
            cs, ss = oracle.shadow_refresh(r.ckpt[s], oracle.SHADOW_E4M3, lib=lib)
            if not (torch.equal(r.shadow[s], cs) and torch.equal(r.shadow_scale[s], ss)):
                raise AssertionError("a fold must rewrite the read copy from the new checkpoint")
            continue
        if not (torch.equal(r.shadow[s], codes[s]) and torch.equal(r.shadow_scale[s], scale[s])):
            raise AssertionError("a step that does not fold must not write the read copy")
        # |dy| <= gate * gamma * sum_n (2^-4 |S_n| + 2^-10 scale) |C_n|
        g = sc["slot_of"]
        Cb = sc["C"][b].double()
        heads_per_group = ck.shape[1] // Cb.shape[0]
        gamma = (plain.y_exact[b] - r.y_exact[b]).abs()
        for h in range(ck.shape[1]):
            Cg = Cb[h // heads_per_group]
            err = (ck[s, h].double().abs() * 2.0 ** -4 + 2.0 ** -10 * scale[s, h].double()[:, None]) @ Cg.abs()
            zz = sc["z"][b, h].double()
            gate = (zz / (1 + torch.exp(-zz))).abs()
            if not torch.all(gamma[h] <= gate * err * (1 + 1e-9) + 1e-12):
                raise AssertionError("read-copy error above its bound")
        if float(gamma.max()) > 0:
            moved = True
    if not moved:
        raise AssertionError("the readout did not use the read copy")


def _ssd_run(w, lib, **kw):
    args = dict(D=w.D, z=w.z, dt_bias=w.dt_bias, dt_softplus=w.dt_softplus, dt_limit=w.dt_limit,
                initial_states=w.initial_states, lib=lib)
    args.update(kw)
    return oracle.ssd(w.x, w.dt, w.A, w.B, w.C, w.cu_chunk_seqlens, w.seq_idx, w.nseq, **args)


def pin_ssd_equals_token_loop(lib):
    """The SSD prefill over packed sequences is the selective state update
    run token by token over each sequence from its initial state: y and the
    final states equal the packed update's (same double arithmetic), for any
    chunk size."""
    lengths = [5, 37, 16, 1]
    for q in (4, 16):
        w = workloads.ssd_problem(51, lengths, heads=4, dim=3, dstate=8, groups=2, chunk_size=q,
                                  state_dtype=torch.float32)
        r = _ssd_run(w, lib)
        width = max(lengths)
        tab = torch.arange(w.nseq, dtype=torch.int64).view(-1, 1).repeat(1, width)
        ref = oracle.ssu(w.initial_states, w.x, w.dt, w.A, w.B, w.C, D=w.D, z=w.z, dt_bias=w.dt_bias,
                         dt_softplus=True, read=oracle.Table.of(tab), cu_seqlens=w.cu_seqlens.to(torch.int64),
                         lib=lib)
        if not torch.equal(r.y_exact, ref.y_exact):
            raise AssertionError("SSD y differs from the token loop")
        last = w.last_chunk_indices.long()
        if not torch.equal(r.states[last], ref.state):
            raise AssertionError("SSD final states differ from the token loop")


def _ssd_chunked_numpy(w):
    """The five stages of the chunked evaluation, in float64 numpy: per chunk
    the cumulative decay, the chunk's own state contribution, the state
    passed between chunks (seq_idx decides where a sequence opens), C . B^T
    and the chunk scan.  Returns (y, states at chunk ends)."""
    x, dt, B, C = (w.x.double().numpy(), w.dt.double().numpy(), w.B.double().numpy(), w.C.double().numpy())
    A = w.A.double().numpy()
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    hpg = H // G
    d = dt + (w.dt_bias.double().numpy() if w.dt_bias is not None else 0.0)
    if w.dt_softplus:
        d = np.logaddexp(0.0, d)
    d = np.clip(d, w.dt_limit[0], w.dt_limit[1])
    cu = w.cu_chunk_seqlens.long().numpy()
    si = w.seq_idx.long().numpy()
    init = None if w.initial_states is None else w.initial_states.double().numpy()
    y = np.zeros((T, H, P))
    states = np.zeros((len(si), H, P, N))
    S = np.zeros((H, P, N))
    for c in range(len(si)):
        t0, t1 = cu[c], cu[c + 1]
        if c == 0 or si[c] != si[c - 1]:
            S = init[si[c]].copy() if init is not None else np.zeros((H, P, N))
        for h in range(H):
            g = h // hpg
            acs = np.cumsum(A[h] * d[t0:t1, h])                       # stage 1
            Bc, Cc, xc, dc = B[t0:t1, g], C[t0:t1, g], x[t0:t1, h], d[t0:t1, h]
            wgt = np.exp(acs[-1] - acs) * dc if t1 > t0 else np.zeros(0)
            Sc = (xc * wgt[:, None]).T @ Bc                             # stage 2: [P, N]
            CB = Cc @ Bc.T                                               # stage 4: [L, L]
            L = np.tril(np.exp(acs[:, None] - acs[None, :]))
            yc = np.exp(acs)[:, None] * (Cc @ S[h].T) + (CB * L) @ (xc * dc[:, None])   # stage 5
            if w.D is not None:
                yc = yc + w.D[h].item() * xc
            if w.z is not None:
                zz = w.z[t0:t1, h].double().numpy()
                yc = yc * zz / (1 + np.exp(-zz))
            y[t0:t1, h] = yc
            S[h] = (np.exp(acs[-1]) if t1 > t0 else 1.0) * S[h] + Sc       # stage 3
        states[c] = S
    return y, states


def pin_ssd_chunked_form(lib):
    """The oracle's token loop equals the chunked five-stage evaluation
    (written out independently in numpy) to double rounding, for y and the
    state at the end of every chunk, with ragged last chunks, several
    sequences, a clamped dt and without initial states."""
    cases = [dict(lengths=[9, 33, 2], chunk_size=8),
             dict(lengths=[17, 17], chunk_size=16, dt_limit=(0.02, 0.3), with_init=False),
             dict(lengths=[50], chunk_size=64, with_z=False, with_D=False)]
    for i, kw in enumerate(cases):
        lengths = kw.pop("lengths")
        w = workloads.ssd_problem(52 + i, lengths, heads=4, dim=3, dstate=8, groups=2, state_dtype=torch.float64,
                                  **kw)
        r = _ssd_run(w, lib, state_dtype=torch.float64)
        y, st = _ssd_chunked_numpy(w)
        _close(r.y_exact.numpy(), y, rtol=1e-10, atol=1e-12, what=f"SSD y, case {i}")
        _close(r.states.numpy(), st, rtol=1e-10, atol=1e-12, what=f"SSD states, case {i}")


def pin_ssd_seq_idx_authority(lib):
    """seq_idx alone decides where a sequence opens: re-labelling chunk 2
    as sequence 1's makes it start from sequence 1's initial state, whatever
    last_chunk_indices says, and chunk 3 continue from it."""
    w = workloads.ssd_problem(55, [40, 40], heads=2, dim=2, dstate=4, groups=1, chunk_size=16,
                              state_dtype=torch.float64)
    relabel = w.seq_idx.clone()
    relabel[2] = 1
    r = _ssd_run(w, lib, **{})
    r2 = oracle.ssd(w.x, w.dt, w.A, w.B, w.C, w.cu_chunk_seqlens, relabel, w.nseq, D=w.D, z=w.z,
                    dt_bias=w.dt_bias, dt_softplus=True, initial_states=w.initial_states, lib=lib)
    if not torch.equal(r.states[:2], r2.states[:2]):
        raise AssertionError("chunks before the relabelled one must not change")
    # chunk 2 alone from sequence 1's initial state, via the token loop
    t0, t1 = int(w.cu_chunk_seqlens[2]), int(w.cu_chunk_seqlens[3])
    sub = slice(t0, t1)
    tab = torch.ones((1, t1 - t0), dtype=torch.int64)
    ref = oracle.ssu(w.initial_states, w.x[sub], w.dt[sub], w.A, w.B[sub], w.C[sub], D=w.D, z=w.z[sub],
                     dt_bias=w.dt_bias, dt_softplus=True, read=oracle.Table.of(tab),
                     cu_seqlens=torch.tensor([0, t1 - t0]), lib=lib)
    if not torch.equal(r2.states[2], ref.state[1]):
        raise AssertionError("a relabelled chunk must open from its sequence's initial state")
    if torch.equal(r2.states[3], r.states[3]):
        raise AssertionError("the chunk after a relabelled one continues from it")


def pin_ssd_dt_limit(lib):
    """x = 0 leaves only the decay: the state at the end is
    exp(A sum_t clamp(softplus(dt + bias), lo, hi)) times the initial state
    (closed form, with values below, inside and above the limits)."""
    w = workloads.ssd_problem(56, [30], heads=3, dim=2, dstate=4, groups=1, chunk_size=8, state_dtype=torch.float64,
                              dt_limit=(0.2, 0.6))
    w.x = torch.zeros_like(w.x)
    r = _ssd_run(w, lib)
    d = np.clip(np.logaddexp(0.0, w.dt.double().numpy() + w.dt_bias.double().numpy()), 0.2, 0.6)
    if not (np.any(d == 0.2) and np.any(d == 0.6) and np.any((d > 0.2) & (d < 0.6))):
        raise AssertionError("the case must exercise both limits")
    decay = np.exp(w.A.double().numpy() * d.sum(axis=0))
    want = decay[:, None, None] * w.initial_states[0].double().numpy()
    _close(r.states[-1].numpy(), want, rtol=1e-12, atol=1e-15, what="dt_limit closed form")


def _verify_scenario(seed, L, T, counts, heads=4, dim=3, dstate=8, groups=2, io=torch.bfloat16,
                     state_dtype=torch.float64, with_z=True, pad_last=False):
    """The replay scenario with T draft tokens per sequence instead of one."""
    sc = _replay_scenario(seed, L, counts, heads, dim, dstate, groups, io, state_dtype, with_z, pad_last)
    g = torch.Generator().manual_seed(seed + 1000)
    nseq = len(counts)
    sc["x"] = torch.randn((nseq, T, heads, dim), generator=g).to(io)
    sc["dt"] = torch.rand((nseq, T, heads, dim), generator=g) * 0.3 - 1.0   # softplus(dt - 0.5) ~ 0.2 .. 0.3
    sc["B"] = torch.randn((nseq, T, groups, dstate), generator=g).to(io)
    sc["C"] = torch.randn((nseq, T, groups, dstate), generator=g).to(io)
    sc["z"] = torch.randn((nseq, T, heads, dim), generator=g).to(io) if with_z else None
    sc["bias"] = torch.full((heads,), 0.5)
    return sc


def _run_verify(sc, lib):
    return oracle.replay_verify(sc["ckpt"], sc["x"], sc["dt"], sc["A"], sc["B"], sc["C"], sc["xbuf"], sc["dtbuf"],
                                sc["Bbuf"], sc["count"], D=sc["D"], z=sc["z"], dt_bias=sc["bias"], dt_softplus=True,
                                slot_of=sc["slot_of"], lib=lib)


def _draft_steps(sc, b):
    """The drafts' processed steps as the buffer stores them: fp32 of
    softplus(dt + bias)."""
    d = np.logaddexp(0.0, f64(sc["dt"][b]) + f64(sc["bias"])[None, :, None])
    return torch.from_numpy(d).to(torch.float32)


def _plain_verify_history(sc, b, ndrafts, lib, extra=None):
    """Sequence b token by token by the plain update from its checkpoint: its
    committed entries, then drafts 0 .. ndrafts-1, then `extra` = (x, dt', B,
    C, z) of one more token; processed steps as dt, softplus off."""
    s = int(sc["slot_of"][b])
    c = int(sc["count"][b])
    d = _draft_steps(sc, b)
    xs = [sc["xbuf"][s, :c], sc["x"][b, :ndrafts]]
    dts = [sc["dtbuf"][s, :c], d[:ndrafts]]
    Bs = [sc["Bbuf"][s, :c], sc["B"][b, :ndrafts]]
    Cs = [sc["C"][b, :1].expand(c, -1, -1), sc["C"][b, :ndrafts]]
    zs = None if sc["z"] is None else [sc["z"][b, :1].expand(c, -1, -1), sc["z"][b, :ndrafts]]
    if extra is not None:
        xs.append(extra[0]); dts.append(extra[1]); Bs.append(extra[2]); Cs.append(extra[3])
        if zs is not None:
            zs.append(extra[4])
    n = c + ndrafts + (1 if extra is not None else 0)
    tab = torch.full((1, n), s, dtype=torch.int64)
    return oracle.ssu(sc["ckpt"], torch.cat(xs), torch.cat(dts), sc["A"], torch.cat(Bs), torch.cat(Cs), D=sc["D"],
                      z=None if zs is None else torch.cat(zs), read=oracle.Table.of(tab),
                      cu_seqlens=torch.tensor([0, n]), lib=lib)


def pin_verify_lossless(lib):
    """Speculative decoding on checkpoint + buffer is lossless: draft k's y
    equals the plain recurrence over the committed entries and drafts
    0 .. k; the flush fires exactly when c + 2T >= L, leaving in the
    checkpoint the state after the committed entries, and nothing is
    committed (count = c, or 0 after the flush)."""
    L, T = 9, 3
    counts = [0, 1, 2, 3, 4, 8, 0]    # c + 2T >= 9 from c = 3 on
    sc = _verify_scenario(61, L, T, counts)
    r = _run_verify(sc, lib)
    for b, c in enumerate(counts):
        h = _plain_verify_history(sc, b, T, lib)
        for k in range(T):
            _close(r.y_exact[b, k].numpy(), h.y_exact[c + k].numpy(), rtol=1e-11, atol=1e-12,
                   what=f"draft {k} y (c={c})")
        s = int(sc["slot_of"][b])
        fold = c + 2 * T >= L
        if fold:
            hc = _plain_verify_history(sc, b, 0, lib) if c > 0 else None
            want = f64(sc["ckpt"][s]) if hc is None else f64(hc.state[s])
            _close(f64(r.ckpt[s]), want, rtol=1e-11, atol=1e-13, what=f"flushed checkpoint (c={c})")
            if int(r.count[b]) != 0:
                raise AssertionError("a flush leaves no committed entry")
        else:
            if not torch.equal(r.ckpt[s], sc["ckpt"][s]):
                raise AssertionError("a step without flush must not write the checkpoint")
            if int(r.count[b]) != c:
                raise AssertionError("verification commits nothing")


def pin_verify_entries(lib):
    """The drafts are appended as entries c .. c+T-1 (0 .. T-1 after a flush):
    x and B with their bits, the processed step in fp32; the committed
    entries below c are untouched."""
    L, T = 8, 2
    counts = [1, 3, 5]                 # the last flushes (5 + 4 >= 8)
    sc = _verify_scenario(62, L, T, counts)
    r = _run_verify(sc, lib)
    for b, c in enumerate(counts):
        s = int(sc["slot_of"][b])
        at = 0 if c + 2 * T >= L else c
        if not torch.equal(r.xbuf[s, at:at + T], sc["x"][b]) or not torch.equal(r.Bbuf[s, at:at + T], sc["B"][b]):
            raise AssertionError(f"appended drafts (c={c})")
        if not torch.equal(r.dtbuf[s, at:at + T], _draft_steps(sc, b)):
            raise AssertionError("appended processed steps")
        if at and not (torch.equal(r.xbuf[s, :c], sc["xbuf"][s, :c]) and torch.equal(r.Bbuf[s, :c], sc["Bbuf"][s, :c])):
            raise AssertionError("committed entries changed")


def pin_verify_rollback(lib):
    """Rollback is moving the count: after verifying T drafts and accepting
    the first a, the next plain replay step (count = c + a) gives the y of
    the plain recurrence over the committed entries, drafts 0 .. a-1 and the
    new token -- the rejected drafts leave no trace."""
    L, T = 12, 3
    counts = [0, 2, 4]
    sc = _verify_scenario(63, L, T, counts)
    r = _run_verify(sc, lib)
    g = torch.Generator().manual_seed(64)
    heads, dim = sc["x"].shape[2], sc["x"].shape[3]
    groups, dstate = sc["B"].shape[2], sc["B"].shape[3]
    for a in range(T + 1):
        nx = torch.randn((len(counts), heads, dim), generator=g).to(sc["x"].dtype)
        nd = torch.rand((len(counts), heads, dim), generator=g) * 0.3
        nB = torch.randn((len(counts), groups, dstate), generator=g).to(sc["x"].dtype)
        nC = torch.randn((len(counts), groups, dstate), generator=g).to(sc["x"].dtype)
        nz = torch.randn((len(counts), heads, dim), generator=g).to(sc["x"].dtype)
        step = oracle.replay(r.ckpt, nx, nd, sc["A"], nB, nC, r.xbuf, r.dtbuf, r.Bbuf, r.count + a, D=sc["D"], z=nz,
                             slot_of=sc["slot_of"], lib=lib)
        for b in range(len(counts)):
            h = _plain_verify_history(sc, b, a, lib,
                                      extra=(nx[b:b + 1], nd[b:b + 1], nB[b:b + 1], nC[b:b + 1], nz[b:b + 1]))
            _close(step.y_exact[b].numpy(), h.y_exact[counts[b] + a].numpy(), rtol=1e-11, atol=1e-12,
                   what=f"step after accepting {a} of {T} drafts (c={counts[b]})")


def pin_verify_pad(lib):
    """A pad slot: the drafts run from a zero state with no history (the
    first draft's y is the zero-state closed form), nothing is written and
    the count is 0."""
    sc = _verify_scenario(65, 6, 2, [1, 2], with_z=False, pad_last=True)
    r = _run_verify(sc, lib)
    b = 1
    gi = np.arange(sc["x"].shape[2]) // (sc["x"].shape[2] // sc["B"].shape[2])
    d = _draft_steps(sc, b)[0].double().numpy()
    xn = f64(sc["x"][b, 0])
    bc = np.einsum("hn,hn->h", f64(sc["B"][b, 0])[gi], f64(sc["C"][b, 0])[gi])
    _close(r.y_exact[b, 0].numpy(), d * bc[:, None] * xn + f64(sc["D"])[:, None] * xn, what="pad draft y")
    if not torch.equal(r.ckpt, sc["ckpt"]) or int(r.count[b]) != 0:
        raise AssertionError("a pad sequence writes nothing and keeps no entry")
    s0 = int(sc["slot_of"][0])
    untouched = [s for s in range(sc["ckpt"].shape[0]) if s != s0]
    if not torch.equal(r.xbuf[untouched], sc["xbuf"][untouched]):
        raise AssertionError("a pad sequence must not append")


ALL_PINS = [pin_conversions, pin_scalar_functions, pin_hand_worked, pin_dt_zero, pin_zero_state,
            pin_A_zero, pin_decay_only, pin_unrolled, pin_basis_vectors, pin_group_map,
            pin_page_examples, pin_pad_never_written, pin_disable_and_untouched, pin_table_forms,
            pin_seed_position, pin_seed_position_per_row, pin_per_head_dt, pin_aliasing_refused,
            pin_replay_lossless, pin_replay_buffer_entries, pin_replay_buffer_len_one,
            pin_replay_pad_and_aliasing, pin_empty_sequences, pin_bounded_decay, pin_e4m3_codes,
            pin_shadow_refresh, pin_replay_read_copy, pin_e2m1_codes, pin_nvfp4_refresh,
            pin_replay_nvfp4_read_copy, pin_ssd_equals_token_loop, pin_ssd_chunked_form,
            pin_ssd_seq_idx_authority, pin_ssd_dt_limit, pin_verify_lossless, pin_verify_entries,
            pin_verify_rollback, pin_verify_pad]
