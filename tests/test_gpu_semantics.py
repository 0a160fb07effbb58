"""Slot semantics, equivalences between call forms, device status bits,
determinism and graph capture, all through libssu's C ABI."""
import pytest
import torch

import selective_state_update_gb300 as ssu
import workloads
from gpu_harness import DEV, full_check, run_gpu
from dataclasses import replace

pytestmark = pytest.mark.gpu

F32, F16, BF16 = torch.float32, torch.float16, torch.bfloat16


def _gpu(w):
    return w.to(DEV)


@pytest.mark.parametrize("state_dtype", [F32, F16, BF16])
def test_packed_lengths_one_equals_onetoken_bitwise(libssu, state_dtype):
    w = workloads.random_problem(11, kind="onetoken", slots=64, heads=8, groups=2, dim=64, dstate=128,
                                 nseq=12, state_dtype=state_dtype, tables="distinct")
    a = _gpu(w)
    ya = run_gpu(a)
    b = _gpu(replace(w, kind="packed", cu_seqlens=torch.arange(13, dtype=torch.int32),
                     read=w.read.view(12, 1), dst=w.dst.view(12, 1)))
    yb = run_gpu(b)
    torch.cuda.synchronize()
    assert torch.equal(ya, yb) and torch.equal(a.state, b.state)


@pytest.mark.parametrize("state_dtype", [F32, F16])
def test_long_and_short_sequence_kernels_agree_bitwise(libssu, state_dtype):
    """The same sequences through the long-sequence kernel (six or more
    tokens a sequence on average) and, with empty sequences appended to the
    call, through the persistent short-sequence kernel: the same per-row
    functions give the same bits."""
    w = workloads.random_problem(31, kind="packed", slots=128, heads=8, groups=2, dim=64, dstate=128, nseq=6,
                                 min_len=6, max_len=9, tables="distinct", pad_frac=0.1, state_dtype=state_dtype)
    a = _gpu(w)
    ya = run_gpu(a)
    extra = 6
    cu = torch.cat([w.cu_seqlens, w.cu_seqlens[-1:].repeat(extra)])
    width = w.read.shape[1]
    pad = torch.full((extra, width), w.pad_slot_id, dtype=w.read.dtype)
    b = _gpu(replace(w, cu_seqlens=cu, read=torch.cat([w.read, pad]), dst=torch.cat([w.dst, pad]),
                     num_accepted=torch.cat([w.num_accepted, torch.ones(extra, dtype=w.num_accepted.dtype)]),
                     meta={"lengths": w.meta["lengths"] + [0] * extra}))
    assert w.rows >= 6 * w.nseq and w.rows < 6 * (w.nseq + extra)
    yb = run_gpu(b)
    torch.cuda.synchronize()
    assert torch.equal(ya, yb) and torch.equal(a.state, b.state)


def test_dense_equals_uniform_cu_bitwise(libssu):
    w = workloads.random_problem(12, kind="packed", slots=64, heads=4, groups=2, dim=64, dstate=128,
                                 nseq=5, max_len=3, dense=True)
    a = _gpu(w)
    ya = run_gpu(a)
    b = _gpu(replace(w, dense_steps=0, cu_seqlens=torch.arange(0, 16, 3, dtype=torch.int32)))
    yb = run_gpu(b)
    torch.cuda.synchronize()
    assert torch.equal(ya, yb) and torch.equal(a.state, b.state)


def test_flat_2d_and_per_row_name_the_same_entries(libssu):
    """MATE "Mamba / SSU": with one sequence per call the flat [rows] table
    and the 2-D [1, rows] table name the same entries."""
    w = workloads.random_problem(13, kind="packed", slots=32, heads=4, groups=2, dim=16, dstate=64,
                                 nseq=1, max_len=7, allow_empty=False, tables="inplace", pad_slot_id=0)
    flat = w.read.reshape(-1).clone()
    forms = [dict(read=flat, dst=flat.clone(), slot_mode=workloads.SLOTS_STRIDED),
             dict(read=flat.view(1, -1), dst=flat.view(1, -1).clone(), slot_mode=workloads.SLOTS_STRIDED),
             dict(read=flat, dst=flat.clone(), slot_mode=workloads.SLOTS_PER_ROW)]
    outs = []
    for f in forms:
        g = _gpu(replace(w, **f))
        outs.append((run_gpu(g), g.state))
    torch.cuda.synchronize()
    for y, s in outs[1:]:
        assert torch.equal(y, outs[0][0]) and torch.equal(s, outs[0][1])
    full_check(replace(w, read=flat, dst=flat.clone()))


@pytest.mark.parametrize("kind", ["onetoken", "packed"])
def test_disable_state_update(libssu, kind):
    w = workloads.random_problem(14, kind=kind, slots=64, heads=4, groups=2, dim=64, dstate=128,
                                 nseq=6, max_len=3)
    a = _gpu(w)
    ya = run_gpu(a)
    b = _gpu(replace(w, disable_state_update=True))
    yb = run_gpu(b)
    torch.cuda.synchronize()
    assert torch.equal(b.state.cpu(), w.state)
    assert torch.equal(ya, yb)


def test_empty_sequences_and_empty_calls(libssu):
    w = workloads.random_problem(15, kind="packed", slots=64, heads=4, groups=2, dim=16, dstate=64,
                                 nseq=4, max_len=2)
    g = _gpu(replace(w, cu_seqlens=torch.zeros(5, dtype=torch.int32), x=w.x[:0], dt=w.dt[:0],
                     B=w.B[:0], C=w.C[:0], z=w.z[:0], meta={"lengths": [0] * 4}))
    y = run_gpu(g)
    torch.cuda.synchronize()
    assert y.numel() == 0 and torch.equal(g.state.cpu(), w.state)
    # nseq == 0
    g = _gpu(replace(w, cu_seqlens=torch.zeros(1, dtype=torch.int32), x=w.x[:0], dt=w.dt[:0],
                     B=w.B[:0], C=w.C[:0], z=w.z[:0], read=w.read[:0], dst=w.dst[:0],
                     num_accepted=w.num_accepted[:0], meta={"lengths": []}))
    run_gpu(g)
    torch.cuda.synchronize()
    assert torch.equal(g.state.cpu(), w.state)


def test_device_status_bad_slot_skips_only_that_unit(libssu):
    w = workloads.random_problem(16, kind="onetoken", slots=32, heads=4, groups=2, dim=16, dstate=64,
                                 nseq=6, tables="distinct", pad_frac=0.0)
    bad = w.read.clone()
    bad[2] = 1000                                   # outside the pool, not the pad id
    g = _gpu(replace(w, read=bad))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = run_gpu(g, status=status, y_fill=7.0)
    torch.cuda.synchronize()
    assert int(status.item()) == ssu.DEV_BAD_SLOT
    assert torch.all(y[2].float() == 7.0), "the skipped unit's y was written"
    assert torch.equal(g.state[int(w.dst[2])].cpu(), w.state[int(w.dst[2])])
    ok = _gpu(w)
    y_ok = run_gpu(ok)
    torch.cuda.synchronize()
    keep = [0, 1, 3, 4, 5]
    assert torch.equal(y[keep], y_ok[keep])


def test_device_status_bad_entry_and_seqlens(libssu):
    w = workloads.random_problem(17, kind="packed", slots=64, heads=4, groups=2, dim=16, dstate=64,
                                 nseq=4, max_len=3, allow_empty=False, tables="distinct")
    # num_accepted far past the table: the seed entry is outside the table
    acc = w.num_accepted.clone()
    acc[1] = 50
    g = _gpu(replace(w, num_accepted=acc))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    run_gpu(g, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == ssu.DEV_BAD_ENTRY
    # decreasing cu_seqlens
    cu = w.cu_seqlens.clone()
    cu[2] = cu[1] - 1
    g = _gpu(replace(w, cu_seqlens=cu))
    status.zero_()
    run_gpu(g, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & ssu.DEV_BAD_SEQLEN


def test_per_row_seed_past_the_sequence_is_flagged(libssu):
    """With a per-row table, num_accepted past a sequence's length would seed
    from another sequence's entry: the kernel flags BAD_ENTRY and skips that
    sequence (no y, no state written); every other sequence is unchanged."""
    w = workloads.random_problem(21, kind="packed", slots=256, heads=4, groups=2, dim=64, dstate=128, nseq=9,
                                 max_len=4, allow_empty=False, slot_mode=workloads.SLOTS_PER_ROW, tables="read",
                                 pad_frac=0.0)
    lens = w.meta["lengths"]
    b = 4
    acc = w.num_accepted.clone()
    acc[b] = lens[b] + 1
    g = _gpu(replace(w, num_accepted=acc))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = run_gpu(g, status=status, y_fill=7.0)
    ok = _gpu(w)
    y_ok = run_gpu(ok)
    torch.cuda.synchronize()
    assert int(status.item()) == ssu.DEV_BAD_ENTRY
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    rows_b = list(range(cu[b], cu[b + 1]))
    others = [r for r in range(cu[-1]) if r not in rows_b]
    assert torch.all(y[rows_b].float() == 7.0), "the skipped sequence's y was written"
    assert torch.equal(y[others], y_ok[others])
    own = [int(w.read[r]) for r in rows_b]
    assert torch.equal(g.state[own].cpu(), w.state[own]), "the skipped sequence wrote its slots"
    rest = [s for s in range(w.state.shape[0]) if s not in own]
    assert torch.equal(g.state[rest], ok.state[rest])


def test_int64_tables_and_meta(libssu):
    w = workloads.random_problem(18, kind="packed", slots=64, heads=4, groups=2, dim=16, dstate=64,
                                 nseq=5, max_len=3)
    a = _gpu(w)
    ya = run_gpu(a)
    b = _gpu(replace(w, read=w.read.long(), dst=w.dst.long(), cu_seqlens=w.cu_seqlens.long(),
                     num_accepted=w.num_accepted.long()))
    yb = run_gpu(b)
    torch.cuda.synchronize()
    assert torch.equal(ya, yb) and torch.equal(a.state, b.state)


def test_strided_inputs(libssu):
    """Non-contiguous x, dt, z, B, C views give the contiguous result bit for bit."""
    w = workloads.random_problem(19, kind="packed", slots=64, heads=4, groups=2, dim=16, dstate=64,
                                 nseq=5, max_len=3)
    a = _gpu(w)
    ya = run_gpu(a)
    wide = lambda t: torch.cat([t, torch.zeros_like(t)], dim=-1)[..., : t.shape[-1]]
    tr = lambda t: t.transpose(1, 2).contiguous().transpose(1, 2)
    b = _gpu(w)
    b = replace(b, x=wide(b.x), dt=wide(b.dt), z=wide(b.z), B=tr(b.B), C=wide(b.C))
    assert not b.x.is_contiguous() and not b.B.is_contiguous()
    yb = run_gpu(b)
    torch.cuda.synchronize()
    assert torch.equal(ya, yb) and torch.equal(a.state, b.state)


def test_repeat_runs_are_bit_identical(libssu):
    """Ten runs from the same snapshot give the same bytes (no races)."""
    w = workloads.random_problem(20, kind="packed", slots=128, heads=8, groups=2, dim=64, dstate=128,
                                 nseq=8, max_len=4, tables="read", slot_mode=workloads.SLOTS_PER_ROW)
    first = None
    for _ in range(10):
        g = _gpu(w)
        y = run_gpu(g)
        torch.cuda.synchronize()
        if first is None:
            first = (y, g.state)
        else:
            assert torch.equal(y, first[0]) and torch.equal(g.state, first[1])


def test_guard_slots_keep_their_pattern(libssu):
    """Slots nobody addresses, filled with a pattern (i % 251), stay byte-identical."""
    w = workloads.random_problem(21, kind="packed", slots=96, heads=4, groups=2, dim=16, dstate=64,
                                 nseq=4, max_len=3, state_dtype=BF16)
    pattern = (torch.arange(w.state.numel()) % 251).to(BF16).view(w.state.shape)
    used = set(w.read.reshape(-1).tolist()) | set(w.dst.reshape(-1).tolist())
    state = w.state.clone()
    guards = [s for s in range(96) if s not in used]
    state[guards] = pattern[guards]
    g = _gpu(replace(w, state=state))
    run_gpu(g)
    torch.cuda.synchronize()
    assert torch.equal(g.state[guards].cpu(), pattern[guards])


def test_graph_capture_replay(libssu):
    w = workloads.random_problem(22, kind="packed", slots=64, heads=4, groups=2, dim=64, dstate=128,
                                 nseq=4, max_len=3)
    ssu.ssu_prewarm(state_dtype=w.state.dtype, io_dtype=w.x.dtype, heads=4, dim=64, dstate=128,
                    groups=2, packed=True)
    eager = _gpu(w)
    y_eager = run_gpu(eager)
    g = _gpu(w)
    snapshot = g.state.clone()
    out = torch.empty_like(g.x)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            ssu.ssu_update_packed(g.state, g.x, g.dt, g.A, g.B, g.C, D=g.D, z=g.z, dt_bias=g.dt_bias,
                                  dt_softplus=g.dt_softplus, state_batch_indices=g.read,
                                  dst_state_batch_indices=g.dst, cu_seqlens=g.cu_seqlens,
                                  num_accepted_tokens=g.num_accepted, pad_slot_id=g.pad_slot_id,
                                  out=out)
    g.state.copy_(snapshot)        # capture does not run the kernel; start from the snapshot
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, y_eager) and torch.equal(g.state, eager.state)


def test_mate_shaped_entry_point(libssu):
    """The MATE-shaped call picks the kernel from the call shape, and arguments
    without semantics here raise NotImplementedError (MATE "Mamba / SSU",
    Stochastic rounding row)."""
    w = workloads.random_problem(23, kind="onetoken", slots=16, heads=8, groups=2, dim=8, dstate=128,
                                 nseq=2, tables="inplace", pad_frac=0.0, with_z=False, with_D=False,
                                 with_bias=False, dt_softplus=False)
    a = _gpu(w)
    y = ssu.selective_state_update(a.state, a.x, a.dt, a.A, a.B, a.C, None,
                                   state_batch_indices=a.read, dst_state_batch_indices=a.dst)
    b = _gpu(w)
    y2 = run_gpu(b)
    torch.cuda.synchronize()
    assert torch.equal(y, y2) and torch.equal(a.state, b.state)
    with pytest.raises(NotImplementedError):
        ssu.selective_state_update(a.state, a.x, a.dt, a.A, a.B, a.C, None,
                                   rand_seed=torch.zeros(1, device=DEV))
    with pytest.raises(NotImplementedError):
        ssu.selective_state_update(a.state, a.x, a.dt, a.A, a.B, a.C, None, cache_steps=2)
    # MTP form: 4-D x goes to the packed kernel
    p = workloads.random_problem(24, kind="packed", slots=64, heads=4, groups=2, dim=16, dstate=64,
                                 nseq=3, max_len=4, dense=True)
    g1 = _gpu(p)
    d4 = lambda t: None if t is None else t.view(3, 4, *t.shape[1:])
    y4 = ssu.selective_state_update(g1.state, d4(g1.x), d4(g1.dt), g1.A, d4(g1.B), d4(g1.C), g1.D,
                                    z=d4(g1.z), dt_bias=g1.dt_bias, dt_softplus=True,
                                    state_batch_indices=g1.read, dst_state_batch_indices=g1.dst,
                                    num_accepted_tokens=g1.num_accepted)
    g2 = _gpu(p)
    y_ref = run_gpu(g2)
    torch.cuda.synchronize()
    assert torch.equal(y4.view(12, *y4.shape[2:]), y_ref) and torch.equal(g1.state, g2.state)
