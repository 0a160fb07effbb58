"""The packed variable-length SSD prefill (MATE "Mamba / SSU", SSD packed
prefill; ssd_combined_fwd_varlen) on the GPU, through libssu's C ABI, against
the oracle's token recurrence.

Tolerances.  y: the chunk scan multiplies the decayed C . B^T weights as
fp16 (rounded to 2^-12 relative; x, staged as fp16 beside them, is exact),
the entering state as a bf16 high and low part (2^-17), and y itself is
stored in bf16 (2^-9).  The rounding errors of one output element add up
over the terms of its sum, which are shared by the 64 dim rows of the same
token (the same weights and entering-state rows), so the error is a small
multiple of 2^-9 times the size of that token's terms; y is held to
|d| <= 1e-2 |ref| + 1e-2 max_p |ref[t, h, :]| + 1e-3 (max over the token's
dim rows, which cancellation in one element does not make small).
States: the chunk states come from a two-part bf16 split of the
decay-weighted x (residual 2^-17 relative per term), fp32 accumulation of up
to chunk_size terms and decays exp() of fp32 sums of up to chunk_size terms;
together a few 1e-5 of the largest state magnitude, so states are held to
|d| <= 1e-4 |ref| + 1e-4 max|ref| (max over the state tensor)."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_update_gb300 as ssu
import workloads
from ssu_testlib import f64, ulp_of

pytestmark = pytest.mark.gpu
DEV = "cuda"


def assert_ssd_y_close(got, ref_exact, what="y"):
    g, r = f64(got), ref_exact.detach().cpu().numpy()
    row = np.abs(r).max(axis=-1, keepdims=True)
    d = np.abs(g - r)
    bad = d > 1e-2 * np.abs(r) + 1e-2 * row + 1e-3
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; first at {i}: "
                             f"got {g[i]!r} ref {r[i]!r} (row max {row[i[:-1]][0]:.3g}, max |d| {d.max():.3g})")


def assert_ssd_states_close(got, ref, what="states"):
    assert got.dtype == ref.dtype and got.shape == ref.shape, (got.dtype, ref.dtype, got.shape, ref.shape)
    g, r = f64(got), f64(ref)
    scale = np.abs(r).max() if r.size else 0.0
    d = np.abs(g - r)
    tol = 1e-4 * np.abs(r) + 1e-4 * scale
    if got.dtype != torch.float32:  # 16-bit states: one unit in the last place on top
        tol = tol + ulp_of(np.maximum(np.abs(g), np.abs(r)), got.dtype)
    bad = d > tol
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} out of tolerance; first at {i}: "
                             f"got {g[i]!r} ref {r[i]!r} (max |d| {d.max():.3g}, scale {scale:.3g})")


def run_gpu_ssd(w, intermediate=False, status=None, seq_idx=None):
    g = w.to(DEV)
    y, states = ssu.ssu_ssd_prefill(g.x, g.dt, g.A, g.B, g.C, g.chunk_size, g.cu_chunk_seqlens,
                                    g.seq_idx if seq_idx is None else seq_idx.to(DEV), g.last_chunk_indices,
                                    D=g.D, z=g.z, dt_bias=g.dt_bias, dt_softplus=g.dt_softplus,
                                    dt_limit=g.dt_limit, initial_states=g.initial_states,
                                    return_intermediate_states=intermediate, state_dtype=g.state_dtype,
                                    nseq=w.nseq, status=status)
    torch.cuda.synchronize()
    return y, states


def run_oracle_ssd(w, seq_idx=None):
    return oracle.ssd(w.x, w.dt, w.A, w.B, w.C, w.cu_chunk_seqlens, w.seq_idx if seq_idx is None else seq_idx,
                      w.nseq, D=w.D, z=w.z, dt_bias=w.dt_bias, dt_softplus=w.dt_softplus, dt_limit=w.dt_limit,
                      initial_states=w.initial_states, state_dtype=w.state_dtype)


def check(w, intermediate=False):
    ref = run_oracle_ssd(w)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y, states = run_gpu_ssd(w, intermediate, status)
    assert int(status.item()) == 0
    assert_ssd_y_close(y, ref.y_exact)
    want = ref.states if intermediate else ref.states[w.last_chunk_indices.long()]
    assert_ssd_states_close(states, want)


@pytest.mark.parametrize("chunk_size", [64, 128, 256])
@pytest.mark.parametrize("dstate", [64, 128])
def test_ssd_against_oracle(libssu, chunk_size, dstate):
    lengths = [1, chunk_size - 1, chunk_size, chunk_size + 1, 2 * chunk_size + 37, 300]
    w = workloads.ssd_problem(200 + chunk_size + dstate, lengths, heads=4, dim=64, dstate=dstate, groups=2,
                              chunk_size=chunk_size)
    check(w)


def test_ssd_intermediate_states(libssu):
    w = workloads.ssd_problem(210, [130, 5, 257], heads=4, dim=64, dstate=128, groups=2, chunk_size=64)
    check(w, intermediate=True)


@pytest.mark.parametrize("flags", [dict(with_init=False), dict(with_z=False, with_D=False, with_bias=False),
                                   dict(dt_softplus=False), dict(dt_limit=(0.2, 0.6))])
def test_ssd_flags(libssu, flags):
    w = workloads.ssd_problem(220, [70, 200, 33], heads=4, dim=64, dstate=64, groups=1, chunk_size=64, **flags)
    check(w)


@pytest.mark.parametrize("state_dtype", [torch.float16, torch.bfloat16])
def test_ssd_16bit_states(libssu, state_dtype):
    w = workloads.ssd_problem(230, [100, 160], heads=4, dim=64, dstate=128, groups=2, chunk_size=64,
                              state_dtype=state_dtype)
    check(w)


def test_ssd_seq_idx_is_the_authority(libssu):
    """Re-labelling a chunk as the next sequence's makes it open from that
    sequence's initial state on the GPU as in the oracle."""
    w = workloads.ssd_problem(240, [150, 150], heads=4, dim=64, dstate=64, groups=2, chunk_size=64)
    relabel = w.seq_idx.clone()
    relabel[2] = 1
    ref = run_oracle_ssd(w, relabel)
    y, states = run_gpu_ssd(w, intermediate=True, seq_idx=relabel)
    assert_ssd_y_close(y, ref.y_exact)
    assert_ssd_states_close(states, ref.states)


def test_ssd_many_heads_and_groups(libssu):
    w = workloads.ssd_problem(250, [97, 256, 511], heads=16, dim=64, dstate=128, groups=4, chunk_size=128)
    check(w)


def test_ssd_full_size_sampled_heads(libssu):
    """The 16k-token prefill workload (heads 128, groups 8, chunk 256) in one
    call; heads 0, 77 and 127 checked against the oracle run on those heads
    alone (each with its group's B and C)."""
    w = workloads.ssd_prefill_16k_bf16()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y, states = run_gpu_ssd(w, status=status)
    assert int(status.item()) == 0
    hpg = 128 // 8
    for h in (0, 77, 127):
        g = h // hpg
        sub = workloads.SsdWorkload(
            "sub", w.x[:, h:h + 1].contiguous(), w.dt[:, h:h + 1].contiguous(), w.A[h:h + 1],
            w.B[:, g:g + 1].contiguous(), w.C[:, g:g + 1].contiguous(), w.cu_seqlens, w.cu_chunk_seqlens,
            w.seq_idx, w.last_chunk_indices, w.chunk_size, D=w.D[h:h + 1], z=w.z[:, h:h + 1].contiguous(),
            dt_bias=w.dt_bias[h:h + 1], dt_softplus=w.dt_softplus, dt_limit=w.dt_limit,
            initial_states=w.initial_states[:, h:h + 1].contiguous(), state_dtype=w.state_dtype)
        ref = run_oracle_ssd(sub)
        assert_ssd_y_close(y[:, h:h + 1].cpu(), ref.y_exact, what=f"y head {h}")
        assert_ssd_states_close(states[:, h:h + 1], ref.states[w.last_chunk_indices.long()], what=f"states head {h}")


def test_ssd_unsupported_shapes_raise(libssu):
    w = workloads.ssd_problem(260, [10], heads=2, dim=32, dstate=64, groups=1, chunk_size=64).to(DEV)
    with pytest.raises(NotImplementedError):
        ssu.ssu_ssd_prefill(w.x, w.dt, w.A, w.B, w.C, 64, w.cu_chunk_seqlens, w.seq_idx, w.last_chunk_indices)


def test_ssd_malformed_chunks_are_flagged(libssu):
    """A chunk longer than chunk_size, a seq_idx past nseq and a
    last_chunk_indices entry past nchunks each set their status bit; the
    well-formed chunks before them are still computed."""
    w = workloads.ssd_problem(270, [64, 64, 64], heads=4, dim=64, dstate=64, groups=2, chunk_size=64)
    ref = run_oracle_ssd(w)
    g = w.to(DEV)
    for name, edit, bit in [("cu_chunk_seqlens", lambda t: t.copy_(torch.tensor([0, 64, 64, 192], dtype=t.dtype)),
                             ssu.DEV_BAD_SEQLEN),
                            ("seq_idx", lambda t: t.copy_(torch.tensor([0, 1, 7], dtype=t.dtype)), ssu.DEV_BAD_ENTRY),
                            ("last_chunk_indices", lambda t: t.copy_(torch.tensor([0, 1, 9], dtype=t.dtype)),
                             ssu.DEV_BAD_ENTRY)]:
        args = {k: getattr(g, k).clone() for k in ("cu_chunk_seqlens", "seq_idx", "last_chunk_indices")}
        edit(args[name])
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        y, _ = ssu.ssu_ssd_prefill(g.x, g.dt, g.A, g.B, g.C, 64, args["cu_chunk_seqlens"], args["seq_idx"],
                                   args["last_chunk_indices"], D=g.D, z=g.z, dt_bias=g.dt_bias,
                                   dt_softplus=g.dt_softplus, initial_states=g.initial_states, nseq=3,
                                   status=status)
        torch.cuda.synchronize()
        assert int(status.item()) & bit, name
        assert_ssd_y_close(y[:64], ref.y_exact[:64], what=f"y of chunk 0 with a bad {name}")


def test_ssd_combined_fwd_varlen_signature(libssu):
    """The MATE-shaped call writes y into ``out`` and returns the states."""
    w = workloads.ssd_problem(280, [90, 40], heads=4, dim=64, dstate=128, groups=2, chunk_size=128)
    ref = run_oracle_ssd(w)
    g = w.to(DEV)
    out = torch.empty_like(g.x)
    states = ssu.ssd_combined_fwd_varlen(g.x, g.dt, g.A, g.B, g.C, 128, g.cu_seqlens, g.cu_chunk_seqlens,
                                         g.last_chunk_indices, g.seq_idx, out=out, D=g.D, z=g.z,
                                         dt_bias=g.dt_bias, dt_softplus=True, initial_states=g.initial_states)
    torch.cuda.synchronize()
    assert_ssd_y_close(out, ref.y_exact)
    assert_ssd_states_close(states, ref.states[w.last_chunk_indices.long()])
    with pytest.raises(NotImplementedError):
        ssu.ssd_combined_fwd_varlen(g.x, g.dt, g.A, g.B, g.C, 128, g.cu_seqlens, g.cu_chunk_seqlens,
                                    g.last_chunk_indices, g.seq_idx, checkpoint_states=g.initial_states)


@pytest.mark.parametrize("scale_x,scale_bc,dt_shift", [(1e5, 1.0, 0.0), (1e-7, 1.0, 0.0), (1.0, 40.0, 3.0),
                                                      (3e4, 20.0, 0.0)])
def test_ssd_operands_outside_fp16_range(libssu, scale_x, scale_bc, dt_shift):
    """x beyond fp16's largest value (65504) or deep in its subnormal range,
    and weights (C . B^T) dt' beyond 65504: the scan stages its fp16
    operands with power-of-two scales picked per chunk and head, so y and the
    states match the oracle relative to their own size."""
    w = workloads.ssd_problem(290, [200, 77], heads=4, dim=64, dstate=128, groups=2, chunk_size=128)
    w.x = (w.x.float() * scale_x).to(w.x.dtype)
    w.B = (w.B.float() * scale_bc).to(w.B.dtype)
    w.C = (w.C.float() * scale_bc).to(w.C.dtype)
    w.dt = w.dt + dt_shift
    ref = run_oracle_ssd(w)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y, states = run_gpu_ssd(w, status=status)
    assert int(status.item()) == 0
    k = 1.0 / float(ref.y_exact.abs().max())
    assert_ssd_y_close(y.double().cpu() * k, ref.y_exact * k, what=f"y / {1 / k:.3g}")
    assert_ssd_states_close(states, ref.states[w.last_chunk_indices.long()])


@pytest.mark.parametrize("chunk_size,dstate,lengths", [(64, 128, [130, 64, 255, 1, 77]), (256, 128, [300, 513, 77]),
                                                       (128, 64, [129, 400, 3, 250])])
def test_ssd_scan_ranges_cross_chunks_and_groups(libssu, chunk_size, dstate, lengths):
    """More (chunk, group, head) units than SMs: each CTA of the scan takes a
    contiguous range that starts and ends inside a group's heads and crosses
    into the next group or chunk, whose C . B^T it computes afresh."""
    w = workloads.ssd_problem(300 + chunk_size, lengths, heads=32, dim=64, dstate=dstate, groups=2,
                              chunk_size=chunk_size)
    assert int(w.seq_idx.numel()) * 32 > torch.cuda.get_device_properties(0).multi_processor_count
    check(w)
