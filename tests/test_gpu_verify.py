"""Speculative decoding on the checkpoint + buffer form (article "ReplaySSM",
section 投机解码回滚) on the GPU through libssu's C ABI, against the oracle:
the drafts' outputs, the flush one window early, the appended entries and
the committed count; and rollback -- a verify followed by a plain replay
step from count_out + a equals the same on the oracle."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_update_gb300 as ssu
import workloads
from gpu_harness import DEV
from ssu_testlib import STATE_F32_ATOL, STATE_F32_RTOL, assert_state_close, assert_y_close, f64

pytestmark = pytest.mark.gpu


def run_verify_gpu(w, status=None):
    g = w.to(DEV)
    y, cnt = ssu.ssu_replay_verify(g.state, g.x, g.dt, g.A, g.B, g.C, g.xbuf, g.dtbuf, g.Bbuf, g.count, D=g.D,
                                   z=g.z, dt_bias=g.dt_bias, dt_softplus=g.dt_softplus,
                                   state_batch_indices=g.read, pad_slot_id=g.pad_slot_id, status=status)
    torch.cuda.synchronize()
    return g, y, cnt


def run_verify_oracle(w):
    return oracle.replay_verify(w.state, w.x, w.dt, w.A, w.B, w.C, w.xbuf, w.dtbuf, w.Bbuf, w.count, D=w.D, z=w.z,
                                dt_bias=w.dt_bias, dt_softplus=w.dt_softplus, slot_of=w.read,
                                pad_slot_id=w.pad_slot_id)


def check_against_oracle(w):
    ref = run_verify_oracle(w)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    g, y, cnt = run_verify_gpu(w, status)
    assert int(status.item()) == 0
    assert_y_close(y, ref.y_exact)
    assert torch.equal(cnt.cpu().long(), ref.count)
    L, T = w.xbuf.shape[1], w.x.shape[1]
    flushed = torch.zeros(w.state.shape[0], dtype=torch.bool)
    for b in range(w.nseq):
        s = b if w.read is None else int(w.read[b])
        if s != w.pad_slot_id and int(w.count[b]) + 2 * T >= L:
            flushed[s] = True
    got = g.state.cpu()
    assert torch.equal(got[~flushed], w.state[~flushed]), "a checkpoint without a flush changed"
    if flushed.any():
        assert_state_close(got[flushed], ref.ckpt[flushed], what="flushed checkpoint")
    assert torch.equal(g.xbuf.cpu(), ref.xbuf), "x buffer"
    assert torch.equal(g.Bbuf.cpu(), ref.Bbuf), "B buffer"
    d, r = f64(g.dtbuf), f64(ref.dtbuf)
    assert np.all(np.abs(d - r) <= STATE_F32_RTOL * np.abs(r) + STATE_F32_ATOL), "dt buffer"
    return g, y, cnt, ref


@pytest.mark.parametrize("buffer_len,ntok", [(4, 1), (4, 2), (8, 1), (8, 3), (16, 4), (16, 8), (5, 5)])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_verify_against_oracle(libssu, buffer_len, ntok, state_dtype):
    w = workloads.verify_problem(300 + 7 * buffer_len + ntok, ntok=ntok, buffer_len=buffer_len, nseq=9,
                                 slots=24, state_dtype=state_dtype)
    check_against_oracle(w)


@pytest.mark.parametrize("dstate,dim", [(16, 8), (32, 64), (64, 100), (128, 64), (256, 130)])
def test_verify_shapes(libssu, dstate, dim):
    w = workloads.verify_problem(320 + dstate + dim, ntok=3, buffer_len=8, nseq=5, slots=12, heads=4,
                                 dim=dim, dstate=dstate, groups=2)
    check_against_oracle(w)


@pytest.mark.parametrize("io_dtype", [torch.float16, torch.float32])
@pytest.mark.parametrize("flags", [dict(with_z=False, with_D=False), dict(dt_softplus=False, with_bias=False)])
def test_verify_io_and_flags(libssu, io_dtype, flags):
    w = workloads.verify_problem(330, ntok=2, buffer_len=6, nseq=6, slots=16, io_dtype=io_dtype, **flags)
    check_against_oracle(w)


def test_verify_no_table_per_head_dt(libssu):
    """No slot table (sequence b uses slot b) and one step per head ([batch,
    T, heads] dt, broadcast over dim)."""
    w = workloads.verify_problem(340, ntok=2, buffer_len=8, nseq=6, slots=6, tables=False)
    w.dt = w.dt[..., 0].contiguous()
    check_against_oracle(w)


def test_rollback_then_step(libssu):
    """Verify, accept a prefix per sequence (count = count_out + a), then one
    plain replay step: y, checkpoints and buffers equal the oracle's run of
    the same two calls."""
    w = workloads.verify_problem(350, ntok=4, buffer_len=16, nseq=8, slots=20, pad_frac=0.0)
    g, y, cnt, ref = check_against_oracle(w)
    acc = torch.tensor([0, 1, 2, 3, 4, 4, 1, 0], dtype=torch.int32)
    nxt = workloads.replay_problem(351, buffer_len=16, nseq=8, slots=20, pad_frac=0.0)
    count2 = ref.count.to(torch.int32) + acc
    step_ref = oracle.replay(ref.ckpt, nxt.x, nxt.dt, w.A, nxt.B, nxt.C, ref.xbuf, ref.dtbuf, ref.Bbuf, count2,
                             D=w.D, z=nxt.z, dt_bias=w.dt_bias, dt_softplus=w.dt_softplus, slot_of=w.read,
                             pad_slot_id=w.pad_slot_id)
    n = nxt.to(DEV)
    y2, cnt2 = ssu.ssu_replay_update(g.state, n.x, n.dt, g.A, n.B, n.C, g.xbuf, g.dtbuf, g.Bbuf,
                                     (cnt + acc.to(DEV)).contiguous(), D=g.D, z=n.z, dt_bias=g.dt_bias,
                                     dt_softplus=g.dt_softplus, state_batch_indices=g.read,
                                     pad_slot_id=g.pad_slot_id)
    torch.cuda.synchronize()
    assert_y_close(y2, step_ref.y_exact, what="the step after the rollback")
    assert torch.equal(cnt2.cpu().long(), step_ref.count)
    assert_state_close(g.state.cpu(), step_ref.ckpt, what="checkpoints after the step")


def test_bad_count_sets_status(libssu):
    w = workloads.verify_problem(360, ntok=2, buffer_len=4, nseq=4, slots=8, pad_frac=0.0)
    w.count[1] = 4  # outside [0, L)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    run_verify_gpu(w, status)
    assert int(status.item()) & ssu.DEV_BAD_COUNT


def test_ntok_beyond_buffer_raises(libssu):
    w = workloads.verify_problem(361, ntok=5, buffer_len=4, nseq=2, slots=4).to(DEV)
    with pytest.raises(ValueError):
        ssu.ssu_replay_verify(w.state, w.x, w.dt, w.A, w.B, w.C, w.xbuf, w.dtbuf, w.Bbuf, w.count,
                              state_batch_indices=w.read, pad_slot_id=w.pad_slot_id)
