"""The checkpoint + buffer form of the decode state (article "ReplaySSM: Cache
SSM Inputs, Not State", section 核心做法) on the GPU, through libssu's C ABI:
against the oracle element by element, L = 1 against the plain one-token
kernel bit for bit, L steps against L plain steps, and the full-size batch-256
workload on sampled sequences."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import selective_state_update_gb300 as ssu
import workloads
from gpu_harness import DEV, run_gpu
from ssu_testlib import (STATE_F32_ATOL, STATE_F32_RTOL, assert_e4m3_codes_close, assert_nvfp4_close,
                         assert_state_close, assert_y_close, f64)

pytestmark = pytest.mark.gpu


def run_replay_gpu(w, status=None):
    g = w.to(DEV)
    y, cnt = ssu.ssu_replay_update(g.state, g.x, g.dt, g.A, g.B, g.C, g.xbuf, g.dtbuf, g.Bbuf, g.count, D=g.D,
                                   z=g.z, dt_bias=g.dt_bias, dt_softplus=g.dt_softplus,
                                   state_batch_indices=g.read, pad_slot_id=g.pad_slot_id, status=status)
    torch.cuda.synchronize()
    return g, y, cnt


def run_replay_oracle(w):
    return oracle.replay(w.state, w.x, w.dt, w.A, w.B, w.C, w.xbuf, w.dtbuf, w.Bbuf, w.count, D=w.D, z=w.z,
                         dt_bias=w.dt_bias, dt_softplus=w.dt_softplus, slot_of=w.read, pad_slot_id=w.pad_slot_id)


def check_against_oracle(w):
    ref = run_replay_oracle(w)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    g, y, cnt = run_replay_gpu(w, status)
    assert int(status.item()) == 0
    assert_y_close(y, ref.y_exact)
    assert torch.equal(cnt.cpu().long(), ref.count)
    written = torch.zeros(w.state.shape[0], dtype=torch.bool)
    L = w.xbuf.shape[1]
    for b in range(w.nseq):
        s = b if w.read is None else int(w.read[b])
        if s != w.pad_slot_id and int(w.count[b]) + 1 == L:
            written[s] = True
    got = g.state.cpu()
    assert torch.equal(got[~written], w.state[~written]), "a checkpoint that does not fold changed"
    if written.any():
        assert_state_close(got[written], ref.ckpt[written], what="folded checkpoint")
    assert torch.equal(g.xbuf.cpu(), ref.xbuf), "x buffer"
    assert torch.equal(g.Bbuf.cpu(), ref.Bbuf), "B buffer"
    d, r = f64(g.dtbuf), f64(ref.dtbuf)
    assert np.all(np.abs(d - r) <= STATE_F32_RTOL * np.abs(r) + STATE_F32_ATOL), "dt buffer"
    return g, y


@pytest.mark.parametrize("buffer_len", [1, 2, 5, 16])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_replay_against_oracle(libssu, buffer_len, state_dtype):
    w = workloads.replay_problem(10 + buffer_len, slots=40, heads=4, groups=2, dim=16, dstate=64, nseq=12,
                                 buffer_len=buffer_len, state_dtype=state_dtype)
    check_against_oracle(w)


@pytest.mark.parametrize("dstate", [16, 32, 128, 256])
@pytest.mark.parametrize("dim", [8, 64, 100])
def test_replay_shapes(libssu, dstate, dim):
    w = workloads.replay_problem(20 + dstate + dim, slots=24, heads=6, groups=3, dim=dim, dstate=dstate, nseq=5,
                                 buffer_len=6)
    check_against_oracle(w)


@pytest.mark.parametrize("io_dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("flags", [(True, True, True, True), (False, False, False, False), (True, False, True, False)])
def test_replay_io_and_flags(libssu, io_dtype, flags):
    with_D, with_z, with_bias, softplus = flags
    w = workloads.replay_problem(30, slots=32, heads=4, groups=1, dim=16, dstate=128, nseq=8, buffer_len=4,
                                 io_dtype=io_dtype, with_D=with_D, with_z=with_z, with_bias=with_bias,
                                 dt_softplus=softplus)
    check_against_oracle(w)


@pytest.mark.parametrize("state_dtype,io_dtype,buffer_len", [
    (torch.float32, torch.bfloat16, 7), (torch.bfloat16, torch.bfloat16, 16), (torch.float32, torch.float32, 32),
    (torch.float16, torch.float32, 3)])
def test_replay_many_units_per_cta(libssu, state_dtype, io_dtype, buffer_len):
    """Far more (sequence, head, dim tile) units than resident CTAs, so each
    CTA walks many units through its ring of stages, folding and non-folding
    units interleaved; two dim tiles per head."""
    w = workloads.replay_problem(40 + buffer_len, slots=96, heads=24, groups=4, dim=128, dstate=64, nseq=80,
                                 buffer_len=buffer_len, state_dtype=state_dtype, io_dtype=io_dtype, pad_frac=0.1)
    check_against_oracle(w)


def test_replay_largest_stage(libssu):
    """fp32 checkpoints of dstate 256 with the longest fp32 buffers: the
    largest stage, a ring of one stage."""
    w = workloads.replay_problem(41, slots=40, heads=8, groups=2, dim=64, dstate=256, nseq=36, buffer_len=32,
                                 state_dtype=torch.float32, io_dtype=torch.float32, pad_frac=0.1)
    check_against_oracle(w)


def test_replay_no_table_and_pad_zero(libssu):
    check_against_oracle(workloads.replay_problem(31, slots=6, nseq=6, tables=False, buffer_len=3))
    check_against_oracle(workloads.replay_problem(32, slots=20, nseq=8, pad_slot_id=0, pad_frac=0.3))


def test_buffer_len_one_is_the_plain_step_bitwise(libssu):
    """L = 1: every step folds and equals the one-token kernel writing back to
    the read slot, bit for bit (the article's anchor)."""
    w = workloads.replay_problem(33, slots=48, heads=8, groups=2, dim=64, dstate=128, nseq=16, buffer_len=1)
    g, y, cnt = run_replay_gpu(w)
    p = replace(w, kind="onetoken", dst=w.read.clone()).to(DEV)
    y_plain = run_gpu(p)
    torch.cuda.synchronize()
    assert torch.equal(y, y_plain) and torch.equal(g.state, p.state)
    assert int(cnt.abs().sum()) == 0


def test_l_steps_equal_l_plain_steps(libssu):
    """From empty buffers, L steps on the checkpoint + buffer form fold into
    exactly the fp32 state L plain steps produce (bit for bit); the folding
    step's y is bit-identical and the others agree within the output
    tolerance."""
    L, nseq = 6, 10
    base = workloads.replay_problem(34, slots=32, heads=4, groups=2, dim=64, dstate=128, nseq=nseq, buffer_len=L,
                                    pad_frac=0.0)
    gen = torch.Generator().manual_seed(77)
    steps = []
    for t in range(L):
        steps.append(dict(x=torch.randn(base.x.shape, generator=gen).to(base.x.dtype),
                          dt=torch.randn(base.dt.shape, generator=gen),
                          z=torch.randn(base.z.shape, generator=gen).to(base.z.dtype),
                          B=torch.randn(base.B.shape, generator=gen).to(base.B.dtype),
                          C=torch.randn(base.C.shape, generator=gen).to(base.C.dtype)))
    rep = replace(base, count=torch.zeros(nseq, dtype=torch.int32)).to(DEV)
    plain = replace(base, kind="onetoken", dst=base.read.clone()).to(DEV)
    for t, inp in enumerate(steps):
        r = replace(rep, **{k: v.to(DEV) for k, v in inp.items()})
        y_r, cnt = ssu.ssu_replay_update(r.state, r.x, r.dt, r.A, r.B, r.C, r.xbuf, r.dtbuf, r.Bbuf, r.count,
                                         D=r.D, z=r.z, dt_bias=r.dt_bias, dt_softplus=r.dt_softplus,
                                         state_batch_indices=r.read)
        rep = replace(rep, count=cnt)
        pl = replace(plain, **{k: v.to(DEV) for k, v in inp.items()})
        y_p = run_gpu(pl)
        torch.cuda.synchronize()
        if t + 1 < L:
            assert_y_close(y_r, y_p.cpu().double())
            assert int(cnt.cpu().sum()) == (t + 1) * nseq
        else:
            assert torch.equal(y_r, y_p)
            assert torch.equal(rep.state, plain.state), "folded checkpoint differs from the plain steps"
            assert int(cnt.cpu().abs().sum()) == 0


def test_bad_count_sets_status(libssu):
    w = workloads.replay_problem(35, slots=20, nseq=4, buffer_len=4, pad_frac=0.0)
    w.count[2] = 9
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    run_replay_gpu(w, status)
    assert int(status.item()) == ssu.DEV_BAD_COUNT


def test_replay_b256_sampled(libssu):
    """The full-size batch-256 workload: sampled sequences against the oracle
    (compact copies of their slots), the rest by properties: checkpoints of
    sequences that do not fold are unchanged, counts advance."""
    w = workloads.replay_b256_fp32()
    L = w.meta["buffer_len"]
    g = w.to(DEV)
    before = g.state.clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y, cnt = ssu.ssu_replay_update(g.state, g.x, g.dt, g.A, g.B, g.C, g.xbuf, g.dtbuf, g.Bbuf, g.count, D=g.D,
                                   z=g.z, dt_bias=g.dt_bias, dt_softplus=True, state_batch_indices=g.read,
                                   pad_slot_id=g.pad_slot_id, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    expect = torch.where((w.count + 1 == L) | (w.read == w.pad_slot_id), 0, w.count + 1)
    assert torch.equal(cnt.cpu(), expect.to(torch.int32))
    fold_slots = [int(w.read[b]) for b in range(w.nseq) if int(w.read[b]) != 0 and int(w.count[b]) + 1 == L]
    keep = torch.ones(w.state.shape[0], dtype=torch.bool, device=DEV)
    keep[torch.tensor(fold_slots, device=DEV)] = False
    assert torch.equal(before[keep], g.state[keep])
    del before
    sample = [b for b in range(w.nseq) if int(w.count[b]) + 1 == L][:6] + [0, 1, 2, 3, 100, 200]
    sample += [b for b in range(w.nseq) if int(w.read[b]) == 0][:3]
    sample = sorted(set(sample))
    slots = [int(w.read[b]) for b in sample]
    order = [0] + sorted(set(s for s in slots if s != 0))
    m = {s: i for i, s in enumerate(order)}
    idx = torch.tensor(order)
    sub = replace(w, state=w.state[idx], xbuf=w.xbuf[idx], dtbuf=w.dtbuf[idx], Bbuf=w.Bbuf[idx],
                  read=torch.tensor([m[s] if s != 0 else 0 for s in slots], dtype=torch.int32),
                  count=w.count[sample], x=w.x[sample], dt=w.dt[sample], z=w.z[sample], B=w.B[sample],
                  C=w.C[sample])
    ref = run_replay_oracle(sub)
    assert_y_close(y[sample].cpu(), ref.y_exact, what="y (sampled)")
    for i, b in enumerate(sample):
        s = slots[i]
        if s != 0 and int(w.count[b]) + 1 == L:
            assert_state_close(g.state[s].cpu(), ref.ckpt[m[s]], what="folded checkpoint (sampled)")
        if s != 0 and int(w.count[b]) + 1 < L:
            c = int(w.count[b])
            assert torch.equal(g.xbuf[s, c].cpu(), ref.xbuf[m[s], c])


# ---------------------------------------------------------------------------
# The low-precision read copy (article "ReplaySSM", section 低精度读写分离).
# ---------------------------------------------------------------------------
_FMT = {"f16": (oracle.SHADOW_F16, torch.float16), "e4m3": (oracle.SHADOW_E4M3, torch.uint8),
        "nvfp4": (oracle.SHADOW_NVFP4, torch.uint8)}


@pytest.mark.parametrize("fmt", ["f16", "e4m3", "nvfp4"])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.float16, torch.bfloat16])
def test_shadow_refresh_is_the_oracles(libssu, fmt, state_dtype):
    """The GPU's read copy of a pool equals the oracle's: fp16 bit for bit;
    E4M3 row scales bit for bit and codes equal except one step at a tie of
    the fp32 quotient (assert_e4m3_codes_close); NVFP4 row scales bit for
    bit, block and element codes the nearest except one step at such a tie
    (assert_nvfp4_close)."""
    code, dtype = _FMT[fmt]
    g = torch.Generator().manual_seed(70)
    st = (torch.randn((5, 3, 20, 128), generator=g) * torch.rand((5, 3, 20, 1), generator=g) * 3).to(state_dtype)
    st[2, 1, 7] = 0
    st[3, 0, 4, 32:48] *= 1e-6  # a block far below its row's largest
    want, want_scale = oracle.shadow_refresh(st, code)
    if fmt == "nvfp4":
        sh = torch.zeros((*st.shape[:-1], 64), dtype=torch.uint8, device=DEV)
        sc = torch.zeros((*st.shape[:-1], ssu.nvfp4_scale_words(128)), dtype=torch.float32, device=DEV)
    else:
        sh = torch.empty(st.shape, dtype=dtype, device=DEV)
        sc = torch.empty(st.shape[:-1], dtype=torch.float32, device=DEV) if fmt == "e4m3" else None
    ssu.ssu_shadow_refresh(st.to(DEV), sh, sc)
    torch.cuda.synchronize()
    if fmt == "nvfp4":
        assert_nvfp4_close(sh, sc, st)
    elif fmt == "e4m3":
        assert torch.equal(sc.cpu(), want_scale)
        assert_e4m3_codes_close(sh, want, st)
    else:
        assert torch.equal(sh.cpu().view(want.dtype), want)


def _check_read_copy(w, fmt):
    code, dtype = _FMT[fmt]
    sh0, sc0 = oracle.shadow_refresh(w.state, code)
    ref = oracle.replay(w.state, w.x, w.dt, w.A, w.B, w.C, w.xbuf, w.dtbuf, w.Bbuf, w.count, D=w.D, z=w.z,
                        dt_bias=w.dt_bias, dt_softplus=w.dt_softplus, slot_of=w.read, pad_slot_id=w.pad_slot_id,
                        shadow=sh0, shadow_scale=sc0, shadow_format=code)
    g = w.to(DEV)
    sh = sh0.to(DEV).view(dtype)
    sc = None if sc0 is None else sc0.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y, cnt = ssu.ssu_replay_update(g.state, g.x, g.dt, g.A, g.B, g.C, g.xbuf, g.dtbuf, g.Bbuf, g.count, D=g.D,
                                   z=g.z, dt_bias=g.dt_bias, dt_softplus=g.dt_softplus, state_batch_indices=g.read,
                                   pad_slot_id=g.pad_slot_id, status=status, shadow=sh, shadow_scale=sc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_y_close(y, ref.y_exact)
    assert torch.equal(cnt.cpu().long(), ref.count)
    L = w.xbuf.shape[1]
    got = g.state.cpu()
    folded = [int(w.read[b]) if w.read is not None else b for b in range(w.nseq)
              if (int(w.read[b]) if w.read is not None else b) != w.pad_slot_id and int(w.count[b]) + 1 == L]
    keep = torch.ones(w.state.shape[0], dtype=torch.bool)
    keep[folded] = False
    assert torch.equal(got[keep], w.state[keep])
    if folded:
        assert_state_close(got[folded], ref.ckpt[folded], what="folded checkpoint")
    # the read copy: untouched where nothing folds; where a slot folds, the
    # copy of the checkpoint the GPU wrote (same decisions, same fp32 values)
    sh_got = sh.cpu().view(sh0.dtype)
    assert torch.equal(sh_got[keep], sh0[keep]), "a read copy changed without a fold"
    if folded:
        want, want_scale = oracle.shadow_refresh(got[folded], code)
        if fmt == "nvfp4":
            assert_nvfp4_close(sh_got[folded], sc.cpu()[folded], got[folded], "a fold's NVFP4 read copy")
        elif fmt == "e4m3":
            assert_e4m3_codes_close(sh_got[folded], want, got[folded], "a fold's read copy")
        else:
            assert torch.equal(sh_got[folded], want), "a fold's read copy differs from the copy of its checkpoint"
        if fmt == "e4m3":
            assert torch.equal(sc.cpu()[folded], want_scale)
    if sc is not None:
        assert torch.equal(sc.cpu()[keep], sc0[keep])
    assert torch.equal(g.xbuf.cpu(), ref.xbuf) and torch.equal(g.Bbuf.cpu(), ref.Bbuf)


@pytest.mark.parametrize("fmt", ["f16", "e4m3", "nvfp4"])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("buffer_len", [1, 3, 16])
def test_replay_read_copy_against_oracle(libssu, fmt, state_dtype, buffer_len):
    w = workloads.replay_problem(80 + buffer_len, slots=40, heads=4, groups=2, dim=16, dstate=64, nseq=12,
                                 buffer_len=buffer_len, state_dtype=state_dtype)
    _check_read_copy(w, fmt)


@pytest.mark.parametrize("fmt", ["f16", "e4m3", "nvfp4"])
@pytest.mark.parametrize("dstate,dim", [(16, 8), (128, 100), (256, 64)])
def test_replay_read_copy_shapes(libssu, fmt, dstate, dim):
    if fmt == "e4m3" and dim % 4:
        pytest.skip("E4M3 row scales need dim % 4 == 0")
    if fmt == "nvfp4" and dstate < 64:
        pytest.skip("an NVFP4 read copy needs dstate 64, 128 or 256")
    w = workloads.replay_problem(90 + dstate + dim, slots=24, heads=6, groups=3, dim=dim, dstate=dstate, nseq=5,
                                 buffer_len=5)
    _check_read_copy(w, fmt)


@pytest.mark.parametrize("fmt", ["f16", "e4m3", "nvfp4"])
def test_replay_read_copy_many_units(libssu, fmt):
    w = workloads.replay_problem(95, slots=96, heads=24, groups=4, dim=128, dstate=64, nseq=80, buffer_len=7,
                                 pad_frac=0.1)
    _check_read_copy(w, fmt)


def test_read_copy_e4m3_needs_dim_multiple_of_4(libssu):
    w = workloads.replay_problem(96, slots=8, heads=2, groups=1, dim=6, dstate=32, nseq=2, buffer_len=2).to(DEV)
    sh = torch.zeros(w.state.shape, dtype=torch.uint8, device=DEV)
    sc = torch.ones(w.state.shape[:-1], dtype=torch.float32, device=DEV)
    with pytest.raises(NotImplementedError):
        ssu.ssu_replay_update(w.state, w.x, w.dt, w.A, w.B, w.C, w.xbuf, w.dtbuf, w.Bbuf, w.count, D=w.D,
                              z=w.z, state_batch_indices=w.read, shadow=sh, shadow_scale=sc)


def test_read_copy_nvfp4_needs_dstate_64_to_256(libssu):
    w = workloads.replay_problem(97, slots=8, heads=2, groups=1, dim=8, dstate=32, nseq=2, buffer_len=2).to(DEV)
    sh = torch.zeros((*w.state.shape[:-1], 16), dtype=torch.uint8, device=DEV)
    sc = torch.zeros((*w.state.shape[:-1], ssu.nvfp4_scale_words(32)), dtype=torch.float32, device=DEV)
    with pytest.raises(NotImplementedError):
        ssu.ssu_replay_update(w.state, w.x, w.dt, w.A, w.B, w.C, w.xbuf, w.dtbuf, w.Bbuf, w.count, D=w.D,
                              z=w.z, state_batch_indices=w.read, shadow=sh, shadow_scale=sc)
