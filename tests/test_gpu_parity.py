"""GPU vs oracle, element by element, on small seeded problems that span
several dim tiles and a ragged tail, across dtypes, dstate sizes, table forms
and flags.  Every call goes through libssu's C ABI."""
import itertools

import pytest
import torch

import workloads
from gpu_harness import full_check

pytestmark = pytest.mark.gpu

F32, F16, BF16 = torch.float32, torch.float16, torch.bfloat16


@pytest.mark.parametrize("state_dtype", [F32, F16, BF16])
@pytest.mark.parametrize("dstate", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("dim", [8, 64, 100])
def test_onetoken_shapes(libssu, state_dtype, dstate, dim):
    w = workloads.random_problem(100 + dstate + dim, kind="onetoken", slots=24, heads=6, groups=3,
                                 dim=dim, dstate=dstate, nseq=5, state_dtype=state_dtype,
                                 io_dtype=BF16, tables="distinct", pad_frac=0.2)
    full_check(w)


@pytest.mark.parametrize("state_dtype", [F32, F16, BF16])
@pytest.mark.parametrize("dstate", [16, 64, 128, 256])
@pytest.mark.parametrize("dim", [8, 64, 100])
def test_packed_shapes(libssu, state_dtype, dstate, dim):
    w = workloads.random_problem(200 + dstate + dim, kind="packed", slots=64, heads=4, groups=2,
                                 dim=dim, dstate=dstate, nseq=5, max_len=4, state_dtype=state_dtype,
                                 io_dtype=BF16, tables="distinct", pad_frac=0.15)
    full_check(w)


FLAGS = list(itertools.product([True, False], repeat=4))


@pytest.mark.parametrize("with_D,with_z,with_bias,softplus", FLAGS)
@pytest.mark.parametrize("kind", ["onetoken", "packed"])
def test_flag_combinations(libssu, kind, with_D, with_z, with_bias, softplus):
    seed = 300 + sum(v << i for i, v in enumerate((with_D, with_z, with_bias, softplus)))
    w = workloads.random_problem(seed, kind=kind, slots=48, heads=4, groups=2, dim=16, dstate=64,
                                 nseq=4, max_len=3, with_D=with_D, with_z=with_z,
                                 with_bias=with_bias, dt_softplus=softplus, tables="distinct")
    full_check(w)


@pytest.mark.parametrize("io_dtype", [F16, BF16, F32])
@pytest.mark.parametrize("dt_dtype", [F32, F16, BF16])
def test_io_and_dt_dtypes(libssu, io_dtype, dt_dtype):
    w = workloads.random_problem(400, kind="packed", slots=48, heads=4, groups=1, dim=16, dstate=128,
                                 nseq=4, max_len=3, io_dtype=io_dtype, dt_dtype=dt_dtype,
                                 state_dtype=F16, tables="distinct")
    full_check(w)


@pytest.mark.parametrize("tables", ["none", "read", "distinct", "inplace"])
@pytest.mark.parametrize("kind", ["onetoken", "packed"])
@pytest.mark.parametrize("pad_slot_id", [-1, 0])
def test_table_forms(libssu, kind, tables, pad_slot_id):
    w = workloads.random_problem(500, kind=kind, slots=40 if tables != "none" else 6, heads=4,
                                 groups=2, dim=16, dstate=64, nseq=6 if tables != "none" else 6,
                                 max_len=3, tables=tables, pad_slot_id=pad_slot_id, pad_frac=0.2)
    full_check(w)


@pytest.mark.parametrize("mode", [workloads.SLOTS_STRIDED, workloads.SLOTS_PER_ROW])
@pytest.mark.parametrize("tables", ["read", "distinct"])
def test_slot_modes(libssu, mode, tables):
    w = workloads.random_problem(600, kind="packed", slots=80, heads=4, groups=2, dim=16, dstate=64,
                                 nseq=6, max_len=4, tables=tables, slot_mode=mode, pad_frac=0.1)
    full_check(w)


@pytest.mark.parametrize("kind", ["onetoken", "packed"])
def test_per_head_dt(libssu, kind):
    w = workloads.random_problem(700, kind=kind, slots=48, heads=4, groups=2, dim=16, dstate=128,
                                 nseq=4, max_len=3, per_head_dt=True)
    full_check(w)


def test_dense_form(libssu):
    w = workloads.random_problem(800, kind="packed", slots=64, heads=4, groups=2, dim=16, dstate=128,
                                 nseq=4, max_len=3, dense=True)
    full_check(w)


def test_groups_one_per_head(libssu):
    w = workloads.random_problem(900, kind="packed", slots=64, heads=8, groups=8, dim=16, dstate=64,
                                 nseq=3, max_len=3)
    full_check(w)


# Sequences of six tokens or more on average take the long-sequence kernel
# (one CTA per unit); the sweeps above take the persistent short-sequence one.
@pytest.mark.parametrize("state_dtype", [F32, F16, BF16])
@pytest.mark.parametrize("dstate", [16, 128, 256])
@pytest.mark.parametrize("dim", [8, 100])
def test_packed_long_shapes(libssu, state_dtype, dstate, dim):
    w = workloads.random_problem(1000 + dstate + dim, kind="packed", slots=128, heads=4, groups=2, dim=dim,
                                 dstate=dstate, nseq=4, min_len=6, max_len=9, state_dtype=state_dtype,
                                 io_dtype=BF16, tables="distinct", pad_frac=0.15)
    assert w.rows >= 6 * w.nseq
    full_check(w)


@pytest.mark.parametrize("with_D,with_z,with_bias,softplus", FLAGS[::3])
@pytest.mark.parametrize("mode", [workloads.SLOTS_STRIDED, workloads.SLOTS_PER_ROW])
def test_packed_long_flags_and_modes(libssu, mode, with_D, with_z, with_bias, softplus):
    seed = 1100 + sum(v << i for i, v in enumerate((with_D, with_z, with_bias, softplus)))
    w = workloads.random_problem(seed, kind="packed", slots=160, heads=4, groups=2, dim=16, dstate=64, nseq=5,
                                 min_len=6, max_len=10, with_D=with_D, with_z=with_z, with_bias=with_bias,
                                 dt_softplus=softplus, tables="distinct", slot_mode=mode, pad_frac=0.1)
    full_check(w)


def test_dense_form_long(libssu):
    w = workloads.random_problem(1200, kind="packed", slots=96, heads=4, groups=2, dim=16, dstate=128,
                                 nseq=4, max_len=7, dense=True)
    full_check(w)
