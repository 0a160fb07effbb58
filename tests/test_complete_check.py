"""The every-sequence comparison used by the full-size GPU tests, checked on
the CPU with the oracle's own full-workload results standing in for the GPU's:
the chunked sub-problems reproduce them, and a mistake planted in one
sequence's y or in one written slot is found."""
import pytest
import torch

import workloads
from gpu_harness import complete_check
from ssu_testlib import run_oracle


def _as_if_gpu(w):
    ref = run_oracle(w)
    return ref.y_exact.to(w.x.dtype), ref.state.clone()


def _onetoken():
    return workloads.random_problem(2, kind="onetoken", slots=64, heads=4, groups=2, dim=16, dstate=32, nseq=24,
                                    pad_slot_id=0)


def _mtp():
    return workloads.random_problem(4, kind="packed", slots=128, heads=4, groups=2, dim=16, dstate=32, nseq=8,
                                    max_len=6, allow_empty=False)


def _per_row():
    return workloads.random_problem(3, kind="packed", slots=256, heads=4, groups=2, dim=16, dstate=32, nseq=21,
                                    max_len=5, slot_mode=workloads.SLOTS_PER_ROW, tables="read",
                                    state_dtype=torch.float16)


@pytest.mark.parametrize("make", [_onetoken, _mtp, _per_row], ids=["onetoken", "mtp", "per_row"])
def test_oracle_results_pass(make):
    w = make()
    y, st = _as_if_gpu(w)
    assert complete_check(w, y, st, per_chunk=4) == w.nseq


def test_planted_y_error_found():
    w = _onetoken()
    y, st = _as_if_gpu(w)
    y[17, 2, 3] += 0.5
    with pytest.raises(AssertionError, match="sequences 16..19"):
        complete_check(w, y, st, per_chunk=4)


def test_planted_state_error_found():
    w = _mtp()
    y, st = _as_if_gpu(w)
    slot = next(int(s) for s in w.dst[4] if int(s) != w.pad_slot_id)
    st[slot, 3, 1, 7] += 1e-3
    with pytest.raises(AssertionError, match="state"):
        complete_check(w, y, st, per_chunk=2)
