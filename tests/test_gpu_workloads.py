"""The five decode workloads at full size, in the launch configuration the
benchmark times: every sequence is compared with the oracle element by element
(y and every written slot), and properties that hold at any size are checked
on the whole pool (untouched slots bit-identical, pad slot never written, no
device status bits)."""
import pytest
import torch

import workloads
from gpu_harness import (DEV, assert_untouched, complete_check, full_check, run_gpu, written_slots)
from ssu_testlib import assert_y_close, run_oracle

pytestmark = pytest.mark.gpu


def _run_full(w_cpu):
    w = w_cpu.to(DEV)
    before = w.state.clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = run_gpu(w, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_untouched(before, w.state, written_slots(w_cpu))
    del before
    return w, y


def test_tiny_onetoken(libssu):
    full_check(workloads.tiny_onetoken())


@pytest.mark.parametrize("in_place", [False, True])
def test_b256_fp32(libssu, in_place):
    w_cpu = workloads.b256_fp32(in_place=in_place)
    w, y = _run_full(w_cpu)
    assert torch.equal(w.state[0].cpu(), w_cpu.state[0]), "pad slot 0 was written"
    assert complete_check(w_cpu, y, w.state) == 256


def test_b1024_bf16(libssu):
    w_cpu = workloads.b1024_bf16()
    w, y = _run_full(w_cpu)
    assert complete_check(w_cpu, y, w.state) == 1024


def test_mtp_64x7_fp32(libssu):
    w_cpu = workloads.mtp_64x7_fp32()
    w, y = _run_full(w_cpu)
    assert complete_check(w_cpu, y, w.state) == 64


def test_varlen_fp16(libssu):
    w_cpu = workloads.varlen_fp16()
    w, y = _run_full(w_cpu)
    assert complete_check(w_cpu, y, w.state) == 128


@pytest.mark.parametrize("slot_mode", [workloads.SLOTS_PER_ROW, workloads.SLOTS_STRIDED])
def test_varlen_fp16_disable(libssu, slot_mode):
    """disable_state_update on identical inputs: the pool stays bit-identical
    and y equals the updating run's y bit for bit (per-row addressing), or the
    oracle's (page-literal strided flat addressing, only meaningful with the
    update disabled)."""
    w_cpu = workloads.varlen_fp16(disable_state_update=True, slot_mode=slot_mode)
    w = w_cpu.to(DEV)
    before = w.state.clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    y = run_gpu(w, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(before, w.state), "disable_state_update changed the pool"
    if slot_mode == workloads.SLOTS_PER_ROW:
        w2 = workloads.varlen_fp16().to(DEV)
        y2 = run_gpu(w2)
        torch.cuda.synchronize()
        assert torch.equal(y, y2)
    # nothing is written, so the oracle may use the input pool as its output
    ref = run_oracle(w_cpu, state_out=w_cpu.state)
    assert_y_close(y, ref.y_exact)
