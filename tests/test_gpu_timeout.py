"""The kernels' exit path, exercised without any device fault: through
ssu_selftest_timeout one unit's stage is never filled, so the consumers'
bounded wait for it runs out (after a short limit) with no copy pending.  The
kernel must report SSU_DEV_TIMEOUT; the CTA that owned the unit stops, waits
for the copies it had issued and returns; every other unit is computed as
usual; and the context stays usable for the next call."""
import pytest
import torch

import selective_state_update_gb300 as ssu
import workloads
from gpu_harness import DEV, full_check
from ssu_testlib import assert_state_close, assert_y_close, run_oracle

pytestmark = pytest.mark.gpu

SENTINEL = 7.0


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_withheld_unit_times_out(libssu, state_dtype):
    # 64 sequences x 8 heads = 512 units: more units than resident CTAs, so the
    # CTA owning the withheld unit has issued the copies of later units too
    w = workloads.random_problem(41, kind="onetoken", slots=160, heads=8, groups=2, dim=64, dstate=128, nseq=64,
                                 tables="distinct", pad_frac=0.0, state_dtype=state_dtype)
    g = w.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full(g.x.shape, SENTINEL, dtype=g.x.dtype, device=DEV)
    withheld = 5 * 8 + 3  # sequence 5, head 3
    ssu.ssu_selftest_timeout(g.state, g.x, g.dt, g.A, g.B, g.C, withhold_unit=withheld, wait_cycles=2_000_000,
                             D=g.D, z=g.z, dt_bias=g.dt_bias, dt_softplus=g.dt_softplus,
                             state_batch_indices=g.read, dst_state_batch_indices=g.dst,
                             pad_slot_id=g.pad_slot_id, out=out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == ssu.DEV_TIMEOUT
    ref = run_oracle(w)
    y, st = out.cpu(), g.state.cpu()
    skipped = []
    for b in range(w.nseq):
        ws = int(w.dst[b])
        for h in range(8):
            untouched = bool(torch.all(y[b, h].float() == SENTINEL)) and torch.equal(st[ws, h], w.state[ws, h])
            if untouched:
                skipped.append(b * 8 + h)
                continue
            assert_y_close(y[b, h], ref.y_exact[b, h], what=f"y of unit {b * 8 + h}")
            assert_state_close(st[ws, h], ref.state[ws, h], what=f"state of unit {b * 8 + h}")
    assert withheld in skipped
    # only the owning CTA stops: its own units at most (512 units over at least 152 CTAs)
    assert len(skipped) <= 4, skipped
    # the context is still usable: a normal call on a fresh copy is correct
    full_check(w)
