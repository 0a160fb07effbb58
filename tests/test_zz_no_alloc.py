"""ssu_ssd_prefill_static: the SSD prefill on the library's own scratch gives
the bits of ssu_ssd_prefill with a caller workspace, on two calls in a row
(the scratch keeps nothing from one call that the next depends on).  Named
to be collected last; it passes alone and after the other tests."""
import ctypes

import pytest
import torch

import selective_state_update_gb300 as ssu
import workloads


def _problem():
    # 700 tokens in 4 sequences, heads 16, groups 2, dstate 128, chunk 128:
    # 8 chunks, within the scratch
    return workloads.ssd_problem(300, [130, 257, 1, 312], heads=16, dim=64, dstate=128, groups=2, chunk_size=128)


def _call(fn, g, **kw):
    return fn(g.x, g.dt, g.A, g.B, g.C, g.chunk_size, g.cu_chunk_seqlens, g.seq_idx, g.last_chunk_indices,
              D=g.D, z=g.z, dt_bias=g.dt_bias, dt_softplus=g.dt_softplus, dt_limit=g.dt_limit,
              initial_states=g.initial_states, state_dtype=g.state_dtype, nseq=g.nseq, **kw)


@pytest.mark.gpu
def test_static_scratch_matches_the_workspace_call(libssu):
    g = _problem().to("cuda")
    ref_y, ref_s = _call(ssu.ssu_ssd_prefill, g)
    ref_yi, ref_si = _call(ssu.ssu_ssd_prefill, g, return_intermediate_states=True)
    for _ in range(2):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        y, s = _call(ssu.ssu_ssd_prefill_static, g, status=status)
        yi, si = _call(ssu.ssu_ssd_prefill_static, g, return_intermediate_states=True, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(y, ref_y) and torch.equal(s, ref_s)
        assert torch.equal(yi, ref_yi) and torch.equal(si, ref_si)


def test_static_scratch_rejects_a_call_larger_than_the_scratch(libssu):
    """Checked on the host before any device work: a call whose workspace
    exceeds the scratch, and a call that passes a workspace."""
    n = ctypes.c_uint64(0)
    assert libssu.ssu_ssd_workspace_size(16, 128, 8, 64, 128, 256, ctypes.byref(n)) == ssu.OK
    assert n.value > ssu.SSD_STATIC_SCRATCH_BYTES
    a = ssu.SsdArgs(tokens=4096, heads=128, dim=64, dstate=128, groups=8, nseq=1, nchunks=16, chunk_size=256,
                    io_dtype=2, x=256, dt=512, B=768, C=1024, A=1280, cu_chunk_seqlens=1536, seq_idx=1792,
                    last_chunk_indices=2048, y=2304, states=2560)
    assert libssu.ssu_ssd_prefill_static(ctypes.byref(a), None) == ssu.ERR_INVALID
    assert "scratch" in libssu.ssu_last_error().decode()
    a.nchunks, a.workspace, a.workspace_bytes = 4, 4096, 1 << 30
    assert libssu.ssu_ssd_prefill_static(ctypes.byref(a), None) == ssu.ERR_INVALID
    assert "workspace must be NULL" in libssu.ssu_last_error().decode()
