"""The C-ABI library builds, loads and exports what include/ssu.h declares;
host-side argument checks fail before any CUDA call (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

import selective_state_update_gb300 as ssu
from selective_state_update_gb300 import build as ssu_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libssu():
    ssu_build.build()
    return ssu.lib()


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s*(ssu_[a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("ssu_update_onetoken", "ssu_update_packed", "ssu_replay_update", "ssu_batch_copy", "ssu_prewarm",
              "ssu_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(libssu):
    out = subprocess.run(["nm", "-D", "--defined-only", ssu.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)$", out, flags=re.M))
    for n in declared_functions():
        assert n in exported, f"{n} is declared in include/ but not exported"
        assert hasattr(libssu, n)


def test_header_compiles_as_c():
    src = '#include "ssu.h"\nint main(void){ return (int)sizeof(ssu_args) > 0 ? 0 : 1; }\n'
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-x",
                        "c", "-", "-fsyntax-only"], input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_struct_layout_matches_the_header():
    """ctypes mirrors of ssu_args / ssu_slot_table have the C sizes and offsets."""
    probe = r'''
#include <stddef.h>
#include <stdio.h>
#include "ssu.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\n", sizeof(ssu_args), sizeof(ssu_slot_table),
         offsetof(ssu_args, pad_slot_id), offsetof(ssu_args, state), offsetof(ssu_args, x_stride),
         offsetof(ssu_args, d_status), offsetof(ssu_slot_table, s0), sizeof(ssu_replay_buffers),
         offsetof(ssu_replay_buffers, shadow_format), offsetof(ssu_replay_buffers, shadow_scale),
         sizeof(ssu_copy));
  return 0;
}
'''
    exe = os.path.join(ROOT, "selective_state_update_gb300", "_build", "layout_probe")
    os.makedirs(os.path.dirname(exe), exist_ok=True)
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), "-x", "c", "-", "-o", exe],
                   input=probe, text=True, check=True)
    vals = [int(v) for v in subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()]
    A, T, R = ssu.Args, ssu.SlotTable, ssu.ReplayBuffers
    assert vals == [ctypes.sizeof(A), ctypes.sizeof(T), A.pad_slot_id.offset, A.state.offset,
                    A.x_stride.offset, A.d_status.offset, T.s0.offset, ctypes.sizeof(R), R.shadow_format.offset,
                    R.shadow_scale.offset, 24]


def _args(**kw):
    a = ssu.Args(slots=4, heads=4, dim=8, dstate=128, groups=2, state_dtype=0, io_dtype=2, dt_dtype=0,
                 state=16, x=32, dt=48, B=64, C=80, A=96, y=112)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code,needle", [
    (dict(unsupported=ssu.UNSUP_RAND_SEED), ssu.ERR_UNSUPPORTED, "rand_seed"),
    (dict(unsupported=ssu.UNSUP_STATE_SCALE), ssu.ERR_UNSUPPORTED, "state_scale"),
    (dict(groups=3), ssu.ERR_INVALID, "divisible"),
    (dict(dstate=96), ssu.ERR_UNSUPPORTED, "dstate"),
    (dict(state_dtype=7), ssu.ERR_INVALID, "state_dtype"),
    (dict(state=8), ssu.ERR_INVALID, "aligned"),
    (dict(y=32), ssu.ERR_INVALID, "alias"),
    (dict(C=None), ssu.ERR_INVALID, "NULL"),
    (dict(slots=0), ssu.ERR_INVALID, "slots"),
    (dict(reserved0=1), ssu.ERR_INVALID, "reserved0"),
])
def test_host_checks_reject_before_launch(libssu, kw, code, needle):
    a = _args(**kw)
    rc = libssu.ssu_update_onetoken(ctypes.byref(a), 2, None, None, None)
    assert rc == code
    assert needle in libssu.ssu_last_error().decode()


def test_negative_stride_and_bad_table(libssu):
    a = _args()
    a.x_stride[1] = -1
    assert libssu.ssu_update_onetoken(ctypes.byref(a), 2, None, None, None) == ssu.ERR_INVALID
    a = _args()
    t = ssu.SlotTable(entries=128, type=5, mode=0, s0=1, s1=1, extent=2)
    assert libssu.ssu_update_onetoken(ctypes.byref(a), 2, ctypes.byref(t), None, None) == ssu.ERR_INVALID
    t = ssu.SlotTable(entries=128, type=0, mode=9, s0=1, s1=1, extent=2)
    assert libssu.ssu_update_onetoken(ctypes.byref(a), 2, ctypes.byref(t), None, None) == ssu.ERR_INVALID


def test_packed_dense_form_checks(libssu):
    a = _args()
    assert libssu.ssu_update_packed(ctypes.byref(a), 2, 5, None, 2, None, 0, None, None, None) == ssu.ERR_INVALID
    assert "nseq * steps" in libssu.ssu_last_error().decode()
    assert libssu.ssu_update_packed(ctypes.byref(a), 2, 4, None, 0, None, 0, None, None, None) == ssu.ERR_INVALID


def test_empty_calls_launch_nothing(libssu):
    a = _args()
    assert libssu.ssu_update_onetoken(ctypes.byref(a), 0, None, None, None) == ssu.OK
    assert libssu.ssu_update_packed(ctypes.byref(a), 0, 0, None, 1, None, 0, None, None, None) == ssu.OK


def test_prewarm_rejects_unsupported_shapes(libssu):
    assert libssu.ssu_prewarm(0, 2, 0, 8, 8, 100, 2, 0) == ssu.ERR_UNSUPPORTED
    assert libssu.ssu_prewarm(0, 2, 0, 8, 8, 128, 3, 0) == ssu.ERR_INVALID


def test_batch_copy_host_checks(libssu):
    """ssu_batch_copy: argument checks before any launch."""
    assert libssu.ssu_batch_copy(None, -1, 16, None, None) == ssu.ERR_INVALID
    assert libssu.ssu_batch_copy(None, 0, 16, None, None) == ssu.OK
    assert libssu.ssu_batch_copy(None, 3, 0, None, None) == ssu.OK
    assert libssu.ssu_batch_copy(None, 3, 16, None, None) == ssu.ERR_INVALID
    assert "NULL" in libssu.ssu_last_error().decode()
    assert libssu.ssu_batch_copy(12, 3, 16, None, None) == ssu.ERR_INVALID
    assert "aligned" in libssu.ssu_last_error().decode()


def test_shadow_refresh_host_checks(libssu):
    assert libssu.ssu_shadow_refresh(16, 0, 4, 128, 9, 32, 48, None) == ssu.ERR_INVALID     # format
    assert libssu.ssu_shadow_refresh(16, 0, 4, 48, 3, 32, 48, None) == ssu.ERR_UNSUPPORTED  # NVFP4, dstate 48
    assert libssu.ssu_shadow_refresh(16, 0, 4, 128, 3, 32, None, None) == ssu.ERR_INVALID   # NVFP4 without scales
    assert libssu.ssu_shadow_refresh(16, 9, 4, 128, 2, 32, 48, None) == ssu.ERR_INVALID     # state dtype
    assert libssu.ssu_shadow_refresh(16, 0, 0, 128, 2, None, None, None) == ssu.OK          # nothing to do
    assert libssu.ssu_shadow_refresh(16, 0, 4, 128, 2, 32, None, None) == ssu.ERR_INVALID   # E4M3 without scales
    assert "NULL" in libssu.ssu_last_error().decode()


def test_ssd_args_layout_matches_the_header():
    probe = r'''
#include <stddef.h>
#include <stdio.h>
#include "ssu.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu\n", sizeof(ssu_ssd_args), offsetof(ssu_ssd_args, dt_min),
         offsetof(ssu_ssd_args, x), offsetof(ssu_ssd_args, workspace_bytes), offsetof(ssu_ssd_args, d_status));
  return 0;
}
'''
    exe = os.path.join(ROOT, "selective_state_update_gb300", "_build", "ssd_layout_probe")
    os.makedirs(os.path.dirname(exe), exist_ok=True)
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), "-x", "c", "-", "-o", exe],
                   input=probe, text=True, check=True)
    vals = [int(v) for v in subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()]
    S = ssu.SsdArgs
    assert vals == [ctypes.sizeof(S), S.dt_min.offset, S.x.offset, S.workspace_bytes.offset, S.d_status.offset]


def _ssd_args(**kw):
    a = ssu.SsdArgs(tokens=100, heads=4, dim=64, dstate=128, groups=2, nseq=2, nchunks=3, chunk_size=64,
                    io_dtype=2, dt_dtype=0, state_dtype=0, meta_type=0, dt_softplus=1, dt_min=0.0, dt_max=1e30,
                    x=256, dt=512, B=768, C=1024, A=1280, cu_chunk_seqlens=1536, seq_idx=1792,
                    last_chunk_indices=2048, y=2304, states=2560, workspace=4096, workspace_bytes=1 << 30)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code,needle", [
    (dict(io_dtype=0), ssu.ERR_UNSUPPORTED, "bf16"),
    (dict(dim=32), ssu.ERR_UNSUPPORTED, "dim 64"),
    (dict(dstate=96), ssu.ERR_UNSUPPORTED, "dstate"),
    (dict(chunk_size=100), ssu.ERR_UNSUPPORTED, "chunk_size"),
    (dict(groups=3), ssu.ERR_INVALID, "multiple of groups"),
    (dict(meta_type=4), ssu.ERR_INVALID, "meta_type"),
    (dict(dt_min=2.0, dt_max=1.0), ssu.ERR_INVALID, "dt_limit"),
    (dict(B=None), ssu.ERR_INVALID, "NULL"),
    (dict(last_chunk_indices=None), ssu.ERR_INVALID, "NULL"),
    (dict(x=264), ssu.ERR_INVALID, "aligned"),
    (dict(workspace_bytes=1024), ssu.ERR_INVALID, "workspace"),
    (dict(tokens=-1), ssu.ERR_INVALID, "negative"),
])
def test_ssd_host_checks_reject_before_launch(libssu, kw, code, needle):
    a = _ssd_args(**kw)
    assert libssu.ssu_ssd_prefill(ctypes.byref(a), None) == code
    assert needle in libssu.ssu_last_error().decode()


def test_ssd_workspace_size_and_empty_call(libssu):
    n = ctypes.c_uint64(0)
    assert libssu.ssu_ssd_workspace_size(3, 4, 2, 64, 128, 64, ctypes.byref(n)) == ssu.OK
    up = lambda v: (v + 255) // 256 * 256
    # 3 chunks x 4 heads: the chunk states (fp32), prefix sums and dt' per token, one decay,
    # the largest |x| and dt' (16 bytes)
    assert n.value == up(12 * 64 * 128 * 4) + 2 * up(12 * 64 * 4) + up(12 * 4) + up(12 * 16)
    assert libssu.ssu_ssd_workspace_size(3, 0, 2, 64, 128, 64, ctypes.byref(n)) == ssu.ERR_INVALID
    assert libssu.ssu_ssd_workspace_size(3, 4, 0, 64, 128, 64, ctypes.byref(n)) == ssu.ERR_INVALID
    # no chunks: nothing to do, nothing launched, no pointer looked at
    a = _ssd_args(nchunks=0, x=None, B=None, workspace=None)
    assert libssu.ssu_ssd_prefill(ctypes.byref(a), None) == ssu.OK


def _replay_buffers(**kw):
    rb = ssu.ReplayBuffers(len=8, x=4096, dt=8192, B=12288, count_in=16384, count_out=16400)
    for k, v in kw.items():
        setattr(rb, k, v)
    return rb


@pytest.mark.parametrize("rb_kw,args_kw,code,needle", [
    (dict(len=0), {}, ssu.ERR_UNSUPPORTED, "buffer length"),
    (dict(len=33), {}, ssu.ERR_UNSUPPORTED, "buffer length"),
    (dict(count_out=16384), {}, ssu.ERR_INVALID, "alias"),
    (dict(x=None), {}, ssu.ERR_INVALID, "NULL"),
    (dict(count_in=None), {}, ssu.ERR_INVALID, "NULL"),
    (dict(reserved0=1), {}, ssu.ERR_INVALID, "reserved0"),
    (dict(shadow_format=7, shadow=20480), {}, ssu.ERR_INVALID, "SSU_SHADOW"),
    (dict(shadow_format=1, shadow=None), {}, ssu.ERR_INVALID, "read copy"),
    (dict(shadow_format=3, shadow=20480), {}, ssu.ERR_INVALID, "NVFP4 scale records"),
    ({}, dict(disable_state_update=1), ssu.ERR_INVALID, "disable_state_update"),
])
def test_replay_host_checks_reject_before_launch(libssu, rb_kw, args_kw, code, needle):
    a, rb = _args(**args_kw), _replay_buffers(**rb_kw)
    assert libssu.ssu_replay_update(ctypes.byref(a), 2, None, ctypes.byref(rb), None) == code
    assert needle in libssu.ssu_last_error().decode()


def test_replay_empty_call_and_missing_buffers(libssu):
    a = _args()
    assert libssu.ssu_replay_update(ctypes.byref(a), 2, None, None, None) == ssu.ERR_INVALID
    assert libssu.ssu_replay_update(ctypes.byref(a), -1, None, ctypes.byref(_replay_buffers()), None) == ssu.ERR_INVALID
    # nothing to do: no buffer pointer is looked at
    rb = _replay_buffers(x=None, dt=None, B=None, count_in=None, count_out=None)
    assert libssu.ssu_replay_update(ctypes.byref(a), 0, None, ctypes.byref(rb), None) == ssu.OK


@pytest.mark.parametrize("ntok,rb_kw,args_kw,code,needle", [
    (0, {}, {}, ssu.ERR_INVALID, "ntok"),
    (9, {}, {}, ssu.ERR_INVALID, "exceeds the buffer length"),
    (2, dict(len=33), {}, ssu.ERR_UNSUPPORTED, "buffer length"),
    (2, dict(shadow_format=1, shadow=20480), {}, ssu.ERR_UNSUPPORTED, "low-precision copy"),
    (2, dict(count_out=16384), {}, ssu.ERR_INVALID, "alias"),
    (2, dict(B=None), {}, ssu.ERR_INVALID, "NULL"),
    (2, dict(reserved0=3), {}, ssu.ERR_INVALID, "reserved0"),
    (2, {}, dict(disable_state_update=1), ssu.ERR_INVALID, "disable_state_update"),
    (2, {}, dict(groups=3), ssu.ERR_INVALID, "divisible"),
])
def test_verify_host_checks_reject_before_launch(libssu, ntok, rb_kw, args_kw, code, needle):
    """ssu_replay_verify: T drafts must fit the buffer, no read copy, the
    replay buffers' rules; all decided before any launch."""
    a, rb = _args(**args_kw), _replay_buffers(**rb_kw)
    assert libssu.ssu_replay_verify(ctypes.byref(a), 2, ntok, None, ctypes.byref(rb), None) == code
    assert needle in libssu.ssu_last_error().decode()


def test_verify_empty_call_launches_nothing(libssu):
    a = _args()
    rb = _replay_buffers(x=None, dt=None, B=None, count_in=None, count_out=None)
    assert libssu.ssu_replay_verify(ctypes.byref(a), 0, 4, None, ctypes.byref(rb), None) == ssu.OK
    assert libssu.ssu_replay_verify(ctypes.byref(a), -1, 4, None, ctypes.byref(rb), None) == ssu.ERR_INVALID


def test_selftest_timeout_host_checks(libssu):
    a = _args()
    assert libssu.ssu_selftest_timeout(ctypes.byref(a), 2, None, None, 8, 10 ** 6, None) == ssu.ERR_INVALID
    assert "withhold_unit" in libssu.ssu_last_error().decode()
    assert libssu.ssu_selftest_timeout(ctypes.byref(a), 2, None, None, -1, 10 ** 6, None) == ssu.ERR_INVALID
    assert libssu.ssu_selftest_timeout(ctypes.byref(a), 2, None, None, 1, 10, None) == ssu.ERR_INVALID
    assert "wait_cycles" in libssu.ssu_last_error().decode()
    assert libssu.ssu_selftest_timeout(ctypes.byref(a), 2, None, None, 1, 10 ** 10, None) == ssu.ERR_INVALID
    assert libssu.ssu_selftest_timeout(ctypes.byref(a), 0, None, None, 0, 10 ** 6, None) == ssu.ERR_INVALID
