"""ssu_batch_copy on the GPU against the memmove oracle (oracle/memcopy.py),
following the test method of the digest of vLLM PR #50729 (实现拆解 item 5):
every result is compared with the copies applied to an unmodified snapshot
of the buffer, never with a second implementation of the kernel."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_update_gb300 as ssu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(buf: torch.Tensor, copies, max_bytes=None, status=None):
    """Apply (src offset, dst offset, bytes) copies to the uint8 CUDA buffer."""
    base = buf.data_ptr()
    table = ssu.copy_table([(base + s, base + d, n) for s, d, n in copies], DEV)
    mb = max((n for _, _, n in copies), default=0) if max_bytes is None else max_bytes
    ssu.ssu_batch_copy(table, mb, status=status)
    torch.cuda.synchronize()


def _check(buf_gpu: torch.Tensor, snapshot: np.ndarray, copies):
    ref = oracle.batch_copy(snapshot, copies)
    got = buf_gpu.cpu().numpy()
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[0]}"


def _random_buffer(nbytes, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, 256, (nbytes,), generator=g, dtype=torch.uint8).to(DEV)


def test_left_overlap_rows_repeatedly(libssu):
    """128 rows of 32 KiB, each shifted left by 16 bytes inside itself, ten
    rounds in a row (the PR's regression test shape)."""
    rows, row = 128, 32 * 1024
    buf = _random_buffer(rows * row, 1)
    copies = [(r * row + 16, r * row, row - 16) for r in range(rows)]
    for _ in range(10):
        snap = buf.cpu().numpy()
        _run(buf, copies)
        _check(buf, snap, copies)


@pytest.mark.parametrize("shift", [1, 3, 16, 100, 4096, 40000])
def test_right_and_left_overlap_shifts(libssu, shift):
    """Shifts smaller and larger than a piece of the ordered path, both
    directions, aligned and unaligned."""
    n = 200 * 1024 + 5
    buf = _random_buffer(2 * (n + shift) + 64, 2 + shift)
    copies = [(0, shift, n),                       # right overlap (dst above src)
              (n + shift + 32 + shift, n + shift + 32, n)]  # left overlap (dst below src)
    snap = buf.cpu().numpy()
    _run(buf, copies)
    _check(buf, snap, copies)


@pytest.mark.parametrize("seed", range(6))
def test_random_mixed_batches(libssu, seed):
    """Random lengths (0 B .. 300 KiB) and alignments, each copy in its own
    region: disjoint copies inside or between regions, overlapping shifts."""
    rng = np.random.default_rng(100 + seed)
    region = 640 * 1024
    nreg = 48
    buf = _random_buffer(region * nreg, 10 + seed)
    copies = []
    for r in range(nreg):
        lo = r * region
        kind = rng.integers(0, 3)
        n = int(rng.choice([0, 1, 15, 16, 17, 4095, 65536, 65537, int(rng.integers(1, 300 * 1024))]))
        if kind == 0:    # disjoint inside the region
            s = lo + int(rng.integers(0, 32))
            d = lo + region // 2 + int(rng.integers(0, 32))
        else:            # overlapping shift
            shift = int(rng.integers(1, max(2, n)))
            s = lo + int(rng.integers(0, 64))
            d = s + shift if kind == 1 else s
            s = s if kind == 1 else s + shift
        copies.append((s, d, n))
    snap = buf.cpu().numpy()
    _run(buf, copies)
    _check(buf, snap, copies)


def test_longer_than_the_tile_grid(libssu):
    """A copy of more tiles than the grid has tile slots (the tile loop)."""
    n = 300 * 1024 * 1024 + 48
    buf = torch.empty(2 * n + 4096, dtype=torch.uint8, device=DEV)
    buf[:n].random_(0, 256, generator=torch.Generator(device=DEV).manual_seed(3))
    before = buf[:n].clone()
    _run(buf, [(0, n + 16, n)])
    assert torch.equal(buf[n + 16:2 * n + 16], before)
    assert torch.equal(buf[:n], before)


def test_edge_cases_and_bound(libssu):
    buf = _random_buffer(1 << 20, 4)
    snap = buf.cpu().numpy()
    # nothing to do
    ssu.ssu_batch_copy(torch.empty((0, 3), dtype=torch.int64, device=DEV), 0)
    _run(buf, [(0, 0, 1000), (100, 5000, 0)])
    _check(buf, snap, [])
    # a copy longer than max_bytes is skipped and flagged; the others run
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    copies = [(0, 500000, 4096), (10000, 700000, 64)]
    _run(buf, copies, max_bytes=1024, status=status)
    assert int(status.item()) == ssu.DEV_BAD_COPY
    _check(buf, snap, [copies[1]])


def test_full_size_slot_copies(libssu):
    """256 whole-slot copies of 4 MiB in a 512-slot fp32 pool (heads 128,
    dim 64, dstate 128), from random slots to other random slots: every
    destination holds its source's bits, every other slot is unchanged."""
    g = torch.Generator().manual_seed(5)
    pool = torch.randn((512, 128, 64, 128), generator=torch.Generator(device=DEV).manual_seed(5), device=DEV)
    perm = torch.randperm(512, generator=g)
    src, dst = perm[:256], perm[256:]
    before = pool.clone()
    table = ssu.slot_copies(pool, src, dst)
    ssu.ssu_batch_copy(table, pool[0].numel() * 4)
    torch.cuda.synchronize()
    assert torch.equal(pool[dst.to(DEV)], before[src.to(DEV)])
    keep = torch.ones(512, dtype=torch.bool)
    keep[dst] = False
    assert torch.equal(pool[keep.to(DEV)], before[keep.to(DEV)])
