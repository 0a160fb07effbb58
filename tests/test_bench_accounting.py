"""bench.py's byte and flop accounting (SSD prefill, speculative verification), against counts
worked out by hand for small problems (CPU only)."""
import bench
import torch
import workloads


def test_ssd_accounting_one_chunk():
    # 16 tokens, heads 2, dim 8, dstate 16, groups 1, chunk 16: one full chunk
    w = workloads.ssd_problem(1, [16], heads=2, dim=8, dstate=16, groups=1, chunk_size=16)
    a = bench.ssd_accounting(w)
    x = 16 * 2 * 8 * 2            # bf16 x (z and y the same size)
    dt = 16 * 2 * 4               # fp32 dt
    bc = 2 * 16 * 1 * 16 * 2      # bf16 B and C
    st = 1 * 2 * 8 * 16 * 4       # one fp32 state per sequence
    meta = (2 + 1 + 1) * 4        # cu_chunk_seqlens, seq_idx, last_chunk_indices (int32)
    assert a["inputs"] == 2 * x + dt + bc + st + meta
    assert a["outputs"] == x + st
    assert a["total"] == a["inputs"] + a["outputs"]
    # per head: chunk state 2TPN, C . S_in^T 2TNP, and one 16 x 16 causal tile
    # for C . B^T (2 * 256 * N) and W . X (2 * 256 * P)
    assert a["flops"] == 2 * (2 * 16 * 8 * 16 + 2 * 16 * 16 * 8 + 2 * 256 * 16 + 2 * 256 * 8)
    # the chunk states cross the workspace four times; C . B^T stays on chip
    assert a["workspace"] == 4 * 1 * 2 * 8 * 16 * 4
    assert a["tokens"] == 16


def test_ssd_accounting_ragged_tiles():
    # a 17-token chunk of a 32-token chunk size counts two 16-row tiles: 16 + 32 columns
    w = workloads.ssd_problem(2, [17], heads=1, dim=8, dstate=16, groups=1, chunk_size=32, with_z=False,
                              with_init=False)
    a = bench.ssd_accounting(w)
    causal = (16 + 32) * 16
    assert a["flops"] == 2 * 17 * 8 * 16 * 2 + 2 * causal * 16 + 2 * causal * 8
    assert a["outputs"] == 17 * 8 * 2 + 8 * 16 * 4


def test_verify_bytes_by_hand():
    # 3 sequences, T = 2, L = 6, heads 2, dim 4, dstate 8, groups 1, bf16 io, fp32 pool;
    # counts 0 (no flush), 2 (2 + 4 >= 6: flush), pad
    w = workloads.verify_problem(5, ntok=2, buffer_len=6, nseq=3, slots=8, heads=2, dim=4, dstate=8, groups=1)
    w.read = torch.tensor([1, 2, -1], dtype=torch.int32)
    count = torch.tensor([0, 2, 0], dtype=torch.int32)
    a = bench.verify_bytes(w, count)
    sb = 2 * 4 * 8 * 4                     # one fp32 checkpoint
    entry = 2 * 4 * (2 + 4) + 1 * 8 * 2    # x (bf16) + dt' (fp32) of every head row, B of the group
    draft_in = 2 * 4 * (2 * 2 + 4) + 2 * 8 * 2   # x, z (bf16), dt (fp32); B, C (bf16)
    draft_out = 2 * 4 * 2
    per_seq = 2 * (draft_in + draft_out) + 12
    want = 3 * per_seq + (sb + 0 + 2 * entry) + (sb + 2 * entry + 2 * entry + sb)
    assert a["total"] == want


def _tiny(kind, rows, heads=2, dim=4, dstate=16, groups=1, slots=12, **kw):
    """A hand-sized workload: fp32 pool, bf16 x/B/C, fp32 dt, A, no optional operands."""
    return workloads.Workload(
        name="tiny", kind=kind, state=torch.zeros(slots, heads, dim, dstate),
        x=torch.zeros(rows, heads, dim, dtype=torch.bfloat16), dt=torch.zeros(rows, heads, dim),
        A=torch.zeros(heads), B=torch.zeros(rows, groups, dstate, dtype=torch.bfloat16),
        C=torch.zeros(rows, groups, dstate, dtype=torch.bfloat16), **kw)


def test_onetoken_bytes_by_hand():
    # 3 sequences: read [5, pad, 7], dst [pad, 2, 3]; a (slot, all heads) state is 2*4*16*4 B
    w = _tiny("onetoken", 3, read=torch.tensor([5, -1, 7], dtype=torch.int32),
              dst=torch.tensor([-1, 2, 3], dtype=torch.int32))
    a = bench.algorithmic_bytes(w)
    sb = 2 * 4 * 16 * 4
    x = 3 * 2 * 4 * 2                                  # bf16 x, and y the same
    small = x + 3 * 2 * 4 * 4 + 2 * (3 * 16 * 2) + 2 * 4 + 2 * 3 * 4 + x   # x, dt, B, C, A, tables, y
    assert (a["seeds"], a["writes"]) == (2, 2)
    assert a["state_read"] == 2 * sb and a["state_write"] == 2 * sb
    assert a["small"] == small and a["total"] == 4 * sb + small


def test_packed_bytes_by_hand():
    # two sequences of 3 tokens (dense 2-D tables): seeds at max(acc-1, 0) = 1 and 0,
    # one pad seed (sequence 1's entry 0), one pad destination
    read = torch.tensor([[4, 9, 6], [-1, 8, 10]], dtype=torch.int32)
    dst = torch.tensor([[1, 2, 3], [5, -1, 11]], dtype=torch.int32)
    w = _tiny("packed", 6, read=read, dst=dst, dense_steps=3, num_accepted=torch.tensor([2, 1], dtype=torch.int32))
    a = bench.algorithmic_bytes(w)
    assert (a["seeds"], a["writes"]) == (1, 5)        # seq 0 seeds at slot 9; seq 1's seed entry is pad
    w.disable_state_update = True
    assert bench.algorithmic_bytes(w)["writes"] == 0


def test_replay_bytes_by_hand():
    # L = 4; counts [0, 3 (folds: 3 + 1 == L), 2, pad]; one (slot, entry) entry is
    # x (bf16) + dt' (fp32) per head row and B per group
    L, heads, dim, dstate, groups = 4, 2, 4, 16, 1
    slots = 8
    w = _tiny("replay", 4, heads=heads, dim=dim, dstate=dstate, groups=groups, slots=slots,
              read=torch.tensor([1, 2, 3, -1], dtype=torch.int32),
              xbuf=torch.zeros(slots, L, heads, dim, dtype=torch.bfloat16),
              dtbuf=torch.zeros(slots, L, heads, dim), Bbuf=torch.zeros(slots, L, groups, dstate, dtype=torch.bfloat16),
              count=torch.tensor([0, 3, 2, 0], dtype=torch.int32))
    a = bench.algorithmic_bytes(w)
    sb = heads * dim * dstate * 4
    entry = heads * dim * (2 + 4) + groups * dstate * 2
    assert a["folds"] == 1
    assert a["state_read"] == 3 * sb + (0 + 3 + 2) * entry      # every live checkpoint, its entries
    assert a["state_write"] == sb + 2 * entry                  # the fold's checkpoint, one entry each other


def test_threaded_oracle_rate_runs_the_oracle_on_several_threads():
    """The CPU baseline on all host cores: the unchanged oracle on several
    threads at once over one-sequence samples, a positive rate."""
    w = workloads.b256_fp32(device="cpu", seed=1002, batch=6)
    rate, desc = bench.oracle_rate_threaded(w, 0.5, 2)
    assert rate > 0 and "on 2 threads" in desc
    assert bench.host_threads() >= 1
