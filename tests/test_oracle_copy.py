"""Pins of the memmove-semantics copy oracle (oracle/memcopy.py) against
C's memmove (through ctypes, an independent implementation), hand-worked
byte strings, and its refusals.  CPU only."""
import ctypes

import numpy as np
import pytest

import oracle


def _libc_memmove(buf: np.ndarray, copies):
    """The copies applied one after another with C's memmove."""
    out = bytearray(buf.tobytes())
    base = ctypes.addressof((ctypes.c_char * len(out)).from_buffer(out))
    for s, d, n in copies:
        ctypes.memmove(base + d, base + s, n)
    return np.frombuffer(bytes(out), dtype=np.uint8)


def test_hand_worked_shifts():
    b = np.frombuffer(b"abcdefgh", dtype=np.uint8)
    assert bytes(oracle.batch_copy(b, [(2, 0, 6)])) == b"cdefghgh"   # left overlap: memmove, not memcpy
    assert bytes(oracle.batch_copy(b, [(0, 2, 6)])) == b"ababcdef"   # right overlap
    assert bytes(oracle.batch_copy(b, [(0, 4, 4)])) == b"abcdabcd"   # adjacent, disjoint
    assert bytes(oracle.batch_copy(b, [(3, 3, 5), (1, 0, 0)])) == b"abcdefgh"  # src == dst, empty
    assert bytes(oracle.batch_copy(b, [(6, 0, 2), (2, 4, 2)])) == b"ghcdcdgh"  # two disjoint copies


@pytest.mark.parametrize("seed", range(20))
def test_single_copies_equal_memmove(seed):
    rng = np.random.default_rng(seed)
    size = int(rng.integers(1, 5000))
    buf = rng.integers(0, 256, size, dtype=np.uint8)
    n = int(rng.integers(0, size + 1))
    s = int(rng.integers(0, size - n + 1))
    d = int(rng.integers(0, size - n + 1))
    assert np.array_equal(oracle.batch_copy(buf, [(s, d, n)]), _libc_memmove(buf, [(s, d, n)]))


def test_disjoint_batches_equal_memmove_in_sequence():
    rng = np.random.default_rng(7)
    buf = rng.integers(0, 256, 64 * 1024, dtype=np.uint8)
    copies = []
    for r in range(16):  # each copy inside its own 4 KiB region, some overlapping themselves
        lo = r * 4096
        n = int(rng.integers(1, 2048))
        s = lo + int(rng.integers(0, 4096 - n))
        d = lo + int(rng.integers(0, 4096 - n))
        copies.append((s, d, n))
    assert np.array_equal(oracle.batch_copy(buf, copies), _libc_memmove(buf, copies))


def test_refusals():
    b = np.zeros(100, dtype=np.uint8)
    with pytest.raises(ValueError):
        oracle.batch_copy(b, [(0, 50, 30), (60, 10, 10)])   # the second reads what the first writes
    with pytest.raises(ValueError):
        oracle.batch_copy(b, [(0, 10, 20), (50, 20, 5)])    # both write bytes 20..24
    with pytest.raises(ValueError):
        oracle.batch_copy(b, [(90, 0, 20)])                 # outside the buffer
    with pytest.raises(ValueError):
        oracle.batch_copy(b.astype(np.int16), [])


def _forward_bytewise(buf, copies):
    """A plausible wrong definition: memcpy as a forward byte loop over the
    live buffer (what a parallel copy without ordering can produce)."""
    out = buf.copy()
    for s, d, n in copies:
        for k in range(n):
            out[d + k] = out[s + k]
    return out


def _backward_bytewise(buf, copies):
    out = buf.copy()
    for s, d, n in copies:
        for k in reversed(range(n)):
            out[d + k] = out[s + k]
    return out


@pytest.mark.parametrize("wrong", [_forward_bytewise, _backward_bytewise])
def test_pins_reject_unordered_copies(wrong):
    """Each plausible wrong definition fails one of the hand-worked pins."""
    b = np.frombuffer(b"abcdefgh", dtype=np.uint8)
    cases = [([(2, 0, 6)], b"cdefghgh"), ([(0, 2, 6)], b"ababcdef")]
    assert any(bytes(wrong(b, c)) != e for c, e in cases)
    assert all(bytes(oracle.batch_copy(b, c)) == e for c, e in cases)
