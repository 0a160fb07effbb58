"""Batched byte copies with memmove semantics, on the host.

TEST INFRASTRUCTURE ONLY (see the package docstring): the plain definition
the GPU's ``ssu_batch_copy`` is compared with.

Digest of vLLM PR #50729, section 实现拆解 (items 1-4): speculative decoding
moves and shifts slot state inside one buffer, a copy's source and
destination may overlap, and a copy must then behave like memmove -- the
destination receives the bytes the source held before the copy.  The PR's
tests compare against an unmodified snapshot of the buffer rather than
against a second implementation; so does this definition: every copy reads
the snapshot.  That is memmove applied copy by copy, because different copies
of one call may not overlap one another (checked here, refused with
ValueError, as the C ABI leaves that case undefined).
"""
from __future__ import annotations

from typing import Iterable, Tuple

import numpy as np


def batch_copy(buf: np.ndarray, copies: Iterable[Tuple[int, int, int]]) -> np.ndarray:
    """``buf`` a 1-D uint8 array; ``copies`` (source offset, destination
    offset, bytes) triples.  Returns the buffer after the copies; ``buf`` is
    not modified."""
    if buf.dtype != np.uint8 or buf.ndim != 1:
        raise ValueError("buf must be a 1-D uint8 array")
    copies = [(int(s), int(d), int(n)) for s, d, n in copies]
    for s, d, n in copies:
        if n < 0 or s < 0 or d < 0 or s + n > buf.size or d + n > buf.size:
            raise ValueError(f"copy ({s}, {d}, {n}) outside the buffer")
    # no copy may touch bytes another copy writes
    live = [(s, d, n) for s, d, n in copies if n > 0 and s != d]
    for i, (s1, d1, n1) in enumerate(live):
        for s2, d2, n2 in live[i + 1:]:
            for a, an in ((s1, n1), (d1, n1)):
                if a < d2 + n2 and d2 < a + an:
                    raise ValueError("two copies overlap")
            if s2 < d1 + n1 and d1 < s2 + n2:
                raise ValueError("two copies overlap")
    out = buf.copy()
    for s, d, n in copies:
        out[d:d + n] = buf[s:s + n]
    return out
