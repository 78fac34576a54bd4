"""Exhaustive pin of the oracle's binary32 -> bfloat16 / binary16 rounding:
all 2^32 input patterns against torch's CPU casts (IEEE round-to-nearest-
even, gradual underflow, overflow to infinity), NaN inputs against the
canonical quiet NaN the oracle defines.  Spread over worker processes
(spawned, so no state is shared with the test process)."""
import multiprocessing as mp
import os

import numpy as np
import pytest

SPAN = 1 << 29      # patterns per job
CHUNK = 1 << 22     # patterns per step inside a job (buffers reused)


def _check_span(args):
    out, start = args
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import torch
    from oracle import oracle as O
    step = np.arange(CHUNK, dtype=np.uint32)
    bits = np.empty(CHUNK, dtype=np.uint32)
    canon = 0x7FC0 if out == "BF16" else 0x7E00
    tdt = torch.bfloat16 if out == "BF16" else torch.float16
    bad, first = 0, None
    for base in range(start, start + SPAN, CHUNK):
        np.add(step, np.uint32(base), out=bits)
        got = O.convert("F32", out, bits.view(np.uint8)).view(np.uint16)
        f = bits.view(np.float32)
        want = torch.from_numpy(f).to(tdt).view(torch.int16).numpy().view(np.uint16)
        want = np.where(np.isnan(f), np.uint16(canon), want)
        diff = np.nonzero(got != want)[0]
        if diff.size:
            bad += int(diff.size)
            first = first if first is not None else int(bits[diff[0]])
    return bad, first


@pytest.mark.parametrize("out", ["BF16", "F16"])
def test_every_f32_pattern_rounds_like_torch(oracle, out):
    jobs = [(out, s) for s in range(0, 1 << 32, SPAN)]
    workers = max(1, min(8, os.cpu_count() or 1))
    with mp.get_context("spawn").Pool(workers) as pool:
        results = pool.map(_check_span, jobs)
    bad = sum(n for n, _ in results)
    first = next((f for n, f in results if n), None)
    assert bad == 0, f"{bad} patterns differ, first 0x{first:08x}"
