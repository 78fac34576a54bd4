"""The parity harness itself, on the CPU: the guard-band check finds a byte
written outside the outputs, and the whole-output comparison finds one wrong
byte anywhere (element ranges split across threads and batches), so that a
green GPU parity run means what it says."""
import numpy as np
import pytest

from conftest import small_file
from oracle_compare import FILL, assert_guards, compare_full, gap_ranges

torch = pytest.importorskip("torch")


def test_gap_ranges():
    starts, stops = gap_ranges(100, [40, 10, 70], [20, 5, 30])
    assert list(zip(starts, stops)) == [(0, 10), (15, 40), (60, 70)]
    starts, stops = gap_ranges(10, [0, 5], [5, 0])
    assert list(zip(starts, stops)) == [(5, 10)]
    with pytest.raises(AssertionError):
        gap_ranges(100, [0, 4], [8, 8])


@pytest.mark.parametrize("max_gather", [3, 1 << 20])
def test_assert_guards_finds_a_stray_write(max_gather):
    offsets, sizes = [16, 64, 300], [40, 100, 7]
    arena = torch.full((400,), FILL, dtype=torch.uint8)
    for o, n in zip(offsets, sizes):
        arena[o:o + n] = 7                                   # the outputs' own bytes may be anything
    assert_guards(arena, offsets, sizes, max_gather=max_gather)
    for pos in (0, 15, 56, 63, 164, 299, 307, 399):         # padding, gaps and the tail
        bad = arena.clone()
        bad[pos] = FILL ^ 1
        with pytest.raises(AssertionError, match=f"offset {pos} "):
            assert_guards(bad, offsets, sizes, max_gather=max_gather)


class _Result:
    def __init__(self, outs):
        self.outs = [torch.from_numpy(o.copy()) for o in outs]

    def raw(self, i):
        return self.outs[i]


@pytest.mark.parametrize("span,batch", [(1 << 22, 1 << 31), (3, 5)])
def test_compare_full_finds_one_wrong_byte(oracle, span, batch):
    g, f = small_file()
    img = np.frombuffer(f, dtype=np.uint8).copy()
    ix = oracle.parse(img)
    sel = ix.select(dst="BF16", scale_suffix=(".weight", ".scale_weight"))
    data = img[8 + ix.header_len:]
    want = [sel.materialize(i, data) for i in range(len(sel))]
    total = sum(w.size for w in want)
    assert compare_full(sel, data, {"a": _Result(want), "b": _Result(want)}, threads=3, span=span,
                        batch_bytes=batch) == total
    for i, w in enumerate(want):
        for pos in sorted({0, w.size // 2, w.size - 1}):
            if w.size == 0:
                continue
            bad = [x.copy() for x in want]
            bad[i][pos] ^= 0x40
            with pytest.raises(AssertionError, match=f"b: output {sel.output(i)['name']} element"):
                compare_full(sel, data, {"a": _Result(want), "b": _Result(bad)}, threads=3, span=span,
                             batch_bytes=batch)
