"""Whole-output parity helpers for the GPU tests: every element of every
output against the oracle, on all host cores, and guard-band checks of the
destination arenas.

The oracle is plain single-threaded C.  Its ctypes calls release the GIL, so
a thread pool runs one oracle call per host core, each over an element range
of one output (OPlan.materialize_range); the oracle's value for a range is
computed once and compared with the same range of every GPU result given
(several kernel builds, say).  GPU outputs come back to pinned host memory in
batches of a few GiB, so host memory stays bounded at any checkpoint size.

Guard bands: GuardedOutputs places the outputs in one device arena filled
with FILL, with guard bytes before the first output and after the last;
assert_guards checks that every byte no output owns still holds FILL, so a
write past an output's end (into alignment padding, a neighbour's gap or the
tail) fails the test even when every output is right.
"""
import concurrent.futures as cf
import os

import numpy as np
import torch

FILL = 0xA5


def host_threads():
    return max(1, len(os.sched_getaffinity(0)))


class GuardedOutputs:
    """Destinations for a plan: one device arena filled with FILL, each
    output at the plan's `align`-byte arena offset shifted by `guard` bytes,
    and `guard` more bytes after the end."""

    def __init__(self, plan, align=256, guard=4096):
        self.infos = plan.outputs()
        offs, total = plan.arena(align)
        self.offsets = [guard + o for o in offs]
        self.arena = torch.full((guard + total + guard,), FILL, dtype=torch.uint8, device="cuda")
        base = self.arena.data_ptr()
        self.ptrs = torch.tensor([base + o for o in self.offsets] or [0], dtype=torch.int64, device="cuda")

    def raw(self, i):
        return self.arena[self.offsets[i]:self.offsets[i] + self.infos[i]["bytes"]]

    def tensor(self, i):
        """Output i as a typed, shaped tensor (a view into the arena)."""
        from safetensors_materialization_gb300.stmat import torch_dtype
        info = self.infos[i]
        return self.raw(i).view(torch_dtype(info["dtype"])).view(info["shape"])

    def check_guards(self):
        assert_guards(self.arena, self.offsets, [o["bytes"] for o in self.infos])


def gap_ranges(size, offsets, sizes):
    """[start, stop) ranges of [0, size) that no (offset, bytes) output covers."""
    order = np.argsort(np.asarray(offsets, dtype=np.int64), kind="stable")
    starts, stops, at = [], [], 0
    for k in order:
        o, n = int(offsets[k]), int(sizes[k])
        if n == 0:
            continue
        assert o >= at, "outputs overlap in the arena"
        if o > at:
            starts.append(at)
            stops.append(o)
        at = o + n
    if at < size:
        starts.append(at)
        stops.append(size)
    return np.asarray(starts, dtype=np.int64), np.asarray(stops, dtype=np.int64)


def assert_guards(arena, offsets, sizes, fill=FILL, max_gather=1 << 26):
    """Every byte of `arena` (a device uint8 tensor) outside the outputs'
    [offset, offset + bytes) ranges still equals `fill`."""
    starts, stops = gap_ranges(arena.numel(), offsets, sizes)
    lengths = stops - starts
    k = 0
    while k < lengths.size:
        # gather the gap bytes of as many ranges as fit in one index tensor
        j, acc = k, 0
        while j < lengths.size and (acc == 0 or acc + lengths[j] <= max_gather):
            acc += int(min(lengths[j], max_gather))
            j += 1
        st, ln = starts[k:j], np.minimum(lengths[k:j], max_gather)
        if ln.size == 1 and lengths[k] > max_gather:     # one long range: check it in slices
            a, b = int(starts[k]), int(stops[k])
            for s in range(a, b, max_gather):
                seg = arena[s:min(b, s + max_gather)]
                bad = torch.nonzero(seg != fill)
                assert bad.numel() == 0, f"guard byte at arena offset {s + int(bad[0])} was overwritten"
            k = j
            continue
        first = np.repeat(st - (np.cumsum(ln) - ln), ln)
        idx = torch.from_numpy(np.arange(int(ln.sum()), dtype=np.int64) + first).to(arena.device)
        vals = arena[idx]
        bad = torch.nonzero(vals != fill)
        if bad.numel():
            pos = int(idx[int(bad[0])])
            raise AssertionError(f"guard byte at arena offset {pos} was overwritten "
                                 f"({int(bad.numel())} of {idx.numel()} guard bytes in this batch)")
        k = j


def assert_device_equals_host(dev, host, chunk=1 << 30):
    """A device uint8 tensor equals a host uint8 array (numpy or torch),
    compared on the GPU in chunks."""
    h = torch.from_numpy(host) if isinstance(host, np.ndarray) else host
    assert dev.numel() == h.numel()
    for s in range(0, h.numel(), chunk):
        e = min(h.numel(), s + chunk)
        part = h[s:e].to(dev.device, non_blocking=False)
        if not torch.equal(dev[s:e], part):
            bad = int(torch.nonzero(dev[s:e] != part)[0])
            raise AssertionError(f"device bytes differ from the host copy at {s + bad}")


def compare_full(sel, data, results, threads=None, span=1 << 22, batch_bytes=1 << 31):
    """Compares every byte of every output of each GPU result with the
    oracle.  sel: oracle selection (OPlan) of the same outputs in the same
    order; data: the data section the oracle reads (numpy uint8); results:
    {label: object with raw(i) -> device uint8 view of output i}.  Returns the
    number of output bytes compared per result; raises AssertionError with
    the first mismatches."""
    threads = threads or host_threads()
    data = np.ascontiguousarray(data, dtype=np.uint8)
    outs = sel.outputs()
    sizes = [o["bytes"] for o in outs]
    isz = [o["bytes"] // o["numel"] if o["numel"] else 1 for o in outs]
    cap = max([batch_bytes] + sizes)
    labels = list(results)
    cuda = torch.cuda.is_available()
    bufs = {lab: torch.empty(max(1, cap), dtype=torch.uint8, pin_memory=cuda) for lab in labels}
    views = {lab: bufs[lab].numpy() for lab in labels}
    bad = []

    def job(ranges):
        out = []
        for i, off, first, count in ranges:
            want = sel.materialize_range(i, data, first, count)
            a, b = off + first * isz[i], off + (first + count) * isz[i]
            for lab in labels:
                got = views[lab][a:b]
                if not np.array_equal(got, want):
                    k = int(np.flatnonzero(got != want)[0])
                    e = k // isz[i]
                    out.append(f"{lab}: output {outs[i]['name']} element {first + e}: got "
                               f"{got[e * isz[i]:(e + 1) * isz[i]].tobytes().hex()} want "
                               f"{want[e * isz[i]:(e + 1) * isz[i]].tobytes().hex()}")
        return out

    compared = 0
    with cf.ThreadPoolExecutor(threads) as ex:
        i = 0
        while i < len(outs) and not bad:
            # one batch of outputs that fits the host buffers
            batch, at = [], 0
            while i < len(outs) and (not batch or at + sizes[i] <= cap):
                batch.append((i, at))
                at += sizes[i]
                i += 1
            for lab in labels:
                for j, off in batch:
                    if sizes[j]:
                        bufs[lab][off:off + sizes[j]].copy_(results[lab].raw(j), non_blocking=True)
            if cuda:
                torch.cuda.synchronize()
            # element ranges of at most `span` elements; small outputs share a job
            futs, group, elems = [], [], 0
            for j, off in batch:
                n = outs[j]["numel"]
                for first in range(0, n, span):
                    count = min(span, n - first)
                    group.append((j, off, first, count))
                    elems += count
                    if elems >= span:
                        futs.append(ex.submit(job, group))
                        group, elems = [], 0
            if group:
                futs.append(ex.submit(job, group))
            for f in futs:
                bad += f.result()
            compared += at
    assert not bad, "GPU output differs from the oracle:\n" + "\n".join(bad[:8])
    return compared
