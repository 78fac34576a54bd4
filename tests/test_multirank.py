"""Multi-rank path on CPU (gloo, world size 2): each rank plans its own part
of a checkpoint with st_selection.part/n_parts (host-only plans, no GPU), the
parts are exchanged over the process group, and their union must be every
output exactly once, in order, with the same bytes as the oracle's parts.
The step-time reduction bench.py uses (max over ranks) is checked too, and
that each rank's loads copy only its part's source bytes.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    try:
        import sys
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        sys.path.insert(0, root)
        from safetensors_materialization_gb300 import stmat, synth
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        lay = synth.unet().files[0]
        ix = stmat.Index.from_header(lay.header, lay.data_bytes).view_rename([("model.diffusion_model.", "unet.")])
        plan = ix.plan(dst="BF16", part=rank, n_parts=world, workers=1024, host_only=True)
        mine = ([(o["name"], o["bytes"]) for o in plan.outputs()], plan.copy_bytes()[0], lay.data_bytes,
                plan.copy_ranges())
        parts = [None] * world
        dist.all_gather_object(parts, mine)
        t = torch.tensor([1.5 + rank])        # a stand-in step time per rank
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        q.put((rank, parts, float(t.item())))
        dist.destroy_process_group()
    except Exception as e:  # noqa: BLE001 - reported to the parent
        q.put((rank, repr(e), None))


def test_two_ranks_partition_outputs(stmat, oracle):
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    for rank, parts, tmax in results:
        assert not isinstance(parts, str), parts
        assert tmax == 2.5                      # max over ranks
    assert results[1][1] == results[0][1]       # every rank sees the same split
    # each rank stages only its part's source bytes: under three quarters of the data section each,
    # together the whole of it (plus at most a merged gap at the boundary)
    data_bytes = results[0][1][0][2]
    copied = [c for _, c, _, _ in results[0][1]]
    assert all(c < data_bytes * 3 // 4 for c in copied)
    assert data_bytes <= sum(copied) <= data_bytes + 65536
    parts = [p for p, _, _, _ in results[0][1]]
    ranges = [r for _, _, _, r in results[0][1]]
    from safetensors_materialization_gb300 import synth
    lay = synth.unet().files[0]
    full = stmat.Index.from_header(lay.header, lay.data_bytes).view_rename(
        [("model.diffusion_model.", "unet.")]).plan(dst="BF16", workers=1024, host_only=True)
    everything = [(o["name"], o["bytes"]) for o in full.outputs()]
    assert parts[0] + parts[1] == everything    # disjoint, contiguous, complete
    total = sum(b for _, b in everything)
    biggest = max(b for _, b in everything)
    for p in parts:
        assert abs(sum(b for _, b in p) - total / world) <= biggest
    # the oracle's parts are the same, and each rank copies exactly its outputs' source extents
    # (taken from the oracle's index), merged across gaps under 64 KiB
    oix = oracle.parse_header(lay.header, lay.data_bytes).view_rename([("model.diffusion_model.", "unet.")])
    for r in range(world):
        sel = oix.select(dst="BF16", part=r, nparts=world)
        assert [(o["name"], o["bytes"]) for o in sel.outputs()] == parts[r]
        ext = sorted((oix.entry(o["entry"])["begin"], oix.entry(o["entry"])["end"]) for o in sel.outputs())
        merged = []
        for a, b in ext:
            if merged and a <= merged[-1][1] + 65536:
                merged[-1][1] = max(merged[-1][1], b)
            else:
                merged.append([a, b])
        assert [tuple(m) for m in merged] == ranges[r]
        assert sum(b - a for a, b in ranges[r]) == copied[r]
