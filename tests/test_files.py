"""Shard files on disk: st_index_open (header only), st_files_open/read
(range reads with pread, several threads) against the bytes the files were
written from, the error statuses, and (GPU) st_load_files, the disk -> pinned
-> device -> materialize pipeline, against the oracle.

"Disk tier safetensors streaming design audit (ComfyUI)", "Range reads and
tiering": Disk->RAM->GPU reads only the ranges asked for into (pinned) host
memory and copies them to the GPU."""
import os

import numpy as np
import pytest

from oracle_compare import GuardedOutputs
from safetensors_materialization_gb300 import synth


def write_shards(tmp_path, w):
    """Writes every shard of workload `w`; returns (paths, data sections)."""
    paths, datas = [], []
    for k, lay in enumerate(w.files):
        img = synth.build_workload_file(w, k)
        path = os.path.join(tmp_path, f"shard{k}.safetensors")
        img.tofile(path)
        paths.append(path)
        datas.append(img[lay.data_start:])
    return paths, datas


def small_llm():
    return synth.llm8b(seed=7, layers=4, hidden=128, inter=352, vocab=500, kv=32, shards=4)


def test_index_open_reads_only_the_header(stmat, oracle, tmp_path):
    w = small_llm()
    paths, datas = write_shards(str(tmp_path), w)
    for path, lay in zip(paths, w.files):
        ix, off = stmat.Index.open(path)
        assert off == lay.data_start
        assert ix.sizes() == (lay.header_len, lay.data_bytes)
        assert ix.entries() == stmat.Index.from_header(lay.header, lay.data_bytes).entries()


@pytest.mark.parametrize("threads", [1, 3, 8])
def test_files_read_the_joined_arena(stmat, tmp_path, threads):
    w = small_llm()
    paths, datas = write_shards(str(tmp_path), w)
    files, ix = stmat.Files.of_checkpoint(paths)
    _, bases = stmat.Index.concat([stmat.Index.open(p)[0] for p in paths])
    total = ix.sizes()[1]
    want = np.zeros(total, np.uint8)
    for b, d in zip(bases, datas):
        want[b:b + d.size] = d
    got = np.zeros(total, np.uint8)
    files.read(0, total, got, threads=threads)
    assert np.array_equal(got, want)
    rng = np.random.Generator(np.random.PCG64(threads))
    for _ in range(20):                       # ranges crossing shard boundaries
        a = int(rng.integers(0, total))
        n = int(rng.integers(0, min(3 << 20, total - a) + 1))
        part = np.full(n, 0xEE, np.uint8)
        files.read(a, n, part, threads=threads)
        # gap bytes between shards are left untouched
        ref = want[a:a + n].copy()
        covered = np.zeros(total, bool)
        for b, d in zip(bases, datas):
            covered[b:b + d.size] = True
        ref[~covered[a:a + n]] = 0xEE
        assert np.array_equal(part, ref)


def test_concurrent_reads_share_the_reader_pool(stmat, tmp_path):
    """Several host threads read different ranges of one files object at
    once (each read split over the object's reader threads); every read gets
    its own bytes."""
    import threading
    rng = np.random.Generator(np.random.PCG64(3))
    data = rng.integers(0, 256, size=24 << 20, dtype=np.uint8)
    path = os.path.join(str(tmp_path), "big.bin")
    data.tofile(path)
    files = stmat.Files([(path, 0, data.size, 0)])
    errors = []

    def worker(seed):
        r = np.random.Generator(np.random.PCG64(seed))
        for _ in range(12):
            begin = int(r.integers(0, data.size - 1))
            n = int(r.integers(1, min(data.size - begin, 5 << 20) + 1))
            got = np.empty(n, np.uint8)
            files.read(begin, n, got, threads=int(r.integers(1, 9)))
            if not np.array_equal(got, data[begin:begin + n]):
                errors.append((seed, begin, n))

    ts = [threading.Thread(target=worker, args=(s,)) for s in range(6)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors
    files.close()


def test_file_errors(stmat, tmp_path):
    w = small_llm()
    paths, datas = write_shards(str(tmp_path), w)
    with pytest.raises(stmat.StmatError) as e:
        stmat.Index.open(os.path.join(str(tmp_path), "missing.safetensors"))
    assert e.value.status == "ST_E_IO"
    short = os.path.join(str(tmp_path), "short.safetensors")
    with open(paths[0], "rb") as f:
        head = f.read(100)
    with open(short, "wb") as f:
        f.write(head)
    with pytest.raises(stmat.StmatError) as e:
        stmat.Index.open(short)
    assert e.value.status == "ST_E_TRUNCATED"
    size0 = os.path.getsize(paths[0])
    with pytest.raises(stmat.StmatError) as e:          # the file is shorter than the part
        stmat.Files([(paths[0], 0, size0 + 1, 0)])
    assert e.value.status == "ST_E_IO"
    with pytest.raises(stmat.StmatError) as e:          # parts overlap in the arena
        stmat.Files([(paths[0], 0, 100, 0), (paths[1], 0, 100, 50)])
    assert e.value.status == "ST_E_INVAL"
    files = stmat.Files([(paths[0], 0, 100, 0)])
    with pytest.raises(stmat.StmatError) as e:          # beyond the arena
        files.read(50, 51, np.zeros(51, np.uint8))
    assert e.value.status == "ST_E_INVAL"
    # a file truncated after opening: the read fails with the OS's story
    victim = os.path.join(str(tmp_path), "victim.safetensors")
    with open(paths[1], "rb") as f:
        blob = f.read()
    with open(victim, "wb") as f:
        f.write(blob)
    files = stmat.Files([(victim, 0, len(blob), 0)])
    os.truncate(victim, len(blob) // 2)
    with pytest.raises(stmat.StmatError) as e:
        files.read(0, len(blob), np.zeros(len(blob), np.uint8), threads=2)
    assert e.value.status == "ST_E_IO"


@pytest.mark.parametrize("threads", [0, 1, 3])
def test_prefetch_and_its_guard(stmat, tmp_path, threads):
    """st_files_prefetch faults the mappings in (the step ring-less loads take
    before each copy); a file that shrank after opening is ST_E_IO there, so a
    ring-less load stops before queueing a copy of missing pages."""
    w = small_llm()
    paths, datas = write_shards(str(tmp_path), w)
    files, ix = stmat.Files.of_checkpoint(paths)
    total = ix.sizes()[1]
    files.prefetch(threads=threads)
    files.prefetch(total // 3, total // 3, threads=threads)
    files.prefetch(total, 0)
    got = np.zeros(total, np.uint8)
    files.read(0, total, got, threads=2)                  # unchanged by the prefetch
    with pytest.raises(stmat.StmatError) as e:
        files.prefetch(total - 10, 11)
    assert e.value.status == "ST_E_INVAL"
    files.close()
    blob = os.path.join(str(tmp_path), "blob.bin")
    np.arange(3 << 20, dtype=np.uint32).astype(np.uint8).tofile(blob)
    bf = stmat.Files([(blob, 4096, (3 << 20) - 4096, 0)])
    bf.prefetch(threads=threads)
    os.truncate(blob, 1 << 20)                            # drops 2 MiB: many whole pages of any size
    with pytest.raises(stmat.StmatError) as e:
        bf.prefetch(threads=threads)
    assert e.value.status == "ST_E_IO" and "shrink" in str(e.value)
    bf.prefetch(0, (1 << 19), threads=threads)            # the part still in the file is fine
    bf.close()


@pytest.mark.gpu
@pytest.mark.parametrize("chunk,slots", [(0, 1), (1 << 16, 2), (1 << 20, 3), (3 << 20, 2),
                                         (0, 0), (1 << 16, 0), (3 << 20, 0)])
def test_load_files_matches_oracle(stmat, oracle, tmp_path, chunk, slots):
    """slots == 0: ring-less, every chunk copied from the files' mappings."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    w = small_llm()
    paths, datas = write_shards(str(tmp_path), w)
    files, ix = stmat.Files.of_checkpoint(paths)
    total = ix.sizes()[1]
    for dst in ("BF16", "F16"):
        plan = ix.plan(dst=dst, chunk_bytes=chunk)
        C = chunk or total
        ring = torch.empty(C * slots, dtype=torch.uint8).pin_memory() if slots else None
        dev = torch.full((total,), 0xA5, dtype=torch.uint8, device="cuda")
        outs = GuardedOutputs(plan)
        copy = torch.cuda.Stream()
        plan.load_files(files, dev, outs.ptrs, ring, threads=4, copy_stream=copy,
                        compute_stream=torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert plan.check() == 0
        oix, obases = oracle.concat([oracle.parse_header(l.header, l.data_bytes) for l in w.files])
        arena = np.zeros(total, np.uint8)
        for b, d in zip(obases, datas):
            arena[b:b + d.size] = d
        sel = oix.select(dst=dst)
        for i in range(len(sel)):
            assert np.array_equal(outs.raw(i).cpu().numpy(), sel.materialize(i, arena)), sel.output(i)["name"]
        outs.check_guards()


@pytest.mark.gpu
def test_load_files_ringless_block_scaled_and_errors(stmat, oracle, tmp_path):
    """Ring-less loads of block-scaled weights through a view (scales read by
    the kernel from chunks landed earlier), a ring pointer without a size and
    the reverse, and the files closed right after a load returns."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    assert isinstance(stmat.reads_pageable(0), bool)
    import test_blockscale as TB
    img, quant = TB.quant_file(70, lead=3)
    path = os.path.join(str(tmp_path), "q.safetensors")
    img.tofile(path)
    oix = oracle.parse(img)
    data = img[8 + oix.header_len:]
    for chunk in (0, 1 << 12, 5000):
        files, ix = stmat.Files.of_checkpoint([path])
        names, q = TB.selection(ix, quant)
        plan = ix.plan(dst="BF16", names=names, quant=q, chunk_bytes=chunk)
        dev = torch.empty(data.size, dtype=torch.uint8, device="cuda")
        outs = GuardedOutputs(plan)
        plan.load_files(files, dev, outs.ptrs, None, copy_stream=torch.cuda.Stream(),
                        compute_stream=torch.cuda.current_stream())
        files.close()                                      # the copies are done when load_files returns
        torch.cuda.synchronize()
        assert plan.check() == 0
        sel = oix.select(names=names, dst="BF16", quant=q)
        for i in range(len(sel)):
            assert np.array_equal(outs.raw(i).cpu().numpy(), sel.materialize(i, data)), sel.output(i)["name"]
        outs.check_guards()
    files, ix = stmat.Files.of_checkpoint([path])
    plan = ix.plan(dst="F32")
    dev = torch.empty(data.size, dtype=torch.uint8, device="cuda")
    outs = GuardedOutputs(plan)
    ring = torch.empty(1 << 20, dtype=torch.uint8).pin_memory()
    for args in ((None, 4096), (ring, 0)):
        with pytest.raises(stmat.StmatError) as e:
            plan.load_files(files, dev, outs.ptrs, args[0], ring_bytes=args[1])
        assert e.value.status == "ST_E_INVAL"
    torch.cuda.synchronize()


@pytest.mark.gpu
def test_load_files_empty_data_sections(stmat, tmp_path):
    """Checkpoints whose data sections are empty (a header alone; zero-size
    tensors): both load modes queue nothing and succeed."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import json
    import struct
    for k, ents in enumerate(({}, {"z": {"dtype": "F16", "shape": [0, 4], "data_offsets": [0, 0]}})):
        h = json.dumps(ents).encode()
        path = os.path.join(str(tmp_path), f"e{k}.safetensors")
        with open(path, "wb") as f:
            f.write(struct.pack("<Q", len(h)) + h)
        files, ix = stmat.Files.of_checkpoint([path])
        assert ix.sizes()[1] == 0
        plan = ix.plan(dst="BF16", chunk_bytes=1 << 20)
        outs = GuardedOutputs(plan)
        dev = torch.empty(16, dtype=torch.uint8, device="cuda")
        ring = torch.empty(1 << 20, dtype=torch.uint8).pin_memory()
        plan.load_files(files, dev, outs.ptrs)
        plan.load_files(files, dev, outs.ptrs, ring)
        torch.cuda.synchronize()
        assert plan.check() == 0
        files.close()


@pytest.mark.gpu
def test_host_affinity_binds_to_the_gpu_socket(stmat):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    before = os.sched_getaffinity(0)
    try:
        cpus = stmat.host_affinity(0, apply=False)
        assert cpus and cpus[0].isdigit()
        assert os.sched_getaffinity(0) == before          # apply=False changes nothing
        stmat.host_affinity(0, apply=True)
        now = os.sched_getaffinity(0)
        listed = set()
        for item in cpus.split(","):
            a, _, b = item.partition("-")
            listed |= set(range(int(a), int(b or a) + 1))
        assert now == listed
    finally:
        os.sched_setaffinity(0, before)


@pytest.mark.gpu
@pytest.mark.parametrize("chunk", [0, 1 << 20, 3 << 20])
def test_tensor_parallel_rank_copies_only_its_ranges(stmat, oracle, tmp_path, chunk):
    """A tensor-parallel rank's plan reads under three quarters of the data
    section, so st_load and both st_load_files modes copy only the byte
    ranges it reads (bytes outside them keep the device buffer's fill); the
    outputs equal the oracle's sliced outputs."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    w = synth.llm8b(seed=8, layers=2, hidden=1024, inter=2816, vocab=4000, kv=256, shards=2)
    paths, datas = write_shards(str(tmp_path), w)
    files, ix = stmat.Files.of_checkpoint(paths)
    total = ix.sizes()[1]
    oix, obases = oracle.concat([oracle.parse_header(l.header, l.data_bytes) for l in w.files])
    arena = np.zeros(total, np.uint8)
    for b, d in zip(obases, datas):
        arena[b:b + d.size] = d
    host = torch.from_numpy(arena).pin_memory()
    entries = [e for lay in w.files for e in lay.entries]
    probe = "model.layers.0.mlp.up_proj.weight"          # split on dim 0: rank 0 never reads its last rows
    probe_end = [e for e in ix.entries() if e["name"] == probe][0]["end"]
    for rank in (0, 3):
        tp = synth.tp_slices(entries, 4, rank)
        names = list(tp)
        slices = [tp[n] for n in names]
        plan = ix.plan(dst="BF16", names=names, slices=slices, chunk_bytes=chunk)
        sel = oix.select(names=names, dst="BF16", slices=slices)
        want = [sel.materialize(i, arena) for i in range(len(sel))]
        for mode in ("pinned", "ringless", "ring"):
            dev = torch.full((total,), 0xA5, dtype=torch.uint8, device="cuda")
            outs = GuardedOutputs(plan)
            copy = torch.cuda.Stream()
            cur = torch.cuda.current_stream()
            if mode == "pinned":
                plan.load(host, dev, outs.ptrs, copy_stream=copy, compute_stream=cur)
            elif mode == "ringless":
                plan.load_files(files, dev, outs.ptrs, None, copy_stream=copy, compute_stream=cur)
            else:
                C = chunk or total
                ring = torch.empty(2 * C, dtype=torch.uint8).pin_memory()
                plan.load_files(files, dev, outs.ptrs, ring, threads=4, copy_stream=copy, compute_stream=cur)
            torch.cuda.synchronize()
            assert plan.check() == 0
            for i in range(len(want)):
                assert np.array_equal(outs.raw(i).cpu().numpy(), want[i]), (mode, sel.output(i)["name"])
            outs.check_guards()
            if rank == 0:
                assert int(dev[probe_end - 1].item()) == 0xA5, mode   # never copied: the plan does not read it
    files.close()
