"""The lazy single-tensor path and its RAM tier ("Disk tier safetensors
streaming design audit (ComfyUI)": a streaming mapping that loads a tensor
when it is accessed; an LRU cache of RAM-resident weights with a maximum
number of bytes, whose eviction keeps only the disk reference).

CPU: the cache's LRU rules (hits, misses, eviction order, the bound, held
entries, entries above the bound), its bytes against the file, and the
mapping's metadata-only side.  GPU: every tensor of a sharded checkpoint
through StreamStateDict (st_load_tensors) against the oracle, with and
without the cache, per-tensor scaled FP8 and block-scaled weights."""
import os

import numpy as np
import pytest

from safetensors_materialization_gb300 import synth


def blob_file(tmp_path, n=1 << 20, seed=0):
    rng = np.random.Generator(np.random.PCG64(seed))
    data = rng.integers(0, 256, size=n, dtype=np.uint8)
    path = os.path.join(str(tmp_path), "blob.bin")
    data.tofile(path)
    return path, data


def test_cache_lru_rules(stmat, tmp_path):
    import ctypes
    path, data = blob_file(tmp_path)
    files = stmat.Files([(path, 0, data.size, 0)])
    c = stmat.Cache(10_000, pinned=False)

    def read(addr, n):
        return np.ctypeslib.as_array((ctypes.c_uint8 * n).from_address(addr))

    a = c.get(files, 0, 4000)
    assert np.array_equal(read(a, 4000), data[:4000])
    c.release(a)
    b = c.get(files, 5000, 4000)
    c.release(b)
    assert c.stats() == {"bytes": 8000, "max_bytes": 10_000, "entries": 2, "hits": 0, "misses": 2, "evictions": 0}
    a2 = c.get(files, 0, 4000)                 # a hit: the same copy, now the most recent
    assert a2 == a and c.stats()["hits"] == 1
    c.release(a2)
    d = c.get(files, 20_000, 3000)             # needs room: evicts b, the least recently used
    st = c.stats()
    assert st["evictions"] == 1 and st["entries"] == 2 and st["bytes"] == 7000
    assert np.array_equal(read(d, 3000), data[20_000:23_000])
    c.release(d)
    b2 = c.get(files, 5000, 4000)              # b was evicted: a miss, read again
    assert c.stats()["misses"] == 4
    assert np.array_equal(read(b2, 4000), data[5000:9000])
    # eviction skips held entries: b2 is held, so d (the older unheld one) goes
    e = c.get(files, 100_000, 6000)
    st = c.stats()
    assert st["bytes"] == 10_000 and st["entries"] == 2
    c.release(b2)
    c.release(e)
    big = c.get(files, 0, 50_000)              # above the bound: read, not kept
    assert np.array_equal(read(big, 50_000), data[:50_000])
    assert c.stats()["entries"] == 2
    c.release(big)
    with pytest.raises(stmat.StmatError):
        c.release(big)                         # freed on release
    c.clear()
    assert c.stats()["entries"] == 0 and c.stats()["bytes"] == 0
    with pytest.raises(stmat.StmatError) as err:
        c.get(files, data.size - 10, 11)
    assert err.value.status == "ST_E_INVAL"


def test_cache_under_held_pressure(stmat, tmp_path):
    """When everything kept is held, a new entry is still read and kept; the
    bound is restored as holds are released and entries age out."""
    path, data = blob_file(tmp_path, seed=1)
    files = stmat.Files([(path, 0, data.size, 0)])
    c = stmat.Cache(8192, pinned=False)
    held = [c.get(files, k * 4096, 4096) for k in range(3)]
    assert c.stats()["bytes"] == 3 * 4096    # over the bound while held
    for h in held:
        c.release(h)
    x = c.get(files, 600_000, 4096)
    c.release(x)
    assert c.stats()["bytes"] <= 8192


def write_shards(tmp_path, w):
    paths = []
    for k, lay in enumerate(w.files):
        path = os.path.join(str(tmp_path), f"m{k}.safetensors")
        synth.build_workload_file(w, k).tofile(path)
        paths.append(path)
    return paths


def small_llm():
    return synth.llm8b(seed=9, layers=3, hidden=128, inter=352, vocab=400, kv=32, shards=3)


def test_stream_state_dict_metadata_only(stmat, tmp_path):
    torch = pytest.importorskip("torch")
    w = small_llm()
    paths = write_shards(tmp_path, w)
    sd = stmat.StreamStateDict(paths, dst="F16", pinned=False, ram_cache_bytes=1 << 20,
                               rename=[("model.", "")])
    names = [e.name.replace("model.", "", 1) if e.name.startswith("model.") else e.name
             for lay in w.files for e in lay.entries]
    assert sd.keys() == names and len(sd) == len(names)
    assert "layers.0.mlp.up_proj.weight" in sd and "model.norm.weight" not in sd
    m = sd.meta("layers.1.self_attn.q_proj.weight")
    assert m.device.type == "meta" and tuple(m.shape) == (128, 128) and m.dtype == torch.float16
    assert sd.metadata() == {"format": "pt"}
    assert sd.cache.stats()["misses"] == 0     # nothing read so far


def gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return torch


def oracle_joined(oracle, w, paths):
    oix, bases = oracle.concat([oracle.parse_header(l.header, l.data_bytes) for l in w.files])
    arena = np.zeros(oix.data_bytes, np.uint8)
    for k, (b, lay) in enumerate(zip(bases, w.files)):
        img = synth.build_workload_file(w, k)
        arena[b:b + lay.data_bytes] = img[lay.data_start:]
    return oix, arena


@pytest.mark.gpu
@pytest.mark.parametrize("cache_bytes", [0, 1 << 14, 1 << 30])
def test_stream_state_dict_loads_every_tensor(stmat, oracle, tmp_path, cache_bytes):
    torch = gpu()
    w = small_llm()
    paths = write_shards(tmp_path, w)
    sd = stmat.StreamStateDict(paths, dst="BF16", ram_cache_bytes=cache_bytes)
    oix, arena = oracle_joined(oracle, w, paths)
    for rounds in range(2):
        for name in sd.keys():
            t = sd[name]
            torch.cuda.synchronize()
            sel = oix.select(names=[name], dst="BF16")
            assert np.array_equal(t.view(torch.uint8).reshape(-1).cpu().numpy(), sel.materialize(0, arena)), name
    assert sd.check() == 0                                 # no device flag left in the static array
    if cache_bytes:
        st = sd.cache.stats()
        assert st["bytes"] <= cache_bytes
        if cache_bytes == 1 << 30:
            assert st["hits"] == len(sd) and st["misses"] == len(sd)   # the second round hit every tensor


@pytest.mark.gpu
def test_lazy_scaled_and_block_scaled(stmat, oracle, tmp_path):
    torch = gpu()
    import test_blockscale as TB
    img, quant = TB.quant_file(50, lead=5)
    path = os.path.join(str(tmp_path), "q.safetensors")
    img.tofile(path)
    oix = oracle.parse(img)
    data = img[8 + oix.header_len:]
    for dst in ("BF16", "F32"):
        sd = stmat.StreamStateDict([path], dst=dst, quant=quant, ram_cache_bytes=1 << 22)
        for name in ("a.weight", "b.weight", "mid"):
            t = sd[name]
            torch.cuda.synchronize()
            sel = oix.select(names=[name], dst=dst, quant=[quant.get(name)])
            assert np.array_equal(t.view(torch.uint8).reshape(-1).cpu().numpy(), sel.materialize(0, data)), name
    # per-tensor scaled FP8 through the suffix pairing
    w = synth.scaled_fp8(blocks=1)
    lay = w.files[0]
    spath = os.path.join(str(tmp_path), "s.safetensors")
    simg = synth.build_workload_file(w, 0)
    simg.tofile(spath)
    sd = stmat.StreamStateDict([spath], dst="BF16", scale_suffix=w.scale_suffix)
    soix = oracle.parse(simg)
    name = [e.name for e in lay.entries if e.name.endswith(".weight")][3]
    t = sd[name]
    torch.cuda.synchronize()
    sel = soix.select(names=[name], dst="BF16", scale_suffix=w.scale_suffix)
    assert np.array_equal(t.view(torch.uint8).reshape(-1).cpu().numpy(), sel.materialize(0, simg[lay.data_start:]))


@pytest.mark.gpu
def test_lazy_rejects_bad_destinations(stmat, tmp_path):
    torch = gpu()
    w = small_llm()
    paths = write_shards(tmp_path, w)
    files, ix = stmat.Files.of_checkpoint(paths)
    staging = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
    out = torch.empty(4096, dtype=torch.uint8, device="cuda")
    name = "model.norm.weight"
    for bad in (0, out.data_ptr() + 1):
        with pytest.raises(stmat.StmatError) as e:
            ix.load_tensors(files, [bad], staging, names=[name], dst="F32")
        assert e.value.status == "ST_E_INVAL"
    with pytest.raises(stmat.StmatError) as e:       # staging too small
        ix.load_tensors(files, [out.data_ptr()], staging[:16], names=[name], dst="BF16")
    assert e.value.status == "ST_E_INVAL" and "staging needs" in str(e.value)


@pytest.mark.gpu
@pytest.mark.parametrize("cache_kind", ["one_tensor", "none_kept", "all"])
def test_back_to_back_loads_keep_entries_until_copied(stmat, oracle, tmp_path, cache_kind):
    """Loads every tensor without synchronizing in between: a RAM-tier entry
    stays held until the staging copy that reads it has finished, so a small
    tier cannot evict (or free) bytes still in flight; the holds are dropped
    by later cache calls."""
    torch = gpu()
    w = small_llm()
    paths = write_shards(tmp_path, w)
    largest = max(e.nbytes for lay in w.files for e in lay.entries)
    bound = {"one_tensor": largest + largest // 2, "none_kept": 64, "all": 1 << 30}[cache_kind]
    sd = stmat.StreamStateDict(paths, dst="F16", ram_cache_bytes=bound)
    oix, arena = oracle_joined(oracle, w, paths)
    got = {name: sd[name] for name in sd.keys()}          # no synchronization between loads
    torch.cuda.synchronize()
    for name, t in got.items():
        sel = oix.select(names=[name], dst="F16")
        assert np.array_equal(t.view(torch.uint8).reshape(-1).cpu().numpy(), sel.materialize(0, arena)), name
    st = sd.cache.stats()                                 # finds every copy finished: no holds left
    assert st["misses"] == len(got)
    sd.cache.clear()
    assert sd.cache.stats()["entries"] == 0 and sd.cache.stats()["bytes"] == 0


def test_cache_entries_belong_to_their_files_object(stmat, tmp_path):
    """Entries are keyed by the files object's own id, not its address: a
    files object opened after another was closed (the allocator often hands
    out the same address again) never hits the closed one's entries."""
    import ctypes
    rng = np.random.Generator(np.random.PCG64(10))
    paths, datas = [], []
    for k in range(2):
        data = rng.integers(0, 256, size=1 << 16, dtype=np.uint8)
        path = os.path.join(str(tmp_path), f"blob{k}.bin")
        data.tofile(path)
        paths.append(path)
        datas.append(data)
    c = stmat.Cache(1 << 20, pinned=False)
    for k in range(8):
        files = stmat.Files([(paths[k % 2], 0, 1 << 16, 0)])
        h = c.get(files, 100, 4000)
        got = np.ctypeslib.as_array((ctypes.c_uint8 * 4000).from_address(h)).copy()
        c.release(h)
        assert np.array_equal(got, datas[k % 2][100:4100]), k
        files.close()
    assert c.stats()["misses"] == 8 and c.stats()["hits"] == 0


@pytest.mark.gpu
def test_holds_released_when_copies_finish_late(stmat, oracle, tmp_path):
    """RAM-tier hits queued behind a long kernel: the next call finds the
    previous call's copies still in flight (their holds must be kept, not
    lost) and the holds are dropped once the copies are done, so clear() then
    empties the tier."""
    torch = gpu()
    w = small_llm()
    paths = write_shards(tmp_path, w)
    sd = stmat.StreamStateDict(paths, dst="BF16", ram_cache_bytes=1 << 30)
    oix, arena = oracle_joined(oracle, w, paths)
    names = sd.keys()[:6]
    for n in names:                            # misses: each allocates its page-locked entry
        sd[n]
    torch.cuda.synchronize()
    torch.cuda._sleep(200_000_000)             # about 0.1 s of a bounded spin on the current stream
    got = [sd[n] for n in names]              # hits (nothing allocated): their copies queue behind it
    torch.cuda.synchronize()
    st = sd.cache.stats()
    assert st["misses"] == len(names) and st["hits"] == len(names) and st["entries"] == len(names)
    sd.cache.clear()
    assert sd.cache.stats()["entries"] == 0 and sd.cache.stats()["bytes"] == 0
    for n, t in zip(names, got):
        sel = oix.select(names=[n], dst="BF16")
        assert np.array_equal(t.view(torch.uint8).reshape(-1).cpu().numpy(), sel.materialize(0, arena)), n


def scaled_fp8_file(tmp_path):
    """Two E4M3 weights with their one-element F32 scales and an F16 tensor."""
    import test_blockscale as TB
    rng = np.random.Generator(np.random.PCG64(12))
    ents = []
    for k in range(2):
        ents.append((f"l{k}.weight", "F8_E4M3", [24, 40], rng.integers(0, 0x7F, size=960, dtype=np.uint8).tobytes()))
        ents.append((f"l{k}.scale_weight", "F32", [], np.float32(rng.uniform(1e-3, 1e-1)).tobytes()))
    ents.append(("norm", "F16", [40], rng.standard_normal(40).astype(np.float16).tobytes()))
    img = TB.image(ents, lead=3)
    path = os.path.join(str(tmp_path), "s.safetensors")
    img.tofile(path)
    return path, img, (".weight", ".scale_weight")


def test_load_many_batches_check_their_outputs(stmat, tmp_path):
    """A batch whose names include a scale that another name of the batch
    consumes has fewer outputs than names: the host-only plan load_many
    checks each batch with shows it (the batch is then loaded name by name)."""
    path, img, suffix = scaled_fp8_file(tmp_path)
    sd = stmat.StreamStateDict([path], dst="BF16", scale_suffix=suffix, pinned=False)
    outs = sd.index.plan(dst="BF16", names=["l0.weight", "l0.scale_weight"], workers=1, host_only=True,
                         scale_suffix=suffix).outputs()
    assert [o["name"] for o in outs] == ["l0.weight"]       # the scale is consumed: one output for two names
    outs = sd.index.plan(dst="BF16", names=["l0.weight", "norm"], workers=1, host_only=True,
                         scale_suffix=suffix).outputs()
    assert [o["name"] for o in outs] == ["l0.weight", "norm"]


@pytest.mark.gpu
@pytest.mark.parametrize("cache_bytes", [0, 1 << 30])
def test_load_many_matches_oracle(stmat, oracle, tmp_path, cache_bytes):
    """load_many over every tensor (batches split by count and bytes) equals
    the oracle; with a scale suffix, a batch holding a weight and its scale
    falls back to one name at a time."""
    torch = gpu()
    w = small_llm()
    paths = write_shards(tmp_path, w)
    sd = stmat.StreamStateDict(paths, dst="F16", ram_cache_bytes=cache_bytes)
    oix, arena = oracle_joined(oracle, w, paths)
    for kw in (dict(), dict(max_batch=5), dict(max_batch_bytes=1 << 16)):
        got = sd.load_many(sd.keys(), **kw)
        torch.cuda.synchronize()
        assert list(got) == sd.keys()
        for name, t in got.items():
            sel = oix.select(names=[name], dst="F16")
            assert np.array_equal(t.view(torch.uint8).reshape(-1).cpu().numpy(), sel.materialize(0, arena)), name
        assert sd.check() == 0
    spath, simg, suffix = scaled_fp8_file(tmp_path)
    sds = stmat.StreamStateDict([spath], dst="BF16", scale_suffix=suffix)
    soix = oracle.parse(simg)
    names = sds.keys()                                     # weights and their scales together
    got = sds.load_many(names)
    torch.cuda.synchronize()
    data = simg[8 + soix.header_len:]
    for name in names:
        sel = soix.select(names=[name], dst="BF16", scale_suffix=suffix)
        assert np.array_equal(got[name].reshape(-1).view(torch.uint8).cpu().numpy(), sel.materialize(0, data)), name


@pytest.mark.gpu
@pytest.mark.parametrize("cache_bytes", [0, 1 << 30])
def test_lazy_slices_match_oracle(stmat, oracle, tmp_path, cache_bytes):
    """sd.slice(name, dim, start, stop): one tensor-parallel rank's rows or
    columns read and gathered on access, on every 2-D tensor of a sharded
    checkpoint along both dimensions, against the oracle's sliced outputs."""
    torch = gpu()
    w = small_llm()
    paths = write_shards(tmp_path, w)
    sd = stmat.StreamStateDict(paths, dst="BF16", ram_cache_bytes=cache_bytes)
    oix, arena = oracle_joined(oracle, w, paths)
    checked = 0
    for name in sd.keys():
        shape, _ = sd.info(name)
        if len(shape) != 2:
            continue
        for dim in (0, 1):
            n = shape[dim]
            start, stop = n // 4, n // 4 + max(1, n // 3)
            t = sd.slice(name, dim, start, stop)
            torch.cuda.synchronize()
            want_shape = list(shape)
            want_shape[dim] = stop - start
            assert list(t.shape) == want_shape
            sel = oix.select(names=[name], dst="BF16", slices=[(dim, start, stop)])
            assert np.array_equal(t.reshape(-1).view(torch.uint8).cpu().numpy(), sel.materialize(0, arena)), (name, dim)
            checked += 1
    assert checked >= 20


@pytest.mark.gpu
def test_lazy_row_slice_reads_only_its_rows(stmat, oracle, tmp_path):
    """A dim-0 slice stages only its rows: the RAM tier then holds exactly
    those bytes (a tensor-parallel rank reads its share of the file), and the
    output still equals the oracle's."""
    torch = gpu()
    w = small_llm()
    paths = write_shards(tmp_path, w)
    sd = stmat.StreamStateDict(paths, dst="BF16", ram_cache_bytes=1 << 30)
    oix, arena = oracle_joined(oracle, w, paths)
    name = "model.layers.1.mlp.up_proj.weight"
    shape, _ = sd.info(name)
    rows = shape[0]
    t = sd.slice(name, 0, rows // 4, rows // 2)
    torch.cuda.synchronize()
    e = sd.index.entry(sd._pos[name])
    row_bytes = (e["end"] - e["begin"]) // rows
    assert sd.cache.stats()["bytes"] == (rows // 2 - rows // 4) * row_bytes
    sel = oix.select(names=[name], dst="BF16", slices=[(0, rows // 4, rows // 2)])
    assert np.array_equal(t.reshape(-1).view(torch.uint8).cpu().numpy(), sel.materialize(0, arena))


def test_cache_is_thread_safe(stmat, tmp_path):
    """Six host threads get and release random ranges of one file through one
    small RAM tier (evictions all the time): every copy holds its bytes, and
    once nothing is held the tier is within its bound and its counters add
    up."""
    import ctypes
    import threading
    path, data = blob_file(tmp_path, n=4 << 20, seed=5)
    files = stmat.Files([(path, 0, data.size, 0)])
    c = stmat.Cache(1 << 20, pinned=False)
    errors, calls = [], []

    def worker(seed):
        r = np.random.Generator(np.random.PCG64(seed))
        k = 0
        for _ in range(150):
            begin = int(r.integers(0, 64)) * 65536               # a few distinct ranges: hits and misses
            n = int(r.integers(1, 8)) * 16384
            n = min(n, data.size - begin)
            h = c.get(files, begin, n, threads=int(r.integers(1, 4)))
            got = np.ctypeslib.as_array((ctypes.c_uint8 * n).from_address(h)).copy()
            c.release(h)
            k += 1
            if not np.array_equal(got, data[begin:begin + n]):
                errors.append((seed, begin, n))
        calls.append(k)

    ts = [threading.Thread(target=worker, args=(s,)) for s in range(6)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors
    st = c.stats()
    assert st["bytes"] <= st["max_bytes"]
    assert st["hits"] + st["misses"] == sum(calls) == 900
    c.clear()
    assert c.stats()["entries"] == 0
    files.close()


@pytest.mark.gpu
def test_items_in_batches_match_oracle(stmat, oracle, tmp_path):
    """StreamStateDict.items(): every tensor in key order, loaded in batches,
    equals the oracle's output."""
    torch = gpu()
    w = small_llm()
    paths = write_shards(tmp_path, w)
    sd = stmat.StreamStateDict(paths, dst="BF16", ram_cache_bytes=1 << 30)
    oix, arena = oracle_joined(oracle, w, paths)
    names = []
    for name, t in sd.items(batch=7):
        names.append(name)
        torch.cuda.synchronize()
        sel = oix.select(names=[name], dst="BF16")
        assert np.array_equal(t.reshape(-1).view(torch.uint8).cpu().numpy(), sel.materialize(0, arena)), name
    assert names == sd.keys()


@pytest.mark.gpu
@pytest.mark.parametrize("cache_bytes", [0, 1 << 30])
def test_lazy_batch_into_guarded_arena(stmat, oracle, tmp_path, cache_bytes):
    """One st_load_tensors call for every tensor of a checkpoint into one
    guard-banded arena: every output equals the oracle's and no byte outside
    the outputs is written."""
    torch = gpu()
    from oracle_compare import GuardedOutputs
    w = small_llm()
    paths = write_shards(tmp_path, w)
    sd = stmat.StreamStateDict(paths, dst="BF16", ram_cache_bytes=cache_bytes)
    oix, arena = oracle_joined(oracle, w, paths)
    names = sd.keys()
    plan = sd.index.plan(dst="BF16", names=names, workers=1, host_only=True)
    outs = GuardedOutputs(plan)
    staging = torch.empty(2 * arena.size + (1 << 20), dtype=torch.uint8, device="cuda")
    ptrs = [outs.arena.data_ptr() + o for o in outs.offsets]
    sd.index.load_tensors(sd.files, ptrs, staging, names, dst="BF16", cache=sd.cache,
                          stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert sd.check() == 0
    outs.check_guards()
    sel = oix.select(names=names, dst="BF16")
    for i in range(len(sel)):
        assert np.array_equal(outs.raw(i).cpu().numpy(), sel.materialize(i, arena)), names[i]
