"""CPU model of the materialize kernel's address arithmetic (no GPU).

Restates, per piece, how the kernel splits a piece into a scalar head, a
vector body of SB-byte source steps (16, 8 or 4 bytes by class) and a
scalar tail, and checks that for
the plans the GPU tests and the benchmark run, every byte the kernel reads
lies in the data section, every byte it writes lies in the piece's output,
and head + body + tail cover the piece's elements exactly once.  Data bases
are taken at every residue mod 16 and destinations at 256-byte and at
itemsize-only alignment.  The item sizes and lane steps it uses are checked
against the library's st_class_step (which the kernels' codecs are checked
against at compile time); the address arithmetic restates csrc/st_kernels.cu
(run_piece; produce and consume_seg of the TMA builds, whose bulk copies also
need 16-byte aligned windows inside the data section that fit the warp's
shared-memory slot).
"""
import numpy as np
import pytest

# class -> (source itemsize, output itemsize) in counted units
CLS = {0: (1, 1), 1: (4, 2), 2: (4, 2), 3: (2, 2), 4: (2, 4), 5: (2, 2), 6: (2, 4),
       7: (1, 2), 8: (1, 2), 9: (1, 4), 10: (1, 2), 11: (1, 2), 12: (1, 4),
       # block-scaled: fp8 elements (13-18), NVFP4 bytes of two elements (19-21)
       13: (1, 2), 14: (1, 2), 15: (1, 4), 16: (1, 2), 17: (1, 2), 18: (1, 4), 19: (1, 4), 20: (1, 4), 21: (1, 8)}
NVFP4 = (19, 20, 21)


def step_shape(cls):
    """(SB, KS, OS) of a class's lane step in the TMA consumer."""
    si, so = CLS[cls]
    if cls >= 13:
        sb = 4 if cls in NVFP4 or so == 4 else 8
        return sb, sb, sb * so
    sb = 16 * si // so if so > si else 16
    return sb, sb // si, (sb // si) * so


def stream_step(si, so):
    """(SB, KS, OS) of a per-tensor class's lane step in the streaming body."""
    sb = 16 * si // so if so > si else 16
    return sb, sb // si, (sb // si) * so


def test_model_steps_match_the_library(stmat):
    """The model's item sizes and lane steps are the constants the library
    exports (which its kernels' codecs are checked against when compiled), so
    the model cannot drift from the kernels silently."""
    for cls, (si, so) in CLS.items():
        lib = stmat.class_step(cls)
        assert lib[:2] == (si, so), cls
        assert lib[2:] == step_shape(cls), cls
        if cls < 13:
            assert lib[2:] == stream_step(si, so), cls
    with pytest.raises(stmat.StmatError):
        stmat.class_step(len(CLS))


def split(src, dst, n, si, so, lo, hi):
    """Mirror of run_piece: returns (head, steps, elements per step, source
    window of the vector body, destination range of the body, its alignment)."""
    SB, KS, OS = stream_step(si, so)   # source bytes, elements and output bytes per lane step
    A = OS
    head = ((A - (dst & (A - 1))) & (A - 1)) // so
    head = min(head, n)
    nst = (n - head) // KS
    sa = src + head * si
    r = sa & (SB - 1)
    if r and nst:
        if (sa & ~(SB - 1)) < lo:
            head += KS
            nst -= 1
            sa += SB
        if nst and (sa & ~(SB - 1)) + SB * nst + SB > hi:
            nst -= 1
    sbase = sa & ~(SB - 1)
    win = (sbase, sbase + SB * nst + (SB if r else 0)) if nst else None
    dbase = dst + head * so
    return head, nst, KS, win, (dbase, dbase + nst * OS) if nst else None, A


def _tma_consts():
    """Segment size and slots of the TMA build, read from the kernel source."""
    import os
    import re
    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "safetensors_materialization_gb300", "csrc", "st_kernels.cu")).read()
    seg = int(re.search(r"#define ST_TMA_SEG (\d+)", src).group(1))
    slots = int(re.search(r"#define ST_TMA_SLOTS (\d+)", src).group(1))
    return seg, slots


SEG, SLOTS = _tma_consts()
SLOT_BYTES = SEG + 32


def tma_run(src, dst, n, si, so, lo, hi):
    """Mirror of the TMA build on one run (materialize_tma's produce and
    consume_seg): yields per segment the bulk-copy window, the global scalar
    reads, the shared-memory reads and the stores, and checks each against
    the rules a bulk copy and the slot impose."""
    SB = 16 * si // so if so > si else 16
    KS = SB // si
    OS = KS * so
    lo16 = (lo + 15) & ~15
    hi16 = hi & ~15
    covered = []
    e = 0
    while e < n:
        ln = min(SEG // si, n - e)
        s = src + e * si
        A, Z = 0, ln
        if s < lo16:
            A = min(ln, (lo16 - s + si - 1) // si)
        if s + ln * si > hi16:
            Z = (hi16 - s) // si if hi16 > s else 0
        Z = max(Z, A)
        nbytes, off = 0, 0
        if Z > A:
            w0 = (s + A * si) & ~15
            w1 = (s + Z * si + 15) & ~15
            nbytes, off = w1 - w0, s + A * si - w0
            assert w0 % 16 == 0 and nbytes % 16 == 0 and 0 < nbytes <= SEG + 16
            assert lo <= lo16 <= w0 and w1 <= hi16 <= hi, (w0, w1, lo16, hi16)
            assert 0 <= off < 16
        for x in list(range(0, A)) + list(range(Z, ln)):   # byte loads from the data section
            assert lo <= s + x * si and s + (x + 1) * si <= hi
        m = Z - A
        dp = dst + (e + A) * so
        h = min(((OS - (dp & (OS - 1))) & (OS - 1)) // so, m)
        nst = (m - h) // KS
        t0 = h + nst * KS
        for x in list(range(0, h)) + list(range(t0, m)):   # scalar reads from the slot
            assert off + (x + 1) * si <= nbytes
        if nst:
            q = off + h * si
            r = q & (SB - 1)
            end = (q - r) + (nst + (1 if r else 0)) * SB
            assert end <= SLOT_BYTES
            assert q + nst * SB <= nbytes          # the bytes used were copied
            assert (dp + h * so) % OS == 0
        covered.append((e, e + ln))
        e += ln
    return covered


def consume_model(off, ln, a, z, nbytes, dst, si, so, cls=None):
    """Mirror of consume_seg / consume_quant for one slot: the slot reads
    stay inside the slot and inside the copied bytes; vector stores aligned."""
    if cls is not None:
        SB, KS, OS = step_shape(cls)
    else:
        SB = 16 * si // so if so > si else 16
        KS = SB // si
        OS = KS * so
    m = z - a
    dp = dst + a * so
    h = min(((OS - (dp & (OS - 1))) & (OS - 1)) // so, m)
    if dp & (so - 1):          # 8-byte units at a 4-aligned destination: element by element
        h = m
    nst = (m - h) // KS
    t0 = h + nst * KS
    for x in list(range(0, h)) + list(range(t0, m)):   # scalar reads from the slot
        assert off + (x + 1) * si <= nbytes
    if nst:
        q = off + h * si
        r = q & (SB - 1)
        assert (q - r) + (nst + (1 if r else 0)) * SB <= SLOT_BYTES
        assert q + nst * SB <= nbytes
        assert (dp + h * so) % OS == 0


def tma_warp(plan, pieces, bases, data_base, lo, hi, quant=None):
    """Mirror of materialize_tma's producer over one warp's pieces (batches of
    32, segments of at most SEG source bytes): every bulk copy is 16-byte
    aligned, inside the 16-byte aligned interior of the data section and fits
    its slot; every element of every run is produced exactly once."""
    lo16, hi16 = (lo + 15) & ~15, hi & ~15
    done = {}
    for b0 in range(0, len(pieces), 32):
        batch = pieces[b0:b0 + 32]
        i, r, e = 0, 0, 0
        while i < len(batch):
            p = batch[i]
            if p["count"] == 0 or r >= p["rows"]:
                i, r, e = i + 1, 0, 0
                continue
            si, so = CLS[p["cls"]]
            cnt = p["count"]
            ln = min(SEG // si, cnt - e)
            if p["cls"] >= 13:   # block-scaled: one row, scales fit the slot's scale area
                q = quant[p["output"]]
                nv = p["cls"] in NVFP4
                u = p["dst"] // so + e
                row, colu = divmod(u, q["row_units"])
                ln = min(ln, q["row_units"] - colu)
                col0 = 2 * colu if nv else colu
                ss = 1 if nv else 4
                bc = 1 << q["bc_shift"]
                max_el = (256 if nv else 32) * bc - (col0 & (bc - 1))
                ln = min(ln, max_el // 2 if nv else max_el)
                el = 2 * ln if nv else ln
                b0 = col0 >> q["bc_shift"]
                nblk = ((col0 + el - 1) >> q["bc_shift"]) - b0 + 1
                g = data_base + q["scale"] + ((row >> q["br_shift"]) * q["scols"] + b0) * ss
                sw0, sw1 = g & ~15, (g + nblk * ss + 15) & ~15
                if sw0 >= lo16 and sw1 <= hi16:
                    assert sw1 - sw0 <= 288 and (sw1 - sw0) % 16 == 0
                else:
                    assert lo <= g and g + nblk * ss <= hi
                assert ln >= 1
            s = data_base + p["src"] + r * p["pitch"] + e * si
            A, Z = 0, ln
            if s < lo16:
                A = min(ln, (lo16 - s + si - 1) // si)
            if s + ln * si > hi16:
                Z = (hi16 - s) // si if hi16 > s else 0
            Z = max(Z, A)
            nbytes = off = w0 = 0
            if Z > A:
                w0 = (s + A * si) & ~15
                w1 = (s + Z * si + 15) & ~15
                nbytes, off = w1 - w0, s + A * si - w0
            for x in list(range(0, A)) + list(range(Z, ln)):
                assert lo <= s + x * si and s + (x + 1) * si <= hi
            dst0 = bases[p["output"]] + p["dst"] + (r * cnt + e) * so
            subs = [(off, ln, A, Z, dst0, si, so, p["cls"])]
            done.setdefault((id(p), r), []).append((e, e + ln))
            e += ln
            if e == cnt:
                e = 0
                r += 1
                if r == p["rows"]:
                    r = 0
                    i += 1
            if nbytes:
                assert w0 % 16 == 0 and nbytes % 16 == 0 and 0 < nbytes <= SEG + 16
                assert lo <= lo16 <= w0 and w0 + nbytes <= hi16 <= hi
            for (o, ln2, a2, z2, d2, si2, so2, c2) in subs:
                consume_model(o, ln2, a2, z2, nbytes, d2, si2, so2, c2)
    for p in pieces:
        for r in range(p["rows"]):
            got = sorted(done.get((id(p), r), []))
            pos = 0
            for a_, b_ in got:
                assert a_ == pos
                pos = b_
            assert pos == p["count"]


def check_plan(plan, data_base, dst_align, data_bytes):
    outs = plan.outputs()
    st = plan.stats()
    # output bases: consecutive, each aligned to dst_align (>= itemsize)
    bases, at = [], 1 << 20
    for o in outs:
        isz = max(1, o["bytes"] // max(1, o["numel"]))
        a = max(dst_align, isz)
        at = (at + a - 1) // a * a
        if dst_align < 16:
            at += isz if (at // isz) % 2 == 0 else 0  # deliberately not 16-byte aligned
        bases.append(at)
        at += o["bytes"]
    lo, hi = data_base, data_base + data_bytes
    pieces = [plan.piece(k) for k in range(st["pieces"])]
    for p in pieces:
        for r in range(p["rows"]):
            check_run(p, r, bases, outs, data_base, lo, hi)
    for c in range(st["chunks"]):
        # each warp's own share, then the claimed pieces (any warp may take a
        # claimed batch; the windows depend on the piece alone)
        for w in range(st["workers"] + 1):
            a, b = plan.worker(c, w)
            tma_warp(plan, pieces[a:b], bases, data_base, lo, hi)
    # grid: blocks of 8 warps cover every worker; parts arrays have workers + 1 entries
    blocks = (st["workers"] + 7) // 8
    assert blocks * 8 >= st["workers"]
    for c in range(st["chunks"]):
        a, b = plan.worker(c, st["workers"])
        assert plan.worker(c, st["workers"] - 1)[1] == a and b <= st["pieces"]


def check_run(p, r, bases, outs, data_base, lo, hi):
    """Run r of piece p (the kernel's run_rows: source + r * pitch, output +
    r * count * itemsize) against the data section and its output."""
    if True:
        si, so = CLS[p["cls"]]
        n = p["count"]
        src = data_base + p["src"] + r * p["pitch"]
        out_base = bases[p["output"]]
        assert out_base % so == 0
        dst = out_base + p["dst"] + r * n * so
        head, nch, K, win, drange, A = split(src, dst, n, si, so, lo, hi)
        assert 0 <= head <= n and head + nch * K <= n
        # scalar elements read [src + e si, +si) for e in head ∪ tail, all inside the piece's bytes
        assert lo <= src and src + n * si <= hi
        if win:
            assert lo <= win[0] and win[1] <= hi, (k, win, lo, hi)
            assert drange[0] % A == 0
            assert out_base <= drange[0] and drange[1] <= out_base + outs[p["output"]]["bytes"]
        assert dst + n * so <= out_base + outs[p["output"]]["bytes"]
        if p["scale"] != (1 << 64) - 1:
            assert lo <= data_base + p["scale"] and data_base + p["scale"] + 4 <= hi


def _plan(stmat, wl, workers, chunk=0, dst=None, kernel=0):
    from safetensors_materialization_gb300 import synth
    w = synth.WORKLOADS[wl]()
    lay = w.files[0]
    ix = stmat.Index.from_header(lay.header, lay.data_bytes)
    if w.rename:
        ix = ix.view_rename(w.rename)
    if w.prefix:
        ix = ix.view_prefix(w.prefix)
    return ix.plan(dst=dst or w.dst[0], scale_suffix=w.scale_suffix, workers=workers, chunk_bytes=chunk,
                   host_only=True, kernel=kernel), lay


@pytest.mark.parametrize("wl,workers,chunk", [("tiny", 664, 0), ("stress", 9728, 0), ("stress", 777, 1 << 26)])
@pytest.mark.parametrize("residue", [0, 1, 7, 8, 15])
def test_workload_accesses_stay_in_bounds(stmat, wl, workers, chunk, residue):
    for kernel in (0, 3):   # class-major and source unit order
        plan, lay = _plan(stmat, wl, workers, chunk, kernel=kernel)
        base = (1 << 32) + residue + (lay.data_start if residue == 7 else 0)
        for dst_align in (256, 2):
            check_plan(plan, base, dst_align, lay.data_bytes)


@pytest.mark.parametrize("residue", [0, 3, 8, 13])
def test_special_value_files_in_bounds(stmat, residue):
    """Files like the GPU edge tests build: every class, tiny to multi-chunk
    tensors, at the start and the end of the data section."""
    import json
    import struct
    ents, off = {}, 0
    rng = np.random.Generator(np.random.PCG64(residue))
    dts = ["F32", "F16", "BF16", "F8_E4M3", "F8_E5M2", "I64", "BOOL", "U8"]
    isz = {"F32": 4, "F16": 2, "BF16": 2, "F8_E4M3": 1, "F8_E5M2": 1, "I64": 8, "BOOL": 1, "U8": 1}
    for i in range(120):
        dt = dts[i % len(dts)]
        n = int(rng.choice([1, 2, 3, 5, 15, 16, 17, 31, 33, 255, 257, 4097, 70001]))
        ents[f"t{i:03d}"] = {"dtype": dt, "shape": [n], "data_offsets": [off, off + n * isz[dt]]}
        off += n * isz[dt]
    h = json.dumps(ents).encode()
    ix = stmat.Index.from_header(struct.pack("<Q", len(h)) + h, off)
    for dst in ("BF16", "F16", "F32", "KEEP"):
        for workers, kernel in ((1, 0), (3, 3), (64, 0), (64, 3)):
            plan = ix.plan(dst=dst, workers=workers, host_only=True, kernel=kernel)
            for dst_align in (256, 2, 1):
                check_plan(plan, (1 << 32) + residue, dst_align, off)


@pytest.mark.parametrize("residue", [0, 5, 8])
def test_sliced_plans_in_bounds(stmat, residue):
    """Slices on every dimension (multi-run pieces with a source pitch)."""
    import json
    import struct
    rng = np.random.Generator(np.random.PCG64(10 + residue))
    shapes = [[64, 300], [9, 40, 33], [3, 5, 7, 11], [4096, 96], [2, 70000]]
    dts = ["F32", "F16", "F8_E4M3", "BF16", "I64"]
    isz = {"F32": 4, "F16": 2, "BF16": 2, "F8_E4M3": 1, "I64": 8}
    ents, off = {}, 0
    for i, (shp, dt) in enumerate(zip(shapes, dts)):
        n = int(np.prod(shp))
        ents[f"s{i}"] = {"dtype": dt, "shape": shp, "data_offsets": [off, off + n * isz[dt]]}
        off += n * isz[dt]
    h = json.dumps(ents).encode()
    ix = stmat.Index.from_header(struct.pack("<Q", len(h)) + h, off)
    names = [f"s{i}" for i in range(len(shapes))]
    for trial in range(6):
        slices = []
        for shp in shapes:
            d = int(rng.integers(0, len(shp)))
            a = int(rng.integers(0, shp[d]))
            b = int(rng.integers(a, shp[d] + 1))
            slices.append((d, a, b))
        for dst in ("BF16", "F32", "KEEP"):
            for workers in (1, 5, 128):
                plan = ix.plan(dst=dst, names=names, slices=slices, workers=workers, host_only=True,
                               unit_bytes=[4096, 32768][trial % 2], kernel=[0, 3][trial % 2])
                for dst_align in (256, 2):
                    check_plan(plan, (1 << 32) + residue, dst_align, off)


def test_tma_windows_on_tiny_data_sections():
    """Data sections of 1..80 bytes at every residue mod 16, cut into two or
    three tensors of every class: the TMA build's windows stay inside the
    16-byte aligned interior (or are skipped) and the byte loads inside the
    section."""
    for nbytes in range(1, 81):
        for residue in range(16):
            lo = (1 << 32) + residue
            hi = lo + nbytes
            for cls, (si, so) in CLS.items():
                n = nbytes // si
                for cut in sorted({0, n // 3, n // 2, n}):
                    for a, b in ((0, cut), (cut, n)):
                        if b > a:
                            segs = tma_run(lo + a * si, (1 << 40) + 256 + a * so, b - a, si, so, lo, hi)
                            assert segs[-1][1] == b - a


@pytest.mark.parametrize("lead", [0, 1, 3, 8])
def test_blockscaled_plans_in_bounds(stmat, lead):
    """Block FP8 and NVFP4 weights (ragged rows, blocks of 16..512 columns,
    unaligned weight and scale offsets): every TMA window, scale window and
    slot read of the block-scaled consumer stays in bounds."""
    import test_blockscale as TB
    for fp8 in (("F8_E4M3", 257, 300, (128, 128)), ("F8_E5M2", 64, 48, (16, 16)), ("F8_E4M3", 3, 2000, (1, 16)),
                ("F8_E4M3", 130, 1030, (64, 512))):
        img, quant = TB.quant_file(lead, lead=lead, fp8=fp8, nv=(7, 2064))
        ix = stmat.Index.from_file(img)
        names, q = TB.selection(ix, quant)
        hlen, dbytes = ix.sizes()
        ents = {e["name"]: e for e in ix.entries()}
        for workers, dst, odd in ((1, "BF16", False), (7, "BF16", True), (64, "BF16", False), (7, "F32", True),
                                  (64, "F32", False)):
            plan = ix.plan(dst=dst, names=names, quant=q, workers=workers, host_only=True)
            outs = plan.outputs()
            qinfo = {}
            for i, o in enumerate(outs):
                if not o["quant"]:
                    continue
                sc = ents[o["scale"]]
                nv = o["quant"] == "nvfp4"
                br, bc = (1, 16) if nv else quant[o["name"]][3]
                qinfo[i] = {"scale": sc["begin"], "row_units": o["shape"][1] // (2 if nv else 1),
                            "scols": sc["shape"][1], "br_shift": br.bit_length() - 1, "bc_shift": bc.bit_length() - 1}
            st = plan.stats()
            pieces = [plan.piece(k) for k in range(st["pieces"])]
            for residue in (0, 5, 11):
                base = (1 << 32) + residue
                bases, at = [], 1 << 20
                for o in outs:
                    # odd: itemsize-aligned only (an F32 output of NVFP4 at 4 mod 8)
                    at = (at + 255) // 256 * 256 + ({"BF16": 2, "F32": 4}[dst] if odd else 0)
                    bases.append(at)
                    at += o["bytes"]
                for w in range(st["workers"] + 1):
                    a, b = plan.worker(0, w)
                    tma_warp(plan, pieces[a:b], bases, base, base, base + dbytes, quant=qinfo)
