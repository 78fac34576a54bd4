"""Thin Python binding of libstmat (ctypes): the C ABI's names, with
arguments marshalled from Python objects and torch tensors, and
StreamStateDict, the lazy mapping on top of st_load_tensors (keys from the
headers, sd[name], slices and batches on access).

Every step of the path (header parse, views, planning, staging copies and
the materialize kernel) runs inside libstmat; PyTorch only provides device
memory and streams.  There is no fallback: if libstmat.so is missing or a
call fails, a StmatError is raised.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libstmat.so")

DTYPES = ["BOOL", "U8", "I8", "I16", "U16", "I32", "U32", "I64", "U64", "F16", "BF16", "F32", "F64",
          "F8_E4M3", "F8_E5M2", "KEEP"]
STATUS = ["ST_OK", "ST_E_INVAL", "ST_E_TRUNCATED", "ST_E_HEADER_JSON", "ST_E_HEADER_TOO_LARGE",
          "ST_E_DUP_KEY", "ST_E_DTYPE", "ST_E_SHAPE", "ST_E_OFFSETS", "ST_E_NOT_FOUND",
          "ST_E_UNSUPPORTED_CAST", "ST_E_ALIGN", "ST_E_NOMEM", "ST_E_CUDA", "ST_E_DEVICE", "ST_E_IO"]

# Every symbol the C ABI exports (include/stmat.h).
EXPORTS = [
    "st_header_size", "st_index_build", "st_index_build_file", "st_index_free", "st_index_count",
    "st_index_get", "st_index_find", "st_index_sizes", "st_index_numel", "st_index_metadata_count",
    "st_index_metadata_get", "st_view_prefix", "st_view_filter", "st_view_rename", "st_index_concat",
    "st_plan",
    "st_plan_free", "st_plan_count", "st_plan_output", "st_plan_arena", "st_plan_stats",
    "st_plan_piece", "st_plan_worker", "st_plan_copy_bytes", "st_plan_copy_range", "st_class_step", "st_materialize", "st_stage_h2d", "st_load", "st_plan_check",
    "st_materialize_noalloc", "st_static_check", "st_index_open", "st_files_open", "st_files_close", "st_files_read",
    "st_load_files", "st_cache_create", "st_cache_free", "st_cache_get", "st_cache_release",
    "st_cache_stats", "st_cache_clear", "st_load_tensors", "st_host_affinity", "st_device_reads_pageable",
    "st_files_prefetch",
    "st_last_error", "st_status_name", "st_dtype_size", "st_dtype_name", "st_version",
]


class StmatError(RuntimeError):
    def __init__(self, code, msg=""):
        self.code = code
        self.status = STATUS[code] if 0 <= code < len(STATUS) else str(code)
        super().__init__(f"{self.status}: {msg}")


class TensorInfo(C.Structure):
    _fields_ = [("name", C.c_char_p), ("dtype", C.c_int), ("ndim", C.c_int32),
                ("shape", C.POINTER(C.c_int64)), ("numel", C.c_uint64), ("begin", C.c_uint64),
                ("end", C.c_uint64)]


class OutputInfo(C.Structure):
    _fields_ = [("name", C.c_char_p), ("dtype", C.c_int), ("src_dtype", C.c_int), ("ndim", C.c_int32),
                ("shape", C.POINTER(C.c_int64)), ("numel", C.c_uint64), ("bytes", C.c_uint64),
                ("src_begin", C.c_uint64), ("scale_name", C.c_char_p), ("slice_dim", C.c_int32),
                ("slice_start", C.c_int64), ("slice_stop", C.c_int64), ("quant_kind", C.c_int32)]


class Slice(C.Structure):
    _fields_ = [("dim", C.c_int32), ("start", C.c_int64), ("stop", C.c_int64)]


class CacheInfo(C.Structure):
    _fields_ = [("bytes", C.c_uint64), ("max_bytes", C.c_uint64), ("entries", C.c_uint64), ("hits", C.c_uint64),
                ("misses", C.c_uint64), ("evictions", C.c_uint64)]


class FilePart(C.Structure):
    _fields_ = [("path", C.c_char_p), ("offset", C.c_uint64), ("bytes", C.c_uint64), ("base", C.c_uint64)]


class BlockQuant(C.Structure):
    _fields_ = [("kind", C.c_int32), ("scale", C.c_char_p), ("scale2", C.c_char_p),
                ("block_rows", C.c_uint32), ("block_cols", C.c_uint32)]


QUANT_KINDS = {"block_fp8": 2, "nvfp4": 3}


class Selection(C.Structure):
    _fields_ = [("names", C.POINTER(C.c_char_p)), ("n_names", C.c_size_t),
                ("scale_names", C.POINTER(C.c_char_p)), ("scale_suffix_from", C.c_char_p),
                ("scale_suffix_to", C.c_char_p), ("part", C.c_uint32), ("n_parts", C.c_uint32),
                ("slices", C.POINTER(Slice)), ("quant", C.POINTER(BlockQuant))]


class PlanOptions(C.Structure):
    _fields_ = [("workers", C.c_uint32), ("chunk_bytes", C.c_uint64), ("host_only", C.c_int32),
                ("blocks_per_sm", C.c_uint32), ("unit_bytes", C.c_uint64), ("kernel", C.c_uint32),
                ("order", C.c_uint32)]


_lib = None


def lib():
    """The loaded libstmat (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise StmatError(1, f"{LIB_PATH} is missing; build it with "
                                "safetensors_materialization_gb300.build.build()")
        L = C.CDLL(LIB_PATH)
        P, U64, U32, S, I = C.c_void_p, C.c_uint64, C.c_uint32, C.c_size_t, C.c_int
        PP = C.POINTER(P)
        sig = {
            "st_header_size": [P, S, C.POINTER(U64)],
            "st_index_build": [P, S, U64, PP],
            "st_index_build_file": [P, U64, PP],
            "st_index_count": [P, C.POINTER(S)],
            "st_index_get": [P, S, C.POINTER(TensorInfo)],
            "st_index_find": [P, C.c_char_p, C.POINTER(S)],
            "st_index_sizes": [P, C.POINTER(U64), C.POINTER(U64)],
            "st_index_numel": [P, C.POINTER(U64), C.POINTER(U64)],
            "st_index_metadata_count": [P, C.POINTER(S)],
            "st_index_metadata_get": [P, S, C.POINTER(C.c_char_p), C.POINTER(C.c_char_p)],
            "st_view_prefix": [P, C.c_char_p, PP],
            "st_view_filter": [P, C.POINTER(C.c_char_p), S, PP],
            "st_view_rename": [P, C.POINTER(C.c_char_p), C.POINTER(C.c_char_p), S, PP],
            "st_index_concat": [C.POINTER(P), S, U64, C.POINTER(U64), PP],
            "st_plan": [P, C.POINTER(Selection), I, C.POINTER(PlanOptions), PP],
            "st_plan_count": [P, C.POINTER(S)],
            "st_plan_output": [P, S, C.POINTER(OutputInfo)],
            "st_plan_arena": [P, U64, C.POINTER(U64), C.POINTER(U64)],
            "st_plan_stats": [P, C.POINTER(U32), C.POINTER(U32), C.POINTER(U64), C.POINTER(U32)],
            "st_plan_piece": [P, U64, C.POINTER(U64), C.POINTER(U64), C.POINTER(U64), C.POINTER(U32),
                              C.POINTER(U32), C.POINTER(U32), C.POINTER(U32), C.POINTER(U64)],
            "st_plan_worker": [P, U32, U32, C.POINTER(U64), C.POINTER(U64)],
            "st_plan_copy_bytes": [P, C.POINTER(U64), C.POINTER(U32)],
            "st_plan_copy_range": [P, U32, C.POINTER(U64), C.POINTER(U64)],
            "st_class_step": [U32] + [C.POINTER(U32)] * 5,
            "st_materialize": [P, P, P, P, P],
            "st_materialize_noalloc": [P, P, P, P, P],
            "st_stage_h2d": [P, P, U64, U64, P, P],
            "st_load": [P, P, P, P, P, P, P],
            "st_plan_check": [P, P, C.POINTER(U32)],
            "st_static_check": [P, C.POINTER(U32)],
            "st_index_open": [C.c_char_p, PP, C.POINTER(U64)],
            "st_files_open": [C.POINTER(FilePart), S, PP],
            "st_files_read": [P, U64, U64, P, U32],
            "st_load_files": [P, P, P, P, P, P, U64, U32, P, P],
            "st_cache_create": [U64, C.c_int32, PP],
            "st_cache_get": [P, P, U64, U64, U32, PP],
            "st_cache_release": [P, P],
            "st_cache_stats": [P, C.POINTER(CacheInfo)],
            "st_cache_clear": [P],
            "st_load_tensors": [P, P, P, C.POINTER(Selection), I, P, P, U64, U32, P],
            "st_host_affinity": [I, C.c_int32, C.c_char_p, S],
            "st_device_reads_pageable": [I, C.POINTER(C.c_int32)],
            "st_files_prefetch": [P, U64, U64, U32],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = I
        for name in ("st_index_free", "st_plan_free", "st_files_close", "st_cache_free"):
            getattr(L, name).argtypes = [P]
            getattr(L, name).restype = None
        L.st_last_error.restype = C.c_char_p
        L.st_status_name.restype = C.c_char_p
        L.st_status_name.argtypes = [I]
        L.st_dtype_size.restype = S
        L.st_dtype_size.argtypes = [I]
        L.st_dtype_name.restype = C.c_char_p
        L.st_dtype_name.argtypes = [I]
        L.st_version.restype = U32
        _lib = L
    return _lib


def _check(code):
    if code != 0:
        raise StmatError(code, lib().st_last_error().decode(errors="replace"))


def _strs(names):
    arr = (C.c_char_p * max(1, len(names)))()
    for i, n in enumerate(names):
        arr[i] = None if n is None else n.encode()
    return arr


def _addr(obj):
    """Address of a numpy array, bytes object or torch tensor."""
    if obj is None:
        return None
    if isinstance(obj, int):
        return obj
    if hasattr(obj, "data_ptr"):
        return obj.data_ptr()
    if isinstance(obj, np.ndarray):
        return obj.ctypes.data
    raise TypeError(f"cannot take the address of {type(obj)}")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return s if isinstance(s, int) else s.cuda_stream


def header_size(first8: bytes) -> int:
    n = C.c_uint64()
    _check(lib().st_header_size(first8, len(first8), C.byref(n)))
    return n.value


def _selection(names=None, scale_names=None, scale_suffix=None, part=0, n_parts=0, slices=None, quant=None):
    """An st_selection and the ctypes objects it points into (keep them alive)."""
    sel = Selection()
    keep = []
    if names is not None:
        arr = _strs(names)
        keep.append(arr)
        sel.names, sel.n_names = C.cast(arr, C.POINTER(C.c_char_p)), len(names)
    if scale_names is not None:
        arr = _strs(scale_names)
        keep.append(arr)
        sel.scale_names = C.cast(arr, C.POINTER(C.c_char_p))
    if scale_suffix:
        sel.scale_suffix_from, sel.scale_suffix_to = scale_suffix[0].encode(), scale_suffix[1].encode()
    sel.part, sel.n_parts = part, n_parts
    if slices is not None:
        arr = (Slice * max(1, len(slices)))()
        for i, x in enumerate(slices):
            arr[i] = Slice(*(x if x is not None else (-1, 0, 0)))
        keep.append(arr)
        sel.slices = C.cast(arr, C.POINTER(Slice))
    if quant is not None:
        arr = (BlockQuant * max(1, len(quant)))()
        for i, q in enumerate(quant):
            if q:
                br, bc = q[3] if len(q) > 3 and q[3] else (0, 0)
                arr[i] = BlockQuant(QUANT_KINDS.get(q[0], 99), q[1].encode() if q[1] else None,
                                    q[2].encode() if q[2] else None, br, bc)
        keep.append(arr)
        sel.quant = C.cast(arr, C.POINTER(BlockQuant))
    return sel, keep


class Index:
    """A parsed header or a view (st_index_t)."""

    def __init__(self, handle, keep=None):
        self._h = C.c_void_p(handle)
        self._keep = keep

    @classmethod
    def from_file(cls, image):
        """Index of a whole file image (bytes or uint8 numpy array)."""
        arr = np.frombuffer(image, dtype=np.uint8) if isinstance(image, (bytes, bytearray)) else image
        out = C.c_void_p()
        _check(lib().st_index_build_file(_addr(arr), arr.size, C.byref(out)))
        return cls(out.value)

    @classmethod
    def from_header(cls, header, data_bytes):
        """Index from the first 8 + N bytes and the data section size."""
        arr = np.frombuffer(header, dtype=np.uint8) if isinstance(header, (bytes, bytearray)) else header
        out = C.c_void_p()
        _check(lib().st_index_build(_addr(arr), arr.size, data_bytes, C.byref(out)))
        return cls(out.value)

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value and _lib is not None:
            _lib.st_index_free(self._h)
            self._h = C.c_void_p(None)

    @property
    def handle(self):
        return self._h

    def __len__(self):
        n = C.c_size_t()
        _check(lib().st_index_count(self._h, C.byref(n)))
        return n.value

    def entry(self, i):
        info = TensorInfo()
        _check(lib().st_index_get(self._h, i, C.byref(info)))
        return {"name": info.name.decode(), "dtype": DTYPES[info.dtype],
                "shape": [info.shape[d] for d in range(info.ndim)], "numel": info.numel,
                "begin": info.begin, "end": info.end}

    def entries(self):
        return [self.entry(i) for i in range(len(self))]

    def find(self, name):
        i = C.c_size_t()
        _check(lib().st_index_find(self._h, name.encode(), C.byref(i)))
        return i.value

    def sizes(self):
        h, d = C.c_uint64(), C.c_uint64()
        _check(lib().st_index_sizes(self._h, C.byref(h), C.byref(d)))
        return h.value, d.value

    def numel(self):
        total = C.c_uint64()
        counts = (C.c_uint64 * 15)()
        _check(lib().st_index_numel(self._h, C.byref(total), counts))
        return total.value, {DTYPES[d]: counts[d] for d in range(15) if counts[d]}

    def metadata(self):
        n = C.c_size_t()
        _check(lib().st_index_metadata_count(self._h, C.byref(n)))
        out = {}
        for i in range(n.value):
            k, v = C.c_char_p(), C.c_char_p()
            _check(lib().st_index_metadata_get(self._h, i, C.byref(k), C.byref(v)))
            out[k.value.decode()] = v.value.decode()
        return out

    def view_prefix(self, prefix):
        out = C.c_void_p()
        _check(lib().st_view_prefix(self._h, prefix.encode(), C.byref(out)))
        return Index(out.value)

    def view_filter(self, names):
        out = C.c_void_p()
        _check(lib().st_view_filter(self._h, _strs(names), len(names), C.byref(out)))
        return Index(out.value)

    def view_rename(self, rules):
        out = C.c_void_p()
        _check(lib().st_view_rename(self._h, _strs([a for a, _ in rules]), _strs([b for _, b in rules]),
                                    len(rules), C.byref(out)))
        return Index(out.value)

    @classmethod
    def open(cls, path):
        """st_index_open: the index of a file on disk (reads its header only);
        returns (index, data-section offset in the file)."""
        out, off = C.c_void_p(), C.c_uint64()
        _check(lib().st_index_open(os.fsencode(path), C.byref(out), C.byref(off)))
        return cls(out.value), off.value

    @classmethod
    def concat(cls, parts, align=256):
        """st_index_concat: one index over shard indexes; returns (index, bases),
        shard k's data section belonging at arena offset bases[k]."""
        n = len(parts)
        hs = (C.c_void_p * max(1, n))(*[p.handle.value for p in parts])
        bases = (C.c_uint64 * max(1, n))()
        out = C.c_void_p()
        _check(lib().st_index_concat(hs, n, align, bases, C.byref(out)))
        return cls(out.value), [int(b) for b in bases[:n]]

    def load_tensors(self, files, dst_ptrs, staging, names, dst="BF16", cache=None, threads=16, stream=None,
                     scale_names=None, scale_suffix=None, quant=None, slices=None):
        """st_load_tensors: the lazy path for a few named tensors (read through
        `cache`, staged in `staging`, one launch on `stream`); dst_ptrs: one
        device address per output, in output order; slices as for plan().
        Its tables go into the library's static device array, shared with
        every other lazy load and st_materialize_noalloc call: keep them on
        one stream.  Device flags: static_check()."""
        sel, keep = _selection(names, scale_names, scale_suffix, 0, 0, slices, quant)
        ptrs = (C.c_void_p * max(1, len(dst_ptrs)))(*dst_ptrs)
        nbytes = staging.numel() if hasattr(staging, "numel") else len(staging)
        _check(lib().st_load_tensors(self._h, files.handle, cache.handle if cache else None, C.byref(sel),
                                     DTYPES.index(dst), ptrs, _addr(staging), nbytes, threads, _stream(stream)))

    def plan(self, dst="BF16", names=None, scale_names=None, scale_suffix=None, part=0, n_parts=0,
             workers=0, chunk_bytes=0, host_only=False, blocks_per_sm=0, unit_bytes=0, kernel=0, order=0,
             slices=None, quant=None):
        """st_plan: outputs and device work for a selection.  quant: per name
        None or (kind, block-scales name, global-scale name or None,
        (block rows, block cols) or None), kind "block_fp8" or "nvfp4"."""
        sel, keep = _selection(names, scale_names, scale_suffix, part, n_parts, slices, quant)
        opts = PlanOptions(workers, chunk_bytes, 1 if host_only else 0, blocks_per_sm, unit_bytes, kernel, order)
        out = C.c_void_p()
        _check(lib().st_plan(self._h, C.byref(sel), DTYPES.index(dst), C.byref(opts), C.byref(out)))
        return Plan(out.value, self)


class Files:
    """st_files_t: shard files addressed as one arena.  parts: (path, file
    offset of the data section, bytes, arena base) per file."""

    def __init__(self, parts):
        self._paths = [os.fsencode(p[0]) for p in parts]
        arr = (FilePart * max(1, len(parts)))()
        for i, (path, off, n, base) in enumerate(parts):
            arr[i] = FilePart(self._paths[i], off, n, base)
        out = C.c_void_p()
        _check(lib().st_files_open(arr, len(parts), C.byref(out)))
        self._h = C.c_void_p(out.value)
        self.arena_bytes = max((base + n for _, _, n, base in parts), default=0)

    @classmethod
    def of_checkpoint(cls, paths, align=256):
        """Opens the shard files of one checkpoint: returns (Files, joined
        Index) with each shard's data section at its st_index_concat base."""
        opened = [Index.open(p) for p in paths]
        ix, bases = Index.concat([o[0] for o in opened], align)
        parts = [(p, off, o.sizes()[1], b) for p, (o, off), b in zip(paths, opened, bases)]
        return cls(parts), ix

    def close(self):
        """st_files_close (also on garbage collection)."""
        if getattr(self, "_h", None) and self._h.value and _lib is not None:
            _lib.st_files_close(self._h)
            self._h = C.c_void_p(None)

    def __del__(self):
        self.close()

    @property
    def handle(self):
        if not self._h.value:
            raise StmatError(1, "the files are closed")
        return self._h

    def prefetch(self, begin=0, nbytes=None, threads=4):
        """st_files_prefetch: fault arena bytes into the mappings' page tables
        (reads uncached pages from disk); default the whole arena."""
        if nbytes is None:
            nbytes = self.arena_bytes - begin
        _check(lib().st_files_prefetch(self.handle, begin, nbytes, threads))

    def read(self, begin, nbytes, host, threads=4):
        """st_files_read into `host` (a numpy uint8 array or torch tensor)."""
        _check(lib().st_files_read(self.handle, begin, nbytes, _addr(host), threads))


class Cache:
    """st_cache_t: the LRU RAM tier (host copies of file ranges, at most
    `max_bytes`; pinned memory unless pinned=False)."""

    def __init__(self, max_bytes, pinned=True):
        out = C.c_void_p()
        _check(lib().st_cache_create(max_bytes, 1 if pinned else 0, C.byref(out)))
        self._h = C.c_void_p(out.value)

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value and _lib is not None:
            _lib.st_cache_free(self._h)
            self._h = C.c_void_p(None)

    @property
    def handle(self):
        return self._h

    def get(self, files, begin, nbytes, threads=4):
        """Holds the host copy of arena bytes [begin, begin + nbytes); returns
        its address (release it with release())."""
        out = C.c_void_p()
        _check(lib().st_cache_get(self._h, files.handle, begin, nbytes, threads, C.byref(out)))
        return out.value

    def release(self, addr):
        _check(lib().st_cache_release(self._h, addr))

    def stats(self):
        info = CacheInfo()
        _check(lib().st_cache_stats(self._h, C.byref(info)))
        return {k: getattr(info, k) for k, _ in CacheInfo._fields_}

    def clear(self):
        _check(lib().st_cache_clear(self._h))


class StreamStateDict:
    """A read-only mapping name -> tensor over a checkpoint's shard files, in
    the manner of the streaming mapping of "Disk tier safetensors streaming
    design audit (ComfyUI)": keys, shapes, dtypes and metadata come from the
    headers alone; sd[name] reads that tensor (and its scales) through the
    RAM tier and materializes it on the GPU with st_load_tensors; meta(name)
    is a device='meta' stand-in (the disk reference stays in the index).

    paths: shard files; dst: output float dtype; rename/prefix: views;
    scale_suffix / quant: as for Index.plan (quant: name -> (kind, scales,
    global scale, block)).

    Every load runs on torch's current stream and takes its kernel's tables
    from the library's one static device array, which st_materialize_noalloc
    uses too: keep every lazy load and allocation-free call of a process on
    one stream, or they race on that array.  check() reads the device flags
    the loads left there."""

    def __init__(self, paths, dst="BF16", device="cuda", ram_cache_bytes=1 << 30, pinned=True, threads=16,
                 rename=None, prefix=None, scale_suffix=None, quant=None, align=256):
        self.files, root = Files.of_checkpoint(list(paths), align)
        view = root
        if rename:
            view = view.view_rename(rename)
        if prefix:
            view = view.view_prefix(prefix)
        self.index, self._root = view, root
        self.dst, self.device, self.threads = dst, device, threads
        self.scale_suffix, self.quant = scale_suffix, dict(quant or {})
        self.cache = Cache(ram_cache_bytes, pinned) if ram_cache_bytes else None
        self._staging = None
        self._names = [e["name"] for e in view.entries()]
        self._pos = {n: i for i, n in enumerate(self._names)}
        self._info = {}  # name -> (shape, dtype, staging bytes), filled on first use

    def keys(self):
        return list(self._names)

    def check(self):
        """Device flags of the loads so far (st_static_check on torch's
        current stream, which it waits for); 0 when every load completed."""
        import torch
        return static_check(torch.cuda.current_stream())

    def __iter__(self):
        return iter(self._names)

    def __len__(self):
        return len(self._names)

    def __contains__(self, name):
        return name in self._pos

    def metadata(self):
        return self.index.metadata()

    def _lookup(self, name):
        got = self._info.get(name)
        if got is None:
            o = self._plan(name, host_only=True).outputs()[0]
            e = self.index.entry(self._pos[name])
            got = (o["shape"], o["dtype"], int((e["end"] - e["begin"]) * 1.25) + (1 << 16))
            self._info[name] = got
        return got

    def info(self, name):
        """Shape and dtype of sd[name] (header only)."""
        shape, dt, _ = self._lookup(name)
        return shape, dt

    def meta(self, name):
        import torch
        shape, dt = self.info(name)
        return torch.empty(shape, dtype=torch_dtype(dt), device="meta")

    def _sel(self, name):
        q = self.quant.get(name)
        return dict(names=[name], scale_suffix=self.scale_suffix, quant=[q] if q else None)

    def _plan(self, name, host_only):
        return self.index.plan(dst=self.dst, workers=1, host_only=host_only, **self._sel(name))

    def __getitem__(self, name):
        import torch
        if name not in self._pos:
            raise KeyError(name)
        shape, dt, need = self._lookup(name)
        out = torch.empty(shape, dtype=torch_dtype(dt), device=self.device)
        if self._staging is None or self._staging.numel() < need:
            self._staging = torch.empty(need, dtype=torch.uint8, device=self.device)
        self.index.load_tensors(self.files, [out.data_ptr()], self._staging, dst=self.dst, cache=self.cache,
                                threads=self.threads, stream=torch.cuda.current_stream(), **self._sel(name))
        return out

    def slice(self, name, dim, start, stop):
        """sd[name][..., start:stop, ...] along `dim`, read and cast on access
        (a tensor-parallel rank's rows or columns): one st_load_tensors with a
        slice, the gather done by the kernel."""
        import torch
        if name not in self._pos:
            raise KeyError(name)
        q = self.quant.get(name)
        kw = dict(names=[name], scale_suffix=self.scale_suffix, quant=[q] if q else None,
                  slices=[(dim, start, stop)])
        o = self.index.plan(dst=self.dst, workers=1, host_only=True, **kw).outputs()[0]
        out = torch.empty(o["shape"], dtype=torch_dtype(o["dtype"]), device=self.device)
        need = self._lookup(name)[2]
        if self._staging is None or self._staging.numel() < need:
            self._staging = torch.empty(need, dtype=torch.uint8, device=self.device)
        self.index.load_tensors(self.files, [out.data_ptr()], self._staging, dst=self.dst, cache=self.cache,
                                threads=self.threads, stream=torch.cuda.current_stream(), **kw)
        return out

    def load_many(self, names, max_batch_bytes=256 << 20, max_batch=1024, alone_bytes=32 << 20):
        """Several tensors at once: one st_load_tensors (one staging copy, one
        launch) per batch of at most max_batch tensors or max_batch_bytes of
        staged bytes; a tensor of alone_bytes or more is loaded on its own
        (large tensors already fill the host link one at a time, and batching
        them only loses the overlap).  Returns {name: tensor}."""
        import torch
        out, batch, staged = {}, [], 0

        def flush():
            if not batch:
                return
            quant = [self.quant.get(n) for n in batch]
            kw = dict(names=list(batch), scale_suffix=self.scale_suffix, quant=quant if any(quant) else None)
            # A name that another name of the batch consumes (its scale) is no
            # output of the batch: then the destinations would not line up.
            got = [o["name"] for o in self.index.plan(dst=self.dst, workers=1, host_only=True, **kw).outputs()]
            if got != batch:
                for n in batch:
                    out[n] = self[n]
                return
            need = sum(self._lookup(n)[2] for n in batch)
            if self._staging is None or self._staging.numel() < need:
                self._staging = torch.empty(need, dtype=torch.uint8, device=self.device)
            ts = [torch.empty(self._lookup(n)[0], dtype=torch_dtype(self._lookup(n)[1]), device=self.device)
                  for n in batch]
            self.index.load_tensors(self.files, [t.data_ptr() for t in ts], self._staging, dst=self.dst,
                                    cache=self.cache, threads=self.threads, stream=torch.cuda.current_stream(), **kw)
            out.update(zip(batch, ts))

        for n in names:
            if n not in self._pos:
                raise KeyError(n)
            need = self._lookup(n)[2]
            if need >= alone_bytes:
                out[n] = self[n]
                continue
            if batch and (len(batch) >= max_batch or staged + need > max_batch_bytes):
                flush()
                batch, staged = [], 0
            batch.append(n)
            staged += need
        flush()
        return {n: out[n] for n in names}

    def items(self, batch=64):
        """(name, tensor) in key order, loaded `batch` names at a time with
        load_many (one staging pass and one launch per batch)."""
        for k in range(0, len(self._names), max(1, batch)):
            yield from self.load_many(self._names[k:k + max(1, batch)]).items()


class Plan:
    """st_plan_t: the outputs of a selection and their device work."""

    def __init__(self, handle, index):
        self._h = C.c_void_p(handle)
        self.index = index

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value and _lib is not None:
            _lib.st_plan_free(self._h)
            self._h = C.c_void_p(None)

    @property
    def handle(self):
        return self._h

    def __len__(self):
        n = C.c_size_t()
        _check(lib().st_plan_count(self._h, C.byref(n)))
        return n.value

    def output(self, i):
        o = OutputInfo()
        _check(lib().st_plan_output(self._h, i, C.byref(o)))
        return {"name": o.name.decode(), "dtype": DTYPES[o.dtype], "src_dtype": DTYPES[o.src_dtype],
                "shape": [o.shape[d] for d in range(o.ndim)], "numel": o.numel, "bytes": o.bytes,
                "begin": o.src_begin, "scale": o.scale_name.decode() if o.scale_name else None,
                "slice": None if o.slice_dim < 0 else (o.slice_dim, o.slice_start, o.slice_stop),
                "quant": {2: "block_fp8", 3: "nvfp4"}.get(o.quant_kind)}

    def outputs(self):
        return [self.output(i) for i in range(len(self))]

    def arena(self, align=256):
        n = len(self)
        offs = (C.c_uint64 * max(1, n))()
        total = C.c_uint64()
        _check(lib().st_plan_arena(self._h, align, offs, C.byref(total)))
        return [offs[i] for i in range(n)], total.value

    def stats(self):
        w, c, p, k = C.c_uint32(), C.c_uint32(), C.c_uint64(), C.c_uint32()
        _check(lib().st_plan_stats(self._h, C.byref(w), C.byref(c), C.byref(p), C.byref(k)))
        return {"workers": w.value, "chunks": c.value, "pieces": p.value,
                "kernel": {1: "stream", 2: "latency", 3: "tma", 4: "tma_wide"}.get(k.value, str(k.value))}

    def piece(self, k):
        v = [C.c_uint64(), C.c_uint64(), C.c_uint64(), C.c_uint32(), C.c_uint32(), C.c_uint32(), C.c_uint32(),
             C.c_uint64()]
        _check(lib().st_plan_piece(self._h, k, *[C.byref(x) for x in v]))
        return dict(zip(["src", "dst", "scale", "count", "output", "cls", "rows", "pitch"], [x.value for x in v]))

    def worker(self, chunk, w):
        a, b = C.c_uint64(), C.c_uint64()
        _check(lib().st_plan_worker(self._h, chunk, w, C.byref(a), C.byref(b)))
        return a.value, b.value

    # ------------------------------------------------------------- device
    def materialize(self, data, dst_ptrs, scales=None, stream=None):
        """st_materialize.  data: device uint8 tensor (or address) of the data
        section; dst_ptrs: device int64 tensor of output addresses."""
        _check(lib().st_materialize(_addr(data), self._h, _addr(dst_ptrs), _addr(scales), _stream(stream)))

    def materialize_noalloc(self, data, dst_ptrs, scales=None, stream=None):
        """st_materialize_noalloc: as materialize(), with the plan's tables in
        the library's static device scratch instead of allocated memory (plan
        with host_only=True).  The scratch is one array shared by every such
        call and every lazy load: keep them all on one stream.  Device flags
        are read with static_check()."""
        _check(lib().st_materialize_noalloc(_addr(data), self._h, _addr(dst_ptrs), _addr(scales),
                                            _stream(stream)))

    def load(self, data_host, data_dev, dst_ptrs, scales=None, copy_stream=None, compute_stream=None):
        """st_load: staged copy of the data section overlapped with materialize."""
        _check(lib().st_load(_addr(data_host), _addr(data_dev), self._h, _addr(dst_ptrs), _addr(scales),
                             _stream(copy_stream), _stream(compute_stream)))

    def load_files(self, files, data_dev, dst_ptrs, ring_host=None, ring_bytes=None, threads=8, scales=None,
                   copy_stream=None, compute_stream=None):
        """st_load_files: disk -> pinned ring -> device, each chunk materialized
        as soon as it lands; with ring_host None, each chunk is copied straight
        from the files' mappings (the fast path where reads_pageable() holds)."""
        if ring_bytes is None and ring_host is None:
            ring_bytes = 0
        elif ring_bytes is None:
            ring_bytes = ring_host.numel() if hasattr(ring_host, "numel") else len(ring_host)
        _check(lib().st_load_files(files.handle, _addr(data_dev), self._h, _addr(dst_ptrs), _addr(scales),
                                   _addr(ring_host), ring_bytes, threads, _stream(copy_stream),
                                   _stream(compute_stream)))

    def copy_bytes(self):
        """st_plan_copy_bytes: (bytes the loaders copy for this plan, ranges)."""
        b, r = C.c_uint64(), C.c_uint32()
        _check(lib().st_plan_copy_bytes(self._h, C.byref(b), C.byref(r)))
        return b.value, r.value

    def copy_ranges(self):
        """st_plan_copy_range for every range: [(begin, end)] of the data
        section that the loaders copy."""
        out = []
        for i in range(self.copy_bytes()[1]):
            a, b = C.c_uint64(), C.c_uint64()
            _check(lib().st_plan_copy_range(self._h, i, C.byref(a), C.byref(b)))
            out.append((a.value, b.value))
        return out

    def check(self, stream=None):
        flags = C.c_uint32()
        code = lib().st_plan_check(self._h, _stream(stream), C.byref(flags))
        if code not in (0, 14):
            _check(code)
        return flags.value


def class_step(cls):
    """st_class_step: (source itemsize, output itemsize, lane-step source
    bytes, counted units, output bytes) of conversion class `cls`."""
    v = [C.c_uint32() for _ in range(5)]
    _check(lib().st_class_step(cls, *[C.byref(x) for x in v]))
    return tuple(x.value for x in v)


def static_check(stream=None):
    """st_static_check: reads and clears the device flags that
    st_materialize_noalloc and st_load_tensors calls left in the library's
    static array on the current device (waits for `stream` first); 0 when
    none (bit 0: bad destination, bit 1: a wait for a staged copy gave up)."""
    flags = C.c_uint32()
    code = lib().st_static_check(_stream(stream), C.byref(flags))
    if code not in (0, 14):
        _check(code)
    return flags.value


def host_affinity(device=0, apply=True):
    """st_host_affinity: the GPU's local CPU list; with apply, binds the
    calling thread to it (do this before allocating pinned memory)."""
    buf = C.create_string_buffer(4096)
    _check(lib().st_host_affinity(device, 1 if apply else 0, buf, len(buf)))
    return buf.value.decode()


def reads_pageable(device=0):
    """st_device_reads_pageable: whether the GPU reads pageable host memory
    through the host's page tables (ring-less file loads are then copy-engine
    reads of the page cache)."""
    yes = C.c_int32()
    _check(lib().st_device_reads_pageable(device, C.byref(yes)))
    return bool(yes.value)


def stage_h2d(dst_dev, src_host, nbytes, chunk_bytes=0, stream=None, done_event=None):
    """st_stage_h2d: chunked host->device copies on `stream`."""
    ev = None if done_event is None else done_event.cuda_event
    _check(lib().st_stage_h2d(_addr(dst_dev), _addr(src_host), nbytes, chunk_bytes, _stream(stream), ev))


# ----------------------------------------------------------- torch helpers

def torch_dtype(name):
    import torch
    return {"BOOL": torch.bool, "U8": torch.uint8, "I8": torch.int8, "I16": torch.int16,
            "U16": torch.uint16, "I32": torch.int32, "U32": torch.uint32, "I64": torch.int64,
            "U64": torch.uint64, "F16": torch.float16, "BF16": torch.bfloat16, "F32": torch.float32,
            "F64": torch.float64, "F8_E4M3": torch.float8_e4m3fn, "F8_E5M2": torch.float8_e5m2}[name]


class Outputs:
    """Destination buffers for a plan: one device arena carved into the
    outputs (each 256-byte aligned) and the device array of their addresses."""

    def __init__(self, plan: Plan, device="cuda", align=256):
        import torch
        self.plan = plan
        self.infos = plan.outputs()
        offs, total = plan.arena(align)
        self.offsets = offs
        self.arena = torch.empty(max(total, 1), dtype=torch.uint8, device=device)
        base = self.arena.data_ptr()
        self.ptrs = torch.tensor([base + o for o in offs] or [0], dtype=torch.int64, device=device)

    def raw(self, i):
        """Output i as uint8 bytes (a view into the arena)."""
        return self.arena[self.offsets[i]:self.offsets[i] + self.infos[i]["bytes"]]

    def tensor(self, i):
        """Output i as a typed, shaped tensor (a view into the arena)."""
        info = self.infos[i]
        return self.raw(i).view(torch_dtype(info["dtype"])).view(info["shape"])

    def tensors(self):
        return {info["name"]: self.tensor(i) for i, info in enumerate(self.infos)}
