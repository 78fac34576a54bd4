"""ctypes wrapper around the plain C oracle (``stmat_oracle.c``).

Test infrastructure only: the tests, the smoke check and the benchmark's CPU
baseline use it; the product path never does.
"""
import ctypes as C

import numpy as np

from . import build as _build

DTYPES = ["BOOL", "U8", "I8", "I16", "U16", "I32", "U32", "I64", "U64",
          "F16", "BF16", "F32", "F64", "F8_E4M3", "F8_E5M2", "KEEP"]
ITEMSIZE = {"BOOL": 1, "U8": 1, "I8": 1, "I16": 2, "U16": 2, "I32": 4, "U32": 4, "I64": 8,
            "U64": 8, "F16": 2, "BF16": 2, "F32": 4, "F64": 8, "F8_E4M3": 1, "F8_E5M2": 1}
STATUS = ["OK", "INVAL", "TRUNCATED", "HEADER_JSON", "HEADER_TOO_LARGE", "DUP_KEY", "DTYPE",
          "SHAPE", "OFFSETS", "NOT_FOUND", "UNSUPPORTED_CAST", "ALIGN", "NOMEM"]


class OracleError(Exception):
    def __init__(self, code):
        self.code = code
        self.status = STATUS[code] if 0 <= code < len(STATUS) else str(code)
        super().__init__(f"oracle status {self.status}")


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = C.CDLL(_build.build())
        P, U64, I64, I = C.c_void_p, C.c_uint64, C.c_int64, C.c_int
        sig = {
            "or_parse": (I, [C.c_char_p, U64, C.POINTER(P)]),
            "or_parse_header": (I, [C.c_char_p, U64, U64, C.POINTER(P)]),
            "or_index_free": (None, [P]),
            "or_count": (U64, [P]), "or_header_len": (U64, [P]), "or_data_bytes": (U64, [P]),
            "or_name": (C.c_char_p, [P, U64]), "or_dtype": (I, [P, U64]), "or_ndim": (I, [P, U64]),
            "or_dim": (I64, [P, U64, I]), "or_numel": (U64, [P, U64]),
            "or_begin": (U64, [P, U64]), "or_end": (U64, [P, U64]),
            "or_meta_count": (U64, [P]), "or_meta_key": (C.c_char_p, [P, U64]),
            "or_meta_val": (C.c_char_p, [P, U64]), "or_find": (I64, [P, C.c_char_p]),
            "or_view_prefix": (I, [P, C.c_char_p, C.POINTER(P)]),
            "or_view_filter": (I, [P, C.POINTER(C.c_char_p), U64, C.POINTER(P)]),
            "or_view_rename": (I, [P, C.POINTER(C.c_char_p), C.POINTER(C.c_char_p), U64, C.POINTER(P)]),
            "or_concat": (I, [C.POINTER(P), U64, U64, C.POINTER(U64), C.POINTER(P)]),
            "or_out_dtype": (I, [I, I]),
            "or_convert": (I, [I, I, C.c_char_p, U64, I, C.c_float, P]),
            "or_select": (I, [P, C.POINTER(C.c_char_p), U64, C.POINTER(C.c_char_p), C.c_char_p,
                              C.c_char_p, I, U64, U64, C.POINTER(I64), C.POINTER(P)]),
            "or_select_q": (I, [P, C.POINTER(C.c_char_p), U64, C.POINTER(C.c_char_p), C.c_char_p,
                                C.c_char_p, I, U64, U64, C.POINTER(I64), C.POINTER(C.c_int),
                                C.POINTER(C.c_char_p), C.POINTER(C.c_char_p), C.POINTER(I64), C.POINTER(P)]),
            "or_plan_quant": (I, [P, U64]), "or_plan_qscale": (I64, [P, U64]),
            "or_plan_qscale2": (I64, [P, U64]),
            "or_plan_numel": (U64, [P, U64]), "or_plan_ndim": (I, [P, P, U64]),
            "or_plan_dim": (I64, [P, P, U64, I]),
            "or_plan_free": (None, [P]), "or_plan_count": (U64, [P]),
            "or_plan_name": (C.c_char_p, [P, U64]), "or_plan_entry": (U64, [P, U64]),
            "or_plan_dtype": (I, [P, U64]), "or_plan_scale": (I64, [P, U64]),
            "or_plan_bytes": (U64, [P, P, U64]),
            "or_materialize": (I, [P, P, U64, P, U64, P]),
            "or_materialize_range": (I, [P, P, U64, P, U64, U64, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(code):
    if code != 0:
        raise OracleError(code)


def _strs(names):
    arr = (C.c_char_p * max(1, len(names)))()
    for i, n in enumerate(names):
        arr[i] = n.encode() if n is not None else None
    return arr


def _ptr(buf):
    """Address of a numpy array / bytes-like object's first byte."""
    if isinstance(buf, np.ndarray):
        return buf.ctypes.data
    return C.cast(C.c_char_p(bytes(buf)), C.c_void_p).value


class OIndex:
    """Oracle index (or view): entries in index order."""

    def __init__(self, handle, keep=None):
        self._h = C.c_void_p(handle)
        self._keep = keep

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value:
            lib().or_index_free(self._h)
            self._h = C.c_void_p(None)

    @property
    def handle(self):
        return self._h

    def __len__(self):
        return lib().or_count(self._h)

    @property
    def header_len(self):
        return lib().or_header_len(self._h)

    @property
    def data_bytes(self):
        return lib().or_data_bytes(self._h)

    def entry(self, i):
        L = lib()
        return {
            "name": L.or_name(self._h, i).decode(),
            "dtype": DTYPES[L.or_dtype(self._h, i)],
            "shape": [L.or_dim(self._h, i, d) for d in range(L.or_ndim(self._h, i))],
            "numel": L.or_numel(self._h, i),
            "begin": L.or_begin(self._h, i),
            "end": L.or_end(self._h, i),
        }

    def entries(self):
        return [self.entry(i) for i in range(len(self))]

    def metadata(self):
        L = lib()
        return {L.or_meta_key(self._h, i).decode(): L.or_meta_val(self._h, i).decode()
                for i in range(L.or_meta_count(self._h))}

    def find(self, name):
        return lib().or_find(self._h, name.encode())

    def view_prefix(self, prefix):
        out = C.c_void_p()
        _check(lib().or_view_prefix(self._h, prefix.encode(), C.byref(out)))
        return OIndex(out.value, keep=self)

    def view_filter(self, names):
        out = C.c_void_p()
        _check(lib().or_view_filter(self._h, _strs(names), len(names), C.byref(out)))
        return OIndex(out.value, keep=self)

    def view_rename(self, pairs):
        out = C.c_void_p()
        fr = _strs([a for a, _ in pairs])
        to = _strs([b for _, b in pairs])
        _check(lib().or_view_rename(self._h, fr, to, len(pairs), C.byref(out)))
        return OIndex(out.value, keep=self)

    def select(self, names=None, dst="BF16", scale_names=None, scale_suffix=None,
               part=0, nparts=1, slices=None, quant=None):
        """slices: per name None or (dim, start, stop).  quant: per name None or
        (kind, scale name, global scale name or None, (block rows, block cols)),
        kind "block_fp8" or "nvfp4"."""
        out = C.c_void_p()
        nm = _strs(names) if names is not None else None
        sn = _strs(scale_names) if scale_names is not None else None
        fr, to = (scale_suffix if scale_suffix else (None, None))
        sl = None
        if slices is not None:
            flat = []
            for x in slices:
                flat += list(x) if x is not None else [-1, 0, 0]
            sl = (C.c_int64 * max(1, len(flat)))(*flat)
        qk = qs = qs2 = qb = None
        if quant is not None:
            kinds = {"block_fp8": 2, "nvfp4": 3}
            qk = (C.c_int * max(1, len(quant)))(*[kinds.get(q[0], 99) if q else 0 for q in quant])
            qs = _strs([q[1] if q else None for q in quant])
            qs2 = _strs([q[2] if q else None for q in quant])
            blocks = []
            for q in quant:
                blocks += list(q[3]) if q and len(q) > 3 and q[3] else [0, 0]
            qb = (C.c_int64 * max(1, len(blocks)))(*blocks)
        _check(lib().or_select_q(self._h, nm, len(names) if names is not None else 0, sn,
                                 fr.encode() if fr else None, to.encode() if to else None,
                                 DTYPES.index(dst), part, nparts, sl, qk, qs, qs2, qb, C.byref(out)))
        return OPlan(out.value, self)


class OPlan:
    """Oracle selection: outputs in order, each with dtype, bytes and scale entry."""

    def __init__(self, handle, index):
        self._h = C.c_void_p(handle)
        self.index = index

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value:
            lib().or_plan_free(self._h)
            self._h = C.c_void_p(None)

    def __len__(self):
        return lib().or_plan_count(self._h)

    def output(self, i):
        L = lib()
        e = self.index.entry(L.or_plan_entry(self._h, i))
        sc = L.or_plan_scale(self._h, i)
        if L.or_plan_quant(self._h, i):
            sc = L.or_plan_qscale(self._h, i)   # the block scales
        return {
            "name": L.or_plan_name(self._h, i).decode(),
            "entry": L.or_plan_entry(self._h, i),
            "dtype": DTYPES[L.or_plan_dtype(self._h, i)],
            "src_dtype": e["dtype"],
            "shape": [L.or_plan_dim(self.index.handle, self._h, i, d)
                      for d in range(L.or_plan_ndim(self.index.handle, self._h, i))],
            "numel": L.or_plan_numel(self._h, i),
            "begin": e["begin"],
            "scale": None if sc < 0 else self.index.entry(sc)["name"],
            "bytes": L.or_plan_bytes(self.index.handle, self._h, i),
            "quant": {0: None, 2: "block_fp8", 3: "nvfp4"}[L.or_plan_quant(self._h, i)],
        }

    def outputs(self):
        return [self.output(i) for i in range(len(self))]

    def materialize(self, i, data):
        """Output i as a uint8 numpy array; `data` is the data section (numpy uint8)."""
        data = np.ascontiguousarray(data, dtype=np.uint8)
        n = lib().or_plan_bytes(self.index.handle, self._h, i)
        dst = np.empty(max(1, n), dtype=np.uint8)
        _check(lib().or_materialize(self.index.handle, self._h, i, data.ctypes.data, data.size,
                                    dst.ctypes.data))
        return dst[:n]

    def materialize_range(self, i, data, first, count):
        """Elements [first, first + count) of output i, as uint8 bytes."""
        data = np.ascontiguousarray(data, dtype=np.uint8)
        so = ITEMSIZE[DTYPES[lib().or_plan_dtype(self._h, i)]]
        dst = np.empty(max(1, count * so), dtype=np.uint8)
        _check(lib().or_materialize_range(self.index.handle, self._h, i, data.ctypes.data, first,
                                          count, dst.ctypes.data))
        return dst[:count * so]


def parse(file_bytes):
    """Parses a whole file image (bytes or uint8 numpy array)."""
    arr = np.frombuffer(bytes(file_bytes), dtype=np.uint8) if not isinstance(file_bytes, np.ndarray) \
        else np.ascontiguousarray(file_bytes, dtype=np.uint8)
    out = C.c_void_p()
    _check(lib().or_parse(C.cast(arr.ctypes.data, C.c_char_p), arr.size, C.byref(out)))
    return OIndex(out.value)


def concat(parts, align=256):
    """Joined index over shard indexes; returns (index, bases)."""
    n = len(parts)
    hs = (C.c_void_p * max(1, n))(*[p.handle.value for p in parts])
    bases = (C.c_uint64 * max(1, n))()
    out = C.c_void_p()
    _check(lib().or_concat(hs, n, align, bases, C.byref(out)))
    return OIndex(out.value, keep=list(parts)), [int(b) for b in bases[:n]]


def parse_header(header, data_bytes):
    """Index from the first 8 + N bytes of a file and its data section size."""
    arr = np.frombuffer(bytes(header), dtype=np.uint8)
    out = C.c_void_p()
    _check(lib().or_parse_header(C.cast(arr.ctypes.data, C.c_char_p), arr.size, data_bytes, C.byref(out)))
    return OIndex(out.value)


def out_dtype(src, req):
    d = lib().or_out_dtype(DTYPES.index(src), DTYPES.index(req))
    return None if d < 0 else DTYPES[d]


def convert(src, out, data, scale=None):
    """Converts the raw little-endian elements in `data` (bytes or numpy) from
    dtype `src` to `out`; returns uint8 numpy bytes."""
    raw = np.frombuffer(bytes(data), dtype=np.uint8) if not isinstance(data, np.ndarray) \
        else np.ascontiguousarray(data).view(np.uint8).reshape(-1)
    n = raw.size // ITEMSIZE[src]
    dst = np.empty(max(1, n * ITEMSIZE[out]), dtype=np.uint8)
    _check(lib().or_convert(DTYPES.index(src), DTYPES.index(out), C.cast(raw.ctypes.data, C.c_char_p),
                            n, 1 if scale is not None else 0,
                            C.c_float(scale if scale is not None else 1.0), dst.ctypes.data))
    return dst[:n * ITEMSIZE[out]]
