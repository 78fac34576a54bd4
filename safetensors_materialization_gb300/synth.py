"""Seeded synthetic safetensors checkpoints for tests and benchmarks.

This module only builds inputs: tensor names/shapes/dtypes, the file layout
(8-byte little-endian header length, JSON header, contiguous data section)
and the bytes.  It holds none of the materialization arithmetic: values are
drawn in binary32 with numpy's PCG64 and turned into the file dtype by library
casts (numpy for binary16, torch CPU for bfloat16); fp8 tensors are uniform
over the non-NaN bit patterns, int64 tensors uniform over 64-bit patterns,
bool tensors uniform over {0, 1}.

Large tensors are filled from a seeded pool of 2^20 draws per dtype, copied in
seeded random windows of 2^16 elements, so that multi-GB checkpoints build in
seconds; every element is still a draw of the stated distribution.

The workloads mirror the checkpoints the streaming-loader design targets
("Disk tier safetensors streaming design audit (ComfyUI)": UNet checkpoints,
scaled-FP8 checkpoints, sharded LLM checkpoints, many small tensors).
"""
from __future__ import annotations

import json
import struct
from dataclasses import dataclass, field

import numpy as np

ITEMSIZE = {"BOOL": 1, "U8": 1, "I8": 1, "I16": 2, "U16": 2, "I32": 4, "U32": 4, "I64": 8,
            "U64": 8, "F16": 2, "BF16": 2, "F32": 4, "F64": 8, "F8_E4M3": 1, "F8_E5M2": 1}

POOL = 1 << 20
WINDOW = 1 << 16


@dataclass
class Entry:
    name: str
    dtype: str
    shape: list
    begin: int = 0
    end: int = 0

    @property
    def numel(self):
        n = 1
        for d in self.shape:
            n *= d
        return n

    @property
    def nbytes(self):
        return self.numel * ITEMSIZE[self.dtype]


@dataclass
class FileLayout:
    """One safetensors file: header bytes (length prefix + JSON + padding) and
    entries with their [begin, end) offsets in the data section."""
    header: bytes
    entries: list
    data_bytes: int

    @property
    def header_len(self):
        return len(self.header) - 8

    @property
    def data_start(self):
        return len(self.header)

    @property
    def file_bytes(self):
        return len(self.header) + self.data_bytes


def make_layout(entries, metadata=None, data_start_mod=(8, 0)):
    """Packs `entries` contiguously in the given order and writes the header.

    The header is padded with spaces until 8 + N == data_start_mod[1]
    (mod data_start_mod[0]); the format's writers pad to a multiple of 8.
    """
    off = 0
    for e in entries:
        e.begin = off
        off += e.nbytes
        e.end = off
    hdr = {}
    if metadata is not None:
        hdr["__metadata__"] = metadata
    for e in entries:
        hdr[e.name] = {"dtype": e.dtype, "shape": list(e.shape), "data_offsets": [e.begin, e.end]}
    js = json.dumps(hdr, separators=(",", ":")).encode()
    mod, rem = data_start_mod
    pad = (rem - (8 + len(js))) % mod
    js += b" " * pad
    return FileLayout(struct.pack("<Q", len(js)) + js, entries, off)


class Pools:
    """Per-dtype pools of seeded draws (bytes), built lazily."""

    def __init__(self, seed):
        self.seed = seed
        self._p = {}

    def get(self, dtype):
        if dtype not in self._p:
            rng = np.random.Generator(np.random.PCG64([self.seed, 7919, list(ITEMSIZE).index(dtype)]))
            self._p[dtype] = draw(rng, dtype, POOL)
        return self._p[dtype]


def draw(rng, dtype, n):
    """n elements of `dtype` as little-endian bytes (uint8 numpy array)."""
    if dtype in ("F32", "F16", "BF16", "F64"):
        x = rng.standard_normal(n, dtype=np.float32) * np.float32(0.02)
        if dtype == "F32":
            return x.view(np.uint8)
        if dtype == "F64":
            return x.astype(np.float64).view(np.uint8)
        if dtype == "F16":
            return x.astype(np.float16).view(np.uint8)
        import torch
        return torch.from_numpy(x).to(torch.bfloat16).view(torch.uint8).numpy()
    if dtype in ("F8_E4M3", "F8_E5M2"):
        if dtype == "F8_E4M3":   # NaN patterns are 0x7F and 0xFF
            v = rng.integers(0, 254, size=n, dtype=np.uint16)
            v = v + (v >= 127)
        else:                    # NaN patterns are 0x7D-0x7F and 0xFD-0xFF
            v = rng.integers(0, 250, size=n, dtype=np.uint16)
            v = v + 3 * (v >= 125)
        return v.astype(np.uint8)
    if dtype == "BOOL":
        return rng.integers(0, 2, size=n, dtype=np.uint8)
    return rng.integers(0, 256, size=n * ITEMSIZE[dtype], dtype=np.uint8)


def fill(layout: FileLayout, data: np.ndarray, seed: int):
    """Writes the data section of `layout` into `data` (uint8, data_bytes long)."""
    assert data.dtype == np.uint8 and data.size >= layout.data_bytes
    pools = Pools(seed)
    rng = np.random.Generator(np.random.PCG64([seed, 104729]))
    for e in layout.entries:
        si = ITEMSIZE[e.dtype]
        pool = pools.get(e.dtype)
        n = e.numel
        pos = 0
        while pos < n:
            k = min(WINDOW, n - pos)
            o = int(rng.integers(0, POOL - k + 1))
            data[e.begin + pos * si:e.begin + (pos + k) * si] = pool[o * si:(o + k) * si]
            pos += k


def build_file(layout: FileLayout, seed: int, out: np.ndarray | None = None):
    """Whole file image (header + data) as a uint8 numpy array."""
    buf = out if out is not None else np.empty(layout.file_bytes, dtype=np.uint8)
    hb = np.frombuffer(layout.header, dtype=np.uint8)
    buf[:hb.size] = hb
    fill(layout, buf[hb.size:hb.size + layout.data_bytes], seed)
    return buf


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    files: list                    # FileLayout per shard
    seeds: list                    # seed per shard
    dst: list                      # target dtype(s), one materialization run each
    prefix: str | None = None      # prefix view
    rename: list = field(default_factory=list)   # rename view rules
    scale_suffix: tuple | None = None            # (weight suffix, scale suffix)
    whole_file_on_device: bool = False           # stage the header too (keeps its misalignment)
    slices: dict | None = None                   # name -> (dim, start, stop) for sliced loads
    quant: dict | None = None                    # name -> (kind, scales, global scale, block) for block-scaled weights

    def view(self, ix):
        """The workload's view of an index (library or oracle: both spell
        view_rename / view_prefix the same way)."""
        if self.rename:
            ix = ix.view_rename(self.rename)
        if self.prefix:
            ix = ix.view_prefix(self.prefix)
        return ix

    def selection(self, ix):
        """Keyword arguments naming the workload's selection of a viewed index:
        explicit names with slices or block-scale descriptions where it has
        them, else {} (every entry, in index order)."""
        if not self.slices and not self.quant:
            return {}
        names = [e["name"] for e in ix.entries()]
        sel = {"names": names}
        if self.slices:
            sel["slices"] = [self.slices.get(n) for n in names]
        if self.quant:
            sel["quant"] = [self.quant.get(n) for n in names]
        return sel


def tiny(seed=0):
    """16 tensors model.t{i}: shapes from {[64],[256,256],[128,64,3,3],[1024,32]},
    dtypes from {F32, F16, BF16}; prefix view 'model.' to BF16."""
    rng = np.random.Generator(np.random.PCG64(seed))
    shapes = [[64], [256, 256], [128, 64, 3, 3], [1024, 32]]
    dts = ["F32", "F16", "BF16"]
    ents = [Entry(f"model.t{i}", dts[int(rng.integers(0, 3))], shapes[int(rng.integers(0, 4))])
            for i in range(16)]
    lay = make_layout(ents, metadata={"format": "pt"})
    return Workload("tiny_16_mixed", [lay], [seed], ["BF16"], prefix="model.")


def unet(seed=1, n1280=38):
    """UNet-shaped fp16 checkpoint (716 tensors, 1.334 G params) under
    'model.diffusion_model.'; rename view to 'unet.' and BF16.  n1280 sets the
    number of 1280-channel resblocks (38 in the full checkpoint)."""
    p = "model.diffusion_model."
    ents = []
    for C, n in ((320, 6), (640, 6), (1280, n1280)):
        for i in range(n):
            b = f"{p}res_{C}_{i:02d}."
            ents += [Entry(b + "conv1.weight", "F16", [C, C, 3, 3]), Entry(b + "conv1.bias", "F16", [C]),
                     Entry(b + "conv2.weight", "F16", [C, C, 3, 3]), Entry(b + "conv2.bias", "F16", [C]),
                     Entry(b + "norm1.weight", "F16", [C]), Entry(b + "norm1.bias", "F16", [C]),
                     Entry(b + "norm2.weight", "F16", [C]), Entry(b + "norm2.bias", "F16", [C])]
    for C, n in ((320, 4), (640, 4), (1280, 20)):
        for i in range(n):
            b = f"{p}attn_{C}_{i:02d}."
            ents += [Entry(b + f"to_{k}.weight", "F16", [C, C]) for k in ("q", "k", "v", "out")]
            ents += [Entry(b + "to_out.bias", "F16", [C])]
            ents += [Entry(b + f"norm{j}.{w}", "F16", [C]) for j in (1, 2, 3) for w in ("weight", "bias")]
    for j, (co, ci) in enumerate(((640, 320), (1280, 640), (640, 1280), (320, 640))):
        ents += [Entry(f"{p}transition_{j}.weight", "F16", [co, ci, 3, 3]),
                 Entry(f"{p}transition_{j}.bias", "F16", [co])]
    ents.sort(key=lambda e: e.name)
    lay = make_layout(ents, metadata={"format": "pt"})
    name = "unet_fp16_716" if n1280 == 38 else f"unet_fp16_{len(ents)}"
    return Workload(name, [lay], [seed], ["BF16"], rename=[(p, "unet.")])


def scaled_fp8(seed=2, blocks=57):
    """57 blocks x (6 x [3072,3072] + 4 x [12288,3072]) F8_E4M3 weights, each
    with a scalar F32 'scale_weight' uniform in [1e-3, 1e-1]; BF16."""
    ents = []
    for b in range(blocks):
        for lin, shape in [(f"attn.{k}", [3072, 3072]) for k in ("q", "k", "v", "o")] + \
                          [(f"mod.{k}", [3072, 3072]) for k in ("a", "b")] + \
                          [(f"mlp.fc{k}", [12288, 3072]) for k in (1, 2, 3, 4)]:
            base = f"model.diffusion_model.blocks.{b:02d}.{lin}."
            ents += [Entry(base + "weight", "F8_E4M3", shape), Entry(base + "scale_weight", "F32", [])]
    ents.sort(key=lambda e: e.name)
    lay = make_layout(ents, metadata={"format": "pt", "quantization": "scaled_fp8"})
    return Workload(f"scaled_fp8_e4m3_{blocks}blk", [lay], [seed], ["BF16"],
                    scale_suffix=(".weight", ".scale_weight"))


def fill_scales(layout: FileLayout, data: np.ndarray, seed: int):
    """Overwrites every one-element F32 tensor with a value uniform in [1e-3, 1e-1]."""
    rng = np.random.Generator(np.random.PCG64([seed, 15485863]))
    for e in layout.entries:
        if e.dtype == "F32" and e.numel == 1:
            v = np.float32(rng.uniform(1e-3, 1e-1))
            data[e.begin:e.end] = np.frombuffer(v.tobytes(), dtype=np.uint8)


def llm8b(seed=3, layers=32, hidden=4096, inter=14336, vocab=128256, kv=1024, shards=4):
    """8B LLM-shaped BF16 checkpoint over 4 shard files split at layer
    boundaries; materialized twice: BF16 (copy) and F16 (cast)."""
    groups = [[Entry("model.embed_tokens.weight", "BF16", [vocab, hidden])]]
    for i in range(layers):
        b = f"model.layers.{i}."
        groups.append([
            Entry(b + "self_attn.q_proj.weight", "BF16", [hidden, hidden]),
            Entry(b + "self_attn.k_proj.weight", "BF16", [kv, hidden]),
            Entry(b + "self_attn.v_proj.weight", "BF16", [kv, hidden]),
            Entry(b + "self_attn.o_proj.weight", "BF16", [hidden, hidden]),
            Entry(b + "mlp.gate_proj.weight", "BF16", [inter, hidden]),
            Entry(b + "mlp.up_proj.weight", "BF16", [inter, hidden]),
            Entry(b + "mlp.down_proj.weight", "BF16", [hidden, inter]),
            Entry(b + "input_layernorm.weight", "BF16", [hidden]),
            Entry(b + "post_attention_layernorm.weight", "BF16", [hidden]),
        ])
    groups[-1] += [Entry("model.norm.weight", "BF16", [hidden]),
                   Entry("lm_head.weight", "BF16", [vocab, hidden])]
    total = sum(e.nbytes for g in groups for e in g)
    files, cur, acc, k = [], [], 0, 1
    for g in groups:
        cur += g
        acc += sum(e.nbytes for e in g)
        if acc >= k * total / shards and k < shards:
            files.append(cur)
            cur, k = [], k + 1
    files.append(cur)
    lays = [make_layout(sorted(f, key=lambda e: e.name), metadata={"format": "pt"}) for f in files]
    return Workload("llm8b_bf16_4shard", lays, [seed * 100 + i for i in range(len(lays))], ["BF16", "F16"])


def stress(seed=4, n=100_000):
    """100k tensors, numel uniform in 1..4096, dtypes uniform over
    {F32, F16, BF16, F8_E4M3, F8_E5M2, I64, BOOL}; the header is padded so the
    data section starts at 7 (mod 16) and numels are nudged so that no tensor
    starts on a 16-byte boundary of a 256-byte-aligned file image."""
    rng = np.random.Generator(np.random.PCG64(seed))
    dts = ["F32", "F16", "BF16", "F8_E4M3", "F8_E5M2", "I64", "BOOL"]
    dsel = rng.integers(0, len(dts), size=n)
    numel = rng.integers(1, 4097, size=n)
    ents = [Entry(f"stress.{i:06d}", dts[int(dsel[i])], [int(numel[i])]) for i in range(n)]
    # With the data section at 7 (mod 16), walk the tensors in order; when the
    # next start would land on a 16-byte boundary, grow (or, at 4096, shrink)
    # the previous tensor by one element, which moves the start by its itemsize
    # (1, 2, 4 or 8 bytes) and so off the boundary.
    start_mod = 7
    off = start_mod
    for i, e in enumerate(ents):
        if i > 0 and off % 16 == 0:
            prev = ents[i - 1]
            step = 1 if prev.shape[0] < 4096 else -1
            prev.shape = [prev.shape[0] + step]
            off += step * ITEMSIZE[prev.dtype]
        off += e.nbytes
    lay = make_layout(ents, data_start_mod=(16, start_mod))
    return Workload("stress_100k_misaligned", [lay], [seed], ["BF16"], whole_file_on_device=True)


def tp_slices(entries, tp, rank):
    """Megatron-style tensor-parallel shard `rank` of `tp` for Llama names:
    column-parallel projections (q/k/v, gate/up) and the vocab-parallel
    embedding and head split dim 0; row-parallel ones (o, down) split dim 1
    (a strided gather); norms stay whole."""
    out = {}
    for e in entries:
        n = e.name
        if any(k in n for k in ("q_proj", "k_proj", "v_proj", "gate_proj", "up_proj", "embed_tokens", "lm_head")):
            d = 0
        elif any(k in n for k in ("o_proj", "down_proj")):
            d = 1
        else:
            continue
        size = e.shape[d] // tp
        out[n] = (d, rank * size, (rank + 1) * size)
    return out


def llm8b_tp4(seed=3):
    """Shard file 0 of the 8B LLM checkpoint loaded as tensor-parallel rank 0
    of 4: BF16 copies of the rank's slices."""
    w = llm8b(seed)
    lay = w.files[0]
    return Workload("llm8b_shard0_tp4_rank0", [lay], [w.seeds[0]], ["BF16"],
                    slices=tp_slices(lay.entries, 4, 0))


def _linears(blocks):
    for b in range(blocks):
        for lin, shape in [(f"self_attn.{k}_proj", [3072, 3072]) for k in ("q", "k", "v", "o")] + \
                          [(f"mlp.{k}_proj", [12288, 3072]) for k in ("gate", "up")] + \
                          [("mlp.down_proj", [3072, 12288])]:
            yield f"model.layers.{b:02d}.{lin}.", shape


def block_fp8(seed=5, blocks=40):
    """Block-FP8 transformer weights (the DeepSeek/Qwen FP8 layout): E4M3
    linears with an F32 'weight_scale_inv' per 128 x 128 block; BF16 out.
    40 layers x (4 x [3072,3072] + 3 x [12288,3072]/[3072,12288]): 6.04 GB of
    weights, 12.08 GB of BF16 out."""
    ents, quant = [], {}
    for base, (M, N) in _linears(blocks):
        ents += [Entry(base + "weight", "F8_E4M3", [M, N]),
                 Entry(base + "weight_scale_inv", "F32", [-(-M // 128), -(-N // 128)])]
        quant[base + "weight"] = ("block_fp8", base + "weight_scale_inv", None, (128, 128))
    ents.sort(key=lambda e: e.name)
    lay = make_layout(ents, metadata={"format": "pt", "quantization": "block_fp8"})
    return Workload(f"block_fp8_e4m3_{blocks}layer", [lay], [seed], ["BF16"], quant=quant)


def nvfp4(seed=6, blocks=40):
    """NVFP4 transformer weights (the ModelOpt layout): U8 [M, N/2] packed
    E2M1 pairs, an E4M3 'weight_scale' per 16 elements of a row and an F32
    'weight_scale_2'; the same 40 layers as block_fp8; BF16 out."""
    ents, quant = [], {}
    for base, (M, N) in _linears(blocks):
        ents += [Entry(base + "weight", "U8", [M, N // 2]),
                 Entry(base + "weight_scale", "F8_E4M3", [M, N // 16]),
                 Entry(base + "weight_scale_2", "F32", [])]
        quant[base + "weight"] = ("nvfp4", base + "weight_scale", base + "weight_scale_2", None)
    ents.sort(key=lambda e: e.name)
    lay = make_layout(ents, metadata={"format": "pt", "quantization": "nvfp4"})
    return Workload(f"nvfp4_{blocks}layer", [lay], [seed], ["BF16"], quant=quant)


WORKLOADS = {"tiny": tiny, "unet": unet, "scaled_fp8": scaled_fp8, "llm8b": llm8b, "stress": stress,
             # a 5-block slice of the scaled-fp8 checkpoint (1.04 GB source), for profiling
             "scaled_fp8_5blk": lambda: scaled_fp8(blocks=5),
             # a UNet with 8 of the 38 1280-channel resblocks (0.83 GB source), for profiling
             "unet_small": lambda: unet(n1280=8),
             "llm8b_tp4": llm8b_tp4,
             # the same 4-shard checkpoint cast to F16 (the second run of the LLM config)
             "llm8b_f16": lambda: _with_dst(llm8b(), ["F16"]),
             "block_fp8": block_fp8, "nvfp4": nvfp4,
             # 4-layer slices of the same constructions, for tests and profiling
             "block_fp8_4l": lambda: block_fp8(blocks=4), "nvfp4_4l": lambda: nvfp4(blocks=4)}


def _with_dst(wl: Workload, dst):
    wl.dst = dst
    wl.name += "_to_" + dst[0].lower()
    return wl


def fill_block_scales(wl: Workload, layout: FileLayout, data: np.ndarray, seed: int):
    """Block scales of block-scaled weights: F32 block-FP8 scales uniform in
    [1e-3, 1e-1]; NVFP4 E4M3 scales uniform over the codes of 2^-6 .. 2^2
    (0x08..0x47); NVFP4 global scales uniform in [1e-4, 1e-2]."""
    rng = np.random.Generator(np.random.PCG64([seed, 32452843]))
    by_name = {e.name: e for e in layout.entries}
    for kind, sname, gname, _ in (wl.quant or {}).values():
        e = by_name.get(sname)
        if e is None:
            continue
        if kind == "block_fp8":
            data[e.begin:e.end] = rng.uniform(1e-3, 1e-1, size=e.numel).astype(np.float32).view(np.uint8)
        else:
            data[e.begin:e.end] = rng.integers(0x08, 0x48, size=e.numel, dtype=np.uint8)
            g = by_name[gname]
            data[g.begin:g.end] = np.frombuffer(np.float32(rng.uniform(1e-4, 1e-2)).tobytes(), dtype=np.uint8)


def build_workload_data(wl: Workload, k: int, out: np.ndarray):
    """Data section of shard k of workload `wl` into `out` (uint8, data_bytes long)."""
    lay = wl.files[k]
    fill(lay, out, wl.seeds[k])
    if wl.scale_suffix:
        fill_scales(lay, out, wl.seeds[k])
    if wl.quant:
        fill_block_scales(wl, lay, out, wl.seeds[k])
    return out


def build_workload_file(wl: Workload, k: int, out: np.ndarray | None = None):
    """File image of shard k of workload `wl` (scales filled for scaled-fp8)."""
    lay = wl.files[k]
    buf = build_file(lay, wl.seeds[k], out)
    if wl.scale_suffix:
        fill_scales(lay, buf[lay.data_start:], wl.seeds[k])
    if wl.quant:
        fill_block_scales(wl, lay, buf[lay.data_start:], wl.seeds[k])
    return buf
