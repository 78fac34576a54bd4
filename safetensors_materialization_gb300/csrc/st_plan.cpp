// st_plan.cpp -- selection, output dtypes, scale pairing, byte-balanced work
// partition, device tables, and the stream-ordered entry points
// (st_materialize, st_stage_h2d, st_load).
//
// "Disk tier safetensors streaming design audit (ComfyUI)":
//  - "ComfyUI load path + eager materialization sites": the scaled-FP8
//    conversion (comfy/sd.py) pairs fp8 weights with per-tensor scales;
//    BaseModel.load_model_weights selects tensors by name/prefix;
//  - "VRAM/RAM offload logic": weights are cast at load (comfy_cast_weights);
//  - "Range reads and tiering", Disk->RAM->GPU: only the tensors' byte ranges
//    are staged from (pinned) host memory and copied to the GPU.
//
// Work layout: every output is cut into pieces (element ranges); pieces are
// balanced by bytes (source + destination, plus a fixed per-piece cost) over
// W warps, so that huge tensors and 100k tiny tensors spread evenly over the
// GPU.  With chunking, the data section is split into chunks and each chunk
// has its own balanced partition, so a chunk can be materialized as soon as
// its bytes are on the device.
#include <cuda_runtime_api.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <new>
#include <string>
#include <string_view>
#include <vector>

#include "st_index.h"
#include "st_internal.h"

namespace stmat {
namespace {

constexpr uint64_t kSplitBytes = 2048;      // pieces of one output start at multiples of this many
                                            // source bytes: one full batch of lane steps
constexpr uint64_t kPieceCost = 1024;       // fixed cost of a piece, in bytes of traffic
constexpr uint64_t kMinWorkerCost = 4096;   // no more warps than total cost / this
constexpr uint64_t kMaxPieceUnits = 1ull << 30;
constexpr uint64_t kDefaultUnitBytes = 32768;  // cost of one interleaved unit
// The TMA build's default unit: smaller units make finer pieces for its
// claimed tail (100k tiny tensors 0.867 -> 0.886-0.891 of the copy peak at
// 16 KiB; 8-20 KiB all within 0.88-0.89; block-scaled weights on the wide
// build measured 0.93-0.96 at 16 KiB against 0.96-0.97 at 32 KiB).
constexpr uint64_t kTmaUnitBytes = 16384;
// The TMA build's claimed tail is cut further, into pieces of at most this
// many source bytes (one 2 KiB segment), which its warps claim at least two
// at a time: a warp that claims the last whole 16 KiB unit finishes up to
// 8 segments after the others.  Measured on 100k tiny tensors: 0.899-0.902
// -> 0.912-0.915 of the copy peak; 3 KiB pieces 0.905, 1 KiB 0.843, claims of
// one piece 0.904-0.907, the same claims of whole units 0.886.  The wide
// build keeps whole units (its 40 % tail cut to 2-8 KiB pieces: block FP8
// 0.974 -> 0.945-0.966, NVFP4 0.973 -> 0.934-0.973).
constexpr uint64_t kTmaTailPieceBytes = 2048;
// Single-chunk plans whose source bytes span at most this much of the data
// section (and fill at least half of that span) prefetch their piece table,
// destination array and that span into L2 as the launch starts, so that the
// dependent reads after the warp's first (parts) read hit L2 (16 tiny
// tensors, L2 flushed before each launch: 9.9 -> 8.8 us per launch).  Only
// when the data section and the destination array are this GPU's memory.
constexpr uint64_t kPrefetchMaxBytes = 16ull << 20;
// Percent of a chunk's cost (whole rounds of units) that warps claim while
// they run instead of owning it, by build (measured best, fractions of the
// copy peak): TMA, 100k tiny tensors 8 % (0.851 with fixed shares -> 0.895-0.903;
// 4-6 % 0.89-0.895, 10-12 % 0.886-0.894, 14 % 0.874-0.883); wide TMA, block-scaled
// weights 40 % (block FP8 0.896 -> 0.974, NVFP4 0.843 -> 0.965); streaming,
// long contiguous runs 20 % (scaled FP8 0.972 -> 0.992, LLM 0.968 -> 1.02,
// UNet 0.971 -> 0.977; 30-40 % the same within 0.3 %), short runs (a
// tensor-parallel rank's row slices) 30 % (0.923 at 3 blocks per SM with
// fixed shares -> 0.988 at 2 blocks per SM; 15 % 0.91, 20 % 0.982, 40 % 0.990).
constexpr uint64_t kClaimedPct = 8, kClaimedPctWide = 40, kClaimedPctStream = 20, kClaimedPctStreamShort = 30;
constexpr uint64_t kLazyBytesPerWarp = 16384;  // st_load_tensors: traffic per warp
constexpr uint64_t kLazyMaxWarps = 2432;        // ... and at most this many warps (2 blocks on each of 152 SMs)
constexpr uint32_t kStreamBlocksPerSm = 2;  // streaming build: fewer, deeper warps
constexpr uint64_t kLongRunBytes = 65536;       // mean traffic per contiguous run that counts as long
constexpr uint64_t kSmallOutputBytes = 65536;  // mean traffic per output below which the
                                               // latency build is chosen

bool is_fp8(int d) { return d == ST_F8_E4M3 || d == ST_F8_E5M2; }
bool is_float(int d) {
  return d == ST_F16 || d == ST_BF16 || d == ST_F32 || d == ST_F64 || d == ST_F8_E4M3 || d == ST_F8_E5M2;
}

// Output dtype for a source dtype and a request, or -1.
int out_dtype_of(int src, int req) {
  if (req == ST_KEEP || !is_float(src)) return src;
  if (src == ST_F64) return -1;
  return req;
}

// Conversion class for (source, output); scaled outputs are never copies.
int class_of(int src, int out, bool scaled) {
  if (src == out && !scaled) return CLS_COPY;
  switch (src) {
    case ST_F32: return out == ST_BF16 ? CLS_F32_BF16 : out == ST_F16 ? CLS_F32_F16 : -1;
    case ST_F16: return out == ST_BF16 ? CLS_F16_BF16 : out == ST_F32 ? CLS_F16_F32 : -1;
    case ST_BF16: return out == ST_F16 ? CLS_BF16_F16 : out == ST_F32 ? CLS_BF16_F32 : -1;
    case ST_F8_E4M3:
      return out == ST_BF16 ? CLS_E4M3_BF16 : out == ST_F16 ? CLS_E4M3_F16 : out == ST_F32 ? CLS_E4M3_F32 : -1;
    case ST_F8_E5M2:
      return out == ST_BF16 ? CLS_E5M2_BF16 : out == ST_F16 ? CLS_E5M2_F16 : out == ST_F32 ? CLS_E5M2_F32 : -1;
    default: return -1;
  }
}

std::string cuda_msg(cudaError_t e) {
  return std::string(cudaGetErrorName(e)) + ": " + cudaGetErrorString(e);
}

}  // namespace

struct Output {
  std::string name;
  uint32_t pos;        // position in the index/view
  uint32_t entry;      // core tensor
  int out_dtype;
  int64_t scale = -1;  // core tensor of the scale
  std::vector<uint32_t> reads;  // view positions of every tensor the output reads (itself first)
  uint32_t cls;
  uint64_t numel;      // output elements (after slicing)
  uint64_t units;      // counted units (elements, or bytes for copies)
  std::vector<int64_t> shape;  // output shape
  int32_t sdim = -1;   // slice
  int64_t start = 0, stop = 0;
  // Block-scaled weights: the format and its scale table entry.
  int32_t qkind = ST_QUANT_NONE;
  int64_t qscale_entry = -1;  // core tensor of the block scales
  QuantInfo quant{};
  // Source geometry in counted units: `runs` runs of `run` units; run r
  // starts at data-section byte src0 + r * pitch.  One run unless an inner
  // dimension is sliced.
  uint64_t runs = 1, run = 0, src0 = 0, pitch = 0;
  // Data-section byte of output unit u.
  uint64_t unit_src(uint64_t u) const {
    return runs == 1 ? src0 + u * cls_in_size(cls) : src0 + (u / run) * pitch + (u % run) * cls_in_size(cls);
  }
};

}  // namespace stmat

using namespace stmat;

struct st_plan_s {
  std::shared_ptr<const IndexData> index;
  std::vector<Output> outs;
  uint32_t workers = 1;
  uint32_t kernel = kKernelStream;
  uint64_t chunk_bytes = 0;
  uint64_t unit_bytes = kDefaultUnitBytes;
  bool class_major = false;
  bool long_runs = false;  // the outputs' contiguous runs average kLongRunBytes or more
  uint32_t n_chunks = 1;
  // Data-section byte ranges the plan reads (sorted, merged); `sparse` when
  // they cover under three quarters of it (a tensor-parallel rank's load):
  // the loaders then copy only these.
  std::vector<std::pair<uint64_t, uint64_t>> ranges;
  bool sparse = false;
  uint64_t pf_lo = 0, pf_hi = 0;  // the span a single-chunk launch prefetches (empty: none)
  std::vector<Piece> pieces;
  std::vector<uint32_t> parts;  // n_chunks * (workers + 1)
  std::vector<uint32_t> claim_end;  // per chunk: end of the pieces claimed at run time (TMA builds)
  // device side
  bool on_device = false;
  int device = -1;
  Piece *d_pieces = nullptr;
  uint32_t *d_parts = nullptr;
  uint32_t *d_err = nullptr;
  uint32_t *d_claim = nullptr;
  std::vector<QuantInfo> quant;  // per output, when any output is block-scaled
  QuantInfo *d_quant = nullptr;
  std::vector<cudaEvent_t> events;  // one per chunk + one for st_load's start
  ~st_plan_s() {
    if (!on_device) return;
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != device) cudaSetDevice(device);
    for (cudaEvent_t e : events) cudaEventDestroy(e);
    cudaFree(d_pieces);
    cudaFree(d_parts);
    cudaFree(d_err);
    cudaFree(d_claim);
    cudaFree(d_quant);
    if (cur != device && cur >= 0) cudaSetDevice(cur);
  }
};

namespace {

uint32_t log2_of(uint64_t v) {
  uint32_t k = 0;
  while ((1ull << k) < v) ++k;
  return k;
}

// Checks selected name `p` against its block-scaled format (see st_block_quant)
// and fills the output's format fields; marks the scale tensors consumed.
st_status check_quant(const IndexData &ix, uint32_t p, const st_block_quant &q, Output *o,
                      std::vector<char> *consumed) {
  const Core &core = *ix.core;
  const Tensor &t = core.tensors[ix.ent[p]];
  const char *nm = ix.names[p];
  if (q.kind != ST_QUANT_BLOCK_FP8 && q.kind != ST_QUANT_NVFP4)
    return set_error(ST_E_INVAL, "\"%s\": unknown block-scaled format %d", nm, q.kind);
  if (!q.scale) return set_error(ST_E_INVAL, "\"%s\": no block-scales tensor named", nm);
  auto it = ix.pos.find(std::string_view(q.scale));
  if (it == ix.pos.end()) return set_error(ST_E_NOT_FOUND, "no block-scales tensor named \"%s\"", q.scale);
  const uint32_t sp = it->second;
  const Tensor &sc = core.tensors[ix.ent[sp]];
  if (t.shape.size() != 2) return set_error(ST_E_INVAL, "\"%s\": a block-scaled weight is 2-D", nm);
  const uint64_t M = static_cast<uint64_t>(t.shape[0]);
  uint64_t br = q.block_rows, bc = q.block_cols, N;
  o->quant.scale2 = kNoScale;
  if (q.kind == ST_QUANT_BLOCK_FP8) {
    if (br == 0) br = 128;
    if (bc == 0) bc = 128;
    N = static_cast<uint64_t>(t.shape[1]);
    if (!is_fp8(t.dtype) || (br & (br - 1)) || (bc & (bc - 1)) || bc < 16 || br > (1u << 30) || bc > (1u << 30))
      return set_error(ST_E_INVAL, "\"%s\": block FP8 needs an fp8 weight and power-of-two blocks, >= 16 columns", nm);
    if (sc.dtype != ST_F32 || sc.shape.size() != 2 || static_cast<uint64_t>(sc.shape[0]) != (M + br - 1) / br ||
        static_cast<uint64_t>(sc.shape[1]) != (N + bc - 1) / bc)
      return set_error(ST_E_INVAL, "\"%s\": block scales must be F32 [ceil(M/%llu), ceil(N/%llu)]", q.scale,
                       static_cast<unsigned long long>(br), static_cast<unsigned long long>(bc));
    o->quant.row_units = static_cast<uint32_t>(N);
  } else {
    if (!((br == 0 && bc == 0) || (br == 1 && bc == 16)))
      return set_error(ST_E_INVAL, "\"%s\": NVFP4 blocks are 1 x 16", nm);
    br = 1;
    bc = 16;
    if (t.dtype != ST_U8 || !q.scale2)
      return set_error(ST_E_INVAL, "\"%s\": NVFP4 needs a U8 weight and a global scale", nm);
    auto it2 = ix.pos.find(std::string_view(q.scale2));
    if (it2 == ix.pos.end()) return set_error(ST_E_NOT_FOUND, "no global scale tensor named \"%s\"", q.scale2);
    N = 2 * static_cast<uint64_t>(t.shape[1]);
    if (sc.dtype != ST_F8_E4M3 || sc.shape.size() != 2 || static_cast<uint64_t>(sc.shape[0]) != M ||
        static_cast<uint64_t>(sc.shape[1]) != (N + 15) / 16)
      return set_error(ST_E_INVAL, "\"%s\": NVFP4 scales must be F8_E4M3 [M, ceil(2K/16)]", q.scale);
    const Tensor &g = core.tensors[ix.ent[it2->second]];
    if (g.dtype != ST_F32 || g.numel != 1)
      return set_error(ST_E_INVAL, "\"%s\": the global scale is a one-element F32 tensor", q.scale2);
    (*consumed)[it2->second] = 1;
    o->reads.push_back(it2->second);
    o->quant.scale2 = g.begin;
    o->quant.row_units = static_cast<uint32_t>(t.shape[1]);
  }
  if (N > (1u << 30)) return set_error(ST_E_INVAL, "\"%s\": a block-scaled row holds at most 2^30 elements", nm);
  (*consumed)[sp] = 1;
  o->qkind = q.kind;
  o->qscale_entry = ix.ent[sp];
  o->reads.push_back(sp);
  o->quant.scale = sc.begin;
  o->quant.scols = static_cast<uint32_t>(sc.shape[1]);
  o->quant.br_shift = log2_of(br);
  o->quant.bc_shift = log2_of(bc);
  return ST_OK;
}

// Selection -> outputs (order, dtype, scale), with the part filter.
st_status select_outputs(const IndexData &ix, const st_selection *sel, int req, std::vector<Output> *outs) {
  const Core &core = *ix.core;
  const bool all = !sel || !sel->names;
  const size_t n = all ? ix.ent.size() : sel->n_names;
  uint32_t n_parts = sel ? sel->n_parts : 0, part = sel ? sel->part : 0;
  if (n_parts == 0) n_parts = 1;
  if (part >= n_parts) return set_error(ST_E_INVAL, "part %u of %u", part, n_parts);
  if (req != ST_BF16 && req != ST_F16 && req != ST_F32 && req != ST_KEEP)
    return set_error(ST_E_UNSUPPORTED_CAST, "output dtype must be BF16, F16, F32 or KEEP");
  if (sel && sel->scale_names && all) return set_error(ST_E_INVAL, "scale_names needs names");
  std::vector<uint32_t> pos(n);
  std::vector<char> taken(ix.ent.size(), 0);
  for (size_t i = 0; i < n; ++i) {
    if (all) {
      pos[i] = static_cast<uint32_t>(i);
    } else {
      const char *nm = sel->names[i];
      if (!nm) return set_error(ST_E_INVAL, "NULL name at %zu", i);
      auto it = ix.pos.find(std::string_view(nm));
      if (it == ix.pos.end()) return set_error(ST_E_NOT_FOUND, "no tensor named \"%s\"", nm);
      pos[i] = it->second;
    }
    if (taken[pos[i]]) return set_error(ST_E_DUP_KEY, "\"%s\" selected twice", ix.names[pos[i]]);
    taken[pos[i]] = 1;
  }
  const st_slice *slices = sel ? sel->slices : nullptr;
  if (slices && all) return set_error(ST_E_INVAL, "slices need names");
  for (size_t i = 0; slices && i < n; ++i) {
    const Tensor &t = core.tensors[ix.ent[pos[i]]];
    const st_slice &sl = slices[i];
    if (sl.dim < 0) continue;
    if (sl.dim >= static_cast<int32_t>(t.shape.size()) || sl.start < 0 || sl.start > sl.stop ||
        sl.stop > t.shape[sl.dim])
      return set_error(ST_E_INVAL, "slice (dim %d, %lld..%lld) does not fit \"%s\"", sl.dim,
                       static_cast<long long>(sl.start), static_cast<long long>(sl.stop), ix.names[pos[i]]);
  }
  std::vector<char> consumed(ix.ent.size(), 0);
  // Block-scaled formats (explicit, per name).
  const st_block_quant *quant = sel ? sel->quant : nullptr;
  if (quant && all) return set_error(ST_E_INVAL, "quant needs names");
  std::vector<Output> qout(n);
  for (size_t i = 0; quant && i < n; ++i) {
    const st_block_quant &q = quant[i];
    if (q.kind == ST_QUANT_NONE) continue;
    const char *nm = ix.names[pos[i]];
    if ((slices && slices[i].dim >= 0) || (sel->scale_names && sel->scale_names[i]))
      return set_error(ST_E_INVAL, "\"%s\": a block-scaled output takes no slice and no per-tensor scale", nm);
    if (req == ST_KEEP) return set_error(ST_E_UNSUPPORTED_CAST, "KEEP cannot apply block scales");
    st_status st = check_quant(ix, pos[i], q, &qout[i], &consumed);
    if (st != ST_OK) return st;
  }
  // Scale pairing.
  std::vector<int64_t> scale(n, -1);  // position of the scale in the view
  const char *from = sel ? sel->scale_suffix_from : nullptr;
  const char *to = sel ? sel->scale_suffix_to : nullptr;
  const size_t flen = from ? strlen(from) : 0;
  std::string cand;
  for (size_t i = 0; i < n; ++i) {
    const Tensor &t = core.tensors[ix.ent[pos[i]]];
    if (qout[i].qkind != ST_QUANT_NONE) continue;
    if (sel && sel->scale_names) {
      const char *sn = sel->scale_names[i];
      if (sn) {
        auto it = ix.pos.find(std::string_view(sn));
        if (it == ix.pos.end()) return set_error(ST_E_NOT_FOUND, "no scale tensor named \"%s\"", sn);
        scale[i] = it->second;
      }
    } else if (from && to && is_fp8(t.dtype)) {
      std::string_view nm(ix.names[pos[i]]);
      if (nm.size() >= flen && nm.substr(nm.size() - flen) == from) {
        cand.assign(nm.data(), nm.size() - flen);
        cand += to;
        auto it = ix.pos.find(std::string_view(cand));
        if (it != ix.pos.end()) scale[i] = it->second;
      }
    }
    if (scale[i] >= 0) {
      const Tensor &s = core.tensors[ix.ent[scale[i]]];
      if (!is_fp8(t.dtype) || s.dtype != ST_F32 || s.numel != 1)
        return set_error(ST_E_INVAL, "\"%s\" cannot scale \"%s\": scales are one-element F32 tensors of fp8 weights",
                         ix.names[scale[i]], ix.names[pos[i]]);
      if (req == ST_KEEP) return set_error(ST_E_UNSUPPORTED_CAST, "KEEP cannot apply a scale");
      consumed[scale[i]] = 1;
    }
  }
  for (size_t i = 0; i < n; ++i) {
    if (consumed[pos[i]]) continue;
    const Tensor &t = core.tensors[ix.ent[pos[i]]];
    if (qout[i].qkind != ST_QUANT_NONE) {
      Output o = std::move(qout[i]);
      o.reads.insert(o.reads.begin(), pos[i]);
      o.name = ix.names[pos[i]];
      o.pos = pos[i];
      o.entry = ix.ent[pos[i]];
      o.out_dtype = req;
      const bool nv = o.qkind == ST_QUANT_NVFP4;
      const uint32_t base = nv ? CLS_NVFP4_BF16 : t.dtype == ST_F8_E4M3 ? CLS_QE4M3_BF16 : CLS_QE5M2_BF16;
      o.cls = base + (req == ST_BF16 ? 0 : req == ST_F16 ? 1 : 2);
      o.shape = {t.shape[0], nv ? 2 * t.shape[1] : t.shape[1]};
      o.numel = static_cast<uint64_t>(o.shape[0]) * static_cast<uint64_t>(o.shape[1]);
      o.src0 = t.begin;
      o.units = t.numel;  // elements, or NVFP4 bytes
      o.run = o.units;
      outs->push_back(std::move(o));
      continue;
    }
    int od = out_dtype_of(t.dtype, req);
    if (od < 0)
      return set_error(ST_E_UNSUPPORTED_CAST, "\"%s\": %s cannot be materialized as %s", ix.names[pos[i]],
                       st_dtype_name(static_cast<st_dtype>(t.dtype)), st_dtype_name(static_cast<st_dtype>(req)));
    Output o;
    o.name = ix.names[pos[i]];
    o.pos = pos[i];
    o.entry = ix.ent[pos[i]];
    o.out_dtype = od;
    o.scale = scale[i] >= 0 ? static_cast<int64_t>(ix.ent[scale[i]]) : -1;
    o.reads.push_back(pos[i]);
    if (scale[i] >= 0) o.reads.push_back(static_cast<uint32_t>(scale[i]));
    int c = class_of(t.dtype, od, o.scale >= 0);
    if (c < 0) return set_error(ST_E_UNSUPPORTED_CAST, "no conversion for \"%s\"", o.name.c_str());
    o.cls = static_cast<uint32_t>(c);
    const uint64_t isz = dtype_size(t.dtype), upe = c == CLS_COPY ? isz : 1;  // units per element
    o.shape = t.shape;
    o.numel = t.numel;
    o.src0 = t.begin;
    if (slices && slices[i].dim >= 0) {
      const st_slice &sl = slices[i];
      uint64_t outer = 1, inner = 1;
      for (int32_t d = 0; d < sl.dim; ++d) outer *= static_cast<uint64_t>(t.shape[d]);
      for (size_t d = sl.dim + 1; d < t.shape.size(); ++d) inner *= static_cast<uint64_t>(t.shape[d]);
      const uint64_t D = static_cast<uint64_t>(t.shape[sl.dim]), w = static_cast<uint64_t>(sl.stop - sl.start);
      o.sdim = sl.dim;
      o.start = sl.start;
      o.stop = sl.stop;
      o.shape[sl.dim] = sl.stop - sl.start;
      o.numel = outer * w * inner;
      o.src0 = t.begin + static_cast<uint64_t>(sl.start) * inner * isz;
      if (outer > 1 && w < D && w * inner > 0) {
        o.runs = outer;
        o.run = w * inner * upe;
        o.pitch = D * inner * isz;
      }
    }
    o.units = o.numel * upe;
    if (o.runs == 1) o.run = o.units;
    outs->push_back(std::move(o));
  }
  if (n_parts > 1) {
    // Output i goes to part floor(n_parts * (2 c_i + b_i) / (2 T)).
    unsigned __int128 T = 0, c = 0;
    for (const Output &o : *outs) T += static_cast<unsigned __int128>(o.numel) * dtype_size(o.out_dtype);
    std::vector<Output> kept;
    for (Output &o : *outs) {
      unsigned __int128 b = static_cast<unsigned __int128>(o.numel) * dtype_size(o.out_dtype);
      uint64_t owner = 0;
      if (T > 0) {
        unsigned __int128 q = ((2 * c + b) * n_parts) / (2 * T);
        owner = q >= n_parts ? n_parts - 1 : static_cast<uint64_t>(q);
      }
      c += b;
      if (owner == part) kept.push_back(std::move(o));
    }
    outs->swap(kept);
  }
  if (outs->size() >= kMaxOutputs) return set_error(ST_E_INVAL, "at most %u outputs", kMaxOutputs - 1);
  return ST_OK;
}

struct Segment {
  uint32_t out;
  uint64_t u0, u1;
};

// A piece's cost in the balance: a fixed cost plus its bytes of traffic.
double piece_cost(const Piece &pc) {
  const uint32_t cls = pc.out_cls & ((1u << kClsBits) - 1);
  return double(kPieceCost) + double(pc.count) * pc.rows * (cls_in_size(cls) + cls_out_size(cls));
}

// Cuts `segs` (in source order) into n consecutive units of about equal cost
// (`total` = the segments' cost): appends the units' pieces to *units and the
// n + 1 unit boundaries to *ub.  Cuts inside an output fall on multiples of
// kSplitBytes source bytes, and each cut adds one piece's fixed cost.
void cut_units(const st_plan_s &p, const std::vector<Segment> &segs, uint64_t n, double total,
               std::vector<Piece> *units, std::vector<uint32_t> *ub) {
  const Core &core = *p.index->core;
  units->clear();
  ub->assign(n + 1, 0);
  const double share = (total + double(n - 1) * kPieceCost) / n;
  uint64_t w = 0;
  double used = 0;  // cost assigned so far (units < w and unit w's part)
  // Output units [a, b) as pieces: one contiguous piece per kMaxPieceUnits,
  // or, across the runs of a sliced output, a partial first run, one
  // multi-row piece for the whole runs, and a partial last run.
  auto emit = [&](const Segment &s, uint64_t a, uint64_t b) {
    const Output &o = p.outs[s.out];
    const uint64_t so = cls_out_size(o.cls);
    const uint64_t scale = o.scale >= 0 ? core.tensors[o.scale].begin : kNoScale;
    auto push = [&](uint64_t u, uint64_t count, uint64_t rows) {
      Piece pc;
      pc.src = o.unit_src(u);
      pc.dst = u * so;
      pc.scale = scale;
      pc.count = static_cast<uint32_t>(count);
      pc.out_cls = (s.out << kClsBits) | o.cls;
      pc.rows = static_cast<uint32_t>(rows);
      pc.pad = 0;
      pc.pitch = o.pitch;
      units->push_back(pc);
    };
    auto contiguous = [&](uint64_t x, uint64_t y) {  // [x, y) inside one run
      for (; x < y; x += kMaxPieceUnits) push(x, std::min(y, x + kMaxPieceUnits) - x, 1);
    };
    if (o.runs == 1) {
      contiguous(a, b);
      return;
    }
    const uint64_t L = o.run;
    if (a % L) {
      const uint64_t e = std::min(b, (a / L + 1) * L);
      contiguous(a, e);
      a = e;
    }
    if (b - a >= L && L <= kMaxPieceUnits) {
      uint64_t rows = (b - a) / L;
      while (rows) {
        const uint64_t k = std::min<uint64_t>(rows, 0xFFFFFFFFu);
        push(a, L, k);
        a += k * L;
        rows -= k;
      }
    }
    while (b - a >= L) {  // runs too long for one piece each
      contiguous(a, a + L);
      a += L;
    }
    if (a < b) contiguous(a, b);
  };
  auto next_unit = [&]() {
    ++w;
    (*ub)[w] = static_cast<uint32_t>(units->size());
  };
  for (const Segment &s : segs) {
    const Output &o = p.outs[s.out];
    const double per = cls_in_size(o.cls) + cls_out_size(o.cls);
    // Cuts fall on 2 KiB of source, or between runs when the runs of a sliced
    // output are short enough to keep whole.
    const uint64_t granule = o.runs > 1 && double(o.run) * per <= double(p.unit_bytes)
                                 ? o.run
                                 : kSplitBytes / cls_in_size(o.cls);
    uint64_t u = s.u0;
    while (u < s.u1) {
      double rest = kPieceCost + double(s.u1 - u) * per;
      double room = (w + 1) * share - used;
      if (w + 1 == n || rest <= room + 0.5 * kPieceCost) {
        emit(s, u, s.u1);
        used += rest;
        u = s.u1;
        if (w + 1 < n && used >= (w + 1) * share) next_unit();
        break;
      }
      // Fill the rest of unit w with a prefix that ends on a split boundary.
      double take = std::floor((room - kPieceCost) / per);
      uint64_t cut = take > 0 ? u + static_cast<uint64_t>(take) : u;
      cut -= cut % granule;
      if (cut > u) {
        emit(s, u, cut);
        used += kPieceCost + double(cut - u) * per;
        u = cut;
      }
      // Boundaries are absolute, so the slack this cut left rolls over to
      // the next unit instead of piling up on the last one.
      next_unit();
    }
  }
  while (w < n) next_unit();
}

// Builds pieces and per-chunk worker partitions.
// Appends a one-run piece cut into pieces of at most `bytes` source bytes
// (at least one element each), in order.
void split_piece(const Piece &pc, uint64_t bytes, std::vector<Piece> *out) {
  const uint32_t cls = pc.out_cls & ((1u << kClsBits) - 1);
  const uint64_t si = cls_in_size(cls), so = cls_out_size(cls);
  const uint32_t step = static_cast<uint32_t>(std::max<uint64_t>(1, bytes / si));
  for (uint32_t e = 0; e < pc.count; e += std::min(step, pc.count - e)) {
    Piece x = pc;
    x.count = std::min(step, pc.count - e);
    x.src = pc.src + e * si;
    x.dst = pc.dst + e * so;
    out->push_back(x);
  }
}

void build_pieces(st_plan_s *p) {
  const Core &core = *p->index->core;
  const uint64_t C = p->chunk_bytes;
  const uint64_t data = core.data_bytes;
  p->n_chunks = C ? static_cast<uint32_t>(std::max<uint64_t>(1, (data + C - 1) / C)) : 1;
  std::vector<std::vector<Segment>> per_chunk(p->n_chunks);
  // Outputs in source order.
  std::vector<uint32_t> order(p->outs.size());
  for (uint32_t i = 0; i < order.size(); ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](uint32_t a, uint32_t b) {
    return p->outs[a].src0 < p->outs[b].src0;
  });
  for (uint32_t oi : order) {
    const Output &o = p->outs[oi];
    if (o.units == 0) continue;
    const uint64_t si = cls_in_size(o.cls);
    if (!C) {
      per_chunk[0].push_back({oi, 0, o.units});
      continue;
    }
    uint64_t scale_chunk = o.scale >= 0 ? (core.tensors[o.scale].end - 1) / C : 0;
    if (o.qkind != ST_QUANT_NONE) {  // all of the block scales (and the global scale) staged first
      const Tensor &qs = core.tensors[o.qscale_entry];
      if (qs.end > qs.begin) scale_chunk = std::max(scale_chunk, (qs.end - 1) / C);
      if (o.quant.scale2 != kNoScale) scale_chunk = std::max(scale_chunk, (o.quant.scale2 + 3) / C);
    }
    if (o.runs > 1) {
      // Whole runs go to the chunk holding their last byte.
      uint64_t r0 = 0, k0 = 0;
      for (uint64_t r = 0; r <= o.runs; ++r) {
        const uint64_t k = r < o.runs ? std::max(scale_chunk, (o.src0 + r * o.pitch + o.run * si - 1) / C) : ~0ull;
        if (r > 0 && k != k0) {
          per_chunk[k0].push_back({oi, r0 * o.run, r * o.run});
          r0 = r;
        }
        k0 = k;
      }
      continue;
    }
    uint64_t u = 0;
    for (uint64_t k = o.src0 / C; u < o.units; ++k) {
      // units whose last byte lies before the end of chunk k
      uint64_t end = (k + 1) * C;
      uint64_t ue = end <= o.src0 ? 0 : std::min<uint64_t>(o.units, (end - o.src0) / si);
      if (ue > u) {
        per_chunk[std::max<uint64_t>(k, scale_chunk)].push_back({oi, u, ue});
        u = ue;
      }
    }
  }
  const uint32_t W = p->workers;
  p->pieces.clear();
  p->parts.assign(static_cast<size_t>(p->n_chunks) * (W + 1), 0);
  p->claim_end.assign(p->n_chunks, 0);
  std::vector<Piece> units;
  std::vector<uint32_t> ub;
  for (uint32_t k = 0; k < p->n_chunks; ++k) {
    auto &segs = per_chunk[k];
    // Class-major source order (default): all warps then run the same
    // conversion class at the same time, which keeps the instruction working
    // set small when many small tensors of mixed dtypes interleave (measured
    // on 100k mixed tensors: 65 % -> 76 % of the HBM copy peak).  Plain
    // source order on request.
    const bool by_class = p->class_major;
    std::stable_sort(segs.begin(), segs.end(), [&](const Segment &a, const Segment &b) {
      const Output &oa = p->outs[a.out], &ob = p->outs[b.out];
      if (by_class && oa.cls != ob.cls) return oa.cls < ob.cls;
      return oa.unit_src(a.u0) < ob.unit_src(b.u0);
    });
    double total = 0;
    for (const Segment &s : segs) {
      const Output &o = p->outs[s.out];
      total += kPieceCost + double(s.u1 - s.u0) * (cls_in_size(o.cls) + cls_out_size(o.cls));
    }
    // The chunk is cut, in source order, into N = rounds * W units of equal
    // cost; unit j goes to warp j mod W.  All warps then work through
    // neighbouring units at the same time, so the GPU's accesses at any moment
    // fall in one compact window of the data section (better DRAM row
    // locality than W independent streams), and each warp's share stays
    // within one unit of the mean.
    const uint64_t rounds = std::max<uint64_t>(1, static_cast<uint64_t>(std::llround(total / (double(W) * p->unit_bytes))));
    const uint64_t N = rounds * W;
    cut_units(*p, segs, N, total, &units, &ub);
    uint32_t *parts = &p->parts[static_cast<size_t>(k) * (W + 1)];
    // The last rounds' units are claimed while the kernel runs (in source
    // order, by whichever warps are free) instead of dealt: with fixed
    // shares the warps' finishing times spread by where they run more than
    // by their shares (measured on 100k tiny tensors: blocks' mean end times
    // 155-179 us, the last warp 14 % after the median, each warp's end time
    // repeatable to 0.5 us).
    const uint64_t pct = p->kernel == kKernelTmaWide ? kClaimedPctWide
                         : is_tma_build(p->kernel)   ? kClaimedPct
                         : p->kernel == kKernelStream ? (p->long_runs ? kClaimedPctStream : kClaimedPctStreamShort)
                                                      : 0;
    // The own units are whole rounds up to where the units' cumulative cost
    // reaches (100 - pct) % of the chunk's cost (rounded to the nearest round,
    // leaving at least one round to claim): units are not always filled
    // evenly (a unit below the 2 KiB cut granule takes more than its share,
    // and the last rounds can then be empty), so the tail is found by cost,
    // not by counting rounds.
    uint64_t Ns = N;
    if (rounds >= 2 && pct) {
      const double keep = total * double(100 - pct) / 100.0;
      double acc = 0;
      uint64_t j = 0;
      for (; j < N; ++j) {
        for (uint32_t q = ub[j]; q < ub[j + 1]; ++q) acc += piece_cost(units[q]);
        if (acc >= keep) break;
      }
      Ns = std::min<uint64_t>(rounds - 1, (j + W / 2) / W) * W;
    }
    for (uint32_t w = 0; w < W; ++w) {
      parts[w] = static_cast<uint32_t>(p->pieces.size());
      for (uint64_t j = w; j < Ns; j += W) p->pieces.insert(p->pieces.end(), units.begin() + ub[j], units.begin() + ub[j + 1]);
    }
    parts[W] = static_cast<uint32_t>(p->pieces.size());
    for (size_t q = ub[Ns]; q < ub[N]; ++q) {
      const Piece &pc = units[q];
      if (p->kernel != kKernelTma || pc.rows != 1) {
        p->pieces.push_back(pc);
        continue;
      }
      split_piece(pc, kTmaTailPieceBytes, &p->pieces);
    }
    p->claim_end[k] = static_cast<uint32_t>(p->pieces.size());
  }
}

// The data-section bytes a plan's outputs read: each output's source extent
// (its runs from the first to the last), its per-tensor scale, its block
// scales and global scale; sorted, and merged across gaps under 64 KiB.
void compute_ranges(st_plan_s *p) {
  const Core &core = *p->index->core;
  std::vector<std::pair<uint64_t, uint64_t>> r;
  r.reserve(p->outs.size() * 2);
  auto whole = [&](int64_t entry) {
    if (entry >= 0) r.push_back({core.tensors[entry].begin, core.tensors[entry].end});
  };
  for (const Output &o : p->outs) {
    if (o.units == 0) continue;
    const uint64_t si = cls_in_size(o.cls);
    r.push_back({o.src0, o.src0 + (o.runs - 1) * o.pitch + (o.runs > 1 ? o.run : o.units) * si});
    whole(o.scale);
    if (o.qkind != ST_QUANT_NONE) {
      whole(o.qscale_entry);
      if (o.quant.scale2 != kNoScale) r.push_back({o.quant.scale2, o.quant.scale2 + 4});
    }
  }
  std::sort(r.begin(), r.end());
  constexpr uint64_t kGap = 65536;
  p->ranges.clear();
  uint64_t covered = 0;
  for (const auto &x : r) {
    if (!p->ranges.empty() && x.first <= p->ranges.back().second + kGap)
      p->ranges.back().second = std::max(p->ranges.back().second, x.second);
    else
      p->ranges.push_back(x);
  }
  for (const auto &x : p->ranges) covered += x.second - x.first;
  p->sparse = covered < core.data_bytes / 4 * 3;
  p->pf_lo = p->pf_hi = 0;
  if (!p->ranges.empty()) {
    const uint64_t lo = p->ranges.front().first, hi = p->ranges.back().second;
    if (hi - lo <= kPrefetchMaxBytes && covered * 2 >= hi - lo) {
      p->pf_lo = lo;
      p->pf_hi = hi;
    }
  }
}

// Calls fn(lo, hi) for the plan's read ranges within [off, off + n): all of
// it when the plan is not sparse.
template <class F>
st_status for_each_range(const st_plan_s *p, uint64_t off, uint64_t n, F fn) {
  if (!n) return ST_OK;
  if (!p->sparse) return fn(off, off + n);
  auto it = std::lower_bound(p->ranges.begin(), p->ranges.end(), std::make_pair(off, uint64_t(0)),
                             [](const std::pair<uint64_t, uint64_t> &a, const std::pair<uint64_t, uint64_t> &b) {
                               return a.second <= b.first;
                             });
  for (; it != p->ranges.end() && it->first < off + n; ++it) {
    const uint64_t lo = std::max(off, it->first), hi = std::min(off + n, it->second);
    if (lo < hi) {
      const st_status s = fn(lo, hi);
      if (s != ST_OK) return s;
    }
  }
  return ST_OK;
}

// Selection, kernel build, warps and pieces of a plan (host side only).
st_status plan_host(std::shared_ptr<const IndexData> index, const st_selection *sel, st_dtype dst_dtype,
                    const st_plan_options *opts, st_plan_s *p) {
  p->index = std::move(index);
  st_status s = select_outputs(*p->index, sel, dst_dtype, &p->outs);
  if (s != ST_OK) return s;
  const bool host_only = opts && opts->host_only;
  uint32_t workers = opts ? opts->workers : 0;
  p->chunk_bytes = opts ? opts->chunk_bytes : 0;
  if (opts && opts->unit_bytes) p->unit_bytes = opts->unit_bytes;
  const uint32_t order = opts ? opts->order : 0;
  if (order > 2) return set_error(ST_E_INVAL, "options.order must be 0, 1 or 2");
  uint64_t cost = 0, traffic = 0, nonempty = 0;
  for (const Output &o : p->outs) {
    const uint64_t t = o.units * (cls_in_size(o.cls) + cls_out_size(o.cls));
    cost += kPieceCost + t;
    traffic += t;
    nonempty += t > 0;
  }
  // Many small tensors: the TMA build (reads staged in shared memory, so a
  // warp keeps kilobytes in flight whatever the tensor size); else the
  // streaming build.
  if (opts && opts->kernel) {
    if (opts->kernel < kKernelStream || opts->kernel > kKernelTmaWide)
      return set_error(ST_E_INVAL, "options.kernel must be 0 .. 4");
    p->kernel = opts->kernel;
  } else {
    p->kernel = nonempty && traffic / nonempty < kSmallOutputBytes ? kKernelTma : kKernelStream;
  }
  // Block-scaled outputs are only in the TMA builds (the wide one by default).
  bool has_quant = false;
  for (const Output &o : p->outs) has_quant = has_quant || o.qkind != ST_QUANT_NONE;
  if (has_quant) {
    if (opts && opts->kernel && opts->kernel != kKernelTma && opts->kernel != kKernelTmaWide)
      return set_error(ST_E_INVAL, "block-scaled outputs need a TMA build (options.kernel 0, 3 or 4)");
    if (!(opts && opts->kernel)) p->kernel = kKernelTmaWide;
  }
  if (!(opts && opts->unit_bytes) && p->kernel == kKernelTma) p->unit_bytes = kTmaUnitBytes;
  // Unit order: the register builds run one class at a time (their
  // per-class code is large, and mixing classes stalls on instruction
  // fetch); the TMA build's code is small, and source order keeps DRAM
  // rows local.
  p->class_major = order == 2 || (order == 0 && !is_tma_build(p->kernel));
  {
    uint64_t runs = 0;
    for (const Output &o : p->outs) runs += o.units ? o.runs : 0;
    p->long_runs = runs && traffic / runs >= kLongRunBytes;
  }
  int sms = 0, blocks = 0;
  if (!host_only || workers == 0) {
    if (host_only) return set_error(ST_E_INVAL, "a host-only plan needs options.workers");
    s = kernel_occupancy(p->kernel, &sms, &blocks);
    if (s != ST_OK) return s;
    uint32_t bps = static_cast<uint32_t>(blocks);
    if (opts && opts->blocks_per_sm) bps = std::min(bps, opts->blocks_per_sm);
    else if (p->kernel == kKernelStream) {
      // Measured: the streaming build runs best at 2 blocks per SM (scaled FP8
      // 91.7 -> 95.6 %, 4-shard LLM 96.9 -> 98.0 % against 3); many short runs
      // (row-sliced tensor-parallel shards) did better at 3 with fixed shares
      // (0.92 against 0.90) but best at 2 with a claimed tail (0.988).
      bps = std::min(bps, kStreamBlocksPerSm);
    }
    if (workers == 0) workers = static_cast<uint32_t>(sms) * bps * kWarpsPerBlock;
  }
  // No more warps than the work can use.
  uint64_t cap = std::max<uint64_t>(1, cost / kMinWorkerCost);
  p->workers = static_cast<uint32_t>(std::min<uint64_t>(workers, cap));
  build_pieces(p);
  compute_ranges(p);
  if (has_quant) {
    p->quant.resize(p->outs.size());
    for (size_t i = 0; i < p->outs.size(); ++i) p->quant[i] = p->outs[i].quant;
  }
  return ST_OK;
}

}  // namespace

extern "C" {

st_status st_plan(const st_index_t *index, const st_selection *sel, st_dtype dst_dtype,
                  const st_plan_options *opts, st_plan_t **out) {
  if (!index || !out) return set_error(ST_E_INVAL, "NULL argument");
  *out = nullptr;
  try {
    auto p = std::make_unique<st_plan_s>();
    st_status s = plan_host(index_ref(index), sel, dst_dtype, opts, p.get());
    if (s != ST_OK) return s;
    const bool host_only = opts && opts->host_only;
    if (!host_only) {
      cudaError_t e = cudaGetDevice(&p->device);
      size_t pb = p->pieces.size() * sizeof(Piece), qb = p->parts.size() * sizeof(uint32_t);
      if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void **>(&p->d_pieces), std::max<size_t>(pb, sizeof(Piece)));
      if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void **>(&p->d_parts), qb);
      if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void **>(&p->d_err), sizeof(uint32_t));
      if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void **>(&p->d_claim), 2 * sizeof(uint32_t));
      p->on_device = true;  // from here the destructor releases what was made
      if (e == cudaSuccess && pb) e = cudaMemcpy(p->d_pieces, p->pieces.data(), pb, cudaMemcpyHostToDevice);
      if (e == cudaSuccess) e = cudaMemcpy(p->d_parts, p->parts.data(), qb, cudaMemcpyHostToDevice);
      if (e == cudaSuccess) e = cudaMemset(p->d_err, 0, sizeof(uint32_t));
      if (e == cudaSuccess) e = cudaMemset(p->d_claim, 0, 2 * sizeof(uint32_t));
      if (e == cudaSuccess && !p->quant.empty()) {
        const size_t bytes = p->quant.size() * sizeof(QuantInfo);
        e = cudaMalloc(reinterpret_cast<void **>(&p->d_quant), bytes);
        if (e == cudaSuccess) e = cudaMemcpy(p->d_quant, p->quant.data(), bytes, cudaMemcpyHostToDevice);
      }
      for (uint32_t k = 0; e == cudaSuccess && k <= p->n_chunks; ++k) {
        cudaEvent_t ev;
        e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        if (e == cudaSuccess) p->events.push_back(ev);
      }
      if (e != cudaSuccess)
        return set_error(ST_E_CUDA, "uploading the plan (%zu pieces): %s", p->pieces.size(), cuda_msg(e).c_str());
    }
    *out = p.release();
    return ST_OK;
  } catch (const std::bad_alloc &) {
    return set_error(ST_E_NOMEM, "out of host memory while planning");
  }
}

void st_plan_free(st_plan_t *plan) { delete plan; }

st_status st_plan_count(const st_plan_t *p, size_t *count) {
  if (!p || !count) return set_error(ST_E_INVAL, "NULL argument");
  *count = p->outs.size();
  return ST_OK;
}

st_status st_plan_output(const st_plan_t *p, size_t i, st_output_info *info) {
  if (!p || !info) return set_error(ST_E_INVAL, "NULL argument");
  if (i >= p->outs.size()) return set_error(ST_E_INVAL, "output %zu out of range", i);
  const Output &o = p->outs[i];
  const Tensor &t = p->index->core->tensors[o.entry];
  info->name = o.name.c_str();
  info->dtype = static_cast<st_dtype>(o.out_dtype);
  info->src_dtype = static_cast<st_dtype>(t.dtype);
  info->ndim = static_cast<int32_t>(o.shape.size());
  info->shape = o.shape.data();
  info->numel = o.numel;
  info->bytes = o.numel * dtype_size(o.out_dtype);
  info->src_begin = t.begin;
  const int64_t sc = o.qkind != ST_QUANT_NONE ? o.qscale_entry : o.scale;
  info->scale_name = sc >= 0 ? p->index->core->tensors[sc].name.c_str() : nullptr;
  info->slice_dim = o.sdim;
  info->slice_start = o.start;
  info->slice_stop = o.stop;
  info->quant_kind = o.qkind;
  return ST_OK;
}

st_status st_plan_arena(const st_plan_t *p, uint64_t align, uint64_t *offsets, uint64_t *total) {
  if (!p || (!offsets && !p->outs.empty()) || !total) return set_error(ST_E_INVAL, "NULL argument");
  if (align < 16 || (align & (align - 1))) return set_error(ST_E_INVAL, "alignment %llu is not a power of two >= 16",
                                                            (unsigned long long)align);
  uint64_t at = 0;
  for (size_t i = 0; i < p->outs.size(); ++i) {
    at = (at + align - 1) & ~(align - 1);
    offsets[i] = at;
    at += p->outs[i].numel * dtype_size(p->outs[i].out_dtype);
  }
  *total = at;
  return ST_OK;
}

st_status st_plan_copy_bytes(const st_plan_t *p, uint64_t *bytes, uint32_t *ranges) {
  if (!p || !bytes) return set_error(ST_E_INVAL, "NULL argument");
  if (!p->sparse) {
    *bytes = p->index->core->data_bytes;
    if (ranges) *ranges = 1;
    return ST_OK;
  }
  uint64_t b = 0;
  for (const auto &x : p->ranges) b += x.second - x.first;
  *bytes = b;
  if (ranges) *ranges = static_cast<uint32_t>(p->ranges.size());
  return ST_OK;
}

st_status st_class_step(uint32_t cls, uint32_t *src_item, uint32_t *out_item, uint32_t *step_src,
                        uint32_t *step_units, uint32_t *step_out) {
  if (cls >= CLS_COUNT) return set_error(ST_E_INVAL, "class %u of %u", cls, static_cast<uint32_t>(CLS_COUNT));
  if (src_item) *src_item = static_cast<uint32_t>(cls_in_size(cls));
  if (out_item) *out_item = static_cast<uint32_t>(cls_out_size(cls));
  if (step_src) *step_src = cls_step_src(cls);
  if (step_units) *step_units = cls_step_units(cls);
  if (step_out) *step_out = cls_step_out(cls);
  return ST_OK;
}

st_status st_plan_copy_range(const st_plan_t *p, uint32_t i, uint64_t *begin, uint64_t *end) {
  if (!p || !begin || !end) return set_error(ST_E_INVAL, "NULL argument");
  const size_t n = p->sparse ? p->ranges.size() : 1;
  if (i >= n) return set_error(ST_E_INVAL, "copy range %u of %zu", i, n);
  *begin = p->sparse ? p->ranges[i].first : 0;
  *end = p->sparse ? p->ranges[i].second : p->index->core->data_bytes;
  return ST_OK;
}

st_status st_plan_stats(const st_plan_t *p, uint32_t *workers, uint32_t *chunks, uint64_t *pieces,
                        uint32_t *kernel) {
  if (!p) return set_error(ST_E_INVAL, "NULL plan");
  if (kernel) *kernel = p->kernel;
  if (workers) *workers = p->workers;
  if (chunks) *chunks = p->n_chunks;
  if (pieces) *pieces = p->pieces.size();
  return ST_OK;
}

st_status st_plan_piece(const st_plan_t *p, uint64_t k, uint64_t *src, uint64_t *dst, uint64_t *scale,
                        uint32_t *count, uint32_t *output, uint32_t *cls, uint32_t *rows, uint64_t *pitch) {
  if (!p || !src || !dst || !scale || !count || !output || !cls || !rows || !pitch)
    return set_error(ST_E_INVAL, "NULL argument");
  if (k >= p->pieces.size()) return set_error(ST_E_INVAL, "piece %llu out of range", (unsigned long long)k);
  const Piece &pc = p->pieces[k];
  *src = pc.src;
  *dst = pc.dst;
  *scale = pc.scale;
  *count = pc.count;
  *output = pc.out_cls >> kClsBits;
  *cls = pc.out_cls & ((1u << kClsBits) - 1);
  *rows = pc.rows;
  *pitch = pc.pitch;
  return ST_OK;
}

st_status st_plan_worker(const st_plan_t *p, uint32_t chunk, uint32_t w, uint64_t *first, uint64_t *last) {
  if (!p || !first || !last) return set_error(ST_E_INVAL, "NULL argument");
  if (chunk >= p->n_chunks || w > p->workers) return set_error(ST_E_INVAL, "chunk/worker out of range");
  const uint32_t *parts = &p->parts[static_cast<size_t>(chunk) * (p->workers + 1)];
  *first = parts[w];
  *last = w < p->workers ? parts[w + 1] : p->claim_end[chunk];
  return ST_OK;
}

}  // extern "C"

namespace {

st_status check_device_plan(const st_plan_t *p) {
  if (!p->on_device) return set_error(ST_E_INVAL, "the plan was built host-only");
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return set_error(ST_E_CUDA, "cudaGetDevice: %s", cuda_msg(e).c_str());
  if (cur != p->device) return set_error(ST_E_INVAL, "the plan belongs to device %d, device %d is current", p->device, cur);
  return ST_OK;
}

// The TMA build's bulk copies read the data section: it must be device (or
// managed) memory.
st_status check_tma_source(const st_plan_t *p, const void *data_dev) {
  if ((p->kernel != kKernelTma && p->kernel != kKernelTmaWide) || !data_dev) return ST_OK;
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, data_dev);
  if (e != cudaSuccess) return set_error(ST_E_CUDA, "cudaPointerGetAttributes: %s", cuda_msg(e).c_str());
  if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
    return set_error(ST_E_INVAL, "the TMA build needs the data section in device or managed memory");
  return ST_OK;
}

// Whether `ptr` is device memory of the current device (the L2 prefetch of
// small plans goes through the bulk-copy engine, which is pointed only at
// this GPU's own memory).
bool on_this_device(const void *ptr) {
  cudaPointerAttributes at;
  int dev = 0;
  if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice && at.device == dev;
}

st_status launch_chunk(const st_plan_t *p, uint32_t k, const void *data_dev, void *const *dst, const float *scales,
                       void *stream) {
  if (p->pieces.empty()) return ST_OK;
  const uint32_t *parts = &p->parts[static_cast<size_t>(k) * (p->workers + 1)];
  if (parts[0] == p->claim_end[k]) return ST_OK;  // nothing in this chunk
  LaunchArgs a;
  a.data = static_cast<const uint8_t *>(data_dev);
  a.data_bytes = p->index->core->data_bytes;
  a.pieces = p->d_pieces;
  a.parts = p->d_parts + static_cast<size_t>(k) * (p->workers + 1);
  a.workers = p->workers;
  a.dst = dst;
  a.scales = scales;
  a.err = p->d_err;
  a.quant = p->d_quant;
  a.claim_end = p->claim_end[k];
  a.claim = p->d_claim;
  if (p->n_chunks == 1 && p->pf_hi > p->pf_lo && on_this_device(data_dev) && on_this_device(dst)) {
    a.pf_table = p->d_pieces + parts[0];
    a.pf_table_bytes = static_cast<uint32_t>((p->claim_end[k] - parts[0]) * sizeof(Piece));
    a.pf_dst_bytes = static_cast<uint32_t>(p->outs.size() * sizeof(void *));
    a.pf_data_off = p->pf_lo;
    a.pf_data_bytes = p->pf_hi - p->pf_lo;
  }
  return launch_materialize(a, p->kernel, stream);
}

// A page-locked mirror of the static array, one per device, allocated on first
// use: st_load_tensors packs its tables there and uploads them in one
// asynchronous copy (a copy from pageable memory first waits for the stream,
// which would hold each lazy call until the previous call's kernel is done).
// Two halves used in turn, each reused once the event recorded after its
// last copy has completed: a call then waits for the call before the
// previous one, not for the previous one's staging copy.  (The device array
// itself is single: its reuse is ordered by the stream.)
struct TableMirror {
  uint8_t *host[2] = {nullptr, nullptr};
  cudaEvent_t done[2] = {nullptr, nullptr};
  uint32_t next = 0;
};
std::mutex g_mirror_mu;
std::map<int, TableMirror> g_mirrors;

// Launches a plan whose tables live in the library's static device array:
// pieces | warp ranges | block-scale table | destinations (when given on the
// host), each 256-byte aligned, filled by stream-ordered copies (with
// `mirror`, one copy from the device's page-locked mirror); the error word
// sits at the array's fixed kStaticErrOffset and is not cleared here.
st_status launch_static(const st_plan_t *p, const void *data_dev, void *const *dst_dev, void *const *dst_host,
                        const float *scales, void *stream, bool mirror = false) {
  const size_t pieces_bytes = p->pieces.size() * sizeof(Piece);
  const size_t parts_off = (pieces_bytes + 255) & ~size_t(255);
  const size_t parts_bytes = p->parts.size() * sizeof(uint32_t);
  const size_t quant_off = (parts_off + parts_bytes + 255) & ~size_t(255);
  const size_t quant_bytes = p->quant.size() * sizeof(QuantInfo);
  const size_t dst_off = (quant_off + quant_bytes + 255) & ~size_t(255);
  const size_t dst_bytes = dst_host ? p->outs.size() * sizeof(void *) : 0;
  const size_t need = dst_off + dst_bytes;
  if (need > kStaticErrOffset)
    return set_error(ST_E_INVAL,
                     "the plan needs %zu bytes of static scratch (%zu pieces, %u warps, %u chunks, %zu block-scale "
                     "records) but the library holds %zu for tables; plan with a larger unit_bytes or fewer workers",
                     need, p->pieces.size(), p->workers, p->n_chunks, p->quant.size(), kStaticErrOffset);
  void *scratch = nullptr;
  st_status s = static_scratch(&scratch);
  if (s != ST_OK) return s;
  uint8_t *base = static_cast<uint8_t *>(scratch);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  std::unique_lock<std::mutex> lock(g_mirror_mu, std::defer_lock);
  TableMirror *mp = nullptr;
  if (mirror) {  // the page-locked mirror, or (if it cannot be had) the pageable copies below
    lock.lock();
    int dev = 0;
    e = cudaGetDevice(&dev);
    TableMirror &m = g_mirrors[dev];
    if (e == cudaSuccess && !m.host[0]) {
      void *h = nullptr;
      cudaEvent_t ev[2] = {nullptr, nullptr};
      if (cudaHostAlloc(&h, 2 * kStaticScratchBytes, cudaHostAllocDefault) == cudaSuccess &&
          cudaEventCreateWithFlags(&ev[0], cudaEventDisableTiming) == cudaSuccess &&
          cudaEventCreateWithFlags(&ev[1], cudaEventDisableTiming) == cudaSuccess &&
          cudaEventRecord(ev[0], st) == cudaSuccess && cudaEventRecord(ev[1], st) == cudaSuccess) {
        for (int k = 0; k < 2; ++k) {
          m.host[k] = static_cast<uint8_t *>(h) + k * kStaticScratchBytes;
          m.done[k] = ev[k];
        }
      } else {
        for (cudaEvent_t x : ev)
          if (x) cudaEventDestroy(x);
        if (h) cudaFreeHost(h);
        (void)cudaGetLastError();  // not sticky: fall back to pageable copies
      }
    }
    if (e == cudaSuccess && m.host[0]) mp = &m;
  }
  if (mp) {
    TableMirror &m = *mp;
    const uint32_t k = m.next;
    m.next ^= 1u;
    uint8_t *h = m.host[k];
    e = cudaEventSynchronize(m.done[k]);  // this half's last copy has left it
    if (e == cudaSuccess) {
      std::memcpy(h, p->pieces.data(), pieces_bytes);
      std::memcpy(h + parts_off, p->parts.data(), parts_bytes);
      if (quant_bytes) std::memcpy(h + quant_off, p->quant.data(), quant_bytes);
      if (dst_bytes) std::memcpy(h + dst_off, dst_host, dst_bytes);
      e = cudaMemcpyAsync(base, h, need, cudaMemcpyHostToDevice, st);
    }
    if (e == cudaSuccess) e = cudaEventRecord(m.done[k], st);
  } else if (e == cudaSuccess) {
    e = cudaMemcpyAsync(base, p->pieces.data(), pieces_bytes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(base + parts_off, p->parts.data(), parts_bytes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && quant_bytes)
      e = cudaMemcpyAsync(base + quant_off, p->quant.data(), quant_bytes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && dst_bytes) e = cudaMemcpyAsync(base + dst_off, dst_host, dst_bytes, cudaMemcpyHostToDevice, st);
  }
  if (e != cudaSuccess) return set_error(ST_E_CUDA, "filling the static scratch: %s", cuda_msg(e).c_str());
  for (uint32_t k = 0; k < p->n_chunks; ++k) {
    const uint32_t *parts = &p->parts[static_cast<size_t>(k) * (p->workers + 1)];
    if (parts[0] == p->claim_end[k]) continue;
    LaunchArgs a;
    a.data = static_cast<const uint8_t *>(data_dev);
    a.data_bytes = p->index->core->data_bytes;
    a.pieces = reinterpret_cast<const Piece *>(base);
    a.parts = reinterpret_cast<const uint32_t *>(base + parts_off) + static_cast<size_t>(k) * (p->workers + 1);
    a.workers = p->workers;
    a.dst = dst_host ? reinterpret_cast<void *const *>(base + dst_off) : dst_dev;
    a.scales = scales;
    a.err = reinterpret_cast<uint32_t *>(base + kStaticErrOffset);
    a.claim_end = p->claim_end[k];
    a.claim = reinterpret_cast<uint32_t *>(base + kStaticClaimOffset);
    a.quant = quant_bytes ? reinterpret_cast<const QuantInfo *>(base + quant_off) : nullptr;
    s = launch_materialize(a, p->kernel, stream);
    if (s != ST_OK) return s;
  }
  return ST_OK;
}

}  // namespace

extern "C" {

st_status st_materialize(const void *data_dev, const st_plan_t *p, void *const *dst_ptrs, const float *scales,
                         void *stream) {
  if (!p) return set_error(ST_E_INVAL, "NULL plan");
  st_status s = check_device_plan(p);
  if (s != ST_OK) return s;
  if (p->pieces.empty()) return ST_OK;
  if (!data_dev || !dst_ptrs) return set_error(ST_E_INVAL, "NULL data or destination array");
  s = check_tma_source(p, data_dev);
  if (s != ST_OK) return s;
  for (uint32_t k = 0; k < p->n_chunks; ++k) {
    s = launch_chunk(p, k, data_dev, dst_ptrs, scales, stream);
    if (s != ST_OK) return s;
  }
  return ST_OK;
}

st_status st_stage_h2d(void *dst_dev, const void *src_host, uint64_t bytes, uint64_t chunk_bytes, void *stream,
                       void *done_event) {
  if (bytes && (!dst_dev || !src_host)) return set_error(ST_E_INVAL, "NULL pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint64_t step = chunk_bytes ? chunk_bytes : bytes;
  for (uint64_t off = 0; off < bytes; off += step) {
    uint64_t n = std::min(step, bytes - off);
    cudaError_t e = cudaMemcpyAsync(static_cast<uint8_t *>(dst_dev) + off, static_cast<const uint8_t *>(src_host) + off,
                                    n, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess)
      return set_error(ST_E_CUDA, "copy of %llu bytes at %llu: %s", (unsigned long long)n, (unsigned long long)off,
                       cuda_msg(e).c_str());
  }
  if (done_event) {
    cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(done_event), st);
    if (e != cudaSuccess) return set_error(ST_E_CUDA, "cudaEventRecord: %s", cuda_msg(e).c_str());
  }
  return ST_OK;
}

st_status st_load(const void *data_host, void *data_dev, const st_plan_t *p, void *const *dst_ptrs,
                  const float *scales, void *copy_stream, void *compute_stream) {
  if (!p) return set_error(ST_E_INVAL, "NULL plan");
  st_status s = check_device_plan(p);
  if (s != ST_OK) return s;
  const uint64_t data = p->index->core->data_bytes;
  if ((data && (!data_host || !data_dev)) || !dst_ptrs) return set_error(ST_E_INVAL, "NULL pointer");
  s = check_tma_source(p, data_dev);
  if (s != ST_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(copy_stream), ks = static_cast<cudaStream_t>(compute_stream);
  // The copies overwrite data_dev: order them after work already on the compute stream.
  cudaEvent_t start = p->events[p->n_chunks];
  cudaError_t e = cudaEventRecord(start, ks);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, start, 0);
  if (e != cudaSuccess) return set_error(ST_E_CUDA, "ordering the copy stream: %s", cuda_msg(e).c_str());
  const uint64_t C = p->chunk_bytes ? p->chunk_bytes : (data ? data : 1);
  for (uint32_t k = 0; k < p->n_chunks; ++k) {
    uint64_t off = static_cast<uint64_t>(k) * C;
    uint64_t n = off < data ? std::min(C, data - off) : 0;
    // The whole chunk, or (sparse plan) only the byte ranges the plan reads.
    s = for_each_range(p, off, n, [&](uint64_t lo, uint64_t hi) -> st_status {
      const cudaError_t ce = cudaMemcpyAsync(static_cast<uint8_t *>(data_dev) + lo,
                                             static_cast<const uint8_t *>(data_host) + lo, hi - lo,
                                             cudaMemcpyHostToDevice, cs);
      if (ce != cudaSuccess)
        return set_error(ST_E_CUDA, "copy of chunk %u (%llu bytes): %s", k, (unsigned long long)(hi - lo),
                         cuda_msg(ce).c_str());
      return ST_OK;
    });
    if (s != ST_OK) return s;
    e = cudaEventRecord(p->events[k], cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ks, p->events[k], 0);
    if (e != cudaSuccess) return set_error(ST_E_CUDA, "chunk %u event: %s", k, cuda_msg(e).c_str());
    s = launch_chunk(p, k, data_dev, dst_ptrs, scales, compute_stream);
    if (s != ST_OK) return s;
  }
  return ST_OK;
}

st_status st_load_files(const st_files_t *files, void *data_dev, const st_plan_t *p, void *const *dst_ptrs,
                        const float *scales, void *ring_host, uint64_t ring_bytes, uint32_t threads,
                        void *copy_stream, void *compute_stream) {
  if (!p || !files) return set_error(ST_E_INVAL, "NULL plan or files");
  st_status s = check_device_plan(p);
  if (s != ST_OK) return s;
  const uint64_t data = p->index->core->data_bytes;
  if (files_arena_bytes(files) != data)
    return set_error(ST_E_INVAL, "the files' arena (%llu bytes) is not the plan's data section (%llu bytes)",
                     (unsigned long long)files_arena_bytes(files), (unsigned long long)data);
  // No ring: every chunk is copied straight from the files' mappings.
  const bool direct = !ring_host && ring_bytes == 0;
  if ((data && (!data_dev || (!ring_host && !direct))) || !dst_ptrs) return set_error(ST_E_INVAL, "NULL pointer");
  s = check_tma_source(p, data_dev);
  if (s != ST_OK) return s;
  const uint64_t C = p->chunk_bytes ? p->chunk_bytes : (data ? data : 1);
  const uint64_t slots = direct ? 0 : ring_bytes / C;
  if (data && !direct && slots == 0)
    return set_error(ST_E_INVAL, "the ring (%llu bytes) holds no %llu-byte chunk", (unsigned long long)ring_bytes,
                     (unsigned long long)C);
  cudaStream_t cs = static_cast<cudaStream_t>(copy_stream), ks = static_cast<cudaStream_t>(compute_stream);
  cudaEvent_t start = p->events[p->n_chunks];
  cudaError_t e = cudaEventRecord(start, ks);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, start, 0);
  if (e != cudaSuccess) return set_error(ST_E_CUDA, "ordering the copy stream: %s", cuda_msg(e).c_str());
  uint8_t *ring = static_cast<uint8_t *>(ring_host);
  // Ring-less: one populate thread faults each chunk's pages in ahead of its
  // copy (the copy engine then finds them in the page tables), and a page that
  // cannot be read ends the load before its copy is queued.  Measured on a
  // Grace-attached GPU from the page cache: first loads (fresh mappings) 31 ->
  // 187 GB/s with it; four threads instead of one lose 5-20 % to contention
  // with the copies.
  struct PopGuard {
    Populator *p = nullptr;
    ~PopGuard() { populate_stop(p); }
  } pop;
  if (direct && data && !p->sparse) {  // a sparse plan faults in each range it copies, right before the copy
    pop.p = populate_start(files, 0, data, C, 1);
    if (!pop.p) return set_error(ST_E_NOMEM, "starting the populate threads");
  }
  for (uint32_t k = 0; k < p->n_chunks; ++k) {
    const uint64_t off = static_cast<uint64_t>(k) * C;
    const uint64_t n = off < data ? std::min(C, data - off) : 0;
    if (direct) {
      // On an error the copies already queued still read the mappings: wait
      // for them, so that closing the files afterwards is safe.
      if (n && pop.p) s = populate_wait(pop.p, k);
      if (s == ST_OK)
        s = for_each_range(p, off, n, [&](uint64_t lo, uint64_t hi) -> st_status {
          st_status r = pop.p ? ST_OK : st_files_prefetch(files, lo, hi - lo, 0);
          if (r == ST_OK) r = copy_arena_direct(files, lo, hi - lo, static_cast<uint8_t *>(data_dev) + lo, cs);
          return r;
        });
      if (s == ST_OK) {
        e = cudaEventRecord(p->events[k], cs);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(ks, p->events[k], 0);
        if (e != cudaSuccess) s = set_error(ST_E_CUDA, "chunk %u event: %s", k, cuda_msg(e).c_str());
      }
      if (s == ST_OK) s = launch_chunk(p, k, data_dev, dst_ptrs, scales, compute_stream);
      if (s != ST_OK) {
        cudaStreamSynchronize(cs);
        return s;
      }
      continue;
    }
    uint8_t *slot = ring + (k % (slots ? slots : 1)) * C;
    if (k >= slots && slots) {  // the slot's previous copy must be done
      e = cudaEventSynchronize(p->events[k - slots]);
      if (e != cudaSuccess) return set_error(ST_E_CUDA, "waiting for chunk %llu: %s", (unsigned long long)(k - slots),
                                             cuda_msg(e).c_str());
    }
    // The whole chunk, or (sparse plan) only the byte ranges the plan reads,
    // each read into the slot at its place and copied.
    s = for_each_range(p, off, n, [&](uint64_t lo, uint64_t hi) -> st_status {
      st_status r = read_arena(files, lo, hi - lo, slot + (lo - off), threads);
      if (r != ST_OK) return r;
      const cudaError_t ce = cudaMemcpyAsync(static_cast<uint8_t *>(data_dev) + lo, slot + (lo - off), hi - lo,
                                             cudaMemcpyHostToDevice, cs);
      if (ce != cudaSuccess)
        return set_error(ST_E_CUDA, "copy of chunk %u (%llu bytes): %s", k, (unsigned long long)(hi - lo),
                         cuda_msg(ce).c_str());
      return ST_OK;
    });
    if (s != ST_OK) return s;
    e = cudaEventRecord(p->events[k], cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ks, p->events[k], 0);
    if (e != cudaSuccess) return set_error(ST_E_CUDA, "chunk %u event: %s", k, cuda_msg(e).c_str());
    s = launch_chunk(p, k, data_dev, dst_ptrs, scales, compute_stream);
    if (s != ST_OK) return s;
  }
  // The ring is free (the mappings no longer read) once the last copies finished.
  if (direct && p->n_chunks) {
    e = cudaEventSynchronize(p->events[p->n_chunks - 1]);
    if (e != cudaSuccess) return set_error(ST_E_CUDA, "waiting for the copies: %s", cuda_msg(e).c_str());
    return ST_OK;
  }
  for (uint32_t k = p->n_chunks > slots ? static_cast<uint32_t>(p->n_chunks - slots) : 0; k < p->n_chunks; ++k) {
    e = cudaEventSynchronize(p->events[k]);
    if (e != cudaSuccess) return set_error(ST_E_CUDA, "waiting for chunk %u: %s", k, cuda_msg(e).c_str());
  }
  return ST_OK;
}

st_status st_materialize_noalloc(const void *data_dev, const st_plan_t *p, void *const *dst_ptrs,
                                 const float *scales, void *stream) {
  if (!p) return set_error(ST_E_INVAL, "NULL plan");
  if (p->pieces.empty()) return ST_OK;
  if (!data_dev || !dst_ptrs) return set_error(ST_E_INVAL, "NULL data or destination array");
  st_status s = check_tma_source(p, data_dev);
  if (s != ST_OK) return s;
  return launch_static(p, data_dev, dst_ptrs, nullptr, scales, stream);
}

st_status st_load_tensors(const st_index_t *index, const st_files_t *files, st_cache_t *cache,
                          const st_selection *sel, st_dtype dst_dtype, void *const *dst_host_ptrs,
                          void *staging_dev, uint64_t staging_bytes, uint32_t threads, void *stream) {
  if (!index || !files || !sel || !sel->names) return set_error(ST_E_INVAL, "NULL argument (the selection needs names)");
  try {
    const IndexData &ix = *index_data(index);
    if (files_arena_bytes(files) != ix.core->data_bytes)
      return set_error(ST_E_INVAL, "the files' arena (%llu bytes) is not the index's data section (%llu bytes)",
                       (unsigned long long)files_arena_bytes(files), (unsigned long long)ix.core->data_bytes);
    // The outputs on the real index, and every tensor they read.
    std::vector<Output> outs;
    st_status s = select_outputs(ix, sel, dst_dtype, &outs);
    if (s != ST_OK) return s;
    if (outs.empty()) return ST_OK;
    if (!dst_host_ptrs) return set_error(ST_E_INVAL, "NULL destinations");
    std::vector<uint32_t> need;
    std::vector<char> seen(ix.ent.size(), 0);
    for (const Output &o : outs)
      for (uint32_t q : o.reads)
        if (!seen[q]) {
          seen[q] = 1;
          need.push_back(q);
        }
    // An output that is a dim-0 slice of a tensor no other output reads
    // stages only its rows (a tensor-parallel rank reads its share of the
    // file, not the whole tensor); the staged tensor is then those rows, and
    // the output reads it unsliced.
    std::vector<uint32_t> readers(ix.ent.size(), 0), need_at(ix.ent.size(), 0);
    for (const Output &o : outs)
      for (uint32_t q : o.reads) ++readers[q];
    for (size_t k = 0; k < need.size(); ++k) need_at[need[k]] = static_cast<uint32_t>(k);
    std::vector<uint64_t> sub_lo(need.size(), 0);  // staged range: source bytes [begin + sub_lo, ...)
    std::vector<int64_t> sub_rows(need.size(), -1);  // rows staged, or -1: the whole tensor
    std::vector<st_slice> slices2;                  // the selection's slices, those outputs unsliced
    if (sel->slices) {
      std::vector<int64_t> sel_of(ix.ent.size(), -1);  // view position -> selection entry
      for (size_t j = 0; j < sel->n_names; ++j) {
        auto it = ix.pos.find(std::string_view(sel->names[j]));
        if (it != ix.pos.end()) sel_of[it->second] = static_cast<int64_t>(j);
      }
      for (const Output &o : outs) {
        const uint32_t q = o.reads[0];
        const Tensor &t = ix.core->tensors[ix.ent[q]];
        if (o.sdim != 0 || o.qkind != ST_QUANT_NONE || readers[q] != 1 || sel_of[o.pos] < 0 || t.shape.empty() ||
            t.shape[0] <= 0)
          continue;
        const uint64_t row_bytes = (t.end - t.begin) / static_cast<uint64_t>(t.shape[0]);
        const uint32_t k = need_at[q];
        sub_lo[k] = static_cast<uint64_t>(o.start) * row_bytes;
        sub_rows[k] = o.stop - o.start;
        if (slices2.empty()) slices2.assign(sel->slices, sel->slices + sel->n_names);
        slices2[sel_of[o.pos]].dim = -1;
      }
    }
    st_selection sel2 = *sel;
    if (!slices2.empty()) sel2.slices = slices2.data();
    // Those tensors staged back to back (256-byte aligned) under their view
    // names: a small index whose data section is the staging buffer.
    auto core = std::make_shared<Core>();
    uint64_t at = 0;
    for (size_t k = 0; k < need.size(); ++k) {
      const uint32_t q = need[k];
      Tensor t = ix.core->tensors[ix.ent[q]];
      uint64_t n = t.end - t.begin;
      if (sub_rows[k] >= 0) {
        const uint64_t rows = static_cast<uint64_t>(t.shape[0]);
        n = static_cast<uint64_t>(sub_rows[k]) * (n / rows);
        t.numel = static_cast<uint64_t>(sub_rows[k]) * (t.numel / rows);
        t.shape[0] = sub_rows[k];
      }
      t.name = ix.names[q];
      at = (at + 255) & ~uint64_t(255);
      t.begin = at;
      t.end = at + n;
      at += n;
      core->tensors.push_back(std::move(t));
    }
    core->data_bytes = at;
    if (at > staging_bytes)
      return set_error(ST_E_INVAL, "staging needs %llu bytes, %llu given", (unsigned long long)at,
                       (unsigned long long)staging_bytes);
    if (!staging_dev) return set_error(ST_E_INVAL, "NULL staging buffer");
    // Destinations checked on the host: non-NULL and itemsize-aligned.
    uint64_t traffic = 0;
    for (size_t i = 0; i < outs.size(); ++i) {
      const Output &o = outs[i];
      const uint64_t isz = dtype_size(o.out_dtype);
      if (o.numel && (!dst_host_ptrs[i] || (reinterpret_cast<uintptr_t>(dst_host_ptrs[i]) & (isz - 1))))
        return set_error(ST_E_INVAL, "destination of \"%s\" is NULL or not %llu-byte aligned", o.name.c_str(),
                         (unsigned long long)isz);
      traffic += o.units * (cls_in_size(o.cls) + cls_out_size(o.cls));
    }
    auto mini = make_root(core);
    s = finish_view(mini.get());
    if (s != ST_OK) return s;
    // Units large enough that the tables fit the static array, and warps in
    // proportion to the traffic: the host plan and its tables grow with the
    // warp count, and one tensor's launch needs few warps (its GPU time
    // overlaps the next call's host work).
    st_plan_options po{};
    po.unit_bytes = std::max<uint64_t>(kDefaultUnitBytes, traffic / 32768 + 1);
    po.workers = static_cast<uint32_t>(std::min<uint64_t>(kLazyMaxWarps, (traffic / kLazyBytesPerWarp + 8) & ~7ull));
    st_plan_s plan;
    s = plan_host(mini, &sel2, dst_dtype, &po, &plan);
    if (s != ST_OK) return s;
    s = check_tma_source(&plan, staging_dev);
    if (s != ST_OK) return s;
    // Host bytes (the RAM tier, or a plain read) -> staging, then launch.
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::vector<const void *> held;
    std::vector<std::vector<uint8_t>> plain;
    auto release_all = [&]() {
      for (const void *h : held) st_cache_release(cache, h);
      held.clear();
    };
    // Without a RAM tier the bytes go straight from the files' mappings
    // (faulted in first, so a page that cannot be read is ST_E_IO before its
    // copy); files that could not be mapped are read into host memory.
    const bool direct = !cache && files_mapped(files);
    cudaError_t e = cudaSuccess;
    for (size_t k = 0; k < need.size() && s == ST_OK; ++k) {
      const uint64_t from = ix.core->tensors[ix.ent[need[k]]].begin + sub_lo[k];  // arena byte
      const uint64_t n = core->tensors[k].end - core->tensors[k].begin;
      if (!n) continue;
      uint8_t *to = static_cast<uint8_t *>(staging_dev) + core->tensors[k].begin;
      const void *host = nullptr;
      if (direct) {
        s = st_files_prefetch(files, from, n, 0);
        if (s == ST_OK) s = copy_arena_direct(files, from, n, to, st);
        continue;
      }
      if (cache) {
        s = st_cache_get(cache, files, from, n, threads, &host);
        if (s != ST_OK) break;
        held.push_back(host);
      } else {
        plain.emplace_back(n);
        s = read_arena(files, from, n, plain.back().data(), threads);
        if (s != ST_OK) break;
        host = plain.back().data();
      }
      e = cudaMemcpyAsync(to, host, n, cudaMemcpyHostToDevice, st);
      if (e != cudaSuccess) break;
    }
    if (s != ST_OK) {  // copies already queued still read host memory or the mappings
      cudaStreamSynchronize(st);
      release_all();
      return s;
    }
    cudaEvent_t done = nullptr;
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&done, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(done, st);
    // RAM-tier entries: held until the copies that read them finish, then
    // dropped by a later cache call (no wait here); other sources: wait.
    if (e == cudaSuccess && cache && !held.empty() && cache_release_after(cache, done, held)) {
      held.clear();
      done = nullptr;  // the cache owns the event now
    }
    if (e == cudaSuccess && done) e = cudaEventSynchronize(done);
    if (done) cudaEventDestroy(done);
    release_all();
    if (e != cudaSuccess) return set_error(ST_E_CUDA, "staging the tensors: %s", cuda_msg(e).c_str());
    return launch_static(&plan, staging_dev, nullptr, dst_host_ptrs, nullptr, stream, /*mirror=*/true);
  } catch (const std::bad_alloc &) {
    return set_error(ST_E_NOMEM, "out of host memory");
  }
}

st_status st_plan_check(const st_plan_t *p, void *stream, uint32_t *flags) {
  if (!p || !flags) return set_error(ST_E_INVAL, "NULL argument");
  st_status s = check_device_plan(p);
  if (s != ST_OK) return s;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  uint32_t v = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&v, p->d_err, sizeof v, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && v) e = cudaMemset(p->d_err, 0, sizeof v);
  if (e != cudaSuccess) return set_error(ST_E_CUDA, "reading the error word: %s", cuda_msg(e).c_str());
  *flags = v;
  if (v)
    return set_error(ST_E_DEVICE, "device flags 0x%x:%s%s", v,
                     (v & kErrBadDst) ? " a non-empty output had a NULL or misaligned destination;" : "",
                     (v & kErrTimeout) ? " a wait for a staged copy gave up;" : "");
  return ST_OK;
}

st_status st_static_check(void *stream, uint32_t *flags) {
  if (!flags) return set_error(ST_E_INVAL, "NULL argument");
  void *scratch = nullptr;
  st_status s = static_scratch(&scratch);
  if (s != ST_OK) return s;
  uint32_t *err = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(scratch) + kStaticErrOffset);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, err, sizeof v, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && v) e = cudaMemsetAsync(err, 0, sizeof v, st);
  if (e == cudaSuccess && v) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return set_error(ST_E_CUDA, "reading the static error word: %s", cuda_msg(e).c_str());
  *flags = v;
  if (v)
    return set_error(ST_E_DEVICE, "static-scratch device flags 0x%x:%s%s", v,
                     (v & kErrBadDst) ? " a non-empty output had a NULL or misaligned destination;" : "",
                     (v & kErrTimeout) ? " a wait for a staged copy gave up;" : "");
  return ST_OK;
}

}  // extern "C"
