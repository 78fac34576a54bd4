// st_internal.h -- structures shared by the host library (index, planner,
// C ABI) and the sm_103a kernels.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <vector>

#include "stmat.h"

#if defined(__CUDACC__)
#define ST_HD __host__ __device__
#else
#define ST_HD
#endif

namespace stmat {

// Conversion classes.  A piece of class CLS_COPY counts bytes; every other
// class counts elements of its source dtype.
enum Cls : uint32_t {
  CLS_COPY = 0,
  CLS_F32_BF16,
  CLS_F32_F16,
  CLS_F16_BF16,
  CLS_F16_F32,
  CLS_BF16_F16,
  CLS_BF16_F32,
  CLS_E4M3_BF16,
  CLS_E4M3_F16,
  CLS_E4M3_F32,
  CLS_E5M2_BF16,
  CLS_E5M2_F16,
  CLS_E5M2_F32,
  // Block-scaled weights (a scale per block read from a second tensor):
  // fp8 elements, and NVFP4 bytes (two e2m1 elements per counted byte).
  CLS_QE4M3_BF16,
  CLS_QE4M3_F16,
  CLS_QE4M3_F32,
  CLS_QE5M2_BF16,
  CLS_QE5M2_F16,
  CLS_QE5M2_F32,
  CLS_NVFP4_BF16,
  CLS_NVFP4_F16,
  CLS_NVFP4_F32,
  CLS_COUNT
};
static_assert(CLS_COUNT <= 32, "classes fit kClsBits");

ST_HD constexpr bool cls_quant(uint32_t c) { return c >= CLS_QE4M3_BF16 && c < CLS_COUNT; }
ST_HD constexpr bool cls_nvfp4(uint32_t c) { return c >= CLS_NVFP4_BF16 && c < CLS_COUNT; }

// `rows` runs of `count` elements of one output: the unit a warp processes.
// Run r reads from data + src + r * pitch and writes to the output at
// dst + r * count * out_itemsize (one run unless an inner dimension is sliced).
struct alignas(16) Piece {
  uint64_t src;      // data-section byte offset of the first run's first element
  uint64_t dst;      // byte offset of that element inside its output buffer
  uint64_t scale;    // data-section byte offset of the binary32 scale, or kNoScale
  uint32_t count;    // elements per run (bytes for CLS_COPY)
  uint32_t out_cls;  // output index << kClsBits | class
  uint32_t rows;     // runs
  uint32_t pad;
  uint64_t pitch;    // source bytes between runs
};
static_assert(sizeof(Piece) == 48, "piece layout");

constexpr uint64_t kNoScale = ~0ull;
constexpr uint32_t kClsBits = 5;
constexpr uint32_t kMaxOutputs = 1u << (32 - kClsBits);
constexpr int kWarpsPerBlock = 8;

// Bits of the device error word: an output's destination is NULL or not
// aligned to its itemsize; a bounded wait for a staged copy gave up.
constexpr uint32_t kErrBadDst = 1u;
constexpr uint32_t kErrTimeout = 2u;

// Block scales of a block-scaled output (device table indexed by output).
struct alignas(16) QuantInfo {
  uint64_t scale;      // data-section offset of the block-scales tensor
  uint64_t scale2;     // NVFP4: data-section offset of the F32 global scale; else kNoScale
  uint32_t row_units;  // counted units per weight row (N elements, or K bytes for NVFP4)
  uint32_t scols;      // scale tensor columns
  uint32_t br_shift;   // log2 block rows
  uint32_t bc_shift;   // log2 block columns, in elements
};
static_assert(sizeof(QuantInfo) == 32, "quant layout");

struct LaunchArgs {
  const uint8_t *data;     // data section on the device
  uint64_t data_bytes;
  const Piece *pieces;     // all pieces of the plan
  const uint32_t *parts;   // workers + 1 piece indices: worker w owns [parts[w], parts[w+1])
  uint32_t workers;
  void *const *dst;        // device array: output index -> destination
  const float *scales;     // device array of per-output scales, or nullptr
  uint32_t *err;           // device error word
  const QuantInfo *quant;  // device array indexed by output (block-scaled outputs), or nullptr
  // TMA builds: pieces [parts[workers], claim_end) are claimed while the
  // launch runs, in source order, through two device words that are zero
  // before the launch (pieces claimed, warps done); the last warp to finish
  // sets them back to zero.
  uint32_t claim_end;
  uint32_t *claim;
  // Small single-chunk plans: the launch's piece table and destination array
  // (block 0) and the data-section bytes [pf_data_off, pf_data_off +
  // pf_data_bytes) (a slice per block) are prefetched into L2 as it starts;
  // pf_data_bytes 0: nothing.
  const void *pf_table = nullptr;
  uint32_t pf_table_bytes = 0;
  uint32_t pf_dst_bytes = 0;
  uint64_t pf_data_off = 0;
  uint64_t pf_data_bytes = 0;
};

// Bytes written per counted unit of a class.
ST_HD constexpr int cls_out_size(uint32_t c) {
  switch (c) {
    case CLS_COPY: return 1;
    case CLS_F32_BF16: case CLS_F32_F16: case CLS_F16_BF16: case CLS_BF16_F16:
    case CLS_E4M3_BF16: case CLS_E4M3_F16: case CLS_E5M2_BF16: case CLS_E5M2_F16:
    case CLS_QE4M3_BF16: case CLS_QE4M3_F16: case CLS_QE5M2_BF16: case CLS_QE5M2_F16: return 2;
    case CLS_NVFP4_F32: return 8;
    default: return 4;
  }
}

// Itemsize of a class's output dtype (the alignment its destination needs).
ST_HD constexpr int cls_out_item(uint32_t c) { return cls_nvfp4(c) ? cls_out_size(c) / 2 : cls_out_size(c); }

// Source itemsize of a class (bytes read per counted unit).
ST_HD constexpr int cls_in_size(uint32_t c) {
  switch (c) {
    case CLS_COPY: return 1;
    case CLS_F32_BF16: case CLS_F32_F16: return 4;
    case CLS_F16_BF16: case CLS_F16_F32: case CLS_BF16_F16: case CLS_BF16_F32: return 2;
    default: return 1;
  }
}

// log2 of the two sizes per counted unit (0..3), packed two bits per class,
// for shift-only address arithmetic in the kernels.
constexpr uint64_t pack_shifts(bool out) {
  uint64_t v = 0;
  for (uint32_t c = 0; c < CLS_COUNT; ++c) {
    const int size = out ? cls_out_size(c) : cls_in_size(c);
    v |= static_cast<uint64_t>(size == 8 ? 3 : size == 4 ? 2 : size == 2 ? 1 : 0) << (2 * c);
  }
  return v;
}
static_assert(2 * CLS_COUNT <= 64, "shift tables fit 64 bits");
constexpr uint64_t kInShifts = pack_shifts(false), kOutShifts = pack_shifts(true);
ST_HD constexpr uint32_t cls_in_shift(uint32_t c) { return static_cast<uint32_t>(kInShifts >> (2 * c)) & 3u; }
ST_HD constexpr uint32_t cls_out_shift(uint32_t c) { return static_cast<uint32_t>(kOutShifts >> (2 * c)) & 3u; }

// A lane step of a class in the kernels' vector bodies reads cls_step_src
// source bytes (cls_step_units counted units) and writes cls_step_out bytes,
// one 16- or 8-byte vector: widening classes read fewer source bytes.
// Block-scaled classes step over 8 fp8 bytes (4 for F32 outputs) or 4 NVFP4
// bytes.  The kernels' codec types are checked against these at compile time.
ST_HD constexpr uint32_t cls_step_src(uint32_t c) {
  return cls_nvfp4(c)   ? 4u
         : cls_quant(c) ? (cls_out_size(c) == 4 ? 4u : 8u)
         : cls_out_size(c) > cls_in_size(c) ? static_cast<uint32_t>(16 * cls_in_size(c) / cls_out_size(c))
                                            : 16u;
}
ST_HD constexpr uint32_t cls_step_units(uint32_t c) { return cls_step_src(c) / cls_in_size(c); }
ST_HD constexpr uint32_t cls_step_out(uint32_t c) { return cls_step_units(c) * cls_out_size(c); }

// Kernel builds (st_kernels.cu): deep unroll for large tensors, higher
// occupancy for many small tensors, or source bytes staged in shared memory
// by the bulk-copy (TMA) engine.
constexpr uint32_t kKernelStream = 1;
constexpr uint32_t kKernelLatency = 2;
constexpr uint32_t kKernelTma = 3;
constexpr uint32_t kKernelTmaWide = 4;  // the TMA build with fewer slots per warp and more warps per SM
constexpr bool is_tma_build(uint32_t variant) { return variant == kKernelTma || variant == kKernelTmaWide; }

// Resident 256-thread blocks per SM for a kernel build, and the SM count of
// the current device.
st_status kernel_occupancy(uint32_t variant, int *sms, int *blocks_per_sm);
// Launches the materialize kernel over `a.workers` warps.
st_status launch_materialize(const LaunchArgs &a, uint32_t variant, void *stream);

// Size of the device array behind st_materialize_noalloc, and its device
// address on the current device (looked up on first use per device).  Its
// last 256 bytes hold the error word of every launch from the array; the
// kernels only OR bits into it, so it keeps every call's flags until
// st_static_check reads and clears it.  The tables take the bytes before.
constexpr size_t kStaticScratchBytes = size_t(4) << 20;
constexpr size_t kStaticErrOffset = kStaticScratchBytes - 256;
constexpr size_t kStaticClaimOffset = kStaticErrOffset + 64;
st_status static_scratch(void **addr);

// Shard-file reads (st_io.cpp): arena bytes [begin, begin + bytes) into host.
st_status read_arena(const st_files_s *f, uint64_t begin, uint64_t bytes, void *host, uint32_t threads);
uint64_t files_arena_bytes(const st_files_s *f);
bool files_mapped(const st_files_s *f);  // every non-empty part has its read-only mapping
// Arena bytes [begin, begin + bytes) from the files' read-only mappings to
// device memory dev[0, bytes) with cudaMemcpyAsync on `stream` (a
// cudaStream_t); bytes no part covers are not written.
st_status copy_arena_direct(const st_files_s *f, uint64_t begin, uint64_t bytes, void *dev, void *stream);
// Populate threads for a load from the files' mappings: `threads` workers
// fault the arena's pages into the page tables (MADV_POPULATE_READ, which
// reads uncached pages from disk) in chunk order, ahead of the copies;
// chunk k is arena bytes [begin + k * chunk, ...) (one chunk when chunk is 0).
// populate_wait(k) blocks until chunk k's bytes are in (ST_E_IO when a page
// could not be read: the file shrank or an I/O error; ST_OK at once where the
// kernel lacks the call); populate_stop ends the workers and frees.
struct Populator;
// Hands one hold on each of `hosts` (entries of `cache`) over to be dropped
// once `event` (a cudaEvent_t recorded after the copies that read them; the
// cache destroys it) has completed: the next st_cache_get or st_cache_stats
// that finds it complete drops them, st_cache_clear and st_cache_free wait
// for it.  False (nothing handed over) when out of host memory.
bool cache_release_after(st_cache_s *cache, void *event, const std::vector<const void *> &hosts);
Populator *populate_start(const st_files_s *f, uint64_t begin, uint64_t bytes, uint64_t chunk,
                          uint32_t threads);
st_status populate_wait(Populator *p, uint64_t k);
void populate_stop(Populator *p);

// Error reporting shared by the host files.
st_status set_error(st_status s, const char *fmt, ...);

}  // namespace stmat
