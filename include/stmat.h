/*
 * stmat.h -- C ABI of libstmat: materialize tensors from a safetensors
 * checkpoint on one GB300 GPU (sm_103a).
 *
 * What the library computes follows "Disk tier safetensors streaming design
 * audit (ComfyUI)":
 *   - "FastSageTensors (fastsafetensors) capability audit": the header is parsed
 *     into per-tensor dtype, shape and data_offsets without allocating tensors
 *     (st_index_build and the index queries);
 *   - "Strategy summary (implemented)", "Streaming safetensors mapping": a
 *     metadata-only index with lazy Prefix/Filter/Rename views (st_view_*);
 *   - "Range reads and tiering", Disk->RAM->GPU: read the byte range into
 *     (pinned) host memory and copy it to the GPU (st_stage_h2d, st_load);
 *   - "ComfyUI load path + eager materialization sites" (scaled-FP8
 *     conversion in comfy/sd.py) and "VRAM/RAM offload logic"
 *     (comfy_cast_weights): each selected tensor is gathered from its byte
 *     range and cast, fp8 weights dequantized by their per-tensor scale
 *     (st_plan, st_materialize).
 * The byte layout is not printed on the pages; the library reads the public
 * safetensors layout: bytes [0,8) hold N, an unsigned 64-bit little-endian
 * header length; bytes [8, 8+N) hold a UTF-8 JSON object mapping each tensor
 * name to {"dtype", "shape", "data_offsets": [begin, end]} plus an optional
 * "__metadata__" object of strings; the data section starts at byte 8+N and
 * [begin, end) are offsets into it.
 *
 * Element conversion (bit-exact, deterministic):
 *   - float sources (F32, F16, BF16, F8_E4M3, F8_E5M2) are decoded exactly,
 *     fp8 values are multiplied by their per-tensor binary32 scale in one IEEE
 *     binary32 multiply, and the result is rounded to the output dtype with
 *     round-to-nearest-even, gradual underflow and overflow to infinity;
 *   - any NaN result becomes the output's positive quiet NaN (BF16 0x7FC0,
 *     F16 0x7E00, F32 0x7FC00000);
 *   - integer and BOOL tensors, and tensors whose output dtype equals their
 *     own dtype (without a scale), are copied byte for byte.
 *
 * Conventions: every call returns an st_status; ST_OK is 0.  On failure the
 * thread-local message from st_last_error() says what failed, with the numbers
 * involved.  No call throws, aborts or traps, and nothing falls back to the
 * CPU: a CUDA failure is ST_E_CUDA.  Handles are not thread-safe; distinct
 * handles may be used from different threads.
 */
#ifndef STMAT_H_
#define STMAT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum st_status {
  ST_OK = 0,
  ST_E_INVAL = 1,            /* bad argument (NULL pointer, bad option, bad handle use) */
  ST_E_TRUNCATED = 2,        /* fewer than 8 bytes, or 8 + N beyond the bytes given */
  ST_E_HEADER_JSON = 3,      /* header is not the JSON the format requires */
  ST_E_HEADER_TOO_LARGE = 4, /* N > 100,000,000 */
  ST_E_DUP_KEY = 5,          /* a tensor name (or output name) appears twice */
  ST_E_DTYPE = 6,            /* unknown dtype string */
  ST_E_SHAPE = 7,            /* dimension not a non-negative integer, or size overflow */
  ST_E_OFFSETS = 8,          /* offsets invalid, out of range, wrong size, overlap, hole */
  ST_E_NOT_FOUND = 9,        /* a named tensor does not exist */
  ST_E_UNSUPPORTED_CAST = 10,/* the requested output dtype cannot be produced */
  ST_E_ALIGN = 11,           /* a pointer is not aligned as required */
  ST_E_NOMEM = 12,           /* host allocation failed */
  ST_E_CUDA = 13,            /* a CUDA runtime call failed (message has the CUDA error) */
  ST_E_DEVICE = 14,          /* the kernel reported a bad destination or a wait that gave up (st_plan_check) */
  ST_E_IO = 15               /* a file could not be opened or read (the message has the OS error) */
} st_status;

/* Dtypes in the header's spelling; ST_KEEP is only an output request. */
typedef enum st_dtype {
  ST_BOOL = 0, ST_U8 = 1, ST_I8 = 2, ST_I16 = 3, ST_U16 = 4, ST_I32 = 5, ST_U32 = 6,
  ST_I64 = 7, ST_U64 = 8, ST_F16 = 9, ST_BF16 = 10, ST_F32 = 11, ST_F64 = 12,
  ST_F8_E4M3 = 13, ST_F8_E5M2 = 14, ST_KEEP = 15
} st_dtype;

typedef struct st_index st_index_t; /* a parsed header, or a view of one */
typedef struct st_plan_s st_plan_t; /* a selection turned into device work */
typedef struct st_files_s st_files_t; /* open shard files addressed as one arena */
typedef struct st_cache_s st_cache_t; /* LRU RAM tier of host copies of file ranges */

/* ---------------------------------------------------------------- header */

/* Reads N from the first 8 bytes of a file.  len < 8 -> ST_E_TRUNCATED;
 * N > 100,000,000 -> ST_E_HEADER_TOO_LARGE. */
st_status st_header_size(const uint8_t *first8, size_t len, uint64_t *header_len);

/* Builds the metadata-only index from the first 8 + N bytes of a file
 * (`header_bytes`, `len` bytes; the caller keeps ownership, the index copies
 * what it needs) and the size of the data section (`data_bytes` = file size -
 * 8 - N).  Validates: JSON syntax and schema, unique names, known dtypes,
 * shapes, end - begin == numel * itemsize, end <= data_bytes, and that the
 * ranges, sorted by offset, tile [0, data_bytes) with no hole or overlap.
 * Errors: ST_E_TRUNCATED (len < 8 + N), ST_E_HEADER_TOO_LARGE, then the
 * first defect: JSON syntax first, then per member in document order
 * (duplicate name, schema, dtype, shape, offsets), then the tiling.
 * Index order: ascending (begin, end, name bytewise). */
st_status st_index_build(const uint8_t *header_bytes, size_t len, uint64_t data_bytes,
                         st_index_t **out);

/* Same, from a whole in-memory file image of `file_len` bytes. */
st_status st_index_build_file(const uint8_t *file, uint64_t file_len, st_index_t **out);

/* Releases an index or view.  Views and plans stay valid after their parent
 * is freed (they share the parsed header by reference count). */
void st_index_free(st_index_t *index);

typedef struct st_tensor_info {
  const char *name;      /* the name under this index/view; UTF-8, NUL-terminated */
  st_dtype dtype;
  int32_t ndim;
  const int64_t *shape;  /* ndim entries */
  uint64_t numel;        /* product of shape; 1 for [] */
  uint64_t begin, end;   /* [begin, end) in the data section */
} st_tensor_info;
/* Pointers in st_tensor_info stay valid while `index` lives. */

st_status st_index_count(const st_index_t *index, size_t *count);
st_status st_index_get(const st_index_t *index, size_t i, st_tensor_info *info);
/* Position of `name` in this index/view; ST_E_NOT_FOUND if absent. */
st_status st_index_find(const st_index_t *index, const char *name, size_t *i);
/* N and data_bytes of the underlying file (a joined index: 0 and the arena size). */
st_status st_index_sizes(const st_index_t *index, uint64_t *header_len, uint64_t *data_bytes);
/* Sum of numel, and per-dtype element counts (counts[15], may be NULL):
 * metadata-only parameter count and dominant dtype ("Pipeline refactors":
 * calculate_parameters / weight_dtype made metadata-aware). */
st_status st_index_numel(const st_index_t *index, uint64_t *total, uint64_t *counts);
/* "__metadata__" entries, in document order. */
st_status st_index_metadata_count(const st_index_t *index, size_t *count);
st_status st_index_metadata_get(const st_index_t *index, size_t i, const char **key,
                                const char **value);

/* ----------------------------------------------------------------- views */
/* Views are new indexes over the same header, in the parent's order: they
 * narrow or rename the metadata and never read tensor bytes.  The caller
 * frees them with st_index_free. */

/* Keeps names that start with `prefix` and strips the prefix. */
st_status st_view_prefix(const st_index_t *parent, const char *prefix, st_index_t **out);
/* Keeps the `n` listed names; each must exist (ST_E_NOT_FOUND). */
st_status st_view_filter(const st_index_t *parent, const char *const *names, size_t n,
                         st_index_t **out);
/* Ordered prefix rules from[i] -> to[i]: the first rule whose `from` starts
 * the name replaces that prefix; names no rule matches are kept.  Two
 * entries mapping to one name -> ST_E_DUP_KEY (state_dict_prefix_replace). */
st_status st_view_rename(const st_index_t *parent, const char *const *from, const char *const *to,
                         size_t n, st_index_t **out);

/* One index over several shard files ("Disk tier safetensors streaming
 * design audit (ComfyUI)", "Strategy summary (implemented)": a
 * checkpoint split over shard files is loaded through one streaming
 * mapping), so that one plan and one launch cover every shard.
 *   parts   n >= 1 indexes or views, one per shard, in arena order.
 *   align   power of two: shard k's data section is placed in one arena at
 *           bases[k] = the end of shard k-1's rounded up to `align`
 *           (bases[0] = 0); the bytes between shards are never read.
 *   bases   caller array of n entries, written on success.  The caller
 *           places shard k's data section at arena + bases[k] and passes the
 *           arena as data_dev / data_host.
 * The joined index lists part 0's entries, then part 1's, ..., each in its
 * part's order under its part's names, with offsets shifted by the part's
 * base; data_bytes = bases[n-1] + data_bytes of part n-1; header_len = 0;
 * metadata keeps each key's first occurrence in part order.  Names must be
 * unique across parts (ST_E_DUP_KEY); ST_E_INVAL on NULL or a bad align.
 * The parts may be freed afterwards. */
st_status st_index_concat(const st_index_t *const *parts, size_t n, uint64_t align, uint64_t *bases,
                          st_index_t **out);

/* ------------------------------------------------------------------ plan */

/* A range along one dimension (the slicing metadata a TensorFrame carries,
 * "Disk tier safetensors streaming design audit (ComfyUI)", "FastSageTensors
 * (fastsafetensors) capability audit"):
 * the output keeps indices [start, stop) of dimension `dim` and all of the
 * others, row-major, so its shape is the tensor's with shape[dim] =
 * stop - start.  dim < 0: the whole tensor.  0 <= dim < ndim and
 * 0 <= start <= stop <= shape[dim], else ST_E_INVAL.  Slicing the outer
 * dimension gives one contiguous source range; slicing an inner one gives
 * one run per outer index (a strided gather, e.g. a row-parallel
 * tensor-parallel shard). */
typedef struct st_slice {
  int32_t dim;
  int64_t start, stop;
} st_slice;

/* A block-scaled weight format (the resident-LLM architecture page, "Current
 * Backend Boundary", names block-FP8 and NVFP4 checkpoints but not their
 * layouts; these are the readings the library implements):
 *   ST_QUANT_BLOCK_FP8: an F8_E4M3 or F8_E5M2 [M, N] weight and an F32
 *     [ceil(M/br), ceil(N/bc)] tensor of block scales; output element (i, j)
 *     = weight (i, j) * scale (i/br, j/bc), one binary32 multiply, rounded to
 *     the output dtype.  br, bc powers of two, bc >= 16; 0 means 128.
 *   ST_QUANT_NVFP4: a U8 [M, K] weight holding M x 2K OCP MX E2M1 values
 *     (element 2c in the low nibble of byte c, 2c+1 in the high nibble), an
 *     F8_E4M3 [M, ceil(2K/16)] tensor of scales for 16 elements of a row,
 *     and a one-element F32 global scale; output element (i, j) = e2m1 *
 *     (scale (i, j/16) * global), each product one binary32 multiply; the
 *     output has shape [M, 2K].  block_rows/block_cols must be 0 (or 1/16).
 * The output dtype must be BF16, F16 or F32; a block-scaled output takes no
 * slice and no per-tensor scale; its scale tensors are consumed.  Plans with
 * block-scaled outputs run a TMA kernel build (4 unless 3 is asked for). */
typedef enum st_quant_kind { ST_QUANT_NONE = 0, ST_QUANT_BLOCK_FP8 = 2, ST_QUANT_NVFP4 = 3 } st_quant_kind;

typedef struct st_block_quant {
  int32_t kind;            /* st_quant_kind */
  const char *scale;       /* the block-scales tensor */
  const char *scale2;      /* ST_QUANT_NVFP4: the global scale tensor; else NULL */
  uint32_t block_rows, block_cols;
} st_block_quant;

typedef struct st_selection {
  /* Names to materialize, in output order; NULL selects every tensor of the
   * index in index order. */
  const char *const *names;
  size_t n_names;
  /* Optional, n_names entries: scale tensor name per selected name (NULL
   * entry: unscaled).  Requires `names`. */
  const char *const *scale_names;
  /* Optional pairing by name when scale_names is NULL: an fp8 tensor
   * "<stem><scale_suffix_from>" uses "<stem><scale_suffix_to>" if present. */
  const char *scale_suffix_from;
  const char *scale_suffix_to;
  /* Keep part `part` of `n_parts` (0/0 or 0/1: everything): outputs are
   * split into contiguous runs balanced by output bytes; output i (b_i bytes,
   * c_i bytes before it, T in total) belongs to part
   * floor(n_parts * (2 c_i + b_i) / (2 T)). */
  uint32_t part, n_parts;
  /* Optional, n_names entries (requires names): a slice per selected name.
   * Parts (above) weigh outputs by their sliced bytes. */
  const st_slice *slices;
  /* Optional, n_names entries (requires names): a block-scaled format per
   * selected name (kind ST_QUANT_NONE: an ordinary tensor). */
  const st_block_quant *quant;
} st_selection;
/* A scale must be a one-element F32 tensor and may scale only an fp8 tensor
 * (ST_E_INVAL otherwise); scale tensors are consumed, not output.  Output
 * dtype: integers and BOOL keep theirs, ST_KEEP keeps every dtype (no
 * scales allowed), float sources take dst_dtype (ST_BF16, ST_F16, ST_F32);
 * F64 -> 16/32-bit floats is ST_E_UNSUPPORTED_CAST. */

typedef struct st_plan_options {
  uint32_t workers;       /* warps to balance over; 0 = blocks_per_sm resident 8-warp blocks
                             on every SM of the current device */
  uint64_t chunk_bytes;   /* 0 = one launch over the whole data section; otherwise the data
                             section is split in chunks of this size for st_load's pipeline */
  int32_t host_only;      /* nonzero: build the plan without touching the GPU (requires workers) */
  uint32_t blocks_per_sm; /* 0 = 2 for the streaming build; the most that fit for the other
                             builds */
  uint64_t unit_bytes;    /* traffic per interleaved unit; 0 = 16384 for the TMA build, 32768
                             otherwise */
  uint32_t kernel;        /* 0 = choose: the TMA build when outputs average under 64 KiB of
                             traffic (many small tensors), else the streaming build; 1 = streaming
                             build (deep unroll); 2 = latency build (high occupancy); 3 = TMA
                             build (source bytes staged in shared memory by bulk copies; the
                             data section must then be device or managed memory, else
                             st_materialize returns ST_E_INVAL); 4 = the TMA build with fewer
                             copies in flight per warp and more warps per SM, the default for
                             plans with block-scaled outputs */
  uint32_t order;         /* unit order within a chunk: 0 = the build's default (2 for builds 1
                             and 2, 1 for the TMA build); 1 = source order (the TMA build then
                             fetches adjacent small tensors with one bulk copy); 2 = grouped by
                             conversion class, then source order (all warps run one class at a
                             time) */
} st_plan_options;

/* Builds the plan: outputs, then pieces (output element ranges).  Each chunk
 * is cut, in the unit order of `order`, into units of about unit_bytes of
 * traffic (source plus destination bytes) in rounds of `workers` units, and
 * unit j is given to warp j mod workers, so that all warps sweep the data
 * section together; the last rounds, about a share of the chunk's cost (8 %
 * for the TMA build, 40 % for the wide TMA build, 20 % for the streaming
 * build when the outputs' contiguous runs average 64 KiB of traffic or more,
 * else 30 %; none for the latency build), are left as a claimed tail that
 * whichever warps finish their own units first take while the kernel runs
 * (the TMA build's tail cut further into pieces of at most 2 KiB of source,
 * claimed at least two at a time).  Unless host_only, allocates the
 * plan's device tables on the current device (cudaMalloc) and uploads them
 * synchronously.  opts may be NULL. */
st_status st_plan(const st_index_t *index, const st_selection *sel, st_dtype dst_dtype,
                  const st_plan_options *opts, st_plan_t **out);
void st_plan_free(st_plan_t *plan);

typedef struct st_output_info {
  const char *name;       /* output name */
  st_dtype dtype;         /* output dtype */
  st_dtype src_dtype;
  int32_t ndim;
  const int64_t *shape;   /* the output's shape (sliced when a slice was given) */
  uint64_t numel;         /* elements of the output */
  uint64_t bytes;         /* numel * itemsize(dtype) */
  uint64_t src_begin;     /* data-section offset of the source tensor */
  const char *scale_name; /* scale tensor (block scales for a block-scaled output), or NULL */
  int32_t slice_dim;      /* the slice, or -1 */
  int64_t slice_start, slice_stop;
  int32_t quant_kind;     /* st_quant_kind of the output */
} st_output_info;

st_status st_plan_count(const st_plan_t *plan, size_t *count);
st_status st_plan_output(const st_plan_t *plan, size_t i, st_output_info *info);
/* Offsets of every output in one buffer, each aligned to `align` (a power of
 * two >= 16); offsets has st_plan_count entries.  `total` is the size. */
st_status st_plan_arena(const st_plan_t *plan, uint64_t align, uint64_t *offsets, uint64_t *total);
/* Piece/worker layout and kernel build (1 streaming, 2 latency, 3 TMA, 4 wide TMA), for tests and
 * tuning; any pointer may be NULL. */
st_status st_plan_stats(const st_plan_t *plan, uint32_t *workers, uint32_t *chunks, uint64_t *pieces,
                        uint32_t *kernel);
/* The data-section bytes st_load and st_load_files copy for this plan: all of
 * it, or, when the outputs read under three quarters of it (a
 * tensor-parallel rank's slices), only the byte ranges they read (each
 * output's source extent and its scales, merged across gaps under 64 KiB),
 * in *ranges pieces (may be NULL). */
st_status st_plan_copy_bytes(const st_plan_t *plan, uint64_t *bytes, uint32_t *ranges);
/* The range reads of "Range reads and tiering" (Disk tier safetensors
 * streaming design audit) as the loaders perform them for a plan.  Range
 * i < *ranges of st_plan_copy_bytes: data-section bytes [begin, end),
 * ascending and disjoint (more than 64 KiB apart).  ST_E_INVAL for i out of
 * range. */
st_status st_plan_copy_range(const st_plan_t *plan, uint32_t i, uint64_t *begin, uint64_t *end);
/* Piece k (host copy): `rows` runs of `count` counted units; run r reads
 * from data-section offset src + r * pitch and writes output bytes from
 * dst + r * count * out_itemsize; scale offset (or ~0), output, class. */
st_status st_plan_piece(const st_plan_t *plan, uint64_t k, uint64_t *src, uint64_t *dst,
                        uint64_t *scale, uint32_t *count, uint32_t *output, uint32_t *cls,
                        uint32_t *rows, uint64_t *pitch);
/* No counterpart on the pages (a description of the kernels' work split).
 * Conversion class `cls` (st_plan_piece's class, 0 .. 21): bytes per counted
 * unit read (src_item) and written (out_item), and one lane step of the
 * kernels' vector bodies: step_src source bytes, step_units counted units,
 * step_out output bytes (one 16- or 8-byte vector).  The kernels' codecs are
 * checked against these when the library is compiled.  Any pointer may be
 * NULL; ST_E_INVAL for an unknown class. */
st_status st_class_step(uint32_t cls, uint32_t *src_item, uint32_t *out_item, uint32_t *step_src,
                        uint32_t *step_units, uint32_t *step_out);
/* Pieces of worker w < workers in chunk c: [first, last), the warp's own
 * share; w == workers gives the chunk's claimed pieces, which the warps take
 * in source order while the kernel runs, whichever warp is free (empty for
 * plans without a claimed tail).  The ranges of w = 0 .. workers cover the
 * chunk's pieces once. */
st_status st_plan_worker(const st_plan_t *plan, uint32_t chunk, uint32_t w, uint64_t *first,
                         uint64_t *last);

/* ------------------------------------------------------------ device path */

/* ------------------------------------------------------------- files */
/* "Range reads and tiering" (Disk->RAM->GPU): bytes are read from the files
 * with pread into host memory, only the ranges asked for. */

/* Parses the header of the safetensors file at `path` (reads 8 + N bytes)
 * into an index; *data_offset (may be NULL) = 8 + N, the file offset of the
 * data section.  ST_E_IO when the file cannot be opened or read; the header
 * errors of st_index_build otherwise. */
st_status st_index_open(const char *path, st_index_t **out, uint64_t *data_offset);

/* One file's data section placed in an arena: arena bytes [base, base +
 * bytes) are the file's bytes [offset, offset + bytes).  For a checkpoint
 * joined by st_index_concat: offset = data_offset of shard k, bytes = its
 * data section size, base = bases[k]. */
typedef struct st_file_part {
  const char *path;
  uint64_t offset, bytes, base;
} st_file_part;

/* Opens the files of `n` parts (read-only) and checks each holds its range;
 * the parts must not overlap in the arena.  Each file is also mapped
 * read-only (shared) for ring-less st_load_files; a file that cannot be
 * mapped is still opened (only ring-less loads of its bytes then fail).
 * ST_E_IO on open/stat failures or a file too short, ST_E_INVAL on overlap.
 * The paths are copied.  A file must not shrink while it is open.  Reads
 * with several threads use reader threads the files object keeps until it is
 * closed: a process forked after they started must not use the object. */
st_status st_files_open(const st_file_part *parts, size_t n, st_files_t **out);
void st_files_close(st_files_t *files);
/* Reads arena bytes [begin, begin + bytes) into host[0, bytes) with up to
 * `threads` reader threads (0 or 1: the calling thread); bytes of the range
 * that no part covers are left as they are.  Synchronous.  ST_E_INVAL when
 * the range leaves the arena, ST_E_IO on a failed read. */
st_status st_files_read(const st_files_t *files, uint64_t begin, uint64_t bytes, void *host,
                        uint32_t threads);

/* The CPUs local to GPU `device` (from the PCI device's local_cpulist in
 * sysfs), written to cpulist (len bytes, NUL-terminated, e.g. "0-71").  With
 * apply != 0 the calling thread is also bound to them (threads it starts
 * later inherit the binding), so that pinned host memory it allocates lands
 * on the GPU's own socket: copies from another socket's memory cross the CPU
 * interconnect.  Changes nothing outside the calling process.  ST_E_CUDA
 * (no such device), ST_E_IO (sysfs unreadable), ST_E_INVAL (bad list). */
st_status st_host_affinity(int device, int32_t apply, char *cpulist, size_t len);

/* Faults arena bytes [begin, begin + bytes) into the page tables of the
 * files' read-only mappings, reading pages that are not in the page cache
 * from disk (madvise MADV_POPULATE_READ), on up to `threads` host threads
 * (0: the calling thread); synchronous.  A prefetch: ring-less st_load_files does the same per chunk
 * ahead of its copies.  ST_E_INVAL when the range leaves the arena, ST_E_IO
 * when a page cannot be read (a file that shrank after it was opened, an I/O
 * error); ST_OK without effect where the kernel lacks MADV_POPULATE_READ or a
 * file could not be mapped. */
st_status st_files_prefetch(const st_files_t *files, uint64_t begin, uint64_t bytes, uint32_t threads);

/* *yes = 1 when GPU `device` reads pageable host memory through the host's
 * page tables (cudaDevAttrPageableMemoryAccessUsesHostPageTables, e.g. a GPU
 * attached to its CPU by a coherent link): copies from mapped files then go
 * from the page cache to the device with no CPU copy, and ring-less
 * st_load_files is the fast path.  Otherwise 0 (ring-less loads still work;
 * the driver then stages each copy through its own buffers).  ST_E_CUDA when
 * the device cannot be queried. */
st_status st_device_reads_pageable(int device, int32_t *yes);

/* Materializes every output of the plan on `stream` (a cudaStream_t; NULL is
 * the legacy default stream), asynchronously, with no host synchronization.
 *   data_dev  device pointer to the data section (any alignment; the plan's
 *             data_bytes bytes must be readable).  Only bytes inside it are read.
 *   dst_ptrs  DEVICE array of st_plan_count pointers: output i is written to
 *             dst_ptrs[i], which must be aligned to the output's itemsize and
 *             hold st_output_info.bytes bytes.  A NULL or misaligned pointer
 *             of a non-empty output is skipped and recorded for st_plan_check.
 *   scales    NULL, or a DEVICE array of st_plan_count binary32 values that
 *             replace the file's scale for fp8 outputs (entries of other
 *             outputs are ignored).  With NULL, fp8 outputs use their paired
 *             scale tensor's value from the data section, or 1.0.
 * Errors: ST_E_INVAL (NULL plan/data/dst_ptrs, host-only plan), ST_E_CUDA
 * (launch failure).  Outputs may not overlap each other or the data section.
 * Launches of one plan (this call, st_load, st_load_files) must not overlap
 * on the GPU: the TMA builds' warps claim pieces through two words the plan
 * owns, which each launch leaves at zero for the next (order them on one
 * stream, or with events). */
st_status st_materialize(const void *data_dev, const st_plan_t *plan, void *const *dst_ptrs,
                         const float *scales, void *stream);

/* Copies `bytes` from host memory to device memory on `stream` in chunks of
 * `chunk_bytes` (0 = one copy) with cudaMemcpyAsync, then records
 * `done_event` (a cudaEvent_t; may be NULL) on `stream`.  src_host should be
 * pinned (page-locked) for the copies to be asynchronous.  ST_E_INVAL on NULL
 * pointers with bytes > 0. */
st_status st_stage_h2d(void *dst_dev, const void *src_host, uint64_t bytes, uint64_t chunk_bytes,
                       void *stream, void *done_event);

/* Stages the data section from host memory (pinned, data_bytes long) into
 * data_dev on `copy_stream` chunk by chunk (the plan's chunk_bytes) and
 * materializes each chunk's pieces on `compute_stream` as soon as that
 * chunk's copy completes, so copies and kernels overlap.  A plan whose
 * outputs read under three quarters of the data section copies only the
 * ranges they read (st_plan_copy_bytes); data_dev's other bytes are left as
 * they are.  The first copy waits for work already queued on compute_stream.
 * Arguments as for st_materialize.  Returns without synchronizing. */
st_status st_load(const void *data_host, void *data_dev, const st_plan_t *plan, void *const *dst_ptrs,
                  const float *scales, void *copy_stream, void *compute_stream);

/* ------------------------------------------------------------ RAM tier */
/* "Disk tier integration" (Disk tier safetensors streaming design audit):
 * an LRU cache of host copies of tensors read from disk with a configurable
 * maximum number of bytes; eviction drops a host copy (the index still
 * describes the tensor, which is read again on its next use).  Thread-safe. */

typedef struct st_cache_info {
  uint64_t bytes, max_bytes;   /* bytes held by kept entries, and the bound */
  uint64_t entries;            /* kept entries */
  uint64_t hits, misses, evictions;
} st_cache_info;

/* pinned != 0: entries live in page-locked memory (cudaHostAlloc), so
 * copies from them to the GPU are asynchronous; else pageable malloc. */
st_status st_cache_create(uint64_t max_bytes, int32_t pinned, st_cache_t **out);
/* Waits for the copies of st_load_tensors calls that still read entries,
 * then frees every entry, held or not: release all holds first. */
void st_cache_free(st_cache_t *cache);
/* The host copy of arena bytes [begin, begin + bytes) of `files`: a hit
 * returns the kept copy (now the most recently used); a miss reads it with
 * pread (`threads` reader threads), evicting least-recently-used entries
 * that nobody holds until it fits the bound.  The entry is held, and *host
 * stays valid, until st_cache_release(cache, *host).  An entry larger than
 * the bound is read but not kept: it is freed on release.  Entries belong
 * to the st_files_t they were read from (each open gets an id of its own):
 * files opened again, even at the same address, never hit them; entries of
 * closed files age out.  Errors: ST_E_INVAL, ST_E_NOMEM, ST_E_IO. */
st_status st_cache_get(st_cache_t *cache, const st_files_t *files, uint64_t begin, uint64_t bytes,
                       uint32_t threads, const void **host);
st_status st_cache_release(st_cache_t *cache, const void *host);
st_status st_cache_stats(const st_cache_t *cache, st_cache_info *info);
/* Waits for the copies of st_load_tensors calls that still read entries
 * (releasing their holds), then drops every entry nobody holds. */
st_status st_cache_clear(st_cache_t *cache);

/* The lazy path for a few tensors ("Streaming safetensors mapping": a tensor
 * is loaded when it is accessed): the selected outputs of `sel` on `index`
 * (whose offsets are the arena of `files`), with the tensors they read
 * (their scales and block scales), are taken from `cache` (read from the
 * files on a miss; cache may be NULL: then copied straight from the files'
 * read-only mappings after st_files_prefetch of their bytes, or read when a
 * file could not be mapped), copied into staging_dev
 * (each at a 256-byte aligned offset; staging_bytes must hold them all, else
 * ST_E_INVAL with the size needed; an output that is a dim-0 slice of a
 * tensor no other output reads stages only its rows) and materialized by one
 * launch on
 * `stream`, with the plan's tables in the library's static device array as
 * for st_materialize_noalloc (no device allocation; calls whose work
 * overlaps on the GPU race on that array: order them on one stream).  The
 * tables go up in one asynchronous copy from a page-locked host mirror of
 * that array (two 4 MiB halves used in turn), allocated by the first call on
 * each device and kept until the process exits.
 *   dst_host_ptrs  HOST array of one destination (device) pointer per output,
 *                  in the selection's output order; each non-NULL and aligned
 *                  to the output's itemsize (ST_E_INVAL otherwise).
 * With a cache: returns once the staging copies are queued; the entries
 * they read stay held until the copies finish and are released by the next
 * st_cache_get or st_cache_stats on that cache that finds them finished
 * (st_cache_clear and st_cache_free wait for them), so the bound may be
 * exceeded meanwhile.  Without a cache: blocks until the copies are done
 * (the files may then be closed).  The kernel runs asynchronously on
 * `stream`; staging_dev is in use until it has run.  Output dtypes,
 * errors and bit-exact results are those of st_plan + st_materialize.  The
 * kernel's device flags (a wait for a staged copy that gave up; lazy
 * destinations are checked on the host) go to the static array's error word:
 * read them with st_static_check. */
st_status st_load_tensors(const st_index_t *index, const st_files_t *files, st_cache_t *cache,
                          const st_selection *sel, st_dtype dst_dtype, void *const *dst_host_ptrs,
                          void *staging_dev, uint64_t staging_bytes, uint32_t threads, void *stream);

/* The disk -> pinned RAM -> device -> materialize pipeline: for each chunk of
 * the plan (its chunk_bytes; one chunk when 0) reads the chunk's arena bytes
 * from `files` into a slot of the host ring with `threads` reader threads,
 * copies the slot to data_dev on copy_stream, and runs that chunk's pieces on
 * compute_stream once its copy is done, so reading chunk k + 1 overlaps the
 * copy and kernel of chunk k.  ring_host: ring_bytes of host memory, pinned
 * for the copies to be asynchronous, holding at least one chunk (two or more
 * for overlap); a slot is reused only after its previous copy finished.
 * Ring-less (ring_host NULL and ring_bytes 0): each chunk is copied to
 * data_dev straight from the files' read-only mappings (cudaMemcpyAsync from
 * pageable memory).  One host thread faults the chunks' pages into the page
 * tables ahead of the copies (madvise MADV_POPULATE_READ, which reads pages
 * not in the page cache from disk; `threads` is unused), and a page that
 * cannot be read (a file that shrank, an I/O error) ends the load with
 * ST_E_IO before that chunk's copy is queued.  On a GPU for which
 * st_device_reads_pageable reports 1 the copy engine then reads the page
 * cache directly.  Bytes of the arena that no file covers (gaps between
 * joined shards) get no defined value in either mode.  A plan whose outputs
 * read under three quarters of the arena (a tensor-parallel rank) reads and
 * copies only those ranges (st_plan_copy_bytes), in both modes; ring-less,
 * each range is then faulted in right before its copy.
 * The first copy waits for work already queued on compute_stream.  Blocks
 * the calling thread until every chunk is read and its copy finished (the
 * ring is then free, the mappings no longer read: the files may be closed),
 * also when it returns an error after queueing copies; the kernels may still
 * be running on compute_stream.  The plan's index must describe the files'
 * arena (data_bytes = the arena size).  Errors: ST_E_INVAL (arguments, ring
 * too small, arena size), ST_E_IO (reads; a file that could not be mapped,
 * ring-less), ST_E_CUDA. */
st_status st_load_files(const st_files_t *files, void *data_dev, const st_plan_t *plan,
                        void *const *dst_ptrs, const float *scales, void *ring_host, uint64_t ring_bytes,
                        uint32_t threads, void *copy_stream, void *compute_stream);

/* Allocation-free st_materialize.  No counterpart on the pages: it exists for
 * callers that cannot allocate device memory, for example a plugin or
 * library running inside a host application whose device memory is entirely
 * held by that application's own allocator (a framework's caching pool, a
 * serving engine's preallocated arena), so that cudaMalloc fails although
 * the pool has room; or code that must not allocate once it is running,
 * because cudaMalloc can block on the device and can fail at a point where
 * the caller has no way to recover.  Such a caller builds the plan with
 * host_only set (st_plan then touches no GPU memory) and calls this instead
 * of st_materialize; arguments are as for st_materialize.
 *   - Scratch: the plan's tables (piece table, per-chunk warp ranges and, for
 *     block-scaled outputs, the block-scale table) are copied
 *     (cudaMemcpyAsync from the plan's host memory) into one static device
 *     array of 4 MiB built into the library.  Every GPU that loads the
 *     library holds those 4 MiB until the process exits.  The tables may take
 *     4 MiB - 256 bytes (the last 256 hold the error word and the claim
 *     words of the TMA builds, which every launch leaves at zero): 48 bytes per
 *     piece, plus 4 bytes per warp and chunk (plus 4 per chunk), plus 32
 *     bytes per output for block-scaled plans, each part rounded up to 256
 *     bytes (st_load_tensors adds 8 bytes per output for its destination
 *     array).  A plan that needs more is rejected with ST_E_INVAL before
 *     anything is queued; plan with a larger unit_bytes or fewer workers to
 *     shrink it.
 *   - Set-up: the first call on a device, with that device current, looks up
 *     the array's device address (cudaGetSymbolAddress) once for that device.
 *   - Sharing: every call, on every stream, uses the same array, and it keeps
 *     the last call's tables.  Calls whose work overlaps on the GPU (different
 *     streams, or threads) race on the array and corrupt each other: order
 *     them on one stream.  The tables are rewritten by every call; nothing
 *     in them needs to start at zero.
 *   - Device flags: a NULL or misaligned destination is skipped as in
 *     st_materialize, and a wait of the TMA build for a staged copy that gives
 *     up stops that warp early (outputs incomplete).  Either sets a bit in the
 *     array's error word, which keeps the bits of every call (and of
 *     st_load_tensors) until st_static_check reads and clears it.
 *   - No cudaMalloc, cudaFree or other allocating CUDA or library routine is
 *     called.
 * Returns without synchronizing. */
st_status st_materialize_noalloc(const void *data_dev, const st_plan_t *plan, void *const *dst_ptrs,
                                 const float *scales, void *stream);

/* No counterpart on the pages (the library's own status for the two calls
 * that use its static array).  Reads and clears the error word of the
 * library's static device array on the current device: the device flags of
 * every st_materialize_noalloc and st_load_tensors call since the last read
 * (bits as for st_plan_check).
 * Copies the word to the host on `stream` and waits for the stream, so every
 * such call queued on it before has finished; calls on other streams are
 * seen only once they have finished.  Allocates nothing.  Returns
 * ST_E_DEVICE when any flag was set, ST_E_CUDA if the copy failed. */
st_status st_static_check(void *stream, uint32_t *flags);

/* Waits for `stream`, then reads and clears the plan's device error flags:
 * bit 0 = a non-empty output had a NULL or misaligned destination;
 * bit 1 = the TMA build gave up a bounded wait for a staged copy (its warp
 * stopped early; outputs are incomplete).
 * Returns ST_E_DEVICE when any flag was set. */
st_status st_plan_check(const st_plan_t *plan, void *stream, uint32_t *flags);

/* ----------------------------------------------------------------- misc */

/* Message of the calling thread's last failure ("" if none). */
const char *st_last_error(void);
/* "ST_OK", "ST_E_INVAL", ... */
const char *st_status_name(st_status status);
/* Itemsize in bytes of a dtype (0 for ST_KEEP / unknown). */
size_t st_dtype_size(st_dtype dtype);
/* Header spelling of a dtype ("F32", ...; "KEEP"), or NULL. */
const char *st_dtype_name(st_dtype dtype);
/* Library version, e.g. 0x000100 for 0.1.0. */
uint32_t st_version(void);

#ifdef __cplusplus
}
#endif

#endif /* STMAT_H_ */
