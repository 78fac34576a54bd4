// st_kernels.cu -- the materialize kernel for GB300 (sm_103a).
//
// Gathers every selected tensor's byte range from the device copy of the data
// section and writes it, converted, to its destination ("Disk tier
// safetensors streaming design audit (ComfyUI)": the Disk->RAM->GPU range
// reads of "Range reads and tiering", the weight casting of "VRAM/RAM offload
// logic", and the scaled-FP8 conversion of "ComfyUI load path + eager
// materialization sites").  The pages run this as one torch cast per tensor;
// here one launch covers every tensor.
//
// Design (HBM-bound; no tensor cores, there is no contraction):
//  - the planner cut outputs into pieces and balanced them by bytes over W
//    warps; warp w walks its own pieces [parts[w], parts[w+1]) with no
//    inter-warp synchronization and no waits, so the kernel cannot stall on a
//    peer, then claims pieces of the plan's tail [parts[W], claim_end) in
//    source order from a claim word (warps that ran fast take more, so all
//    finish together; the last one out zeroes the word; launches without a
//    tail leave it alone).  Small plans (a source span of at most 16 MiB)
//    first prefetch that span, the piece table and the destination array
//    into L2, one slice per block, so the reads that follow a warp's first
//    one hit L2.  A warp stages up to
//    32 piece descriptors at a time in shared memory (one per lane), with
//    their destination pointers and scales, so the dependent loads of a piece
//    are paid once per 32 pieces;
//  - each lane moves one 16-byte source chunk per step (K = 16 / itemsize
//    elements) with 16-byte vector loads; consecutive lanes take consecutive
//    chunks, so every warp access is one contiguous run; a batch of up to 4
//    chunks per lane is loaded before any is converted;
//  - a source whose address is not 16-byte aligned is read as the two
//    aligned 16-byte words covering each chunk; the misalignment r is the
//    same for every chunk of a piece, so the realignment is two uniform word
//    selects (r & 8, r & 4) and four funnel shifts by 8 * (r & 3);
//  - destinations are written with aligned vector stores (8 or 16 bytes);
//    elements before the first aligned destination chunk, after the last, or
//    whose source window would leave the data section are converted one by
//    one with byte loads, so no byte outside the data section is read;
//  - conversions work on element pairs: exact decode to binary32 (cvt of
//    f16x2 and e4m3x2, bit placement for bf16 and e5m2), one __fmul_rn by
//    the scale for fp8, then cvt.rn to bf16x2/f16x2 (round to nearest even,
//    subnormals kept); NaN results become the output's positive quiet NaN.
//  - code size matters: one kernel serves every class, and workloads that
//    mix classes (many small tensors) otherwise stall on instruction fetch,
//    so each class has just an aligned and a misaligned body.
// Four builds share the codecs: streaming (deep register batches, for large
// tensors and sliced runs), latency (shallow batches at high occupancy, on
// request) and two shapes of the TMA build (source bytes staged in shared
// memory by bulk copies: four slots per warp for many small tensors, two
// slots at more warps per SM for block-scaled weights; see "the TMA build"
// below).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <string>

#include "st_internal.h"

namespace stmat {
namespace {

constexpr int kThreads = kWarpsPerBlock * 32;
constexpr uint32_t kNanBF16 = 0x7FC0u, kNanF16 = 0x7E00u, kNanF32 = 0x7FC00000u;

// ------------------------------------------------------------ element codecs

enum Src { S_F32, S_F16, S_BF16, S_E4M3, S_E5M2 };
enum Dst { D_BF16, D_F16, D_F32 };

template <int S> struct SrcInfo;
template <> struct SrcInfo<S_F32> { static constexpr int kSize = 4; };
template <> struct SrcInfo<S_F16> { static constexpr int kSize = 2; };
template <> struct SrcInfo<S_BF16> { static constexpr int kSize = 2; };
template <> struct SrcInfo<S_E4M3> { static constexpr int kSize = 1; };
template <> struct SrcInfo<S_E5M2> { static constexpr int kSize = 1; };

template <int D> struct DstInfo { static constexpr int kSize = D == D_F32 ? 4 : 2; };

// One element (for the scalar path): raw bits -> binary32.
template <int S>
__device__ __forceinline__ float decode1(uint32_t b) {
  if constexpr (S == S_F32) return __uint_as_float(b);
  if constexpr (S == S_F16) return __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
  if constexpr (S == S_BF16) return __uint_as_float(b << 16);
  if constexpr (S == S_E4M3) {
    __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
    return __half2float(__half(h));
  }
  // an e5m2 value is the upper byte of its binary16 encoding
  return __half2float(__ushort_as_half(static_cast<unsigned short>(b << 8)));
}

// One element: binary32 -> raw bits of the output dtype.
template <int D>
__device__ __forceinline__ uint32_t encode1(float x) {
  if constexpr (D == D_BF16) return x != x ? kNanBF16 : static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
  if constexpr (D == D_F16) return x != x ? kNanF16 : static_cast<uint32_t>(__half_as_ushort(__float2half_rn(x)));
  return x != x ? kNanF32 : __float_as_uint(x);
}

// Element pair j of a source step held in words s[] -> two binary32.
template <int S, int NS>
__device__ __forceinline__ float2 decode2(const uint32_t (&s)[NS], int j) {
  if constexpr (S == S_F32) {
    return make_float2(__uint_as_float(s[2 * j]), __uint_as_float(s[2 * j + 1]));
  } else if constexpr (S == S_F16) {
    __half2_raw h;
    h.x = static_cast<unsigned short>(s[j] & 0xFFFFu);
    h.y = static_cast<unsigned short>(s[j] >> 16);
    return __half22float2(__half2(h));
  } else if constexpr (S == S_BF16) {
    return make_float2(__uint_as_float(s[j] << 16), __uint_as_float(s[j] & 0xFFFF0000u));
  } else if constexpr (S == S_E4M3) {
    const uint32_t pair = (s[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(pair), __NV_E4M3);
    return __half22float2(__half2(h));
  } else {
    // bytes 2j, 2j+1 become the high bytes of two binary16 values
    const uint32_t bits = __byte_perm(s[j >> 1], 0u, (j & 1) ? 0x3424u : 0x1404u);
    __half2_raw h;
    h.x = static_cast<unsigned short>(bits & 0xFFFFu);
    h.y = static_cast<unsigned short>(bits >> 16);
    return __half22float2(__half2(h));
  }
}

// Two binary32 -> one packed 16-bit pair (lower address in the low half).
// A converted half is NaN exactly when its input was (rounding keeps
// infinities and never makes a NaN), so one packed unordered compare of the
// result with itself marks the NaN halves, which become the canonical NaN.
template <int D>
__device__ __forceinline__ uint32_t encode2_16(float2 f) {
  uint32_t r, m;
  if constexpr (D == D_BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(f.x, f.y);
    r = *reinterpret_cast<uint32_t *>(&v);
    m = __hneu2_mask(v, v);
    return (r & ~m) | (m & (kNanBF16 | (kNanBF16 << 16)));
  } else {
    __half2 v = __floats2half2_rn(f.x, f.y);
    r = *reinterpret_cast<uint32_t *>(&v);
    m = __hneu2_mask(v, v);
    return (r & ~m) | (m & (kNanF16 | (kNanF16 << 16)));
  }
}

// A conversion class.  One lane step reads SB source bytes (KS elements) and
// writes OS <= 16 output bytes: classes that widen read fewer source bytes per
// step so that every lane stores one contiguous 16-byte (or 8-byte) vector
// and a warp's store is one contiguous run.
template <int S, int D>
struct Conv {
  static constexpr int SI = SrcInfo<S>::kSize, SO = DstInfo<D>::kSize;
  static constexpr int SB = SO > SI ? 16 * SI / SO : 16;  // source bytes per lane step
  static constexpr int KS = SB / SI;                       // elements per lane step
  static constexpr int OS = KS * SO;                       // output bytes per lane step
  static constexpr bool kScaled = (S == S_E4M3 || S == S_E5M2);

  __device__ static uint32_t one(uint32_t bits, float scale) {
    float x = decode1<S>(bits);
    if constexpr (kScaled) x = __fmul_rn(x, scale);
    return encode1<D>(x);
  }

  __device__ static void step(const uint32_t (&s)[SB / 4], float scale, uint32_t (&o)[OS / 4]) {
#pragma unroll
    for (int j = 0; j < KS / 2; ++j) {
      float2 f = decode2<S, SB / 4>(s, j);
      if constexpr (kScaled) {
        f.x = __fmul_rn(f.x, scale);
        f.y = __fmul_rn(f.y, scale);
      }
      if constexpr (D == D_F32) {
        o[2 * j] = encode1<D_F32>(f.x);
        o[2 * j + 1] = encode1<D_F32>(f.y);
      } else {
        o[j] = encode2_16<D>(f);
      }
    }
  }
};

struct CopyBytes {
  static constexpr int SI = 1, SO = 1, SB = 16, KS = 16, OS = 16;
  __device__ static uint32_t one(uint32_t bits, float) { return bits; }
  __device__ static void step(const uint32_t (&s)[4], float, uint32_t (&o)[4]) {
    o[0] = s[0]; o[1] = s[1]; o[2] = s[2]; o[3] = s[3];
  }
};

// Two builds of the kernel share all code but the unroll depth (lane steps
// per batch for 16-, 8- and 4-byte source steps) and the register budget:
//  - StreamCfg: about 64 source bytes in flight per lane, <= 64 registers;
//    for checkpoints of large tensors, run at 3 blocks per SM;
//  - LatencyCfg: half the depth, <= 40 registers (6 blocks per SM); for
//    many small tensors, where per-piece latency dominates and more resident
//    warps hide it.
#ifndef ST_STREAM_U16
#define ST_STREAM_U16 4
#endif
#ifndef ST_STREAM_U8
#define ST_STREAM_U8 8
#endif
#ifndef ST_STREAM_U4
#define ST_STREAM_U4 16
#endif
struct StreamCfg {
  static constexpr int kU16 = ST_STREAM_U16, kU8 = ST_STREAM_U8, kU4 = ST_STREAM_U4;
};
// Compile-time tuning knobs for the latency build (defaults measured best).
#ifndef ST_LAT_U16
#define ST_LAT_U16 2
#endif
#ifndef ST_LAT_U8
#define ST_LAT_U8 4
#endif
#ifndef ST_LAT_U4
#define ST_LAT_U4 8
#endif
#ifndef ST_LAT_MIN_BLOCKS
#define ST_LAT_MIN_BLOCKS 6
#endif
struct LatencyCfg {
  static constexpr int kU16 = ST_LAT_U16, kU8 = ST_LAT_U8, kU4 = ST_LAT_U4;
};

template <class Cfg, class CV>
struct Unroll {
  static constexpr int value = CV::SB == 16 ? Cfg::kU16 : CV::SB == 8 ? Cfg::kU8 : Cfg::kU4;
};

// ------------------------------------------------------------- data moves

// Read-only loads of N 32-bit words (N = 1, 2, 4) from an N*4-aligned address,
// kept in program order with the other batch loads.
template <int N>
__device__ __forceinline__ void ldw(const uint8_t *p, uint32_t (&v)[N]) {
  if constexpr (N == 4) {
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]) : "l"(p));
  } else if constexpr (N == 2) {
    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v[0]), "=r"(v[1]) : "l"(p));
  } else {
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v[0]) : "l"(p));
  }
}

__device__ __forceinline__ uint4 ld16(const uint8_t *p) {
  uint32_t v[4];
  ldw<4>(p, v);
  return make_uint4(v[0], v[1], v[2], v[3]);
}

// N source words starting at byte offset r (1 .. 4N-1) of the 2N-word window
// {a, b}: drop whole words (r / 4), then funnel-shift by 8 * (r % 4).
template <int N>
__device__ __forceinline__ void realign(const uint32_t (&a)[N], const uint32_t (&b)[N], uint32_t r,
                                        uint32_t (&s)[N]) {
  uint32_t w[N + 1];
#pragma unroll
  for (int i = 0; i < N; ++i) w[i] = a[i];
  w[N] = b[0];
  if constexpr (N == 4) {
    if (r & 8) { w[0] = a[2]; w[1] = a[3]; w[2] = b[0]; w[3] = b[1]; w[4] = b[2]; }
    if (r & 4) { w[0] = w[1]; w[1] = w[2]; w[2] = w[3]; w[3] = w[4]; w[4] = (r & 8) ? b[3] : b[1]; }
  } else if constexpr (N == 2) {
    if (r & 4) { w[0] = a[1]; w[1] = b[0]; w[2] = b[1]; }
  }
  const uint32_t sh = (r & 3) * 8;
#pragma unroll
  for (int i = 0; i < N; ++i) s[i] = __funnelshift_r(w[i], w[i + 1], sh);
}

template <int NW>
__device__ __forceinline__ void store_out(uint8_t *p, const uint32_t (&o)[NW]) {
  if constexpr (NW == 2) {
    *reinterpret_cast<uint2 *>(p) = make_uint2(o[0], o[1]);
  } else if constexpr (NW == 4) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(o[0], o[1], o[2], o[3]);
  } else {
    *reinterpret_cast<uint4 *>(p) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4 *>(p + 16) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

template <class CV, bool kMis>
__device__ __forceinline__ void do_step(uint8_t *dbase, uint64_t c, const uint32_t (&a)[CV::SB / 4],
                                        const uint32_t (&b)[CV::SB / 4], uint32_t r, float scale) {
  constexpr int N = CV::SB / 4;
  uint32_t s[N];
  if constexpr (kMis) {
    realign<N>(a, b, r, s);
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) s[i] = a[i];
  }
  uint32_t o[CV::OS / 4];
  CV::step(s, scale, o);
  store_out<CV::OS / 4>(dbase + c * CV::OS, o);
}

// The word after a lane's step window is the next lane's first word; lane 31
// (and the lane of the last step) loads it itself.
template <int N>
__device__ __forceinline__ void next_words(const uint32_t (&a)[N], uint32_t (&b)[N], bool load_own,
                                           const uint8_t *p) {
#pragma unroll
  for (int i = 0; i < N; ++i) b[i] = __shfl_down_sync(0xFFFFFFFFu, a[i], 1);
  if (load_own) ldw<N>(p, b);
}

// Vector body over lane steps [0, nst): step c's SB bytes start at byte r of
// the SB-aligned word sbase + SB c (r == 0 when not kMis).  Every lane runs
// the same number of iterations (shuffles need the whole warp).
// One batch of U lane steps: issue every load, then convert and store.
template <class CV, int U>
__device__ __forceinline__ void load_batch(const uint8_t *sbase, uint64_t base, uint32_t lane,
                                           uint32_t (&a)[U][CV::SB / 4]) {
#pragma unroll
  for (int u = 0; u < U; ++u) ldw<CV::SB / 4>(sbase + (base + 32 * u + lane) * CV::SB, a[u]);
}

template <class CV, bool kMis, int U>
__device__ __forceinline__ void process_batch(const uint8_t *sbase, uint32_t r, uint8_t *dbase, uint64_t base,
                                              float scale, uint32_t lane, const uint32_t (&a)[U][CV::SB / 4]) {
  constexpr int N = CV::SB / 4;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const uint64_t c = base + 32 * u + lane;
    if constexpr (kMis) {
      uint32_t b[N];
      next_words<N>(a[u], b, lane == 31, sbase + (c + 1) * CV::SB);
      do_step<CV, true>(dbase, c, a[u], b, r, scale);
    } else {
      do_step<CV, false>(dbase, c, a[u], a[u], r, scale);
    }
  }
}

// Vector body over lane steps [0, nst): step c's SB bytes start at byte r of
// the SB-aligned word sbase + SB c (r == 0 when not kMis).  Every lane runs
// the same number of iterations (shuffles need the whole warp).
template <class Cfg, class CV, bool kMis>
__device__ __forceinline__ void body(const uint8_t *sbase, uint32_t r, uint8_t *dbase, uint64_t nst, float scale,
                                     uint32_t lane) {
  constexpr int U = Unroll<Cfg, CV>::value;
  constexpr int N = CV::SB / 4;
  constexpr uint64_t B = 32 * U;
  const uint64_t nb = nst / B;  // full batches
  for (uint64_t i = 0; i < nb; ++i) {
    uint32_t x[U][N];
    load_batch<CV, U>(sbase, i * B, lane, x);
    process_batch<CV, kMis, U>(sbase, r, dbase, i * B, scale, lane, x);
  }
  for (uint64_t base = nb * B; base < nst; base += 32) {
    const uint64_t c = base + lane;
    const bool valid = c < nst;
    uint32_t a[N];
#pragma unroll
    for (int i = 0; i < N; ++i) a[i] = 0;
    if (valid) ldw<N>(sbase + c * CV::SB, a);
    uint32_t b[N];
    if constexpr (kMis) next_words<N>(a, b, valid && (lane == 31 || c + 1 == nst), sbase + (c + 1) * CV::SB);
    if (valid) do_step<CV, kMis>(dbase, c, a, kMis ? b : a, r, scale);
  }
}

// Elements [0, head) and [tail, n) one per lane, with byte loads (any source
// alignment); one loop serves both ends so each class has one copy of it.
template <class CV>
__device__ __forceinline__ void scalar_ends(const uint8_t *src, uint8_t *dst, uint64_t head, uint64_t tail,
                                            uint64_t n, float scale, uint32_t lane) {
  const uint64_t count = head + (n - tail);
  for (uint64_t i = lane; i < count; i += 32) {
    const uint64_t e = i < head ? i : tail + (i - head);
    const uint8_t *p = src + e * CV::SI;
    uint32_t bits = 0;
#pragma unroll
    for (int i = 0; i < CV::SI; ++i) bits |= static_cast<uint32_t>(p[i]) << (8 * i);
    const uint32_t y = CV::one(bits, scale);
    uint8_t *q = dst + e * CV::SO;
    if constexpr (CV::SO == 1) *q = static_cast<uint8_t>(y);
    else if constexpr (CV::SO == 2) *reinterpret_cast<uint16_t *>(q) = static_cast<uint16_t>(y);
    else *reinterpret_cast<uint32_t *>(q) = y;
  }
}

template <class Cfg, class CV>
__device__ __forceinline__ void run_piece(const uint8_t *data, uint64_t data_bytes, const uint8_t *src, uint8_t *dst,
                                          uint64_t n, float scale, uint32_t lane) {
  constexpr int KS = CV::KS, SB = CV::SB;
  constexpr int A = CV::OS;  // destination alignment of the vector body (8 or 16)
  uint64_t head = ((A - (reinterpret_cast<uintptr_t>(dst) & (A - 1))) & (A - 1)) / CV::SO;
  if (head > n) head = n;
  uint64_t nst = (n - head) / KS;
  uintptr_t sa = reinterpret_cast<uintptr_t>(src + head * CV::SI);
  const uint32_t r = static_cast<uint32_t>(sa & (SB - 1));
  if (r && nst) {
    // Keep every 2*SB-byte window inside the data section.
    const uintptr_t lo = reinterpret_cast<uintptr_t>(data), hi = lo + data_bytes;
    if ((sa & ~uintptr_t(SB - 1)) < lo) {
      head += KS;
      --nst;
      sa += SB;
    }
    if (nst && (sa & ~uintptr_t(SB - 1)) + SB * nst + SB > hi) --nst;
  }
  const uint64_t tail = head + nst * KS;
  if (head || tail < n) scalar_ends<CV>(src, dst, head, tail, n, scale, lane);
  if (nst) {
    const uint8_t *sbase = reinterpret_cast<const uint8_t *>(sa & ~uintptr_t(SB - 1));
    uint8_t *dbase = dst + head * CV::SO;
    if (r) body<Cfg, CV, true>(sbase, r, dbase, nst, scale, lane);
    else body<Cfg, CV, false>(sbase, 0, dbase, nst, scale, lane);
  }
}

// Binary32 from 4 little-endian bytes at any alignment.
__device__ __forceinline__ float load_f32_le(const uint8_t *p) {
  return __uint_as_float(static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 8) |
                         (static_cast<uint32_t>(p[2]) << 16) | (static_cast<uint32_t>(p[3]) << 24));
}

__device__ __forceinline__ Piece load_piece(const Piece *p) {
  const uint4 *q = reinterpret_cast<const uint4 *>(p);
  const uint4 x = ld16(reinterpret_cast<const uint8_t *>(q));
  const uint4 y = ld16(reinterpret_cast<const uint8_t *>(q + 1));
  const uint4 z = ld16(reinterpret_cast<const uint8_t *>(q + 2));
  Piece pc;
  pc.src = (static_cast<uint64_t>(x.y) << 32) | x.x;
  pc.dst = (static_cast<uint64_t>(x.w) << 32) | x.z;
  pc.scale = (static_cast<uint64_t>(y.y) << 32) | y.x;
  pc.count = y.z;
  pc.out_cls = y.w;
  pc.rows = z.x;
  pc.pad = z.y;
  pc.pitch = (static_cast<uint64_t>(z.w) << 32) | z.z;
  return pc;
}

// The runs of a piece, one after the other (one run unless an inner
// dimension of the output is sliced).
template <class Cfg, class CV>
__device__ __forceinline__ void run_rows(const LaunchArgs &a, const volatile Piece *sp, uint8_t *dst, float scale,
                                         uint32_t lane) {
  // The piece's fields are re-read from its staged copy in shared memory for
  // every run (volatile), so no descriptor state stays live in registers
  // across run_piece.
  for (uint32_t r = 0; r < sp->rows; ++r) {
    const uint64_t cnt = sp->count;
    run_piece<Cfg, CV>(a.data, a.data_bytes, a.data + sp->src + r * sp->pitch, dst + r * cnt * CV::SO, cnt, scale,
                       lane);
  }
}

// Per-warp staging of up to 32 pieces: descriptor, destination and scale.
struct Staged {
  Piece piece[32];
  uint8_t *dst[32];
  float scale[32];
};

__device__ __forceinline__ void release_claims(const LaunchArgs &a, uint32_t lane);
// A claim takes about (pieces left to claim) / (kClaimSpread * warps) pieces,
// at least one and at most 32: larger claims early, single pieces at the end.
constexpr uint32_t kClaimSpread = 8;

// L2 prefetch of the 16-byte-aligned interior of [p, p + bytes).
__device__ __forceinline__ void l2_prefetch(const void *p, uint64_t bytes) {
  uintptr_t lo = (reinterpret_cast<uintptr_t>(p) + 15) & ~uintptr_t(15);
  const uintptr_t hi = (reinterpret_cast<uintptr_t>(p) + bytes) & ~uintptr_t(15);
  while (lo < hi) {
    const uint32_t n = static_cast<uint32_t>(hi - lo < 65536 ? hi - lo : 65536);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(lo), "r"(n) : "memory");
    lo += n;
  }
}
__device__ __forceinline__ void prefetch_inputs(const LaunchArgs &a) {
  if (threadIdx.x != 0 || a.pf_data_bytes == 0) return;
  if (blockIdx.x == 0) {
    l2_prefetch(a.pf_table, a.pf_table_bytes);
    l2_prefetch(a.dst, a.pf_dst_bytes);
  }
  const uint64_t slice = (a.pf_data_bytes + gridDim.x - 1) / gridDim.x;
  const uint64_t b0 = a.pf_data_bytes < slice * blockIdx.x ? a.pf_data_bytes : slice * blockIdx.x;
  l2_prefetch(a.data + a.pf_data_off + b0, slice < a.pf_data_bytes - b0 ? slice : a.pf_data_bytes - b0);
}

template <class Cfg>
__device__ __forceinline__ void materialize_body(const LaunchArgs &a) {
  __shared__ Staged stage[kWarpsPerBlock];
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t wib = threadIdx.x >> 5;
  const uint32_t w = blockIdx.x * kWarpsPerBlock + wib;
  prefetch_inputs(a);
  if (w >= a.workers) return;
  const uint32_t p0 = a.parts[w], p1 = a.parts[w + 1];
  const uint32_t dyn0 = a.parts[a.workers], dtotal = a.claim_end - dyn0;
  const uint32_t spread = kClaimSpread * a.workers;
  Staged &st = stage[wib];
  // Own pieces [p0, p1) in batches of 32, then batches claimed from the tail
  // [dyn0, dyn0 + dtotal); each claim is asked for one batch ahead.
  uint32_t next_at = 0, next_k = 0;  // lane 0: the claim in flight
  bool claiming = false;
  auto start_claim = [&](uint32_t from) {
    if (lane == 0) {
      const uint32_t left = from < dtotal ? dtotal - from : 0;
      next_k = max(1u, min(32u, left / spread));
      next_at = atomicAdd(a.claim, next_k);
    }
    claiming = true;
  };
  uint32_t base = p0;
  if (p0 == p1 && dtotal) start_claim(0);
  for (;;) {
    uint32_t n;
    if (base < p1) {
      n = min(32u, p1 - base);
      if (base + n == p1 && dtotal) start_claim(0);
    } else {
      if (!claiming) break;
      claiming = false;
      const uint32_t at = __shfl_sync(0xFFFFFFFFu, next_at, 0), k = __shfl_sync(0xFFFFFFFFu, next_k, 0);
      if (at >= dtotal) break;
      base = dyn0 + at;
      n = min(k, dtotal - at);
      start_claim(at + k);
    }
    // Lane i fetches piece base+i, then its destination and scale: two
    // dependent round trips shared by up to 32 pieces.
    __syncwarp();
    if (lane < n) {
      const Piece pc = load_piece(a.pieces + base + lane);
      const uint32_t out = pc.out_cls >> kClsBits, cls = pc.out_cls & ((1u << kClsBits) - 1);
      float scale = 1.0f;
      if (cls >= CLS_E4M3_BF16) {
        if (a.scales) scale = a.scales[out];
        else if (pc.scale != kNoScale) scale = load_f32_le(a.data + pc.scale);
      }
      st.piece[lane] = pc;
      st.dst[lane] = static_cast<uint8_t *>(a.dst[out]);
      st.scale[lane] = scale;
    }
    __syncwarp();
    for (uint32_t i = 0; i < n; ++i) {
      const uint32_t cls = st.piece[i].out_cls & ((1u << kClsBits) - 1);
      uint8_t *dst = st.dst[i];
      const float scale = st.scale[i];
      const int so = cls_out_size(cls);
      if (dst == nullptr || (reinterpret_cast<uintptr_t>(dst) & (so - 1))) {
        if (lane == 0) atomicOr(a.err, kErrBadDst);
        continue;
      }
      dst += st.piece[i].dst;
      switch (cls) {
        case CLS_COPY: run_rows<Cfg, CopyBytes>(a, &st.piece[i], dst, scale, lane); break;
        case CLS_F32_BF16: run_rows<Cfg, Conv<S_F32, D_BF16>>(a, &st.piece[i], dst, scale, lane); break;
        case CLS_F32_F16: run_rows<Cfg, Conv<S_F32, D_F16>>(a, &st.piece[i], dst, scale, lane); break;
        case CLS_F16_BF16: run_rows<Cfg, Conv<S_F16, D_BF16>>(a, &st.piece[i], dst, scale, lane); break;
        case CLS_F16_F32: run_rows<Cfg, Conv<S_F16, D_F32>>(a, &st.piece[i], dst, scale, lane); break;
        case CLS_BF16_F16: run_rows<Cfg, Conv<S_BF16, D_F16>>(a, &st.piece[i], dst, scale, lane); break;
        case CLS_BF16_F32: run_rows<Cfg, Conv<S_BF16, D_F32>>(a, &st.piece[i], dst, scale, lane); break;
        case CLS_E4M3_BF16: run_rows<Cfg, Conv<S_E4M3, D_BF16>>(a, &st.piece[i], dst, scale, lane); break;
        case CLS_E4M3_F16: run_rows<Cfg, Conv<S_E4M3, D_F16>>(a, &st.piece[i], dst, scale, lane); break;
        case CLS_E4M3_F32: run_rows<Cfg, Conv<S_E4M3, D_F32>>(a, &st.piece[i], dst, scale, lane); break;
        case CLS_E5M2_BF16: run_rows<Cfg, Conv<S_E5M2, D_BF16>>(a, &st.piece[i], dst, scale, lane); break;
        case CLS_E5M2_F16: run_rows<Cfg, Conv<S_E5M2, D_F16>>(a, &st.piece[i], dst, scale, lane); break;
        case CLS_E5M2_F32: run_rows<Cfg, Conv<S_E5M2, D_F32>>(a, &st.piece[i], dst, scale, lane); break;
        default:
          if (lane == 0) atomicOr(a.err, kErrBadDst);
      }
    }
    base += n;
  }
  if (dtotal) release_claims(a, lane);
}

__global__ void __launch_bounds__(kThreads) materialize_stream(const LaunchArgs a) { materialize_body<StreamCfg>(a); }

__global__ void __launch_bounds__(kThreads, ST_LAT_MIN_BLOCKS) materialize_latency(const LaunchArgs a) {
  materialize_body<LatencyCfg>(a);
}

// ------------------------------------------------------------ the TMA build
//
// Source bytes travel through shared memory instead of registers: each warp
// cuts its pieces into segments of up to kSeg source bytes and keeps kSlots
// of them in flight, each fetched by one bulk copy (cp.async.bulk, the TMA
// engine) into a slot of the warp's shared memory and tracked by an mbarrier.
// The bytes a warp has in flight no longer cost registers, so an SM keeps
// about kWarps * kSlots * kSeg bytes of reads outstanding however small the
// tensors are; the registers-only builds hold far less while a warp walks
// many small tensors one dependent round trip at a time.
//  - A bulk copy needs 16-byte aligned global and shared addresses and a
//    multiple of 16 bytes, so a segment is fetched as the aligned window
//    covering it, clipped to the 16-byte aligned interior of the data
//    section; the few elements outside that interior (only at the two ends
//    of the data section) are read with byte loads.  No byte outside the
//    data section is read.
//  - The consumer reads the window from shared memory: lane c takes source
//    step c (SB bytes) as two aligned words and realigns them by the
//    window's byte offset, converts, and stores one 16- or 8-byte vector;
//    elements before the first aligned destination vector or after the
//    last are converted one by one from shared memory.
//  - Piece descriptors arrive the same way, up to 32 at a time, one batch
//    ahead: first the warp's own pieces (its interleaved units), then pieces
//    of the plan's claimed tail, taken in source order from the launch's
//    claim word (a warp asks for the batch after next as it enters a batch,
//    so the answer is there when needed), so warps that run fast take more
//    and all finish together.  The last warp to finish zeroes the claim
//    words for the next launch.
//  - One warp is both producer and consumer, so a slot is refilled only
//    after the warp has finished reading it (program order, __syncwarp and
//    a proxy fence).  Every wait is bounded: a wait that gives up sets
//    kErrTimeout, waits (bounded) for the warp's copies still in flight and
//    ends the warp.
#ifndef ST_TMA_SEG
#define ST_TMA_SEG 2048
#endif
// Two shapes of the build: many small tensors run best with 4 slots per warp
// at 2 blocks per SM (deep per-warp queues); block-scaled weights, whose
// consumer is busier, with 2 slots at 3 blocks per SM (more warps to issue).
#ifndef ST_TMA_SLOTS
#define ST_TMA_SLOTS 4
#endif
#ifndef ST_TMA_MIN_BLOCKS
#define ST_TMA_MIN_BLOCKS 2
#endif
#ifndef ST_TMA_WIDE_SLOTS
#define ST_TMA_WIDE_SLOTS 2
#endif
#ifndef ST_TMA_WIDE_MIN_BLOCKS
#define ST_TMA_WIDE_MIN_BLOCKS 3
#endif
constexpr uint32_t kSeg = ST_TMA_SEG;
constexpr uint32_t kBatch = 32;  // piece descriptors fetched per bulk copy (one per lane)
constexpr uint32_t kSlotBytes = kSeg + 32;  // a clipped window is at most kSeg + 16 bytes
constexpr uint32_t kSpinLimit = 1u << 22;
static_assert(kSeg % 16 == 0 && kSeg >= 64, "segment size");

// One staged segment: a run of one piece, elements [0, len); elements
// [a, z) are in the slot, the rest are read with byte loads.
struct alignas(16) SegMeta {
  uint8_t *dst;         // output address of element 0
  const uint8_t *gsrc;  // data-section address of element 0
  uint32_t len;         // elements (bytes for CLS_COPY)
  uint32_t a, z;
  uint32_t off;         // slot offset of element a
  float scale;          // per-tensor scale (fp8), or the NVFP4 global scale
  uint32_t cls;
  // Block-scaled segments: the scale of the block holding element column
  // col0 is at sptr (the slot's scale area, or the data section itself when
  // the scales sit at an unaligned end of it); blocks are 1 << bcs columns.
  uint32_t col0, bcs;
  const uint8_t *sptr;
  uint64_t pad;
};
static_assert(sizeof(SegMeta) == 64, "segment metadata: four 16-byte words");

// Segment metadata moves between the producer and the consumer as 16-byte
// shared-memory words (the fourth only for block-scaled segments).
__device__ __forceinline__ void put_meta(SegMeta *m, const SegMeta &v, bool quant) {
  const uint4 *src = reinterpret_cast<const uint4 *>(&v);
  uint4 *dst = reinterpret_cast<uint4 *>(m);
  dst[0] = src[0];
  dst[1] = src[1];
  dst[2] = src[2];
  if (quant) dst[3] = src[3];
}
__device__ __forceinline__ SegMeta get_meta(const SegMeta *m) {
  SegMeta v;
  const uint4 *src = reinterpret_cast<const uint4 *>(m);
  uint4 *dst = reinterpret_cast<uint4 *>(&v);
  dst[0] = src[0];
  dst[1] = src[1];
  dst[2] = src[2];
  if (cls_quant(v.cls)) dst[3] = src[3];
  return v;
}

// A segment of a block-scaled weight brings at most this many bytes of block
// scales (the producer shortens the segment to fit), fetched with the
// segment into the slot's scale area: 256 NVFP4 scales cover a whole 2 KiB
// segment; block-FP8 segments are held to kQscMax F32 scales, which the
// consumer decodes into the warp's table.
constexpr uint32_t kScalePayload = 256;
constexpr uint32_t kScaleBytes = kScalePayload + 32;
constexpr uint32_t kQscMax = 32;

template <int kSlots>
struct alignas(128) WarpSmem {
  uint8_t buf[kSlots][kSlotBytes];
  uint8_t sbuf[kSlots][kScaleBytes];
  Piece desc[2][kBatch];
  uint8_t *dstp[2][kBatch];
  float scl[2][kBatch];
  SegMeta meta[kSlots];
  uint64_t bar[kSlots];
  uint64_t dbar[2];
  float qsc[kQscMax];  // the consumed block-FP8 segment's scales as binary32 (any alignment in the slot)
};
static_assert(sizeof(WarpSmem<ST_TMA_SLOTS>) * kWarpsPerBlock * ST_TMA_MIN_BLOCKS <= 226 * 1024, "blocks per SM fit");
static_assert(sizeof(WarpSmem<ST_TMA_WIDE_SLOTS>) * kWarpsPerBlock * ST_TMA_WIDE_MIN_BLOCKS <= 226 * 1024,
              "blocks per SM fit");
static_assert(offsetof(WarpSmem<ST_TMA_SLOTS>, sbuf) % 16 == 0 && offsetof(WarpSmem<ST_TMA_WIDE_SLOTS>, sbuf) % 16 == 0 &&
                  kScaleBytes % 16 == 0, "scale bulk-copy destinations");
static_assert(offsetof(WarpSmem<ST_TMA_SLOTS>, desc) % 16 == 0 && offsetof(WarpSmem<ST_TMA_WIDE_SLOTS>, desc) % 16 == 0 &&
                  kSlotBytes % 16 == 0, "bulk-copy destinations");

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void proxy_fence() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// Lane 0: one arrival that also expects `bytes` of copies, then the copy.
__device__ __forceinline__ void bulk_load(void *sdst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
  if (bytes == 0) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
    return;
  }
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(sdst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
// Lane 0: one arrival expecting `bytes`, then the copies that deliver them.
__device__ __forceinline__ void mbar_expect(uint64_t *bar, uint32_t bytes) {
  if (bytes == 0) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
    return;
  }
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_copy(void *sdst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(sdst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  for (uint32_t it = 0; it < kSpinLimit; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}

template <int N>
__device__ __forceinline__ void lds(const uint8_t *p, uint32_t (&v)[N]) {
  if constexpr (N == 4) {
    const uint4 x = *reinterpret_cast<const uint4 *>(p);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  } else if constexpr (N == 2) {
    const uint2 x = *reinterpret_cast<const uint2 *>(p);
    v[0] = x.x; v[1] = x.y;
  } else {
    v[0] = *reinterpret_cast<const uint32_t *>(p);
  }
}

template <class CV>
__device__ __forceinline__ void convert_one(const uint8_t *p, uint8_t *q, float scale) {
  uint32_t bits = 0;
#pragma unroll
  for (int i = 0; i < CV::SI; ++i) bits |= static_cast<uint32_t>(p[i]) << (8 * i);
  const uint32_t y = CV::one(bits, scale);
  if constexpr (CV::SO == 1) *q = static_cast<uint8_t>(y);
  else if constexpr (CV::SO == 2) *reinterpret_cast<uint16_t *>(q) = static_cast<uint16_t>(y);
  else *reinterpret_cast<uint32_t *>(q) = y;
}

// A staged segment: elements [a, z) from the slot (element a at slot offset
// `off`), the rest from global with byte loads.
template <class CV>
__device__ __forceinline__ void consume_seg(const uint8_t *buf, const SegMeta &m, uint32_t lane) {
  constexpr int SI = CV::SI, SO = CV::SO, SB = CV::SB, KS = CV::KS, OS = CV::OS, N = SB / 4;
  const float scale = m.scale;
  uint8_t *const dst = m.dst;
  const uint32_t len = m.len, off = m.off, a = m.a, z = m.z;
  const uint32_t edge = a + (len - z);  // elements outside the staged window: only at the data section's ends
  if (edge) {
    for (uint32_t t = lane; t < edge; t += 32) {
      const uint32_t e = t < a ? t : z + (t - a);
      convert_one<CV>(m.gsrc + static_cast<uint64_t>(e) * SI, dst + static_cast<uint64_t>(e) * SO, scale);
    }
  }
  const uint32_t n = z - a;
  const uint8_t *sp = buf + off;
  uint8_t *dp = dst + static_cast<uint64_t>(a) * SO;
  uint32_t h = static_cast<uint32_t>(((OS - (reinterpret_cast<uintptr_t>(dp) & (OS - 1))) & (OS - 1)) / SO);
  if (h > n) h = n;
  const uint32_t nst = (n - h) / KS, t0 = h + nst * KS;
  const uint32_t ends = h + (n - t0);
  for (uint32_t t = lane; t < ends; t += 32) {
    const uint32_t e = t < h ? t : t0 + (t - h);
    convert_one<CV>(sp + e * SI, dp + e * SO, scale);
  }
  const uint32_t q = off + h * SI, r = q & (SB - 1);
  const uint8_t *wb = buf + (q - r);
  uint8_t *db = dp + h * SO;
  for (uint32_t c = lane; c < nst; c += 32) {
    uint32_t x[N], sv[N];
    lds<N>(wb + c * SB, x);
    if (r) {
      uint32_t y[N];
      lds<N>(wb + (c + 1) * SB, y);
      realign<N>(x, y, r, sv);
    } else {
#pragma unroll
      for (int i = 0; i < N; ++i) sv[i] = x[i];
    }
    uint32_t o[OS / 4];
    CV::step(sv, scale, o);
    store_out<OS / 4>(db + c * OS, o);
  }
}

// ----------------------------------------------------- block-scaled weights

constexpr int S_NV = 100;  // NVFP4 source marker for QConv

// OCP MX E2M1: magnitudes x 2 of codes 0..7 are 0, 1, 2, 3, 4, 6, 8, 12
// (nibbles of 0xC8643210); the sign is bit 3.  Exact in binary32.
__device__ __forceinline__ float e2m1_value(uint32_t nib) {
  const float mag = static_cast<float>((0xC8643210u >> ((nib & 7u) * 4u)) & 15u) * 0.5f;
  return __uint_as_float(__float_as_uint(mag) | ((nib & 8u) << 28));
}

// Block scale k of a segment as binary32: an F32 block scale (block FP8,
// any alignment), or an E4M3 block scale times the global scale g (NVFP4).
template <bool kNv>
__device__ __forceinline__ float decode_scale(const uint8_t *sptr, uint32_t k, float g) {
  if constexpr (kNv) {
    return __fmul_rn(decode1<S_E4M3>(sptr[k]), g);
  } else {
    const uint8_t *p = sptr + 4 * k;
    return __uint_as_float(static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 8) |
                           (static_cast<uint32_t>(p[2]) << 16) | (static_cast<uint32_t>(p[3]) << 24));
  }
}

// A block-scaled class: counted units are bytes (an fp8 element, or two
// NVFP4 elements); a lane step reads SB bytes and writes one 16-byte vector
// (two for NVFP4 to F32).
template <int S, int D>
struct QConv {
  static constexpr bool kNv = S == S_NV;
  static constexpr int EPU = kNv ? 2 : 1;             // elements per unit
  static constexpr int ES = DstInfo<D>::kSize;        // output element size
  static constexpr int SO = EPU * ES;
  static constexpr int SB = kNv ? 4 : (ES == 4 ? 4 : 8);
  static constexpr int KS = SB, OS = KS * SO, KE = KS * EPU;

  // Block FP8: whether any element of the step could give a NaN product
  // (E4M3: a NaN code, the low seven bits all set; E5M2: exponent all ones,
  // infinity included since infinity times a zero scale is NaN),
  // byte-parallel on the words.
  __device__ static bool has_nan(const uint32_t (&w)[SB / 4]) {
    uint32_t any = 0;
#pragma unroll
    for (int i = 0; i < SB / 4; ++i) {
      const uint32_t t = w[i] & 0x7F7F7F7Fu;
      any |= (t + (S == S_E4M3 ? 0x01010101u : 0x04040404u)) & 0x80808080u;
    }
    return any != 0;
  }

  // Elements 2j, 2j+1 of a step's words as binary32 (NVFP4: one hardware
  // e2m1x2 -> f16x2 conversion, exact, then f16 -> f32, exact).
  __device__ static float2 pair(const uint32_t (&w)[SB / 4], int j) {
    if constexpr (kNv) {
      const uint16_t byte = static_cast<uint16_t>((w[j >> 2] >> (8 * (j & 3))) & 0xFFu);
      uint32_t h2;
      asm("{\n .reg .b8 t;\n cvt.u8.u16 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(h2) : "h"(byte));
      __half2_raw r;
      r.x = static_cast<unsigned short>(h2 & 0xFFFFu);
      r.y = static_cast<unsigned short>(h2 >> 16);
      return __half22float2(__half2(r));
    } else {
      return decode2<S, SB / 4>(w, j);
    }
  }
  // One unit at p (any memory) to q; `col` = its first element's column
  // relative to the segment's first block; the scales are the table qsc
  // (block FP8) or the E4M3 bytes at sptr times g (NVFP4).
  __device__ static void one(const uint8_t *p, uint8_t *q, uint32_t col, uint32_t bcs, const float *qsc,
                             const uint8_t *sptr, float g) {
    const uint32_t byte = *p;
#pragma unroll
    for (int k = 0; k < EPU; ++k) {
      const float v = kNv ? e2m1_value(k ? byte >> 4 : byte & 15u) : decode1<S>(byte);
      const uint32_t blk = (col + k) >> bcs;
      const float sc = kNv ? decode_scale<true>(sptr, blk, g) : qsc[blk];
      const uint32_t y = encode1<D>(__fmul_rn(v, sc));
      if constexpr (ES == 2) reinterpret_cast<uint16_t *>(q)[k] = static_cast<uint16_t>(y);
      else reinterpret_cast<uint32_t *>(q)[k] = y;
    }
  }
  // KE elements; elements [0, kb) take scale lo, the rest hi (a step crosses
  // at most one block boundary: blocks hold >= 16 elements).  kClean: no
  // product can be NaN (NVFP4 values are finite and the segment's scales
  // are finite), so the NaN canonicalization is skipped.
  template <bool kClean>
  __device__ static void step(const uint32_t (&w)[SB / 4], float lo, float hi, uint32_t kb,
                              uint32_t (&o)[OS / 4]) {
#pragma unroll
    for (int j = 0; j < KE / 2; ++j) {
      float2 f = pair(w, j);
      f.x = __fmul_rn(f.x, static_cast<uint32_t>(2 * j) < kb ? lo : hi);
      f.y = __fmul_rn(f.y, static_cast<uint32_t>(2 * j + 1) < kb ? lo : hi);
      if constexpr (D == D_F32) {
        o[2 * j] = kClean ? __float_as_uint(f.x) : encode1<D_F32>(f.x);
        o[2 * j + 1] = kClean ? __float_as_uint(f.y) : encode1<D_F32>(f.y);
      } else if constexpr (kClean && D == D_BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(f.x, f.y);
        o[j] = *reinterpret_cast<uint32_t *>(&v);
      } else if constexpr (kClean) {
        __half2 v = __floats2half2_rn(f.x, f.y);
        o[j] = *reinterpret_cast<uint32_t *>(&v);
      } else {
        o[j] = encode2_16<D>(f);
      }
    }
  }
};

// A block-scaled segment: its block scales are decoded once into the warp's
// table, then elements [a, z) come from the slot and the rest from global.
template <class QV>
__device__ __forceinline__ void consume_quant(const uint8_t *buf, const SegMeta &m, float *qsc, uint32_t lane) {
  constexpr int SO = QV::SO, SB = QV::SB, KS = QV::KS, OS = QV::OS, N = SB / 4, EPU = QV::EPU;
  uint8_t *const dst = m.dst;
  const uint8_t *const gsrc = m.gsrc;
  const uint32_t len = m.len, off = m.off, a = m.a, z = m.z, bcs = m.bcs;
  const uint32_t cbase = m.col0 & ((1u << bcs) - 1);  // column of unit 0 relative to its block's start
  const uint32_t nblk = ((cbase + len * EPU - 1) >> bcs) + 1;
  const uint8_t *const sptr = m.sptr;
  const float g = m.scale;
  // Block FP8: the F32 scales (any alignment) decoded once into the table.
  // NVFP4: scales are decoded per step from the slot; here only checked.
  bool finite = true;
  for (uint32_t k = lane; k < nblk; k += 32) {
    const float v = decode_scale<QV::kNv>(sptr, k, g);
    finite = finite && isfinite(v);
    if constexpr (!QV::kNv) qsc[k] = v;
  }
  __syncwarp();
  // NVFP4: no product can be NaN when the scales are finite.  Block FP8: also
  // needs NaN-free elements, checked per step below.
  const bool clean = __all_sync(0xFFFFFFFFu, finite);
  auto scale_at = [&](uint32_t blk) -> float {
    if constexpr (QV::kNv) return decode_scale<true>(sptr, blk, g);
    else return qsc[blk];
  };
  const uint32_t edge = a + (len - z);
  for (uint32_t t = lane; t < edge; t += 32) {
    const uint32_t e = t < a ? t : z + (t - a);
    QV::one(gsrc + e, dst + static_cast<uint64_t>(e) * SO, cbase + e * EPU, bcs, qsc, sptr, g);
  }
  const uint32_t n = z - a;
  const uint8_t *sp = buf + off;
  uint8_t *dp = dst + static_cast<uint64_t>(a) * SO;
  uint32_t h = static_cast<uint32_t>(((OS - (reinterpret_cast<uintptr_t>(dp) & (OS - 1))) & (OS - 1)) / SO);
  // An NVFP4 unit is two elements (4 bytes of BF16/F16, 8 of F32) and a
  // destination is only aligned to the itemsize: at 2 mod 4 (4 mod 8) whole
  // units never reach vector alignment, so every unit is written element by
  // element.
  if (h > n || (reinterpret_cast<uintptr_t>(dp) & (SO - 1))) h = n;
  const uint32_t nst = (n - h) / KS, t0 = h + nst * KS;
  const uint32_t ends = h + (n - t0);
  for (uint32_t t = lane; t < ends; t += 32) {
    const uint32_t e = t < h ? t : t0 + (t - h);
    QV::one(sp + e, dp + e * SO, cbase + (a + e) * EPU, bcs, qsc, sptr, g);
  }
  const uint32_t q = off + h, r = q & (SB - 1);
  const uint8_t *wb = buf + (q - r);
  uint8_t *db = dp + h * SO;
  const uint32_t bc = 1u << bcs;
  const uint32_t col1 = cbase + (a + h) * EPU;  // the first step's first element, block-relative
  // Steps that start on a multiple of KE columns never cross a block boundary
  // (blocks are powers of two >= 16 >= KE): one scale per step.
  const uint32_t kb_all = (col1 & (QV::KE - 1)) == 0 ? static_cast<uint32_t>(QV::KE) : 0u;
  for (uint32_t c = lane; c < nst; c += 32) {
    const uint32_t col = col1 + c * KS * EPU;
    const uint32_t kb = kb_all ? kb_all : bc - (col & (bc - 1));
    const float lo = scale_at(col >> bcs);
    const float hi = kb < static_cast<uint32_t>(QV::KE) ? scale_at((col >> bcs) + 1) : lo;
    uint32_t x[N], sv[N];
    lds<N>(wb + c * SB, x);
    if (r) {
      uint32_t y[N];
      lds<N>(wb + (c + 1) * SB, y);
      realign<N>(x, y, r, sv);
    } else {
#pragma unroll
      for (int i = 0; i < N; ++i) sv[i] = x[i];
    }
    uint32_t o[OS / 4];
    bool fast = clean;
    if constexpr (!QV::kNv) fast = fast && __all_sync(__activemask(), !QV::has_nan(sv));
    if (kb_all) {
      if (fast) QV::template step<true>(sv, lo, lo, QV::KE, o);
      else QV::template step<false>(sv, lo, lo, QV::KE, o);
    } else {
      if (fast) QV::template step<true>(sv, lo, hi, kb, o);
      else QV::template step<false>(sv, lo, hi, kb, o);
    }
    store_out<OS / 4>(db + c * OS, o);
  }
}

// The codec types' lane steps are the ones the host describes (cls_step_*).
template <class CV, uint32_t C>
constexpr bool step_is() {
  return CV::SB == cls_step_src(C) && CV::KS == cls_step_units(C) && CV::OS == cls_step_out(C);
}
static_assert(step_is<CopyBytes, CLS_COPY>() && step_is<Conv<S_F32, D_BF16>, CLS_F32_BF16>() &&
                  step_is<Conv<S_F32, D_F16>, CLS_F32_F16>() && step_is<Conv<S_F16, D_BF16>, CLS_F16_BF16>() &&
                  step_is<Conv<S_F16, D_F32>, CLS_F16_F32>() && step_is<Conv<S_BF16, D_F16>, CLS_BF16_F16>() &&
                  step_is<Conv<S_BF16, D_F32>, CLS_BF16_F32>() && step_is<Conv<S_E4M3, D_BF16>, CLS_E4M3_BF16>() &&
                  step_is<Conv<S_E4M3, D_F16>, CLS_E4M3_F16>() && step_is<Conv<S_E4M3, D_F32>, CLS_E4M3_F32>() &&
                  step_is<Conv<S_E5M2, D_BF16>, CLS_E5M2_BF16>() && step_is<Conv<S_E5M2, D_F16>, CLS_E5M2_F16>() &&
                  step_is<Conv<S_E5M2, D_F32>, CLS_E5M2_F32>(),
              "per-tensor codec steps");
static_assert(step_is<QConv<S_E4M3, D_BF16>, CLS_QE4M3_BF16>() && step_is<QConv<S_E4M3, D_F16>, CLS_QE4M3_F16>() &&
                  step_is<QConv<S_E4M3, D_F32>, CLS_QE4M3_F32>() && step_is<QConv<S_E5M2, D_BF16>, CLS_QE5M2_BF16>() &&
                  step_is<QConv<S_E5M2, D_F16>, CLS_QE5M2_F16>() && step_is<QConv<S_E5M2, D_F32>, CLS_QE5M2_F32>() &&
                  step_is<QConv<S_NV, D_BF16>, CLS_NVFP4_BF16>() && step_is<QConv<S_NV, D_F16>, CLS_NVFP4_F16>() &&
                  step_is<QConv<S_NV, D_F32>, CLS_NVFP4_F32>(),
              "block-scaled codec steps");

__device__ __forceinline__ void consume_any(const uint8_t *buf, const SegMeta &m, float *qsc, uint32_t lane) {
  switch (m.cls) {
    case CLS_COPY: consume_seg<CopyBytes>(buf, m, lane); break;
    case CLS_F32_BF16: consume_seg<Conv<S_F32, D_BF16>>(buf, m, lane); break;
    case CLS_F32_F16: consume_seg<Conv<S_F32, D_F16>>(buf, m, lane); break;
    case CLS_F16_BF16: consume_seg<Conv<S_F16, D_BF16>>(buf, m, lane); break;
    case CLS_F16_F32: consume_seg<Conv<S_F16, D_F32>>(buf, m, lane); break;
    case CLS_BF16_F16: consume_seg<Conv<S_BF16, D_F16>>(buf, m, lane); break;
    case CLS_BF16_F32: consume_seg<Conv<S_BF16, D_F32>>(buf, m, lane); break;
    case CLS_E4M3_BF16: consume_seg<Conv<S_E4M3, D_BF16>>(buf, m, lane); break;
    case CLS_E4M3_F16: consume_seg<Conv<S_E4M3, D_F16>>(buf, m, lane); break;
    case CLS_E4M3_F32: consume_seg<Conv<S_E4M3, D_F32>>(buf, m, lane); break;
    case CLS_E5M2_BF16: consume_seg<Conv<S_E5M2, D_BF16>>(buf, m, lane); break;
    case CLS_E5M2_F16: consume_seg<Conv<S_E5M2, D_F16>>(buf, m, lane); break;
    case CLS_E5M2_F32: consume_seg<Conv<S_E5M2, D_F32>>(buf, m, lane); break;
    case CLS_QE4M3_BF16: consume_quant<QConv<S_E4M3, D_BF16>>(buf, m, qsc, lane); break;
    case CLS_QE4M3_F16: consume_quant<QConv<S_E4M3, D_F16>>(buf, m, qsc, lane); break;
    case CLS_QE4M3_F32: consume_quant<QConv<S_E4M3, D_F32>>(buf, m, qsc, lane); break;
    case CLS_QE5M2_BF16: consume_quant<QConv<S_E5M2, D_BF16>>(buf, m, qsc, lane); break;
    case CLS_QE5M2_F16: consume_quant<QConv<S_E5M2, D_F16>>(buf, m, qsc, lane); break;
    case CLS_QE5M2_F32: consume_quant<QConv<S_E5M2, D_F32>>(buf, m, qsc, lane); break;
    case CLS_NVFP4_BF16: consume_quant<QConv<S_NV, D_BF16>>(buf, m, qsc, lane); break;
    case CLS_NVFP4_F16: consume_quant<QConv<S_NV, D_F16>>(buf, m, qsc, lane); break;
    case CLS_NVFP4_F32: consume_quant<QConv<S_NV, D_F32>>(buf, m, qsc, lane); break;
    default: break;
  }
}

// Producer cursor over a warp's pieces: batch, piece in batch, run, element.
struct Cursor {
  uint32_t b, i, r, n;  // n = pieces in batch b
  uint32_t e;
};

// kInterior: compute per piece whether it lies inside the data section's
// aligned interior, so its segments skip the clipping arithmetic (measured:
// +2 % on many small tensors with the 4-slot shape; -1..3 % on the
// register-capped wide shape, which keeps the general path).
// The last warp of a launch to finish zeroes its claim words (every warp has
// made its last claim by then).  Launches without a claimed tail never touch
// them and skip this (its fence and atomic cost a warp about 1 us, the 16
// tiny tensors' launch 10 %).
__device__ __forceinline__ void release_claims(const LaunchArgs &a, uint32_t lane) {
  if (lane == 0) {
    __threadfence();
    if (atomicAdd(a.claim + 1, 1u) == a.workers - 1) {
      atomicExch(a.claim, 0u);
      atomicExch(a.claim + 1, 0u);
    }
  }
}

template <int kSlots, bool kInterior>
__device__ __forceinline__ void tma_body(const LaunchArgs &a, uint8_t *smem) {
  const uint32_t lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const uint32_t w = blockIdx.x * kWarpsPerBlock + wib;
  prefetch_inputs(a);
  if (w >= a.workers) return;
  WarpSmem<kSlots> &ws = reinterpret_cast<WarpSmem<kSlots> *>(smem)[wib];
  // The warp's own pieces [p0, p1), then pieces of the claimed tail
  // [dyn0, dyn0 + dtotal), in batches of at most kBatch.
  const uint32_t p0 = a.parts[w], p1 = a.parts[w + 1];
  const uint32_t dyn0 = a.parts[a.workers], dtotal = a.claim_end - dyn0;
  const uint32_t spread = kClaimSpread * a.workers;
  // The 4-slot build (kInterior) gets tail pieces of at most one segment
  // (the planner cuts them so); its warps claim two or more at a time.
  constexpr uint32_t kClaimMin = kInterior ? 2 : 1;
  uint32_t sp = p0;                // the next own piece not yet in a batch
  bool claiming = false;           // a claim has been made and not yet taken
  uint32_t next_at = 0, next_k = 0;  // lane 0: that claim
  auto start_claim = [&](uint32_t from) {  // claim about (left) / spread pieces, from = claimed so far
    if (lane == 0) {
      const uint32_t left = from < dtotal ? dtotal - from : 0;
      next_k = max(kClaimMin, min(kBatch, left / spread));
      next_at = atomicAdd(a.claim, next_k);
    }
    claiming = true;
  };
  // The next batch: own pieces first; the claim for the tail's first batch
  // goes out with the last own batch, and each claimed batch makes the next
  // claim, so a claim's answer is read one batch after it was asked for.
  auto next_batch = [&](uint32_t &start) -> uint32_t {
    if (sp < p1) {
      start = sp;
      const uint32_t n = min(kBatch, p1 - sp);
      sp += n;
      if (sp == p1 && dtotal) start_claim(0);
      return n;
    }
    if (!claiming) return 0;
    claiming = false;
    const uint32_t at = __shfl_sync(0xFFFFFFFFu, next_at, 0), k = __shfl_sync(0xFFFFFFFFu, next_k, 0);
    if (at >= dtotal) return 0;
    start = dyn0 + at;
    start_claim(at + k);
    return min(k, dtotal - at);
  };
  if (p0 == p1 && dtotal) start_claim(0);
  uint32_t bs0 = 0, bs1 = 0, bn0 = 0, bn1 = 0;  // the batches in the two descriptor slots
  bn0 = next_batch(bs0);
  if (bn0 == 0) {
    if (dtotal) release_claims(a, lane);
    return;
  }
  const uintptr_t lo16 = (reinterpret_cast<uintptr_t>(a.data) + 15) & ~uintptr_t(15);
  const uintptr_t hi16 = (reinterpret_cast<uintptr_t>(a.data) + a.data_bytes) & ~uintptr_t(15);

  auto issue_desc = [&](uint32_t bb) {  // lane 0
    bulk_load(ws.desc[bb & 1], a.pieces + ((bb & 1) ? bs1 : bs0),
              ((bb & 1) ? bn1 : bn0) * static_cast<uint32_t>(sizeof(Piece)), &ws.dbar[bb & 1]);
  };
  if (lane == 0) {
    for (int k = 0; k < kSlots; ++k) mbar_init(&ws.bar[k]);
    mbar_init(&ws.dbar[0]);
    mbar_init(&ws.dbar[1]);
    mbar_init_fence();
    issue_desc(0);
  }
  uint32_t dissued = 1, dseen = 0;  // descriptor batches fetched / waited for
  bool later = true;                // a batch follows the one entered last (known once it is entered)
  __syncwarp();

  // Waits for descriptor batch b, resolves its destinations and scales, and
  // fetches batch b + 1 into the other descriptor slot.
  auto enter_batch = [&](uint32_t b) -> bool {
    if (!mbar_wait(&ws.dbar[b & 1], (b >> 1) & 1)) return false;
    dseen = b + 1;
    const uint32_t cnt = (b & 1) ? bn1 : bn0;
    if (lane < cnt) {
      const Piece &pc = ws.desc[b & 1][lane];
      const uint32_t out = pc.out_cls >> kClsBits, cls = pc.out_cls & ((1u << kClsBits) - 1);
      uint8_t *d = static_cast<uint8_t *>(a.dst[out]);
      float scale = 1.0f;
      if (cls_nvfp4(cls)) {
        scale = load_f32_le(a.data + a.quant[out].scale2);  // the global scale
      } else if (cls >= CLS_E4M3_BF16 && !cls_quant(cls)) {
        if (a.scales) scale = a.scales[out];
        else if (pc.scale != kNoScale) scale = load_f32_le(a.data + pc.scale);
      }
      if (d == nullptr || cls >= CLS_COUNT ||
          (reinterpret_cast<uintptr_t>(d) & static_cast<uintptr_t>(cls_out_item(cls) - 1))) {
        atomicOr(a.err, kErrBadDst);
        d = nullptr;
      }
      ws.dstp[b & 1][lane] = d;
      ws.scl[b & 1][lane] = scale;
    }
    __syncwarp();
    uint32_t st = 0;
    const uint32_t n = next_batch(st);
    later = n > 0;
    if (later) {
      if ((b + 1) & 1) {
        bs1 = st;
        bn1 = n;
      } else {
        bs0 = st;
        bn0 = n;
      }
      if (lane == 0) {
        proxy_fence();
        issue_desc(b + 1);
      }
      dissued = b + 2;
    }
    return true;
  };

  // The piece being cut into segments: its fields are loaded once, when the
  // cursor reaches it, and the run's source/output addresses advance by the
  // pitch / run size, so a segment costs no divisions or multiplications.
  Cursor cur{0, 0, 0, bn0, 0};
  const uint8_t *run_src = nullptr;  // source of the current run's element 0
  uint8_t *run_dst = nullptr;        // output address of the current run's element 0
  uint64_t pitch = 0;
  uint32_t count = 0, rows = 0, cls = 0, sis = 0, sos = 0;
  float scale = 1.0f;
  bool loaded = false;
  bool interior = false;  // every byte of the piece lies in [lo16, hi16): no clipping
  // Block-scaled pieces: the output's scale table entry and the output unit
  // index of the piece's first unit.
  QuantInfo qi{};
  uint32_t q_row = 0, q_colu = 0;  // weight row and column (in units) of the cursor
  auto load_piece_state = [&]() -> bool {  // false: skip this piece
    const Piece &pc = ws.desc[cur.b & 1][cur.i];
    uint8_t *dp = ws.dstp[cur.b & 1][cur.i];
    count = pc.count;
    rows = pc.rows;
    if (dp == nullptr || count == 0 || rows == 0) return false;
    cls = pc.out_cls & ((1u << kClsBits) - 1);
    sis = cls_in_shift(cls);
    sos = cls_out_shift(cls);
    pitch = pc.pitch;
    run_src = a.data + pc.src;
    run_dst = dp + pc.dst;
    scale = ws.scl[cur.b & 1][cur.i];
    if constexpr (kInterior) {
      const uintptr_t lo = reinterpret_cast<uintptr_t>(run_src);
      const uintptr_t hi = lo + static_cast<uint64_t>(rows - 1) * pitch + (static_cast<uint64_t>(count) << sis);
      interior = lo >= lo16 && hi <= hi16;
    }
    if (cls_quant(cls)) {
      qi = a.quant[pc.out_cls >> kClsBits];
      const uint64_t unit0 = pc.dst >> sos;  // one division per piece
      q_row = static_cast<uint32_t>(unit0 / qi.row_units);
      q_colu = static_cast<uint32_t>(unit0 - static_cast<uint64_t>(q_row) * qi.row_units);
    }
    return true;
  };
  auto produce = [&](int slot) -> int {  // 1 issued, 0 done, -1 timed out
    for (;;) {
      if (cur.i == cur.n) {
        if (!later) return 0;
        ++cur.b;
        cur.i = 0;
        cur.r = 0;
        cur.e = 0;
        if (!enter_batch(cur.b)) return -1;
        cur.n = (cur.b & 1) ? bn1 : bn0;
        continue;
      }
      if (!loaded) {
        if (!load_piece_state()) {
          ++cur.i;
          continue;
        }
        loaded = true;
      }
      uint32_t len = min(kSeg >> sis, count - cur.e);
      // Block-scaled: the segment stays in one weight row and its block scales
      // fit the slot's scale area; they are fetched with it when they lie in
      // the aligned interior of the data section (else read in place).
      uint32_t col0 = 0, sbytes = 0;
      const uint8_t *sptr = nullptr;
      uintptr_t sw0 = 0;
      if (cls_quant(cls)) {
        const bool nv = cls_nvfp4(cls);
        const uint32_t row = q_row, colu = q_colu;
        len = min(len, qi.row_units - colu);
        col0 = nv ? 2 * colu : colu;
        const uint32_t ss = nv ? 1 : 4;  // bytes per block scale
        const uint32_t bc = 1u << qi.bc_shift, maxblk = nv ? kScalePayload : kQscMax;
        const uint32_t max_el = maxblk * bc - (col0 & (bc - 1));
        len = min(len, nv ? max_el / 2 : max_el);
        const uint32_t el = nv ? 2 * len : len;
        const uint32_t b0 = col0 >> qi.bc_shift, nblk = ((col0 + el - 1) >> qi.bc_shift) - b0 + 1;
        const uint8_t *sg = a.data + qi.scale + (static_cast<uint64_t>(row >> qi.br_shift) * qi.scols + b0) * ss;
        q_colu += len;  // the next segment: same row, or the next one
        if (q_colu == qi.row_units) {
          q_colu = 0;
          ++q_row;
        }
        const uintptr_t g = reinterpret_cast<uintptr_t>(sg);
        sw0 = g & ~uintptr_t(15);
        const uintptr_t sw1 = (g + nblk * ss + 15) & ~uintptr_t(15);
        if (sw0 >= lo16 && sw1 <= hi16) {
          sbytes = static_cast<uint32_t>(sw1 - sw0);
          sptr = ws.sbuf[slot] + (g - sw0);
        } else {
          sptr = sg;
        }
      }
      const uint8_t *s0 = run_src + (static_cast<uint64_t>(cur.e) << sis);
      const uintptr_t s = reinterpret_cast<uintptr_t>(s0);
      const uintptr_t send = s + (static_cast<uint64_t>(len) << sis);
      uint32_t A = 0, Z = len, bytes, off;
      uintptr_t w0;
      if (kInterior && interior) {
        w0 = s & ~uintptr_t(15);
        bytes = static_cast<uint32_t>(((send + 15) & ~uintptr_t(15)) - w0);
        off = static_cast<uint32_t>(s - w0);
      } else {  // the first or last piece of the data section: clip to [lo16, hi16)
        if (s < lo16) A = min(len, static_cast<uint32_t>((lo16 - s + (1u << sis) - 1) >> sis));
        if (send > hi16) Z = hi16 > s ? static_cast<uint32_t>((hi16 - s) >> sis) : 0;
        if (Z < A) Z = A;
        bytes = 0;
        off = 0;
        w0 = 0;
        if (Z > A) {
          const uintptr_t sa = s + (static_cast<uint64_t>(A) << sis);
          w0 = sa & ~uintptr_t(15);
          bytes = static_cast<uint32_t>(((s + (static_cast<uint64_t>(Z) << sis) + 15) & ~uintptr_t(15)) - w0);
          off = static_cast<uint32_t>(sa - w0);
        }
      }
      if (lane == 0) {
        SegMeta m;
        m.dst = run_dst + (static_cast<uint64_t>(cur.e) << sos);
        m.gsrc = s0;
        m.len = len;
        m.a = A;
        m.z = Z;
        m.off = off;
        m.scale = scale;
        m.cls = cls;
        m.col0 = col0;
        m.bcs = qi.bc_shift;
        m.sptr = sptr;
        put_meta(&ws.meta[slot], m, cls_quant(cls));
        proxy_fence();
        mbar_expect(&ws.bar[slot], bytes + sbytes);
        if (bytes) bulk_copy(ws.buf[slot], reinterpret_cast<const void *>(w0), bytes, &ws.bar[slot]);
        if (sbytes) bulk_copy(ws.sbuf[slot], reinterpret_cast<const void *>(sw0), sbytes, &ws.bar[slot]);
      }
      cur.e += len;
      if (cur.e == count) {
        cur.e = 0;
        run_src += pitch;
        run_dst += static_cast<uint64_t>(count) << sos;
        if (++cur.r == rows) {
          cur.r = 0;
          ++cur.i;
          loaded = false;
        }
      }
      return 1;
    }
  };

  bool ok = enter_batch(0);
  uint32_t jp = 0, jc = 0;
  bool more = ok;
  while (ok) {
    while (more && jp - jc < static_cast<uint32_t>(kSlots)) {
      const int got = produce(static_cast<int>(jp % kSlots));
      if (got > 0) ++jp;
      else {
        more = false;
        ok = got == 0;
      }
    }
    if (!ok || jc == jp) break;
    const int slot = static_cast<int>(jc % kSlots);
    if (!mbar_wait(&ws.bar[slot], (jc / kSlots) & 1)) {
      ok = false;
      break;
    }
    __syncwarp();
    {
      const SegMeta m = get_meta(&ws.meta[slot]);
      consume_any(ws.buf[slot], m, ws.qsc, lane);
    }
    __syncwarp();
    ++jc;
  }
  if (!ok) {
    // A wait gave up: record it, then give the warp's outstanding copies a
    // bounded chance to land before the warp (and its shared memory) ends.
    if (lane == 0) atomicOr(a.err, kErrTimeout);
    for (; jc < jp; ++jc) mbar_wait(&ws.bar[jc % kSlots], (jc / kSlots) & 1);
    for (; dseen < dissued; ++dseen) mbar_wait(&ws.dbar[dseen & 1], (dseen >> 1) & 1);
  }
  if (dtotal) release_claims(a, lane);
}

__global__ void __launch_bounds__(kThreads, ST_TMA_MIN_BLOCKS) materialize_tma(const LaunchArgs a) {
  extern __shared__ __align__(128) uint8_t tma_smem[];
  tma_body<ST_TMA_SLOTS, true>(a, tma_smem);
}

__global__ void __launch_bounds__(kThreads, ST_TMA_WIDE_MIN_BLOCKS) materialize_tma_wide(const LaunchArgs a) {
  extern __shared__ __align__(128) uint8_t tma_smem[];
  tma_body<ST_TMA_WIDE_SLOTS, false>(a, tma_smem);
}

std::string cuda_msg(cudaError_t e) { return std::string(cudaGetErrorName(e)) + ": " + cudaGetErrorString(e); }

}  // namespace

namespace {
constexpr size_t kTmaSmem = sizeof(WarpSmem<ST_TMA_SLOTS>) * kWarpsPerBlock;
constexpr size_t kTmaWideSmem = sizeof(WarpSmem<ST_TMA_WIDE_SLOTS>) * kWarpsPerBlock;
constexpr int kMaxDevices = 256;
std::mutex g_attr_mu;
bool g_tma_attr[2][kMaxDevices] = {};

// The TMA builds' dynamic shared memory exceeds the default 48 KiB: raise
// each kernel's limit once per device.
cudaError_t tma_attr(int dev, bool wide) {
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  if (g_tma_attr[wide][dev]) return cudaSuccess;
  cudaError_t e = wide ? cudaFuncSetAttribute(materialize_tma_wide, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(kTmaWideSmem))
                       : cudaFuncSetAttribute(materialize_tma, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(kTmaSmem));
  if (e == cudaSuccess) g_tma_attr[wide][dev] = true;
  return e;
}
}  // namespace

st_status kernel_occupancy(uint32_t variant, int *sms, int *blocks_per_sm) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess && (variant == kKernelTma || variant == kKernelTmaWide)) e = tma_attr(dev, variant == kKernelTmaWide);
  if (e == cudaSuccess) {
    switch (variant) {
      case kKernelLatency:
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, materialize_latency, kThreads, 0);
        break;
      case kKernelTma:
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, materialize_tma, kThreads, kTmaSmem);
        break;
      case kKernelTmaWide:
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, materialize_tma_wide, kThreads, kTmaWideSmem);
        break;
      default:
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, materialize_stream, kThreads, 0);
    }
  }
  if (e != cudaSuccess) return set_error(ST_E_CUDA, "querying the device: %s", cuda_msg(e).c_str());
  if (*blocks_per_sm < 1) *blocks_per_sm = 1;
  return ST_OK;
}

st_status launch_materialize(const LaunchArgs &a, uint32_t variant, void *stream) {
  const uint32_t blocks = (a.workers + kWarpsPerBlock - 1) / kWarpsPerBlock;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (variant == kKernelTma || variant == kKernelTmaWide) {
    const bool wide = variant == kKernelTmaWide;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = tma_attr(dev, wide);
    if (e != cudaSuccess)
      return set_error(ST_E_CUDA, "enabling %zu bytes of shared memory: %s", wide ? kTmaWideSmem : kTmaSmem,
                       cuda_msg(e).c_str());
    if (wide) materialize_tma_wide<<<blocks, kThreads, kTmaWideSmem, st>>>(a);
    else materialize_tma<<<blocks, kThreads, kTmaSmem, st>>>(a);
  } else if (variant == kKernelLatency) {
    materialize_latency<<<blocks, kThreads, 0, st>>>(a);
  } else {
    materialize_stream<<<blocks, kThreads, 0, st>>>(a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(ST_E_CUDA, "materialize launch (%u blocks): %s", blocks, cuda_msg(e).c_str());
  return ST_OK;
}

// ------------------------------------------------ allocation-free scratch
//
// Scratch for st_materialize_noalloc: the plan's piece table, warp ranges and
// error word are copied here instead of into memory the library allocates.
// The array is part of the module image, so every device that loads the
// library holds these bytes until the process exits.  In host code the name
// g_static_scratch is only a host-side stand-in, never a device address: the
// device address comes from cudaGetSymbolAddress, looked up once per device
// with that device current.
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {
std::mutex g_static_mu;
void *g_static_addr[kMaxDevices] = {};
}  // namespace

st_status static_scratch(void **addr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(ST_E_CUDA, "cudaGetDevice: %s", cuda_msg(e).c_str());
  if (dev < 0 || dev >= kMaxDevices) return set_error(ST_E_INVAL, "device %d is beyond the %d supported", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p)
      return set_error(ST_E_CUDA, "looking up the static scratch on device %d: %s", dev, cuda_msg(e).c_str());
    g_static_addr[dev] = p;
  }
  *addr = g_static_addr[dev];
  return ST_OK;
}

}  // namespace stmat
