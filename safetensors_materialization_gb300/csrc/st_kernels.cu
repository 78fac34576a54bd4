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
//    warps; warp w walks pieces [parts[w], parts[w+1]) with no inter-warp
//    synchronization and no waits, so the kernel cannot stall on a peer.  A
//    warp stages up to 32 piece descriptors at a time in shared memory (one
//    per lane), with their destination pointers and scales, so the dependent
//    loads of a piece are paid once per 32 pieces;
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
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

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
template <int D>
__device__ __forceinline__ uint32_t encode2_16(float2 f) {
  uint32_t r;
  if constexpr (D == D_BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(f.x, f.y);
    r = *reinterpret_cast<uint32_t *>(&v);
    const uint32_t lo = f.x != f.x ? kNanBF16 : (r & 0xFFFFu);
    const uint32_t hi = f.y != f.y ? kNanBF16 : (r >> 16);
    return lo | (hi << 16);
  } else {
    __half2 v = __floats2half2_rn(f.x, f.y);
    r = *reinterpret_cast<uint32_t *>(&v);
    const uint32_t lo = f.x != f.x ? kNanF16 : (r & 0xFFFFu);
    const uint32_t hi = f.y != f.y ? kNanF16 : (r >> 16);
    return lo | (hi << 16);
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
struct StreamCfg {
  static constexpr int kU16 = 4, kU8 = 8, kU4 = 16;
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
  if constexpr (NW == 2) *reinterpret_cast<uint2 *>(p) = make_uint2(o[0], o[1]);
  else *reinterpret_cast<uint4 *>(p) = make_uint4(o[0], o[1], o[2], o[3]);
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

template <class Cfg>
__device__ __forceinline__ void materialize_body(const LaunchArgs &a) {
  __shared__ Staged stage[kWarpsPerBlock];
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t wib = threadIdx.x >> 5;
  const uint32_t w = blockIdx.x * kWarpsPerBlock + wib;
  if (w >= a.workers) return;
  const uint32_t p0 = a.parts[w], p1 = a.parts[w + 1];
  Staged &st = stage[wib];
  for (uint32_t base = p0; base < p1; base += 32) {
    const uint32_t n = min(32u, p1 - base);
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
  }
}

__global__ void __launch_bounds__(kThreads) materialize_stream(const LaunchArgs a) { materialize_body<StreamCfg>(a); }

__global__ void __launch_bounds__(kThreads, ST_LAT_MIN_BLOCKS) materialize_latency(const LaunchArgs a) {
  materialize_body<LatencyCfg>(a);
}

std::string cuda_msg(cudaError_t e) { return std::string(cudaGetErrorName(e)) + ": " + cudaGetErrorString(e); }

}  // namespace

st_status kernel_occupancy(uint32_t variant, int *sms, int *blocks_per_sm) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = variant == kKernelLatency
            ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, materialize_latency, kThreads, 0)
            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, materialize_stream, kThreads, 0);
  if (e != cudaSuccess) return set_error(ST_E_CUDA, "querying the device: %s", cuda_msg(e).c_str());
  if (*blocks_per_sm < 1) *blocks_per_sm = 1;
  return ST_OK;
}

st_status launch_materialize(const LaunchArgs &a, uint32_t variant, void *stream) {
  const uint32_t blocks = (a.workers + kWarpsPerBlock - 1) / kWarpsPerBlock;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (variant == kKernelLatency) materialize_latency<<<blocks, kThreads, 0, st>>>(a);
  else materialize_stream<<<blocks, kThreads, 0, st>>>(a);
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
constexpr int kMaxDevices = 256;
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
