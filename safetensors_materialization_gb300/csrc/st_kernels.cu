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
//    synchronization and no waits, so the kernel cannot stall on a peer;
//  - each lane moves one 16-byte source chunk per step (K = 16 / itemsize
//    elements) with 16-byte vector loads; consecutive lanes take consecutive
//    chunks, so every warp access is one contiguous run;
//  - a source whose address is not 16-byte aligned is read as the two
//    aligned 16-byte words covering the chunk and shifted into place with
//    funnel shifts (the misalignment is the same for every chunk of a piece,
//    so the word offset is a template parameter and the bit shift uniform);
//  - destinations are written with aligned vector stores (8 or 16 bytes);
//    elements before the first aligned destination chunk, after the last, or
//    whose 16-byte source window would leave the data section are converted
//    one by one with byte loads, so no byte outside the data section is read;
//  - conversions: exact decode to binary32 (hardware cvt for f16 and e4m3,
//    bit placement for bf16 and e5m2), one __fmul_rn by the scale for fp8,
//    then cvt.rn to bf16/f16 (round to nearest even, subnormals kept);
//    NaN results are replaced by the output's positive quiet NaN.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "st_internal.h"

namespace stmat {
namespace {

constexpr int kThreads = kWarpsPerBlock * 32;
constexpr int kUnroll = 4;  // chunks in flight per lane

// ---------------------------------------------------------------- codecs

struct DecF32 {
  static constexpr int kSize = 4;
  __device__ static float dec(uint32_t b) { return __uint_as_float(b); }
};
struct DecF16 {
  static constexpr int kSize = 2;
  __device__ static float dec(uint32_t b) { return __half2float(__ushort_as_half(static_cast<unsigned short>(b))); }
};
struct DecBF16 {
  static constexpr int kSize = 2;
  __device__ static float dec(uint32_t b) { return __uint_as_float(b << 16); }
};
struct DecE4M3 {
  static constexpr int kSize = 1;
  __device__ static float dec(uint32_t b) {
    __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
    return __half2float(__half(h));
  }
};
struct DecE5M2 {
  static constexpr int kSize = 1;  // an e5m2 value is the upper byte of its binary16 encoding
  __device__ static float dec(uint32_t b) { return __half2float(__ushort_as_half(static_cast<unsigned short>(b << 8))); }
};

struct EncBF16 {
  static constexpr int kSize = 2;
  __device__ static uint32_t enc(float x) {
    return x != x ? 0x7FC0u : static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
  }
};
struct EncF16 {
  static constexpr int kSize = 2;
  __device__ static uint32_t enc(float x) {
    return x != x ? 0x7E00u : static_cast<uint32_t>(__half_as_ushort(__float2half_rn(x)));
  }
};
struct EncF32 {
  static constexpr int kSize = 4;
  __device__ static uint32_t enc(float x) { return x != x ? 0x7FC00000u : __float_as_uint(x); }
};

template <class D, class E, bool kScaled>
struct Conv {
  static constexpr int SI = D::kSize, SO = E::kSize;
  static constexpr bool kCopy = false;
  __device__ static uint32_t one(uint32_t bits, float s) {
    float x = D::dec(bits);
    if (kScaled) x = __fmul_rn(x, s);
    return E::enc(x);
  }
};

struct CopyBytes {
  static constexpr int SI = 1, SO = 1;
  static constexpr bool kCopy = true;
  __device__ static uint32_t one(uint32_t bits, float) { return bits; }
};

// ------------------------------------------------------------- data moves

__device__ __forceinline__ uint4 ld16(const uint8_t *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }

// Read-only 16-byte load kept in program order with the other batch loads.
__device__ __forceinline__ uint4 ld16_batch(const uint8_t *p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16 source bytes starting at word offset Q (0..3) of the 32-byte window
// {a, b}, shifted right by `sh` bits (8 * (misalignment % 4)).
template <int Q>
__device__ __forceinline__ void realign(const uint4 &a, const uint4 &b, uint32_t sh, uint32_t (&s)[4]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) s[i] = __funnelshift_r(w[Q + i], w[Q + i + 1], sh);
}

// Converts one 16-byte source chunk (16 / SI elements) into OB output bytes.
template <class CV>
__device__ __forceinline__ void convert16(const uint32_t (&s)[4], float scale,
                                          uint32_t (&o)[(16 / CV::SI) * CV::SO / 4]) {
  constexpr int K = 16 / CV::SI;
  constexpr int NW = K * CV::SO / 4;
  if constexpr (CV::kCopy) {
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = s[i];
  } else {
#pragma unroll
    for (int i = 0; i < NW; ++i) o[i] = 0;
#pragma unroll
    for (int j = 0; j < K; ++j) {
      constexpr uint32_t kMask = CV::SI == 4 ? 0xFFFFFFFFu : (1u << (8 * CV::SI)) - 1;
      const uint32_t bits = (s[(j * CV::SI) / 4] >> (8 * ((j * CV::SI) % 4))) & kMask;
      const uint32_t y = CV::one(bits, scale);
      o[(j * CV::SO) / 4] |= y << (8 * ((j * CV::SO) % 4));
    }
  }
}

template <int NW>
__device__ __forceinline__ void store_out(uint8_t *p, const uint32_t (&o)[NW]) {
  if constexpr (NW == 2) {
    *reinterpret_cast<uint2 *>(p) = make_uint2(o[0], o[1]);
  } else {
#pragma unroll
    for (int i = 0; i < NW / 4; ++i)
      reinterpret_cast<uint4 *>(p)[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
  }
}

// Vector body: chunks [0, nch) of 16 source bytes each.  Q < 0: the source
// base is 16-byte aligned; otherwise chunk c's bytes start at word Q of the
// aligned window sbase + 16 c, shifted by sh bits.
template <class CV, int Q>
__device__ __forceinline__ void chunk(const uint8_t *sbase, uint32_t sh, uint8_t *dbase, uint64_t c, const uint4 &a,
                                      const uint4 &b, float scale) {
  constexpr int OB = (16 / CV::SI) * CV::SO;
  uint32_t s[4];
  if constexpr (Q >= 0) {
    realign<Q>(a, b, sh, s);
  } else {
    s[0] = a.x; s[1] = a.y; s[2] = a.z; s[3] = a.w;
  }
  uint32_t o[OB / 4];
  convert16<CV>(s, scale, o);
  store_out<OB / 4>(dbase + c * OB, o);
}

template <class CV, int Q>
__device__ __forceinline__ void body(const uint8_t *sbase, uint32_t sh, uint8_t *dbase, uint64_t nch, float scale,
                                     int lane) {
  uint64_t c = lane;
  // Full batches: kUnroll chunks per lane in flight.
  for (; c + 32 * (kUnroll - 1) < nch; c += 32 * kUnroll) {
    uint4 a[kUnroll], b[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      a[u] = ld16_batch(sbase + (c + 32 * u) * 16);
      if constexpr (Q >= 0) b[u] = ld16_batch(sbase + (c + 32 * u) * 16 + 16);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) chunk<CV, Q>(sbase, sh, dbase, c + 32 * u, a[u], b[u], scale);
  }
  for (; c < nch; c += 32) {
    uint4 a = ld16(sbase + c * 16), b = a;
    if constexpr (Q >= 0) b = ld16(sbase + c * 16 + 16);
    chunk<CV, Q>(sbase, sh, dbase, c, a, b, scale);
  }
}

// Elements [a, b) one per lane, with byte loads (any source alignment).
template <class CV>
__device__ __forceinline__ void scalar_range(const uint8_t *src, uint8_t *dst, uint64_t a, uint64_t b, float scale,
                                             int lane) {
  for (uint64_t e = a + lane; e < b; e += 32) {
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

template <class CV>
__device__ void run_piece(const uint8_t *data, uint64_t data_bytes, const uint8_t *src, uint8_t *dst, uint64_t n,
                          float scale, int lane) {
  constexpr int K = 16 / CV::SI;
  constexpr int OB = K * CV::SO;
  constexpr int A = OB < 16 ? OB : 16;  // destination alignment of the vector body
  uint64_t head = ((A - (reinterpret_cast<uintptr_t>(dst) & (A - 1))) & (A - 1)) / CV::SO;
  if (head > n) head = n;
  uint64_t nch = (n - head) / K;
  uintptr_t sa = reinterpret_cast<uintptr_t>(src + head * CV::SI);
  const uint32_t r = static_cast<uint32_t>(sa & 15);
  if (r && nch) {
    // Keep every 32-byte window inside the data section.
    const uintptr_t lo = reinterpret_cast<uintptr_t>(data), hi = lo + data_bytes;
    if ((sa & ~uintptr_t(15)) < lo) {
      head += K;
      --nch;
      sa += 16;
    }
    if (nch && (sa & ~uintptr_t(15)) + 16 * nch + 16 > hi) --nch;
  }
  scalar_range<CV>(src, dst, 0, head, scale, lane);
  scalar_range<CV>(src, dst, head + nch * K, n, scale, lane);
  if (!nch) return;
  const uint8_t *sbase = reinterpret_cast<const uint8_t *>(sa & ~uintptr_t(15));
  uint8_t *dbase = dst + head * CV::SO;
  const uint32_t sh = 8 * (r & 3);
  if (r == 0) {
    body<CV, -1>(sbase, 0, dbase, nch, scale, lane);
  } else {
    switch (r >> 2) {
      case 0: body<CV, 0>(sbase, sh, dbase, nch, scale, lane); break;
      case 1: body<CV, 1>(sbase, sh, dbase, nch, scale, lane); break;
      case 2: body<CV, 2>(sbase, sh, dbase, nch, scale, lane); break;
      default: body<CV, 3>(sbase, sh, dbase, nch, scale, lane); break;
    }
  }
}

// Binary32 from 4 little-endian bytes at any alignment.
__device__ __forceinline__ float load_f32_le(const uint8_t *p) {
  return __uint_as_float(static_cast<uint32_t>(p[0]) | (static_cast<uint32_t>(p[1]) << 8) |
                         (static_cast<uint32_t>(p[2]) << 16) | (static_cast<uint32_t>(p[3]) << 24));
}

__global__ void __launch_bounds__(kThreads) materialize_kernel(const LaunchArgs a) {
  const int lane = threadIdx.x & 31;
  const uint32_t w = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  if (w >= a.workers) return;
  const uint32_t p0 = a.parts[w], p1 = a.parts[w + 1];
  for (uint32_t k = p0; k < p1; ++k) {
    const Piece pc = a.pieces[k];
    const uint32_t out = pc.out_cls >> kClsBits, cls = pc.out_cls & ((1u << kClsBits) - 1);
    uint8_t *dst = static_cast<uint8_t *>(a.dst[out]);
    const int so = cls_out_size(cls);
    if (dst == nullptr || (reinterpret_cast<uintptr_t>(dst) & (so - 1))) {
      if (lane == 0) atomicOr(a.err, kErrBadDst);
      continue;
    }
    dst += pc.dst;
    const uint8_t *src = a.data + pc.src;
    float scale = 1.0f;
    if (cls >= CLS_E4M3_BF16) {
      if (a.scales) scale = a.scales[out];
      else if (pc.scale != kNoScale) scale = load_f32_le(a.data + pc.scale);
    }
    const uint64_t n = pc.count;
    switch (cls) {
      case CLS_COPY: run_piece<CopyBytes>(a.data, a.data_bytes, src, dst, n, scale, lane); break;
      case CLS_F32_BF16: run_piece<Conv<DecF32, EncBF16, false>>(a.data, a.data_bytes, src, dst, n, scale, lane); break;
      case CLS_F32_F16: run_piece<Conv<DecF32, EncF16, false>>(a.data, a.data_bytes, src, dst, n, scale, lane); break;
      case CLS_F16_BF16: run_piece<Conv<DecF16, EncBF16, false>>(a.data, a.data_bytes, src, dst, n, scale, lane); break;
      case CLS_F16_F32: run_piece<Conv<DecF16, EncF32, false>>(a.data, a.data_bytes, src, dst, n, scale, lane); break;
      case CLS_BF16_F16: run_piece<Conv<DecBF16, EncF16, false>>(a.data, a.data_bytes, src, dst, n, scale, lane); break;
      case CLS_BF16_F32: run_piece<Conv<DecBF16, EncF32, false>>(a.data, a.data_bytes, src, dst, n, scale, lane); break;
      case CLS_E4M3_BF16: run_piece<Conv<DecE4M3, EncBF16, true>>(a.data, a.data_bytes, src, dst, n, scale, lane); break;
      case CLS_E4M3_F16: run_piece<Conv<DecE4M3, EncF16, true>>(a.data, a.data_bytes, src, dst, n, scale, lane); break;
      case CLS_E4M3_F32: run_piece<Conv<DecE4M3, EncF32, true>>(a.data, a.data_bytes, src, dst, n, scale, lane); break;
      case CLS_E5M2_BF16: run_piece<Conv<DecE5M2, EncBF16, true>>(a.data, a.data_bytes, src, dst, n, scale, lane); break;
      case CLS_E5M2_F16: run_piece<Conv<DecE5M2, EncF16, true>>(a.data, a.data_bytes, src, dst, n, scale, lane); break;
      case CLS_E5M2_F32: run_piece<Conv<DecE5M2, EncF32, true>>(a.data, a.data_bytes, src, dst, n, scale, lane); break;
      default:
        if (lane == 0) atomicOr(a.err, kErrBadDst);
    }
  }
}

std::string cuda_msg(cudaError_t e) { return std::string(cudaGetErrorName(e)) + ": " + cudaGetErrorString(e); }

}  // namespace

st_status kernel_occupancy(int *sms, int *blocks_per_sm) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, materialize_kernel, kThreads, 0);
  if (e != cudaSuccess) return set_error(ST_E_CUDA, "querying the device: %s", cuda_msg(e).c_str());
  if (*blocks_per_sm < 1) *blocks_per_sm = 1;
  return ST_OK;
}

st_status launch_materialize(const LaunchArgs &a, void *stream) {
  const uint32_t blocks = (a.workers + kWarpsPerBlock - 1) / kWarpsPerBlock;
  materialize_kernel<<<blocks, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(ST_E_CUDA, "materialize launch (%u blocks): %s", blocks, cuda_msg(e).c_str());
  return ST_OK;
}

}  // namespace stmat
