// Shared device code of the ReplaySSM kernels: the store view, the register tile of a
// (sequence, head) slab, vector loads and stores for each storage type, warp reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/replayssm.h"

namespace rssm {

constexpr int kThreads = 256;  // one CTA per (sequence, head) slab: 8 warps
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCap = 64;    // ring records a sequence can hold (2 per lane)
constexpr int kDtStage = 1024; // dt values a prep CTA stages in shared memory at once
constexpr unsigned kFull = 0xffffffffu;
// Dynamic shared memory above this opts the kernel in to more than the default 48 KB per CTA,
// a cap that counts static shared memory too (at most about 6 KB in these kernels).
constexpr size_t kSmemNoOptIn = 40 * 1024;
constexpr float kE4M3Max = 448.0f;

// Resident CTAs per SM the register budget is sized for: a P=64 slab tile is 8 rows x N/32
// columns per thread, so wide states (N = 256) trade occupancy for registers.
template <int N>
constexpr int kMinBlocks = N >= 256 ? 2 : 4;

using bf16 = __nv_bfloat16;

// Everything a kernel needs to find a store's regions (passed by value).
struct StoreView {
  float* h0;      // [batch][H][P][N]
  void* rc;       // read copy, bf16, e4m3 or fp16 [batch][H][P][N]
  float* scale;   // [batch][H] (e4m3 and nvfp4 copies)
  uint8_t* bscale;  // [batch][H][P][N/16] e4m3 block scales (nvfp4 copy)
  void* xbuf;     // [batch][H][cap][P]
  void* bbuf;     // [batch][G][cap][N]
  void* dtbuf;    // [batch][H][cap]
  int4* meta;     // [batch] {start, n, pending, epoch of the next checkpoint write}
  int* arrive;    // [batch]
  int* status;
  int4* plan;     // [batch] {start, n, kind, 0} of the step in flight
  float* coef;    // [batch][H][cap + 1]
  const float* A;
  const float* D;
  int batch, H, G, hpg, L, cap, tmax;
  int shared;     // 1: the read copy is the checkpoint (no FP32 checkpoint)
  int ckpt16;     // 1: h0 holds FP16 values written by stochastic rounding (not FP32)
  int sms;        // SMs of the device the store lives on (0: unknown, no L2 prefetch)
  int prep_appends;  // 1: a step's prep kernel appends the token's B and dt records (stores
                     // with a read copy, whose steps overlap); 0: the per-head kernels do
};

// Bulk prefetch of `bytes` (a multiple of 16, from a 16-byte aligned address) into L2: one
// instruction, no registers held, nothing to wait for. A per-head kernel CTA prefetches the
// state a CTA one wave later will read, so DRAM keeps streaming while the resident CTAs
// compute (their own loads are bounded by the registers that receive them).
__device__ __forceinline__ void prefetch_l2(const void* p, unsigned int bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ------------------------------------------------------------------ element conversion
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(bf16 v) { return __bfloat162float(v); }

// Load VEC consecutive elements (16-byte or smaller vector loads) and widen to float.
template <int VEC>
__device__ __forceinline__ void ldv(const float* p, float (&o)[VEC]) {
  static_assert(VEC == 2 || VEC == 4, "vec");
  if constexpr (VEC == 4) {
    float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  } else {
    float2 v = *reinterpret_cast<const float2*>(p);
    o[0] = v.x; o[1] = v.y;
  }
}
template <int VEC>
__device__ __forceinline__ void ldv(const bf16* p, float (&o)[VEC]) {
  static_assert(VEC == 2 || VEC == 4, "vec");
  if constexpr (VEC == 4) {
    uint2 v = *reinterpret_cast<const uint2*>(p);
    float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v.x));
    float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v.y));
    o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
  } else {
    uint32_t v = *reinterpret_cast<const uint32_t*>(p);
    float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v));
    o[0] = a.x; o[1] = a.y;
  }
}

// Streaming (evict-first) FP32 loads for state slabs, which are read once per call.
template <int VEC>
__device__ __forceinline__ void ldv_stream(const float* p, float (&o)[VEC]) {
  if constexpr (VEC == 4) {
    float4 v = __ldcs(reinterpret_cast<const float4*>(p));
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  } else {
    float2 v = __ldcs(reinterpret_cast<const float2*>(p));
    o[0] = v.x; o[1] = v.y;
  }
}
template <int VEC>
__device__ __forceinline__ void stv_stream(float* p, const float (&v)[VEC]) {
  if constexpr (VEC == 4) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
  } else {
    __stcs(reinterpret_cast<float2*>(p), make_float2(v[0], v[1]));
  }
}

// Read-copy element types. A "pack" is VEC elements: 8 or 4 bytes (bf16), 4 or 2 (e4m3).
template <int VEC>
__device__ __forceinline__ void ld_bf16_stream(const bf16* p, float (&o)[VEC]) {
  if constexpr (VEC == 4) {
    uint2 v = __ldcs(reinterpret_cast<const uint2*>(p));
    float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v.x));
    float2 b = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v.y));
    o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
  } else {
    unsigned int v = __ldcs(reinterpret_cast<const unsigned int*>(p));
    float2 a = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v));
    o[0] = a.x; o[1] = a.y;
  }
}
template <int VEC>
__device__ __forceinline__ void st_bf16_stream(bf16* p, const float (&v)[VEC]) {
  if constexpr (VEC == 4) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
    __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
    uint2 u;
    u.x = *reinterpret_cast<unsigned int*>(&a);
    u.y = *reinterpret_cast<unsigned int*>(&b);
    __stcs(reinterpret_cast<uint2*>(p), u);
  } else {
    __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
    __stcs(reinterpret_cast<unsigned int*>(p), *reinterpret_cast<unsigned int*>(&a));
  }
}

__device__ __forceinline__ float2 e4m3x2_to_float2(unsigned short v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  return __half22float2(hh);
}
__device__ __forceinline__ unsigned short float2_to_e4m3x2(float a, float b) {
  return static_cast<unsigned short>(
      __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

template <int VEC>
__device__ __forceinline__ void ld_e4m3_stream(const uint8_t* p, float scale, float (&o)[VEC]) {
  if constexpr (VEC == 4) {
    unsigned int v = __ldcs(reinterpret_cast<const unsigned int*>(p));
    float2 a = e4m3x2_to_float2(static_cast<unsigned short>(v & 0xffffu));
    float2 b = e4m3x2_to_float2(static_cast<unsigned short>(v >> 16));
    o[0] = a.x * scale; o[1] = a.y * scale; o[2] = b.x * scale; o[3] = b.y * scale;
  } else {
    unsigned short v = __ldcs(reinterpret_cast<const unsigned short*>(p));
    float2 a = e4m3x2_to_float2(v);
    o[0] = a.x * scale; o[1] = a.y * scale;
  }
}
// Codes are decided in FP32 with an IEEE division by the scale, as the format defines. (A
// multiply by the reciprocal with an exact fallback near the code boundaries was measured: the
// boundary tests cost as many instructions as the division and added branch stalls.)
template <int VEC>
__device__ __forceinline__ void st_e4m3_stream(uint8_t* p, float scale, const float (&v)[VEC]) {
  if constexpr (VEC == 4) {
    unsigned int lo = float2_to_e4m3x2(__fdiv_rn(v[0], scale), __fdiv_rn(v[1], scale));
    unsigned int hi = float2_to_e4m3x2(__fdiv_rn(v[2], scale), __fdiv_rn(v[3], scale));
    __stcs(reinterpret_cast<unsigned int*>(p), lo | (hi << 16));
  } else {
    unsigned short c = float2_to_e4m3x2(__fdiv_rn(v[0], scale), __fdiv_rn(v[1], scale));
    __stcs(reinterpret_cast<unsigned short*>(p), c);
  }
}

// NVFP4 copies (dstate 128): E2M1 codes, one E4M3 scale per 16 consecutive elements of a row
// ([P][N/16], row-major), one FP32 scale per slab. Code layout of a row (64 bytes): quarter q
// (0..3) of every block holds columns 4q..4q+3 of the block; the 8 blocks' quarter-q units sit
// together at bytes 16q + 2b, 16q + 2b + 1. A unit's byte 0 holds columns 4q (slot A) and
// 4q + 2 (slot B), byte 1 columns 4q + 1 (A) and 4q + 3 (B). Slot A keeps a code's sign in
// bit 7 and its magnitude in bits 3..1, slot B the sign in bit 0 and the magnitude in bits
// 6..4. So a lane that owns a row's quarter reads all 8 blocks of it with one 16-byte load,
// and slot A is already the high byte of an FP16 equal to the E2M1 value times 2^-14.
constexpr float kE2M1Max = 6.0f;
constexpr int kFp4Block = 16;
__device__ __forceinline__ float2 e2m1x2_to_float2(unsigned int byte) {
  const __half2_raw r = __nv_cvt_fp4x2_to_halfraw2(static_cast<__nv_fp4x2_storage_t>(byte & 0xffu), __NV_E2M1);
  return __half22float2(*reinterpret_cast<const __half2*>(&r));
}
__device__ __forceinline__ unsigned int float2_to_e2m1x2(float a, float b) {
  return __nv_cvt_float2_to_fp4x2(make_float2(a, b), __NV_E2M1, cudaRoundNearest);
}
__device__ __forceinline__ float e4m3_to_float(unsigned int code) {
  return e4m3x2_to_float2(static_cast<unsigned short>(code & 0xffu)).x;
}
// E2M1 code (sign bit 3, magnitude bits 2..0) <-> the two byte slots
__device__ __forceinline__ unsigned int fp4_slot_a(unsigned int c) { return ((c & 8u) << 4) | ((c & 7u) << 1); }
__device__ __forceinline__ unsigned int fp4_slot_b(unsigned int c) { return ((c & 8u) >> 3) | ((c & 7u) << 4); }
__device__ __forceinline__ unsigned int fp4_code_a(unsigned int byte) { return ((byte >> 4) & 8u) | ((byte >> 1) & 7u); }
__device__ __forceinline__ unsigned int fp4_code_b(unsigned int byte) { return ((byte & 1u) << 3) | ((byte >> 4) & 7u); }
// Byte offset of the unit of row `row`, block `b`, quarter `q` inside a slab's codes.
__device__ __forceinline__ int fp4_unit(int row, int b, int q) { return row * 64 + q * 16 + b * 2; }

// Read-copy "packs": the raw bytes of VEC consecutive copy elements, kept packed in registers
// until they are used (so a thread can hold several heads' tiles), and their widening.
template <int RC, int VEC> struct PackOf;
template <> struct PackOf<REPLAY_RC_BF16, 4> { using type = uint2; };
template <> struct PackOf<REPLAY_RC_BF16, 2> { using type = unsigned int; };
template <> struct PackOf<REPLAY_RC_FP8E4M3, 4> { using type = unsigned int; };
template <> struct PackOf<REPLAY_RC_FP8E4M3, 2> { using type = unsigned short; };
template <> struct PackOf<REPLAY_RC_FP16, 4> { using type = uint2; };
template <> struct PackOf<REPLAY_RC_FP16, 2> { using type = unsigned int; };

template <int RC, int VEC>
__device__ __forceinline__ typename PackOf<RC, VEC>::type ld_pack(const void* rc, size_t elem) {
  using PT = typename PackOf<RC, VEC>::type;
  constexpr int esz = RC == REPLAY_RC_FP8E4M3 ? 1 : 2;
  return __ldcs(reinterpret_cast<const PT*>(static_cast<const char*>(rc) + elem * esz));
}
template <int RC, int VEC>
__device__ __forceinline__ void unpack(typename PackOf<RC, VEC>::type v, float scale, float (&o)[VEC]) {
  if constexpr (RC == REPLAY_RC_BF16) {
    if constexpr (VEC == 4) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
      o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
    } else {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
      o[0] = a.x; o[1] = a.y;
    }
  } else if constexpr (RC == REPLAY_RC_FP16) {
    if constexpr (VEC == 4) {
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
      o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
    } else {
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v));
      o[0] = a.x; o[1] = a.y;
    }
  } else {
    if constexpr (VEC == 4) {
      const float2 a = e4m3x2_to_float2(static_cast<unsigned short>(v & 0xffffu));
      const float2 b = e4m3x2_to_float2(static_cast<unsigned short>(v >> 16));
      o[0] = a.x * scale; o[1] = a.y * scale; o[2] = b.x * scale; o[3] = b.y * scale;
    } else {
      const float2 a = e4m3x2_to_float2(v);
      o[0] = a.x * scale; o[1] = a.y * scale;
    }
  }
}

// The same VEC values as VEC / 2 pairs for packed FP32 arithmetic, without the E4M3 slab
// scale (a caller applies it once to a sum). bf16 widens by shifts: a bf16 is the top half of
// an FP32.
template <int RC, int VEC>
__device__ __forceinline__ void unpack_pairs(typename PackOf<RC, VEC>::type v, float2 (&o)[VEC / 2]) {
  unsigned w[VEC / 2];
  if constexpr (sizeof(v) == 8) {
    w[0] = v.x;
    w[1] = v.y;
  } else if constexpr (VEC == 4) {
    w[0] = v & 0xffffu;  // E4M3: two codes per pair
    w[1] = v >> 16;
  } else {
    w[0] = v;
  }
#pragma unroll
  for (int j = 0; j < VEC / 2; ++j) {
    if constexpr (RC == REPLAY_RC_BF16)
      o[j] = make_float2(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xffff0000u));
    else if constexpr (RC == REPLAY_RC_FP16)
      o[j] = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
    else
      o[j] = e4m3x2_to_float2(static_cast<unsigned short>(w[j]));
  }
}

// ------------------------------------------------------------------ slab register tile
// A P x N slab is spread over 8 warps: warp w owns rows w*RPW .. w*RPW+RPW-1; in each row a
// lane owns NVEC vectors of VEC columns, vector v at column v*32*VEC + lane*VEC. Every
// vector load of a warp therefore covers a contiguous 32*VEC-element run of one row.
template <int P, int N>
struct Tile {
  static_assert(P % kWarps == 0, "P must be a multiple of 8");
  static_assert(N == 64 || N == 128 || N == 256, "N must be 64, 128 or 256");
  static constexpr int RPW = P / kWarps;
  static constexpr int VEC = N >= 128 ? 4 : 2;
  static constexpr int NVEC = N / (32 * VEC);
  static constexpr int E = VEC * NVEC;  // columns per lane
  __device__ static __forceinline__ int row(int warp, int i) { return warp * RPW + i; }
  __device__ static __forceinline__ int col(int lane, int v) { return v * 32 * VEC + lane * VEC; }
};

// Load the lane's E columns of a length-N vector (C or B), widened to float.
template <int P, int N, class T>
__device__ __forceinline__ void load_cols(const T* vec, int lane, float (&o)[Tile<P, N>::E]) {
  using TL = Tile<P, N>;
#pragma unroll
  for (int v = 0; v < TL::NVEC; ++v) {
    float t[TL::VEC];
    ldv<TL::VEC>(vec + TL::col(lane, v), t);
#pragma unroll
    for (int e = 0; e < TL::VEC; ++e) o[v * TL::VEC + e] = t[e];
  }
}

template <int P, int N>
__device__ __forceinline__ void load_tile_f32(const float* slab, int warp, int lane,
                                              float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E]) {
  using TL = Tile<P, N>;
#pragma unroll
  for (int i = 0; i < TL::RPW; ++i)
#pragma unroll
    for (int v = 0; v < TL::NVEC; ++v) {
      float t[TL::VEC];
      ldv_stream<TL::VEC>(slab + TL::row(warp, i) * N + TL::col(lane, v), t);
#pragma unroll
      for (int e = 0; e < TL::VEC; ++e) hv[i][v * TL::VEC + e] = t[e];
    }
}

// The same tile from a row-major FP32 slab in shared memory (a warp's access covers one row:
// conflict-free).
template <int P, int N>
__device__ __forceinline__ void load_tile_smem(const float* slab, int warp, int lane,
                                               float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E]) {
  using TL = Tile<P, N>;
#pragma unroll
  for (int i = 0; i < TL::RPW; ++i)
#pragma unroll
    for (int v = 0; v < TL::NVEC; ++v) {
      float t[TL::VEC];
      ldv<TL::VEC>(slab + TL::row(warp, i) * N + TL::col(lane, v), t);
#pragma unroll
      for (int e = 0; e < TL::VEC; ++e) hv[i][v * TL::VEC + e] = t[e];
    }
}

template <int P, int N>
__device__ __forceinline__ void store_tile_f32(float* slab, int warp, int lane,
                                               const float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E]) {
  using TL = Tile<P, N>;
#pragma unroll
  for (int i = 0; i < TL::RPW; ++i)
#pragma unroll
    for (int v = 0; v < TL::NVEC; ++v) {
      float t[TL::VEC];
#pragma unroll
      for (int e = 0; e < TL::VEC; ++e) t[e] = hv[i][v * TL::VEC + e];
      stv_stream<TL::VEC>(slab + TL::row(warp, i) * N + TL::col(lane, v), t);
    }
}

// FP16 copies: loads, round-to-nearest-even stores, and stochastic rounding.
template <int VEC>
__device__ __forceinline__ void ld_f16_stream(const __half* p, float (&o)[VEC]) {
  if constexpr (VEC == 4) {
    uint2 v = __ldcs(reinterpret_cast<const uint2*>(p));
    const float2 a = __half22float2(*reinterpret_cast<__half2*>(&v.x));
    const float2 b = __half22float2(*reinterpret_cast<__half2*>(&v.y));
    o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
  } else {
    unsigned int v = __ldcs(reinterpret_cast<const unsigned int*>(p));
    const float2 a = __half22float2(*reinterpret_cast<__half2*>(&v));
    o[0] = a.x; o[1] = a.y;
  }
}
template <int VEC>
__device__ __forceinline__ void st_f16_stream(__half* p, const float (&v)[VEC]) {
  if constexpr (VEC == 4) {
    __half2 a = __floats2half2_rn(v[0], v[1]), b = __floats2half2_rn(v[2], v[3]);
    uint2 u;
    u.x = *reinterpret_cast<unsigned int*>(&a);
    u.y = *reinterpret_cast<unsigned int*>(&b);
    __stcs(reinterpret_cast<uint2*>(p), u);
  } else {
    __half2 a = __floats2half2_rn(v[0], v[1]);
    __stcs(reinterpret_cast<unsigned int*>(p), *reinterpret_cast<unsigned int*>(&a));
  }
}

// The draws of stochastic rounding, 16 bits each: draw idx is 16-bit chunk idx mod 4 (most
// significant first) of output idx / 4 of the splitmix64 sequence (Steele, Lea and Flood, "Fast
// splittable pseudorandom number generators", OOPSLA 2014) started at kSrSeed; u = chunk / 2^16.
constexpr unsigned long long kSrSeed = 0x2545F4914F6CDD1Dull;
__device__ __forceinline__ unsigned long long splitmix64_at(unsigned long long seed, unsigned long long idx) {
  unsigned long long z = seed + (idx + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
// FP32 -> FP16 code by stochastic rounding: with lo the FP16 value toward zero and hi the
// next one away from zero, take hi iff u < (|v| - |lo|) / (|hi| - |lo|). Both differences
// are exact and the step is a power of two, so the ratio is exact. Saturates at 65504.
__device__ __forceinline__ unsigned short f16_sr(float v, float u) {
  const unsigned short lb = __half_as_ushort(__float2half_rz(v));
  if ((lb & 0x7FFFu) >= 0x7BFFu) return static_cast<unsigned short>((lb & 0x8000u) | 0x7BFFu);
  const unsigned short hb = static_cast<unsigned short>(lb + 1u);
  const float lo = fabsf(__half2float(__ushort_as_half(lb)));
  const float hi = fabsf(__half2float(__ushort_as_half(hb)));
  const float frac = __fdiv_rn(fabsf(v) - lo, hi - lo);
  return u < frac ? hb : lb;
}

// Read-copy tile loads/stores. RC is REPLAY_RC_BF16, REPLAY_RC_FP8E4M3 or REPLAY_RC_FP16.
template <int P, int N, int RC>
__device__ __forceinline__ void load_tile_rc(const void* rc, size_t slab, float scale, int warp,
                                             int lane, float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E],
                                             const uint8_t* bscale = nullptr) {
  using TL = Tile<P, N>;
#pragma unroll
  for (int i = 0; i < TL::RPW; ++i)
#pragma unroll
    for (int v = 0; v < TL::NVEC; ++v) {
      float t[TL::VEC];
      const size_t off = slab * P * N + TL::row(warp, i) * N + TL::col(lane, v);
      if constexpr (RC == REPLAY_RC_NVFP4) {
        // the lane's 4 columns are one unit (block lane / 4, quarter lane % 4); value =
        // decode(q) * (s_b * s_g)
        static_assert(N == 128 && TL::VEC == 4, "the NVFP4 copy is laid out for dstate 128");
        const float es = __fmul_rn(e4m3_to_float(__ldcs(bscale + off / kFp4Block)), scale);
        const unsigned int u = __ldcs(reinterpret_cast<const unsigned short*>(
            static_cast<const uint8_t*>(rc) + slab * P * N / 2 + fp4_unit(TL::row(warp, i), lane >> 2, lane & 3)));
        const unsigned int b0 = u & 0xffu, b1 = u >> 8;
        const float2 f01 = e2m1x2_to_float2(fp4_code_a(b0) | (fp4_code_a(b1) << 4));
        const float2 f23 = e2m1x2_to_float2(fp4_code_b(b0) | (fp4_code_b(b1) << 4));
        t[0] = f01.x * es;
        t[1] = f01.y * es;
        t[2] = f23.x * es;
        t[3] = f23.y * es;
      } else if constexpr (RC == REPLAY_RC_BF16)
        ld_bf16_stream<TL::VEC>(static_cast<const bf16*>(rc) + off, t);
      else if constexpr (RC == REPLAY_RC_FP16)
        ld_f16_stream<TL::VEC>(static_cast<const __half*>(rc) + off, t);
      else
        ld_e4m3_stream<TL::VEC>(static_cast<const uint8_t*>(rc) + off, scale, t);
#pragma unroll
      for (int e = 0; e < TL::VEC; ++e) hv[i][v * TL::VEC + e] = t[e];
    }
}

// One row of a copy tile: the lane's E values of row `row` (columns Tile::col(lane, v)).
template <int P, int N, int RC>
__device__ __forceinline__ void store_row_rc(void* rc, size_t slab, float scale, int row, int lane,
                                             const float (&vals)[Tile<P, N>::E]) {
  using TL = Tile<P, N>;
#pragma unroll
  for (int v = 0; v < TL::NVEC; ++v) {
    float t[TL::VEC];
#pragma unroll
    for (int e = 0; e < TL::VEC; ++e) t[e] = vals[v * TL::VEC + e];
    const size_t off = slab * P * N + static_cast<size_t>(row) * N + TL::col(lane, v);
    if constexpr (RC == REPLAY_RC_BF16)
      st_bf16_stream<TL::VEC>(static_cast<bf16*>(rc) + off, t);
    else if constexpr (RC == REPLAY_RC_FP16)
      st_f16_stream<TL::VEC>(static_cast<__half*>(rc) + off, t);
    else
      st_e4m3_stream<TL::VEC>(static_cast<uint8_t*>(rc) + off, scale, t);
  }
}

template <int P, int N, int RC>
__device__ __forceinline__ void store_tile_rc(void* rc, size_t slab, float scale, int warp, int lane,
                                              const float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E]) {
  using TL = Tile<P, N>;
#pragma unroll
  for (int i = 0; i < TL::RPW; ++i) store_row_rc<P, N, RC>(rc, slab, scale, TL::row(warp, i), lane, hv[i]);
}

// An NVFP4 row with slab scale sg: each 16-element block of the row (4 consecutive lanes)
// takes s_b = e4m3(block absmax / (6 sg)) and codes e2m1(h / (s_b sg)), every step one FP32
// operation; a block whose scale is 0 stores zero codes. Lane l's 4 columns are the unit of
// block l / 4, quarter l % 4 (layout above). The whole warp calls it (block maxima by shuffles).
template <int P, int N>
__device__ __forceinline__ void store_row_nvfp4(void* rc, uint8_t* bscale, size_t slab, float sg, int row, int lane,
                                                const float (&t)[Tile<P, N>::E]) {
  static_assert(N == 128 && Tile<P, N>::E == 4, "the NVFP4 copy is laid out for dstate 128");
  const float unit = __fmul_rn(kE2M1Max, sg);
  float bm = fmaxf(fmaxf(fabsf(t[0]), fabsf(t[1])), fmaxf(fabsf(t[2]), fabsf(t[3])));
  bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 1));
  bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 2));
  const unsigned int sb = float2_to_e4m3x2(__fdiv_rn(bm, unit), 0.f) & 0xffu;
  const float es = __fmul_rn(e4m3_to_float(sb), sg);
  unsigned int c01 = 0, c23 = 0;  // E2M1 codes of columns (0, 1) and (2, 3), low nibble first
  if (es > 0.f) {
    c01 = float2_to_e2m1x2(__fdiv_rn(t[0], es), __fdiv_rn(t[1], es));
    c23 = float2_to_e2m1x2(__fdiv_rn(t[2], es), __fdiv_rn(t[3], es));
  }
  const unsigned int b0 = fp4_slot_a(c01 & 15u) | fp4_slot_b(c23 & 15u);
  const unsigned int b1 = fp4_slot_a(c01 >> 4) | fp4_slot_b(c23 >> 4);
  __stcs(reinterpret_cast<unsigned short*>(static_cast<uint8_t*>(rc) + slab * P * N / 2 +
                                           fp4_unit(row, lane >> 2, lane & 3)),
         static_cast<unsigned short>(b0 | (b1 << 8)));
  if ((lane & 3) == 0) __stcs(bscale + (slab * P + row) * (N / kFp4Block) + (lane >> 2), static_cast<uint8_t>(sb));
}

template <int P, int N>
__device__ __forceinline__ void store_tile_nvfp4(void* rc, uint8_t* bscale, size_t slab, float sg, int warp,
                                                 int lane, const float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E]) {
  using TL = Tile<P, N>;
#pragma unroll
  for (int i = 0; i < TL::RPW; ++i) store_row_nvfp4<P, N>(rc, bscale, slab, sg, TL::row(warp, i), lane, hv[i]);
}

// The same decision with a 16-bit draw u16 (u = u16 / 2^16), in integers for FP16 normals:
// truncating an FP32 at or above 2^-14 to FP16 drops its 13 low fraction bits t, the fraction of
// the spacing is t / 2^13 exactly, and u < t / 2^13 iff u16 < 8 t. Magnitudes from 65504 up
// saturate; FP16 subnormals and zero take the general routine.
__device__ __forceinline__ unsigned short f16_sr16(float v, unsigned u16) {
  const unsigned b = __float_as_uint(v), a = b & 0x7fffffffu;
  const unsigned sign = (b >> 16) & 0x8000u;
  if (a >= 0x38800000u) {
    const unsigned mag = (a >> 13) - 0x1C000u;  // FP16 exponent and fraction, truncated
    if (mag >= 0x7BFFu) return static_cast<unsigned short>(sign | 0x7BFFu);
    return static_cast<unsigned short>(sign | (mag + (u16 < ((a & 0x1fffu) << 3) ? 1u : 0u)));
  }
  return f16_sr(v, static_cast<float>(u16) * 0x1p-16f);
}

// An FP16 row by stochastic rounding: element e of slab `slab` (of num_slabs) written by flush
// `epoch` takes draw (epoch * num_slabs + slab) * P*N + e. A lane's VEC columns start at a
// multiple of VEC, so they share one generator output (two lanes share it when VEC is 2).
template <int P, int N>
__device__ __forceinline__ void store_row_f16_sr(void* rc, size_t slab, unsigned long long epoch,
                                                 unsigned long long num_slabs, int row, int lane,
                                                 const float (&vals)[Tile<P, N>::E]) {
  using TL = Tile<P, N>;
  static_assert(TL::VEC == 2 || TL::VEC == 4, "a lane's columns lie within one generator output");
  const unsigned long long base = (epoch * num_slabs + slab) * static_cast<unsigned long long>(P * N);
#pragma unroll
  for (int v = 0; v < TL::NVEC; ++v) {
    const int e0 = row * N + TL::col(lane, v);
    const unsigned long long z = splitmix64_at(kSrSeed, (base + e0) >> 2);
    unsigned short c[TL::VEC];
#pragma unroll
    for (int e = 0; e < TL::VEC; ++e) {
      const int chunk = (e0 + e) & 3;  // base is a multiple of 4
      c[e] = f16_sr16(vals[v * TL::VEC + e], static_cast<unsigned>(z >> (48 - 16 * chunk)) & 0xffffu);
    }
    __half* p = static_cast<__half*>(rc) + slab * P * N + e0;
    if constexpr (TL::VEC == 4) {
      uint2 w;
      w.x = c[0] | (static_cast<unsigned int>(c[1]) << 16);
      w.y = c[2] | (static_cast<unsigned int>(c[3]) << 16);
      __stcs(reinterpret_cast<uint2*>(p), w);
    } else {
      __stcs(reinterpret_cast<unsigned int*>(p), c[0] | (static_cast<unsigned int>(c[1]) << 16));
    }
  }
}

template <int P, int N>
__device__ __forceinline__ void store_tile_f16_sr(void* rc, size_t slab, unsigned long long epoch,
                                                  unsigned long long num_slabs, int warp, int lane,
                                                  const float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E]) {
  using TL = Tile<P, N>;
#pragma unroll
  for (int i = 0; i < TL::RPW; ++i) store_row_f16_sr<P, N>(rc, slab, epoch, num_slabs, TL::row(warp, i), lane, hv[i]);
}

// ------------------------------------------------------------------ warp reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, off));
  return v;
}

// Sum M per-lane values over the 32 lanes at once ("transpose reduction"): each halving
// step trades half of the values with the lane `off` away, so M sums cost
// M-1 + log2(32/M) shuffles instead of 5M. Lane l ends with the sum of value
// transpose_index<M>(l); the lanes with (l & (32/M - 1)) == 0 hold distinct values.
template <int M>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[M], int lane) {
  static_assert(M >= 1 && M <= 32 && (M & (M - 1)) == 0, "M must be a power of two <= 32");
#pragma unroll
  for (int w = M / 2, off = 16; w >= 1; w >>= 1, off >>= 1) {
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? v[i] : v[i + w];
      const float keep = up ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, off);
    }
  }
  float s = v[0];
#pragma unroll
  for (int off = 16 / M; off >= 1; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
  return s;
}
template <int M>
__device__ __forceinline__ int transpose_index(int lane) {
  int idx = 0;
#pragma unroll
  for (int w = M / 2, off = 16; w >= 1; w >>= 1, off >>= 1)
    if (lane & off) idx += w;
  return idx;
}
template <int M>
__device__ __forceinline__ bool transpose_leader(int lane) {
  return (lane & (32 / M - 1)) == 0;
}

// ------------------------------------------------------------------ small helpers
// Load RPW consecutive elements of one record row (rows w*RPW.. of an x vector).
template <int RPW, class T>
__device__ __forceinline__ void load_rows(const T* p, float (&o)[RPW]) {
#pragma unroll
  for (int i = 0; i < RPW; i += 4) {
    float t[4];
    ldv<4>(p + i, t);
#pragma unroll
    for (int e = 0; e < 4; ++e) o[i + e] = t[e];
  }
}

// One 16-byte chunk (8 bf16 or 4 FP32 values) widened to float, and its FP32 store.
template <class T>
__device__ __forceinline__ void load16(const T* p, float (&o)[16 / sizeof(T)]) {
  if constexpr (sizeof(T) == 4) {
    ldv<4>(reinterpret_cast<const float*>(p), o);
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const unsigned w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      o[2 * i] = f.x;
      o[2 * i + 1] = f.y;
    }
  }
}
template <int EPC>
__device__ __forceinline__ void store16f(float* p, const float (&v)[EPC]) {
#pragma unroll
  for (int i = 0; i < EPC; i += 4) *reinterpret_cast<float4*>(p + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
}

__device__ __forceinline__ int ring_slot(int start, int s, int cap) {
  int v = start + s;
  return v >= cap ? v - cap : v;
}

__device__ __forceinline__ void set_status(int* status, int bit) { atomicOr(status, bit); }

// 16-byte asynchronous global -> shared copy (L2 only), and the wait for all of a thread's
// outstanding copies. Both addresses must be 16-byte aligned.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }
// cp.async groups: commit the copies issued so far as one group; wait until at most N groups
// are still in flight.
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// One-shot bulk copy global -> shared by the tensor memory accelerator, tracked by an
// mbarrier in shared memory: one thread initialises the barrier (count 1), arms it with the
// byte count, issues the copy and later waits on phase 0 while the others wait at a CTA
// barrier (spinning warps would take issue slots from the SM's other CTAs). The data never passes
// through registers or L1, so a CTA keeps its whole slab in flight however few registers it
// has. Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return static_cast<unsigned>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(unsigned long long* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(bar)) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
// The copy is marked evict-first in L2 (read once per call), like the streaming loads, so
// the state stream does not push the ring records out of L2.
__device__ __forceinline__ void bulk_load(void* smem, const void* gmem, unsigned int bytes, unsigned long long* bar) {
  unsigned long long policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(policy));
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::"r"(
          smem_u32(smem)),
      "l"(gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}
// Wait for phase `parity` of the barrier for at most about `ns` nanoseconds of the global
// timer (and a fixed number of polls); false if it has not completed by then.
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, unsigned int parity, unsigned long long ns) {
  const unsigned a = smem_u32(bar);
  unsigned long long t0 = 0;
  for (int it = 0; it < (1 << 28); ++it) {
    unsigned done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
    if ((it & 255) == 0) {
      const unsigned long long t = global_ns();
      if (it == 0) t0 = t;
      else if (t - t0 > ns) return false;
    }
  }
  return false;
}
constexpr unsigned long long kCopyWaitNs = 1000000000ull;  // 1 s: far beyond any copy's time

// Programmatic dependent launch: a primary kernel lets its dependent start early; the
// dependent waits, where it first needs the primary's results, until the primary grid has
// completed and its writes are visible. Without the launch attribute both are no-ops.
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

// Last-CTA-done update of a sequence's metadata: every CTA of sequence b calls this once,
// from its single reader thread, after the value it read from meta[b] has been consumed
// (written to shared memory and past a CTA barrier), so its read is complete; the last of
// the H arrivals writes the new value and re-arms the counter. The new value is only read
// by later launches. Nothing waits, so nothing can hang.
__device__ __forceinline__ void arrive_and_publish(const StoreView& sv, int b, int4 next, int count) {
  const int old = atomicAdd(&sv.arrive[b], 1);
  if (old == count - 1) {
    sv.arrive[b] = 0;
    sv.meta[b] = next;
  }
}

}  // namespace rssm
