// replay_step for stores with a read copy (bf16, FP16, E4M3 or NVFP4 at dstate 128) when the
// host knows that no sequence flushes: one persistent kernel that streams the copy.
//
// Source: "ReplaySSM: Rethinking State Storage for Faster Hybrid-Model Decoding" (NVIDIA
// Developer blog), sections "How ReplaySSM represents the state" (a non-flush step computes
// y_k = Gamma_k (h0 . C_k) + sum_s gamma(k,s) dt_s (B_s . C_k) x_s + D x_k from the checkpoint
// and the buffered records, and writes only the new record) and "Benefit 3" (non-flush steps
// read the low-precision copy of the checkpoint).
//
// Why a different kernel: a non-flush read-copy step only reads, and its copy slabs are 2-8x
// smaller than the FP32 ones, so a one-shot CTA per few heads keeps too few bytes in flight
// and pays a load-then-compute latency per CTA (the per-head kernels reach 0.5-0.8 of the
// copy bandwidth). Here one CTA per SM runs a pipeline over "units" (U consecutive heads of one
// group of one sequence, about 16 KB of copy):
//   - a producer thread issues, per unit, bulk copies (cp.async.bulk, the tensor memory
//     accelerator) of everything the unit reads -- the copy slabs (and NVFP4 block scales),
//     the slab scales, the live x records of its heads, the group's live B records, the
//     current x, B, C, the heads' dt ring and current dt -- into one of S shared-memory stages,
//     completing on the stage's "full" mbarrier;
//   - two consumer halves of 8 warps take alternate units: they compute the group's B_s . C
//     dots and the heads' record weights themselves (so no prep kernel runs before this one),
//     then the outputs, append the record, release the stage on its "empty" mbarrier and
//     arrive on the sequence's counter (the last of its units publishes the new ring pointer).
// Every wait is bounded (1 s of the global timer): a copy that does not land sets
// REPLAY_DEV_COPY_TIMEOUT and gives NaN outputs. A sequence whose ring is full (a flush plan,
// the host's hint being wrong) is folded by the consumers from global memory.
#include <algorithm>

#include "launch.h"
#include "replay_core.cuh"

namespace rssm {
namespace {

constexpr int kHalf = 256;                    // threads of one consumer half (8 warps)
constexpr int kStreamThreads = 2 * kHalf + 32;  // two halves and the producer warp
constexpr int kMaxStages = 12;
constexpr int kMaxU = 4;

// Heads per unit: about 16 KB of copy (plus 2 KB of NVFP4 block scales).
template <int RC>
constexpr int stream_heads() {
  return RC == REPLAY_RC_NVFP4 ? 4 : (RC == REPLAY_RC_FP8E4M3 ? 2 : 1);
}

// Byte layout of one stage (every part 128-byte aligned) and the work split, computed on the
// host.
struct StreamPlan {
  int U, upg, nunits, per_cta, stages, lrec;  // lrec: x/B record slots kept per head (L - 1)
  unsigned stage;                             // bytes per stage
  unsigned o_state, o_bsc, o_sc, o_xr, o_br, o_xc, o_bc, o_c, o_dtr, o_dtc;
  unsigned state_bytes, bsc_bytes;            // per unit: copy codes, NVFP4 block scales
};

__device__ __forceinline__ void bar_half(int h) {  // named barrier of one consumer half
  asm volatile("bar.sync %0, %1;" ::"r"(h + 1), "n"(kHalf) : "memory");
}
struct HalfSync {
  int h;
  __device__ void operator()() const { bar_half(h); }
};

__device__ __forceinline__ void mbar_init_count(unsigned long long* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive1(unsigned long long* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// Bulk copy global -> shared completing on `bar` (16-byte aligned addresses, size a multiple
// of 16), evict-first in L2 when `stream` (data read once per call), else normal.
__device__ __forceinline__ void bulk_g2s(void* smem, const void* gmem, unsigned bytes, unsigned long long* bar,
                                         unsigned long long policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::"r"(
          smem_u32(smem)),
      "l"(gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// The 16-byte aligned window [a & ~15, ...) covering `bytes` bytes at address a.
__device__ __forceinline__ unsigned window_bytes(const void* a, unsigned bytes) {
  const unsigned off = static_cast<unsigned>(reinterpret_cast<uintptr_t>(a) & 15u);
  return (off + bytes + 15u) & ~15u;
}
__device__ __forceinline__ const void* window_base(const void* a) {
  return reinterpret_cast<const void*>(reinterpret_cast<uintptr_t>(a) & ~static_cast<uintptr_t>(15));
}

// Scratch of one consumer half (static shared memory).
template <int N>
struct HalfScratch {
  float bc[kMaxCap];                 // B_s . C of the unit's group
  float coef[kMaxU][32];             // c_s = w_s (B_s . C), per head
  float gam[kMaxU];                  // Gamma_k, per head
  float red[kWarps];
  float cmax[4];
  int ok;
  __half ch[2][N];                   // NVFP4: C scaled by 2^sc, high and low FP16 parts
  float ys[kWarps][32];              // NVFP4: h0 . C of each warp's 32 rows
};

// ---- the flush of one unit when its plan says so (not expected on this path): head by head,
// from the checkpoint (or, for a shared checkpoint, the copy) and the records in global memory.
template <int P, int N, class T, int RC>
__device__ __noinline__ void stream_flush_unit(const StoreView& sv, const T* __restrict__ x,
                                               const T* __restrict__ B, const T* __restrict__ C,
                                               const T* __restrict__ dt, float* __restrict__ y, int b, int g,
                                               int h0, int U, int start, int n, int epoch, int hf,
                                               HalfScratch<N>& hs) {
  using TL = Tile<P, N>;
  constexpr int RPW = TL::RPW, E = TL::E;
  const int lt = threadIdx.x & (kHalf - 1), warp = lt >> 5, lane = lt & 31;
  const int cap = sv.cap, k = n + 1;
  const size_t bo = (static_cast<size_t>(b) * sv.G + g) * N;
  const int myrow = warp * RPW + transpose_index<RPW>(lane);
  float cv[E];
  load_cols<P, N>(C + bo, lane, cv);
  for (int hh = 0; hh < U; ++hh) {
    const int h = h0 + hh;
    const size_t slab = static_cast<size_t>(b) * sv.H + h;
    const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
    const size_t xo = slab * P;
    auto x_of = [&](int s) { return s < n ? ring.x + static_cast<size_t>(ring_slot(start, s, cap)) * P : x + xo; };
    auto b_of = [&](int s) { return s < n ? ring.b + static_cast<size_t>(ring_slot(start, s, cap)) * N : B + bo; };
    if (warp == 0) {
      auto dt_of = [&](int s) { return to_f(s < n ? ring.dt[ring_slot(start, s, cap)] : dt[slab]); };
      const float d0 = lane < k ? dt_of(lane) : 0.f;
      const float d1 = lane + 32 < k ? dt_of(lane + 32) : 0.f;
      const RecordWeights rw = record_weights(d0, d1, k, sv.A[h], lane);
      if (lane < k) hs.bc[lane] = rw.w0;
      if (lane + 32 < k) hs.bc[lane + 32] = rw.w1;
      if (lane == 0) hs.gam[0] = rw.gam;
    }
    float hv[RPW][E];
    if (sv.shared) {
      const float scale = RC == REPLAY_RC_FP8E4M3 || RC == REPLAY_RC_NVFP4 ? sv.scale[slab] : 1.f;
      load_tile_rc<P, N, RC>(sv.rc, slab, scale, warp, lane, hv, sv.bscale);
    } else {
      load_checkpoint<P, N>(sv, slab, warp, lane, hv);
    }
    bar_half(hf);
    const float gam = hs.gam[0];
#pragma unroll
    for (int i = 0; i < RPW; ++i)
#pragma unroll
      for (int e = 0; e < E; ++e) hv[i][e] *= gam;
    for (int s = 0; s < k; ++s) {
      float u[RPW], bv[E];
      load_rows<RPW>(x_of(s) + warp * RPW, u);
      load_cols<P, N>(b_of(s), lane, bv);
      const float w = hs.bc[s];
#pragma unroll
      for (int i = 0; i < RPW; ++i)
#pragma unroll
        for (int e = 0; e < E; ++e) hv[i][e] = fmaf(w * u[i], bv[e], hv[i][e]);
    }
    float zero[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) zero[i] = 0.f;
    const float sum = tile_rows_dot<P, N>(hv, cv, 1.f, zero, lane);
    if (transpose_leader<RPW>(lane)) y[xo + myrow] = fmaf(sv.D[h], to_f(x[xo + myrow]), sum);
    write_checkpoint<P, N, RC, HalfSync>(sv, slab, hs.red, hv, epoch, HalfSync{hf});
    bar_half(hf);  // the weights are read before the next head's are written
  }
}

// ---- outputs of a unit from the stage (bf16, FP16, E4M3 copies): warp w takes RW rows of
// head (w * RW) / P; lane l columns 4l .. 4l+3; the k records' share on lanes s < k.
template <int P, int N, class T, int RC, int U>
__device__ __forceinline__ void stream_outputs_packed(const StreamPlan& pl, const uint8_t* stg, float* y,
                                                      size_t slab0, int n, HalfScratch<N>& hs, const float* Dh,
                                                      const float* scl) {
  static_assert(N == 128, "stage rows hold 128 columns");
  constexpr int ESZ = RC == REPLAY_RC_FP8E4M3 ? 1 : 2;
  constexpr int RW = U * P / kWarps;  // rows per warp
  using PT = typename PackOf<RC, 4>::type;
  const int lt = threadIdx.x & (kHalf - 1), warp = lt >> 5, lane = lt & 31;
  const int hh = warp * RW / P, r0 = (warp * RW) % P, k = n + 1;
  const T* cst = reinterpret_cast<const T*>(stg + pl.o_c);
  float2 cv2[2];
  {
    float cv[4];
    ldv<4>(cst + 4 * lane, cv);
    cv2[0] = make_float2(cv[0], cv[1]);
    cv2[1] = make_float2(cv[2], cv[3]);
  }
  // the records' share: lane s holds record s (the current record is s = n)
  float ex[RW];
  if (lane < k) {
    const T* xs = lane < n ? reinterpret_cast<const T*>(stg + pl.o_xr) + (static_cast<size_t>(hh) * pl.lrec + lane) * P
                           : reinterpret_cast<const T*>(stg + pl.o_xc) + hh * P;
    load_rows<RW>(xs + r0, ex);
    const float c = hs.coef[hh][lane];
#pragma unroll
    for (int i = 0; i < RW; ++i) ex[i] *= c;
  } else {
#pragma unroll
    for (int i = 0; i < RW; ++i) ex[i] = 0.f;
  }
  const float gs = hs.gam[hh] * scl[hh];
  const uint8_t* rows = stg + pl.o_state + (static_cast<size_t>(hh) * P * N + static_cast<size_t>(r0) * N + 4 * lane) * ESZ;
  float part[RW];
#pragma unroll
  for (int i = 0; i < RW; ++i) {
    float2 w[2];
    unpack_pairs<RC, 4>(*reinterpret_cast<const PT*>(rows + static_cast<size_t>(i) * N * ESZ), w);
    float2 hc = __ffma2_rn(w[0], cv2[0], make_float2(0.f, 0.f));
    hc = __ffma2_rn(w[1], cv2[1], hc);
    part[i] = fmaf(gs, hc.x + hc.y, ex[i]);
  }
  const float sum = warp_transpose_reduce<RW>(part, lane);
  if (transpose_leader<RW>(lane)) {
    const int row = r0 + transpose_index<RW>(lane);
    const T* xc = reinterpret_cast<const T*>(stg + pl.o_xc) + hh * P;
    y[(slab0 + hh) * P + row] = fmaf(Dh[hh], to_f(xc[row]), sum);
  }
}

// ---- outputs of a unit from an NVFP4 stage: two warps per head, 32 rows each; h0 . C on the
// tensor cores (mma.sync m16n8k16, f16 in, FP32 accumulate) as in the per-head NVFP4 kernel:
// codes placed as FP16 by integer ops, scaled by their block scale, C split into an FP16 high
// and low part (columns 0 and 1 of the B operand).
__device__ __forceinline__ void mma16816(float (&d)[4], unsigned a0, unsigned a1, unsigned a2, unsigned a3,
                                         unsigned b0, unsigned b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ unsigned prmt_b32(unsigned a, unsigned b, unsigned sel) {
  unsigned d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ unsigned placed_a(unsigned w) { return w & 0x8E8E8E8Eu; }
__device__ __forceinline__ unsigned placed_b(unsigned w) { return ((w >> 3) & 0x0E0E0E0Eu) | ((w << 7) & 0x80808080u); }
template <int I>
__device__ __forceinline__ unsigned fp16_pair_of(unsigned x) {
  return prmt_b32(x, 0u, 4u | (I << 4) | (4u << 8) | ((I + 1) << 12));
}
template <int I>
__device__ __forceinline__ __half2 scale_pair_of(unsigned w) {
  const unsigned t = (prmt_b32(w, 0u, I | (4u << 4) | ((I + 1) << 8) | (4u << 12)) << 7) & 0x3F803F80u;
  return __hmul2(*reinterpret_cast<const __half2*>(&t), __float2half2_rn(256.f));
}
__device__ __forceinline__ unsigned times(unsigned p, __half s) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&p), __half2half2(s));
  return *reinterpret_cast<const unsigned*>(&r);
}

template <int P, int N, class T>
__device__ __forceinline__ void stream_outputs_nvfp4(const StreamPlan& pl, const uint8_t* stg, float* y,
                                                     size_t slab0, int n, HalfScratch<N>& hs, const float* Dh,
                                                     const float* scl, float down) {
  static_assert(P == 64 && N == 128, "64 x 128 slabs");
  constexpr int NB = N / kFp4Block, CODE = P * N / 2, SCB = P * NB;
  const int lt = threadIdx.x & (kHalf - 1), warp = lt >> 5, lane = lt & 31;
  const int gq = lane >> 2, q = lane & 3, hh = warp >> 1, rbase = (warp & 1) * 32, k = n + 1;
  unsigned bf[NB][2];
#pragma unroll
  for (int bk = 0; bk < NB; ++bk)
#pragma unroll
    for (int j = 0; j < 2; ++j)
      bf[bk][j] = gq < 2 ? *reinterpret_cast<const unsigned*>(&hs.ch[gq][bk * kFp4Block + 4 * q + 2 * j]) : 0u;
  const uint8_t* codes = stg + pl.o_state + static_cast<size_t>(hh) * CODE;
  const uint8_t* scales = stg + pl.o_bsc + static_cast<size_t>(hh) * SCB;
#pragma unroll
  for (int m = 0; m < 2; ++m) {
    const int r0 = rbase + m * 16 + gq;
    const uint4 W0 = *reinterpret_cast<const uint4*>(codes + fp4_unit(r0, 0, q));
    const uint4 W1 = *reinterpret_cast<const uint4*>(codes + fp4_unit(r0 + 8, 0, q));
    const uint2 S0 = *reinterpret_cast<const uint2*>(scales + r0 * NB);
    const uint2 S1 = *reinterpret_cast<const uint2*>(scales + (r0 + 8) * NB);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
      const unsigned w0 = wd == 0 ? W0.x : wd == 1 ? W0.y : wd == 2 ? W0.z : W0.w;
      const unsigned w1 = wd == 0 ? W1.x : wd == 1 ? W1.y : wd == 2 ? W1.z : W1.w;
      const unsigned sw0 = wd < 2 ? S0.x : S0.y, sw1 = wd < 2 ? S1.x : S1.y;
      const __half2 sc0 = (wd & 1) ? scale_pair_of<2>(sw0) : scale_pair_of<0>(sw0);
      const __half2 sc1 = (wd & 1) ? scale_pair_of<2>(sw1) : scale_pair_of<0>(sw1);
      const unsigned a0 = placed_a(w0), b0 = placed_b(w0), a1 = placed_a(w1), b1 = placed_b(w1);
      {
        const __half s0 = __low2half(sc0), s1 = __low2half(sc1);
        mma16816(acc, times(fp16_pair_of<0>(a0), s0), times(fp16_pair_of<0>(a1), s1), times(fp16_pair_of<0>(b0), s0),
                 times(fp16_pair_of<0>(b1), s1), bf[2 * wd][0], bf[2 * wd][1]);
      }
      {
        const __half s0 = __high2half(sc0), s1 = __high2half(sc1);
        mma16816(acc, times(fp16_pair_of<2>(a0), s0), times(fp16_pair_of<2>(a1), s1), times(fp16_pair_of<2>(b0), s0),
                 times(fp16_pair_of<2>(b1), s1), bf[2 * wd + 1][0], bf[2 * wd + 1][1]);
      }
    }
    if (q == 0) {
      hs.ys[warp][m * 16 + gq] = acc[0] + acc[1];
      hs.ys[warp][m * 16 + gq + 8] = acc[2] + acc[3];
    }
  }
  __syncwarp();
  // row rbase + lane: records' share, then y
  const int row = rbase + lane;
  float ex = 0.f;
  const T* xr = reinterpret_cast<const T*>(stg + pl.o_xr) + static_cast<size_t>(hh) * pl.lrec * P + row;
  for (int s = 0; s < n; ++s) ex = fmaf(hs.coef[hh][s], to_f(xr[static_cast<size_t>(s) * P]), ex);
  const float xcur = to_f(reinterpret_cast<const T*>(stg + pl.o_xc)[hh * P + row]);
  ex = fmaf(hs.coef[hh][n], xcur, ex);
  const float gsc = hs.gam[hh] * scl[hh] * down;
  y[(slab0 + hh) * P + row] = fmaf(Dh[hh], xcur, fmaf(gsc, hs.ys[warp][lane], ex));
  (void)k;
}

template <int P, int N, class T, int RC>
__global__ void __launch_bounds__(kStreamThreads, 1)
replay_step_stream_kernel(StoreView sv, const T* __restrict__ x, const T* __restrict__ B,
                          const T* __restrict__ C, const T* __restrict__ dt, float* __restrict__ y,
                          StreamPlan pl) {
  constexpr int U = stream_heads<RC>();
  constexpr int ESZ = sizeof(T);
  constexpr unsigned SLAB = RC == REPLAY_RC_NVFP4 ? P * N / 2 : P * N * (RC == REPLAY_RC_FP8E4M3 ? 1 : 2);
  constexpr bool SCALED = RC == REPLAY_RC_FP8E4M3 || RC == REPLAY_RC_NVFP4;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) unsigned long long s_full[kMaxStages], s_empty[kMaxStages];
  __shared__ int4 s_hdr[kMaxStages];  // {start, n, epoch, 1 = records copied / 0 = bad meta / 2 = flush}
  __shared__ HalfScratch<N> s_half[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = pl.stages;
  const int first = blockIdx.x * pl.per_cta;
  const int mine = max(0, min(pl.per_cta, pl.nunits - first));
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init_count(&s_full[s], 2);   // the producer's two arrivals: state, then records
      mbar_init_count(&s_empty[s], 1);  // the consumer half's leader
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  const int cap = sv.cap;
  auto unit_of = [&](int u, int& b, int& g, int& h0) {
    const int hc = u % pl.upg, bg = u / pl.upg;
    g = bg % sv.G;
    b = bg / sv.G;
    h0 = g * sv.hpg + hc * U;
  };

  if (warp == 2 * kWarps) {  // ---------------------------------------------- producer
    if (lane != 0) return;
    unsigned long long stream_pol, keep_pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(stream_pol));
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(keep_pol));
    int cur_b = -1;
    int4 m = make_int4(0, 0, 0, 0);
    for (int j = 0; j < mine; ++j) {
      const int st = j % S;
      if (j >= S && !mbar_wait(&s_empty[st], ((j / S) - 1) & 1, kCopyWaitNs)) {
        set_status(sv.status, REPLAY_DEV_COPY_TIMEOUT);
        return;  // consumers time out on the stages never filled
      }
      int b, g, h0;
      unit_of(first + j, b, g, h0);
      const size_t slab0 = static_cast<size_t>(b) * sv.H + h0;
      uint8_t* sb = smem + static_cast<size_t>(st) * pl.stage;
      const float* scw = sv.scale + slab0;
      const unsigned sc_bytes = SCALED ? window_bytes(scw, U * 4u) : 0u;
      mbar_arrive_tx(&s_full[st], pl.state_bytes + pl.bsc_bytes + sc_bytes);
      bulk_g2s(sb + pl.o_state, static_cast<const uint8_t*>(sv.rc) + slab0 * SLAB, pl.state_bytes, &s_full[st],
               stream_pol);
      if (RC == REPLAY_RC_NVFP4)
        bulk_g2s(sb + pl.o_bsc, sv.bscale + slab0 * (P * N / kFp4Block), pl.bsc_bytes, &s_full[st], stream_pol);
      if (SCALED) bulk_g2s(sb + pl.o_sc, window_base(scw), sc_bytes, &s_full[st], keep_pol);
      if (b != cur_b) {
        m = sv.meta[b];
        cur_b = b;
      }
      const int start = m.x, n = m.y;
      const bool ok = n >= 0 && n < cap && start >= 0 && start < cap;
      const bool flush = ok && n + 1 >= sv.L;
      s_hdr[st] = make_int4(start, n, m.w, ok ? (flush ? 2 : 1) : 0);
      if (!ok || flush) {  // nothing more to copy: the consumers read global memory
        mbar_arrive1(&s_full[st]);
        continue;
      }
      const T* dtc = dt + slab0;
      const unsigned dtc_bytes = window_bytes(dtc, U * ESZ);
      const int run1 = min(n, cap - start), run2 = n - run1;
      const unsigned xrec = P * ESZ, brec = N * ESZ;
      const unsigned bytes = static_cast<unsigned>(U * n) * xrec + n * brec + U * xrec + 2 * brec +
                             U * cap * ESZ + dtc_bytes;
      mbar_arrive_tx(&s_full[st], bytes);
      const T* xring = static_cast<const T*>(sv.xbuf) + slab0 * cap * P;
      for (int hh = 0; hh < U; ++hh) {
        uint8_t* dst = sb + pl.o_xr + static_cast<size_t>(hh) * pl.lrec * xrec;
        const T* src = xring + static_cast<size_t>(hh) * cap * P;
        if (run1 > 0) bulk_g2s(dst, src + static_cast<size_t>(start) * P, run1 * xrec, &s_full[st], keep_pol);
        if (run2 > 0) bulk_g2s(dst + run1 * xrec, src, run2 * xrec, &s_full[st], keep_pol);
      }
      const T* bring = static_cast<const T*>(sv.bbuf) + (static_cast<size_t>(b) * sv.G + g) * cap * N;
      if (run1 > 0) bulk_g2s(sb + pl.o_br, bring + static_cast<size_t>(start) * N, run1 * brec, &s_full[st], keep_pol);
      if (run2 > 0) bulk_g2s(sb + pl.o_br + run1 * brec, bring, run2 * brec, &s_full[st], keep_pol);
      const size_t bo = (static_cast<size_t>(b) * sv.G + g) * N;
      bulk_g2s(sb + pl.o_xc, x + slab0 * P, U * xrec, &s_full[st], keep_pol);
      bulk_g2s(sb + pl.o_bc, B + bo, brec, &s_full[st], keep_pol);
      bulk_g2s(sb + pl.o_c, C + bo, brec, &s_full[st], keep_pol);
      bulk_g2s(sb + pl.o_dtr, static_cast<const T*>(sv.dtbuf) + slab0 * cap, U * cap * ESZ, &s_full[st], keep_pol);
      bulk_g2s(sb + pl.o_dtc, window_base(dtc), dtc_bytes, &s_full[st], keep_pol);
    }
    return;
  }

  // ---------------------------------------------------------------- consumer halves
  const int hf = warp / kWarps, lt = tid & (kHalf - 1), lw = lt >> 5;
  HalfScratch<N>& hs = s_half[hf];
  const int units_per_seq = sv.G * pl.upg;
  for (int j = hf; j < mine; j += 2) {
    const int st = j % S;
    const uint8_t* stg = smem + static_cast<size_t>(st) * pl.stage;
    if (lt == 0) {
      bool ok = mbar_wait(&s_full[st], (j / S) & 1, kCopyWaitNs);
      if (!ok) {
        set_status(sv.status, REPLAY_DEV_COPY_TIMEOUT);
        ok = mbar_wait(&s_full[st], (j / S) & 1, kCopyWaitNs) && false;  // no copy outlives the CTA
      }
      hs.ok = ok;
    }
    bar_half(hf);
    int b, g, h0;
    unit_of(first + j, b, g, h0);
    const size_t slab0 = static_cast<size_t>(b) * sv.H + h0;
    const int4 hd = s_hdr[st];
    const int start = hd.x, n = hd.y, k = n + 1;
    const bool landed = hs.ok;
    if (!landed || hd.w == 0) {
      // bad metadata (the sequence's state is left alone, like every kernel does), or a copy
      // past its wait limit (REPLAY_DEV_COPY_TIMEOUT already set; the store needs a reset)
      for (int i = lt; i < U * P; i += kHalf) y[slab0 * P + i] = __int_as_float(0x7fc00000);
      bar_half(hf);
      if (lt == 0) {
        if (landed) set_status(sv.status, REPLAY_DEV_BAD_META);
        mbar_arrive1(&s_empty[st]);
      }
      if (!landed) return;  // the stages after it may never fill
      continue;
    }
    if (hd.w == 2) {  // a flush plan (the host expected none): fold from global memory
      stream_flush_unit<P, N, T, RC>(sv, x, B, C, dt, y, b, g, h0, U, start, n, hd.z, hf, hs);
      if (lt == 0) {
        arrive_and_publish(sv, b, make_int4(ring_slot(start, k, cap), 0, 0, hd.z + 1), units_per_seq);
        mbar_arrive1(&s_empty[st]);
      }
      continue;
    }
    const T* cst = reinterpret_cast<const T*>(stg + pl.o_c);
    // -- phase A: the group's B_s . C (records s < n from the ring, s = n the current B); for
    // NVFP4 also the partial maxima of |C|
    for (int s = lw; s < k; s += kWarps) {
      const T* bs = s < n ? reinterpret_cast<const T*>(stg + pl.o_br) + static_cast<size_t>(s) * N
                          : reinterpret_cast<const T*>(stg + pl.o_bc);
      float bv[4], cv[4];
      ldv<4>(bs + 4 * lane, bv);
      ldv<4>(cst + 4 * lane, cv);
      float d = bv[0] * cv[0];
      d = fmaf(bv[1], cv[1], d);
      d = fmaf(bv[2], cv[2], d);
      d = fmaf(bv[3], cv[3], d);
      d = warp_sum(d);
      if (lane == 0) hs.bc[s] = d;
    }
    if constexpr (RC == REPLAY_RC_NVFP4) {
      if (lw < 4) {
        const float mx = warp_max(fabsf(to_f(cst[lt])));
        if (lane == 0) hs.cmax[lw] = mx;
      }
    }
    bar_half(hf);
    // -- phase B: record weights of each head (warp hh), and for NVFP4 the split of C
    if (lw < U) {
      const T* dtr = reinterpret_cast<const T*>(stg + pl.o_dtr) + lw * cap;
      const T* dtcw = reinterpret_cast<const T*>(
          stg + pl.o_dtc + (reinterpret_cast<uintptr_t>(dt + slab0) & 15u));
      const float d0 = lane < n ? to_f(dtr[ring_slot(start, lane, cap)]) : (lane == n ? to_f(dtcw[lw]) : 0.f);
      const RecordWeights rw = record_weights(d0, 0.f, k, sv.A[h0 + lw], lane);
      if (lane < k) hs.coef[lw][lane] = rw.w0 * hs.bc[lane];
      if (lane == 0) hs.gam[lw] = rw.gam;
    }
    float down = 1.f;
    if constexpr (RC == REPLAY_RC_NVFP4) {
      const float cmax = fmaxf(fmaxf(hs.cmax[0], hs.cmax[1]), fmaxf(hs.cmax[2], hs.cmax[3]));
      const int ce = cmax > 0.f ? min(max(((__float_as_int(cmax) >> 23) & 0xff) - 127, -100), 100) : 0;
      down = __int_as_float((127 + 1 + ce) << 23);  // 2^14 / 2^sc
      if (lw >= 4) {
        const int c = lt - 128;
        const float cs = to_f(cst[c]) * __int_as_float((127 + 13 - ce) << 23);
        const __half hi = __float2half_rn(cs);
        hs.ch[0][c] = hi;
        hs.ch[1][c] = __float2half_rn(cs - __half2float(hi));
      }
    }
    bar_half(hf);
    // -- phase C: outputs, then the appends of this token's record at slot start + n
    float Dh[U], scl[U];
    const float* scw = reinterpret_cast<const float*>(stg + pl.o_sc + (reinterpret_cast<uintptr_t>(sv.scale + slab0) & 15u));
#pragma unroll
    for (int hh = 0; hh < U; ++hh) {
      Dh[hh] = sv.D[h0 + hh];
      scl[hh] = SCALED ? scw[hh] : 1.f;
    }
    if constexpr (RC == REPLAY_RC_NVFP4)
      stream_outputs_nvfp4<P, N, T>(pl, stg, y, slab0, n, hs, Dh, scl, down);
    else
      stream_outputs_packed<P, N, T, RC, U>(pl, stg, y, slab0, n, hs, Dh, scl);
    {
      const int slot = ring_slot(start, n, cap);
      constexpr int EPC = 16 / ESZ, XC = P / EPC, BC = N / EPC;
      T* xring = static_cast<T*>(sv.xbuf) + slab0 * cap * P;
      const T* xc = reinterpret_cast<const T*>(stg + pl.o_xc);
      if (lt < U * XC) {
        const int hh = lt / XC, c = lt - hh * XC;
        *reinterpret_cast<uint4*>(xring + (static_cast<size_t>(hh) * cap + slot) * P + c * EPC) =
            *reinterpret_cast<const uint4*>(xc + hh * P + c * EPC);
      } else if (h0 % sv.hpg == 0 && lt < U * XC + BC) {  // B once per group
        const int c = lt - U * XC;
        T* bring = static_cast<T*>(sv.bbuf) + (static_cast<size_t>(b) * sv.G + g) * cap * N;
        *reinterpret_cast<uint4*>(bring + static_cast<size_t>(slot) * N + c * EPC) =
            *reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(stg + pl.o_bc) + c * EPC);
      } else if (lt >= kHalf - U) {
        const int hh = lt - (kHalf - U);
        const T* dtcw = reinterpret_cast<const T*>(stg + pl.o_dtc + (reinterpret_cast<uintptr_t>(dt + slab0) & 15u));
        static_cast<T*>(sv.dtbuf)[(slab0 + hh) * cap + slot] = dtcw[hh];
      }
    }
    bar_half(hf);  // every read of the stage and of the half's scratch is done
    if (lt == 0) {
      mbar_arrive1(&s_empty[st]);
      arrive_and_publish(sv, b, make_int4(start, k, 0, hd.z), units_per_seq);
    }
  }
}

constexpr unsigned align128u(unsigned v) { return (v + 127u) & ~127u; }

template <int P, int N, class T, int RC>
int launch_stream(const StoreView& sv, const void* x, const void* B, const void* C, const void* dt, float* y,
                  cudaStream_t stream) {
  constexpr int U = stream_heads<RC>();
  constexpr unsigned ESZ = sizeof(T);
  constexpr unsigned SLAB = RC == REPLAY_RC_NVFP4 ? P * N / 2 : P * N * (RC == REPLAY_RC_FP8E4M3 ? 1 : 2);
  StreamPlan pl{};
  pl.U = U;
  pl.upg = sv.hpg / U;
  pl.nunits = sv.batch * sv.G * pl.upg;
  pl.lrec = sv.L - 1;
  pl.state_bytes = U * SLAB;
  pl.bsc_bytes = RC == REPLAY_RC_NVFP4 ? U * P * (N / kFp4Block) : 0;
  unsigned off = 0;
  auto take = [&](unsigned bytes) {
    const unsigned at = off;
    off = align128u(off + bytes);
    return at;
  };
  pl.o_state = take(pl.state_bytes);
  pl.o_bsc = take(pl.bsc_bytes);
  pl.o_sc = take(32);
  pl.o_xr = take(U * pl.lrec * P * ESZ);
  pl.o_br = take(pl.lrec * N * ESZ);
  pl.o_xc = take(U * P * ESZ);
  pl.o_bc = take(N * ESZ);
  pl.o_c = take(N * ESZ);
  pl.o_dtr = take(U * sv.cap * ESZ);
  pl.o_dtc = take(32);
  pl.stage = off;
  int dev = 0, smem_max = 0, sms = sv.sms;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return REPLAY_ECUDA;
  const unsigned static_bytes = 2 * sizeof(HalfScratch<N>) + kMaxStages * (16 + 16) + 256;
  // an even count: each consumer half then owns the stages of its parity, so a half never
  // waits on a stage a full round ahead of the one the other half is still filling
  const int stages = std::min(kMaxStages, static_cast<int>((smem_max - static_bytes) / pl.stage)) & ~1;
  if (stages < 4 || sms <= 0) return REPLAY_EUNSUPPORTED;
  pl.stages = stages;
  const int grid = std::min(sms, pl.nunits);
  pl.per_cta = (pl.nunits + grid - 1) / grid;
  const size_t smem = static_cast<size_t>(stages) * pl.stage;
  auto kern = replay_step_stream_kernel<P, N, T, RC>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return REPLAY_ECUDA;
  kern<<<grid, kStreamThreads, smem, stream>>>(sv, static_cast<const T*>(x), static_cast<const T*>(B),
                                                static_cast<const T*>(C), static_cast<const T*>(dt), y, pl);
  return cudaGetLastError() == cudaSuccess ? REPLAY_OK : REPLAY_ECUDA;
}

}  // namespace

bool step_streams(const StoreView& sv, const Shape& sh, int all_n, const void* dt) {
  if (sh.P != 64 || sh.N != 128) return false;
  const int rc = sh.read_copy;
  if (rc != REPLAY_RC_BF16 && rc != REPLAY_RC_FP16 && rc != REPLAY_RC_FP8E4M3 && rc != REPLAY_RC_NVFP4) return false;
  if (all_n < 0 || all_n + 1 >= sv.L || sv.L > 33 || sv.sms <= 0) return false;
  const int U = rc == REPLAY_RC_NVFP4 ? 4 : (rc == REPLAY_RC_FP8E4M3 ? 2 : 1);
  const int esz = sh.in_dtype == REPLAY_F32 ? 4 : 2;
  if (sv.hpg % U != 0) return false;
  if ((sv.cap * esz) % 16 != 0) return false;                   // the dt ring of a unit's heads
  if ((static_cast<long long>(sv.H) * esz) % 16 != 0 || (sv.H * 4) % 16 != 0) return false;  // windows
  if (reinterpret_cast<uintptr_t>(dt) % 16 != 0) return false;
  return true;
}

int launch_step_stream(const StoreView& sv, const Shape& sh, const void* x, const void* B, const void* C,
                       const void* dt, float* y, cudaStream_t stream) {
#define RSSM_STREAM(TT, RCC)                                                         \
  if (sh.in_dtype == RSSM_DTYPE_OF(TT) && sh.read_copy == RCC)                      \
    return launch_stream<64, 128, TT, RCC>(sv, x, B, C, dt, y, stream);
  RSSM_STREAM(float, REPLAY_RC_BF16) RSSM_STREAM(bf16, REPLAY_RC_BF16)
  RSSM_STREAM(float, REPLAY_RC_FP16) RSSM_STREAM(bf16, REPLAY_RC_FP16)
  RSSM_STREAM(float, REPLAY_RC_FP8E4M3) RSSM_STREAM(bf16, REPLAY_RC_FP8E4M3)
  RSSM_STREAM(float, REPLAY_RC_NVFP4) RSSM_STREAM(bf16, REPLAY_RC_NVFP4)
#undef RSSM_STREAM
  return REPLAY_EUNSUPPORTED;
}

}  // namespace rssm
