// Device routines shared by the step, verify and flush kernels: staging a slab's records
// in shared memory, folding them into a checkpoint tile, writing a new checkpoint with its
// read copy, and the per-warp record weights.
#pragma once

#include "common.cuh"

namespace rssm {

// Pointers to one (sequence, head) slab's ring records in global memory.
template <class T>
struct SlabRing {
  T* x;   // [cap][P] of this head
  T* b;   // [cap][N] of this head's group
  T* dt;  // [cap] of this head
};

template <int P, int N, class T>
__device__ __forceinline__ SlabRing<T> slab_ring(const StoreView& sv, int b, int h, int g) {
  const size_t slab = static_cast<size_t>(b) * sv.H + h;
  SlabRing<T> r;
  r.x = static_cast<T*>(sv.xbuf) + slab * sv.cap * P;
  r.b = static_cast<T*>(sv.bbuf) + (static_cast<size_t>(b) * sv.G + g) * sv.cap * N;
  r.dt = static_cast<T*>(sv.dtbuf) + slab * sv.cap;
  return r;
}

// Shared-memory image of a slab's records. In a ring image the slots are those of the global
// ring, so record s of the window sits at slot (start + s) mod cap in both.
template <class T>
struct RingImage {
  T* x;       // [slots][P]
  T* b;       // [slots][N]
  float* dt;  // [slots]
};

template <int P, int N, class T>
__host__ __device__ constexpr size_t ring_image_bytes(int cap) {
  return static_cast<size_t>(cap) * (P + N) * sizeof(T) + static_cast<size_t>(cap) * sizeof(float);
}

template <int P, int N, class T>
__device__ __forceinline__ RingImage<T> ring_image(void* smem, int cap) {
  RingImage<T> im;
  im.x = static_cast<T*>(smem);
  im.b = im.x + static_cast<size_t>(cap) * P;
  im.dt = reinterpret_cast<float*>(im.b + static_cast<size_t>(cap) * N);
  return im;
}

// Where the records of a window come from: s < nring are ring slots; s >= nring are "extra"
// records held by the caller's input arrays (the drafts of a verify), extra record e at
// x + e*xstride, b + e*bstride, dt[e*dtstride].
template <class T>
struct ExtraRecords {
  const T* x;
  const T* b;
  const T* dt;
  size_t xstride, bstride, dtstride;
};

// Copy records s = 0..K-1 of the window into the ring image with 16-byte cp.async chunks
// (all threads), and their dt values as FP32. The caller waits with cp_async_wait_all() and
// a CTA barrier before reading the image.
template <int P, int N, class T>
__device__ __forceinline__ void stage_records(const SlabRing<T>& ring, const RingImage<T>& im,
                                              int start, int cap, int K, int nring,
                                              const ExtraRecords<T>& ex) {
  constexpr int EPC = 16 / sizeof(T);  // elements per 16-byte chunk
  constexpr int XC = P / EPC, BC = N / EPC;
  static_assert(P % EPC == 0 && N % EPC == 0, "records must be whole 16-byte chunks");
  const int nx = K * XC, total = K * (XC + BC);
  for (int c = threadIdx.x; c < total; c += kThreads) {
    if (c < nx) {
      const int s = c / XC, off = (c - s * XC) * EPC;
      const int slot = ring_slot(start, s, cap);
      const T* src = s < nring ? ring.x + static_cast<size_t>(slot) * P : ex.x + (s - nring) * ex.xstride;
      cp_async16(im.x + slot * P + off, src + off);
    } else {
      const int c2 = c - nx;
      const int s = c2 / BC, off = (c2 - s * BC) * EPC;
      const int slot = ring_slot(start, s, cap);
      const T* src = s < nring ? ring.b + static_cast<size_t>(slot) * N : ex.b + (s - nring) * ex.bstride;
      cp_async16(im.b + slot * N + off, src + off);
    }
  }
  for (int s = threadIdx.x; s < K; s += kThreads)
    im.dt[ring_slot(start, s, cap)] =
        to_f(s < nring ? ring.dt[ring_slot(start, s, cap)] : ex.dt[(s - nring) * ex.dtstride]);
}

// Copy one record (x of this head, B of this group if `with_b`) from image slot `from` to
// global ring slot `to` with 16-byte vectors, and dt from `dtv`.
template <int P, int N, class T>
__device__ __forceinline__ void append_record(const SlabRing<T>& ring, const RingImage<T>& im, int from,
                                              int to, bool with_b, T dtv) {
  constexpr int EPC = 16 / sizeof(T);
  constexpr int XC = P / EPC, BC = N / EPC;
  const int t = threadIdx.x;
  if (t < XC) {
    *reinterpret_cast<uint4*>(ring.x + static_cast<size_t>(to) * P + t * EPC) =
        *reinterpret_cast<const uint4*>(im.x + from * P + t * EPC);
  } else if (with_b && t < XC + BC) {
    const int c = t - XC;
    *reinterpret_cast<uint4*>(ring.b + static_cast<size_t>(to) * N + c * EPC) =
        *reinterpret_cast<const uint4*>(im.b + from * N + c * EPC);
  } else if (t == XC + BC) {
    ring.dt[to] = dtv;
  }
}

// Load the checkpoint tile of a slab: FP32, or FP16 widened when the checkpoint is kept in
// FP16 (the caller handles a shared checkpoint, which is the read copy itself).
template <int P, int N>
__device__ __forceinline__ void load_checkpoint(const StoreView& sv, size_t slab, int warp, int lane,
                                                float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E]) {
  if constexpr (N <= 128) {
    if (sv.ckpt16) {
      load_tile_rc<P, N, REPLAY_RC_FP16>(sv.h0, slab, 1.f, warp, lane, hv);
      return;
    }
  }
  load_tile_f32<P, N>(sv.h0 + slab * P * N, warp, lane, hv);
}

// Write a new checkpoint tile: FP32 (or FP16 by stochastic rounding, when the checkpoint is
// kept in FP16), and the read copy cast independently from the same FP32 values ("Benefit 3:
// Limit error accumulation with separate precisions"). The E4M3 copy takes one FP32 scale per
// slab, absmax / 448 (1 for an all-zero slab). An FP16 copy rounds to nearest even, except when
// it is itself the checkpoint: then it is rounded stochastically, with draws indexed by the
// sequence's flush count `epoch` (the FP16 recurrence checkpoint with stochastic rounding the
// post's section "State quantization" cites); an FP16 checkpoint beside a read copy takes the
// same draws. Contains CTA barriers when the copy is E4M3 or NVFP4.
// The barrier of a whole CTA; kernels whose warps split into groups pass their own.
struct CtaSync {
  __device__ void operator()() const { __syncthreads(); }
};

// (tid: the thread's index among the kThreads threads that write the tile)
template <int P, int N, int RC, class Sync = CtaSync>
__device__ __forceinline__ void write_checkpoint(const StoreView& sv, size_t slab, float* s_red,
                                                 const float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E],
                                                 int epoch, Sync sync = Sync()) {
  using TL = Tile<P, N>;
  const int tid = threadIdx.x & (kThreads - 1), warp = tid >> 5, lane = tid & 31;
  if (!sv.shared) {  // shared: the copy only
    bool done = false;
    if constexpr (N <= 128 && RC != REPLAY_RC_NONE && RC != REPLAY_RC_FP16) {
      if (sv.ckpt16) {  // the FP16 checkpoint, rounded stochastically (draws of write `epoch`)
        store_tile_f16_sr<P, N>(sv.h0, slab, static_cast<unsigned int>(epoch),
                                static_cast<unsigned long long>(sv.batch) * sv.H, warp, lane, hv);
        done = true;
      }
    }
    if (!done) store_tile_f32<P, N>(sv.h0 + slab * P * N, warp, lane, hv);
  }
  if constexpr (RC == REPLAY_RC_BF16) {
    store_tile_rc<P, N, RC>(sv.rc, slab, 1.f, warp, lane, hv);
  } else if constexpr (RC == REPLAY_RC_FP16) {
    if (sv.shared)
      store_tile_f16_sr<P, N>(sv.rc, slab, static_cast<unsigned int>(epoch),
                              static_cast<unsigned long long>(sv.batch) * sv.H, warp, lane, hv);
    else
      store_tile_rc<P, N, RC>(sv.rc, slab, 1.f, warp, lane, hv);
  } else if constexpr (RC == REPLAY_RC_FP8E4M3 || RC == REPLAY_RC_NVFP4) {
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < TL::RPW; ++i)
#pragma unroll
      for (int e = 0; e < TL::E; ++e) m = fmaxf(m, fabsf(hv[i][e]));
    m = warp_max(m);
    sync();  // s_red may hold an earlier phase's values
    if (lane == 0) s_red[warp] = m;
    sync();
    float amax = s_red[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) amax = fmaxf(amax, s_red[w]);
    if constexpr (RC == REPLAY_RC_FP8E4M3) {
      const float scale = amax > 0.f ? __fdiv_rn(amax, kE4M3Max) : 1.f;
      if (tid == 0) sv.scale[slab] = scale;
      store_tile_rc<P, N, RC>(sv.rc, slab, scale, warp, lane, hv);
    } else {
      const float sg = amax > 0.f ? __fdiv_rn(amax, kE4M3Max * kE2M1Max) : 1.f;
      if (tid == 0) sv.scale[slab] = sg;
      store_tile_nvfp4<P, N>(sv.rc, sv.bscale, slab, sg, warp, lane, hv);
    }
  }
}

// The records' share of a non-flush output for the warp's RPW rows: record s (< k) sits on
// lane s (and lane s + 32) and contributes c_s x_s[row]; each lane returns its partial per
// row, to be summed over the warp.
template <int RPW, class T, class XOf>
__device__ __forceinline__ void record_terms(XOf x_of, const float* cf, int k, int warp, int lane,
                                             float (&ex)[RPW]) {
  if (lane < k) {
    load_rows<RPW>(x_of(lane) + warp * RPW, ex);
    const float c0 = cf[lane];
#pragma unroll
    for (int i = 0; i < RPW; ++i) ex[i] *= c0;
  } else {
#pragma unroll
    for (int i = 0; i < RPW; ++i) ex[i] = 0.f;
  }
  if (lane + 32 < k) {
    float x1[RPW];
    load_rows<RPW>(x_of(lane + 32) + warp * RPW, x1);
    const float c1 = cf[lane + 32];
#pragma unroll
    for (int i = 0; i < RPW; ++i) ex[i] = fmaf(c1, x1[i], ex[i]);
  }
}

// Output of the tile's rows against the lane's columns of c: gam * (h . c)[row] + extra[row],
// reduced across the warp; the transpose leader of each row gets the value.
template <int P, int N>
__device__ __forceinline__ float tile_rows_dot(const float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E],
                                               const float (&cv)[Tile<P, N>::E], float gam,
                                               const float (&extra)[Tile<P, N>::RPW], int lane) {
  using TL = Tile<P, N>;
  float part[TL::RPW];
#pragma unroll
  for (int i = 0; i < TL::RPW; ++i) {
    float hc = 0.f;
#pragma unroll
    for (int e = 0; e < TL::E; ++e) hc = fmaf(hv[i][e], cv[e], hc);
    part[i] = fmaf(gam, hc, extra[i]);
  }
  return warp_transpose_reduce<TL::RPW>(part, lane);
}

// The same output with the tile read row by row from a row-major FP32 slab in shared
// memory: a row's E values are live at a time, not the whole tile.
template <int P, int N>
__device__ __forceinline__ float smem_rows_dot(const float* slab, const float (&cv)[Tile<P, N>::E], float gam,
                                               const float (&extra)[Tile<P, N>::RPW], int warp, int lane) {
  using TL = Tile<P, N>;
  float part[TL::RPW];
#pragma unroll
  for (int i = 0; i < TL::RPW; ++i) {
    float2 hc = make_float2(0.f, 0.f);
#pragma unroll
    for (int v = 0; v < TL::NVEC; ++v) {
      float t[TL::VEC];
      ldv<TL::VEC>(slab + TL::row(warp, i) * N + TL::col(lane, v), t);
#pragma unroll
      for (int e = 0; e < TL::VEC; e += 2)
        hc = __ffma2_rn(make_float2(t[e], t[e + 1]), make_float2(cv[v * TL::VEC + e], cv[v * TL::VEC + e + 1]), hc);
    }
    part[i] = fmaf(gam, hc.x + hc.y, extra[i]);
  }
  return warp_transpose_reduce<TL::RPW>(part, lane);
}

// Weights of the records of one query, one record per lane (record s = lane, and lane+32
// when k > 32): w_s = exp(A sum_{r=s+1..k-1} dt_r) * dt_s, Gamma = exp(A sum_{r<k} dt_r).
// The suffix sums are warp scans (tree order) over the records' dt, each over its own range.
// exp is the fast hardware exponential (__expf): its relative error, a few 1e-7 at the
// exponents met here, is far inside the 1e-4 output bound.
struct RecordWeights {
  float w0, w1, gam;
};
__device__ __forceinline__ float suffix_scan(float v, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float a = __shfl_down_sync(kFull, v, off);
    if (lane + off < 32) v += a;
  }
  return v;  // inclusive: sum over lanes >= lane
}
__device__ __forceinline__ RecordWeights record_weights(float dt0, float dt1, int k, float A, int lane) {
  // dt0: record lane (0 if lane >= k); dt1: record lane + 32 (0 if lane + 32 >= k)
  RecordWeights r;
  const float in0 = suffix_scan(dt0, lane);
  float ex0 = __shfl_down_sync(kFull, in0, 1);  // exclusive: the records after s
  if (lane == 31) ex0 = 0.f;
  float tot1 = 0.f;
  r.w1 = 0.f;
  if (k > 32) {  // warp-uniform
    const float in1 = suffix_scan(dt1, lane);
    float ex1 = __shfl_down_sync(kFull, in1, 1);
    if (lane == 31) ex1 = 0.f;
    tot1 = __shfl_sync(kFull, in1, 0);
    ex0 += tot1;  // records 32..k-1 follow every record of the lower half
    r.w1 = lane + 32 < k ? __expf(A * ex1) * dt1 : 0.f;
  }
  r.w0 = lane < k ? __expf(A * ex0) * dt0 : 0.f;
  r.gam = __expf(A * (__shfl_sync(kFull, in0, 0) + tot1));
  return r;
}

// The same for two heads at once when k <= 16: lanes 0..15 carry records 0..15 of one head,
// lanes 16..31 those of the other, with each half-warp's own A. Suffix sums stay within a
// half-warp; w is the weight of the lane's record, gam its head's cumulative decay.
struct HalfWeights {
  float w, gam;
};
__device__ __forceinline__ HalfWeights record_weights_pair(float dtv, int k, float A, int lane) {
  const int hl = lane & 15;
  float in = dtv;
#pragma unroll
  for (int off = 1; off < 16; off <<= 1) {
    const float a = __shfl_down_sync(kFull, in, off, 16);
    if (hl + off < 16) in += a;
  }
  float ex = __shfl_down_sync(kFull, in, 1, 16);  // exclusive: the records after s
  if (hl == 15) ex = 0.f;
  HalfWeights r;
  r.w = hl < k ? __expf(A * ex) * dtv : 0.f;
  r.gam = __expf(A * __shfl_sync(kFull, in, lane & 16));
  return r;
}

// Fold K records into the register tile of the checkpoint, record s at image slot
// slot_of(s) ("How ReplaySSM represents the state": the state after a window is the
// cumulative decay times the state before it, plus the buffered records):
//     h <- Gamma_K * h + sum_{s<K} w_s x_s B_s^T,  w_s = exp(A sum_{r=s+1..K-1} dt_r) dt_s.
// Warp 0 forms the weights by warp scans; the CTA then stages u_s = w_s x_s and B_s in FP32
// (sm_u [K][P], sm_b [K][N]) so the rank-K update is three 16-byte shared loads and 32 FFMA
// per record per thread. Contains CTA barriers; s_w holds kMaxCap + 1 floats.
template <int P, int N, class T, class SlotOf>
__device__ __forceinline__ void fold_tile(const RingImage<T>& im, SlotOf slot_of, int K, float A,
                                          float* sm_u, float* sm_b, float* s_w,
                                          float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E]) {
  using TL = Tile<P, N>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {
    const float dt0 = lane < K ? im.dt[slot_of(lane)] : 0.f;
    const float dt1 = lane + 32 < K ? im.dt[slot_of(lane + 32)] : 0.f;
    const RecordWeights rw = record_weights(dt0, dt1, K, A, lane);
    if (lane < K) s_w[lane] = rw.w0;
    if (lane + 32 < K) s_w[lane + 32] = rw.w1;
    if (lane == 0) s_w[kMaxCap] = rw.gam;
  }
  __syncthreads();
  for (int idx = tid; idx < K * P; idx += kThreads) {
    const int s = idx / P, p = idx - s * P;
    sm_u[idx] = s_w[s] * to_f(im.x[slot_of(s) * P + p]);
  }
  for (int idx = tid; idx < K * N; idx += kThreads) {
    const int s = idx / N, c = idx - s * N;
    sm_b[idx] = to_f(im.b[slot_of(s) * N + c]);
  }
  __syncthreads();
  const float Gam = s_w[kMaxCap];
#pragma unroll
  for (int i = 0; i < TL::RPW; ++i)
#pragma unroll
    for (int e = 0; e < TL::E; ++e) hv[i][e] *= Gam;
  for (int s = 0; s < K; ++s) {
    float u[TL::RPW], bv[TL::E];
    load_rows<TL::RPW>(sm_u + s * P + warp * TL::RPW, u);
    load_cols<P, N>(sm_b + s * N, lane, bv);
#pragma unroll
    for (int i = 0; i < TL::RPW; ++i)
#pragma unroll
      for (int e = 0; e < TL::E; e += 2) {  // packed FP32 FMAs, two columns at a time
        const float2 r = __ffma2_rn(make_float2(u[i], u[i]), make_float2(bv[e], bv[e + 1]),
                                    make_float2(hv[i][e], hv[i][e + 1]));
        hv[i][e] = r.x;
        hv[i][e + 1] = r.y;
      }
  }
}

template <int P, int N>
__host__ __device__ constexpr size_t fold_staging_bytes(int K) {
  return static_cast<size_t>(K) * (P + N) * sizeof(float);
}

// Shared-memory plan of a kernel: a record image of `image_bytes`, then (128-byte aligned)
// the FP32 staging of a fold of up to `cap` records.
__host__ __device__ constexpr size_t align128(size_t v) { return (v + 127) / 128 * 128; }
template <int P, int N>
__host__ __device__ constexpr size_t smem_plan_bytes(size_t image_bytes, int cap) {
  return align128(image_bytes) + fold_staging_bytes<P, N>(cap);
}
__device__ __forceinline__ float* fold_staging(void* smem, size_t image_bytes) {
  return reinterpret_cast<float*>(static_cast<char*>(smem) + align128(image_bytes));
}

// Stage K records for a fold straight from global memory, in 16-byte chunks (all threads):
// sm_u[s][p] = w[s] * x_s[p] and sm_b[s][c] = B_s[c] in FP32; x_of(s) and b_of(s) give the
// record's x (this head) and B (this group). The caller puts a CTA barrier after it.
template <int P, int N, class T, class XOf, class BOf>
__device__ __forceinline__ void stage_weighted(XOf x_of, BOf b_of, const float* w, int K, float* sm_u,
                                               float* sm_b) {
  constexpr int EPC = 16 / sizeof(T), XC = P / EPC, BC = N / EPC;
  for (int c = threadIdx.x; c < K * (XC + BC); c += kThreads) {
    float v[EPC];
    if (c < K * XC) {
      const int s = c / XC, off = (c - s * XC) * EPC;
      load16<T>(x_of(s) + off, v);
      const float ws = w[s];
#pragma unroll
      for (int e = 0; e < EPC; ++e) v[e] *= ws;
      store16f<EPC>(sm_u + s * P + off, v);
    } else {
      const int c2 = c - K * XC;
      const int s = c2 / BC, off = (c2 - s * BC) * EPC;
      load16<T>(b_of(s) + off, v);
      store16f<EPC>(sm_b + s * N + off, v);
    }
  }
}

// The rank-K update of a checkpoint tile from staged records: h <- gam * h + sum_s u_s B_s^T.
template <int P, int N>
__device__ __forceinline__ void fold_staged(const float* sm_u, const float* sm_b, int K, float gam,
                                            float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E]) {
  using TL = Tile<P, N>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < TL::RPW; ++i)
#pragma unroll
    for (int e = 0; e < TL::E; ++e) hv[i][e] *= gam;
  for (int s = 0; s < K; ++s) {
    float u[TL::RPW], bv[TL::E];
    load_rows<TL::RPW>(sm_u + s * P + warp * TL::RPW, u);
    load_cols<P, N>(sm_b + s * N, lane, bv);
#pragma unroll
    for (int i = 0; i < TL::RPW; ++i)
#pragma unroll
      for (int e = 0; e < TL::E; e += 2) {  // packed FP32 FMAs, two columns at a time
        const float2 r = __ffma2_rn(make_float2(u[i], u[i]), make_float2(bv[e], bv[e + 1]),
                                    make_float2(hv[i][e], hv[i][e + 1]));
        hv[i][e] = r.x;
        hv[i][e + 1] = r.y;
      }
  }
}

// Weights of a fold of K records for one head, written by one warp: w[s] for s < K and
// Gamma_K at w[cap]. dt_of(s) gives record s's dt.
template <class DtOf>
__device__ __forceinline__ void write_fold_weights(DtOf dt_of, int K, float A, float* w, int cap, int lane) {
  const float d0 = lane < K ? dt_of(lane) : 0.f;
  const float d1 = lane + 32 < K ? dt_of(lane + 32) : 0.f;
  const RecordWeights rw = record_weights(d0, d1, K, A, lane);
  if (lane < K) w[lane] = rw.w0;
  if (lane + 32 < K) w[lane + 32] = rw.w1;
  if (lane == 0) w[cap] = rw.gam;
}

}  // namespace rssm
