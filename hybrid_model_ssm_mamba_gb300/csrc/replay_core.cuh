// Device routines shared by the step, verify and flush kernels: folding buffered records
// into a checkpoint tile, and writing a new checkpoint with its read copy.
#pragma once

#include "common.cuh"

namespace rssm {

// Pointers to one (sequence, head) slab's ring records.
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

// Fold K records into the register tile of the checkpoint ("How ReplaySSM represents the
// state": the state after a window is the cumulative decay times the state before it plus
// the buffered records):
//     h <- Gamma_K * h + sum_{s<K} w_s x_s B_s^T,  w_s = exp(A sum_{r=s+1..K-1} dt_r) dt_s,
//     Gamma_K = exp(A sum_{r<K} dt_r).
// Records s < nring are ring slots (start + s) mod cap; record s == nring, when K > nring,
// is the current token (xcur, bcur, dtcur). The records are staged in shared memory as FP32
// (sm_x [K][P], sm_b [K][N], sm_dt [K]); every thread then forms its own w_s, so the suffix
// sums of dt are taken directly over each range, as in the definition. Starts and ends with
// a CTA barrier.
template <int P, int N, class T>
__device__ __forceinline__ void fold_records(const SlabRing<T>& ring, int start, int cap, int K,
                                             int nring, const T* xcur, const T* bcur, T dtcur,
                                             float A, float* sm_x, float* sm_b, float* sm_dt,
                                             float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E]) {
  using TL = Tile<P, N>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __syncthreads();  // shared staging buffers may still be read by an earlier phase
  for (int idx = tid; idx < K * P; idx += kThreads) {
    const int s = idx / P, p = idx - s * P;
    sm_x[idx] = s < nring ? to_f(ring.x[static_cast<size_t>(ring_slot(start, s, cap)) * P + p])
                          : to_f(xcur[p]);
  }
  for (int idx = tid; idx < K * N; idx += kThreads) {
    const int s = idx / N, c = idx - s * N;
    sm_b[idx] = s < nring ? to_f(ring.b[static_cast<size_t>(ring_slot(start, s, cap)) * N + c])
                          : to_f(bcur[c]);
  }
  if (tid < K) sm_dt[tid] = tid < nring ? to_f(ring.dt[ring_slot(start, tid, cap)]) : to_f(dtcur);
  __syncthreads();

  float tot = 0.f;
  for (int r = 0; r < K; ++r) tot += sm_dt[r];
  const float Gam = expf(A * tot);
#pragma unroll
  for (int i = 0; i < TL::RPW; ++i)
#pragma unroll
    for (int e = 0; e < TL::E; ++e) hv[i][e] *= Gam;

  float suf = 0.f;  // sum of dt over records after s
  for (int s = K - 1; s >= 0; --s) {
    const float dts = sm_dt[s];
    const float w = expf(A * suf) * dts;
    suf += dts;
    float u[TL::RPW];
#pragma unroll
    for (int i = 0; i < TL::RPW; i += 4) {
      const float4 t = *reinterpret_cast<const float4*>(sm_x + s * P + warp * TL::RPW + i);
      u[i] = w * t.x; u[i + 1] = w * t.y; u[i + 2] = w * t.z; u[i + 3] = w * t.w;
    }
    float bv[TL::E];
#pragma unroll
    for (int v = 0; v < TL::NVEC; ++v) {
      float t[TL::VEC];
      ldv<TL::VEC>(sm_b + s * N + TL::col(lane, v), t);
#pragma unroll
      for (int e = 0; e < TL::VEC; ++e) bv[v * TL::VEC + e] = t[e];
    }
#pragma unroll
    for (int i = 0; i < TL::RPW; ++i)
#pragma unroll
      for (int e = 0; e < TL::E; ++e) hv[i][e] = fmaf(u[i], bv[e], hv[i][e]);
  }
  __syncthreads();
}

// Write a new checkpoint tile: FP32 always, and the read copy cast independently from the
// same FP32 values ("Benefit 3: Limit error accumulation with separate precisions"). The
// E4M3 copy takes one FP32 scale per slab, absmax / 448 (1 for an all-zero slab).
template <int P, int N, int RC>
__device__ __forceinline__ void write_checkpoint(const StoreView& sv, size_t slab, float* s_red,
                                                 const float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E]) {
  using TL = Tile<P, N>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  store_tile_f32<P, N>(sv.h0 + slab * P * N, warp, lane, hv);
  if constexpr (RC == REPLAY_RC_BF16) {
    store_tile_rc<P, N, RC>(sv.rc, slab, 1.f, warp, lane, hv);
  } else if constexpr (RC == REPLAY_RC_FP8E4M3) {
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < TL::RPW; ++i)
#pragma unroll
      for (int e = 0; e < TL::E; ++e) m = fmaxf(m, fabsf(hv[i][e]));
    m = warp_max(m);
    __syncthreads();  // s_red may hold an earlier phase's values
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    float amax = s_red[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) amax = fmaxf(amax, s_red[w]);
    const float scale = amax > 0.f ? __fdiv_rn(amax, kE4M3Max) : 1.f;
    if (tid == 0) sv.scale[slab] = scale;
    store_tile_rc<P, N, RC>(sv.rc, slab, scale, warp, lane, hv);
  }
}

// Output of the tile's rows against the lane's columns of c: y[row] = gam * (h . c)[row]
// + extra[row], reduced across the warp; the transpose leader of each row gets the value.
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

}  // namespace rssm
