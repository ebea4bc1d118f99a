// Conventional baselines: the load-update-store decode step and the snapshot-per-draft
// verify.
//
// Source: "ReplaySSM: Rethinking State Storage for Faster Hybrid-Model Decoding" (NVIDIA
// Developer blog), sections "Why SSM layers can become a decoding bottleneck" (each step
// loads the state, applies the decay and a rank-1 update, reads the output with C and
// stores the state back) and "Rollback for speculative decoding" (a snapshot after every
// draft: one read and T writes per step, the accepted prefix's snapshot is picked).
//
// Same slab tiling as the replay kernels (one CTA per (sequence, head), coalesced 16-byte
// streaming loads and stores), so the comparison measures the method, not the tiling.
#include "launch.h"
#include "replay_core.cuh"

namespace rssm {

template <int P, int N, class S>
__device__ __forceinline__ void load_state(const S* base, size_t slab, int warp, int lane,
                                           float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E]) {
  if constexpr (std::is_same<S, float>::value)
    load_tile_f32<P, N>(base + slab * P * N, warp, lane, hv);
  else
    load_tile_rc<P, N, REPLAY_RC_BF16>(base, slab, 1.f, warp, lane, hv);
}
template <int P, int N, class S>
__device__ __forceinline__ void store_state(S* base, size_t slab, int warp, int lane,
                                            const float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E]) {
  if constexpr (std::is_same<S, float>::value)
    store_tile_f32<P, N>(base + slab * P * N, warp, lane, hv);
  else
    store_tile_rc<P, N, REPLAY_RC_BF16>(base, slab, 1.f, warp, lane, hv);
}

// h <- exp(dt A) h + (dt x) B^T on the register tile; returns y for the transpose leader.
template <int P, int N, class T>
__device__ __forceinline__ float update_and_read(float (&hv)[Tile<P, N>::RPW][Tile<P, N>::E],
                                                 const T* x, const T* Bv, const T* Cv, float dtv,
                                                 float A, int warp, int lane) {
  using TL = Tile<P, N>;
  float bv[TL::E], cv[TL::E], xr[TL::RPW];
  load_cols<P, N>(Bv, lane, bv);
  load_cols<P, N>(Cv, lane, cv);
  load_rows<TL::RPW>(x + warp * TL::RPW, xr);
  const float a = expf(dtv * A);
#pragma unroll
  for (int i = 0; i < TL::RPW; ++i) {
    const float u = dtv * xr[i];
#pragma unroll
    for (int e = 0; e < TL::E; ++e) hv[i][e] = fmaf(a, hv[i][e], u * bv[e]);
  }
  float zero[TL::RPW];
#pragma unroll
  for (int i = 0; i < TL::RPW; ++i) zero[i] = 0.f;
  return tile_rows_dot<P, N>(hv, cv, 1.f, zero, lane);
}

template <int P, int N, class T, class S>
__global__ void __launch_bounds__(kThreads, kMinBlocks<N>)
conv_step_kernel(S* __restrict__ state, const float* __restrict__ Av, const float* __restrict__ Dv,
                 const T* __restrict__ x, const T* __restrict__ B, const T* __restrict__ C,
                 const T* __restrict__ dt, float* __restrict__ y, int H, int G) {
  using TL = Tile<P, N>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slab = blockIdx.x;
  const int b = slab / H, h = slab - b * H, g = h / (H / G);
  float hv[TL::RPW][TL::E];
  load_state<P, N, S>(state, slab, warp, lane, hv);
  const size_t xo = static_cast<size_t>(slab) * P, bo = (static_cast<size_t>(b) * G + g) * N;
  const float sum = update_and_read<P, N, T>(hv, x + xo, B + bo, C + bo, to_f(dt[slab]), Av[h], warp, lane);
  if (transpose_leader<TL::RPW>(lane)) {
    const int row = warp * TL::RPW + transpose_index<TL::RPW>(lane);
    y[xo + row] = fmaf(Dv[h], to_f(x[xo + row]), sum);
  }
  store_state<P, N, S>(state, slab, warp, lane, hv);
}

template <int P, int N, class T>
__global__ void __launch_bounds__(kThreads, kMinBlocks<N>)
conv_verify_kernel(float* __restrict__ snaps, const int* __restrict__ cur, const float* __restrict__ Av,
                   const float* __restrict__ Dv, const T* __restrict__ x, const T* __restrict__ B,
                   const T* __restrict__ C, const T* __restrict__ dt, float* __restrict__ y, int H,
                   int G, int TT) {
  using TL = Tile<P, N>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slab = blockIdx.x;
  const int b = slab / H, h = slab - b * H, g = h / (H / G);
  const int c0 = cur[b];
  auto snap = [&](int slot) { return (static_cast<size_t>(b) * (TT + 1) + slot) * H + h; };
  auto xoff = [&](int j) { return ((static_cast<size_t>(b) * TT + j) * H + h) * P; };
  auto boff = [&](int j) { return ((static_cast<size_t>(b) * TT + j) * G + g) * N; };
  if (c0 < 0 || c0 > TT) {
    for (int j = 0; j < TT; ++j)
      if (tid < P) y[xoff(j) + tid] = __int_as_float(0x7fc00000);
    return;
  }
  float hv[TL::RPW][TL::E];
  load_tile_f32<P, N>(snaps + snap(c0) * P * N, warp, lane, hv);
  const float A = Av[h], Dh = Dv[h];
  for (int j = 0; j < TT; ++j) {
    const float dtv = to_f(dt[(static_cast<size_t>(b) * TT + j) * H + h]);
    const float sum = update_and_read<P, N, T>(hv, x + xoff(j), B + boff(j), C + boff(j), dtv, A, warp, lane);
    if (transpose_leader<TL::RPW>(lane)) {
      const int row = warp * TL::RPW + transpose_index<TL::RPW>(lane);
      y[xoff(j) + row] = fmaf(Dh, to_f(x[xoff(j) + row]), sum);
    }
    int slot = c0 + 1 + j;
    if (slot > TT) slot -= TT + 1;
    store_tile_f32<P, N>(snaps + snap(slot) * P * N, warp, lane, hv);
  }
}

__global__ void conv_commit_kernel(int batch, int TT, int* __restrict__ cur, const int* __restrict__ accept,
                                   int* __restrict__ status) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int a = accept[b];
  if (a < 0 || a > TT) {
    if (status != nullptr) atomicOr(status, REPLAY_DEV_BAD_ACCEPT);
    return;
  }
  int c = cur[b] + a;
  if (c > TT) c -= TT + 1;
  cur[b] = c;
}

int launch_conv_step(const Shape& sh, int batch, int H, int G, void* state, int state_dtype,
                     const float* A, const float* D, const void* x, const void* B, const void* C,
                     const void* dt, float* y, cudaStream_t stream) {
#define RSSM_CONV(NN, TT, SS)                                                                    \
  if (sh.N == NN && sh.in_dtype == RSSM_DTYPE_OF(TT) && state_dtype == RSSM_DTYPE_OF(SS)) {     \
    conv_step_kernel<64, NN, TT, SS><<<batch * H, kThreads, 0, stream>>>(                       \
        static_cast<SS*>(state), A, D, static_cast<const TT*>(x), static_cast<const TT*>(B),      \
        static_cast<const TT*>(C), static_cast<const TT*>(dt), y, H, G);                         \
    return cudaGetLastError() == cudaSuccess ? REPLAY_OK : REPLAY_ECUDA;                         \
  }
  RSSM_CONV(64, float, float) RSSM_CONV(64, float, bf16) RSSM_CONV(64, bf16, float) RSSM_CONV(64, bf16, bf16)
  RSSM_CONV(128, float, float) RSSM_CONV(128, float, bf16) RSSM_CONV(128, bf16, float) RSSM_CONV(128, bf16, bf16)
  RSSM_CONV(256, float, float) RSSM_CONV(256, float, bf16) RSSM_CONV(256, bf16, float) RSSM_CONV(256, bf16, bf16)
#undef RSSM_CONV
  return REPLAY_EUNSUPPORTED;
}

int launch_conv_verify(const Shape& sh, int batch, int H, int G, int T, float* snaps,
                       const int* cur, const float* A, const float* D, const void* x,
                       const void* B, const void* C, const void* dt, float* y,
                       cudaStream_t stream) {
#define RSSM_CONVV(NN, TT)                                                                  \
  if (sh.N == NN && sh.in_dtype == RSSM_DTYPE_OF(TT)) {                                     \
    conv_verify_kernel<64, NN, TT><<<batch * H, kThreads, 0, stream>>>(                     \
        snaps, cur, A, D, static_cast<const TT*>(x), static_cast<const TT*>(B),             \
        static_cast<const TT*>(C), static_cast<const TT*>(dt), y, H, G, T);                 \
    return cudaGetLastError() == cudaSuccess ? REPLAY_OK : REPLAY_ECUDA;                    \
  }
  RSSM_CONVV(64, float) RSSM_CONVV(64, bf16) RSSM_CONVV(128, float) RSSM_CONVV(128, bf16)
  RSSM_CONVV(256, float) RSSM_CONVV(256, bf16)
#undef RSSM_CONVV
  return REPLAY_EUNSUPPORTED;
}

int launch_conv_commit(int batch, int T, int* cur, const int* accept, int* status, cudaStream_t stream) {
  const int threads = 256;
  conv_commit_kernel<<<(batch + threads - 1) / threads, threads, 0, stream>>>(batch, T, cur, accept, status);
  return cudaGetLastError() == cudaSuccess ? REPLAY_OK : REPLAY_ECUDA;
}

}  // namespace rssm
