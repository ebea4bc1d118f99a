// replay_step: one decode token for every sequence -- non-flush or flush per sequence.
//
// Source: "ReplaySSM: Rethinking State Storage for Faster Hybrid-Model Decoding" (NVIDIA
// Developer blog), sections "How ReplaySSM represents the state" (non-flush and flush
// steps) and "Benefit 1: Reduce state memory traffic" (a non-flush step reads the
// checkpoint and writes only the new record; the checkpoint is written once per window).
//
// One CTA per (sequence, head) slab. The checkpoint tile (P x N FP32, or its read copy)
// is loaded into registers with coalesced 16-byte streaming loads issued before anything
// else, so they are in flight while the CTA reads its metadata and records. A non-flush
// step then needs one CTA barrier: warps compute the B_s . C dot products of the records
// (warp-strided) while lane s of every warp holds record s's x values for the warp's rows,
// so the record term sum_s w_s x_s[p] joins the h0 . C partial sums of the same warp
// reduction.
#include "launch.h"
#include "replay_core.cuh"

namespace rssm {

template <int P, int N, class T, int RC>
__global__ void __launch_bounds__(kThreads, kMinBlocks<N>)
replay_step_kernel(StoreView sv, const T* __restrict__ x, const T* __restrict__ B,
                   const T* __restrict__ C, const T* __restrict__ dt, float* __restrict__ y) {
  using TL = Tile<P, N>;
  constexpr int RPW = TL::RPW, E = TL::E;
  extern __shared__ float4 smem4[];
  float* smem = reinterpret_cast<float*>(smem4);
  __shared__ int4 s_meta;
  __shared__ float s_dt[kMaxCap];
  __shared__ float s_bc[kMaxCap];
  __shared__ float s_red[kWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slab = blockIdx.x;
  const int b = slab / sv.H, h = slab - b * sv.H, g = h / sv.hpg;
  const int cap = sv.cap;
  const size_t xo = static_cast<size_t>(slab) * P;  // x[b][h][:] and y[b][h][:]
  const size_t bo = (static_cast<size_t>(b) * sv.G + g) * N;

  if (tid == 0) s_meta = sv.meta[b];
  float hv[RPW][E];
  if constexpr (RC == REPLAY_RC_NONE)
    load_tile_f32<P, N>(sv.h0 + static_cast<size_t>(slab) * P * N, warp, lane, hv);
  float cv[E];
  load_cols<P, N>(C + bo, lane, cv);
  __syncthreads();

  const int start = s_meta.x, n = s_meta.y;
  const int k = n + 1;  // records including this token
  if (n < 0 || k > cap || start < 0 || start >= cap) {
    if (tid < P) y[xo + tid] = __int_as_float(0x7fc00000);
    if (tid == 0) set_status(sv.status, REPLAY_DEV_BAD_META);
    return;
  }
  const float A = sv.A[h], Dh = sv.D[h];
  const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
  const T* xcur = x + xo;
  const T* bcur = B + bo;
  const T dtcur = dt[slab];
  int4 next;

  if (k >= sv.L) {
    // ---------------- flush: fold the k records into h0, write it once, read y from it
    if constexpr (RC != REPLAY_RC_NONE)
      load_tile_f32<P, N>(sv.h0 + static_cast<size_t>(slab) * P * N, warp, lane, hv);
    float* sm_x = smem;
    float* sm_b = smem + cap * P;
    fold_records<P, N, T>(ring, start, cap, k, n, xcur, bcur, dtcur, A, sm_x, sm_b, s_dt, hv);
    float dx[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) dx[i] = 0.f;
    const float sum = tile_rows_dot<P, N>(hv, cv, 1.f, dx, lane);
    if (transpose_leader<RPW>(lane)) {
      const int row = warp * RPW + transpose_index<RPW>(lane);
      y[xo + row] = fmaf(Dh, to_f(xcur[row]), sum);
    }
    write_checkpoint<P, N, RC>(sv, slab, s_red, hv);
    next = make_int4(ring_slot(start, k, cap), 0, 0, 0);
  } else {
    // ---------------- non-flush: y from checkpoint + records; append; no state write
    if constexpr (RC != REPLAY_RC_NONE) {
      const float scale = RC == REPLAY_RC_FP8E4M3 ? sv.scale[slab] : 1.f;
      load_tile_rc<P, N, RC>(sv.rc, slab, scale, warp, lane, hv);
    }
    if (warp == kWarps - 1)
      for (int s = lane; s < k; s += 32)
        s_dt[s] = s < n ? to_f(ring.dt[ring_slot(start, s, cap)]) : to_f(dtcur);
    for (int s = warp; s < k; s += kWarps) {
      const T* bs = s < n ? ring.b + static_cast<size_t>(ring_slot(start, s, cap)) * N : bcur;
      float bv[E];
      load_cols<P, N>(bs, lane, bv);
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) d = fmaf(bv[e], cv[e], d);
      d = warp_sum(d);
      if (lane == 0) s_bc[s] = d;
    }
    float xr[RPW];  // record `lane`: x values of this warp's rows
    const int s0 = lane;
    if (s0 < k) {
      const T* xs = s0 < n ? ring.x + static_cast<size_t>(ring_slot(start, s0, cap)) * P : xcur;
      load_rows<RPW>(xs + warp * RPW, xr);
    } else {
#pragma unroll
      for (int i = 0; i < RPW; ++i) xr[i] = 0.f;
    }
    __syncthreads();

    float tot = 0.f;
    for (int r = 0; r < k; ++r) tot += s_dt[r];
    const float Gam = expf(A * tot);
    float c0 = 0.f;
    if (s0 < k) {
      float suf = 0.f;
      for (int r = s0 + 1; r < k; ++r) suf += s_dt[r];
      c0 = expf(A * suf) * s_dt[s0] * s_bc[s0];
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) xr[i] *= c0;
    if (k > 32) {  // records 32..63 (rings longer than 32 records)
      const int s1 = lane + 32;
      if (s1 < k) {
        const T* xs = s1 < n ? ring.x + static_cast<size_t>(ring_slot(start, s1, cap)) * P : xcur;
        float x1[RPW];
        load_rows<RPW>(xs + warp * RPW, x1);
        float suf = 0.f;
        for (int r = s1 + 1; r < k; ++r) suf += s_dt[r];
        const float c1 = expf(A * suf) * s_dt[s1] * s_bc[s1];
#pragma unroll
        for (int i = 0; i < RPW; ++i) xr[i] = fmaf(c1, x1[i], xr[i]);
      }
    }
    const float sum = tile_rows_dot<P, N>(hv, cv, Gam, xr, lane);
    if (transpose_leader<RPW>(lane)) {
      const int row = warp * RPW + transpose_index<RPW>(lane);
      y[xo + row] = fmaf(Dh, to_f(xcur[row]), sum);
    }
    // append this token's record at ring slot start + n
    const int slot = ring_slot(start, n, cap);
    T* xw = ring.x + static_cast<size_t>(slot) * P;
    for (int p = tid; p < P; p += kThreads) xw[p] = xcur[p];
    if (h % sv.hpg == 0) {
      T* bw = ring.b + static_cast<size_t>(slot) * N;
      for (int c = tid; c < N; c += kThreads) bw[c] = bcur[c];
    }
    if (tid == 0) ring.dt[slot] = dtcur;
    next = make_int4(start, k, 0, 0);
  }
  if (tid == 0) arrive_and_publish(sv, b, next);
}

template <int P, int N, class T, int RC>
static int launch(const StoreView& sv, const void* x, const void* B, const void* C, const void* dt,
                  float* y, cudaStream_t stream) {
  auto kern = replay_step_kernel<P, N, T, RC>;
  const size_t smem = static_cast<size_t>(sv.cap) * (P + N) * sizeof(float);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess)
    return REPLAY_ECUDA;
  kern<<<sv.batch * sv.H, kThreads, smem, stream>>>(sv, static_cast<const T*>(x),
                                                   static_cast<const T*>(B), static_cast<const T*>(C),
                                                   static_cast<const T*>(dt), y);
  return cudaGetLastError() == cudaSuccess ? REPLAY_OK : REPLAY_ECUDA;
}

int launch_step(const StoreView& sv, const Shape& sh, const void* x, const void* B, const void* C,
                const void* dt, float* y, cudaStream_t stream) {
#define RSSM_STEP(NN, TT, RCC)                                                              \
  if (sh.N == NN && sh.in_dtype == RSSM_DTYPE_OF(TT) && sh.read_copy == RCC)                 \
    return launch<64, NN, TT, RCC>(sv, x, B, C, dt, y, stream);
  RSSM_FOR_EACH_CONFIG(RSSM_STEP)
#undef RSSM_STEP
  return REPLAY_EUNSUPPORTED;
}

}  // namespace rssm
