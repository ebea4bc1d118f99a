// replay_step: one decode token for every sequence -- non-flush or flush per sequence.
//
// Source: "ReplaySSM: Rethinking State Storage for Faster Hybrid-Model Decoding" (NVIDIA
// Developer blog), sections "How ReplaySSM represents the state" (non-flush and flush
// steps) and "Benefit 1: Reduce state memory traffic" (a non-flush step reads the
// checkpoint and writes only the new record; the checkpoint is written once per window).
//
// One CTA per (sequence, head) slab; the grid is (heads per group, groups, batch), so a
// CTA's indices need no division and consecutive CTAs are the heads of one group (their
// shared B records stay in L2). At entry every thread issues, before anything else, its
// coalesced 16-byte streaming loads of the checkpoint tile (FP32, or the read copy) and its
// share of cp.async copies of the slab's whole ring (x of the head, B of the group, dt)
// plus the current token's record into a shared-memory image; nothing waits on the ring
// pointer, which one thread reads meanwhile. After one barrier the CTA publishes the
// sequence's next pointer (last-CTA-done counter) and branches:
//  - non-flush: the B_s . C dots (warp-strided), the decay weights (warp scans), and then
//    one warp reduction per warp that sums h0 . C and the record term: lane s of every warp
//    carries w_s (B_s . C) x_s for the warp's rows;
//  - flush: the records are folded into the tile (rank-k FFMA update from FP32 staging),
//    y is read from the new state, and the checkpoint (and read copy) is written once.
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
  __shared__ int4 s_meta;
  __shared__ float s_bc[kMaxCap];
  __shared__ float s_w[kMaxCap + 1];
  __shared__ float s_red[kWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y, b = blockIdx.z;
  const int h = g * sv.hpg + blockIdx.x;
  const int slab = b * sv.H + h;
  const int cap = sv.cap;
  const size_t xo = static_cast<size_t>(slab) * P;  // x[b][h][:] and y[b][h][:]
  const size_t bo = (static_cast<size_t>(b) * sv.G + g) * N;

  if (tid == 0) s_meta = sv.meta[b];
  float hv[RPW][E];
  if constexpr (RC == REPLAY_RC_NONE) {
    load_tile_f32<P, N>(sv.h0 + static_cast<size_t>(slab) * P * N, warp, lane, hv);
  } else {
    const float scale = RC == REPLAY_RC_FP8E4M3 ? sv.scale[slab] : 1.f;
    load_tile_rc<P, N, RC>(sv.rc, slab, scale, warp, lane, hv);
  }
  const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
  const RingImage<T> im = whole_image<P, N, T>(smem4, cap);
  const T dtcur = dt[slab];
  stage_whole_ring<P, N, T>(ring, im, cap, x + xo, B + bo, dtcur);
  float cv[E];
  load_cols<P, N>(C + bo, lane, cv);
  const int myrow = warp * RPW + transpose_index<RPW>(lane);
  const float xk_row = to_f(x[xo + myrow]);
  const float A = sv.A[h], Dh = sv.D[h];
  cp_async_wait_all();
  __syncthreads();

  const int start = s_meta.x, n = s_meta.y;
  const int k = n + 1;  // records including this token
  if (n < 0 || k > cap || start < 0 || start >= cap) {
    if (tid < P) y[xo + tid] = __int_as_float(0x7fc00000);
    if (tid == 0) set_status(sv.status, REPLAY_DEV_BAD_META);
    return;
  }
  const bool flush = k >= sv.L;
  if (tid == 0)
    arrive_and_publish(sv, b, flush ? make_int4(ring_slot(start, k, cap), 0, 0, 0) : make_int4(start, k, 0, 0));
  // record s of the window: ring slot start + s, or the current token (image slot cap)
  auto slot_of = [&](int s) { return s < n ? ring_slot(start, s, cap) : cap; };

  if (flush) {
    // ---------------- flush: fold the k records into h0, write it once, read y from it
    if constexpr (RC != REPLAY_RC_NONE)  // a flush starts from the FP32 checkpoint
      load_tile_f32<P, N>(sv.h0 + static_cast<size_t>(slab) * P * N, warp, lane, hv);
    float* sm_u = fold_staging(smem4, whole_image_bytes<P, N, T>(cap));
    fold_tile<P, N, T>(im, slot_of, k, A, sm_u, sm_u + cap * P, s_w, hv);
    float zero[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) zero[i] = 0.f;
    const float sum = tile_rows_dot<P, N>(hv, cv, 1.f, zero, lane);
    if (transpose_leader<RPW>(lane)) y[xo + myrow] = fmaf(Dh, xk_row, sum);
    write_checkpoint<P, N, RC>(sv, slab, s_red, hv);
    return;
  }

  // ---------------- non-flush: y from checkpoint + records; no state write
  for (int s = warp; s < k; s += kWarps) {
    float bv[E];
    load_cols<P, N>(im.b + slot_of(s) * N, lane, bv);
    float d = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) d = fmaf(bv[e], cv[e], d);
    d = warp_sum(d);
    if (lane == 0) s_bc[s] = d;
  }
  __syncthreads();
  const float dt0 = lane < k ? im.dt[slot_of(lane)] : 0.f;
  const float dt1 = lane + 32 < k ? im.dt[slot_of(lane + 32)] : 0.f;
  const RecordWeights rw = record_weights(dt0, dt1, k, A, lane);
  float xr[RPW];
  if (lane < k) {
    load_rows<RPW>(im.x + slot_of(lane) * P + warp * RPW, xr);
    const float c0 = rw.w0 * s_bc[lane];
#pragma unroll
    for (int i = 0; i < RPW; ++i) xr[i] *= c0;
  } else {
#pragma unroll
    for (int i = 0; i < RPW; ++i) xr[i] = 0.f;
  }
  if (lane + 32 < k) {
    float x1[RPW];
    load_rows<RPW>(im.x + slot_of(lane + 32) * P + warp * RPW, x1);
    const float c1 = rw.w1 * s_bc[lane + 32];
#pragma unroll
    for (int i = 0; i < RPW; ++i) xr[i] = fmaf(c1, x1[i], xr[i]);
  }
  const float sum = tile_rows_dot<P, N>(hv, cv, rw.gam, xr, lane);
  if (transpose_leader<RPW>(lane)) y[xo + myrow] = fmaf(Dh, xk_row, sum);
  // append this token's record (image slot cap) at ring slot start + n
  append_record<P, N, T>(ring, im, cap, ring_slot(start, n, cap), blockIdx.x == 0, dtcur);
}

template <int P, int N, class T, int RC>
static int launch(const StoreView& sv, const void* x, const void* B, const void* C, const void* dt,
                  float* y, cudaStream_t stream) {
  auto kern = replay_step_kernel<P, N, T, RC>;
  const size_t smem = smem_plan_bytes<P, N>(whole_image_bytes<P, N, T>(sv.cap), sv.cap);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess)
    return REPLAY_ECUDA;
  const dim3 grid(sv.hpg, sv.G, sv.batch);
  kern<<<grid, kThreads, smem, stream>>>(sv, static_cast<const T*>(x), static_cast<const T*>(B),
                                         static_cast<const T*>(C), static_cast<const T*>(dt), y);
  return cudaGetLastError() == cudaSuccess ? REPLAY_OK : REPLAY_ECUDA;
}

int launch_step(const StoreView& sv, const Shape& sh, const void* x, const void* B, const void* C,
                const void* dt, float* y, cudaStream_t stream) {
#define RSSM_STEP(NN, TT, RCC)                                                  \
  if (sh.N == NN && sh.in_dtype == RSSM_DTYPE_OF(TT) && sh.read_copy == RCC)    \
    return launch<64, NN, TT, RCC>(sv, x, B, C, dt, y, stream);
  RSSM_FOR_EACH_CONFIG(RSSM_STEP)
#undef RSSM_STEP
  return REPLAY_EUNSUPPORTED;
}

}  // namespace rssm
