// replay_verify and replay_commit: speculative verify of T drafts with buffer-truncate
// rollback.
//
// Source: "ReplaySSM: Rethinking State Storage for Faster Hybrid-Model Decoding" (NVIDIA
// Developer blog), section "Benefit 2: Simplify rollback and speed up verification": the
// drafts' inputs are appended beyond the commit pointer before verification, the accepted
// prefix is committed by advancing the pointer, records beyond it are ignored and later
// overwritten, and a flush folds only committed records. The T outputs are computed by
// output-only evaluation: the checkpoint is read once for all T queries and every other
// term is a scalar (B_s . C_j, times a decay) scaling a cached x_s -- no state is formed.
//
// One CTA per (sequence, head) slab, as in the step kernel: the checkpoint tile is loaded
// into registers first; the committed records and the drafts are staged in a shared-memory
// image of the ring (the drafts at the slots they are appended to); when n >= L committed
// records are waiting they are folded into the tile and written as the new checkpoint
// before the drafts are evaluated.
#include "launch.h"
#include "replay_core.cuh"

namespace rssm {

constexpr int kMaxDrafts = 8;

template <int P, int N, class T, int RC>
__global__ void __launch_bounds__(kThreads, kMinBlocks<N> == 4 ? 3 : 2)
replay_verify_kernel(StoreView sv, int TT, const T* __restrict__ x, const T* __restrict__ B,
                     const T* __restrict__ C, const T* __restrict__ dt, float* __restrict__ y) {
  using TL = Tile<P, N>;
  constexpr int RPW = TL::RPW, E = TL::E;
  extern __shared__ float4 smem4[];
  __shared__ int4 s_meta;
  __shared__ float s_bc[kMaxDrafts][kMaxCap];
  __shared__ float s_w[kMaxCap + 1];
  __shared__ float s_red[kWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = sv.H, G = sv.G;
  const int g = blockIdx.y, b = blockIdx.z;
  const int h = g * sv.hpg + blockIdx.x;
  const int slab = b * H + h;
  const int cap = sv.cap;
  // draft j of sequence b: x/y at ((b*TT + j)*H + h)*P, B/C at ((b*TT + j)*G + g)*N
  auto xoff = [&](int j) { return (static_cast<size_t>(b) * TT + j) * H * P + static_cast<size_t>(h) * P; };
  auto boff = [&](int j) { return (static_cast<size_t>(b) * TT + j) * G * N + static_cast<size_t>(g) * N; };
  auto doff = [&](int j) { return (static_cast<size_t>(b) * TT + j) * H + h; };

  if (tid == 0) s_meta = sv.meta[b];
  float hv[RPW][E];
  if constexpr (RC == REPLAY_RC_NONE) {
    load_tile_f32<P, N>(sv.h0 + static_cast<size_t>(slab) * P * N, warp, lane, hv);
  } else {
    const float scale = RC == REPLAY_RC_FP8E4M3 ? sv.scale[slab] : 1.f;
    load_tile_rc<P, N, RC>(sv.rc, slab, scale, warp, lane, hv);
  }
  const int myrow = warp * RPW + transpose_index<RPW>(lane);
  const float A = sv.A[h], Dh = sv.D[h];
  __syncthreads();

  const int start = s_meta.x, n = s_meta.y;
  if (n < 0 || start < 0 || start >= cap || n + TT > cap) {
    for (int j = 0; j < TT; ++j)
      if (tid < P) y[xoff(j) + tid] = __int_as_float(0x7fc00000);
    if (tid == 0) set_status(sv.status, REPLAY_DEV_BAD_META);
    return;
  }
  const bool prefold = n >= sv.L;  // fold the committed records first (flush of committed only)
  const int start2 = prefold ? ring_slot(start, n, cap) : start;
  const int n2 = prefold ? 0 : n;
  const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
  const RingImage<T> im = ring_image<P, N, T>(smem4, cap);
  const ExtraRecords<T> drafts{x + xoff(0), B + boff(0), dt + doff(0), static_cast<size_t>(H) * P,
                               static_cast<size_t>(G) * N, static_cast<size_t>(H)};
  stage_records<P, N, T>(ring, im, start, cap, n + TT, n, drafts);
  if (tid == 0) arrive_and_publish(sv, b, make_int4(start2, n2, TT, 0), H);
  if constexpr (RC != REPLAY_RC_NONE) {
    if (prefold) load_tile_f32<P, N>(sv.h0 + static_cast<size_t>(slab) * P * N, warp, lane, hv);
  }
  cp_async_wait_all();
  __syncthreads();

  if (prefold) {
    auto slot_of = [&](int s) { return ring_slot(start, s, cap); };
    float* sm_u = fold_staging(smem4, ring_image_bytes<P, N, T>(cap));
    fold_tile<P, N, T>(im, slot_of, n, A, sm_u, sm_u + cap * P, s_w, hv);
    write_checkpoint<P, N, RC>(sv, slab, s_red, hv);
  }
  const int kk = n2 + TT;  // committed records, then the drafts, from slot start2
  // B_s . C_j for every record s a draft j sees (s <= n2 + j); the pair loop is warp-strided
  for (int pi = warp; pi < TT * kk; pi += kWarps) {
    const int j = pi / kk, s = pi - j * kk;
    if (s > n2 + j) continue;
    float bv[E], cj[E];
    load_cols<P, N>(im.b + ring_slot(start2, s, cap) * N, lane, bv);
    load_cols<P, N>(C + boff(j), lane, cj);
    float d = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) d = fmaf(bv[e], cj[e], d);
    d = warp_sum(d);
    if (lane == 0) s_bc[j][s] = d;
  }
  __syncthreads();

  float xr0[RPW], xr1[RPW];  // records lane and lane + 32: x values of this warp's rows
#pragma unroll
  for (int i = 0; i < RPW; ++i) xr0[i] = xr1[i] = 0.f;
  if (lane < kk) load_rows<RPW>(im.x + ring_slot(start2, lane, cap) * P + warp * RPW, xr0);
  if (lane + 32 < kk) load_rows<RPW>(im.x + ring_slot(start2, lane + 32, cap) * P + warp * RPW, xr1);
  const float dt0 = lane < kk ? im.dt[ring_slot(start2, lane, cap)] : 0.f;
  const float dt1 = lane + 32 < kk ? im.dt[ring_slot(start2, lane + 32, cap)] : 0.f;
  for (int j = 0; j < TT; ++j) {
    const int k = n2 + j + 1;  // records draft j sees, itself included
    const RecordWeights rw = record_weights(lane < k ? dt0 : 0.f, lane + 32 < k ? dt1 : 0.f, k, A, lane);
    const float c0 = lane < k ? rw.w0 * s_bc[j][lane] : 0.f;
    const float c1 = lane + 32 < k ? rw.w1 * s_bc[j][lane + 32] : 0.f;
    float ex[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) ex[i] = fmaf(c1, xr1[i], c0 * xr0[i]);
    float cq[E];
    load_cols<P, N>(C + boff(j), lane, cq);
    const float sum = tile_rows_dot<P, N>(hv, cq, rw.gam, ex, lane);
    if (transpose_leader<RPW>(lane)) {
      const float xj = to_f(im.x[ring_slot(start2, n2 + j, cap) * P + myrow]);
      y[xoff(j) + myrow] = fmaf(Dh, xj, sum);
    }
  }
  // the drafts' records go to the ring beyond the committed ones; the pointer stays
  for (int j = 0; j < TT; ++j) {
    const int slot = ring_slot(start2, n2 + j, cap);
    append_record<P, N, T>(ring, im, slot, slot, blockIdx.x == 0, dt[doff(j)]);
  }
}

template <int P, int N, class T, int RC>
static int launch(const StoreView& sv, int TT, const void* x, const void* B, const void* C,
                  const void* dt, float* y, cudaStream_t stream) {
  auto kern = replay_verify_kernel<P, N, T, RC>;
  const size_t smem = smem_plan_bytes<P, N>(ring_image_bytes<P, N, T>(sv.cap), sv.cap);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess)
    return REPLAY_ECUDA;
  const dim3 grid(sv.hpg, sv.G, sv.batch);
  kern<<<grid, kThreads, smem, stream>>>(sv, TT, static_cast<const T*>(x), static_cast<const T*>(B),
                                         static_cast<const T*>(C), static_cast<const T*>(dt), y);
  return cudaGetLastError() == cudaSuccess ? REPLAY_OK : REPLAY_ECUDA;
}

int launch_verify(const StoreView& sv, const Shape& sh, int T, const void* x, const void* B,
                  const void* C, const void* dt, float* y, cudaStream_t stream) {
  if (T < 1 || T > kMaxDrafts) return REPLAY_ECAPACITY;
#define RSSM_VERIFY(NN, TT, RCC)                                                  \
  if (sh.N == NN && sh.in_dtype == RSSM_DTYPE_OF(TT) && sh.read_copy == RCC)      \
    return launch<64, NN, TT, RCC>(sv, T, x, B, C, dt, y, stream);
  RSSM_FOR_EACH_CONFIG(RSSM_VERIFY)
#undef RSSM_VERIFY
  return REPLAY_EUNSUPPORTED;
}

// Commit: one thread per sequence advances the pointer over the accepted drafts.
__global__ void replay_commit_kernel(StoreView sv, const int* __restrict__ accept) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= sv.batch) return;
  int4 m = sv.meta[b];
  const int a = accept[b];
  if (a < 0 || a > m.z) {
    set_status(sv.status, REPLAY_DEV_BAD_ACCEPT);
  } else {
    m.y += a;
  }
  m.z = 0;
  sv.meta[b] = m;
}

int launch_commit(const StoreView& sv, const int* accept, cudaStream_t stream) {
  const int threads = 256;
  replay_commit_kernel<<<(sv.batch + threads - 1) / threads, threads, 0, stream>>>(sv, accept);
  return cudaGetLastError() == cudaSuccess ? REPLAY_OK : REPLAY_ECUDA;
}

}  // namespace rssm
