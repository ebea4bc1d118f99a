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
  float* smem = reinterpret_cast<float*>(smem4);
  __shared__ int4 s_meta;
  __shared__ float s_dt[kMaxCap];
  __shared__ float s_bc[kMaxDrafts][kMaxCap];
  __shared__ float s_red[kWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slab = blockIdx.x;
  const int H = sv.H, G = sv.G;
  const int b = slab / H, h = slab - b * H, g = h / sv.hpg;
  const int cap = sv.cap;
  // draft j of sequence b: x/y at ((b*TT + j)*H + h)*P, B/C at ((b*TT + j)*G + g)*N
  auto xoff = [&](int j) { return (static_cast<size_t>(b) * TT + j) * H * P + static_cast<size_t>(h) * P; };
  auto boff = [&](int j) { return (static_cast<size_t>(b) * TT + j) * G * N + static_cast<size_t>(g) * N; };
  auto doff = [&](int j) { return (static_cast<size_t>(b) * TT + j) * H + h; };

  if (tid == 0) s_meta = sv.meta[b];
  float hv[RPW][E];
  if constexpr (RC == REPLAY_RC_NONE)
    load_tile_f32<P, N>(sv.h0 + static_cast<size_t>(slab) * P * N, warp, lane, hv);
  __syncthreads();

  const int start = s_meta.x, n = s_meta.y;
  if (n < 0 || start < 0 || start >= cap || n + TT > cap) {
    for (int j = 0; j < TT; ++j)
      if (tid < P) y[xoff(j) + tid] = __int_as_float(0x7fc00000);
    if (tid == 0) set_status(sv.status, REPLAY_DEV_BAD_META);
    return;
  }
  const float A = sv.A[h], Dh = sv.D[h];
  const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
  int start2 = start, n2 = n;
  if (n >= sv.L) {
    // fold the committed records first (a flush of committed records only)
    if constexpr (RC != REPLAY_RC_NONE)
      load_tile_f32<P, N>(sv.h0 + static_cast<size_t>(slab) * P * N, warp, lane, hv);
    fold_records<P, N, T>(ring, start, cap, n, n, nullptr, nullptr, T(0.f), A, smem, smem + cap * P,
                          s_dt, hv);
    write_checkpoint<P, N, RC>(sv, slab, s_red, hv);
    start2 = ring_slot(start, n, cap);
    n2 = 0;
    __syncthreads();  // s_dt is reused below
  } else {
    if constexpr (RC != REPLAY_RC_NONE) {
      const float scale = RC == REPLAY_RC_FP8E4M3 ? sv.scale[slab] : 1.f;
      load_tile_rc<P, N, RC>(sv.rc, slab, scale, warp, lane, hv);
    }
  }

  const int kk = n2 + TT;  // committed records, then the drafts
  if (warp == kWarps - 1)
    for (int s = lane; s < kk; s += 32)
      s_dt[s] = s < n2 ? to_f(ring.dt[ring_slot(start2, s, cap)]) : to_f(dt[doff(s - n2)]);
  // B_s . C_j for every record s a draft j sees (s <= n2 + j); the pair loop is warp-strided
  for (int pi = warp; pi < TT * kk; pi += kWarps) {
    const int j = pi / kk, s = pi - j * kk;
    if (s > n2 + j) continue;
    const T* bs = s < n2 ? ring.b + static_cast<size_t>(ring_slot(start2, s, cap)) * N : B + boff(s - n2);
    float bv[E], cj[E];
    load_cols<P, N>(bs, lane, bv);
    load_cols<P, N>(C + boff(j), lane, cj);
    float d = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) d = fmaf(bv[e], cj[e], d);
    d = warp_sum(d);
    if (lane == 0) s_bc[j][s] = d;
  }
  float xr[RPW];  // record `lane`: x values of this warp's rows
  const int s0 = lane;
  if (s0 < kk) {
    const T* xs = s0 < n2 ? ring.x + static_cast<size_t>(ring_slot(start2, s0, cap)) * P : x + xoff(s0 - n2);
    load_rows<RPW>(xs + warp * RPW, xr);
  } else {
#pragma unroll
    for (int i = 0; i < RPW; ++i) xr[i] = 0.f;
  }
  __syncthreads();

  for (int j = 0; j < TT; ++j) {
    const int k = n2 + j + 1;  // records draft j sees, itself included
    float tot = 0.f;
    for (int r = 0; r < k; ++r) tot += s_dt[r];
    const float Gam = expf(A * tot);
    float c0 = 0.f;
    if (s0 < k) {
      float suf = 0.f;
      for (int r = s0 + 1; r < k; ++r) suf += s_dt[r];
      c0 = expf(A * suf) * s_dt[s0] * s_bc[j][s0];
    }
    float ex[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) ex[i] = c0 * xr[i];
    if (k > 32) {
      const int s1 = lane + 32;
      if (s1 < k) {
        const T* xs = s1 < n2 ? ring.x + static_cast<size_t>(ring_slot(start2, s1, cap)) * P : x + xoff(s1 - n2);
        float x1[RPW];
        load_rows<RPW>(xs + warp * RPW, x1);
        float suf = 0.f;
        for (int r = s1 + 1; r < k; ++r) suf += s_dt[r];
        const float c1 = expf(A * suf) * s_dt[s1] * s_bc[j][s1];
#pragma unroll
        for (int i = 0; i < RPW; ++i) ex[i] = fmaf(c1, x1[i], ex[i]);
      }
    }
    float cq[E];
    load_cols<P, N>(C + boff(j), lane, cq);
    const float sum = tile_rows_dot<P, N>(hv, cq, Gam, ex, lane);
    if (transpose_leader<RPW>(lane)) {
      const int row = warp * RPW + transpose_index<RPW>(lane);
      y[xoff(j) + row] = fmaf(Dh, to_f(x[xoff(j) + row]), sum);
    }
  }
  // the drafts' records go beyond the committed ones; the pointer stays
  for (int j = 0; j < TT; ++j) {
    const int slot = ring_slot(start2, n2 + j, cap);
    for (int p = tid; p < P; p += kThreads) ring.x[static_cast<size_t>(slot) * P + p] = x[xoff(j) + p];
    if (h % sv.hpg == 0)
      for (int c = tid; c < N; c += kThreads) ring.b[static_cast<size_t>(slot) * N + c] = B[boff(j) + c];
    if (tid == 0) ring.dt[slot] = dt[doff(j)];
  }
  if (tid == 0) arrive_and_publish(sv, b, make_int4(start2, n2, TT, 0));
}

template <int P, int N, class T, int RC>
static int launch(const StoreView& sv, int TT, const void* x, const void* B, const void* C,
                  const void* dt, float* y, cudaStream_t stream) {
  auto kern = replay_verify_kernel<P, N, T, RC>;
  const size_t smem = static_cast<size_t>(sv.cap) * (P + N) * sizeof(float);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess)
    return REPLAY_ECUDA;
  kern<<<sv.batch * sv.H, kThreads, smem, stream>>>(sv, TT, static_cast<const T*>(x),
                                                   static_cast<const T*>(B), static_cast<const T*>(C),
                                                   static_cast<const T*>(dt), y);
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
