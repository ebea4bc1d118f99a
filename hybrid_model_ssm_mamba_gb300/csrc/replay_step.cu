// replay_step: one decode token for every sequence -- non-flush or flush per sequence.
//
// Source: "ReplaySSM: Rethinking State Storage for Faster Hybrid-Model Decoding" (NVIDIA
// Developer blog), sections "How ReplaySSM represents the state" (non-flush and flush
// steps) and "Benefit 1: Reduce state memory traffic" (a non-flush step reads the
// checkpoint and writes only the new record; the checkpoint is written once per window).
//
// Two kernels per step.
//  1. replay_step_prep_kernel, one CTA per (sequence, group): reads the ring pointer,
//     records it as the step's plan, publishes the next pointer (last-CTA-done counter over
//     the G groups), computes the B_s . C dots of the group's k records once, and for each
//     head of the group the record coefficients by warp scans over dt:
//        non-flush: c_s = exp(A sum_{r=s+1..k-1} dt_r) dt_s (B_s . C),   flush: w_s (no dot)
//     plus Gamma_k = exp(A sum_{r<k} dt_r). This work is shared by the H/G heads of a group
//     (B and C are per group), so doing it here removes it from every head's CTA.
//  2. replay_step_kernel, one CTA per (sequence, head) slab, grid (heads per group, groups,
//     batch), launched as a programmatic dependent of the prep kernel: its checkpoint tile
//     loads (coalesced 16-byte streaming loads into registers) are issued before it waits
//     for the prep results. A non-flush step is then barrier-free: lane s of every warp loads
//     c_s and record s's x values for the warp's rows, and one warp reduction per warp sums
//     Gamma_k h0 . C and sum_s c_s x_s. A flush stages u_s = w_s x_s and B_s in FP32 shared
//     memory, applies the rank-k update, reads y from the new state and writes the
//     checkpoint (and read copy) once.
#include "launch.h"
#include "replay_core.cuh"

namespace rssm {

constexpr int kPlanNonFlush = 0, kPlanFlush = 1, kPlanBad = -1;

template <int P, int N, class T>
__global__ void __launch_bounds__(kThreads)
replay_step_prep_kernel(StoreView sv, const T* __restrict__ B, const T* __restrict__ C,
                        const T* __restrict__ dt) {
  using TL = Tile<P, N>;
  __shared__ int4 s_meta;
  __shared__ float s_bc[kMaxCap];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x, b = blockIdx.y;
  const int cap = sv.cap;
  griddep_launch_dependents();  // the head CTAs may start their checkpoint loads now
  if (tid == 0) s_meta = sv.meta[b];
  __syncthreads();
  const int start = s_meta.x, n = s_meta.y;
  const int k = n + 1;
  if (n < 0 || k > cap || start < 0 || start >= cap) {
    if (tid == 0) {
      if (g == 0) sv.plan[b] = make_int4(start, n, kPlanBad, 0);
      set_status(sv.status, REPLAY_DEV_BAD_META);
    }
    return;
  }
  const bool flush = k >= sv.L;
  if (tid == 0) {
    if (g == 0) sv.plan[b] = make_int4(start, n, flush ? kPlanFlush : kPlanNonFlush, 0);
    arrive_and_publish(sv, b, flush ? make_int4(ring_slot(start, k, cap), 0, 0, 0) : make_int4(start, k, 0, 0),
                       sv.G);
  }
  const size_t bo = (static_cast<size_t>(b) * sv.G + g) * N;
  if (!flush) {
    // stage the k records' B and this token's C in shared memory (one round trip)
    extern __shared__ float4 smem4[];
    T* sb = reinterpret_cast<T*>(smem4);  // [k][N] B, then [N] C
    const T* bring = static_cast<const T*>(sv.bbuf) + (static_cast<size_t>(b) * sv.G + g) * cap * N;
    constexpr int EPC = 16 / sizeof(T), BC = N / EPC;
    for (int c = tid; c < (k + 1) * BC; c += kThreads) {
      const int r = c / BC, off = (c - r * BC) * EPC;
      const T* src = r == k ? C + bo : (r < n ? bring + static_cast<size_t>(ring_slot(start, r, cap)) * N : B + bo);
      cp_async16(sb + static_cast<size_t>(r) * N + off, src + off);
    }
    cp_async_wait_all();
    __syncthreads();
    float cv[TL::E];
    load_cols<P, N>(sb + static_cast<size_t>(k) * N, lane, cv);
    for (int s = warp; s < k; s += kWarps) {
      float bv[TL::E];
      load_cols<P, N>(sb + static_cast<size_t>(s) * N, lane, bv);
      float d = 0.f;
#pragma unroll
      for (int e = 0; e < TL::E; ++e) d = fmaf(bv[e], cv[e], d);
      d = warp_sum(d);
      if (lane == 0) s_bc[s] = d;
    }
  }
  __syncthreads();
  for (int hh = warp; hh < sv.hpg; hh += kWarps) {
    const int h = g * sv.hpg + hh;
    const size_t slab = static_cast<size_t>(b) * sv.H + h;
    const T* dtr = static_cast<const T*>(sv.dtbuf) + slab * cap;
    auto dt_of = [&](int s) { return to_f(s < n ? dtr[ring_slot(start, s, cap)] : dt[slab]); };
    const float dt0 = lane < k ? dt_of(lane) : 0.f;
    const float dt1 = lane + 32 < k ? dt_of(lane + 32) : 0.f;
    const RecordWeights rw = record_weights(dt0, dt1, k, sv.A[h], lane);
    float* cf = sv.coef + slab * (cap + 1);
    if (lane < k) cf[lane] = flush ? rw.w0 : rw.w0 * s_bc[lane];
    if (lane + 32 < k) cf[lane + 32] = flush ? rw.w1 : rw.w1 * s_bc[lane + 32];
    if (lane == 0) cf[cap] = rw.gam;
  }
}

template <int P, int N, class T, int RC>
__global__ void __launch_bounds__(kThreads, kMinBlocks<N>)
replay_step_kernel(StoreView sv, const T* __restrict__ x, const T* __restrict__ B,
                   const T* __restrict__ C, const T* __restrict__ dt, float* __restrict__ y) {
  using TL = Tile<P, N>;
  constexpr int RPW = TL::RPW, E = TL::E;
  constexpr int EPC = 16 / sizeof(T), XC = P / EPC, BC = N / EPC;  // 16-byte chunks per record
  extern __shared__ float4 smem4[];
  __shared__ float s_red[kWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y, b = blockIdx.z;
  const int h = g * sv.hpg + blockIdx.x;
  const int slab = b * sv.H + h;
  const int cap = sv.cap;
  const size_t xo = static_cast<size_t>(slab) * P;  // x[b][h][:] and y[b][h][:]
  const size_t bo = (static_cast<size_t>(b) * sv.G + g) * N;

  // Independent of the prep kernel: the slab a non-flush step reads, C, x for D x.
  float hv[RPW][E];
  if constexpr (RC == REPLAY_RC_NONE) {
    load_tile_f32<P, N>(sv.h0 + static_cast<size_t>(slab) * P * N, warp, lane, hv);
  } else {
    const float scale = RC == REPLAY_RC_FP8E4M3 ? sv.scale[slab] : 1.f;
    load_tile_rc<P, N, RC>(sv.rc, slab, scale, warp, lane, hv);
  }
  float cv[E];
  load_cols<P, N>(C + bo, lane, cv);
  const int myrow = warp * RPW + transpose_index<RPW>(lane);
  const float xk_row = to_f(x[xo + myrow]);
  const float Dh = sv.D[h];

  griddep_wait();  // plan and coefficients of this step are written
  const int4 pl = sv.plan[b];
  const int start = pl.x, n = pl.y;
  if (pl.z == kPlanBad) {
    if (tid < P) y[xo + tid] = __int_as_float(0x7fc00000);
    return;
  }
  const int k = n + 1;
  const float* cf = sv.coef + static_cast<size_t>(slab) * (cap + 1);
  const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
  auto x_of = [&](int s) { return s < n ? ring.x + static_cast<size_t>(ring_slot(start, s, cap)) * P : x + xo; };

  if (pl.z == kPlanNonFlush) {
    float xr[RPW];
    if (lane < k) {
      load_rows<RPW>(x_of(lane) + warp * RPW, xr);
      const float c0 = cf[lane];
#pragma unroll
      for (int i = 0; i < RPW; ++i) xr[i] *= c0;
    } else {
#pragma unroll
      for (int i = 0; i < RPW; ++i) xr[i] = 0.f;
    }
    if (lane + 32 < k) {
      float x1[RPW];
      load_rows<RPW>(x_of(lane + 32) + warp * RPW, x1);
      const float c1 = cf[lane + 32];
#pragma unroll
      for (int i = 0; i < RPW; ++i) xr[i] = fmaf(c1, x1[i], xr[i]);
    }
    const float sum = tile_rows_dot<P, N>(hv, cv, cf[cap], xr, lane);
    if (transpose_leader<RPW>(lane)) y[xo + myrow] = fmaf(Dh, xk_row, sum);
    // append this token's record at ring slot start + n (B once per group, by its first head)
    const int slot = ring_slot(start, n, cap);
    if (tid < XC) {
      *reinterpret_cast<uint4*>(ring.x + static_cast<size_t>(slot) * P + tid * EPC) =
          *reinterpret_cast<const uint4*>(x + xo + tid * EPC);
    } else if (blockIdx.x == 0 && tid < XC + BC) {
      const int c = tid - XC;
      *reinterpret_cast<uint4*>(ring.b + static_cast<size_t>(slot) * N + c * EPC) =
          *reinterpret_cast<const uint4*>(B + bo + c * EPC);
    } else if (tid == XC + BC) {
      ring.dt[slot] = dt[slab];
    }
    return;
  }

  // ---------------- flush: fold the k records into h0, write it once, read y from it
  if constexpr (RC != REPLAY_RC_NONE)  // a flush starts from the FP32 checkpoint
    load_tile_f32<P, N>(sv.h0 + static_cast<size_t>(slab) * P * N, warp, lane, hv);
  float* sm_u = reinterpret_cast<float*>(smem4);  // [k][P]: w_s x_s
  float* sm_b = sm_u + cap * P;                   // [k][N]: B_s
  auto b_of = [&](int s) { return s < n ? ring.b + static_cast<size_t>(ring_slot(start, s, cap)) * N : B + bo; };
  stage_weighted<P, N, T>(x_of, b_of, cf, k, sm_u, sm_b);
  __syncthreads();
  fold_staged<P, N>(sm_u, sm_b, k, cf[cap], hv);
  float zero[RPW];
#pragma unroll
  for (int i = 0; i < RPW; ++i) zero[i] = 0.f;
  const float sum = tile_rows_dot<P, N>(hv, cv, 1.f, zero, lane);
  if (transpose_leader<RPW>(lane)) y[xo + myrow] = fmaf(Dh, xk_row, sum);
  write_checkpoint<P, N, RC>(sv, slab, s_red, hv);
}

template <int P, int N, class T, int RC>
static int launch(const StoreView& sv, const void* x, const void* B, const void* C, const void* dt,
                  float* y, cudaStream_t stream) {
  auto prep = replay_step_prep_kernel<P, N, T>;
  const size_t psmem = static_cast<size_t>(sv.cap + 1) * N * sizeof(T);
  if (psmem > 48 * 1024 &&
      cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(psmem)) !=
          cudaSuccess)
    return REPLAY_ECUDA;
  prep<<<dim3(sv.G, sv.batch), kThreads, psmem, stream>>>(sv, static_cast<const T*>(B), static_cast<const T*>(C),
                                                          static_cast<const T*>(dt));
  if (cudaGetLastError() != cudaSuccess) return REPLAY_ECUDA;
  auto kern = replay_step_kernel<P, N, T, RC>;
  const size_t smem = fold_staging_bytes<P, N>(sv.cap);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess)
    return REPLAY_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sv.hpg, sv.G, sv.batch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, sv, static_cast<const T*>(x), static_cast<const T*>(B),
                                           static_cast<const T*>(C), static_cast<const T*>(dt), y);
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? REPLAY_OK : REPLAY_ECUDA;
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
