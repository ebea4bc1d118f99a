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

// The prep CTAs must all be resident before the per-head kernel can start (programmatic
// dependent launch), so they are kept small: 128 threads.
constexpr int kPrepThreads = 128, kPrepWarps = kPrepThreads / 32;

template <int P, int N, class T>
__global__ void __launch_bounds__(kPrepThreads)
replay_step_prep_kernel(StoreView sv, const T* __restrict__ B, const T* __restrict__ C,
                        const T* __restrict__ dt) {
  using TL = Tile<P, N>;
  extern __shared__ float4 smem4[];
  __shared__ int4 s_meta;
  __shared__ float s_bc[kMaxCap];
  __shared__ float s_dt[kDtStage];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x, b = blockIdx.y;
  const int cap = sv.cap;
  griddep_launch_dependents();  // the head CTAs may start their checkpoint loads now
  if (tid == 0) s_meta = sv.meta[b];
  __syncthreads();
  const int start = s_meta.x, n = s_meta.y, epoch = s_meta.w;
  const int k = n + 1;
  if (n < 0 || k > cap || start < 0 || start >= cap) {
    if (tid == 0) {
      if (g == 0) sv.plan[b] = make_int4(start, n, kPlanBad, epoch);
      set_status(sv.status, REPLAY_DEV_BAD_META);
    }
    return;
  }
  const bool flush = k >= sv.L;
  if (tid == 0) {
    if (g == 0) sv.plan[b] = make_int4(start, n, flush ? kPlanFlush : kPlanNonFlush, epoch);
    arrive_and_publish(sv, b,
                       flush ? make_int4(ring_slot(start, k, cap), 0, 0, epoch + 1) : make_int4(start, k, 0, epoch),
                       sv.G);
  }
  const size_t bo = (static_cast<size_t>(b) * sv.G + g) * N;
  // One round trip for everything: the k records' B and this token's C go to shared memory by
  // cp.async (non-flush only), and meanwhile every head's k dt values (when they fit).
  T* sb = reinterpret_cast<T*>(smem4);  // [k][N] B, then [N] C
  if (!flush) {
    const T* bring = static_cast<const T*>(sv.bbuf) + (static_cast<size_t>(b) * sv.G + g) * cap * N;
    constexpr int EPC = 16 / sizeof(T), BC = N / EPC;
    for (int c = tid; c < (k + 1) * BC; c += kPrepThreads) {
      const int r = c / BC, off = (c - r * BC) * EPC;
      const T* src = r == k ? C + bo : (r < n ? bring + static_cast<size_t>(ring_slot(start, r, cap)) * N : B + bo);
      cp_async16(sb + static_cast<size_t>(r) * N + off, src + off);
    }
  }
  const bool stage_dt = sv.hpg * k <= kDtStage;
  if (stage_dt) {
    for (int idx = tid; idx < sv.hpg * k; idx += kPrepThreads) {
      const int hh = idx / k, s = idx - hh * k;
      const size_t slab = static_cast<size_t>(b) * sv.H + g * sv.hpg + hh;
      const T* dtr = static_cast<const T*>(sv.dtbuf) + slab * cap;
      s_dt[idx] = to_f(s < n ? dtr[ring_slot(start, s, cap)] : dt[slab]);
    }
  }
  if (!flush) {
    cp_async_wait_all();
    __syncthreads();
    float cv[TL::E];
    load_cols<P, N>(sb + static_cast<size_t>(k) * N, lane, cv);
    for (int s = warp; s < k; s += kPrepWarps) {
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
  for (int hh = warp; hh < sv.hpg; hh += kPrepWarps) {
    const int h = g * sv.hpg + hh;
    const size_t slab = static_cast<size_t>(b) * sv.H + h;
    const T* dtr = static_cast<const T*>(sv.dtbuf) + slab * cap;
    auto dt_of = [&](int s) {
      return stage_dt ? s_dt[hh * k + s] : to_f(s < n ? dtr[ring_slot(start, s, cap)] : dt[slab]);
    };
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
  if constexpr (RC != REPLAY_RC_NONE) {  // a flush starts from the FP32 checkpoint
    if (!sv.shared)                      // (a shared copy is the checkpoint: already loaded)
      load_tile_f32<P, N>(sv.h0 + static_cast<size_t>(slab) * P * N, warp, lane, hv);
  }
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
  write_checkpoint<P, N, RC>(sv, slab, s_red, hv, pl.w);
}

// ---------------------------------------------------------------------------------------
// With a read copy the slab a non-flush step reads is 2x (bf16) or 4x (E4M3) smaller, so a
// one-head CTA would keep that much less in flight. This variant gives a CTA HPC heads of
// one group: their copy tiles are loaded packed (about 32 registers in all, like one FP32
// tile) before the prep wait, and widened head by head when used. A flush handles the CTA's
// heads one after another from their FP32 checkpoints.
template <int N, int RC>
constexpr int heads_per_cta() {
  constexpr int VEC = N >= 128 ? 4 : 2, NVEC = N / (32 * VEC);
  constexpr int words = (sizeof(typename PackOf<RC, VEC>::type) + 3) / 4;
  constexpr int h = 32 / (8 * NVEC * words);
  return h < 1 ? 1 : h;
}

template <int P, int N, class T, int RC, int HPC>
__global__ void __launch_bounds__(kThreads, kMinBlocks<N>)
replay_step_copy_kernel(StoreView sv, const T* __restrict__ x, const T* __restrict__ B,
                        const T* __restrict__ C, const T* __restrict__ dt, float* __restrict__ y) {
  using TL = Tile<P, N>;
  constexpr int RPW = TL::RPW, E = TL::E, VEC = TL::VEC, NVEC = TL::NVEC;
  constexpr int EPC = 16 / sizeof(T), XC = P / EPC, BC = N / EPC;
  using PT = typename PackOf<RC, VEC>::type;
  extern __shared__ float4 smem4[];
  __shared__ float s_red[kWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y, b = blockIdx.z;
  const int hfirst = g * sv.hpg + blockIdx.x * HPC;
  const int slab0 = b * sv.H + hfirst;
  const int cap = sv.cap;
  const size_t bo = (static_cast<size_t>(b) * sv.G + g) * N;

  PT pk[HPC][RPW][NVEC];
  float scl[HPC];
#pragma unroll
  for (int hh = 0; hh < HPC; ++hh) {
    scl[hh] = RC == REPLAY_RC_FP8E4M3 ? sv.scale[slab0 + hh] : 1.f;
#pragma unroll
    for (int i = 0; i < RPW; ++i)
#pragma unroll
      for (int v = 0; v < NVEC; ++v)
        pk[hh][i][v] = ld_pack<RC, VEC>(
            sv.rc, static_cast<size_t>(slab0 + hh) * P * N + TL::row(warp, i) * N + TL::col(lane, v));
  }
  float cv[E];
  load_cols<P, N>(C + bo, lane, cv);
  const int myrow = warp * RPW + transpose_index<RPW>(lane);

  griddep_wait();  // plan and coefficients of this step are written
  const int4 pl = sv.plan[b];
  const int start = pl.x, n = pl.y;
  if (pl.z == kPlanBad) {
    for (int hh = 0; hh < HPC; ++hh)
      if (tid < P) y[static_cast<size_t>(slab0 + hh) * P + tid] = __int_as_float(0x7fc00000);
    return;
  }
  const int k = n + 1;

  if (pl.z == kPlanNonFlush) {
    const int slot = ring_slot(start, n, cap);
#pragma unroll
    for (int hh = 0; hh < HPC; ++hh) {
      const int h = hfirst + hh, slab = slab0 + hh;
      const size_t xo = static_cast<size_t>(slab) * P;
      const float* cf = sv.coef + static_cast<size_t>(slab) * (cap + 1);
      const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
      auto x_of = [&](int s) { return s < n ? ring.x + static_cast<size_t>(ring_slot(start, s, cap)) * P : x + xo; };
      float ex[RPW];
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
      const float gam = cf[cap];
      float part[RPW];
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        float hc = 0.f;
#pragma unroll
        for (int v = 0; v < NVEC; ++v) {
          float w[VEC];
          unpack<RC, VEC>(pk[hh][i][v], scl[hh], w);
#pragma unroll
          for (int e = 0; e < VEC; ++e) hc = fmaf(w[e], cv[v * VEC + e], hc);
        }
        part[i] = fmaf(gam, hc, ex[i]);
      }
      const float sum = warp_transpose_reduce<RPW>(part, lane);
      if (transpose_leader<RPW>(lane)) y[xo + myrow] = fmaf(sv.D[h], to_f(x[xo + myrow]), sum);
      // append this head's record at ring slot start + n (B once per group)
      if (tid < XC) {
        *reinterpret_cast<uint4*>(ring.x + static_cast<size_t>(slot) * P + tid * EPC) =
            *reinterpret_cast<const uint4*>(x + xo + tid * EPC);
      } else if (blockIdx.x == 0 && hh == 0 && tid < XC + BC) {
        const int c = tid - XC;
        *reinterpret_cast<uint4*>(ring.b + static_cast<size_t>(slot) * N + c * EPC) =
            *reinterpret_cast<const uint4*>(B + bo + c * EPC);
      } else if (tid == XC + BC) {
        ring.dt[slot] = dt[slab];
      }
    }
    return;
  }

  // ---------------- flush, head by head from the FP32 checkpoints
  float* sm_u = reinterpret_cast<float*>(smem4);
  float* sm_b = sm_u + cap * P;
  for (int hh = 0; hh < HPC; ++hh) {
    const int h = hfirst + hh, slab = slab0 + hh;
    const size_t xo = static_cast<size_t>(slab) * P;
    const float* cf = sv.coef + static_cast<size_t>(slab) * (cap + 1);
    const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
    float hv[RPW][E];
    if (sv.shared) {  // the copy is the checkpoint: widen the packed tile already loaded
#pragma unroll
      for (int i = 0; i < RPW; ++i)
#pragma unroll
        for (int v = 0; v < NVEC; ++v) {
          float w[VEC];
          unpack<RC, VEC>(pk[hh][i][v], scl[hh], w);
#pragma unroll
          for (int e = 0; e < VEC; ++e) hv[i][v * VEC + e] = w[e];
        }
    } else {
      load_tile_f32<P, N>(sv.h0 + static_cast<size_t>(slab) * P * N, warp, lane, hv);
    }
    auto x_of = [&](int s) { return s < n ? ring.x + static_cast<size_t>(ring_slot(start, s, cap)) * P : x + xo; };
    auto b_of = [&](int s) { return s < n ? ring.b + static_cast<size_t>(ring_slot(start, s, cap)) * N : B + bo; };
    if (hh > 0) __syncthreads();  // the previous head's staging has been read
    stage_weighted<P, N, T>(x_of, b_of, cf, k, sm_u, sm_b);
    __syncthreads();
    fold_staged<P, N>(sm_u, sm_b, k, cf[cap], hv);
    float zero[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) zero[i] = 0.f;
    const float sum = tile_rows_dot<P, N>(hv, cv, 1.f, zero, lane);
    if (transpose_leader<RPW>(lane)) y[xo + myrow] = fmaf(sv.D[h], to_f(x[xo + myrow]), sum);
    write_checkpoint<P, N, RC>(sv, slab, s_red, hv, pl.w);
  }
}

// ---------------------------------------------------------------------------------------
// Small calls (few slabs, so few waves): one fused kernel. Each head's CTA copies its slab's
// whole ring (x of the head, B of the group, dt) and the current record into a shared-memory
// image with cp.async while its checkpoint loads are in flight -- nothing waits on the ring
// pointer -- then forms its own coefficients. One launch and one round trip, instead of the
// prep -> per-head chain whose latency the large calls hide behind their checkpoint reads.
// Image slots 0..cap-1 mirror the ring; slot cap holds the current token's record.
template <int P, int N, class T>
__host__ __device__ constexpr size_t whole_image_bytes(int cap) {
  return static_cast<size_t>(cap + 1) * (P + N) * sizeof(T) + static_cast<size_t>(cap + 1) * sizeof(float);
}

template <int P, int N, class T, int RC>
__global__ void __launch_bounds__(kThreads, kMinBlocks<N>)
replay_step_fused_kernel(StoreView sv, const T* __restrict__ x, const T* __restrict__ B,
                         const T* __restrict__ C, const T* __restrict__ dt, float* __restrict__ y) {
  using TL = Tile<P, N>;
  constexpr int RPW = TL::RPW, E = TL::E;
  constexpr int EPC = 16 / sizeof(T), XC = P / EPC, BC = N / EPC;
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
  const size_t xo = static_cast<size_t>(slab) * P;
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
  RingImage<T> im;
  im.x = reinterpret_cast<T*>(smem4);
  im.b = im.x + static_cast<size_t>(cap + 1) * P;
  im.dt = reinterpret_cast<float*>(im.b + static_cast<size_t>(cap + 1) * N);
  const T dtcur = dt[slab];
  for (int c = tid; c < (cap + 1) * (XC + BC); c += kThreads) {
    if (c < (cap + 1) * XC) {
      const int s = c / XC, off = (c - s * XC) * EPC;
      cp_async16(im.x + s * P + off, (s < cap ? ring.x + static_cast<size_t>(s) * P : x + xo) + off);
    } else {
      const int c2 = c - (cap + 1) * XC;
      const int s = c2 / BC, off = (c2 - s * BC) * EPC;
      cp_async16(im.b + s * N + off, (s < cap ? ring.b + static_cast<size_t>(s) * N : B + bo) + off);
    }
  }
  for (int s = tid; s <= cap; s += kThreads) im.dt[s] = to_f(s < cap ? ring.dt[s] : dtcur);
  float cv[E];
  load_cols<P, N>(C + bo, lane, cv);
  const int myrow = warp * RPW + transpose_index<RPW>(lane);
  const float xk_row = to_f(x[xo + myrow]);
  const float A = sv.A[h], Dh = sv.D[h];
  cp_async_wait_all();
  __syncthreads();

  const int start = s_meta.x, n = s_meta.y, epoch = s_meta.w;
  const int k = n + 1;
  if (n < 0 || k > cap || start < 0 || start >= cap) {
    if (tid < P) y[xo + tid] = __int_as_float(0x7fc00000);
    if (tid == 0) set_status(sv.status, REPLAY_DEV_BAD_META);
    return;
  }
  const bool flush = k >= sv.L;
  if (tid == 0)
    arrive_and_publish(sv, b,
                       flush ? make_int4(ring_slot(start, k, cap), 0, 0, epoch + 1) : make_int4(start, k, 0, epoch),
                       sv.H);
  auto slot_of = [&](int s) { return s < n ? ring_slot(start, s, cap) : cap; };

  if (flush) {
    if constexpr (RC != REPLAY_RC_NONE) {
      if (!sv.shared) load_tile_f32<P, N>(sv.h0 + static_cast<size_t>(slab) * P * N, warp, lane, hv);
    }
    float* sm_u = fold_staging(smem4, whole_image_bytes<P, N, T>(cap));
    fold_tile<P, N, T>(im, slot_of, k, A, sm_u, sm_u + cap * P, s_w, hv);
    float zero[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) zero[i] = 0.f;
    const float sum = tile_rows_dot<P, N>(hv, cv, 1.f, zero, lane);
    if (transpose_leader<RPW>(lane)) y[xo + myrow] = fmaf(Dh, xk_row, sum);
    write_checkpoint<P, N, RC>(sv, slab, s_red, hv, epoch);
    return;
  }
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
  append_record<P, N, T>(ring, im, cap, ring_slot(start, n, cap), blockIdx.x == 0, dtcur);
}

// Calls with at most this many (sequence, head) slabs take the fused kernel.
constexpr long long kFusedMaxSlabs = 1024;

template <int P, int N, class T, int RC>
static int launch(const StoreView& sv, const void* x, const void* B, const void* C, const void* dt,
                  float* y, cudaStream_t stream) {
  if (static_cast<long long>(sv.batch) * sv.H <= kFusedMaxSlabs) {
    auto fused = replay_step_fused_kernel<P, N, T, RC>;
    const size_t fsmem = smem_plan_bytes<P, N>(whole_image_bytes<P, N, T>(sv.cap), sv.cap);
    if (fsmem > 48 * 1024 &&
        cudaFuncSetAttribute(fused, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(fsmem)) !=
            cudaSuccess)
      return REPLAY_ECUDA;
    fused<<<dim3(sv.hpg, sv.G, sv.batch), kThreads, fsmem, stream>>>(
        sv, static_cast<const T*>(x), static_cast<const T*>(B), static_cast<const T*>(C),
        static_cast<const T*>(dt), y);
    return cudaGetLastError() == cudaSuccess ? REPLAY_OK : REPLAY_ECUDA;
  }
  auto prep = replay_step_prep_kernel<P, N, T>;
  const size_t psmem = static_cast<size_t>(sv.cap + 1) * N * sizeof(T);
  if (psmem > 48 * 1024 &&
      cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(psmem)) !=
          cudaSuccess)
    return REPLAY_ECUDA;
  prep<<<dim3(sv.G, sv.batch), kPrepThreads, psmem, stream>>>(sv, static_cast<const T*>(B), static_cast<const T*>(C),
                                                          static_cast<const T*>(dt));
  if (cudaGetLastError() != cudaSuccess) return REPLAY_ECUDA;
  auto kern = replay_step_kernel<P, N, T, RC>;
  int heads = 1;  // heads per CTA
  if constexpr (RC != REPLAY_RC_NONE) {
    constexpr int HPC = heads_per_cta<N, RC>();
    if (HPC > 1 && sv.hpg % HPC == 0) {
      kern = replay_step_copy_kernel<P, N, T, RC, HPC>;
      heads = HPC;
    }
  }
  const size_t smem = fold_staging_bytes<P, N>(sv.cap);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess)
    return REPLAY_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sv.hpg / heads, sv.G, sv.batch);
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
