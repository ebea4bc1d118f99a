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
// Which per-head kernel runs is chosen on the host and never changes results (each handles
// any plan): replay_step_read_kernel (FP32 checkpoint, phase known: the slab by one bulk copy
// into shared memory), replay_step_copy_read_kernel / replay_step_copy_kernel (bf16, E4M3,
// FP16 read copies, several heads per CTA), replay_step_fp4_kernel (NVFP4 read copy, h0 . C
// on the tensor cores), replay_step_kernel (the rest: unknown phase, flushes of read-copy
// stores); calls of at most 1024 slabs take replay_step_fused_kernel and no prep. With a
// read copy, a step's prep may run during the previous step's per-head kernel (see launch).
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
                        const T* __restrict__ dt, int overlap) {
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
    if (overlap) griddep_wait();
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
  if (!flush && sv.prep_appends) {  // this token's B (the group's) and dt (each head's) into slot start + n
    // An empty ring means the previous step flushed after all (the host expected it not to):
    // its fold may still be reading this slot, so wait for it to complete first.
    if (overlap && n == 0) griddep_wait();
    constexpr int EPC = 16 / sizeof(T), BC = N / EPC;
    const int slot = ring_slot(start, n, cap);
    T* bslot = static_cast<T*>(sv.bbuf) + ((static_cast<size_t>(b) * sv.G + g) * cap + slot) * N;
    for (int c = tid; c < BC; c += kPrepThreads)
      *reinterpret_cast<uint4*>(bslot + c * EPC) = *reinterpret_cast<const uint4*>(B + bo + c * EPC);
    for (int hh = tid; hh < sv.hpg; hh += kPrepThreads) {
      const size_t slab = static_cast<size_t>(b) * sv.H + g * sv.hpg + hh;
      static_cast<T*>(sv.dtbuf)[slab * cap + slot] = dt[slab];
    }
  }
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
  if (k <= 16) {  // two heads per warp: half-warp scans
    for (int hp = 2 * warp; hp < sv.hpg; hp += 2 * kPrepWarps) {
      const int hh = hp + (lane >> 4), s = lane & 15;
      const bool live = hh < sv.hpg;
      const int h = g * sv.hpg + (live ? hh : hp);
      const size_t slab = static_cast<size_t>(b) * sv.H + h;
      const T* dtr = static_cast<const T*>(sv.dtbuf) + slab * cap;
      float dtv = 0.f;
      if (live && s < k)
        dtv = stage_dt ? s_dt[hh * k + s] : to_f(s < n ? dtr[ring_slot(start, s, cap)] : dt[slab]);
      const HalfWeights rw = record_weights_pair(dtv, k, sv.A[h], lane);
      float* cf = sv.coef + slab * (cap + 1);
      if (live && s < k) cf[s] = flush ? rw.w : rw.w * s_bc[s];
      if (live && s == 0) cf[cap] = rw.gam;
    }
    if (overlap) griddep_wait();  // this grid completes after the previous step's kernels
    return;
  }
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
  if (overlap) griddep_wait();  // this grid completes after the previous step's kernels
}

// The state bytes of slabs [slab, slab + nslab) as a per-head kernel reads them: the
// checkpoint, or the read copy (NVFP4: codes and block scales).
template <int P, int N, int RC>
__device__ __forceinline__ void prefetch_slabs(const StoreView& sv, long long slab, int nslab, bool f32) {
  if (f32) {  // the checkpoint (FP32, or FP16)
    const unsigned esz = sv.ckpt16 ? 2u : 4u;
    prefetch_l2(reinterpret_cast<const uint8_t*>(sv.h0) + slab * P * N * esz, nslab * (P * N * esz));
  } else if constexpr (RC == REPLAY_RC_NVFP4) {
    prefetch_l2(static_cast<const uint8_t*>(sv.rc) + slab * (P * N / 2), nslab * (P * N / 2u));
    prefetch_l2(sv.bscale + slab * (P * N / kFp4Block), nslab * (P * N / static_cast<unsigned>(kFp4Block)));
  } else if constexpr (RC != REPLAY_RC_NONE) {
    constexpr unsigned esz = RC == REPLAY_RC_FP8E4M3 ? 1u : 2u;
    prefetch_l2(static_cast<const uint8_t*>(sv.rc) + slab * P * N * esz, nslab * (P * N * esz));
  }
}

// A CTA covering slabs [slab0, slab0 + nslab) sends to L2 the slabs of the CTA one wave
// (SMs x resident CTAs per SM) after it: CTAs of these grids run in slab order, so that CTA
// starts about when this one ends, and finds its state in L2.
template <int P, int N, int RC>
__device__ __forceinline__ void prefetch_next_wave(const StoreView& sv, int slab0, int nslab, int ctas_per_sm,
                                                   bool f32) {
  if (threadIdx.x != 0 || sv.sms <= 0) return;
  const long long ahead = slab0 + static_cast<long long>(sv.sms) * ctas_per_sm * nslab;
  if (ahead + nslab <= static_cast<long long>(sv.batch) * sv.H) prefetch_slabs<P, N, RC>(sv, ahead, nslab, f32);
}

// expect_flush: the host knows every sequence flushes on this step, so a CTA with a read copy
// loads the FP32 checkpoint (the flush's input) before the prep wait instead of the copy, and
// every CTA sends the slab of the CTA one wave later to L2 (a flush computes between its read
// and its write, so its own loads leave DRAM idle part of the time).
template <int P, int N, class T, int RC>
__global__ void __launch_bounds__(kThreads, kMinBlocks<N>)
replay_step_kernel(StoreView sv, const T* __restrict__ x, const T* __restrict__ B,
                   const T* __restrict__ C, const T* __restrict__ dt, float* __restrict__ y,
                   int expect_flush) {
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

  // Independent of the prep kernel: the slab the step most likely reads, C, x for D x.
  float hv[RPW][E];
  const bool f32_first = RC == REPLAY_RC_NONE || (expect_flush && !sv.shared);
  if (expect_flush) prefetch_next_wave<P, N, RC>(sv, slab, 1, kMinBlocks<N>, f32_first);
  auto load_copy = [&] {
    if constexpr (RC != REPLAY_RC_NONE) {
      const float scale = RC == REPLAY_RC_FP8E4M3 || RC == REPLAY_RC_NVFP4 ? sv.scale[slab] : 1.f;
      load_tile_rc<P, N, RC>(sv.rc, slab, scale, warp, lane, hv, sv.bscale);
    }
  };
  if (f32_first)
    load_checkpoint<P, N>(sv, slab, warp, lane, hv);
  else
    load_copy();
  float cv[E];
  load_cols<P, N>(C + bo, lane, cv);
  const int myrow = warp * RPW + transpose_index<RPW>(lane);
  const float xk_row = to_f(x[xo + myrow]);
  const float Dh = sv.D[h];

  griddep_wait();  // plan and coefficients of this step are written
  // (read-copy stores only: there the next step's prep may overlap this kernel; the trigger
  // instruction, even when not executed, measurably slows these kernels, so FP32 ones lack it)
  if constexpr (RC != REPLAY_RC_NONE) griddep_launch_dependents();
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
    if (RC != REPLAY_RC_NONE && f32_first) load_copy();  // a non-flush step reads the copy
    float xr[RPW];
    record_terms<RPW, T>(x_of, cf, k, warp, lane, xr);
    const float sum = tile_rows_dot<P, N>(hv, cv, cf[cap], xr, lane);
    if (transpose_leader<RPW>(lane)) y[xo + myrow] = fmaf(Dh, xk_row, sum);
    // append this token's record at ring slot start + n (B and dt here unless the prep does)
    const int slot = ring_slot(start, n, cap);
    if (tid < XC) {
      *reinterpret_cast<uint4*>(ring.x + static_cast<size_t>(slot) * P + tid * EPC) =
          *reinterpret_cast<const uint4*>(x + xo + tid * EPC);
    } else if (!sv.prep_appends && blockIdx.x == 0 && tid < XC + BC) {  // B once per group
      const int c = tid - XC;
      *reinterpret_cast<uint4*>(ring.b + static_cast<size_t>(slot) * N + c * EPC) =
          *reinterpret_cast<const uint4*>(B + bo + c * EPC);
    } else if (!sv.prep_appends && tid == XC + BC) {
      ring.dt[slot] = dt[slab];
    }
    return;
  }

  // ---------------- flush: fold the k records into h0, write it once, read y from it
  // (from the FP32 checkpoint; a shared copy is the checkpoint and is already loaded)
  if (!f32_first && !sv.shared) load_checkpoint<P, N>(sv, slab, warp, lane, hv);
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
// replay_step_copy_read_kernel: a bf16, E4M3 or FP16 read-copy step the host knows flushes
// no sequence. The CTA's HPC copy slabs are contiguous, so one bulk copy brings them into
// shared memory (the packed tiles no longer take 32 registers, and the copy is in flight
// without holding registers or L1), and every head's record terms are loaded before the copy
// is waited for, so the HPC heads' record latencies overlap the copy instead of following
// one dot product after another. A flush plan, not expected here, is folded head by head
// from the records in global memory.
// The flush of a read-copy CTA's HPC heads when a flush plan reaches the bulk-copy read
// kernel (the host expected none): head by head, from the FP32 checkpoint (or from the copy
// in shared memory when the copy is the checkpoint), records read from global memory. Kept
// out of line: it holds a whole register tile, the read path does not.
template <int P, int N, class T, int RC, int HPC>
__device__ __noinline__ void copy_read_flush(const StoreView& sv, const T* __restrict__ x, const T* __restrict__ B,
                                             const T* __restrict__ C, float* __restrict__ y, const uint8_t* s_rc,
                                             const float* scl, int start, int n, int epoch, float* s_red) {
  using TL = Tile<P, N>;
  constexpr int RPW = TL::RPW, E = TL::E, VEC = TL::VEC, NVEC = TL::NVEC;
  constexpr int ESZ = RC == REPLAY_RC_FP8E4M3 ? 1 : 2;
  using PT = typename PackOf<RC, VEC>::type;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y, b = blockIdx.z;
  const int hfirst = g * sv.hpg + blockIdx.x * HPC;
  const int slab0 = b * sv.H + hfirst;
  const int cap = sv.cap, k = n + 1;
  const size_t bo = (static_cast<size_t>(b) * sv.G + g) * N;
  const int myrow = warp * RPW + transpose_index<RPW>(lane);
  float cv[E];
  load_cols<P, N>(C + bo, lane, cv);
  for (int hh = 0; hh < HPC; ++hh) {
    const int h = hfirst + hh, slab = slab0 + hh;
    const size_t xo = static_cast<size_t>(slab) * P;
    const float* cf = sv.coef + static_cast<size_t>(slab) * (cap + 1);
    const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
    float hv[RPW][E];
    if (sv.shared) {
#pragma unroll
      for (int i = 0; i < RPW; ++i)
#pragma unroll
        for (int v = 0; v < NVEC; ++v) {
          const size_t elem = static_cast<size_t>(hh) * P * N + TL::row(warp, i) * N + TL::col(lane, v);
          float w[VEC];
          unpack<RC, VEC>(*reinterpret_cast<const PT*>(s_rc + elem * ESZ), scl[hh], w);
#pragma unroll
          for (int e = 0; e < VEC; ++e) hv[i][v * VEC + e] = w[e];
        }
    } else {
      load_checkpoint<P, N>(sv, slab, warp, lane, hv);
    }
    const float gam = cf[cap];
#pragma unroll
    for (int i = 0; i < RPW; ++i)
#pragma unroll
      for (int e = 0; e < E; ++e) hv[i][e] *= gam;
    for (int s = 0; s < k; ++s) {
      const int slot = ring_slot(start, s, cap);
      float u[RPW], bv[E];
      load_rows<RPW>((s < n ? ring.x + static_cast<size_t>(slot) * P : x + xo) + warp * RPW, u);
      load_cols<P, N>(s < n ? ring.b + static_cast<size_t>(slot) * N : B + bo, lane, bv);
      const float w = cf[s];
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
    write_checkpoint<P, N, RC>(sv, slab, s_red, hv, epoch);
  }
}

template <int N, int HPC>
constexpr int kCopyReadCtas = N >= 256 ? 3 : (HPC >= 4 ? 4 : 6);

template <int P, int N, class T, int RC, int HPC>
__global__ void __launch_bounds__(kThreads, kCopyReadCtas<N, HPC>)
replay_step_copy_read_kernel(StoreView sv, const T* __restrict__ x, const T* __restrict__ B,
                             const T* __restrict__ C, const T* __restrict__ dt, float* __restrict__ y) {
  using TL = Tile<P, N>;
  constexpr int RPW = TL::RPW, E = TL::E, VEC = TL::VEC, NVEC = TL::NVEC;
  constexpr int EPC = 16 / sizeof(T), XC = P / EPC, BC = N / EPC;
  constexpr int ESZ = RC == REPLAY_RC_FP8E4M3 ? 1 : 2;
  constexpr unsigned SLAB_BYTES = P * N * ESZ;
  using PT = typename PackOf<RC, VEC>::type;
  extern __shared__ float4 smem4[];
  __shared__ float s_red[kWarps];
  __shared__ __align__(8) unsigned long long s_bar;
  __shared__ int s_landed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y, b = blockIdx.z;
  const int hfirst = g * sv.hpg + blockIdx.x * HPC;
  const int slab0 = b * sv.H + hfirst;
  const int cap = sv.cap;
  const size_t bo = (static_cast<size_t>(b) * sv.G + g) * N;
  const uint8_t* s_rc = reinterpret_cast<const uint8_t*>(smem4);
  if (tid == 0) {
    mbar_init(&s_bar);
    bulk_load(smem4, static_cast<const uint8_t*>(sv.rc) + static_cast<size_t>(slab0) * SLAB_BYTES,
              HPC * SLAB_BYTES, &s_bar);
  }
  const uint8_t* my_rc = s_rc + (TL::row(warp, 0) * N + TL::col(lane, 0)) * ESZ;  // this lane's first pack
  auto tile_pack = [&](int hh, int i, int v) {
    return *reinterpret_cast<const PT*>(my_rc + (hh * P * N + i * N + v * 32 * VEC) * ESZ);
  };
  float scl[HPC];
#pragma unroll
  for (int hh = 0; hh < HPC; ++hh) scl[hh] = RC == REPLAY_RC_FP8E4M3 ? sv.scale[slab0 + hh] : 1.f;
  float cv[E];
  load_cols<P, N>(C + bo, lane, cv);
  float2 cv2[E / 2];
#pragma unroll
  for (int j = 0; j < E / 2; ++j) cv2[j] = make_float2(cv[2 * j], cv[2 * j + 1]);
  const int myrow = warp * RPW + transpose_index<RPW>(lane);

  griddep_wait();  // plan and coefficients of this step are written
  griddep_launch_dependents();  // after the wait: the next step's prep may start
  const int4 pl = sv.plan[b];
  const int start = pl.x, n = pl.y, k = n + 1;
  auto x_of_head = [&](int hh, int s) {
    const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, hfirst + hh, g);
    return s < n ? ring.x + static_cast<size_t>(ring_slot(start, s, cap)) * P
                 : x + static_cast<size_t>(slab0 + hh) * P;
  };
  float ex[HPC][RPW];
  if (pl.z == kPlanNonFlush) {
#pragma unroll
    for (int hh = 0; hh < HPC; ++hh) {
      const float* cf = sv.coef + static_cast<size_t>(slab0 + hh) * (cap + 1);
      record_terms<RPW, T>([&](int s) { return x_of_head(hh, s); }, cf, k, warp, lane, ex[hh]);
    }
  }
  // The copy must have landed before it is read or the CTA exits (bounded wait, see the FP32
  // read kernel).
  if (tid == 0) {
    const bool ok = mbar_wait(&s_bar, 0, kCopyWaitNs);
    if (!ok) {
      set_status(sv.status, REPLAY_DEV_COPY_TIMEOUT);
      mbar_wait(&s_bar, 0, kCopyWaitNs);
    }
    s_landed = ok;
  }
  __syncthreads();
  if (!s_landed || pl.z == kPlanBad) {
    for (int hh = 0; hh < HPC; ++hh)
      if (tid < P) y[static_cast<size_t>(slab0 + hh) * P + tid] = __int_as_float(0x7fc00000);
    return;
  }

  if (pl.z == kPlanNonFlush) {
    const int slot = ring_slot(start, n, cap);
#pragma unroll
    for (int hh = 0; hh < HPC; ++hh) {
      const int h = hfirst + hh, slab = slab0 + hh;
      const size_t xo = static_cast<size_t>(slab) * P;
      // Gamma h . C with the copy's pairs on packed FP32 FMAs; the slab scale once per row
      const float gs = sv.coef[static_cast<size_t>(slab) * (cap + 1) + cap] * scl[hh];
      float part[RPW];
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        float2 hc = make_float2(0.f, 0.f);
#pragma unroll
        for (int v = 0; v < NVEC; ++v) {
          float2 w[VEC / 2];
          unpack_pairs<RC, VEC>(tile_pack(hh, i, v), w);
#pragma unroll
          for (int j = 0; j < VEC / 2; ++j) hc = __ffma2_rn(w[j], cv2[v * VEC / 2 + j], hc);
        }
        part[i] = fmaf(gs, hc.x + hc.y, ex[hh][i]);
      }
      const float sum = warp_transpose_reduce<RPW>(part, lane);
      if (transpose_leader<RPW>(lane)) y[xo + myrow] = fmaf(sv.D[h], to_f(x[xo + myrow]), sum);
      const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
      if (tid < XC) {
        *reinterpret_cast<uint4*>(ring.x + static_cast<size_t>(slot) * P + tid * EPC) =
            *reinterpret_cast<const uint4*>(x + xo + tid * EPC);
      } else if (!sv.prep_appends && blockIdx.x == 0 && hh == 0 && tid < XC + BC) {
        const int c = tid - XC;
        *reinterpret_cast<uint4*>(ring.b + static_cast<size_t>(slot) * N + c * EPC) =
            *reinterpret_cast<const uint4*>(B + bo + c * EPC);
      } else if (!sv.prep_appends && tid == XC + BC) {
        ring.dt[slot] = dt[slab];
      }
    }
    return;
  }

  // flush (not expected): out of line, so that its registers do not weigh on the read path
  copy_read_flush<P, N, T, RC, HPC>(sv, x, B, C, y, s_rc, scl, start, n, pl.w, s_red);
}

// ---------------------------------------------------------------------------------------
// replay_step_e4m3_mma_kernel: the non-flush step of an E4M3 read copy at dstate 128 with the
// codes fed to the tensor cores as they are stored (`mma.sync` m16n8k32, E4M3 x E4M3 -> FP32):
// no code is decoded by an instruction. C must enter as E4M3 too, so it is split into 8 terms,
// one per MMA column: with s0 the power of two that brings max |C| below 256, r_0 = s0 C,
// t_j = e4m3(r_j) (round to nearest even) and r_{j+1} = 16 (r_j - t_j), every step exact in
// FP32, so s0 C = sum_j t_j 16^-j up to 2^-33 of its largest value. Column j of the MMA result
// is then codes . t_j, products exact, and the row's h0 . C is scale / s0 * sum_j D[.][j] 16^-j.
// The CTA takes HR heads of a group (one bulk copy of their codes), two warps per head, 32
// rows each as two 16-row tiles. The MMA's k order is permuted so that lane (g, q) = (lane / 4,
// lane % 4) reads one contiguous 32-byte piece of each row it needs (two 16-byte loads): in
// k-tile kt, MMA k index 4q + i is column 32q + 8kt + i and 16 + 4q + i is column
// 32q + 8kt + 4 + i, for A (the codes) and B (the C terms) alike. A row's 128 products per
// term accumulate over the 4 k-tiles in the MMA accumulators. Lane (g, q) holds terms 2q and
// 2q + 1 of rows g and g + 8: it weights them, adds its share of the record terms (records q,
// q + 4, ... from x staged in shared memory by cp.async beside the copy) and two shuffles sum
// the row's four lanes.
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], const unsigned (&a)[4], unsigned b0, unsigned b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Dynamic shared memory of the E4M3 tensor-core read kernel: the HR copy slabs, the records' x
// of the HR heads ([HR][cap][P + 8], padded rows), their coefficients ([HR][cap + 1]).
template <int P, int N, class T, int HR>
constexpr size_t e4m3_mma_smem(int cap) {
  return static_cast<size_t>(HR) * P * N + static_cast<size_t>(HR) * cap * (P + 8) * sizeof(T) +
         static_cast<size_t>(HR) * (cap + 1) * sizeof(float);
}

template <int P, int N, class T, int HR>
__global__ void __launch_bounds__(kThreads, 5)
replay_step_e4m3_mma_kernel(StoreView sv, const T* __restrict__ x, const T* __restrict__ B,
                            const T* __restrict__ C, const T* __restrict__ dt, float* __restrict__ y) {
  static_assert(P == 64 && N == 128 && HR * 2 == kWarps, "two warps per head, 64 x 128 slabs");
  constexpr int RC = REPLAY_RC_FP8E4M3;
  constexpr int EPC = 16 / sizeof(T), XC = P / EPC, BC = N / EPC, XS = P + 8;
  constexpr unsigned SLAB_BYTES = P * N;
  extern __shared__ float4 smem4[];
  __shared__ float s_red[kWarps];
  __shared__ __align__(16) uint8_t s_terms[8][N];
  __shared__ float s_inv;
  __shared__ __align__(8) unsigned long long s_bar;
  __shared__ int s_landed;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, q = lane & 3;
  const int g = blockIdx.y, b = blockIdx.z;
  const int hfirst = g * sv.hpg + blockIdx.x * HR;
  const int slab0 = b * sv.H + hfirst;
  const int cap = sv.cap;
  const size_t bo = (static_cast<size_t>(b) * sv.G + g) * N;
  const uint8_t* s_rc = reinterpret_cast<const uint8_t*>(smem4);
  if (tid == 0) {
    mbar_init(&s_bar);
    bulk_load(smem4, static_cast<const uint8_t*>(sv.rc) + static_cast<size_t>(slab0) * SLAB_BYTES,
              HR * SLAB_BYTES, &s_bar);
  }
  // C's 8 E4M3 terms (two threads per column find the CTA-wide max |C|; one thread per two
  // columns builds their terms)
  {
    const float c = to_f(C[bo + (tid & (N - 1))]);
    const float m = warp_max(fabsf(c));
    if (lane == 0) s_red[warp] = m;
    __syncthreads();
    float cmax = s_red[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) cmax = fmaxf(cmax, s_red[w]);
    if (tid < N / 2) {  // columns 2 tid, 2 tid + 1
      const int ce = cmax > 0.f ? max(((__float_as_int(cmax) >> 23) & 0xff) - 127, -110) : 0;
      const float s0 = __int_as_float((127 + 7 - ce) << 23);
      float2 r = make_float2(to_f(C[bo + 2 * tid]) * s0, to_f(C[bo + 2 * tid + 1]) * s0);  // |r| < 256
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const unsigned short t2 =
            static_cast<unsigned short>(__nv_cvt_float2_to_fp8x2(r, __NV_SATFINITE, __NV_E4M3));
        *reinterpret_cast<unsigned short*>(&s_terms[j][2 * tid]) = t2;
        const float2 tv = e4m3x2_to_float2(t2);
        r = make_float2((r.x - tv.x) * 16.f, (r.y - tv.y) * 16.f);
      }
      if (tid == 0) s_inv = __int_as_float((127 - 7 + ce) << 23);  // 1 / s0
    }
  }
  __syncthreads();
  const float inv_s0 = s_inv;
  unsigned bt[4][2];  // B fragments: term gq at the lane's columns, per k-tile
#pragma unroll
  for (int kt = 0; kt < 4; ++kt) {
    const uint2 w = *reinterpret_cast<const uint2*>(&s_terms[gq][32 * q + 8 * kt]);
    bt[kt][0] = w.x;
    bt[kt][1] = w.y;
  }
  // the weights of the lane's two terms, 16^-2q and 16^-(2q+1)
  const float w0 = __int_as_float((127 - 8 * q) << 23), w1 = __int_as_float((127 - 8 * q - 4) << 23);

  griddep_wait();  // plan and coefficients of this step are written
  griddep_launch_dependents();  // after the wait: the next step's prep may start
  const int4 pl = sv.plan[b];
  const int start = pl.x, n = pl.y, k = n + 1;
  T* s_x = reinterpret_cast<T*>(smem4 + HR * SLAB_BYTES / 16);  // [HR][cap][XS]
  float* s_cf = reinterpret_cast<float*>(s_x + static_cast<size_t>(HR) * cap * XS);  // [HR][cap + 1]
  const bool nonflush = pl.z == kPlanNonFlush;
  if (nonflush) {  // the k records' x and the coefficients, beside the copy: one round trip
    const int off = (tid % XC) * EPC;
    for (int pr = tid / XC; pr < HR * k; pr += kThreads / XC) {  // (head, record) pairs
      const int hh = pr / k, s = pr - hh * k;
      const T* src = s < n ? slab_ring<P, N, T>(sv, b, hfirst + hh, g).x + static_cast<size_t>(ring_slot(start, s, cap)) * P
                           : x + static_cast<size_t>(slab0 + hh) * P;
      cp_async16(s_x + (static_cast<size_t>(hh) * cap + s) * XS + off, src + off);
    }
    for (int c = tid; c < HR * (cap + 1); c += kThreads)
      s_cf[c] = sv.coef[static_cast<size_t>(slab0) * (cap + 1) + c];  // the HR slabs' rows are consecutive
    cp_async_commit();
  }
  // The copy must have landed before it is read or the CTA exits (bounded wait, see the FP32
  // read kernel).
  if (tid == 0) {
    const bool ok = mbar_wait(&s_bar, 0, kCopyWaitNs);
    if (!ok) {
      set_status(sv.status, REPLAY_DEV_COPY_TIMEOUT);
      mbar_wait(&s_bar, 0, kCopyWaitNs);
    }
    s_landed = ok;
  }
  cp_async_wait_all();
  __syncthreads();
  if (!s_landed || pl.z == kPlanBad) {
    for (int hh = 0; hh < HR; ++hh)
      if (tid < P) y[static_cast<size_t>(slab0 + hh) * P + tid] = __int_as_float(0x7fc00000);
    return;
  }

  if (nonflush) {
    const int hh = warp >> 1, half = warp & 1;
    const int h = hfirst + hh, slab = slab0 + hh;
    const size_t xo = static_cast<size_t>(slab) * P;
    const float* cf = s_cf + hh * (cap + 1);
    const T* sxh = s_x + static_cast<size_t>(hh) * cap * XS;
    float part[4];  // rows 32 half + 16 t + 8 u + gq, index 2t + u
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int r0 = 32 * half + 16 * t + gq;
      const uint8_t* row0 = s_rc + hh * SLAB_BYTES + r0 * N + 32 * q;
      const uint4 lo0 = *reinterpret_cast<const uint4*>(row0), hi0 = *reinterpret_cast<const uint4*>(row0 + 16);
      const uint4 lo1 = *reinterpret_cast<const uint4*>(row0 + 8 * N), hi1 = *reinterpret_cast<const uint4*>(row0 + 8 * N + 16);
      const unsigned ra[8] = {lo0.x, lo0.y, lo0.z, lo0.w, hi0.x, hi0.y, hi0.z, hi0.w};
      const unsigned rb[8] = {lo1.x, lo1.y, lo1.z, lo1.w, hi1.x, hi1.y, hi1.z, hi1.w};
      float acc[4] = {0.f, 0.f, 0.f, 0.f};  // 128 exact products per element, as 4 MMAs
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
        const unsigned a[4] = {ra[2 * kt], rb[2 * kt], ra[2 * kt + 1], rb[2 * kt + 1]};
        mma_e4m3_16832(acc, a, bt[kt][0], bt[kt][1]);
      }
      part[2 * t] = fmaf(acc[1], w1, acc[0] * w0);      // row r0: terms 2q, 2q + 1
      part[2 * t + 1] = fmaf(acc[3], w1, acc[2] * w0);  // row r0 + 8
    }
    const float gs = cf[cap] * sv.scale[slab] * inv_s0;  // Gamma_k, the slab scale, 1 / s0
    float e[4] = {0.f, 0.f, 0.f, 0.f};  // the record terms of this lane's records q, q + 4, ...
    const T* xr = sxh + 32 * half + gq;
    for (int s = q; s < k; s += 4) {
      const float c = cf[s];
#pragma unroll
      for (int i = 0; i < 4; ++i) e[i] = fmaf(c, to_f(xr[s * XS + 16 * (i >> 1) + 8 * (i & 1)]), e[i]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      part[i] = fmaf(gs, part[i], e[i]);
      part[i] += __shfl_xor_sync(kFull, part[i], 1);
      part[i] += __shfl_xor_sync(kFull, part[i], 2);
    }
    // lane q writes its row q of the four: the warp's 32 rows in one 128-byte store
    const int rq = 32 * half + 16 * (q >> 1) + 8 * (q & 1) + gq;
    const float v = q == 0 ? part[0] : q == 1 ? part[1] : q == 2 ? part[2] : part[3];
    y[xo + rq] = fmaf(sv.D[h], to_f(x[xo + rq]), v);
    // this token's record: the warp pair's head
    const int slot = ring_slot(start, n, cap);
    const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
    const int ht = tid & 63;  // thread of the head's warp pair
    if (ht < XC) {
      *reinterpret_cast<uint4*>(ring.x + static_cast<size_t>(slot) * P + ht * EPC) =
          *reinterpret_cast<const uint4*>(x + xo + ht * EPC);
    } else if (!sv.prep_appends && blockIdx.x == 0 && hh == 0 && ht < XC + BC) {
      const int c = ht - XC;
      *reinterpret_cast<uint4*>(ring.b + static_cast<size_t>(slot) * N + c * EPC) =
          *reinterpret_cast<const uint4*>(B + bo + c * EPC);
    } else if (!sv.prep_appends && ht == XC + BC) {
      ring.dt[slot] = dt[slab];
    }
    return;
  }

  // flush (not expected): out of line, so that its registers do not weigh on the read path
  float scl[HR];
#pragma unroll
  for (int hh = 0; hh < HR; ++hh) scl[hh] = sv.scale[slab0 + hh];
  copy_read_flush<P, N, T, RC, HR>(sv, x, B, C, y, s_rc, scl, start, n, pl.w, s_red);
}

// ---------------------------------------------------------------------------------------
// replay_step_read_kernel: the FP32-checkpoint step when the host knows that no sequence
// flushes (the non-flush steps of a window). Such a step only reads, so its speed is the
// bytes an SM keeps in flight. A register tile holds 32 KB per CTA and the register file
// allows 4 such CTAs; loads into registers also pass through L1, which a shared-memory
// carveout shrinks. Here one thread brings the slab into shared memory with one bulk copy
// (neither registers nor L1 hold it in flight), the dot products stream from shared memory
// row by row, and the few registers left let kReadCtas CTAs share an SM.
// FL: the launch is for a step the host knows flushes every sequence. The records are then
// staged in shared memory past the slab while its copy lands, and the fold takes half of a
// warp's rows at a time from shared memory (48 registers: 5 CTAs per SM, against 4 with a
// register tile); the CTA also sends the slab of the CTA one wave later to L2. Without FL a
// flush plan (not expected) folds a quarter of the rows at a time from the records in global
// memory.
template <int N, bool FL>
constexpr int kReadCtas = N >= 256 ? (FL ? 2 : 3) : (FL ? 5 : 6);

// A non-flush plan reaching the flush kernel of a read-copy store (the host expected a flush):
// the output reads the copy, like every non-flush step of such a store. Out of line.
template <int P, int N, class T, int RC>
__device__ __noinline__ void read_copy_nonflush(const StoreView& sv, const T* __restrict__ x,
                                                const T* __restrict__ C, float* __restrict__ y, int b, int g,
                                                int h, int start, int n) {
  using TL = Tile<P, N>;
  constexpr int RPW = TL::RPW, E = TL::E, EPC = 16 / sizeof(T), XC = P / EPC;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slab = b * sv.H + h, cap = sv.cap, k = n + 1;
  const size_t xo = static_cast<size_t>(slab) * P;
  float hv[RPW][E];
  const float scale = RC == REPLAY_RC_FP8E4M3 || RC == REPLAY_RC_NVFP4 ? sv.scale[slab] : 1.f;
  load_tile_rc<P, N, RC>(sv.rc, slab, scale, warp, lane, hv, sv.bscale);
  float cv[E];
  load_cols<P, N>(C + (static_cast<size_t>(b) * sv.G + g) * N, lane, cv);
  const float* cf = sv.coef + static_cast<size_t>(slab) * (cap + 1);
  const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
  auto x_of = [&](int s) { return s < n ? ring.x + static_cast<size_t>(ring_slot(start, s, cap)) * P : x + xo; };
  float xr[RPW];
  record_terms<RPW, T>(x_of, cf, k, warp, lane, xr);
  const float sum = tile_rows_dot<P, N>(hv, cv, cf[cap], xr, lane);
  const int myrow = warp * RPW + transpose_index<RPW>(lane);
  if (transpose_leader<RPW>(lane)) y[xo + myrow] = fmaf(sv.D[h], to_f(x[xo + myrow]), sum);
  if (tid < XC)  // (B and dt: the prep appends them for read-copy stores)
    *reinterpret_cast<uint4*>(ring.x + static_cast<size_t>(ring_slot(start, n, cap)) * P + tid * EPC) =
        *reinterpret_cast<const uint4*>(x + xo + tid * EPC);
}

// RC (the launch is for a flush, FL): besides the FP32 checkpoint, the flush writes the read
// copy RC. bf16 and FP16 rows are cast as they are folded; an E4M3 or NVFP4 copy needs the
// slab's absmax first, so the folded rows go back into the shared slab and are encoded from
// there once the CTA has reduced it.
template <int P, int N, class T, bool FL, int RC = REPLAY_RC_NONE>
__global__ void __launch_bounds__(kThreads, kReadCtas<N, FL>)
replay_step_read_kernel(StoreView sv, const T* __restrict__ x, const T* __restrict__ B,
                        const T* __restrict__ C, const T* __restrict__ dt, float* __restrict__ y) {
  using TL = Tile<P, N>;
  constexpr int RPW = TL::RPW, E = TL::E, VEC = TL::VEC, NVEC = TL::NVEC, HR = FL ? RPW / 2 : RPW / 4;
  constexpr int EPC = 16 / sizeof(T), XC = P / EPC, BC = N / EPC;
  constexpr bool ENC = RC == REPLAY_RC_FP8E4M3 || RC == REPLAY_RC_NVFP4;  // encoded after an absmax
  static_assert(FL || RC == REPLAY_RC_NONE, "copies are written by the flush launch only");
  extern __shared__ float4 smem4[];
  __shared__ __align__(8) unsigned long long s_bar;
  __shared__ int s_landed;
  __shared__ float s_red[kWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y, b = blockIdx.z;
  const int h = g * sv.hpg + blockIdx.x;
  const int slab = b * sv.H + h;
  const int cap = sv.cap;
  const size_t xo = static_cast<size_t>(slab) * P;
  const size_t bo = (static_cast<size_t>(b) * sv.G + g) * N;
  float* s_h = reinterpret_cast<float*>(smem4);
  float* h0 = sv.h0 + static_cast<size_t>(slab) * P * N;
  if (tid == 0) {
    mbar_init(&s_bar);
    bulk_load(s_h, h0, P * N * sizeof(float), &s_bar);
  }
  if (FL) prefetch_next_wave<P, N, REPLAY_RC_NONE>(sv, slab, 1, kReadCtas<N, FL>, true);
  float cv[E];
  load_cols<P, N>(C + bo, lane, cv);
  const int myrow = warp * RPW + transpose_index<RPW>(lane);
  const float xk_row = to_f(x[xo + myrow]);
  const float Dh = sv.D[h];

  griddep_wait();  // plan and coefficients of this step are written
  const int4 pl = sv.plan[b];
  const int start = pl.x, n = pl.y, k = n + 1;
  const float* cf = sv.coef + static_cast<size_t>(slab) * (cap + 1);
  const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
  auto x_of = [&](int s) { return s < n ? ring.x + static_cast<size_t>(ring_slot(start, s, cap)) * P : x + xo; };
  auto b_of = [&](int s) { return s < n ? ring.b + static_cast<size_t>(ring_slot(start, s, cap)) * N : B + bo; };
  float* sm_u = s_h + P * N;     // FL: [k][P] w_s x_s, then [k][N] B_s
  float* sm_b = sm_u + cap * P;
  float xr[RPW];
  if (RC == REPLAY_RC_NONE && pl.z == kPlanNonFlush) record_terms<RPW, T>(x_of, cf, k, warp, lane, xr);
  if (FL && pl.z == kPlanFlush) stage_weighted<P, N, T>(x_of, b_of, cf, k, sm_u, sm_b);
  // The slab must have landed before it is read or the CTA exits; one thread waits, the rest
  // at the barrier (which also publishes a flush's staging). A copy past its limit leaves this
  // slab's y NaN and its state untouched (after a second bounded wait).
  if (tid == 0) {
    const bool ok = mbar_wait(&s_bar, 0, kCopyWaitNs);
    if (!ok) {
      set_status(sv.status, REPLAY_DEV_COPY_TIMEOUT);
      mbar_wait(&s_bar, 0, kCopyWaitNs);
    }
    s_landed = ok;
  }
  __syncthreads();
  if (!s_landed || pl.z == kPlanBad) {
    if (tid < P) y[xo + tid] = __int_as_float(0x7fc00000);
    return;
  }

  if (pl.z == kPlanNonFlush) {
    if constexpr (RC != REPLAY_RC_NONE) {
      read_copy_nonflush<P, N, T, RC>(sv, x, C, y, b, g, h, start, n);
      return;
    } else {
      const float sum = smem_rows_dot<P, N>(s_h, cv, cf[cap], xr, warp, lane);
      if (transpose_leader<RPW>(lane)) y[xo + myrow] = fmaf(Dh, xk_row, sum);
      const int slot = ring_slot(start, n, cap);
      if (tid < XC) {
        *reinterpret_cast<uint4*>(ring.x + static_cast<size_t>(slot) * P + tid * EPC) =
            *reinterpret_cast<const uint4*>(x + xo + tid * EPC);
      } else if (!sv.prep_appends && blockIdx.x == 0 && tid < XC + BC) {  // B once per group
        const int c = tid - XC;
        *reinterpret_cast<uint4*>(ring.b + static_cast<size_t>(slot) * N + c * EPC) =
            *reinterpret_cast<const uint4*>(B + bo + c * EPC);
      } else if (!sv.prep_appends && tid == XC + BC) {
        ring.dt[slot] = dt[slab];
      }
      return;
    }
  }

  // flush: h <- Gamma h + sum_s w_s x_s B_s^T, HR of the warp's rows at a time. The FP32-only
  // store reduces all of the warp's rows at the end (measured faster than a reduction per group
  // of HR rows, despite a few spilled bytes); the copy stores reduce each group as it is done.
  const float gam = cf[cap];
  float amax = 0.f;
  float partall[RPW];
#pragma unroll
  for (int hf = 0; hf < RPW / HR; ++hf) {
    const int r0 = warp * RPW + hf * HR;
    float hv[HR][E];
#pragma unroll
    for (int i = 0; i < HR; ++i)
#pragma unroll
      for (int v = 0; v < NVEC; ++v) {
        float t[VEC];
        ldv<VEC>(s_h + (r0 + i) * N + TL::col(lane, v), t);
#pragma unroll
        for (int e = 0; e < VEC; ++e) hv[i][v * VEC + e] = gam * t[e];
      }
    for (int s = 0; s < k; ++s) {
      float u[HR], bv[E];
      if constexpr (FL) {
        load_rows<HR>(sm_u + s * P + r0, u);
        load_cols<P, N>(sm_b + s * N, lane, bv);
      } else {
        load_cols<P, N>(b_of(s), lane, bv);
        const T* xs = x_of(s) + r0;
        const float w = cf[s];
#pragma unroll
        for (int i = 0; i < HR; ++i) u[i] = w * to_f(xs[i]);
      }
#pragma unroll
      for (int i = 0; i < HR; ++i)
#pragma unroll
        for (int e = 0; e < E; e += 2) {  // packed FP32 FMAs, two columns at a time
          const float2 r = __ffma2_rn(make_float2(u[i], u[i]), make_float2(bv[e], bv[e + 1]),
                                      make_float2(hv[i][e], hv[i][e + 1]));
          hv[i][e] = r.x;
          hv[i][e + 1] = r.y;
        }
    }
    float part[HR];
#pragma unroll
    for (int i = 0; i < HR; ++i) {
      float hc = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) hc = fmaf(hv[i][e], cv[e], hc);
      part[i] = hc;
#pragma unroll
      for (int v = 0; v < NVEC; ++v) {
        float t[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) t[e] = hv[i][v * VEC + e];
        stv_stream<VEC>(h0 + (r0 + i) * N + TL::col(lane, v), t);
      }
      if constexpr (RC == REPLAY_RC_BF16 || RC == REPLAY_RC_FP16) {
        store_row_rc<P, N, RC>(sv.rc, slab, 1.f, r0 + i, lane, hv[i]);
      } else if constexpr (ENC) {  // back into the slab, for the encoding below
#pragma unroll
        for (int v = 0; v < NVEC; ++v) {
          float t[VEC];
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            t[e] = hv[i][v * VEC + e];
            amax = fmaxf(amax, fabsf(t[e]));
          }
          *reinterpret_cast<float4*>(s_h + (r0 + i) * N + TL::col(lane, v)) = make_float4(t[0], t[1], t[2], t[3]);
        }
      }
    }
    if constexpr (RC == REPLAY_RC_NONE) {
#pragma unroll
      for (int i = 0; i < HR; ++i) partall[hf * HR + i] = part[i];
    } else {
      const float sum = warp_transpose_reduce<HR>(part, lane);
      if (transpose_leader<HR>(lane)) {
        const int row = r0 + transpose_index<HR>(lane);
        y[xo + row] = fmaf(Dh, to_f(x[xo + row]), sum);
      }
    }
  }
  if constexpr (RC == REPLAY_RC_NONE) {
    const float sum = warp_transpose_reduce<RPW>(partall, lane);
    if (transpose_leader<RPW>(lane)) y[xo + myrow] = fmaf(Dh, xk_row, sum);
  }
  if constexpr (ENC) {
    // the slab's absmax, its scale, then the codes of the warp's own rows from the slab
    amax = warp_max(amax);
    if (lane == 0) s_red[warp] = amax;
    __syncthreads();
    float m = s_red[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) m = fmaxf(m, s_red[w]);
    const float scale = RC == REPLAY_RC_FP8E4M3 ? (m > 0.f ? __fdiv_rn(m, kE4M3Max) : 1.f)
                                                : (m > 0.f ? __fdiv_rn(m, kE4M3Max * kE2M1Max) : 1.f);
    if (tid == 0) sv.scale[slab] = scale;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const int row = warp * RPW + i;
      float t[E];
#pragma unroll
      for (int v = 0; v < NVEC; ++v) {
        float w4[VEC];
        ldv<VEC>(s_h + row * N + TL::col(lane, v), w4);
#pragma unroll
        for (int e = 0; e < VEC; ++e) t[v * VEC + e] = w4[e];
      }
      if constexpr (RC == REPLAY_RC_FP8E4M3)
        store_row_rc<P, N, RC>(sv.rc, slab, scale, row, lane, t);
      else
        store_row_nvfp4<P, N>(sv.rc, sv.bscale, slab, scale, row, lane, t);
    }
  }
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
  griddep_launch_dependents();  // after the wait: the next step's prep may start
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
      record_terms<RPW, T>(x_of, cf, k, warp, lane, ex);
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
      // append this head's record at ring slot start + n (B and dt here unless the prep does)
      if (tid < XC) {
        *reinterpret_cast<uint4*>(ring.x + static_cast<size_t>(slot) * P + tid * EPC) =
            *reinterpret_cast<const uint4*>(x + xo + tid * EPC);
      } else if (!sv.prep_appends && blockIdx.x == 0 && hh == 0 && tid < XC + BC) {
        const int c = tid - XC;
        *reinterpret_cast<uint4*>(ring.b + static_cast<size_t>(slot) * N + c * EPC) =
            *reinterpret_cast<const uint4*>(B + bo + c * EPC);
      } else if (!sv.prep_appends && tid == XC + BC) {
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
      load_checkpoint<P, N>(sv, slab, warp, lane, hv);
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
// NVFP4 copy (dstate 128). A slab's copy is 4 KiB of codes and 512 B of block scales, so a CTA
// takes 8 heads of a group, one warp per head. h0 . C of a head is a 64 x 128 by 128 product,
// done on the tensor cores with mma.sync m16n8k16 (f16 inputs, FP32 accumulation): one MMA
// per (16-row tile, block), its k dimension one NVFP4 block. The codes become FP16 operands
// with integer ops only: slot A of a stored byte is already the high byte of the FP16 value *
// 2^-14, slot B takes two shifts, and a byte permute with zero places two codes in an FP16
// pair. C enters as the B operand split into an FP16 high and low part, after scaling the
// group's C by a power of two that brings its largest value to [2^13, 2^14): the products are
// exact in FP32 and C keeps about 22 bits. Block bk's MMA puts the two parts in columns
// 2 (bk mod 4) and 2 (bk mod 4) + 1, so each block's unscaled sum lands in a column pair of its
// own and the block scale weights it once per (row, block) afterwards (scaling every operand
// pair cost as many instructions as the decode). Lane (g, q) = (lane / 4, lane % 4) reads quarter q
// of rows g and g + 8 of every 16-row tile (one 16-byte load each) and holds the A fragment
// columns of that quarter; the MMA k index 2q, 2q+1, 2q+8, 2q+9 is block column 4q .. 4q+3.
// d += a b
__device__ __forceinline__ void mma_16816(float (&d)[4], unsigned a0, unsigned a1, unsigned a2, unsigned a3,
                                          unsigned b0, unsigned b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ unsigned prmt(unsigned a, unsigned b, unsigned sel) {
  unsigned d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// The high FP16 bytes of the four slot-A codes, and of the four slot-B codes, of a word.
__device__ __forceinline__ unsigned fp4_placed_a(unsigned w) { return w & 0x8E8E8E8Eu; }
__device__ __forceinline__ unsigned fp4_placed_b(unsigned w) {
  return ((w >> 3) & 0x0E0E0E0Eu) | ((w << 7) & 0x80808080u);
}
// FP16 pair (byte i, byte i + 1 of x as high bytes, zero low bytes)
template <int I>
__device__ __forceinline__ unsigned fp4_pair(unsigned x) {
  return prmt(x, 0u, 4u | (I << 4) | (4u << 8) | ((I + 1) << 12));
}
// Dynamic shared memory of the NVFP4 kernel: per warp (head) its codes and block scales,
// staged by cp.async before the prep wait, then its k records (x) staged after it.
template <int P, int N, class T>
constexpr size_t fp4_stage_bytes(int heads, int cap) {
  return static_cast<size_t>(heads) * (P * N / 2 + P * N / kFp4Block) +
         static_cast<size_t>(heads) * cap * P * sizeof(T);
}

template <int P, int N, class T, int HPC>
__global__ void __launch_bounds__(kThreads, 4)
replay_step_fp4_kernel(StoreView sv, const T* __restrict__ x, const T* __restrict__ B,
                       const T* __restrict__ C, const T* __restrict__ dt, float* __restrict__ y) {
  static_assert(P == 64 && N == 128 && HPC == kWarps && 2 * N == kThreads, "one warp per head, 64 x 128 slabs");
  using TL = Tile<P, N>;
  constexpr int RPW = TL::RPW, E = TL::E;
  constexpr int EPC = 16 / sizeof(T), XC = P / EPC, BC = N / EPC;
  constexpr int NB = N / kFp4Block, MT = P / 16;  // blocks per row, 16-row tiles
  constexpr int CODE_BYTES = P * N / 2, SCALE_BYTES = P * NB;
  extern __shared__ float4 smem4[];
  __shared__ float s_red[kWarps];
  __shared__ float s_y[kWarps][P];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, q = lane & 3;
  const int g = blockIdx.y, b = blockIdx.z;
  const int hfirst = g * sv.hpg + blockIdx.x * HPC;
  const int slab0 = b * sv.H + hfirst;
  const int cap = sv.cap;
  const size_t bo = (static_cast<size_t>(b) * sv.G + g) * N;
  const int hw = hfirst + warp, slabw = slab0 + warp;  // this warp's head
  const size_t xow = static_cast<size_t>(slabw) * P;

  // Independent of the prep kernel: the head's codes and block scales into shared memory,
  // C, x for D x.
  uint8_t* s_codes = reinterpret_cast<uint8_t*>(smem4) + warp * (CODE_BYTES + SCALE_BYTES);
  uint8_t* s_scales = s_codes + CODE_BYTES;
  {
    const uint8_t* codes = static_cast<const uint8_t*>(sv.rc) + static_cast<size_t>(slabw) * CODE_BYTES;
    const uint8_t* scales = sv.bscale + static_cast<size_t>(slabw) * SCALE_BYTES;
#pragma unroll
    for (int c = lane; c < CODE_BYTES / 16; c += 32) cp_async16(s_codes + c * 16, codes + c * 16);
#pragma unroll
    for (int c = lane; c < SCALE_BYTES / 16; c += 32) cp_async16(s_scales + c * 16, scales + c * 16);
    cp_async_commit();
  }
  // The group's C scaled by 2^sc and split into FP16 high and low parts, once per CTA (two
  // threads per column), then each lane's B fragments (column gq: 0 = high, 1 = low, others
  // zero).
  __shared__ __half s_ch[2][N];
  __shared__ float s_cmax[kWarps];
  const int cc = tid & (N - 1);
  const float cval = to_f(C[bo + cc]);
  {
    const float m = warp_max(fabsf(cval));
    if (lane == 0) s_cmax[warp] = m;
  }
  __syncthreads();
  float cmax = s_cmax[0];
#pragma unroll
  for (int w = 1; w < N / 32; ++w) cmax = fmaxf(cmax, s_cmax[w]);
  const int ce = cmax > 0.f ? min(max(((__float_as_int(cmax) >> 23) & 0xff) - 127, -100), 100) : 0;
  const float up = __int_as_float((127 + 13 - ce) << 23);    // 2^sc: largest |C| in [2^13, 2^14)
  const float down = __int_as_float((127 + 1 + ce) << 23);   // 2^14 / 2^sc
  {
    const float cs = cval * up;
    const __half hi = __float2half_rn(cs);
    s_ch[tid / N][cc] = tid < N ? hi : __float2half_rn(cs - __half2float(hi));
  }
  __syncthreads();
  // B operand of block bk's MMA: C's high part in column 2 (bk mod 4), its low part in column
  // 2 (bk mod 4) + 1, zero elsewhere; lane (gq, q) holds column gq.
  unsigned bf[NB][2];
#pragma unroll
  for (int bk = 0; bk < NB; ++bk)
#pragma unroll
    for (int j = 0; j < 2; ++j)
      bf[bk][j] = (gq >> 1) == (bk & 3)
                      ? *reinterpret_cast<const unsigned*>(&s_ch[gq & 1][bk * kFp4Block + 4 * q + 2 * j])
                      : 0u;
  const float xk0 = to_f(x[xow + lane]), xk1 = to_f(x[xow + lane + 32]);

  griddep_wait();  // plan and coefficients of this step are written
  griddep_launch_dependents();  // after the wait: the next step's prep may start
  const int4 pl = sv.plan[b];
  const int start = pl.x, n = pl.y;
  if (pl.z == kPlanBad) {
    if (tid < P)
      for (int hh = 0; hh < HPC; ++hh) y[static_cast<size_t>(slab0 + hh) * P + tid] = __int_as_float(0x7fc00000);
    return;
  }
  const int k = n + 1;

  if (pl.z == kPlanNonFlush) {
    // Stage this head's k records (x) in shared memory by cp.async, and the coefficients in
    // registers (lane s holds c_s and c_{s+32}); the MMAs below hide their latency.
    const float* cf = sv.coef + static_cast<size_t>(slabw) * (cap + 1);
    const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, hw, g);
    T* sx = reinterpret_cast<T*>(reinterpret_cast<uint8_t*>(smem4) + HPC * (CODE_BYTES + SCALE_BYTES)) +
            static_cast<size_t>(warp) * cap * P;
    for (int c = lane; c < k * XC; c += 32) {
      const int s = c / XC, off = (c - s * XC) * EPC;
      const T* src = s < n ? ring.x + static_cast<size_t>(ring_slot(start, s, cap)) * P : x + xow;
      cp_async16(sx + s * P + off, src + off);
    }
    cp_async_commit();
    const float c_lo = lane < k ? cf[lane] : 0.f;
    const float c_hi = lane + 32 < k ? cf[lane + 32] : 0.f;
    const float gsc = cf[cap] * sv.scale[slabw] * down;
    cp_async_wait_group<1>();  // the codes and scales (the records may still be in flight)
    __syncwarp();
    // h0 . C: each block's MMA takes its codes unscaled (FP16 pairs placed by integer ops) and
    // writes its sum over the block's 16 columns into columns 2 (bk mod 4) and 2 (bk mod 4) + 1
    // (C high, low) of accumulator bk / 4; the block scales then weight the 8 block sums of a row
    // once each. Rows gq and gq + 8 of each tile end up in the lanes with q == 0.
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int r0 = mt * 16 + gq;
      const uint4 W0 = *reinterpret_cast<const uint4*>(s_codes + fp4_unit(r0, 0, q));
      const uint4 W1 = *reinterpret_cast<const uint4*>(s_codes + fp4_unit(r0 + 8, 0, q));
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int wd = 0; wd < 4; ++wd) {  // word wd holds blocks 2 wd and 2 wd + 1
        const unsigned w0 = wd == 0 ? W0.x : wd == 1 ? W0.y : wd == 2 ? W0.z : W0.w;
        const unsigned w1 = wd == 0 ? W1.x : wd == 1 ? W1.y : wd == 2 ? W1.z : W1.w;
        const unsigned a0 = fp4_placed_a(w0), b0 = fp4_placed_b(w0);
        const unsigned a1 = fp4_placed_a(w1), b1 = fp4_placed_b(w1);
        mma_16816(acc[wd >> 1], fp4_pair<0>(a0), fp4_pair<0>(a1), fp4_pair<0>(b0), fp4_pair<0>(b1), bf[2 * wd][0],
                  bf[2 * wd][1]);
        mma_16816(acc[wd >> 1], fp4_pair<2>(a0), fp4_pair<2>(a1), fp4_pair<2>(b0), fp4_pair<2>(b1),
                  bf[2 * wd + 1][0], bf[2 * wd + 1][1]);
      }
      // lane (gq, q): blocks q and q + 4 of rows gq and gq + 8, high plus low part
      const float za0 = acc[0][0] + acc[0][1], za1 = acc[1][0] + acc[1][1];
      const float zb0 = acc[0][2] + acc[0][3], zb1 = acc[1][2] + acc[1][3];
      // their block scales (E4M3 bytes q and q + 4 of the rows' scale words), as FP32
      const uint2 S0 = *reinterpret_cast<const uint2*>(s_scales + r0 * NB);
      const uint2 S1 = *reinterpret_cast<const uint2*>(s_scales + (r0 + 8) * NB);
      const float2 sa = e4m3x2_to_float2(static_cast<unsigned short>(prmt(S0.x, S0.y, q | ((q + 4) << 4))));
      const float2 sb = e4m3x2_to_float2(static_cast<unsigned short>(prmt(S1.x, S1.y, q | ((q + 4) << 4))));
      float ta = fmaf(za1, sa.y, za0 * sa.x), tb = fmaf(zb1, sb.y, zb0 * sb.x);
      ta += __shfl_xor_sync(kFull, ta, 1);
      tb += __shfl_xor_sync(kFull, tb, 1);
      ta += __shfl_xor_sync(kFull, ta, 2);
      tb += __shfl_xor_sync(kFull, tb, 2);
      if (q == 0) {
        s_y[warp][mt * 16 + gq] = ta;
        s_y[warp][mt * 16 + gq + 8] = tb;
      }
    }
    cp_async_wait_all();
    __syncwarp();
    // records: lane holds rows lane and lane + 32
    float ex0 = 0.f, ex1 = 0.f;
    for (int s = 0; s < k; ++s) {
      const float c = __shfl_sync(kFull, s < 32 ? c_lo : c_hi, s & 31);
      ex0 = fmaf(c, to_f(sx[s * P + lane]), ex0);
      ex1 = fmaf(c, to_f(sx[s * P + lane + 32]), ex1);
    }
    const float Dh = sv.D[hw];
    y[xow + lane] = fmaf(Dh, xk0, fmaf(gsc, s_y[warp][lane], ex0));
    y[xow + lane + 32] = fmaf(Dh, xk1, fmaf(gsc, s_y[warp][lane + 32], ex1));
    // append this head's record at ring slot start + n (B and dt here unless the prep does)
    const int slot = ring_slot(start, n, cap);
    if (lane < XC)
      *reinterpret_cast<uint4*>(ring.x + static_cast<size_t>(slot) * P + lane * EPC) =
          *reinterpret_cast<const uint4*>(x + xow + lane * EPC);
    if (!sv.prep_appends) {
      if (lane == 31) ring.dt[slot] = dt[slabw];
      if (blockIdx.x == 0 && warp == 0)
        for (int c = lane; c < BC; c += 32)
          *reinterpret_cast<uint4*>(ring.b + static_cast<size_t>(slot) * N + c * EPC) =
              *reinterpret_cast<const uint4*>(B + bo + c * EPC);
    }
    return;
  }

  // ---------------- flush, head by head, the whole CTA on each
  cp_async_wait_all();  // the staged codes share the shared memory the fold stages into
  __syncthreads();
  float cv[E];
  load_cols<P, N>(C + bo, lane, cv);
  const int myrow = warp * RPW + transpose_index<RPW>(lane);
  float* sm_u = reinterpret_cast<float*>(smem4);
  float* sm_b = sm_u + cap * P;
  for (int hh = 0; hh < HPC; ++hh) {
    const int h = hfirst + hh, slab = slab0 + hh;
    const size_t xo = static_cast<size_t>(slab) * P;
    const float* cf = sv.coef + static_cast<size_t>(slab) * (cap + 1);
    const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
    float hv[RPW][E];
    if (sv.shared)
      load_tile_rc<P, N, REPLAY_RC_NVFP4>(sv.rc, slab, sv.scale[slab], warp, lane, hv, sv.bscale);
    else
      load_checkpoint<P, N>(sv, slab, warp, lane, hv);
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
    write_checkpoint<P, N, REPLAY_RC_NVFP4>(sv, slab, s_red, hv, pl.w);
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
    const float scale = RC == REPLAY_RC_FP8E4M3 || RC == REPLAY_RC_NVFP4 ? sv.scale[slab] : 1.f;
    load_tile_rc<P, N, RC>(sv.rc, slab, scale, warp, lane, hv, sv.bscale);
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
      if (!sv.shared) load_checkpoint<P, N>(sv, slab, warp, lane, hv);
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


// Launch a per-head kernel as a programmatic dependent of the prep kernel before it.
template <class... KArgs, class... Args>
static int launch_ex(void (*kern)(KArgs...), dim3 grid, int block, size_t smem, cudaStream_t stream,
                     bool programmatic, Args... args) {
  if (smem > kSmemNoOptIn &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess)
    return REPLAY_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? REPLAY_OK : REPLAY_ECUDA;
}
template <class... KArgs, class... Args>
static int pdl_launch(void (*kern)(KArgs...), dim3 grid, size_t smem, cudaStream_t stream, Args... args) {
  return launch_ex(kern, grid, kThreads, smem, stream, true, args...);
}

// all_n: the ring count every sequence holds before this step when the host knows it (-1
// otherwise). It only picks kernels: every kernel handles any mix of flush and non-flush
// sequences. A step the host knows flushes every sequence takes the one-head-per-CTA kernel
// (more slabs in flight for the FP32 read and write); otherwise a read copy takes the
// several-heads-per-CTA kernels built for the small copy reads.
template <int P, int N, class T, int RC>
static int launch(const StoreView& base, int all_n, int parity, int overlap, const void* x, const void* B,
                  const void* C, const void* dt, float* y, cudaStream_t stream) {
  const T *tx = static_cast<const T*>(x), *tB = static_cast<const T*>(B), *tC = static_cast<const T*>(C),
          *tdt = static_cast<const T*>(dt);
  if (!step_runs_prep(base)) {
    auto fused = replay_step_fused_kernel<P, N, T, RC>;
    const size_t fsmem = smem_plan_bytes<P, N>(whole_image_bytes<P, N, T>(base.cap), base.cap);
    if (fsmem > kSmemNoOptIn &&
        cudaFuncSetAttribute(fused, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(fsmem)) !=
            cudaSuccess)
      return REPLAY_ECUDA;
    fused<<<dim3(base.hpg, base.G, base.batch), kThreads, fsmem, stream>>>(base, tx, tB, tC, tdt, y);
    return cudaGetLastError() == cudaSuccess ? REPLAY_OK : REPLAY_ECUDA;
  }
  StoreView sv = base;  // this step's plan and coefficient buffer (consecutive steps alternate)
  sv.plan += static_cast<size_t>(parity) * sv.batch;
  sv.coef += static_cast<size_t>(parity) * sv.batch * sv.H * (sv.cap + 1);
  // With overlap the prep is a programmatic dependent of the previous step's per-head kernel:
  // it starts as that kernel's CTAs retire and waits for it only before it completes.
  const size_t psmem = static_cast<size_t>(sv.cap + 1) * N * sizeof(T);
  const int prc = launch_ex(replay_step_prep_kernel<P, N, T>, dim3(sv.G, sv.batch), kPrepThreads, psmem, stream,
                            overlap != 0, sv, tB, tC, tdt, overlap);
  if (prc != REPLAY_OK) return prc;
  const size_t smem = fold_staging_bytes<P, N>(sv.cap);
  const bool all_flush = all_n >= 0 && all_n + 1 >= sv.L;
  if constexpr (RC == REPLAY_RC_NVFP4 && N == 128) {
    constexpr int HPC = 8;
    const size_t fsmem = std::max(smem, fp4_stage_bytes<P, N, T>(HPC, sv.cap));
    if (!all_flush && sv.hpg % HPC == 0) {
      // 4 CTAs of 52 KB share an SM only with the largest shared-memory carveout (a preference:
      // set on the current device before every launch, like the dynamic shared-memory size)
      if (cudaFuncSetAttribute(replay_step_fp4_kernel<P, N, T, HPC>, cudaFuncAttributePreferredSharedMemoryCarveout,
                               100) != cudaSuccess)
        return REPLAY_ECUDA;
      return pdl_launch(replay_step_fp4_kernel<P, N, T, HPC>, dim3(sv.hpg / HPC, sv.G, sv.batch), fsmem, stream,
                        sv, tx, tB, tC, tdt, y);
    }
  }
  if constexpr (RC != REPLAY_RC_NONE && N == 128) {  // a known flush of a copy store: bulk-copy flush kernel
    const size_t flsmem = static_cast<size_t>(P) * N * sizeof(float) + smem;
    // (a shared checkpoint, or an FP16 one, measured faster in the register-tile kernel below:
    // there the slab read is the small copy, or the stochastic rounding dominates)
    if (all_flush && !sv.shared && !sv.ckpt16)
      return pdl_launch(replay_step_read_kernel<P, N, T, true, RC>, dim3(sv.hpg, sv.G, sv.batch), flsmem,
                        stream, sv, tx, tB, tC, tdt, y);
  }
  if constexpr (RC == REPLAY_RC_FP8E4M3 && P == 64 && N == 128) {
    constexpr int HR = 4;
    if (all_n >= 0 && !all_flush && sv.hpg % HR == 0) {
      if (cudaFuncSetAttribute(replay_step_e4m3_mma_kernel<P, N, T, HR>,
                               cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
        return REPLAY_ECUDA;
      return pdl_launch(replay_step_e4m3_mma_kernel<P, N, T, HR>, dim3(sv.hpg / HR, sv.G, sv.batch),
                        e4m3_mma_smem<P, N, T, HR>(sv.cap), stream, sv, tx, tB, tC, tdt, y);
    }
  }
  if constexpr (RC != REPLAY_RC_NONE && RC != REPLAY_RC_NVFP4) {
    constexpr int HPC = heads_per_cta<N, RC>();
    // the bulk-copy kernel takes at most 2 heads of E4M3 at dstate 128 (16 KB): 6 CTAs per SM
    // beat 4 with 4 heads each (measured)
    constexpr int HR = RC == REPLAY_RC_FP8E4M3 && HPC == 4 && N == 128 ? 2 : HPC;
    constexpr size_t kCopyBytes = static_cast<size_t>(HR) * P * N * (RC == REPLAY_RC_FP8E4M3 ? 1 : 2);
    if (all_n >= 0 && !all_flush && HR > 1 && sv.hpg % HR == 0)
      return pdl_launch(replay_step_copy_read_kernel<P, N, T, RC, HR>, dim3(sv.hpg / HR, sv.G, sv.batch),
                        kCopyBytes, stream, sv, tx, tB, tC, tdt, y);
    if (!all_flush && HPC > 1 && sv.hpg % HPC == 0)
      return pdl_launch(replay_step_copy_kernel<P, N, T, RC, HPC>, dim3(sv.hpg / HPC, sv.G, sv.batch), smem,
                        stream, sv, tx, tB, tC, tdt, y);
  }
  if constexpr (RC == REPLAY_RC_NONE) {
    const size_t slab_bytes = static_cast<size_t>(P) * N * sizeof(float);
    if (all_flush)
      return pdl_launch(replay_step_read_kernel<P, N, T, true>, dim3(sv.hpg, sv.G, sv.batch), slab_bytes + smem,
                        stream, sv, tx, tB, tC, tdt, y);
    if (all_n >= 0)
      return pdl_launch(replay_step_read_kernel<P, N, T, false>, dim3(sv.hpg, sv.G, sv.batch), slab_bytes, stream,
                        sv, tx, tB, tC, tdt, y);
  }
  return pdl_launch(replay_step_kernel<P, N, T, RC>, dim3(sv.hpg, sv.G, sv.batch), smem, stream, sv, tx, tB, tC,
                    tdt, y, all_flush ? 1 : 0);
}

int launch_step(const StoreView& sv, const Shape& sh, int all_n, int parity, int overlap, const void* x,
                const void* B, const void* C, const void* dt, float* y, cudaStream_t stream) {
#define RSSM_STEP(NN, TT, RCC)                                                  \
  if (sh.N == NN && sh.in_dtype == RSSM_DTYPE_OF(TT) && sh.read_copy == RCC)    \
    return launch<64, NN, TT, RCC>(sv, all_n, parity, overlap, x, B, C, dt, y, stream);
  RSSM_FOR_EACH_CONFIG(RSSM_STEP)
#undef RSSM_STEP
  return REPLAY_EUNSUPPORTED;
}

}  // namespace rssm
