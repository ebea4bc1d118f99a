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
// Two kernels, as for the decode step.
//  1. replay_verify_prep_kernel, one CTA per (sequence, group): reads the ring pointer,
//     records the call's plan, publishes the next pointer (drafts pending beyond it),
//     computes the B_s . C_j dots of the group once (s <= n + j: the committed records and
//     the drafts up to j), and per head the fold weights of the committed records (when
//     n >= L they are folded first) and the query coefficients
//        c_j[s] = exp(A sum_{r=s+1..n+j} dt_r) dt_s (B_s . C_j),  Gamma_j = exp(A sum_{r<=n+j} dt_r).
//  2. replay_verify_kernel, one CTA per (sequence, head) slab, a programmatic dependent of
//     the prep: the checkpoint tile is loaded first; a pre-fold, when planned, stages and
//     folds the committed records and writes the checkpoint; then for each draft j one warp
//     reduction sums Gamma_j h0 . C_j and sum_s c_j[s] x_s (lane s carries record s). The
//     drafts' records are appended beyond the committed ones.
#include "launch.h"
#include "replay_core.cuh"

namespace rssm {

constexpr int kMaxDrafts = 8;
constexpr int kVerifyBad = -1, kVerifyPlain = 0, kVerifyPrefold = 1;
// FP32 checkpoint, dstate 128: the tensor-core kernel handles drafts in groups of 4 (its MMA
// tiles have room for 4 drafts' C split in two), so it pays for whole groups; it takes the calls
// whose draft count fills them (measured at batch 512, 8 heads: T = 4 60.8 vs 64.4 us, T = 8
// 93.2 vs 95.1 us for the packed-FMA kernel), the packed-FMA kernel every other count (T = 1
// 44.6 vs 51.8 us, T = 3 57.6 vs 58.3, T = 6 79.6 vs 83.8).
inline bool verify_takes_tc(int TT) { return TT % 4 == 0; }

// The prep's CTA size: 256 threads when the whole prep grid fits on the GPU at once with room
// to spare (its serial per-head work then spreads over 8 warps), else 128 so that every prep
// CTA is resident before the dependent per-head kernel needs them (as for the step's prep).
constexpr long long kPrepWideMaxThreads = 152LL * 1024;

template <int P, int N, class T, int kPrepThreads>
__global__ void __launch_bounds__(kPrepThreads)
replay_verify_prep_kernel(StoreView sv, int TT, const T* __restrict__ B, const T* __restrict__ C,
                          const T* __restrict__ dt) {
  constexpr int EPC = 16 / sizeof(T), BC = N / EPC;
  __shared__ int4 s_meta;
  __shared__ float s_bc[kMaxDrafts][kMaxCap];
  __shared__ float s_dt[kDtStage];
  extern __shared__ float4 smem4[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x, b = blockIdx.y;
  const int H = sv.H, G = sv.G, cap = sv.cap, hpg = sv.hpg;
  griddep_launch_dependents();  // the head CTAs may start their checkpoint loads now

  // One round trip for everything, the ring pointer included: the group's whole B ring by slot
  // (the committed records are among its slots wherever the pointer is), the drafts' B and C,
  // and every head's dt ring by slot beside the drafts' dt.
  T* sring = reinterpret_cast<T*>(smem4);  // [cap][N] the B ring, by slot
  T* sdb = sring + static_cast<size_t>(cap) * N;  // [TT][N] the drafts' B
  T* sdc = sdb + static_cast<size_t>(TT) * N;     // [TT][N] the drafts' C
  const T* bring = static_cast<const T*>(sv.bbuf) + (static_cast<size_t>(b) * G + g) * cap * N;
  if (tid == 0) s_meta = sv.meta[b];
  for (int c = tid; c < (cap + 2 * TT) * BC; c += kPrepThreads) {
    const int r = c / BC, off = (c - r * BC) * EPC;
    const T* src;
    if (r < cap) {
      src = bring + static_cast<size_t>(r) * N;
    } else {
      const int j = r < cap + TT ? r - cap : r - cap - TT;
      src = (r < cap + TT ? B : C) + (static_cast<size_t>(b) * TT + j) * G * N + static_cast<size_t>(g) * N;
    }
    cp_async16(sring + static_cast<size_t>(r) * N + off, src + off);
  }
  cp_async_commit();
  // s_dt: [hpg][cap] the heads' dt rings by slot, then [hpg][TT] the drafts' dt
  const bool stage_dt = hpg * (cap + TT) <= kDtStage;
  const T* dtring = static_cast<const T*>(sv.dtbuf) + (static_cast<size_t>(b) * H + g * hpg) * cap;
  if (stage_dt) {
    for (int i = tid; i < hpg * cap; i += kPrepThreads) s_dt[i] = to_f(dtring[i]);
    for (int i = tid; i < hpg * TT; i += kPrepThreads) {
      const int j = i / hpg, hh = i - j * hpg;
      s_dt[hpg * cap + hh * TT + j] = to_f(dt[(static_cast<size_t>(b) * TT + j) * H + g * hpg + hh]);
    }
  }
  __syncthreads();
  const int start = s_meta.x, n = s_meta.y, epoch = s_meta.w;
  if (n < 0 || start < 0 || start >= cap || n + TT > cap) {
    if (tid == 0) {
      if (g == 0) sv.plan[b] = make_int4(start, n, kVerifyBad, epoch);
      set_status(sv.status, REPLAY_DEV_BAD_META);
    }
    cp_async_wait_all();
    return;
  }
  const bool prefold = n >= sv.L;
  const int start2 = prefold ? ring_slot(start, n, cap) : start;
  const int n2 = prefold ? 0 : n;
  if (tid == 0) {
    if (g == 0) sv.plan[b] = make_int4(start, n, prefold ? kVerifyPrefold : kVerifyPlain, epoch);
    arrive_and_publish(sv, b, make_int4(start2, n2, TT, epoch + (prefold ? 1 : 0)), G);
  }
  const int kk = n2 + TT;  // committed records after any pre-fold, then the drafts
  const int nf = prefold ? n : 0;
  // dt of head hh's record i: the n pre-folded records from start, then the kk query records
  auto dt_rec = [&](int hh, int i) {
    const int s = i - nf;
    if (i < nf || s < n2) {
      const int slot = i < nf ? ring_slot(start, i, cap) : ring_slot(start2, s, cap);
      return stage_dt ? s_dt[hh * cap + slot] : to_f(dtring[hh * cap + slot]);
    }
    const int j = s - n2;
    return stage_dt ? s_dt[hpg * cap + hh * TT + j]
                    : to_f(dt[(static_cast<size_t>(b) * TT + j) * H + g * hpg + hh]);
  };
  cp_async_wait_all();
  __syncthreads();

  // B_s . C_j for s <= n2 + j, one thread each: a serial sum over the 16-byte chunks, each
  // thread starting at its own chunk so that a warp's loads fall in distinct banks
  for (int p = tid; p < TT * kk; p += kPrepThreads) {
    const int j = p / kk, s = p - j * kk;
    if (s > n2 + j) continue;
    const T* br = s < n2 ? sring + static_cast<size_t>(ring_slot(start2, s, cap)) * N
                         : sdb + static_cast<size_t>(s - n2) * N;
    const T* cr = sdc + static_cast<size_t>(j) * N;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int c = 0; c < BC; ++c) {
      const int off = ((c + tid) % BC) * EPC;
      float bv[EPC], cv[EPC];
      load16(br + off, bv);
      load16(cr + off, cv);
#pragma unroll
      for (int e = 0; e < EPC; ++e) acc[e & 3] = fmaf(bv[e], cv[e], acc[e & 3]);
    }
    s_bc[j][s] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
  }
  __syncthreads();

  // Per head (one warp each): the fold weights of pre-folded records, then the query
  // coefficients. With Q_i = sum_{r<i} dt_r over the kk query records (one warp scan), draft j
  // sees k = n2 + j + 1 records and c_j[s] = exp(A (Q_k - Q_{s+1})) dt_s (B_s . C_j),
  // Gamma_j = exp(A Q_k).
  const int cs = cap + 1;
  for (int hh = warp; hh < hpg; hh += kPrepThreads / 32) {
    const int h = g * hpg + hh;
    const size_t slab = static_cast<size_t>(b) * H + h;
    const float A = sv.A[h];
    float* cf = sv.coef + slab * (sv.tmax + 1) * cs;
    if (prefold) {
      auto dt_fold = [&](int s) { return dt_rec(hh, s); };
      write_fold_weights(dt_fold, n, A, cf, cap, lane);
    }
    const float d0 = lane < kk ? dt_rec(hh, nf + lane) : 0.f;
    const float d1 = lane + 32 < kk ? dt_rec(hh, nf + lane + 32) : 0.f;
    float q0 = d0, q1 = d1;  // inclusive prefix sums: Q_{lane+1}, Q_{lane+33}
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float u0 = __shfl_up_sync(kFull, q0, off), u1 = __shfl_up_sync(kFull, q1, off);
      if (lane >= off) { q0 += u0; q1 += u1; }
    }
    q1 += __shfl_sync(kFull, q0, 31);
    for (int j = 0; j < TT; ++j) {
      const int k = n2 + j + 1;
      const float qk = __shfl_sync(kFull, k <= 32 ? q0 : q1, (k - 1) & 31);
      float* cj = cf + (1 + j) * cs;
      if (lane < k) cj[lane] = __expf(A * (qk - q0)) * d0 * s_bc[j][lane];
      if (lane + 32 < k) cj[lane + 32] = __expf(A * (qk - q1)) * d1 * s_bc[j][lane + 32];
      if (lane == 0) cj[cap] = __expf(A * qk);
    }
  }
}

template <int P, int N, class T, int RC>
__global__ void __launch_bounds__(kThreads, kMinBlocks<N> == 4 ? 3 : 2)
replay_verify_kernel(StoreView sv, int TT, const T* __restrict__ x, const T* __restrict__ B,
                     const T* __restrict__ C, const T* __restrict__ dt, float* __restrict__ y) {
  using TL = Tile<P, N>;
  constexpr int RPW = TL::RPW, E = TL::E;
  constexpr int EPC = 16 / sizeof(T), XC = P / EPC, BC = N / EPC;
  extern __shared__ float4 smem4[];
  __shared__ float s_red[kWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = sv.H, G = sv.G, cap = sv.cap;
  const int g = blockIdx.y, b = blockIdx.z;
  const int h = g * sv.hpg + blockIdx.x;
  const int slab = b * H + h;
  // draft j of sequence b: x/y at ((b*TT + j)*H + h)*P, B/C at ((b*TT + j)*G + g)*N
  auto xoff = [&](int j) { return (static_cast<size_t>(b) * TT + j) * H * P + static_cast<size_t>(h) * P; };
  auto boff = [&](int j) { return (static_cast<size_t>(b) * TT + j) * G * N + static_cast<size_t>(g) * N; };

  float hv[RPW][E];
  if constexpr (RC == REPLAY_RC_NONE) {
    load_tile_f32<P, N>(sv.h0 + static_cast<size_t>(slab) * P * N, warp, lane, hv);
  } else {
    const float scale = RC == REPLAY_RC_FP8E4M3 || RC == REPLAY_RC_NVFP4 ? sv.scale[slab] : 1.f;
    load_tile_rc<P, N, RC>(sv.rc, slab, scale, warp, lane, hv, sv.bscale);
  }
  const int myrow = warp * RPW + transpose_index<RPW>(lane);
  const float Dh = sv.D[h];
  // the drafts' C (this group) and x (this head), staged while the prep kernel runs
  T* sq = reinterpret_cast<T*>(reinterpret_cast<char*>(smem4) + fold_staging_bytes<P, N>(cap));
  T* sx = sq + static_cast<size_t>(TT) * N;
  for (int c = tid; c < TT * (BC + XC); c += kThreads) {
    if (c < TT * BC) {
      const int j = c / BC, off = (c - j * BC) * EPC;
      cp_async16(sq + j * N + off, C + boff(j) + off);
    } else {
      const int c2 = c - TT * BC;
      const int j = c2 / XC, off = (c2 - j * XC) * EPC;
      cp_async16(sx + j * P + off, x + xoff(j) + off);
    }
  }

  griddep_wait();  // plan and coefficients of this call are written
  cp_async_wait_all();
  __syncthreads();
  const int4 pl = sv.plan[b];
  if (pl.z == kVerifyBad) {
    for (int j = 0; j < TT; ++j)
      if (tid < P) y[xoff(j) + tid] = __int_as_float(0x7fc00000);
    return;
  }
  const int start = pl.x, n = pl.y;
  const bool prefold = pl.z == kVerifyPrefold;
  const int start2 = prefold ? ring_slot(start, n, cap) : start;
  const int n2 = prefold ? 0 : n;
  const int cs = cap + 1;
  const float* cf = sv.coef + static_cast<size_t>(slab) * (sv.tmax + 1) * cs;
  const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);

  if (prefold) {  // a flush of the committed records, from the checkpoint
    if constexpr (RC != REPLAY_RC_NONE) {
      if (!sv.shared) load_checkpoint<P, N>(sv, slab, warp, lane, hv);
    }
    float* sm_u = reinterpret_cast<float*>(smem4);
    float* sm_b = sm_u + cap * P;
    auto xf = [&](int s) { return ring.x + static_cast<size_t>(ring_slot(start, s, cap)) * P; };
    auto bf = [&](int s) { return ring.b + static_cast<size_t>(ring_slot(start, s, cap)) * N; };
    stage_weighted<P, N, T>(xf, bf, cf, n, sm_u, sm_b);
    __syncthreads();
    fold_staged<P, N>(sm_u, sm_b, n, cf[cap], hv);
    write_checkpoint<P, N, RC>(sv, slab, s_red, hv, pl.w);
  }

  const int kk = n2 + TT;
  auto x_of = [&](int s) {
    return s < n2 ? ring.x + static_cast<size_t>(ring_slot(start2, s, cap)) * P : x + xoff(s - n2);
  };
  // the drafts' coefficients to shared memory in one round trip (not one per draft)
  float* s_cf = reinterpret_cast<float*>(sx + static_cast<size_t>(TT) * P);
  for (int i = tid; i < TT * cs; i += kThreads) s_cf[i] = cf[cs + i];
  float xr0[RPW], xr1[RPW];  // records lane and lane + 32: x values of this warp's rows
#pragma unroll
  for (int i = 0; i < RPW; ++i) xr0[i] = xr1[i] = 0.f;
  if (lane < kk) load_rows<RPW>(x_of(lane) + warp * RPW, xr0);
  if (lane + 32 < kk) load_rows<RPW>(x_of(lane + 32) + warp * RPW, xr1);
  __syncthreads();
  for (int j = 0; j < TT; ++j) {
    const int k = n2 + j + 1;  // records draft j sees, itself included
    const float* cj = s_cf + j * cs;
    const float c0 = lane < k ? cj[lane] : 0.f;
    const float c1 = lane + 32 < k ? cj[lane + 32] : 0.f;
    float ex[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) ex[i] = fmaf(c1, xr1[i], c0 * xr0[i]);
    float cq[E];
    load_cols<P, N>(sq + j * N, lane, cq);
    const float sum = tile_rows_dot<P, N>(hv, cq, cj[cap], ex, lane);
    if (transpose_leader<RPW>(lane)) y[xoff(j) + myrow] = fmaf(Dh, to_f(sx[j * P + myrow]), sum);
  }
  // the drafts' records go to the ring beyond the committed ones; the pointer stays
  for (int j = 0; j < TT; ++j) {
    const int slot = ring_slot(start2, n2 + j, cap);
    if (tid < XC) {
      *reinterpret_cast<uint4*>(ring.x + static_cast<size_t>(slot) * P + tid * EPC) =
          *reinterpret_cast<const uint4*>(x + xoff(j) + tid * EPC);
    } else if (blockIdx.x == 0 && tid < XC + BC) {
      const int c = tid - XC;
      *reinterpret_cast<uint4*>(ring.b + static_cast<size_t>(slot) * N + c * EPC) =
          *reinterpret_cast<const uint4*>(B + boff(j) + c * EPC);
    } else if (tid == XC + BC) {
      ring.dt[slot] = dt[(static_cast<size_t>(b) * TT + j) * H + h];
    }
  }
}

// ---------------------------------------------------------------------------------------
// FP32 checkpoint, dstate 128: the drafts' h0 . C_j on the tensor cores. h0 . [C_1 .. C_T] is
// a 64 x 128 by 128 x T product per head; on CUDA cores with one warp reduction per draft it
// made the kernel instruction-bound. Here each warp takes 8 rows of the slab and runs
// mma.sync m16n8k8 with TF32 inputs and FP32 accumulation (rows 8..15 of the MMA tile are
// zero padding). For FP32 accuracy both operands are split: h0 = hi + lo with hi the value
// with its low 13 bits cleared (exact in TF32) and lo the exact remainder, and likewise C;
// one MMA multiplies h0_hi and one h0_lo against B columns [C_hi of drafts 0..3 | C_lo of
// drafts 0..3], which covers all four products; hi and lo columns are summed after. Lane
// (g, q) = (lane / 4, lane % 4) holds row 8w + g, columns 16i + 4q .. 16i + 4q + 3 (i = 0..7),
// loaded with one 16-byte load per i (each load of the warp reads 8 rows x 64 contiguous
// bytes); the MMA k index q, q + 4 of k-tile 2i + h is column 16i + 4q + 2h, + 1. After the
// MMAs, lane (g, q) finishes draft 2 (q & 1) + (q >> 1) of row 8w + g: the record terms from
// records staged in shared memory, the decay, the skip term.
__device__ __forceinline__ void mma_tf32_1688(float (&d)[4], unsigned a0, unsigned a2, unsigned b0, unsigned b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
__device__ __forceinline__ unsigned tf32_hi(float v) { return __float_as_uint(v) & 0xFFFFE000u; }
__device__ __forceinline__ unsigned tf32_lo(float v) { return __float_as_uint(v - __uint_as_float(tf32_hi(v))); }

// Dynamic shared memory of the tensor-core verify kernel (bytes), in order: the fold staging
// of a pre-fold; the drafts' C and x; the drafts' coefficients; the B fragments (per group of
// 4 drafts: 16 k-tiles x 32 lanes x 2 words); each warp's 8 rows of the kk records' x.
template <int P, int N, class T>
constexpr size_t tc_verify_smem(int TT, int cap) {
  return fold_staging_bytes<P, N>(cap) + static_cast<size_t>(TT) * (P + N) * sizeof(T) +
         align128(static_cast<size_t>(TT) * (cap + 1) * sizeof(float)) +
         static_cast<size_t>((TT + 3) / 4) * 16 * 32 * 2 * sizeof(unsigned) +
         static_cast<size_t>(cap) * P * sizeof(T);
}

template <int P, int N, class T>
__global__ void __launch_bounds__(kThreads, 4)
replay_verify_tc_kernel(StoreView sv, int TT, const T* __restrict__ x, const T* __restrict__ B,
                        const T* __restrict__ C, const T* __restrict__ dt, float* __restrict__ y) {
  static_assert(P == 64 && N == 128, "rows 8 per warp, 8 x 16 columns per row");
  constexpr int EPC = 16 / sizeof(T), XC = P / EPC, BC = N / EPC;
  extern __shared__ float4 smem4[];
  __shared__ float s_red[kWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, q = lane & 3;
  const int H = sv.H, G = sv.G, cap = sv.cap;
  const int g = blockIdx.y, b = blockIdx.z;
  const int h = g * sv.hpg + blockIdx.x;
  const int slab = b * H + h;
  const int row = warp * 8 + gq;
  const T* xb = x + static_cast<size_t>(b) * TT * H * P + static_cast<size_t>(h) * P;  // draft j: + j H P
  const T* cb = C + static_cast<size_t>(b) * TT * G * N + static_cast<size_t>(g) * N;  // draft j: + j G N
  const T* bb = B + static_cast<size_t>(b) * TT * G * N + static_cast<size_t>(g) * N;
  float* yb = y + static_cast<size_t>(b) * TT * H * P + static_cast<size_t>(h) * P;

  // shared memory regions
  char* base = reinterpret_cast<char*>(smem4);
  T* sq = reinterpret_cast<T*>(base + fold_staging_bytes<P, N>(cap));  // [TT][N] drafts' C
  T* sx = sq + static_cast<size_t>(TT) * N;                                // [TT][P] drafts' x
  float* s_cf = reinterpret_cast<float*>(sx + static_cast<size_t>(TT) * P);
  unsigned* s_bf = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(s_cf) +
                                               align128(static_cast<size_t>(TT) * (cap + 1) * sizeof(float)));
  const int NG = (TT + 3) / 4;
  T* s_rec = reinterpret_cast<T*>(s_bf + NG * 16 * 32 * 2);  // [cap][P] this head's x ring, by slot

  // Independent of the prep kernel: the lane's 32 checkpoint values, the drafts' C and x in
  // shared memory, and each thread's share of the drafts' records to append (x of this
  // head, B of the group by the group's first head, dt) in registers.
  float a[8][4];
  {
    const float* hr = sv.h0 + static_cast<size_t>(slab) * P * N + static_cast<size_t>(row) * N + 4 * q;
#pragma unroll
    for (int i = 0; i < 8; ++i) ldv_stream<4>(hr + 16 * i, a[i]);
  }
  for (int c = tid; c < TT * (BC + XC); c += kThreads) {
    if (c < TT * BC) {
      const int j = c / BC, off = (c - j * BC) * EPC;
      cp_async16(sq + j * N + off, cb + static_cast<size_t>(j) * G * N + off);
    } else {
      const int c2 = c - TT * BC;
      const int j = c2 / XC, off = (c2 - j * XC) * EPC;
      cp_async16(sx + j * P + off, xb + static_cast<size_t>(j) * H * P + off);
    }
  }
  cp_async_commit();
  // This head's whole x ring, by slot: its committed records are among them whatever the
  // ring pointer turns out to be, and the prep does not write them, so the copy need not wait
  // for the plan (the slots past the committed records are copied for nothing).
  const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
  for (int c = tid; c < cap * XC; c += kThreads) cp_async16(s_rec + c * EPC, ring.x + c * EPC);
  cp_async_commit();
  const int nxc = TT * XC, nbc = blockIdx.x == 0 ? TT * BC : 0, napp = nxc + nbc + TT;
  uint4 app[2];
  T appdt[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int c = tid + r * kThreads;
    if (c < nxc) {
      const int j = c / XC, off = (c - j * XC) * EPC;
      app[r] = *reinterpret_cast<const uint4*>(xb + static_cast<size_t>(j) * H * P + off);
    } else if (c < nxc + nbc) {
      const int c2 = c - nxc, j = c2 / BC, off = (c2 - j * BC) * EPC;
      app[r] = *reinterpret_cast<const uint4*>(bb + static_cast<size_t>(j) * G * N + off);
    } else if (c < napp) {
      appdt[r] = dt[(static_cast<size_t>(b) * TT + (c - nxc - nbc)) * H + h];
    }
  }
  const float Dh = sv.D[h];

  griddep_wait();  // plan and coefficients of this call are written
  // the plan and this thread's share of the drafts' coefficients in one round trip
  const int cs = cap + 1;
  const float* cf = sv.coef + static_cast<size_t>(slab) * (sv.tmax + 1) * cs;
  const float cfv = tid < TT * cs ? cf[cs + tid] : 0.f;
  const int4 pl = sv.plan[b];
  if (pl.z == kVerifyBad) {
    cp_async_wait_all();
    for (int j = 0; j < TT; ++j)
      if (tid < P) yb[static_cast<size_t>(j) * H * P + tid] = __int_as_float(0x7fc00000);
    return;
  }
  const int start = pl.x, n = pl.y;
  const bool prefold = pl.z == kVerifyPrefold;
  const int start2 = prefold ? ring_slot(start, n, cap) : start;
  const int n2 = prefold ? 0 : n;
  // the drafts' records go to the ring beyond the committed ones; the pointer stays
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int c = tid + r * kThreads;
    if (c < nxc) {
      const int j = c / XC, off = (c - j * XC) * EPC;
      *reinterpret_cast<uint4*>(ring.x + static_cast<size_t>(ring_slot(start2, n2 + j, cap)) * P + off) = app[r];
    } else if (c < nxc + nbc) {
      const int c2 = c - nxc, j = c2 / BC, off = (c2 - j * BC) * EPC;
      *reinterpret_cast<uint4*>(ring.b + static_cast<size_t>(ring_slot(start2, n2 + j, cap)) * N + off) = app[r];
    } else if (c < napp) {
      const int j = c - nxc - nbc;
      ring.dt[ring_slot(start2, n2 + j, cap)] = appdt[r];
    }
  }

  if (prefold) {  // a flush of the committed records, in the one-tile layout, then reload
    using TL = Tile<P, N>;
    float hv[TL::RPW][TL::E];
    load_tile_f32<P, N>(sv.h0 + static_cast<size_t>(slab) * P * N, warp, lane, hv);
    float* sm_u = reinterpret_cast<float*>(smem4);
    float* sm_b = sm_u + cap * P;
    auto xf = [&](int s) { return ring.x + static_cast<size_t>(ring_slot(start, s, cap)) * P; };
    auto bfn = [&](int s) { return ring.b + static_cast<size_t>(ring_slot(start, s, cap)) * N; };
    stage_weighted<P, N, T>(xf, bfn, cf, n, sm_u, sm_b);
    __syncthreads();
    fold_staged<P, N>(sm_u, sm_b, n, cf[cap], hv);
    write_checkpoint<P, N, REPLAY_RC_NONE>(sv, slab, s_red, hv, pl.w);
    __syncthreads();  // the new checkpoint is written (and visible to the block)
    const float* hr = sv.h0 + static_cast<size_t>(slab) * P * N + static_cast<size_t>(row) * N + 4 * q;
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // L2 reads: the block's own writes of the new checkpoint
      const float4 v = __ldcg(reinterpret_cast<const float4*>(hr + 16 * i));
      a[i][0] = v.x; a[i][1] = v.y; a[i][2] = v.z; a[i][3] = v.w;
    }
  }

  // coefficients and B fragments (the drafts' C, split) into shared memory
  if (tid < TT * cs) s_cf[tid] = cfv;
  for (int i = tid + kThreads; i < TT * cs; i += kThreads) s_cf[i] = cf[cs + i];
  cp_async_wait_group<1>();  // the drafts' C and x
  __syncthreads();
  for (int e = tid; e < NG * 16 * 32 * 2; e += kThreads) {
    const int r = e & 1, L = (e >> 1) & 31, kt = (e >> 6) & 15, set = e >> 10;
    const int gg = L >> 2, t = L & 3;
    const int j = 4 * set + (gg & 3);
    const int col = 16 * (kt >> 1) + 4 * t + 2 * (kt & 1) + r;
    const float c = j < TT ? to_f(sq[j * N + col]) : 0.f;
    s_bf[e] = (gg >> 2) ? tf32_lo(c) : tf32_hi(c);
  }
  cp_async_wait_all();  // the x ring
  __syncthreads();

  // d[set]: the MMA accumulators of drafts 4 set .. 4 set + 3
  float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  const uint2* bfr = reinterpret_cast<const uint2*>(s_bf) + lane;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const float v0 = a[i][2 * hh], v1 = a[i][2 * hh + 1];
      const unsigned h0 = tf32_hi(v0), h1 = tf32_hi(v1), l0 = tf32_lo(v0), l1 = tf32_lo(v1);
#pragma unroll
      for (int set = 0; set < 2; ++set) {
        if (set < NG) {
          const uint2 bb = bfr[(set * 16 + 2 * i + hh) * 32];
          mma_tf32_1688(d[set], h0, h1, bb.x, bb.y);
          mma_tf32_1688(d[set], l0, l1, bb.x, bb.y);
        }
      }
    }
  const int dsel = 2 * (q & 1) + (q >> 1);  // the draft (within a group of 4) this lane finishes
#pragma unroll
  for (int set = 0; set < 2; ++set) {
    if (set >= NG) break;
    // column 2q, 2q + 1 of row gq: q < 2 holds C_hi products of drafts 2q, 2q+1, q >= 2 the
    // C_lo products of drafts 2(q-2), 2(q-2)+1
    const float d0 = d[set][0] + __shfl_xor_sync(kFull, d[set][0], 2);
    const float d1 = d[set][1] + __shfl_xor_sync(kFull, d[set][1], 2);
    const int j = 4 * set + dsel;
    if (j < TT) {
      const float hc = (q >> 1) ? d1 : d0;
      const float* cj = s_cf + j * cs;
      float ex = 0.f;  // records draft j sees: the n2 committed ones, then drafts 0..j
      for (int s = 0; s < n2; ++s) ex = fmaf(cj[s], to_f(s_rec[ring_slot(start2, s, cap) * P + row]), ex);
      for (int s = 0; s <= j; ++s) ex = fmaf(cj[n2 + s], to_f(sx[s * P + row]), ex);
      yb[static_cast<size_t>(j) * H * P + row] = fmaf(Dh, to_f(sx[j * P + row]), fmaf(cj[cap], hc, ex));
    }
  }
}

// ---------------------------------------------------------------------------------------
// FP32 checkpoint, dstate 128: every head's T outputs from one register tile, with few
// instructions per value. Each warp takes 8 rows of the slab; lane (g, q) = (lane / 4, lane % 4)
// holds row 8w + g, columns 16i + 4q .. 16i + 4q + 3 (i = 0..7), loaded with one 16-byte load
// per i (each load of the warp reads 8 rows x 64 contiguous bytes). For draft j the lane forms
// its part of h0 . C_j with packed FP32 FMAs (C_j in shared memory in FP32, the same 16 bytes
// for the 8 lanes of a column quarter: one wavefront per load), scales it by Gamma_j, adds the
// record terms c_j[s] x_s[row] of records s = q, q + 4, ... (x staged in shared memory with
// rows padded to P + 8 values, so the 4 records a warp reads at once fall in distinct banks),
// and two shuffles sum the row's four lanes. A warp-uniform loop over drafts; no warp-wide
// reduction trees, no tensor-core operand splitting.
template <int P, int N, class T>
constexpr int kVerifyRecStride = P + 8;

// Dynamic shared memory of the FP32-checkpoint verify kernel (bytes), in order: the fold
// staging of a pre-fold; the drafts' C (input type); for bf16 inputs the same in FP32; the
// drafts' x; the drafts' coefficients; this head's x ring by slot (padded rows).
template <int P, int N, class T>
constexpr size_t ffma_verify_smem(int TT, int cap) {
  return fold_staging_bytes<P, N>(cap) + static_cast<size_t>(TT) * N * sizeof(T) +
         (sizeof(T) == 4 ? 0 : static_cast<size_t>(TT) * N * sizeof(float)) +
         static_cast<size_t>(TT) * kVerifyRecStride<P, N, T> * sizeof(T) +
         align128(static_cast<size_t>(TT) * (cap + 1) * sizeof(float)) +
         static_cast<size_t>(cap) * kVerifyRecStride<P, N, T> * sizeof(T);
}

template <int P, int N, class T>
__global__ void __launch_bounds__(kThreads, 4)
replay_verify_ffma_kernel(StoreView sv, int TT, const T* __restrict__ x, const T* __restrict__ B,
                          const T* __restrict__ C, const T* __restrict__ dt, float* __restrict__ y) {
  static_assert(P == 64 && N == 128, "rows 8 per warp, 8 x 16 columns per row");
  constexpr int EPC = 16 / sizeof(T), XC = P / EPC, BC = N / EPC, XS = kVerifyRecStride<P, N, T>;
  extern __shared__ float4 smem4[];
  __shared__ float s_red[kWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q = lane & 3;
  const int H = sv.H, G = sv.G, cap = sv.cap;
  const int g = blockIdx.y, b = blockIdx.z;
  const int h = g * sv.hpg + blockIdx.x;
  const int slab = b * H + h;
  const int row = warp * 8 + (lane >> 2);
  const T* xb = x + static_cast<size_t>(b) * TT * H * P + static_cast<size_t>(h) * P;  // draft j: + j H P
  const T* cb = C + static_cast<size_t>(b) * TT * G * N + static_cast<size_t>(g) * N;  // draft j: + j G N
  const T* bb = B + static_cast<size_t>(b) * TT * G * N + static_cast<size_t>(g) * N;
  float* yb = y + static_cast<size_t>(b) * TT * H * P + static_cast<size_t>(h) * P;

  // shared memory regions
  char* p0 = reinterpret_cast<char*>(smem4) + fold_staging_bytes<P, N>(cap);
  T* sq = reinterpret_cast<T*>(p0);  // [TT][N] drafts' C
  p0 += static_cast<size_t>(TT) * N * sizeof(T);
  float* sqf = reinterpret_cast<float*>(sq);  // [TT][N] drafts' C in FP32
  if constexpr (sizeof(T) != 4) {
    sqf = reinterpret_cast<float*>(p0);
    p0 += static_cast<size_t>(TT) * N * sizeof(float);
  }
  T* sx = reinterpret_cast<T*>(p0);  // [TT][XS] drafts' x
  p0 += static_cast<size_t>(TT) * XS * sizeof(T);
  float* s_cf = reinterpret_cast<float*>(p0);  // [TT][cap + 1] drafts' coefficients
  p0 += align128(static_cast<size_t>(TT) * (cap + 1) * sizeof(float));
  T* s_rec = reinterpret_cast<T*>(p0);  // [cap][XS] this head's x ring, by slot

  // Independent of the prep kernel: the lane's 32 checkpoint values, the drafts' C and x and
  // the x ring in shared memory, and each thread's share of the drafts' records to append (x
  // of this head, B of the group by the group's first head, dt) in registers.
  float a[8][4];
  {
    const float* hr = sv.h0 + static_cast<size_t>(slab) * P * N + static_cast<size_t>(row) * N + 4 * q;
#pragma unroll
    for (int i = 0; i < 8; ++i) ldv_stream<4>(hr + 16 * i, a[i]);
  }
  for (int c = tid; c < TT * (BC + XC); c += kThreads) {
    if (c < TT * BC) {
      const int j = c / BC, off = (c - j * BC) * EPC;
      cp_async16(sq + j * N + off, cb + static_cast<size_t>(j) * G * N + off);
    } else {
      const int c2 = c - TT * BC;
      const int j = c2 / XC, off = (c2 - j * XC) * EPC;
      cp_async16(sx + j * XS + off, xb + static_cast<size_t>(j) * H * P + off);
    }
  }
  // This head's whole x ring, by slot: its committed records are among them whatever the
  // ring pointer turns out to be, and the prep does not write them, so the copy need not wait
  // for the plan (the slots past the committed records are copied for nothing).
  const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
  for (int c = tid; c < cap * XC; c += kThreads) {
    const int slot = c / XC, off = (c - slot * XC) * EPC;
    cp_async16(s_rec + slot * XS + off, ring.x + c * EPC);
  }
  cp_async_commit();
  const int nxc = TT * XC, nbc = blockIdx.x == 0 ? TT * BC : 0, napp = nxc + nbc + TT;
  uint4 app[2];
  T appdt[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int c = tid + r * kThreads;
    if (c < nxc) {
      const int j = c / XC, off = (c - j * XC) * EPC;
      app[r] = *reinterpret_cast<const uint4*>(xb + static_cast<size_t>(j) * H * P + off);
    } else if (c < nxc + nbc) {
      const int c2 = c - nxc, j = c2 / BC, off = (c2 - j * BC) * EPC;
      app[r] = *reinterpret_cast<const uint4*>(bb + static_cast<size_t>(j) * G * N + off);
    } else if (c < napp) {
      appdt[r] = dt[(static_cast<size_t>(b) * TT + (c - nxc - nbc)) * H + h];
    }
  }
  const float Dh = sv.D[h];

  griddep_wait();  // plan and coefficients of this call are written
  // the plan and this thread's share of the drafts' coefficients in one round trip
  const int cs = cap + 1;
  const float* cf = sv.coef + static_cast<size_t>(slab) * (sv.tmax + 1) * cs;
  const float cfv = tid < TT * cs ? cf[cs + tid] : 0.f;
  const int4 pl = sv.plan[b];
  if (pl.z == kVerifyBad) {
    cp_async_wait_all();
    for (int j = 0; j < TT; ++j)
      if (tid < P) yb[static_cast<size_t>(j) * H * P + tid] = __int_as_float(0x7fc00000);
    return;
  }
  const int start = pl.x, n = pl.y;
  const bool prefold = pl.z == kVerifyPrefold;
  const int start2 = prefold ? ring_slot(start, n, cap) : start;
  const int n2 = prefold ? 0 : n;
  // the drafts' records go to the ring beyond the committed ones; the pointer stays
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int c = tid + r * kThreads;
    if (c < nxc) {
      const int j = c / XC, off = (c - j * XC) * EPC;
      *reinterpret_cast<uint4*>(ring.x + static_cast<size_t>(ring_slot(start2, n2 + j, cap)) * P + off) = app[r];
    } else if (c < nxc + nbc) {
      const int c2 = c - nxc, j = c2 / BC, off = (c2 - j * BC) * EPC;
      *reinterpret_cast<uint4*>(ring.b + static_cast<size_t>(ring_slot(start2, n2 + j, cap)) * N + off) = app[r];
    } else if (c < napp) {
      const int j = c - nxc - nbc;
      ring.dt[ring_slot(start2, n2 + j, cap)] = appdt[r];
    }
  }

  if (prefold) {  // a flush of the committed records, in the one-tile layout, then reload
    using TL = Tile<P, N>;
    float hv[TL::RPW][TL::E];
    load_tile_f32<P, N>(sv.h0 + static_cast<size_t>(slab) * P * N, warp, lane, hv);
    float* sm_u = reinterpret_cast<float*>(smem4);
    float* sm_b = sm_u + cap * P;
    auto xf = [&](int s) { return ring.x + static_cast<size_t>(ring_slot(start, s, cap)) * P; };
    auto bfn = [&](int s) { return ring.b + static_cast<size_t>(ring_slot(start, s, cap)) * N; };
    stage_weighted<P, N, T>(xf, bfn, cf, n, sm_u, sm_b);
    __syncthreads();
    fold_staged<P, N>(sm_u, sm_b, n, cf[cap], hv);
    write_checkpoint<P, N, REPLAY_RC_NONE>(sv, slab, s_red, hv, pl.w);
    __syncthreads();  // the new checkpoint is written (and visible to the block)
    const float* hr = sv.h0 + static_cast<size_t>(slab) * P * N + static_cast<size_t>(row) * N + 4 * q;
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // L2 reads: the block's own writes of the new checkpoint
      const float4 v = __ldcg(reinterpret_cast<const float4*>(hr + 16 * i));
      a[i][0] = v.x; a[i][1] = v.y; a[i][2] = v.z; a[i][3] = v.w;
    }
  }

  if (tid < TT * cs) s_cf[tid] = cfv;
  for (int i = tid + kThreads; i < TT * cs; i += kThreads) s_cf[i] = cf[cs + i];
  cp_async_wait_all();
  __syncthreads();
  if constexpr (sizeof(T) != 4) {
    for (int e = tid; e < TT * N; e += kThreads) sqf[e] = to_f(sq[e]);
    __syncthreads();
  }

  for (int j = 0; j < TT; ++j) {
    const float* cj = s_cf + j * cs;
    const float4* c4 = reinterpret_cast<const float4*>(sqf + j * N + 4 * q);
    float2 ha = make_float2(0.f, 0.f), hb = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 c = c4[4 * i];  // columns 16i + 4q .. 16i + 4q + 3 of C_j
      ha = __ffma2_rn(make_float2(a[i][0], a[i][1]), make_float2(c.x, c.y), ha);
      hb = __ffma2_rn(make_float2(a[i][2], a[i][3]), make_float2(c.z, c.w), hb);
    }
    float v = cj[cap] * ((ha.x + ha.y) + (hb.x + hb.y));
    const int k = n2 + j + 1;  // records draft j sees: the n2 committed ones, then drafts 0..j
    for (int s = q; s < k; s += 4) {
      const T xs = s < n2 ? s_rec[ring_slot(start2, s, cap) * XS + row] : sx[(s - n2) * XS + row];
      v = fmaf(cj[s], to_f(xs), v);
    }
    v += __shfl_xor_sync(kFull, v, 1);
    v += __shfl_xor_sync(kFull, v, 2);
    if (q == 0) yb[static_cast<size_t>(j) * H * P + row] = fmaf(Dh, to_f(sx[j * XS + row]), v);
  }
}

template <int P, int N, class T, int RC>
static int launch(const StoreView& sv, int TT, const void* x, const void* B, const void* C,
                  const void* dt, float* y, cudaStream_t stream) {
  const bool wide = static_cast<long long>(sv.G) * sv.batch * 256 <= kPrepWideMaxThreads;
  auto prep = wide ? replay_verify_prep_kernel<P, N, T, 256> : replay_verify_prep_kernel<P, N, T, 128>;
  const size_t psmem = static_cast<size_t>(sv.cap + 2 * TT) * N * sizeof(T);
  if (psmem > kSmemNoOptIn &&
      cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(psmem)) !=
          cudaSuccess)
    return REPLAY_ECUDA;
  prep<<<dim3(sv.G, sv.batch), wide ? 256 : 128, psmem, stream>>>(sv, TT, static_cast<const T*>(B),
                                                              static_cast<const T*>(C), static_cast<const T*>(dt));
  if (cudaGetLastError() != cudaSuccess) return REPLAY_ECUDA;
  auto kern = replay_verify_kernel<P, N, T, RC>;
  size_t smem = fold_staging_bytes<P, N>(sv.cap) + static_cast<size_t>(TT) * (P + N) * sizeof(T) +
                static_cast<size_t>(TT) * (sv.cap + 1) * sizeof(float);
  if constexpr (RC == REPLAY_RC_NONE && N == 128) {
    if (!verify_takes_tc(TT)) {
      kern = replay_verify_ffma_kernel<P, N, T>;
      smem = ffma_verify_smem<P, N, T>(TT, sv.cap);
    } else {
      kern = replay_verify_tc_kernel<P, N, T>;
      smem = tc_verify_smem<P, N, T>(TT, sv.cap);
    }
    // 4 CTAs per SM (up to 40 KB each at T = 8) need the largest shared-memory carveout
    if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
      return REPLAY_ECUDA;
  }
  if (smem > kSmemNoOptIn &&
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
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, sv, TT, static_cast<const T*>(x), static_cast<const T*>(B),
                                           static_cast<const T*>(C), static_cast<const T*>(dt), y);
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? REPLAY_OK : REPLAY_ECUDA;
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
