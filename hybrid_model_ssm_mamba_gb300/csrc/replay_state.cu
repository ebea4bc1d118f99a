// replay_flush, replay_export_state, replay_load_state, replay_reset: moving whole states
// in and out of the checkpoint store.
//
// Source: "ReplaySSM: Rethinking State Storage for Faster Hybrid-Model Decoding" (NVIDIA
// Developer blog), sections "How ReplaySSM represents the state" (the state is the
// checkpoint with the buffered records folded in) and "Benefit 3" (every checkpoint write
// casts the FP32 values independently into the read copy).
#include "launch.h"
#include "replay_core.cuh"

namespace rssm {

// mode 0: fold the committed records into h0 and write it (flush); mode 1: write the folded
// state to `out` and leave the store unchanged (export).
template <int P, int N, class T, int RC, int MODE>
__global__ void __launch_bounds__(kThreads, kMinBlocks<N>)
replay_fold_kernel(StoreView sv, float* __restrict__ out) {
  using TL = Tile<P, N>;
  extern __shared__ float4 smem4[];
  __shared__ int4 s_meta;
  __shared__ float s_w[kMaxCap + 1];
  __shared__ float s_red[kWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y, b = blockIdx.z;
  const int h = g * sv.hpg + blockIdx.x;
  const int slab = b * sv.H + h;
  const int cap = sv.cap;

  if (tid == 0) s_meta = sv.meta[b];
  float hv[TL::RPW][TL::E];
  if (RC != REPLAY_RC_NONE && sv.shared) {  // the copy is the checkpoint
    const float scale = RC == REPLAY_RC_FP8E4M3 || RC == REPLAY_RC_NVFP4 ? sv.scale[slab] : 1.f;
    load_tile_rc<P, N, RC == REPLAY_RC_NONE ? REPLAY_RC_BF16 : RC>(sv.rc, slab, scale, warp, lane, hv, sv.bscale);
  } else {
    load_checkpoint<P, N>(sv, slab, warp, lane, hv);
  }
  __syncthreads();
  const int start = s_meta.x, n = s_meta.y;
  if (n < 0 || n > cap || start < 0 || start >= cap) {
    if (tid == 0) set_status(sv.status, REPLAY_DEV_BAD_META);
    if constexpr (MODE == 1) {
#pragma unroll
      for (int i = 0; i < TL::RPW; ++i)
#pragma unroll
        for (int e = 0; e < TL::E; ++e) hv[i][e] = __int_as_float(0x7fc00000);
      store_tile_f32<P, N>(out + static_cast<size_t>(slab) * P * N, warp, lane, hv);
    }
    return;
  }
  const SlabRing<T> ring = slab_ring<P, N, T>(sv, b, h, g);
  const RingImage<T> im = ring_image<P, N, T>(smem4, cap);
  const ExtraRecords<T> none{nullptr, nullptr, nullptr, 0, 0, 0};
  stage_records<P, N, T>(ring, im, start, cap, n, n, none);
  if constexpr (MODE == 0) {
    if (tid == 0) arrive_and_publish(sv, b, make_int4(ring_slot(start, n, cap), 0, 0, s_meta.w + (n > 0)), sv.H);
  }
  cp_async_wait_all();
  __syncthreads();
  if (n > 0) {
    auto slot_of = [&](int s) { return ring_slot(start, s, cap); };
    float* sm_u = fold_staging(smem4, ring_image_bytes<P, N, T>(cap));
    fold_tile<P, N, T>(im, slot_of, n, sv.A[h], sm_u, sm_u + cap * P, s_w, hv);
  }
  if constexpr (MODE == 1) {
    store_tile_f32<P, N>(out + static_cast<size_t>(slab) * P * N, warp, lane, hv);
  } else {
    if (n > 0) write_checkpoint<P, N, RC>(sv, slab, s_red, hv, s_meta.w);
  }
}

// Import h (or zeros) as the checkpoint of the selected sequences, recasting the read copy.
template <int P, int N, int RC>
__global__ void __launch_bounds__(kThreads, kMinBlocks<N>)
replay_load_kernel(StoreView sv, const float* __restrict__ h, const int* __restrict__ mask) {
  using TL = Tile<P, N>;
  __shared__ float s_red[kWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slab = blockIdx.x;
  const int b = slab / sv.H, hd = slab - b * sv.H;
  if (mask != nullptr && mask[b] == 0) return;
  float hv[TL::RPW][TL::E];
  if (h != nullptr) {
    load_tile_f32<P, N>(h + static_cast<size_t>(slab) * P * N, warp, lane, hv);
  } else {
#pragma unroll
    for (int i = 0; i < TL::RPW; ++i)
#pragma unroll
      for (int e = 0; e < TL::E; ++e) hv[i][e] = 0.f;
  }
  write_checkpoint<P, N, RC>(sv, slab, s_red, hv, 0);
  if (hd == 0 && tid == 0) {
    sv.meta[b] = make_int4(0, 0, 0, 1);
    sv.arrive[b] = 0;
  }
}

template <int P, int N, class T, int RC>
static int fold(const StoreView& sv, int mode, float* out, cudaStream_t stream) {
  const size_t smem = smem_plan_bytes<P, N>(ring_image_bytes<P, N, T>(sv.cap), sv.cap);
  auto kern = mode == 0 ? replay_fold_kernel<P, N, T, RC, 0> : replay_fold_kernel<P, N, T, RC, 1>;
  if (smem > kSmemNoOptIn &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess)
    return REPLAY_ECUDA;
  const dim3 grid(sv.hpg, sv.G, sv.batch);
  kern<<<grid, kThreads, smem, stream>>>(sv, out);
  return cudaGetLastError() == cudaSuccess ? REPLAY_OK : REPLAY_ECUDA;
}

int launch_fold(const StoreView& sv, const Shape& sh, int mode, float* out, cudaStream_t stream) {
#define RSSM_FOLD(NN, TT, RCC)                                                  \
  if (sh.N == NN && sh.in_dtype == RSSM_DTYPE_OF(TT) && sh.read_copy == RCC)    \
    return fold<64, NN, TT, RCC>(sv, mode, out, stream);
  RSSM_FOR_EACH_CONFIG(RSSM_FOLD)
#undef RSSM_FOLD
  return REPLAY_EUNSUPPORTED;
}

int launch_load(const StoreView& sv, const Shape& sh, const float* h, const int* mask,
                cudaStream_t stream) {
#define RSSM_LOAD(NN, RCC)                                                                   \
  if (sh.N == NN && sh.read_copy == RCC) {                                                   \
    replay_load_kernel<64, NN, RCC><<<sv.batch * sv.H, kThreads, 0, stream>>>(sv, h, mask);   \
    return cudaGetLastError() == cudaSuccess ? REPLAY_OK : REPLAY_ECUDA;                     \
  }
  RSSM_LOAD(64, REPLAY_RC_NONE) RSSM_LOAD(64, REPLAY_RC_BF16) RSSM_LOAD(64, REPLAY_RC_FP8E4M3)
  RSSM_LOAD(128, REPLAY_RC_NONE) RSSM_LOAD(128, REPLAY_RC_BF16) RSSM_LOAD(128, REPLAY_RC_FP8E4M3)
  RSSM_LOAD(256, REPLAY_RC_NONE) RSSM_LOAD(256, REPLAY_RC_BF16) RSSM_LOAD(256, REPLAY_RC_FP8E4M3)
  RSSM_LOAD(64, REPLAY_RC_FP16) RSSM_LOAD(128, REPLAY_RC_FP16)
  RSSM_LOAD(128, REPLAY_RC_NVFP4)
#undef RSSM_LOAD
  return REPLAY_EUNSUPPORTED;
}

}  // namespace rssm
