// Host-side launchers of the kernel translation units (one per family, so they compile in
// parallel). Each returns a REPLAY_* code; shapes and dtypes without a kernel give
// REPLAY_EUNSUPPORTED.
#pragma once

#include <cuda_runtime.h>

#include <type_traits>

#include "common.cuh"

namespace rssm {

struct Shape {
  int P, N, in_dtype, read_copy;
};

// Every (dstate, input type, read copy) combination with a kernel; headdim is 64. The FP16
// copy has kernels for dstate 64 and 128, the NVFP4 copy for dstate 128.
#define RSSM_FOR_EACH_CONFIG(X)                                                    \
  X(128, float, REPLAY_RC_NONE) X(128, float, REPLAY_RC_BF16) X(128, float, REPLAY_RC_FP8E4M3) \
  X(128, bf16, REPLAY_RC_NONE) X(128, bf16, REPLAY_RC_BF16) X(128, bf16, REPLAY_RC_FP8E4M3)   \
  X(64, float, REPLAY_RC_NONE) X(64, float, REPLAY_RC_BF16) X(64, float, REPLAY_RC_FP8E4M3)    \
  X(64, bf16, REPLAY_RC_NONE) X(64, bf16, REPLAY_RC_BF16) X(64, bf16, REPLAY_RC_FP8E4M3)      \
  X(256, float, REPLAY_RC_NONE) X(256, float, REPLAY_RC_BF16) X(256, float, REPLAY_RC_FP8E4M3) \
  X(256, bf16, REPLAY_RC_NONE) X(256, bf16, REPLAY_RC_BF16) X(256, bf16, REPLAY_RC_FP8E4M3)   \
  X(128, float, REPLAY_RC_FP16) X(128, bf16, REPLAY_RC_FP16) X(64, float, REPLAY_RC_FP16)      \
  X(64, bf16, REPLAY_RC_FP16) X(128, float, REPLAY_RC_NVFP4) X(128, bf16, REPLAY_RC_NVFP4)

#define RSSM_DTYPE_OF(TT) (std::is_same<TT, float>::value ? REPLAY_F32 : REPLAY_BF16)

// all_n: the ring count all sequences share before the step if the host knows it, else -1
// (a kernel-choice hint only).
// parity: which of the two plan and coefficient buffers this step uses (consecutive steps
// alternate). overlap: the previous call on the stream was a step known to flush no sequence
// that ran through the prep kernel; this step's prep may then start while that step's
// per-head kernel still runs.
int launch_step(const StoreView& sv, const Shape& sh, int all_n, int parity, int overlap, const void* x,
                const void* B, const void* C, const void* dt, float* y, cudaStream_t stream);

// Calls with at most this many (sequence, head) slabs take the fused step kernel (no prep).
constexpr long long kFusedMaxSlabs = 1024;
inline bool step_runs_prep(const StoreView& sv) { return static_cast<long long>(sv.batch) * sv.H > kFusedMaxSlabs; }
int launch_verify(const StoreView& sv, const Shape& sh, int T, const void* x, const void* B,
                  const void* C, const void* dt, float* y, cudaStream_t stream);
int launch_commit(const StoreView& sv, const int* accept, cudaStream_t stream);
// mode: 0 = flush committed records into h0 (+ read copy); 1 = export the folded state to out
int launch_fold(const StoreView& sv, const Shape& sh, int mode, float* out, cudaStream_t stream);
// h == nullptr loads zeros; mask (device, may be null) selects the sequences
int launch_load(const StoreView& sv, const Shape& sh, const float* h, const int* mask,
                cudaStream_t stream);

int launch_conv_step(const Shape& sh, int batch, int H, int G, void* state, int state_dtype,
                     const float* A, const float* D, const void* x, const void* B, const void* C,
                     const void* dt, float* y, cudaStream_t stream);
int launch_conv_verify(const Shape& sh, int batch, int H, int G, int T, float* snaps,
                       const int* cur, const float* A, const float* D, const void* x,
                       const void* B, const void* C, const void* dt, float* y,
                       cudaStream_t stream);
int launch_conv_commit(int batch, int T, int* cur, const int* accept, int* status,
                       cudaStream_t stream);

}  // namespace rssm
