// replay_step_static_scratch: the decode step for callers that may not allocate device
// memory.
//
// Some callers cannot call cudaMalloc, or anything that allocates, at the point where they
// decode: an inference-engine plugin that is handed only its input, output and state
// buffers at enqueue time; a process whose device memory is owned up front by another
// framework's pool, so a stray allocation would fail or break its accounting; code that
// runs while a stream is being captured, where allocating is not allowed. They can still
// keep the store (its workspace is memory they were given), but they cannot provide extra
// memory for a kernel's scratch.
//
// replay_step's scratch is what it keeps only for the duration of one step: the
// per-sequence arrival counters (which must read zero when a step starts), the step's plan
// (the ring pointer it runs on) and the per-head record coefficients. Here all three live
// in one fixed array inside the library instead of the store's arrive, plan and coef
// regions: a file-scope device array that every GPU loading the library holds until the
// process exits. The kernels and everything else are replay_step's own.
#include <cstdint>
#include <mutex>

#include "launch.h"
#include "store.h"

namespace {

constexpr size_t kArriveBytes = sizeof(int) * REPLAY_STATIC_MAX_BATCH;
constexpr size_t kPlanBytes = sizeof(int4) * REPLAY_STATIC_MAX_BATCH;
constexpr size_t kCoefBytes = sizeof(float) * static_cast<size_t>(REPLAY_STATIC_MAX_COEFS);
constexpr size_t kScratchBytes = kArriveBytes + kPlanBytes + kCoefBytes;

static __device__ __align__(256) unsigned char g_step_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
unsigned char* g_scratch_ptr[kMaxDevices] = {};  // device address of the array, per device

// Device address of the scratch array on the current device, looked up once per device.
// On the host, g_step_scratch names a host-side stand-in, never the device memory, so the
// address must come from cudaGetSymbolAddress with that device current.
int scratch_on_current_device(unsigned char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return REPLAY_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return REPLAY_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_step_scratch) != cudaSuccess || p == nullptr) return REPLAY_ECUDA;
    g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
  }
  *out = g_scratch_ptr[dev];
  return REPLAY_OK;
}

bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

}  // namespace

extern "C" int replay_step_static_scratch(replay_store* st, const void* x, const void* B, const void* C,
                                          const void* dt, float* y, void* stream) {
  if (st == nullptr || x == nullptr || B == nullptr || C == nullptr || dt == nullptr || y == nullptr)
    return REPLAY_EBADARG;
  if (!aligned16(x) || !aligned16(B) || !aligned16(C)) return REPLAY_EBADARG;
  const size_t coefs = static_cast<size_t>(st->cfg.batch) * st->cfg.nheads * (st->lay.cap + 1);
  if (st->cfg.batch > REPLAY_STATIC_MAX_BATCH || coefs > static_cast<size_t>(REPLAY_STATIC_MAX_COEFS))
    return REPLAY_ECAPACITY;
  unsigned char* scratch = nullptr;
  int rc = scratch_on_current_device(&scratch);
  if (rc != REPLAY_OK) return rc;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps whatever the previous call left: the arrival counters must start at
  // zero (plan and coefficients are written by the step before they are read).
  if (cudaMemsetAsync(scratch, 0, sizeof(int) * static_cast<size_t>(st->cfg.batch), s) != cudaSuccess)
    return REPLAY_ECUDA;
  rssm::StoreView sv = st->sv;
  sv.arrive = reinterpret_cast<int*>(scratch);
  sv.plan = reinterpret_cast<int4*>(scratch + kArriveBytes);
  sv.coef = reinterpret_cast<float*>(scratch + kArriveBytes + kPlanBytes);
  // (one plan and coefficient buffer, and no overlap with the previous step: the memset
  // above already separates the two)
  rc = rssm::launch_step(sv, st->sh, st->all_n, 0, 0, x, B, C, dt, y, s);
  st->prev_nonflush = 0;
  if (rc == REPLAY_OK) st->all_n = advance_all_n(st);
  return rc;
}
