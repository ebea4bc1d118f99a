// The C ABI of the library: argument checks on the host, the workspace layout, and
// dispatch to the kernel launchers. Declarations and the meaning of every call are in
// include/replayssm.h.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <new>

#include "launch.h"
#include "store.h"

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool shape_supported(int P, int N) { return P == 64 && (N == 64 || N == 128 || N == 256); }

int check_shape(const replay_config* c) {
  if (c == nullptr) return REPLAY_EBADARG;
  if (c->batch < 1 || c->nheads < 1 || c->ngroups < 1 || c->headdim < 1 || c->dstate < 1)
    return REPLAY_EBADARG;
  if (c->nheads % c->ngroups != 0) return REPLAY_EBADARG;
  if (c->in_dtype != REPLAY_F32 && c->in_dtype != REPLAY_BF16) return REPLAY_EBADARG;
  if (!shape_supported(c->headdim, c->dstate)) return REPLAY_EUNSUPPORTED;
  if (static_cast<long long>(c->batch) * c->nheads > INT_MAX) return REPLAY_ECAPACITY;
  if (c->batch > 65535 || c->nheads / c->ngroups > 65535) return REPLAY_ECAPACITY;  // grid limits
  return REPLAY_OK;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

int cuda_ok(cudaError_t e) { return e == cudaSuccess ? REPLAY_OK : REPLAY_ECUDA; }

// x, B, C and states are read with 16-byte vector loads and asynchronous copies.
bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

}  // namespace

extern "C" {

int replay_abi_version(void) { return REPLAY_ABI_VERSION; }

const char* replay_strerror(int code) {
  switch (code) {
    case REPLAY_OK: return "ok";
    case REPLAY_EBADARG: return "bad argument";
    case REPLAY_EUNSUPPORTED: return "unsupported shape or dtype";
    case REPLAY_ECAPACITY: return "capacity exceeded";
    case REPLAY_ECUDA: return "CUDA error";
    default: return "unknown error";
  }
}

int replay_layout_of(const replay_config* c, replay_layout* out) {
  if (out == nullptr) return REPLAY_EBADARG;
  int rc = check_shape(c);
  if (rc != REPLAY_OK) return rc;
  if (c->window_L < 1 || c->max_draft_T < 0) return REPLAY_EBADARG;
  if (c->read_copy < REPLAY_RC_NONE || c->read_copy > REPLAY_RC_NVFP4) return REPLAY_EBADARG;
  if (c->read_copy == REPLAY_RC_FP16 && c->dstate > 128) return REPLAY_EUNSUPPORTED;
  if (c->read_copy == REPLAY_RC_NVFP4 && c->dstate != 128) return REPLAY_EUNSUPPORTED;
  if (c->shared_checkpoint != 0 && (c->shared_checkpoint != 1 || c->read_copy == REPLAY_RC_NONE))
    return REPLAY_EBADARG;
  if (c->checkpoint_format != REPLAY_CKPT_F32 && c->checkpoint_format != REPLAY_CKPT_F16_SR) return REPLAY_EBADARG;
  if (c->checkpoint_format == REPLAY_CKPT_F16_SR) {
    if (c->shared_checkpoint != 0 || c->read_copy == REPLAY_RC_NONE || c->read_copy == REPLAY_RC_FP16)
      return REPLAY_EBADARG;
    if (c->dstate > 128) return REPLAY_EUNSUPPORTED;
  }
  if (c->max_draft_T > 8) return REPLAY_ECAPACITY;
  const long long cap = c->max_draft_T > 0 ? static_cast<long long>(c->window_L) + 2LL * c->max_draft_T - 1
                                           : c->window_L;
  if (cap > rssm::kMaxCap) return REPLAY_ECAPACITY;
  const size_t Bn = c->batch, H = c->nheads, G = c->ngroups, P = c->headdim, N = c->dstate;
  const size_t esz = c->in_dtype == REPLAY_F32 ? 4 : 2;
  // read-copy bytes per 2 elements
  const size_t rc2 = c->read_copy == REPLAY_RC_NONE    ? 0
                     : c->read_copy == REPLAY_RC_NVFP4 ? 1
                     : c->read_copy == REPLAY_RC_FP8E4M3 ? 2 : 4;
  const bool slab_scale = c->read_copy == REPLAY_RC_FP8E4M3 || c->read_copy == REPLAY_RC_NVFP4;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes);
    return at;
  };
  replay_layout L;
  L.cap = static_cast<int>(cap);
  const size_t ckpt_bytes = c->shared_checkpoint ? 0 : (c->checkpoint_format == REPLAY_CKPT_F16_SR ? 2 : 4);
  L.h0 = take(Bn * H * P * N * ckpt_bytes);  // no separate checkpoint when shared
  L.rc = take(Bn * H * P * N / 2 * rc2);
  L.scale = take(slab_scale ? Bn * H * 4 : 0);
  L.bscale = take(c->read_copy == REPLAY_RC_NVFP4 ? Bn * H * P * N / 16 : 0);
  L.xbuf = take(Bn * H * cap * P * esz);
  L.bbuf = take(Bn * G * cap * N * esz);
  L.dtbuf = take(Bn * H * cap * esz);
  L.meta = take(Bn * 16);
  L.arrive = take(Bn * 4);
  L.status = take(4);
  L.plan = take(2 * Bn * 16);  // two: a step's plan is written while the previous step reads its own
  L.coef = take(Bn * H * std::max<size_t>(static_cast<size_t>(c->max_draft_T) + 1, 2) * (cap + 1) * 4);
  L.total = off;
  *out = L;
  return REPLAY_OK;
}

int replay_store_bytes(const replay_config* c, size_t* bytes) {
  if (bytes == nullptr) return REPLAY_EBADARG;
  replay_layout L;
  const int rc = replay_layout_of(c, &L);
  if (rc == REPLAY_OK) *bytes = L.total;
  return rc;
}

int replay_alloc(const replay_config* c, void* workspace, size_t workspace_bytes, const float* A,
                 const float* D, void* stream, replay_store** out) {
  if (out == nullptr || workspace == nullptr || A == nullptr || D == nullptr) return REPLAY_EBADARG;
  replay_layout L;
  int rc = replay_layout_of(c, &L);
  if (rc != REPLAY_OK) return rc;
  if (reinterpret_cast<uintptr_t>(workspace) % kAlign != 0) return REPLAY_EBADARG;
  if (workspace_bytes < L.total) return REPLAY_ECAPACITY;
  replay_store* st = new (std::nothrow) replay_store;
  if (st == nullptr) return REPLAY_ECAPACITY;
  st->cfg = *c;
  st->lay = L;
  st->step_parity = 0;
  st->prev_nonflush = 0;
  st->ws = static_cast<char*>(workspace);
  rssm::StoreView& sv = st->sv;
  sv.h0 = reinterpret_cast<float*>(st->ws + L.h0);
  sv.rc = st->ws + L.rc;
  sv.scale = reinterpret_cast<float*>(st->ws + L.scale);
  sv.bscale = reinterpret_cast<uint8_t*>(st->ws + L.bscale);
  sv.xbuf = st->ws + L.xbuf;
  sv.bbuf = st->ws + L.bbuf;
  sv.dtbuf = st->ws + L.dtbuf;
  sv.meta = reinterpret_cast<int4*>(st->ws + L.meta);
  sv.arrive = reinterpret_cast<int*>(st->ws + L.arrive);
  sv.status = reinterpret_cast<int*>(st->ws + L.status);
  sv.plan = reinterpret_cast<int4*>(st->ws + L.plan);
  sv.coef = reinterpret_cast<float*>(st->ws + L.coef);
  sv.A = A;
  sv.D = D;
  sv.batch = c->batch;
  sv.H = c->nheads;
  sv.G = c->ngroups;
  sv.hpg = c->nheads / c->ngroups;
  sv.L = c->window_L;
  sv.cap = L.cap;
  sv.tmax = c->max_draft_T;
  sv.shared = c->shared_checkpoint;
  sv.ckpt16 = c->checkpoint_format == REPLAY_CKPT_F16_SR;
  sv.prep_appends = c->read_copy != REPLAY_RC_NONE;
  int dev = 0;
  sv.sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sv.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    sv.sms = 0;
    (void)cudaGetLastError();
  }
  st->sh = rssm::Shape{c->headdim, c->dstate, c->in_dtype, c->read_copy};
  rc = replay_reset(st, nullptr, stream);
  if (rc != REPLAY_OK) {
    delete st;
    return rc;
  }
  *out = st;
  return REPLAY_OK;
}

int replay_free(replay_store* st) {
  if (st == nullptr) return REPLAY_EBADARG;
  delete st;
  return REPLAY_OK;
}

int replay_reset(replay_store* st, const int* seq_mask, void* stream) {
  if (st == nullptr) return REPLAY_EBADARG;
  if (seq_mask == nullptr) {
    int rc = cuda_ok(cudaMemsetAsync(st->sv.status, 0, sizeof(int), as_stream(stream)));
    if (rc != REPLAY_OK) return rc;
  }
  const int rc = rssm::launch_load(st->sv, st->sh, nullptr, seq_mask, as_stream(stream));
  st->all_n = rc == REPLAY_OK && seq_mask == nullptr ? 0 : -1;
  st->prev_nonflush = 0;
  return rc;
}

int replay_load_state(replay_store* st, const float* h, void* stream) {
  if (st == nullptr || h == nullptr) return REPLAY_EBADARG;
  const int rc = rssm::launch_load(st->sv, st->sh, h, nullptr, as_stream(stream));
  st->all_n = rc == REPLAY_OK ? 0 : -1;
  st->prev_nonflush = 0;
  return rc;
}

int replay_export_state(replay_store* st, float* h_out, void* stream) {
  if (st == nullptr || h_out == nullptr) return REPLAY_EBADARG;
  st->prev_nonflush = 0;
  return rssm::launch_fold(st->sv, st->sh, 1, h_out, as_stream(stream));
}

int replay_step(replay_store* st, const void* x, const void* B, const void* C, const void* dt,
                float* y, void* stream) {
  if (st == nullptr || x == nullptr || B == nullptr || C == nullptr || dt == nullptr || y == nullptr)
    return REPLAY_EBADARG;
  if (!aligned16(x) || !aligned16(B) || !aligned16(C)) return REPLAY_EBADARG;
  const int all_n = st->all_n;
  // (stores without a read copy never overlap steps: one buffer, the per-head kernels append)
  const int parity = st->sv.prep_appends ? st->step_parity : 0;
  const int rc = rssm::launch_step(st->sv, st->sh, all_n, parity, st->prev_nonflush, x, B, C, dt, y,
                                   as_stream(stream));
  st->prev_nonflush = rc == REPLAY_OK && st->sv.prep_appends && all_n >= 0 && all_n + 1 < st->cfg.window_L &&
                      rssm::step_runs_prep(st->sv);
  if (rc == REPLAY_OK) {
    st->all_n = advance_all_n(st);
    st->step_parity ^= 1;
  }
  return rc;
}

int replay_verify(replay_store* st, int T, const void* x, const void* B, const void* C,
                  const void* dt, float* y, void* stream) {
  if (st == nullptr || x == nullptr || B == nullptr || C == nullptr || dt == nullptr || y == nullptr)
    return REPLAY_EBADARG;
  if (T < 1 || !aligned16(x) || !aligned16(B) || !aligned16(C)) return REPLAY_EBADARG;
  if (T > st->cfg.max_draft_T) return REPLAY_ECAPACITY;
  st->all_n = -1;
  st->prev_nonflush = 0;
  return rssm::launch_verify(st->sv, st->sh, T, x, B, C, dt, y, as_stream(stream));
}

int replay_commit(replay_store* st, const int* accept, void* stream) {
  if (st == nullptr || accept == nullptr) return REPLAY_EBADARG;
  st->all_n = -1;
  st->prev_nonflush = 0;
  return rssm::launch_commit(st->sv, accept, as_stream(stream));
}

int replay_flush(replay_store* st, void* stream) {
  if (st == nullptr) return REPLAY_EBADARG;
  st->prev_nonflush = 0;
  const int rc = rssm::launch_fold(st->sv, st->sh, 0, nullptr, as_stream(stream));
  if (rc == REPLAY_OK) st->all_n = 0;
  return rc;
}

int replay_status(replay_store* st, int* status_out, int clear, void* stream) {
  if (st == nullptr || status_out == nullptr) return REPLAY_EBADARG;
  int v = 0;
  int rc = cuda_ok(cudaMemcpyAsync(&v, st->sv.status, sizeof(int), cudaMemcpyDeviceToHost, as_stream(stream)));
  if (rc == REPLAY_OK) rc = cuda_ok(cudaStreamSynchronize(as_stream(stream)));
  if (rc != REPLAY_OK) return rc;
  *status_out = v;
  if (clear) rc = cuda_ok(cudaMemsetAsync(st->sv.status, 0, sizeof(int), as_stream(stream)));
  return rc;
}

int conv_step(const replay_config* c, void* state, int state_dtype, const float* A, const float* D,
              const void* x, const void* B, const void* C, const void* dt, float* y, void* stream) {
  int rc = check_shape(c);
  if (rc != REPLAY_OK) return rc;
  if (state == nullptr || A == nullptr || D == nullptr || x == nullptr || B == nullptr || C == nullptr ||
      dt == nullptr || y == nullptr)
    return REPLAY_EBADARG;
  if (state_dtype != REPLAY_F32 && state_dtype != REPLAY_BF16) return REPLAY_EBADARG;
  if (!aligned16(state) || !aligned16(x) || !aligned16(B) || !aligned16(C)) return REPLAY_EBADARG;
  const rssm::Shape sh{c->headdim, c->dstate, c->in_dtype, REPLAY_RC_NONE};
  return rssm::launch_conv_step(sh, c->batch, c->nheads, c->ngroups, state, state_dtype, A, D, x, B, C,
                                dt, y, as_stream(stream));
}

int conv_verify_snapshot(const replay_config* c, int T, float* snaps, const int* cur, const float* A,
                         const float* D, const void* x, const void* B, const void* C, const void* dt,
                         float* y, void* stream) {
  int rc = check_shape(c);
  if (rc != REPLAY_OK) return rc;
  if (snaps == nullptr || cur == nullptr || A == nullptr || D == nullptr || x == nullptr || B == nullptr ||
      C == nullptr || dt == nullptr || y == nullptr || T < 1)
    return REPLAY_EBADARG;
  if (!aligned16(snaps) || !aligned16(x) || !aligned16(B) || !aligned16(C)) return REPLAY_EBADARG;
  const rssm::Shape sh{c->headdim, c->dstate, c->in_dtype, REPLAY_RC_NONE};
  return rssm::launch_conv_verify(sh, c->batch, c->nheads, c->ngroups, T, snaps, cur, A, D, x, B, C, dt,
                                  y, as_stream(stream));
}

int conv_commit(int batch, int T, int* cur, const int* accept, int* status, void* stream) {
  if (batch < 1 || T < 1 || cur == nullptr || accept == nullptr) return REPLAY_EBADARG;
  return rssm::launch_conv_commit(batch, T, cur, accept, status, as_stream(stream));
}

}  // extern "C"
