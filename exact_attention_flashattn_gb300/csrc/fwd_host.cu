// Prefill with host-resident Q, K, V, O and LSE: the work is cut into chunks of (sequence, KV
// head) units, and each chunk's copies in, kernel and copies out run on three streams, so that
// the transfers of one chunk overlap the kernels and the other direction's transfers of the
// neighbouring chunks. Device staging comes from the caller's workspace (two slots, used
// alternately); the library allocates nothing.
//
// A chunk of units is one contiguous byte range in every tensor: in the [B, H, N, d] layouts,
// unit u = (b, kv head hk) owns query heads hk*g .. hk*g + g - 1 of batch b, which start at
// element u * g * Nq * d of Q and O, u * Nk * d of K and V and u * g * Nq of LSE. A chunk of n
// units is therefore exactly a prefill with B = n, Hq = g, Hkv = 1, and is run as one.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/bwattn.h"
#include "kernels.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kSlots = 2;
constexpr int kMaxChunks = 8;

constexpr int kH2dStreams = 3;  // Q, K and V of a chunk are copied in on streams of their own

struct HostPipe {
  cudaStream_t h2d[kH2dStreams] = {}, comp = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t h2d_done[kMaxChunks][kH2dStreams] = {}, comp_done[kMaxChunks] = {}, d2h_done[kMaxChunks] = {};
  bool ready = false;
};
HostPipe g_pipe[kMaxDevices];
// held while a call enqueues its work: the streams and events above are shared by all calls
std::mutex g_pipe_mu;

cudaError_t make_pipe(HostPipe& p) {
  cudaError_t e;
  const unsigned sf = cudaStreamNonBlocking;
  for (int i = 0; i < kH2dStreams; ++i)
    if ((e = cudaStreamCreateWithFlags(&p.h2d[i], sf)) != cudaSuccess) return e;
  if ((e = cudaStreamCreateWithFlags(&p.comp, sf)) != cudaSuccess) return e;
  if ((e = cudaStreamCreateWithFlags(&p.d2h, sf)) != cudaSuccess) return e;
  const unsigned ef = cudaEventDisableTiming;
  if ((e = cudaEventCreateWithFlags(&p.start, ef)) != cudaSuccess) return e;
  if ((e = cudaEventCreateWithFlags(&p.done, ef)) != cudaSuccess) return e;
  for (int i = 0; i < kMaxChunks; ++i) {
    for (int j = 0; j < kH2dStreams; ++j)
      if ((e = cudaEventCreateWithFlags(&p.h2d_done[i][j], ef)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&p.comp_done[i], ef)) != cudaSuccess) return e;
    if ((e = cudaEventCreateWithFlags(&p.d2h_done[i], ef)) != cudaSuccess) return e;
  }
  p.ready = true;
  return cudaSuccess;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Plan {
  int g = 0, units = 0, per = 0, nchunks = 0;
  size_t es = 0;                       // bytes per element
  size_t q_b = 0, kv_b = 0, lse_b = 0;  // bytes of one chunk (per = units per chunk)
  size_t slot_b = 0;                   // one staging slot: q, k, v, o, lse
};

bool make_plan(int B, int Hq, int Hkv, int Nq, int Nk, int d, int dtype, Plan* p) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk < 0 || d <= 0 || Hq % Hkv != 0) return false;
  if (dtype != BWATTN_DTYPE_BF16 && dtype != BWATTN_DTYPE_FP32) return false;
  p->g = Hq / Hkv;
  p->units = B * Hkv;
  p->nchunks = p->units < kMaxChunks ? p->units : kMaxChunks;
  p->per = (p->units + p->nchunks - 1) / p->nchunks;
  p->nchunks = (p->units + p->per - 1) / p->per;
  p->es = dtype == BWATTN_DTYPE_BF16 ? 2 : 4;
  p->q_b = static_cast<size_t>(p->per) * p->g * Nq * d * p->es;
  p->kv_b = static_cast<size_t>(p->per) * Nk * d * p->es;
  p->lse_b = static_cast<size_t>(p->per) * p->g * Nq * sizeof(float);
  p->slot_b = 2 * align256(p->q_b) + 2 * align256(p->kv_b) + align256(p->lse_b);
  return true;
}

}  // namespace

extern "C" {

size_t attn_fwd_host_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d, int dtype) {
  Plan p;
  if (!make_plan(B, Hq, Hkv, Nq, Nk, d, dtype, &p)) return 0;
  return kSlots * p.slot_b;
}

int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                  int Nk, int d, int causal, float scale, int dtype, void* workspace, size_t workspace_bytes,
                  void* stream) {
  if (B < 0 || Nq < 0 || Nk < 0) return BWATTN_ERR_INVALID_ARG;
  if (B == 0 || Nq == 0) return BWATTN_OK;
  Plan p;
  if (!make_plan(B, Hq, Hkv, Nq, Nk, d, dtype, &p)) {
    return (dtype != BWATTN_DTYPE_BF16 && dtype != BWATTN_DTYPE_FP32) ? BWATTN_ERR_UNSUPPORTED
                                                                      : BWATTN_ERR_INVALID_ARG;
  }
  if (!q || !o || (Nk > 0 && (!k || !v)) || !workspace) return BWATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < kSlots * p.slot_b)
    return BWATTN_ERR_INVALID_ARG;
  // the chunk calls validate the rest (head dim, scale, causal flag) before any CUDA call; an
  // empty call with a chunk's shape reports those errors here, before anything is queued
  {
    const int rc = attn_fwd(nullptr, nullptr, nullptr, nullptr, nullptr, 0, p.g, 1, Nq, Nk, d, causal, scale, dtype,
                            nullptr);
    if (rc != BWATTN_OK) return rc;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    bw::record_cuda_error(e);
    return BWATTN_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return BWATTN_ERR_UNSUPPORTED;

  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe& pp = g_pipe[dev];
  if (!pp.ready && (e = make_pipe(pp)) != cudaSuccess) {
    bw::record_cuda_error(e);
    return BWATTN_ERR_CUDA;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // On an error after work was queued, wait for this call's own streams before returning, so
  // that no copy from or to the caller's host buffers is still running when the caller sees
  // the error (their status is not reported again: the first error is).
  auto drain = [&pp](int rc) {
    for (int i = 0; i < kH2dStreams; ++i) cudaStreamSynchronize(pp.h2d[i]);
    cudaStreamSynchronize(pp.comp);
    cudaStreamSynchronize(pp.d2h);
    return rc;
  };
  auto fail = [&drain](cudaError_t err) {
    bw::record_cuda_error(err);
    return drain(BWATTN_ERR_CUDA);
  };
  // everything starts after the work already queued on the caller's stream
  if ((e = cudaEventRecord(pp.start, st)) != cudaSuccess) return fail(e);
  for (int i = 0; i < kH2dStreams; ++i)
    if ((e = cudaStreamWaitEvent(pp.h2d[i], pp.start, 0)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(pp.comp, pp.start, 0)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(pp.d2h, pp.start, 0)) != cudaSuccess) return fail(e);

  const size_t q_unit = p.q_b / p.per, kv_unit = p.kv_b / p.per, lse_unit = p.lse_b / p.per;
  const auto* hq = static_cast<const uint8_t*>(q);
  const auto* hk = static_cast<const uint8_t*>(k);
  const auto* hv = static_cast<const uint8_t*>(v);
  auto* ho = static_cast<uint8_t*>(o);
  auto* hl = reinterpret_cast<uint8_t*>(lse);
  for (int c = 0; c < p.nchunks; ++c) {
    const int s = c % kSlots;
    const int u0 = c * p.per;
    const int n = (p.units - u0) < p.per ? (p.units - u0) : p.per;
    uint8_t* base = static_cast<uint8_t*>(workspace) + s * p.slot_b;
    uint8_t* dq = base;
    uint8_t* dk = dq + align256(p.q_b);
    uint8_t* dv = dk + align256(p.kv_b);
    uint8_t* dout = dv + align256(p.kv_b);
    float* dl = reinterpret_cast<float*>(dout + align256(p.q_b));
    const size_t qn = q_unit * n, kvn = kv_unit * n, ln = lse_unit * n;
    // copies in: the slot's inputs are free once the kernel of chunk c - kSlots has finished
    const void* src[kH2dStreams] = {hq + q_unit * u0, hk + kv_unit * u0, hv + kv_unit * u0};
    void* dst[kH2dStreams] = {dq, dk, dv};
    const size_t bytes[kH2dStreams] = {qn, kvn, kvn};
    for (int i = 0; i < kH2dStreams; ++i) {
      if (c >= kSlots && (e = cudaStreamWaitEvent(pp.h2d[i], pp.comp_done[c - kSlots], 0)) != cudaSuccess)
        return fail(e);
      if (bytes[i] > 0 &&
          (e = cudaMemcpyAsync(dst[i], src[i], bytes[i], cudaMemcpyHostToDevice, pp.h2d[i])) != cudaSuccess)
        return fail(e);
      if ((e = cudaEventRecord(pp.h2d_done[c][i], pp.h2d[i])) != cudaSuccess) return fail(e);
    }
    // kernel: after its inputs, and after the slot's outputs of chunk c - kSlots were copied out
    for (int i = 0; i < kH2dStreams; ++i)
      if ((e = cudaStreamWaitEvent(pp.comp, pp.h2d_done[c][i], 0)) != cudaSuccess) return fail(e);
    if (c >= kSlots && (e = cudaStreamWaitEvent(pp.comp, pp.d2h_done[c - kSlots], 0)) != cudaSuccess) return fail(e);
    const int rc = attn_fwd(dq, dk, dv, dout, lse ? dl : nullptr, n, p.g, 1, Nq, Nk, d, causal, scale, dtype, pp.comp);
    if (rc != BWATTN_OK) return drain(rc);
    if ((e = cudaEventRecord(pp.comp_done[c], pp.comp)) != cudaSuccess) return fail(e);
    // copies out
    if ((e = cudaStreamWaitEvent(pp.d2h, pp.comp_done[c], 0)) != cudaSuccess) return fail(e);
    if ((e = cudaMemcpyAsync(ho + q_unit * u0, dout, qn, cudaMemcpyDeviceToHost, pp.d2h)) != cudaSuccess)
      return fail(e);
    if (lse && (e = cudaMemcpyAsync(hl + lse_unit * u0, dl, ln, cudaMemcpyDeviceToHost, pp.d2h)) != cudaSuccess)
      return fail(e);
    if ((e = cudaEventRecord(pp.d2h_done[c], pp.d2h)) != cudaSuccess) return fail(e);
  }
  // the caller's stream continues once the last copy out has landed (it follows every kernel)
  if ((e = cudaEventRecord(pp.done, pp.d2h)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(st, pp.done, 0)) != cudaSuccess) return fail(e);
  return BWATTN_OK;
}

}  // extern "C"
