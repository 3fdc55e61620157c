// attn_decode_static: split-K decode for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or pass a workspace: a plugin or inference-engine host
// that hands a kernel only its input and output buffers, code whose device memory is owned by
// another allocator, or a latency-critical loop that cannot take cudaMalloc's implicit device
// synchronisation. For them this entry point runs the same split-K pass and merge as
// attn_decode, with the per-split partial states kept in a fixed file-scope device array
// instead of a caller-provided workspace. The pages have no counterpart to it.
//
// The array is BWATTN_DECODE_STATIC_SCRATCH_BYTES (8 MiB); every GPU that loads the library
// holds it until the process exits. In host code its name is only a host-side stand-in, so
// its device address is looked up with cudaGetSymbolAddress once per device (with that device
// current) on the first call there, and that address is what the kernels receive. Every call
// on a device shares the array and it keeps the last call's contents; nothing needs clearing
// (the split pass writes every partial the merge then reads), but overlapping calls race.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/bwattn.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchFloats = BWATTN_DECODE_STATIC_SCRATCH_BYTES / sizeof(float);
static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on first use there.
cudaError_t scratch_address(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    float* p = nullptr;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" int attn_decode_static(const void* q, const void* kcache, const void* vcache, void* o, const int32_t* nk,
                                  int B, int Hq, int Hkv, int nk_cap, int d, int num_splits, float scale, float* lse,
                                  void* stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || nk_cap < 0 || d <= 0) return BWATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || !(isfinite(scale) && scale > 0.f) || num_splits < 1 || num_splits > 1024)
    return BWATTN_ERR_INVALID_ARG;
  if (B > 65535) return BWATTN_ERR_INVALID_ARG;
  const int g = Hq / Hkv;
  if ((d != 64 && d != 128 && d != 256) || g > 32 || Hkv > 32767) return BWATTN_ERR_UNSUPPORTED;
  if (B == 0) return BWATTN_OK;
  if (!q || !kcache || !vcache || !o || !nk) return BWATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) || !aligned4(nk) ||
      (lse && !aligned4(lse)))
    return BWATTN_ERR_INVALID_ARG;
  // the partials of this call must fit the fixed array
  if (bw::splitk_ws_bytes(B * Hkv, num_splits, g, d) > BWATTN_DECODE_STATIC_SCRATCH_BYTES)
    return BWATTN_ERR_UNSUPPORTED;
  float* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    bw::record_cuda_error(e);
    return BWATTN_ERR_CUDA;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  bw::SplitKArgs a{};
  a.d = d;
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(kcache);
  a.v = static_cast<const uint16_t*>(vcache);
  a.ws = scratch;
  a.nk = nk;
  a.cu_q = a.cu_k = nullptr;
  a.num_seqs = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.g = g;
  a.kv_seq_stride = static_cast<int64_t>(Hkv) * nk_cap * d;
  a.kv_head_stride = static_cast<int64_t>(nk_cap) * d;
  a.kv_key_stride = d;
  a.kv_cap = nk_cap;
  a.total_q = a.total_k = 0;
  a.num_splits = num_splits;
  a.rows_max = g;
  a.group_rows = g <= 8 ? 8 : 16;
  a.row_groups = (g + a.group_rows - 1) / a.group_rows;
  a.causal = 0;
  a.small_rows_limit = g;
  a.ws_o_offset = bw::splitk_o_offset(B * Hkv, num_splits, g);
  a.scale_log2 = scale * bw::kLog2e;
  if ((e = bw::launch_splitk(a, st)) != cudaSuccess) {
    bw::record_cuda_error(e);
    return BWATTN_ERR_CUDA;
  }
  bw::count_launch();
  bw::MergeArgs m{};
  m.d = d;
  m.ws = scratch;
  m.o = static_cast<uint16_t*>(o);
  m.lse = lse;
  m.cu_q = m.cu_k = nullptr;
  m.nk = nk;
  m.num_seqs = B;
  m.Hq = Hq;
  m.Hkv = Hkv;
  m.g = g;
  m.num_splits = num_splits;
  m.rows_max = g;
  m.small_rows_limit = g;
  m.total_q = B;
  m.ws_o_offset = a.ws_o_offset;
  if ((e = bw::launch_merge(m, st)) != cudaSuccess) {
    bw::record_cuda_error(e);
    return BWATTN_ERR_CUDA;
  }
  bw::count_launch();
  return BWATTN_OK;
}
