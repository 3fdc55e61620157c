// C-ABI of libbwattn: argument validation, TMA tensor-map encoding, workspace layout and
// kernel dispatch. See include/bwattn.h for the contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "../../include/bwattn.h"
#include "kernels.h"

namespace {

__device__ unsigned int g_status_word;

constexpr int kMaxDevices = 64;

// Item counters of the persistent prefill kernel: one pair per launch, taken round-robin from
// this ring (one position per device), so launches in flight on different streams never share
// a pair unless 4096 or more prefill launches are in flight on the device at once; a launch
// leaves its pair zeroed when it completes.
constexpr int kSchedSlots = 4096;
__device__ unsigned int g_sched_counters[2 * kSchedSlots];
std::atomic<uint32_t> g_sched_next[kMaxDevices];

// Merge tickets of the split-K kernel: each launch takes a contiguous block (zeroed, and left
// zeroed by the kernel) from this ring (one position per device); the ring holds 2^16 tickets,
// so a block is handed out again only after 2^16 more tickets have been taken on the device.
// Launches still in flight by then (other streams, a captured graph replayed alongside) would
// share it; the header states the limit.
constexpr uint32_t kTicketSlots = 1u << 16;
// Varlen short-query pass: with more splits than this the separate merge kernel (one CTA per
// output row) is faster than letting one CTA per unit walk all the splits. Below it the fused
// merge also saves the merge launch's CTAs for every inactive (sequence, row) of the batch
// (separate merge at 8 splits: 1.000 against 0.949 ms on the 64-sequence append workload).
constexpr int kFusedMergeMaxSplits = 32;
// Dense and paged decode: the separate merge, a programmatic dependent launch, is faster from a
// few splits on (16 splits: bf16 GQA +0.6 %, paged +1.2 %, FP8 GQA +2.5 %, FP8 paged +1.7 %;
// 8 splits, d = 256: +0.5 %); with this many or fewer the fused merge saves the second launch.
constexpr int kFusedMergeMaxSplitsDecode = 4;
__device__ unsigned int g_merge_tickets[kTicketSlots];
uint32_t g_ticket_next[kMaxDevices] = {};

thread_local int t_last_cuda_error = 0;
std::atomic<uint64_t> g_launches{0};
std::atomic<uint64_t> g_timeout_ns{2000000000ull};

std::mutex g_mu;
unsigned int* g_status_ptr[kMaxDevices] = {};
unsigned int* g_sched_ptr[kMaxDevices] = {};
unsigned int* g_ticket_ptr[kMaxDevices] = {};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return BWATTN_ERR_CUDA;
}

// Device address of the status word on the current device (looked up once per device).
cudaError_t status_ptr(unsigned int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return e;
    g_status_ptr[dev] = static_cast<unsigned int*>(p);
  }
  *out = g_status_ptr[dev];
  return cudaSuccess;
}

// A fresh pair of item counters on the current device for one launch of the prefill kernel.
cudaError_t sched_ptr(unsigned int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned int* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sched_ptr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_sched_counters);
      if (e != cudaSuccess) return e;
      g_sched_ptr[dev] = static_cast<unsigned int*>(p);
    }
    base = g_sched_ptr[dev];
  }
  *out = base + 2 * (g_sched_next[dev].fetch_add(1) % kSchedSlots);
  return cudaSuccess;
}

cudaError_t encoder(EncodeTiledFn* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  *out = g_encode;
  return cudaSuccess;
}

// 3-D bf16 map {d, dim1, dim2} with row strides in elements, box {64, box1, box2},
// 128-byte swizzle, zero fill out of bounds.
cudaError_t make_map(CUtensorMap* m, const void* base, int d, int64_t dim1, int64_t dim2, int64_t stride1_elems,
                     int64_t stride2_elems, int box1, int box2) {
  EncodeTiledFn enc = nullptr;
  cudaError_t e = encoder(&enc);
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(dim1),
                              static_cast<cuuint64_t>(dim2)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(stride1_elems) * 2,
                                 static_cast<cuuint64_t>(stride2_elems) * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box1), static_cast<cuuint32_t>(box2)};
  const cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D uint8 map {128, dim1, dim2} with row strides in bytes, box {128, box1, box2}, 128-byte
// swizzle (rows of E4M3 codes at d = 128: one swizzle atom wide), zero fill out of bounds.
cudaError_t make_map_u8(CUtensorMap* m, const void* base, int64_t dim1, int64_t dim2, int64_t stride1_bytes,
                        int64_t stride2_bytes, int box1, int box2) {
  EncodeTiledFn enc = nullptr;
  cudaError_t e = encoder(&enc);
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(dim1), static_cast<cuuint64_t>(dim2)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(stride1_bytes), static_cast<cuuint64_t>(stride2_bytes)};
  const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(box1), static_cast<cuuint32_t>(box2)};
  const cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Units per band of the prefill item list: as many (sequence, head) units as keep their K and V
// (one KV head serves g consecutive query heads) within 16 MB, between 16 and 64. Wider bands
// help short sequences, whose items are many and short (32 units: +5.6 % at 1024 keys, d = 128);
// from 2048 keys on (d = 128) the band stays at 16, where wider ones measured 1-2 % slower. At
// d = 256 the floor is 8 units: 16 units of 4096 keys hold 64 MB of K/V, and the two bands in
// flight then no longer fit in L2 (DRAM reads 1.4x the Q, K, V bytes), while 8 units measured
// as fast.
int band_units_for(int64_t nk, int d, int g) {
  const int64_t unit_bytes = std::max<int64_t>(1, nk * d * 4 / std::max(g, 1));
  const int64_t b = (static_cast<int64_t>(16) << 20) / unit_bytes;
  const int64_t floor_units = d == 256 ? 8 : 16;
  return static_cast<int>(std::min<int64_t>(64, std::max<int64_t>(floor_units, b)));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool good_scale(float s) { return isfinite(s) && s > 0.f; }

constexpr int kSmallRowsLimit = 32;  // varlen: n_q * g at or below this takes the split-K path
// varlen short-query rows are taken 16 at a time in the 16-row MMA form (168 registers, three
// CTAs per SM). Groups of 8 in the transposed form (127 registers, four CTAs; a sequence with
// more rows takes several row-group CTAs, which read its K/V from L2 after the first) measured
// 1.194 against 1.093 ms on the 64-sequence append workload.
constexpr int kVarlenGroupRows = 16;
// Keys per split of the short-query pass, which is also the least a split takes (min_chunk):
// 4096 measured 0.937 ms on the 64-sequence append workload against 0.945 for 2048, 0.984 for
// 1024 and 0.986 for 8192.
constexpr int kVarlenKeysPerSplit = 4096;
constexpr int kVarlenMaxSplits = 64;

int varlen_splits(int max_seqlen_k) {
  int s = (max_seqlen_k + kVarlenKeysPerSplit - 1) / kVarlenKeysPerSplit;
  if (s < 1) s = 1;
  if (s > kVarlenMaxSplits) s = kVarlenMaxSplits;
  return s;
}

}  // namespace

namespace bw {
void record_cuda_error(cudaError_t e) { t_last_cuda_error = static_cast<int>(e); }
void count_launch() { g_launches.fetch_add(1); }

cudaError_t merge_tickets(int n, unsigned int** out) {
  *out = nullptr;
  if (n <= 0 || static_cast<uint32_t>(n) > kTicketSlots / 16) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_ticket_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_merge_tickets);
    if (e != cudaSuccess) return e;
    g_ticket_ptr[dev] = static_cast<unsigned int*>(p);
  }
  uint32_t pos = g_ticket_next[dev];
  if (pos + static_cast<uint32_t>(n) > kTicketSlots) pos = 0;
  g_ticket_next[dev] = pos + static_cast<uint32_t>(n);
  *out = g_ticket_ptr[dev] + pos;
  return cudaSuccess;
}
}  // namespace bw

extern "C" {

int bwattn_version(void) { return 100; }

int bwattn_last_cuda_error(void) { return t_last_cuda_error; }

uint64_t bwattn_launch_count(void) { return g_launches.load(); }

void bwattn_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1); }

const char* bwattn_status_string(int status) {
  switch (status) {
    case BWATTN_OK:
      return "ok";
    case BWATTN_ERR_INVALID_ARG:
      return "invalid argument";
    case BWATTN_ERR_UNSUPPORTED:
      return "unsupported configuration";
    case BWATTN_ERR_CUDA:
      return "CUDA error";
    case BWATTN_ERR_TIMEOUT:
      return "a kernel gave up an internal wait";
    default:
      return "unknown status";
  }
}

int bwattn_get_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned int* p = nullptr;
  if ((e = status_ptr(&p)) != cudaSuccess) return cuda_fail(e);
  unsigned int v = 0;
  if ((e = cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e);
  return (v & bw::kStatusTimeoutBit) ? BWATTN_ERR_TIMEOUT : BWATTN_OK;
}

int bwattn_clear_status(void* stream) {
  unsigned int* p = nullptr;
  cudaError_t e = status_ptr(&p);
  if (e != cudaSuccess) return cuda_fail(e);
  if ((e = cudaMemsetAsync(p, 0, sizeof(unsigned int), static_cast<cudaStream_t>(stream))) != cudaSuccess)
    return cuda_fail(e);
  return BWATTN_OK;
}

int bwattn_test_wait_timeout(void* stream) {
  unsigned int* p = nullptr;
  cudaError_t e = status_ptr(&p);
  if (e != cudaSuccess) return cuda_fail(e);
  e = bw::launch_wait_timeout_probe(g_timeout_ns.load(), p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  g_launches.fetch_add(1);
  return BWATTN_OK;
}

}  // extern "C"

namespace {

int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq, int Nk,
             int d, int causal, float scale, int dtype, int window, void* stream) {
  if (B < 0 || Nq < 0 || Nk < 0 || Hq <= 0 || Hkv <= 0 || d <= 0) return BWATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || !good_scale(scale) || (causal != 0 && causal != 1)) return BWATTN_ERR_INVALID_ARG;
  if (B > 65535 || Hq > 65535) return BWATTN_ERR_INVALID_ARG;
  if (dtype != BWATTN_DTYPE_FP32 && dtype != BWATTN_DTYPE_BF16) return BWATTN_ERR_UNSUPPORTED;
  if ((d != 64 && d != 128 && d != 256) || (d == 256 && dtype == BWATTN_DTYPE_FP32)) return BWATTN_ERR_UNSUPPORTED;
  if (B == 0 || Nq == 0) return BWATTN_OK;
  if (!q || !o || ((!k || !v) && Nk > 0)) return BWATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || (Nk > 0 && (!aligned16(k) || !aligned16(v)))) return BWATTN_ERR_INVALID_ARG;
  if (lse && !aligned4(lse)) return BWATTN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float sl2 = scale * bw::kLog2e;
  cudaError_t e;
  if (dtype == BWATTN_DTYPE_FP32) {
    bw::Fp32FwdArgs a{static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
                      static_cast<float*>(o), lse, B, Hq, Hkv, Nq, Nk, d, causal, sl2, window};
    if ((e = bw::launch_prefill_fp32(a, st)) != cudaSuccess) return cuda_fail(e);
    g_launches.fetch_add(1);
    return BWATTN_OK;
  }
  bw::TcFwdArgs a{};
  const int nk_map = Nk > 0 ? Nk : 1;
  const void* kp = Nk > 0 ? k : q;
  const void* vp = Nk > 0 ? v : q;
  if ((e = make_map(&a.tm_q, q, d, Nq, static_cast<int64_t>(B) * Hq, d, static_cast<int64_t>(Nq) * d, 128, 1)) !=
      cudaSuccess)
    return cuda_fail(e);
  const int64_t kv_heads_map = Nk > 0 ? static_cast<int64_t>(B) * Hkv : static_cast<int64_t>(B) * Hq;
  const int nk_rows = Nk > 0 ? nk_map : Nq;
  const int kv_box = d == 256 ? 64 : 128;  // keys per K/V tile
  if ((e = make_map(&a.tm_k, kp, d, nk_rows, kv_heads_map, d, static_cast<int64_t>(nk_rows) * d, kv_box, 1)) !=
      cudaSuccess)
    return cuda_fail(e);
  if ((e = make_map(&a.tm_v, vp, d, nk_rows, kv_heads_map, d, static_cast<int64_t>(nk_rows) * d, kv_box, 1)) !=
      cudaSuccess)
    return cuda_fail(e);
  a.o = static_cast<uint16_t*>(o);
  a.lse = lse;
  a.cu_q = a.cu_k = nullptr;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.causal = causal;
  a.num_seqs = B;
  a.small_rows_limit = 0;
  // items per unit: d = 256 one query tile each; below, two query tiles of one head, or (d = 128,
  // even group size) one query tile of two heads of the same KV group, whose K/V ranges are equal
  // (+7 % at N = 1024, +2.6 % at 4096, +5.5 % with a window 1024 for 32/8 heads; at d = 64, where
  // the softmax is the limit, the two tiles' softmaxes in lockstep measured 2 % slower)
  a.head_pair = d == 128 && (Hq / Hkv) % 2 == 0;
  a.max_pairs = (d == 256 || a.head_pair) ? (Nq + 127) / 128 : (Nq + 255) / 256;
  a.band_units = band_units_for(Nk, d, a.head_pair ? Hq / Hkv / 2 : Hq / Hkv);
  a.window = window;
  a.scale_log2 = sl2;
  a.timeout_ns = g_timeout_ns.load();
  unsigned int* sp = nullptr;
  unsigned int* sc = nullptr;
  if ((e = status_ptr(&sp)) != cudaSuccess) return cuda_fail(e);
  if ((e = sched_ptr(&sc)) != cudaSuccess) return cuda_fail(e);
  if ((e = (d == 256 ? bw::launch_prefill_tc256(a, sp, sc, st) : bw::launch_prefill_tc(a, sp, sc, st))) !=
      cudaSuccess)
    return cuda_fail(e);
  g_launches.fetch_add(1);
  return BWATTN_OK;
}

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
             int Nk, int d, int causal, float scale, int dtype, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, scale, dtype, 0, stream);
}

int attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Nq,
                    int Nk, int d, int window, float scale, int dtype, void* stream) {
  if (window < 1) return BWATTN_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, 1, scale, dtype, window, stream);
}

size_t attn_decode_workspace_size(int B, int Hq, int d, int num_splits) {
  if (B <= 0 || Hq <= 0 || d <= 0 || num_splits <= 0) return 0;
  // units x rows = B x Hq (rows_max = g per (sequence, KV head))
  return bw::splitk_ws_bytes(B, num_splits, Hq, d);
}

}  // extern "C"

namespace {

// The split-K launch of a decode call, then the separate merge when the splits are not merged
// by the split kernel itself.
int run_decode(bw::SplitKArgs& a, int B, int Hq, int Hkv, int g, int num_splits, const int32_t* nk, void* o,
               float* lse, cudaStream_t st) {
  a.nk = nk;
  a.num_seqs = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.g = g;
  a.num_splits = num_splits;
  a.rows_max = g;
  a.group_rows = g <= 8 ? 8 : 16;
  a.row_groups = (g + a.group_rows - 1) / a.group_rows;
  a.causal = 0;
  a.small_rows_limit = g;
  a.ws_o_offset = bw::splitk_o_offset(B * Hkv, num_splits, g);
  cudaError_t e;
  if (num_splits <= kFusedMergeMaxSplitsDecode &&
      (e = bw::merge_tickets(B * Hkv * a.row_groups, &a.tickets)) != cudaSuccess)
    return cuda_fail(e);
  a.o = static_cast<uint16_t*>(o);
  a.lse = lse;
  if ((e = status_ptr(&a.status)) != cudaSuccess) return cuda_fail(e);
  a.timeout_ns = g_timeout_ns.load();
  if ((e = bw::launch_splitk(a, st)) != cudaSuccess) return cuda_fail(e);
  g_launches.fetch_add(1);
  if (a.tickets) return BWATTN_OK;  // merged by the last CTA of each unit
  bw::MergeArgs m{};
  m.ws = a.ws;
  m.d = a.d;
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
  if ((e = bw::launch_merge(m, st)) != cudaSuccess) return cuda_fail(e);
  g_launches.fetch_add(1);
  return BWATTN_OK;
}

// Contiguous cache [B, Hkv, nk_cap, d]; bf16 (k_scale == v_scale == nullptr, fp8 false) or FP8
// E4M3 codes with per-(KV head, channel) scales.
int decode_contig(const void* q, const void* kcache, const void* vcache, const float* k_scale, const float* v_scale,
                  bool fp8, void* o, const int32_t* nk, int B, int Hq, int Hkv, int nk_cap, int d, int num_splits,
                  float scale, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || nk_cap < 0 || d <= 0) return BWATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || !good_scale(scale) || num_splits < 1 || num_splits > 1024) return BWATTN_ERR_INVALID_ARG;
  if (B > 65535) return BWATTN_ERR_INVALID_ARG;
  const int g = Hq / Hkv;
  if ((d != 64 && d != 128 && d != 256) || (fp8 && d != 128) || g > 32 || Hkv > 32767) return BWATTN_ERR_UNSUPPORTED;
  if (B == 0) return BWATTN_OK;
  if (!q || !kcache || !vcache || !o || !nk || !workspace) return BWATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) || !aligned16(workspace) ||
      !aligned4(nk) || (lse && !aligned4(lse)))
    return BWATTN_ERR_INVALID_ARG;
  if (fp8 && (!k_scale || !v_scale || !aligned16(k_scale) || !aligned16(v_scale))) return BWATTN_ERR_INVALID_ARG;
  // workspace: units = B * Hkv, rows_max = g
  if (workspace_bytes < bw::splitk_ws_bytes(B * Hkv, num_splits, g, d)) return BWATTN_ERR_INVALID_ARG;
  bw::SplitKArgs a{};
  a.d = d;
  a.q = static_cast<const uint16_t*>(q);
  if (fp8) {
    a.k8 = static_cast<const uint8_t*>(kcache);
    a.v8 = static_cast<const uint8_t*>(vcache);
    a.k_scale = k_scale;
    a.v_scale = v_scale;
  } else {
    a.k = static_cast<const uint16_t*>(kcache);
    a.v = static_cast<const uint16_t*>(vcache);
  }
  a.ws = static_cast<float*>(workspace);
  a.cu_q = a.cu_k = nullptr;
  a.kv_seq_stride = static_cast<int64_t>(Hkv) * nk_cap * d;
  a.kv_head_stride = static_cast<int64_t>(nk_cap) * d;
  a.kv_key_stride = d;
  a.kv_cap = nk_cap;
  a.total_q = a.total_k = 0;
  a.scale_log2 = scale * bw::kLog2e;
  if (!fp8 && d == 128 && g > 8 && nk_cap > 0) {
    // the 16-row form's K and V rows by TMA: {128 channels, key, sequence * KV head}, box {64, 16, 1}
    cudaError_t e;
    if ((e = make_map(&a.tm_k16, kcache, d, nk_cap, static_cast<int64_t>(B) * Hkv, d,
                      static_cast<int64_t>(nk_cap) * d, 16, 1)) != cudaSuccess ||
        (e = make_map(&a.tm_v16, vcache, d, nk_cap, static_cast<int64_t>(B) * Hkv, d,
                      static_cast<int64_t>(nk_cap) * d, 16, 1)) != cudaSuccess)
      return cuda_fail(e);
    a.tma16 = 1;
  }
  if (fp8 && nk_cap > 0) {
    // {128 codes, keys, sequence * KV head}: a box is one 16-key step of one KV head
    cudaError_t e;
    if ((e = make_map_u8(&a.tm_k8, kcache, nk_cap, static_cast<int64_t>(B) * Hkv, 128,
                         static_cast<int64_t>(nk_cap) * 128, 16, 1)) != cudaSuccess ||
        (e = make_map_u8(&a.tm_v8, vcache, nk_cap, static_cast<int64_t>(B) * Hkv, 128,
                         static_cast<int64_t>(nk_cap) * 128, 16, 1)) != cudaSuccess)
      return cuda_fail(e);
  }
  return run_decode(a, B, Hq, Hkv, g, num_splits, nk, o, lse, static_cast<cudaStream_t>(stream));
}

// Paged cache [num_pages, page_size, Hkv, d] through a block table; bf16 or FP8 as above.
int decode_paged(const void* q, const void* k_pages, const void* v_pages, const float* k_scale, const float* v_scale,
                 bool fp8, void* o, const int32_t* block_table, const int32_t* nk, int B, int Hq, int Hkv,
                 int page_size, int num_pages, int max_pages_per_seq, int d, int num_splits, float scale, float* lse,
                 void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || num_pages <= 0 || max_pages_per_seq <= 0)
    return BWATTN_ERR_INVALID_ARG;
  if (page_size < 16 || page_size > 1024 || page_size % 16 != 0) return BWATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || !good_scale(scale) || num_splits < 1 || num_splits > 1024) return BWATTN_ERR_INVALID_ARG;
  if (B > 65535 || static_cast<int64_t>(max_pages_per_seq) * page_size > 0x7fffffff) return BWATTN_ERR_INVALID_ARG;
  const int g = Hq / Hkv;
  if ((d != 64 && d != 128 && d != 256) || (fp8 && d != 128) || g > 32 || Hkv > 32767) return BWATTN_ERR_UNSUPPORTED;
  if (B == 0) return BWATTN_OK;
  if (!q || !k_pages || !v_pages || !o || !block_table || !nk || !workspace) return BWATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) || !aligned16(workspace) ||
      !aligned4(block_table) || !aligned4(nk) || (lse && !aligned4(lse)))
    return BWATTN_ERR_INVALID_ARG;
  if (fp8 && (!k_scale || !v_scale || !aligned16(k_scale) || !aligned16(v_scale))) return BWATTN_ERR_INVALID_ARG;
  if (workspace_bytes < bw::splitk_ws_bytes(B * Hkv, num_splits, g, d)) return BWATTN_ERR_INVALID_ARG;
  bw::SplitKArgs a{};
  a.d = d;
  a.q = static_cast<const uint16_t*>(q);
  if (fp8) {
    a.k8 = static_cast<const uint8_t*>(k_pages);
    a.v8 = static_cast<const uint8_t*>(v_pages);
    a.k_scale = k_scale;
    a.v_scale = v_scale;
  } else {
    a.k = static_cast<const uint16_t*>(k_pages);
    a.v = static_cast<const uint16_t*>(v_pages);
  }
  a.ws = static_cast<float*>(workspace);
  a.kv_head_stride = d;
  a.kv_key_stride = static_cast<int64_t>(Hkv) * d;
  a.scale_log2 = scale * bw::kLog2e;
  a.block_table = block_table;
  a.page_size = page_size;
  a.max_pages = max_pages_per_seq;
  a.num_pages = num_pages;
  if (fp8) {
    // {128 codes, KV head, page rows}: a box is 16 consecutive rows of one KV head inside a page
    const int64_t rows = static_cast<int64_t>(num_pages) * page_size;
    cudaError_t e;
    if ((e = make_map_u8(&a.tm_k8, k_pages, Hkv, rows, 128, static_cast<int64_t>(Hkv) * 128, 1, 16)) != cudaSuccess ||
        (e = make_map_u8(&a.tm_v8, v_pages, Hkv, rows, 128, static_cast<int64_t>(Hkv) * 128, 1, 16)) != cudaSuccess)
      return cuda_fail(e);
  }
  return run_decode(a, B, Hq, Hkv, g, num_splits, nk, o, lse, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int attn_decode(const void* q, const void* kcache, const void* vcache, void* o, const int32_t* nk, int B, int Hq,
                int Hkv, int nk_cap, int d, int num_splits, float scale, float* lse, void* workspace,
                size_t workspace_bytes, void* stream) {
  return decode_contig(q, kcache, vcache, nullptr, nullptr, false, o, nk, B, Hq, Hkv, nk_cap, d, num_splits, scale,
                       lse, workspace, workspace_bytes, stream);
}

int attn_decode_fp8(const void* q, const void* kcache, const void* vcache, const float* k_scale,
                    const float* v_scale, void* o, const int32_t* nk, int B, int Hq, int Hkv, int nk_cap, int d,
                    int num_splits, float scale, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_contig(q, kcache, vcache, k_scale, v_scale, true, o, nk, B, Hq, Hkv, nk_cap, d, num_splits, scale,
                       lse, workspace, workspace_bytes, stream);
}

int attn_decode_paged(const void* q, const void* k_pages, const void* v_pages, void* o, const int32_t* block_table,
                      const int32_t* nk, int B, int Hq, int Hkv, int page_size, int num_pages, int max_pages_per_seq,
                      int d, int num_splits, float scale, float* lse, void* workspace, size_t workspace_bytes,
                      void* stream) {
  return decode_paged(q, k_pages, v_pages, nullptr, nullptr, false, o, block_table, nk, B, Hq, Hkv, page_size,
                      num_pages, max_pages_per_seq, d, num_splits, scale, lse, workspace, workspace_bytes, stream);
}

int attn_decode_paged_fp8(const void* q, const void* k_pages, const void* v_pages, const float* k_scale,
                          const float* v_scale, void* o, const int32_t* block_table, const int32_t* nk, int B, int Hq,
                          int Hkv, int page_size, int num_pages, int max_pages_per_seq, int d, int num_splits,
                          float scale, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_paged(q, k_pages, v_pages, k_scale, v_scale, true, o, block_table, nk, B, Hq, Hkv, page_size,
                      num_pages, max_pages_per_seq, d, num_splits, scale, lse, workspace, workspace_bytes, stream);
}

size_t attn_varlen_workspace_size(int num_seqs, int max_seqlen_k, int Hq, int Hkv, int d) {
  if (num_seqs <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || max_seqlen_k < 0) return 0;
  return bw::splitk_ws_bytes(num_seqs * Hkv, varlen_splits(max_seqlen_k), kSmallRowsLimit, d);
}

}  // extern "C"

namespace {

int varlen_impl(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens_q,
                const int32_t* cu_seqlens_k, int num_seqs, int total_q, int total_k, int max_seqlen_q,
                int max_seqlen_k, int Hq, int Hkv, int d, int causal, int window, float scale, void* workspace,
                size_t workspace_bytes, void* stream) {
  if (num_seqs < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0) return BWATTN_ERR_INVALID_ARG;
  if (Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0 || !good_scale(scale) || (causal != 0 && causal != 1))
    return BWATTN_ERR_INVALID_ARG;
  if (num_seqs > 65535 || Hq > 65535) return BWATTN_ERR_INVALID_ARG;
  const int g = Hq / Hkv;
  if ((d != 64 && d != 128 && d != 256) || g > kSmallRowsLimit) return BWATTN_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_q == 0 || max_seqlen_q == 0) return BWATTN_OK;
  if (!q || !o || !cu_seqlens_q || !cu_seqlens_k || !workspace || (total_k > 0 && (!k || !v)))
    return BWATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || !aligned16(workspace) || (total_k > 0 && (!aligned16(k) || !aligned16(v))) ||
      !aligned4(cu_seqlens_q) || !aligned4(cu_seqlens_k) || (lse && !aligned4(lse)))
    return BWATTN_ERR_INVALID_ARG;
  const int splits = varlen_splits(max_seqlen_k);
  const int units = num_seqs * Hkv;
  if (workspace_bytes < bw::splitk_ws_bytes(units, splits, kSmallRowsLimit, d)) return BWATTN_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float sl2 = scale * bw::kLog2e;
  cudaError_t e;
  // 1) sequences with many queries: tcgen05 prefill kernel over the packed layout
  const bool prefill = static_cast<int64_t>(max_seqlen_q) * g > kSmallRowsLimit;
  if (prefill) {
    bw::TcFwdArgs a{};
    // with no keys at all the K/V maps are never used; they point at q so they stay valid
    const void* kp = total_k > 0 ? k : q;
    const void* vp = total_k > 0 ? v : q;
    const int hk_map = total_k > 0 ? Hkv : Hq;
    const int tk_map = total_k > 0 ? total_k : total_q;
    if ((e = make_map(&a.tm_q, q, d, Hq, total_q, d, static_cast<int64_t>(Hq) * d, 1, 128)) != cudaSuccess)
      return cuda_fail(e);
    const int kv_box = d == 256 ? 64 : 128;  // keys per K/V tile
    if ((e = make_map(&a.tm_k, kp, d, hk_map, tk_map, d, static_cast<int64_t>(hk_map) * d, 1, kv_box)) !=
        cudaSuccess)
      return cuda_fail(e);
    if ((e = make_map(&a.tm_v, vp, d, hk_map, tk_map, d, static_cast<int64_t>(hk_map) * d, 1, kv_box)) !=
        cudaSuccess)
      return cuda_fail(e);
    a.o = static_cast<uint16_t*>(o);
    a.lse = lse;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.B = num_seqs;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.Nq = total_q;
    a.Nk = total_k;
    a.d = d;
    a.causal = causal;
    a.num_seqs = num_seqs;
    a.small_rows_limit = kSmallRowsLimit;
    a.head_pair = d == 128 && g % 2 == 0;
    a.max_pairs = (d == 256 || a.head_pair) ? (max_seqlen_q + 127) / 128 : (max_seqlen_q + 255) / 256;
    a.band_units = band_units_for(max_seqlen_k, d, a.head_pair ? g / 2 : g);
    a.window = window;
    a.scale_log2 = sl2;
    a.timeout_ns = g_timeout_ns.load();
    unsigned int* sp = nullptr;
    unsigned int* sc = nullptr;
    if ((e = status_ptr(&sp)) != cudaSuccess) return cuda_fail(e);
    if ((e = sched_ptr(&sc)) != cudaSuccess) return cuda_fail(e);
    if ((e = (d == 256 ? bw::launch_prefill_tc256(a, sp, sc, st) : bw::launch_prefill_tc(a, sp, sc, st))) !=
        cudaSuccess)
      return cuda_fail(e);
    g_launches.fetch_add(1);
  }
  // 2) sequences with few queries: split-K kernel with the (query, head) rows packed, then merge
  bw::SplitKArgs s{};
  s.d = d;
  s.q = static_cast<const uint16_t*>(q);
  s.k = static_cast<const uint16_t*>(k);
  s.v = static_cast<const uint16_t*>(v);
  s.ws = static_cast<float*>(workspace);
  s.nk = nullptr;
  s.cu_q = cu_seqlens_q;
  s.cu_k = cu_seqlens_k;
  s.num_seqs = num_seqs;
  s.Hq = Hq;
  s.Hkv = Hkv;
  s.g = g;
  s.kv_seq_stride = 0;
  s.kv_head_stride = d;
  s.kv_key_stride = static_cast<int64_t>(Hkv) * d;
  s.kv_cap = 0;
  s.total_q = total_q;
  s.total_k = total_k;
  s.num_splits = splits;
  s.rows_max = kSmallRowsLimit;
  s.group_rows = kVarlenGroupRows;
  s.row_groups = kSmallRowsLimit / kVarlenGroupRows;
  s.causal = causal;
  s.window = window;
  s.small_rows_limit = kSmallRowsLimit;
  s.min_chunk = kVarlenKeysPerSplit;  // 1.6 % faster on the varlen workload than slices sized by the longest sequence
  s.ws_o_offset = bw::splitk_o_offset(units, splits, kSmallRowsLimit);
  s.scale_log2 = sl2;
  s.after_prefill = prefill ? 1 : 0;  // runs beside the prefill's last items
  if (splits <= kFusedMergeMaxSplits && (e = bw::merge_tickets(units * s.row_groups, &s.tickets)) != cudaSuccess)
    return cuda_fail(e);
  s.o = static_cast<uint16_t*>(o);
  s.lse = lse;
  if ((e = status_ptr(&s.status)) != cudaSuccess) return cuda_fail(e);
  s.timeout_ns = g_timeout_ns.load();
  if (d == 128 && window == 0 && total_k > 0) {
    // the 16-row form's K and V rows by TMA: {128 channels, KV head, token}, box {64, 1, 16}
    if ((e = make_map(&s.tm_k16, k, d, Hkv, total_k, d, static_cast<int64_t>(Hkv) * d, 1, 16)) != cudaSuccess ||
        (e = make_map(&s.tm_v16, v, d, Hkv, total_k, d, static_cast<int64_t>(Hkv) * d, 1, 16)) != cudaSuccess)
      return cuda_fail(e);
    s.tma16 = 1;
  }
  if ((e = bw::launch_splitk(s, st)) != cudaSuccess) return cuda_fail(e);
  g_launches.fetch_add(1);
  if (s.tickets) return BWATTN_OK;  // merged by the last CTA of each unit
  bw::MergeArgs m{};
  m.ws = s.ws;
  m.d = d;
  m.o = static_cast<uint16_t*>(o);
  m.lse = lse;
  m.cu_q = cu_seqlens_q;
  m.cu_k = cu_seqlens_k;
  m.nk = nullptr;
  m.num_seqs = num_seqs;
  m.Hq = Hq;
  m.Hkv = Hkv;
  m.g = g;
  m.num_splits = splits;
  m.rows_max = kSmallRowsLimit;
  m.small_rows_limit = kSmallRowsLimit;
  m.total_q = total_q;
  m.ws_o_offset = s.ws_o_offset;
  if ((e = bw::launch_merge(m, st)) != cudaSuccess) return cuda_fail(e);
  g_launches.fetch_add(1);
  return BWATTN_OK;
}

}  // namespace

extern "C" {

int attn_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens_q,
                const int32_t* cu_seqlens_k, int num_seqs, int total_q, int total_k, int max_seqlen_q,
                int max_seqlen_k, int Hq, int Hkv, int d, int causal, float scale, void* workspace,
                size_t workspace_bytes, void* stream) {
  return varlen_impl(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k, max_seqlen_q,
                     max_seqlen_k, Hq, Hkv, d, causal, 0, scale, workspace, workspace_bytes, stream);
}

int attn_varlen_window(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* cu_seqlens_q,
                       const int32_t* cu_seqlens_k, int num_seqs, int total_q, int total_k, int max_seqlen_q,
                       int max_seqlen_k, int Hq, int Hkv, int d, int window, float scale, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (window < 1) return BWATTN_ERR_INVALID_ARG;
  return varlen_impl(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k, max_seqlen_q,
                     max_seqlen_k, Hq, Hkv, d, 1, window, scale, workspace, workspace_bytes, stream);
}

}  // extern "C"
