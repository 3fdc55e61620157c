// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bw {

constexpr float kLog2e = 1.4426950408889634f;
// Bit of the device status word (owned by the C-ABI layer, passed to kernels as a pointer)
// that records a wait some kernel gave up.
constexpr unsigned int kStatusTimeoutBit = 1u;
constexpr float kLn2 = 0.6931471805599453f;

// ---- fp32 FMA prefill (any B, heads, lengths; d in {64, 128}) ----
struct Fp32FwdArgs {
  const float* q;
  const float* k;
  const float* v;
  float* o;
  float* lse;
  int B, Hq, Hkv, Nq, Nk, d, causal;
  float scale_log2;  // scale * log2(e)
  int window;        // > 0: sliding window of that many keys ending at the causal limit
};
cudaError_t launch_prefill_fp32(const Fp32FwdArgs& a, cudaStream_t stream);

// ---- split-K pass over the KV axis (decode and small-n_q varlen sequences) ----
// A "unit" is (sequence, KV head, row group); its rows are the (query, head) pairs
// r = i * g + hh of that sequence's queries and the group's query heads, group_rows (8 or 16)
// per row group.
struct SplitKArgs {
  const uint16_t* q;  // bf16 bits; token-major [tokens, Hq, D]
  const uint16_t* k;  // bf16 bits
  const uint16_t* v;
  float* ws;          // partials: (m, l) then o, see splitk_ws_layout()
  const int32_t* nk;  // dense decode: [B] valid keys per sequence (device)
  const int32_t* cu_q;  // varlen: [num_seqs + 1] (device), else null
  const int32_t* cu_k;
  int num_seqs, Hq, Hkv, g;
  int d;              // head dim D: 64 or 128 (128 with an FP8 cache)
  int64_t kv_seq_stride;  // dense: elements between sequences' caches (Hkv * cap * D)
  int64_t kv_head_stride;  // elements between KV heads at the same key (dense: cap * D, varlen: D)
  int64_t kv_key_stride;   // elements between consecutive keys (dense: D, varlen: Hkv * D)
  int kv_cap;         // dense: cache capacity (nk[b] is clamped to it)
  int total_q, total_k;  // varlen: rows of the packed tensors (cu_seqlens are clamped to them)
  int num_splits;
  int rows_max;       // workspace rows per (sequence, KV head)
  int group_rows;     // rows per row group: 8 (transposed 8-row MMA form) or 16 (16-row form)
  int row_groups;     // ceil(rows_max / group_rows)
  int causal;         // varlen: causal aligned to each sequence's end
  int window;         // varlen: > 0 adds a sliding window of that many keys
  int small_rows_limit;  // varlen: a sequence takes this path iff n_q * g <= this
  int min_chunk;         // varlen: a split takes at least this many keys (a multiple of 16; 0: none)
  size_t ws_o_offset;    // splitk_o_offset(num_seqs * Hkv, num_splits, rows_max)
  float scale_log2;
  // paged KV cache (decode only) when block_table is non-null: k, v are [num_pages, page_size,
  // Hkv, D]; key j of sequence b lives in page block_table[b * max_pages + j / page_size],
  // row j % page_size (page_size a multiple of 16, so a 16-key step never crosses a page)
  const int32_t* block_table;
  int page_size, max_pages, num_pages;
  // FP8 KV cache when k8 is non-null (k, v unused): E4M3 codes laid out like k, v; the value of
  // element (head h, channel c) is e4m3(code) * k_scale[h * D + c] (v_scale for V). tm_k8 and
  // tm_v8 are 3-D uint8 maps with a 128-byte swizzle whose box is one 16-key step of one KV
  // head: contiguous {128, cap, B * Hkv}, box {128, 16, 1}; paged {128, Hkv, pages * page_size},
  // box {128, 1, 16}
  CUtensorMap tm_k8, tm_v8;
  // bf16 16-row form at d = 128 (contiguous or packed cache, no window) when tma16 is non-zero:
  // K and V rows arrive by TMA through tm_k16 / tm_v16, 3-D bf16 maps with a 128-byte swizzle
  // whose box is 16 keys x 64 channels of one KV head: contiguous {128, cap, B * Hkv}, box
  // {64, 16, 1}; packed {128, Hkv, total_k}, box {64, 1, 16}
  CUtensorMap tm_k16, tm_v16;
  int tma16;
  const uint8_t* k8;
  const uint8_t* v8;
  const float* k_scale;
  const float* v_scale;
  // fused merge when tickets is non-null: units * row_groups zeroed counters owned by this
  // launch (left zeroed again); the last CTA of each (unit, row group) writes o and lse
  unsigned int* tickets;
  uint16_t* o;
  float* lse;
  // the FP8 instances' copies are waited for with a bounded wait (timeout_ns); one that gives up
  // sets kStatusTimeoutBit in *status (the device status word)
  unsigned int* status;
  uint64_t timeout_ns;
  // varlen: non-zero when the call's prefill kernel was launched just before on the same stream.
  // The pass reads nothing that kernel writes, so it is then a programmatic dependent launch whose
  // CTAs take the SMs the prefill's persistent CTAs leave; its last CTA waits for the prefill grid
  // to complete, so that this grid (and the work queued after it) completes after the prefill
  int after_prefill;
};
cudaError_t launch_splitk(const SplitKArgs& a, cudaStream_t stream);

struct MergeArgs {
  const float* ws;
  uint16_t* o;  // bf16 bits, token-major [tokens, Hq, D]
  float* lse;   // [tokens, Hq] or null
  const int32_t* cu_q;  // varlen or null (dense: one token per sequence)
  const int32_t* cu_k;
  const int32_t* nk;
  int num_seqs, Hq, Hkv, g, num_splits, rows_max, small_rows_limit;
  int d;  // head dim: 64 or 128
  int total_q;  // varlen: rows of the packed q / o (cu_seqlens_q is clamped to it)
  size_t ws_o_offset;
};
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream);

// ---- tcgen05 prefill (bf16, d in {64, 128, 256}) ----
struct TcFwdArgs {
  CUtensorMap tm_q, tm_k, tm_v;  // 3-D maps, box {64, 1 or 128 (d = 256 K/V: 64), ...}, 128-byte swizzle
  uint16_t* o;
  float* lse;
  const int32_t* cu_q;  // varlen (packed) mode if non-null
  const int32_t* cu_k;
  int B, Hq, Hkv, Nq, Nk, d, causal;  // packed mode: Nq, Nk = total rows of q and k
  int num_seqs;
  int small_rows_limit;  // varlen: sequences with n_q * g <= this are skipped here
  int max_pairs;         // work items per (sequence, head): pairs of 128-row query tiles (d = 256: tiles)
  int window;            // > 0: sliding window of that many keys ending at the causal limit
  int band_units;        // (sequence, head) units per band of the item list (at least 1)
  int head_pair;         // d = 128, even g: a work item is one query tile of two heads that share
                         // a KV head (units are head pairs, max_pairs counts query tiles)
  float scale_log2;
  uint64_t timeout_ns;
};
// `sched`: two zeroed device counters (next item, CTAs finished) owned by this launch alone;
// the kernel leaves them zeroed again when it completes.
cudaError_t launch_prefill_tc(const TcFwdArgs& a, unsigned int* status, unsigned int* sched, cudaStream_t stream);
// Head dim 256: one 128-row query tile per item, 64-key K/V tiles (the K/V maps' box is 64 rows
// or tokens high), a.max_pairs = query tiles per (sequence, head).
cudaError_t launch_prefill_tc256(const TcFwdArgs& a, unsigned int* status, unsigned int* sched, cudaStream_t stream);

// Timeout self-test: one CTA waits on a barrier that is never arrived at.
cudaError_t launch_wait_timeout_probe(uint64_t timeout_ns, unsigned int* status, cudaStream_t stream);

// Bookkeeping shared by every entry point (defined in api.cu): record a failed CUDA call for
// bwattn_last_cuda_error(), count a successful launch for bwattn_launch_count().
void record_cuda_error(cudaError_t e);
void count_launch();
// `n` zeroed merge tickets on the current device for one launch of the split-K kernel (null
// when the request exceeds the ticket pool: the caller then launches the merge kernel).
cudaError_t merge_tickets(int n, unsigned int** out);

// Float offset of the o[] block of the split-K workspace (after the (m, l) pairs, 256-byte aligned).
inline size_t splitk_o_offset(int units, int num_splits, int rows_max) {
  return (static_cast<size_t>(units) * num_splits * rows_max * 2 + 63) & ~static_cast<size_t>(63);
}
inline size_t splitk_ws_bytes(int units, int num_splits, int rows_max, int d) {
  return (splitk_o_offset(units, num_splits, rows_max) + static_cast<size_t>(units) * num_splits * rows_max * d) *
         sizeof(float);
}

}  // namespace bw
