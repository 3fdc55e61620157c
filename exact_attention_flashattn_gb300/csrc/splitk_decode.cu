// Split-K attention over the KV axis for few query rows (single-query decode, and the
// short-query sequences of a packed varlen batch), plus the merge of the per-split partial
// states.
//
// Method ("Attention from the kernel's side", Prefill and decode are different problems;
// "Attention kernels", Concept and Maths): the keys of one (sequence, KV head) are cut into
// num_splits slices; each CTA folds its slice into partial states (m, l, o) with the
// online-softmax recurrence and writes them out; a second kernel merges the partials with
// m = max_s m_s, l = sum_s l_s e^{m_s - m}, o = sum_s o_s e^{m_s - m}, and divides.
//
// Layout of the work: a CTA owns one slice for up to 16 "rows", a row being one (query,
// query head) pair of the GQA group that shares the KV head ("Attention Computation in
// Practice", GQA in the kernel), so every K/V byte the CTA reads serves all those rows.
// The two contractions per 16 keys are warp-level bf16 tensor-core MMAs (m16n8k16, fp32
// accumulate): S = Q K^T with the rows as M, then O += P V with the keys as K. Cache reads
// are 16-byte vector loads straight into registers. To make them line up with the MMA
// fragment layout without shared memory, the head-dim index is permuted identically on Q
// and K (a permutation of the contraction index leaves the dot product unchanged), and the
// output-channel index of the P V product is permuted and undone at the write. When a row
// group has at most 8 rows (GQA groups of up to 8 heads) the products are taken transposed:
// S^T = K Q^T with the 16 keys of a step as the MMA rows and the group's heads as the 8 columns,
// then O^T += V^T P^T with 16 head-dim channels as the rows; P^T reaches the operand layout by an
// in-register 8x8 transpose (movmatrix). Half the MMAs of the 16-row form, none of them padding.
//
// FP8 KV cache ("Attention from the kernel's side", Why a quantised cache needs a fused kernel:
// the codes are turned into values inside the tile load, so HBM carries only the codes): the
// cache holds E4M3 codes with a per-(KV head, channel) scale. Each 16-byte load brings 16
// codes; `cvt.rn.f16x2.e4m3x2` turns code pairs into f16 pairs exactly (every E4M3 value is an
// f16 value) and the contractions run as f16 MMAs. The K scale is folded into Q once per CTA
// (s = sum_c (q_c k_scale_c) code_c), with a per-row power of two that keeps q * k_scale in
// f16 range and is given back in the row's score scale; the V scale multiplies each output
// channel of the partial o (o_c = v_scale_c sum_j p_j code_jc).
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bw {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerGroup = 16;
constexpr int kKeysPerStep = 16;
// FP8 cache: each warp's 16-key steps (2 KB of K codes, 2 KB of V codes) arrive by TMA in a ring
// of kFp8Stages shared-memory stages per warp, one mbarrier per stage, so that the bytes in
// flight are bounded by shared memory rather than registers and one lane issues a step's copies
constexpr int kFp8Stages = 3;
constexpr uint32_t kFp8WarpStepBytes = 2 * kKeysPerStep * 128;  // K box + V box
constexpr uint32_t kFp8StageBytes = kWarps * kFp8WarpStepBytes;
constexpr uint32_t kFp8RingBytes = kFp8Stages * kFp8StageBytes;
constexpr uint32_t kFp8SmemBytes = kFp8RingBytes + 1024;  // + slack to align the ring to 1024 B
// bf16 16-row form at d = 128 (varlen short-query sequences, decode with g > 8) with the TMA ring:
// 8 KB per warp step, two stages
constexpr int kT16Stages = 2;
constexpr uint32_t kT16WarpStepBytes = 2 * 2 * kKeysPerStep * 128;
constexpr uint32_t kT16StageBytes = kWarps * kT16WarpStepBytes;
constexpr uint32_t kT16SmemBytes = kT16Stages * kT16StageBytes + 1024;  // + slack to align the ring
constexpr int kMergeThreads = 256;
constexpr int kMergeMaxSplits = 1024;  // the entry points accept at most this many splits

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}


__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}


// Four E4M3 codes (bytes 0..3) to two f16 pairs: bytes 0,1 -> lo, bytes 2,3 -> hi; exact.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t codes, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(codes));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// 8x8 transpose of a b16 matrix held one row pair per thread (mma accumulator layout).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

__device__ __forceinline__ uint32_t word(const uint4& v, int w) {
  return w == 0 ? v.x : (w == 1 ? v.y : (w == 2 ? v.z : v.w));
}

// Output channel held by MMA column position p (0..7) of output n-tile nu (0..D/8 - 1).
__device__ __forceinline__ int dv_of(int nu, int p) { return (nu < 8) ? (8 * p + nu) : (64 + 8 * p + (nu - 8)); }
// Transposed form: the channels held by rows gr (A) and gr + 8 (B) of output m-tile mu. d = 128:
// va (channels 8 gr .. 8 gr + 7) feeds the A rows, vb (64 + 8 gr ..) the B rows; d = 64 has va
// only, so its lo / hi halves feed the A / B rows: channels 8 gr + 2 mu and 8 gr + 2 mu + 1.
template <int D>
__device__ __forceinline__ int chA_of(int gr, int mu) { return D == 128 ? 8 * gr + mu : 8 * gr + 2 * mu; }
template <int D>
__device__ __forceinline__ int chB_of(int gr, int mu) { return D == 128 ? 64 + 8 * gr + mu : 8 * gr + 2 * mu + 1; }
// The same for the FP8 cache, whose V loads are 16-channel chunks: column p of n-tile nu is
// channel 16 p + nu.
__device__ __forceinline__ int dv8_of(int nu, int p) { return 16 * p + nu; }

struct UnitGeom {
  int tok0;     // first query token of the sequence
  int nq;       // queries of the sequence
  int nk;       // keys of the sequence
  int k0;       // varlen: token index of the sequence's first key (0 otherwise)
  int64_t kv0;  // element offset of key 0 of this KV head
  bool active;
};

__device__ __forceinline__ UnitGeom unit_geom(const SplitKArgs& a, int seq, int hkv) {
  UnitGeom u;
  if (a.cu_q) {
    // lengths come from device arrays: clamp them to the packed tensors so no access leaves them
    u.tok0 = min(max(a.cu_q[seq], 0), a.total_q);
    u.nq = min(max(a.cu_q[seq + 1] - u.tok0, 0), a.total_q - u.tok0);
    const int k0 = min(max(a.cu_k[seq], 0), a.total_k);
    u.k0 = k0;
    u.nk = min(max(a.cu_k[seq + 1] - k0, 0), a.total_k - k0);
    u.kv0 = static_cast<int64_t>(k0) * a.kv_key_stride + static_cast<int64_t>(hkv) * a.kv_head_stride;
    u.active = u.nq > 0 && u.nq * a.g <= a.small_rows_limit;
  } else if (a.block_table) {
    // paged cache: kv0 is the head's offset inside a page row; pages come from the block table
    u.tok0 = seq;
    u.nq = 1;
    u.k0 = 0;
    u.nk = min(max(a.nk[seq], 0), a.max_pages * a.page_size);
    u.kv0 = static_cast<int64_t>(hkv) * a.kv_head_stride;
    u.active = true;
  } else {
    u.tok0 = seq;
    u.nq = 1;
    u.k0 = 0;
    u.nk = min(max(a.nk[seq], 0), a.kv_cap);
    u.kv0 = static_cast<int64_t>(seq) * a.kv_seq_stride + static_cast<int64_t>(hkv) * a.kv_head_stride;
    u.active = true;
  }
  return u;
}

// Element offset of the first key row of the 16-key step starting at key kb (relative to the
// unit's kv0): contiguous caches step by rows, paged caches look the page up in the block
// table ("Attention Computation in Practice", PagedAttention's kernel difference).
template <bool kPaged>
__device__ __forceinline__ int64_t step_offset(const SplitKArgs& a, int seq, int kb) {
  if constexpr (!kPaged) return static_cast<int64_t>(kb) * a.kv_key_stride;
  int page = a.block_table[static_cast<int64_t>(seq) * a.max_pages + kb / a.page_size];
  page = min(max(page, 0), a.num_pages - 1);  // a bad entry reads a wrong page, never outside the pool
  return (static_cast<int64_t>(page) * a.page_size + kb % a.page_size) * a.kv_key_stride;
}

// Workspace: for unit (seq, hkv), split s, row r: ml[2] then o[D] are stored as
//   ml: ws[((unit * S + s) * rows_max + r) * 2 + {0, 1}]
//   o : ws[ws_o_offset + ((unit * S + s) * rows_max + r) * D + c]
__device__ __forceinline__ size_t ws_ml_index(const SplitKArgs& a, int unit, int s, int r) {
  return ((static_cast<size_t>(unit) * a.num_splits + s) * a.rows_max + r) * 2;
}

// d = 256: the two warps of a pair (key group kg = 0 or 1) add their partial score tiles, 4 * NH
// scores per lane. Each warp writes its values into its half of the step's slot, meets its
// partner at the pair's named barrier (id 1 + kg, 64 threads) and adds the partner's values; a + b is the
// same float in both warps, so both take the same softmax. The slots alternate with the step
// parity: a warp rewrites a slot two steps later, after the barrier of the step in between,
// which its partner reaches only once it has read that slot.
template <int NH>
__device__ __forceinline__ void pair_sum(float4 (&slot)[2][32][NH], int half, int lane, int kg,
                                         float (&v)[4 * NH]) {
#pragma unroll
  for (int i = 0; i < NH; ++i) slot[half][lane][i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  if (kg == 0)
    asm volatile("bar.sync 1, 64;" ::: "memory");
  else
    asm volatile("bar.sync 2, 64;" ::: "memory");
#pragma unroll
  for (int i = 0; i < NH; ++i) {
    const float4 o = slot[half ^ 1][lane][i];
    v[4 * i] += o.x;
    v[4 * i + 1] += o.y;
    v[4 * i + 2] += o.z;
    v[4 * i + 3] += o.w;
  }
}

// D = head dim (64, 128 or 256; the FP8 cache is 128 only);
// NH = number of 8-row halves of the 16-row MMA tile that carry real rows (1 or 2);
// kPaged: keys are gathered page by page through the block table; kWindow: causal sliding
// window (a separate instance, so the plain causal and paged paths carry no window registers);
// kFp8: FP8 E4M3 cache with per-channel scales (k8, v8, k_scale, v_scale).
template <int D, int NH, bool kPaged, bool kWindow, bool kFp8, bool kTma16 = false>
__global__ void __launch_bounds__(kThreads, NH == 1 ? 4 : 3) splitk_kernel(const __grid_constant__ SplitKArgs a) {
  static_assert(D == 64 || D == 128 || D == 256, "head dim");
  static_assert(!kFp8 || D == 128, "the FP8 cache layout is d = 128");
  static_assert(!kTma16 || (D == 128 && NH == 2 && !kPaged && !kWindow && !kFp8), "TMA ring: 16-row form, d = 128");
  // d = 256: the warps work in pairs on the same 16-key steps, each warp holding 128 of the
  // channels of Q, K, V and O; the pair adds its two partial score tiles through shared memory,
  // so both warps take the same softmax and each accumulates its own half of O
  constexpr bool kPair = D == 256;
  constexpr int DW = kPair ? 128 : D;       // channels per warp
  constexpr int kKG = kPair ? kWarps / 2 : kWarps;  // key groups (warps or warp pairs) per CTA
  constexpr int kSteps = DW / 16;  // k16 steps of S = Q K^T over the warp's channels
  constexpr int kNT = DW / 8;      // output n8 tiles of O (16-row form); 8-row pairs of them transposed
  extern __shared__ __align__(16) uint8_t dsm[];  // FP8: the load ring, then the combine buffer
  // a dependent merge launch may be scheduled from now on (it waits for this grid to complete)
  asm volatile("griddepcontrol.launch_dependents;");
  // after a prefill launch this grid may start before that one completes (it reads nothing the
  // prefill writes); its last CTA waits for it, so that this grid completes after the prefill
  if (a.after_prefill && blockIdx.x == gridDim.x - 1 && blockIdx.y == gridDim.y - 1 && blockIdx.z == gridDim.z - 1)
    asm volatile("griddepcontrol.wait;" ::: "memory");
  // paged caches hold every KV head of a token in one row of a page: their grid runs the heads
  // fastest, so the CTAs that read the same pages run at the same time
  const int split = kPaged ? blockIdx.y : blockIdx.x;
  const int hg = kPaged ? blockIdx.x : blockIdx.y;
  const int hkv = hg % a.Hkv;
  const int grp = hg / a.Hkv;
  const int seq = blockIdx.z;
  const UnitGeom u = unit_geom(a, seq, hkv);
  if (!u.active) return;
  const int R = u.nq * a.g;
  const int row0 = grp * 8 * NH;
  if (row0 >= R) return;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = lane & 3, gr = lane >> 2;
  const int kg = kPair ? warp >> 1 : warp;           // this warp's key group
  const int hoff = kPair ? 128 * (warp & 1) : 0;     // first channel this warp holds

  // Key slice of this split: whole 16-key steps, at least min_chunk keys (varlen: the splits of a
  // short sequence past its last key are empty partials)
  const int per = (u.nk + a.num_splits - 1) / a.num_splits;
  const int chunk = max((per + kKeysPerStep - 1) / kKeysPerStep * kKeysPerStep, a.min_chunk);
  const int kbeg = min(u.nk, split * chunk);
  const int kend = min(u.nk, kbeg + chunk);

  // Rows gr (and gr + 8) of this group: (query i, head hh) and their key limits [lo, lim).
  int lim[2], lo[2];
  uint32_t qa[kSteps][4];
  float sl2[2] = {a.scale_log2, a.scale_log2};  // FP8: the row's score scale (see below)
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int r = row0 + gr + 8 * rr;
    const bool ok = rr < NH && r < R;
    const int i = ok ? r / a.g : 0;
    const int hh = ok ? r % a.g : 0;
    lim[rr] = a.causal ? min(kend, u.nk - u.nq + i + 1) : kend;
    lo[rr] = kWindow ? u.nk - u.nq + i + 1 - a.window : 0;
    if (!ok) {
      lim[rr] = kend;
      lo[rr] = 0;
    }
    const uint16_t* qrow = a.q + (static_cast<int64_t>(u.tok0 + i) * a.Hq + hkv * a.g + hh) * D + hoff;
    if constexpr (!kFp8) {
#pragma unroll
      for (int s = 0; s < DW / 32; ++s) {
        uint4 c = make_uint4(0, 0, 0, 0);
        if (ok) c = *reinterpret_cast<const uint4*>(qrow + 8 * (t + 4 * s));
        // k-step 2s uses words 0,1 of chunk t+4s; k-step 2s+1 words 2,3 (same permutation as K)
        qa[2 * s][rr] = c.x;
        qa[2 * s][rr + 2] = c.y;
        qa[2 * s + 1][rr] = c.z;
        qa[2 * s + 1][rr + 2] = c.w;
      }
    } else {
      // this thread's K loads are the 16-code chunks t and t + 4, so it holds q * k_scale for
      // channels 16t..16t+15 (k-steps 0..3) and 16(t+4)..16(t+4)+15 (k-steps 4..7)
      float qs[32];
      const float* ksc = a.k_scale + hkv * D;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int c0 = 16 * (t + 4 * hf);
#pragma unroll
        for (int s8 = 0; s8 < 2; ++s8) {
          uint4 c = make_uint4(0, 0, 0, 0);
          if (ok) c = *reinterpret_cast<const uint4*>(qrow + c0 + 8 * s8);
          const float4 k0 = *reinterpret_cast<const float4*>(ksc + c0 + 8 * s8);
          const float4 k1 = *reinterpret_cast<const float4*>(ksc + c0 + 8 * s8 + 4);
          const uint32_t wv[4] = {c.x, c.y, c.z, c.w};
          const float kv[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint32_t bits = (e & 1) ? (wv[e >> 1] & 0xFFFF0000u) : (wv[e >> 1] << 16);
            qs[16 * hf + 8 * s8 + e] = __uint_as_float(bits) * kv[e];
          }
        }
      }
      // row scale 2^e so that max |q * k_scale| * 2^-e lies in [8, 16): f16 keeps 11 bits of
      // every significant product and cannot overflow; the scores get the 2^e back
      float amax = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(qs[e]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      int ex = 0;
      if (amax > 0.f && amax <= 3.0e38f) {
        frexpf(amax, &ex);
        ex = min(max(ex - 4, -120), 120);
      }
      const float down = __int_as_float((127 - ex) << 23);  // 2^-ex
      sl2[rr] = a.scale_log2 * __int_as_float((127 + ex) << 23);
#pragma unroll
      for (int kst = 0; kst < 8; ++kst) {
        const int b = 16 * (kst >> 2) + 4 * (kst & 3);
        qa[kst][rr] = pack_f16x2(qs[b] * down, qs[b + 1] * down);
        qa[kst][rr + 2] = pack_f16x2(qs[b + 2] * down, qs[b + 3] * down);
      }
    }
  }
  // transposed form (NH == 1): this thread's scores belong to rows 2t and 2t+1 of the group
  int limT[2], loT[2];
  float sl2T[2];
  if constexpr (NH == 1) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int r = row0 + 2 * t + j;
      const bool ok = r < R;
      const int i = ok ? r / a.g : 0;
      limT[j] = ok ? (a.causal ? min(kend, u.nk - u.nq + i + 1) : kend) : kend;
      loT[j] = (ok && kWindow) ? u.nk - u.nq + i + 1 - a.window : 0;
      // FP8: row 2t+j's Q was normalised by the lanes holding that row (gr = 2t + j)
      sl2T[j] = kFp8 ? __shfl_sync(0xffffffffu, sl2[0], (2 * t + j) * 4) : a.scale_log2;
    }
  }
  // lowest key limit over the CTA's rows: steps ending at or below it need no mask
  int min_lim = kend;
  if (a.causal) min_lim = min(kend, u.nk - u.nq + row0 / a.g + 1);
  // with a sliding window: keys below the first row's window start are skipped (whole 16-key
  // steps, so the step grid is kept), and steps starting below the last row's start are masked
  int kstart = kbeg;
  int max_lo = 0;
  if constexpr (kWindow) {
    kstart = max(kbeg, (u.nk - u.nq + row0 / a.g + 1 - a.window) / kKeysPerStep * kKeysPerStep);
    const int last_r = min(row0 + 8 * NH, R) - 1;
    max_lo = u.nk - u.nq + last_r / a.g + 1 - a.window;
  }

  float oacc[kNT][2 * NH];
#pragma unroll
  for (int nu = 0; nu < kNT; ++nu)
#pragma unroll
    for (int c = 0; c < 2 * NH; ++c) oacc[nu][c] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_part[2] = {0.f, 0.f};

  const uint16_t* kbase = a.k + u.kv0;
  const uint16_t* vbase = a.v + u.kv0;
  const uint8_t* kbase8 = a.k8 + u.kv0;
  const uint8_t* vbase8 = a.v8 + u.kv0;
  const int64_t ks = a.kv_key_stride;

  // ---- scale (log2 units), mask, row max over the quad, online-softmax update of one 16-key
  // step starting at key kb; returns the A fragment of P (rows x 16 keys)
  auto softmax_step = [&](int kb, float (&sacc)[2][4], uint32_t (&pa)[4]) {
    bool need_mask = kb + kKeysPerStep > min_lim;
    if constexpr (kWindow) need_mask = need_mask || kb < max_lo;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int c = 0; c < 2 * NH; ++c) {
        const int rr = c >> 1;
        float s = sacc[nt][c] * (kFp8 ? sl2[rr] : a.scale_log2);
        if (need_mask) {
          const int key = kb + nt * 8 + 2 * t + (c & 1);
          if (key >= lim[rr] || (kWindow && key < lo[rr])) s = -INFINITY;
        }
        sacc[nt][c] = s;
        mx[rr] = fmaxf(mx[rr], s);
      }
#pragma unroll
    for (int rr = 0; rr < NH; ++rr) {
      mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
      mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
    }
    // O is rescaled only when some row's max grew
    float mnew[2], muse[2];
    bool grow = false;
#pragma unroll
    for (int rr = 0; rr < NH; ++rr) {
      mnew[rr] = fmaxf(m_run[rr], mx[rr]);
      grow |= mnew[rr] > m_run[rr];
      muse[rr] = (mnew[rr] == -INFINITY) ? 0.f : mnew[rr];
    }
    if (__any_sync(0xffffffffu, grow)) {
      float al[2];
#pragma unroll
      for (int rr = 0; rr < NH; ++rr) {
        al[rr] = (m_run[rr] == -INFINITY) ? 0.f : ex2(m_run[rr] - muse[rr]);
        l_part[rr] *= al[rr];
      }
#pragma unroll
      for (int nu = 0; nu < kNT; ++nu)
#pragma unroll
        for (int c = 0; c < 2 * NH; ++c) oacc[nu][c] *= al[c >> 1];
    }
#pragma unroll
    for (int rr = 0; rr < NH; ++rr) m_run[rr] = mnew[rr];
    float p[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int c = 0; c < 2 * NH; ++c) {
        p[nt][c] = ex2(sacc[nt][c] - muse[c >> 1]);
        l_part[c >> 1] += p[nt][c];
      }
    // k positions 2t,2t+1 from tile 0, 2t+8,2t+9 from tile 1 (f16 for the FP8 cache)
    pa[0] = kFp8 ? pack_f16x2(p[0][0], p[0][1]) : pack_bf16x2(p[0][0], p[0][1]);
    pa[2] = kFp8 ? pack_f16x2(p[1][0], p[1][1]) : pack_bf16x2(p[1][0], p[1][1]);
    if constexpr (NH == 2) {
      pa[1] = kFp8 ? pack_f16x2(p[0][2], p[0][3]) : pack_bf16x2(p[0][2], p[0][3]);
      pa[3] = kFp8 ? pack_f16x2(p[1][2], p[1][3]) : pack_bf16x2(p[1][2], p[1][3]);
    } else {
      pa[1] = pa[3] = 0u;
    }
  };

  // Transposed form: scores st = S^T (c0: key gr, row 2t; c1: key gr, row 2t+1; c2, c3: key
  // gr + 8); the row max runs over the 8 lanes of equal t. Returns the B fragment of P^T.
  auto softmax_stepT = [&](int kb, float (&st)[4], uint32_t& b0, uint32_t& b1) {
    bool need_mask = kb + kKeysPerStep > min_lim;
    if constexpr (kWindow) need_mask = need_mask || kb < max_lo;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = c & 1;
      float s = st[c] * sl2T[j];
      if (need_mask) {
        const int key = kb + gr + 8 * (c >> 1);
        if (key >= limT[j] || (kWindow && key < loT[j])) s = -INFINITY;
      }
      st[c] = s;
    }
    float mx[2] = {fmaxf(st[0], st[2]), fmaxf(st[1], st[3])};
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 4));
      mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 8));
      mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 16));
    }
    float mnew[2], muse[2];
    bool grow = false;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      mnew[j] = fmaxf(m_run[j], mx[j]);
      grow |= mnew[j] > m_run[j];
      muse[j] = (mnew[j] == -INFINITY) ? 0.f : mnew[j];
    }
    if (__any_sync(0xffffffffu, grow)) {
      float al[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        al[j] = (m_run[j] == -INFINITY) ? 0.f : ex2(m_run[j] - muse[j]);
        l_part[j] *= al[j];
      }
#pragma unroll
      for (int nu = 0; nu < kNT; ++nu)
#pragma unroll
        for (int c = 0; c < 2; ++c) oacc[nu][c] *= al[c];
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) m_run[j] = mnew[j];
    float p[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      p[c] = ex2(st[c] - muse[c & 1]);
      l_part[c & 1] += p[c];
    }
    // P^T of keys gr (and gr + 8) for rows 2t, 2t+1 -> transposed: row gr, keys 2t, 2t+1 (2t+8, 2t+9)
    b0 = movmatrix_trans(kFp8 ? pack_f16x2(p[0], p[1]) : pack_bf16x2(p[0], p[1]));
    b1 = movmatrix_trans(kFp8 ? pack_f16x2(p[2], p[3]) : pack_bf16x2(p[2], p[3]));
  };

  if constexpr (!kFp8) {
    // d = 256: the pairs' exchange slots [key group][step parity][warp of the pair][lane]
    __shared__ float4 xch[kKG][2][2][32][NH];
    // one 16-key step from its K and V fragments: the two contractions and the softmax update
    auto compute_bf16 = [&](int kb, int step, const uint4 (&kk)[2][DW / 32], const uint4 (&va)[4],
                            const uint4 (&vb)[4]) {
      if constexpr (NH == 1) {
        // ---- S^T = K Q^T: rows = keys gr / gr + 8 (the two K rows this thread loaded), DW/16
        // k16 steps over the warp's channels; Q is the B operand (row gr of the group)
        float st[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kst = 0; kst < kSteps; ++kst) {
          const uint4& r0 = kk[0][kst >> 1];
          const uint4& r1 = kk[1][kst >> 1];
          const uint32_t af[4] = {(kst & 1) ? r0.z : r0.x, (kst & 1) ? r1.z : r1.x, (kst & 1) ? r0.w : r0.y,
                                  (kst & 1) ? r1.w : r1.y};
          mma_bf16(st, af, qa[kst][0], qa[kst][2]);
        }
        if constexpr (kPair) pair_sum<NH>(xch[kg][step & 1], warp & 1, lane, kg, st);
        uint32_t b0, b1;
        softmax_stepT(kb, st, b0, b1);
        // ---- O^T += V^T P^T over DW/16 channel tiles: tile mu, rows gr and gr + 8 = channels
        // hoff + chA_of(gr, mu) and hoff + chB_of(gr, mu); keys 2t, 2t+1 | 2t+8, 2t+9
#pragma unroll
        for (int mu = 0; mu < DW / 16; ++mu) {
          uint32_t af[4];
          if constexpr (DW == 128) {
            const int w = mu >> 1;
            const uint32_t sel = (mu & 1) ? 0x7632u : 0x5410u;
            af[0] = __byte_perm(word(va[0], w), word(va[1], w), sel);
            af[1] = __byte_perm(word(vb[0], w), word(vb[1], w), sel);
            af[2] = __byte_perm(word(va[2], w), word(va[3], w), sel);
            af[3] = __byte_perm(word(vb[2], w), word(vb[3], w), sel);
          } else {
            af[0] = __byte_perm(word(va[0], mu), word(va[1], mu), 0x5410u);
            af[1] = __byte_perm(word(va[0], mu), word(va[1], mu), 0x7632u);
            af[2] = __byte_perm(word(va[2], mu), word(va[3], mu), 0x5410u);
            af[3] = __byte_perm(word(va[2], mu), word(va[3], mu), 0x7632u);
          }
          float(&acc)[4] = *reinterpret_cast<float(*)[4]>(&oacc[2 * mu][0]);
          mma_bf16(acc, af, b0, b1);
        }
      } else {
        // ---- S = Q K^T for 16 keys: two n8 tiles, D/16 k16 steps over the head dim
        float sacc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
          for (int kst = 0; kst < kSteps; ++kst) {
            const uint4& c = kk[nt][kst >> 1];
            const uint32_t b0 = (kst & 1) ? c.z : c.x;
            const uint32_t b1 = (kst & 1) ? c.w : c.y;
            mma_bf16(sacc[nt], qa[kst], b0, b1);
          }
        }
        if constexpr (kPair) pair_sum<NH>(xch[kg][step & 1], warp & 1, lane, kg, *reinterpret_cast<float(*)[8]>(&sacc[0][0]));
        uint32_t pa[4];
        softmax_step(kb, sacc, pa);
        // ---- O += P V over DW/8 output n-tiles
#pragma unroll
        for (int nu = 0; nu < kNT; ++nu) {
          const int e = nu & 7;
          const int w = e >> 1;
          const uint32_t sel = (e & 1) ? 0x7632u : 0x5410u;
          const uint32_t w0 = word((nu < 8) ? va[0] : vb[0], w), w1 = word((nu < 8) ? va[1] : vb[1], w);
          const uint32_t w2 = word((nu < 8) ? va[2] : vb[2], w), w3 = word((nu < 8) ? va[3] : vb[3], w);
          float(&acc)[4] = *reinterpret_cast<float(*)[4]>(&oacc[nu][0]);
          mma_bf16(acc, pa, __byte_perm(w0, w1, sel), __byte_perm(w2, w3, sel));
        }
      }
    };
    if constexpr (kTma16) {
      // 16-row form at d = 128 over a contiguous or packed cache: each warp's steps arrive by TMA
      // (one lane issues 4 boxes of 16 key rows x 64 channels: K and V, two channel halves each,
      // 128-byte swizzle) in a kT16Stages-deep ring of the warp's own stages, so that a warp has
      // the next step's 8 KB in flight while it computes this one, and the fragments live in
      // registers only while they are used
      __shared__ __align__(8) uint64_t t16_full[kWarps][kT16Stages];
      uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
      if (lane == 0) {
        for (int s2 = 0; s2 < kT16Stages; ++s2) mbar_init(&t16_full[warp][s2], 1);
        fence_mbar_init();
      }
      __syncwarp();
      auto stage_ptr = [&](int s2) { return ring + s2 * kT16StageBytes + warp * kT16WarpStepBytes; };
      const bool packed = a.cu_q != nullptr;
      auto issue = [&](int kb, int s2) {
        if (kb >= kend) return;
        uint8_t* dst = stage_ptr(s2);
        mbar_arrive_expect_tx(&t16_full[warp][s2], kT16WarpStepBytes);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // boxes: K half 0, K half 1, V half 0, V half 1 (2 KB each)
          if (packed) {
            tma_load_3d(dst + h * 2048, &a.tm_k16, &t16_full[warp][s2], 64 * h, hkv, u.k0 + kb);
            tma_load_3d(dst + 4096 + h * 2048, &a.tm_v16, &t16_full[warp][s2], 64 * h, hkv, u.k0 + kb);
          } else {
            tma_load_3d(dst + h * 2048, &a.tm_k16, &t16_full[warp][s2], 64 * h, kb, seq * a.Hkv + hkv);
            tma_load_3d(dst + 4096 + h * 2048, &a.tm_v16, &t16_full[warp][s2], 64 * h, kb, seq * a.Hkv + hkv);
          }
        }
      };
      // 8 channels (16 bytes) at chunk c (0..15) of row r: box half c / 8, swizzled chunk c % 8
      auto ld_row = [&](const uint8_t* box, int r, int c) {
        uint4 v;
        const uint32_t addr = smem_u32(box + (c >> 3) * 2048) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"(addr));
        return v;
      };
      constexpr int kStride = kWarps * kKeysPerStep;
      const int no_abort = 0;
      bool timed_out = false;
      int kb_next = kstart + warp * kKeysPerStep;
#pragma unroll
      for (int s2 = 0; s2 < kT16Stages - 1; ++s2) {
        issue(kb_next, s2);
        kb_next += kStride;
      }
      int st = 0, n = 0;
      for (int kb = kstart + warp * kKeysPerStep; kb < kend; kb += kStride, ++n) {
        __syncwarp();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        issue(kb_next, st == 0 ? kT16Stages - 1 : st - 1);
        kb_next += kStride;
        if (!__all_sync(0xffffffffu, mbar_wait(&t16_full[warp][st], (n / kT16Stages) & 1, a.timeout_ns, &no_abort))) {
          if (lane == 0 && a.status) atomicOr(a.status, kStatusTimeoutBit);
          timed_out = true;
          break;
        }
        const uint8_t* kbox = stage_ptr(st);
        const uint8_t* vbox = kbox + 4096;
        uint4 kk[2][DW / 32], va[4], vb[4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int s3 = 0; s3 < DW / 32; ++s3) kk[nt][s3] = ld_row(kbox, nt * 8 + gr, t + 4 * s3);
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int r = 2 * t + (x & 1) + 8 * (x >> 1);
          va[x] = ld_row(vbox, r, gr);
          vb[x] = ld_row(vbox, r, 8 + gr);
          // rows past the slice hold other keys (possibly NaN or inf): their P is 0, and 0 * NaN
          // would still reach O, so their values are zeroed (their scores are masked)
          if (kb + r >= kend) va[x] = vb[x] = make_uint4(0u, 0u, 0u, 0u);
        }
        st = (st + 1 == kT16Stages) ? 0 : st + 1;
        compute_bf16(kb, n, kk, va, vb);
      }
      // after a timed-out wait, the copies issued past it must land (bounded) before the ring is
      // reused for the combine below; otherwise every issued step was consumed
      if (timed_out) {
        for (int m = n; m < n + kT16Stages; ++m) {
          const int kbm = kstart + warp * kKeysPerStep + m * kStride;
          if (kbm < kend) mbar_wait(&t16_full[warp][m % kT16Stages], (m / kT16Stages) & 1, a.timeout_ns, &no_abort);
        }
      }
    } else {
      int step = 0;
      for (int kb = kstart + kg * kKeysPerStep; kb < kend; kb += kKG * kKeysPerStep, ++step) {
        // ---- loads: K rows kb + nt*8 + gr (chunks t + 4s); V rows kb + {2t, 2t+1, 2t+8, 2t+9}
        // (chunk gr into va; 128 channels per warp also chunk 8 + gr into vb); all from channel hoff
        const int64_t so = step_offset<kPaged>(a, seq, kb) + hoff;
        uint4 kk[2][DW / 32], va[4], vb[4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int key = kb + nt * 8 + gr;
          const uint16_t* kr = kbase + so + static_cast<int64_t>(nt * 8 + gr) * ks;
#pragma unroll
          for (int s = 0; s < DW / 32; ++s)
            kk[nt][s] = (key < kend) ? ld_stream(kr + 8 * (t + 4 * s)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const int key = kb + 2 * t + (x & 1) + 8 * (x >> 1);
          const uint16_t* vr = vbase + so + static_cast<int64_t>(key - kb) * ks;
          va[x] = (key < kend) ? ld_stream(vr + 8 * gr) : make_uint4(0, 0, 0, 0);
          if constexpr (DW == 128) vb[x] = (key < kend) ? ld_stream(vr + 64 + 8 * gr) : make_uint4(0, 0, 0, 0);
        }
        compute_bf16(kb, step, kk, va, vb);
      }
    }
  } else {
    // FP8: each warp's steps arrive by TMA (one lane issues a K box and a V box, 16 key rows of
    // 128 codes each, 128-byte swizzle) in a kFp8Stages-deep ring of this warp's own stages,
    // kFp8Stages - 1 steps ahead of the one being computed; a stage is refilled only after the
    // warp's reads of it, and each stage's barrier is waited for in step order.
    __shared__ __align__(8) uint64_t fp8_full[kWarps][kFp8Stages];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
    if (lane == 0) {
      for (int s2 = 0; s2 < kFp8Stages; ++s2) mbar_init(&fp8_full[warp][s2], 1);
      fence_mbar_init();
    }
    __syncwarp();
    auto stage_ptr = [&](int s2) { return ring + s2 * kFp8StageBytes + warp * kFp8WarpStepBytes; };
    const int unit_row = seq * a.Hkv + hkv;  // contiguous map: (sequence, KV head) plane
    constexpr int kStride = kWarps * kKeysPerStep;
    // paged: lane l holds the block-table entry of this warp's step 32 b + l, read once per 32
    // steps, so a copy's page is a shuffle away instead of a dependent global load
    int pg_batch = -1, pg_lane = 0;
    auto page_of_step = [&](int ni) -> int {
      if ((ni >> 5) != pg_batch) {
        pg_batch = ni >> 5;
        const int kbl = kstart + warp * kKeysPerStep + (pg_batch * 32 + lane) * kStride;
        pg_lane = (kbl < kend) ? a.block_table[static_cast<int64_t>(seq) * a.max_pages + kbl / a.page_size] : 0;
      }
      return __shfl_sync(0xffffffffu, pg_lane, ni & 31);
    };
    auto issue = [&](int kb, int ni, int s2) {
      if (kb >= kend) return;
      uint8_t* dst = stage_ptr(s2);
      mbar_arrive_expect_tx(&fp8_full[warp][s2], kFp8WarpStepBytes);
      if constexpr (kPaged) {
        int page = page_of_step(ni);
        page = min(max(page, 0), a.num_pages - 1);  // a bad entry reads a wrong page, never outside the pool
        const int tok = page * a.page_size + kb % a.page_size;
        tma_load_3d(dst, &a.tm_k8, &fp8_full[warp][s2], 0, hkv, tok);
        tma_load_3d(dst + kKeysPerStep * 128, &a.tm_v8, &fp8_full[warp][s2], 0, hkv, tok);
      } else {
        tma_load_3d(dst, &a.tm_k8, &fp8_full[warp][s2], 0, kb, unit_row);
        tma_load_3d(dst + kKeysPerStep * 128, &a.tm_v8, &fp8_full[warp][s2], 0, kb, unit_row);
      }
    };
    // 16 bytes at chunk c of row r of a 128-byte-swizzled box (chunk c ^ (r mod 8) holds it)
    auto ld_box = [&](const uint8_t* box, int r, int c) {
      uint4 v;
      const uint32_t addr = smem_u32(box) + r * 128 + ((c ^ (r & 7)) << 4);
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                   : "r"(addr));
      return v;
    };
    const int no_abort = 0;
    bool timed_out = false;
    int kb_next = kstart + warp * kKeysPerStep;
    int n_next = 0;  // this warp's step index of kb_next
#pragma unroll
    for (int s2 = 0; s2 < kFp8Stages - 1; ++s2) {
      issue(kb_next, n_next, s2);
      kb_next += kStride;
      ++n_next;
    }
    int st = 0, n = 0;  // stage and index of this warp's current step
    for (int kb = kstart + warp * kKeysPerStep; kb < kend; kb += kStride, ++n) {
      // refill the stage read one step ago: every lane's reads of it are done (their values were
      // used), and the fence orders them before the copy engine's writes
      __syncwarp();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(kb_next, n_next, st == 0 ? kFp8Stages - 1 : st - 1);
      kb_next += kStride;
      ++n_next;
      // bounded wait: a copy that never lands ends the warp's loop and sets the status word
      if (!__all_sync(0xffffffffu, mbar_wait(&fp8_full[warp][st], (n / kFp8Stages) & 1, a.timeout_ns, &no_abort))) {
        if (lane == 0 && a.status) atomicOr(a.status, kStatusTimeoutBit);
        timed_out = true;
        break;
      }
      const uint8_t* kbox = stage_ptr(st);
      const uint8_t* vbox = kbox + kKeysPerStep * 128;
      uint4 kk[2][2], va[4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        kk[nt][0] = ld_box(kbox, nt * 8 + gr, t);
        kk[nt][1] = ld_box(kbox, nt * 8 + gr, t + 4);
      }
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int r = 2 * t + (x & 1) + 8 * (x >> 1);
        va[x] = ld_box(vbox, r, gr);
        // rows past the slice hold other keys' codes (possibly NaN): their P is 0, and 0 * NaN
        // would still reach O, so their values are zeroed (their scores are masked)
        if (kb + r >= kend) va[x] = make_uint4(0u, 0u, 0u, 0u);
      }
      st = (st + 1 == kFp8Stages) ? 0 : st + 1;
      // k-step kst takes word kst & 3 of chunk kst >> 2: codes (c0, c1) -> k = 2t, 2t+1 and
      // (c2, c3) -> k = 2t+8, 2t+9, the channel order Q was packed in
      if constexpr (NH == 1) {
        float st4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kst = 0; kst < 8; ++kst) {
          uint32_t af[4];
          e4m3x4_to_f16x2x2(word(kk[0][kst >> 2], kst & 3), af[0], af[2]);
          e4m3x4_to_f16x2x2(word(kk[1][kst >> 2], kst & 3), af[1], af[3]);
          mma_f16(st4, af, qa[kst][0], qa[kst][2]);
        }
        uint32_t b0, b1;
        softmax_stepT(kb, st4, b0, b1);
        // tile mu, row gr = channel 16 gr + mu, row gr + 8 = channel 16 gr + 8 + mu: codes mu and
        // 8 + mu of each key's chunk; one byte permute pairs keys (2t, 2t+1) for tiles mu, mu + 1
#pragma unroll
        for (int mu = 0; mu < 8; mu += 2) {
          const int w = mu >> 2, k = mu & 3;
          const uint32_t sel = k | ((4 + k) << 4) | ((k + 1) << 8) | ((5 + k) << 12);
          uint32_t a0[2], a1[2], a2[2], a3[2];
          e4m3x4_to_f16x2x2(__byte_perm(word(va[0], w), word(va[1], w), sel), a0[0], a0[1]);
          e4m3x4_to_f16x2x2(__byte_perm(word(va[0], w + 2), word(va[1], w + 2), sel), a1[0], a1[1]);
          e4m3x4_to_f16x2x2(__byte_perm(word(va[2], w), word(va[3], w), sel), a2[0], a2[1]);
          e4m3x4_to_f16x2x2(__byte_perm(word(va[2], w + 2), word(va[3], w + 2), sel), a3[0], a3[1]);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const uint32_t af[4] = {a0[h2], a1[h2], a2[h2], a3[h2]};
            float(&acc)[4] = *reinterpret_cast<float(*)[4]>(&oacc[2 * (mu + h2)][0]);
            mma_f16(acc, af, b0, b1);
          }
        }
      } else {
        float sacc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
#pragma unroll
          for (int kst = 0; kst < 8; ++kst) {
            uint32_t b0, b1;
            e4m3x4_to_f16x2x2(word(kk[nt][kst >> 2], kst & 3), b0, b1);
            mma_f16(sacc[nt], qa[kst], b0, b1);
          }
        }
        uint32_t pa[4];
        softmax_step(kb, sacc, pa);
        // n-tile nu, column gr = channel 16 gr + nu: code nu of each key's chunk. One byte
        // permute pairs keys (2t, 2t+1) for channels nu and nu + 1 at once; likewise (2t+8, 2t+9).
#pragma unroll
        for (int nu = 0; nu < 16; nu += 2) {
          const int w = nu >> 2, k = nu & 3;
          const uint32_t sel = k | ((4 + k) << 4) | ((k + 1) << 8) | ((5 + k) << 12);
          uint32_t b0v[2], b1v[2];
          e4m3x4_to_f16x2x2(__byte_perm(word(va[0], w), word(va[1], w), sel), b0v[0], b0v[1]);
          e4m3x4_to_f16x2x2(__byte_perm(word(va[2], w), word(va[3], w), sel), b1v[0], b1v[1]);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            float(&acc)[4] = *reinterpret_cast<float(*)[4]>(&oacc[nu + h2][0]);
            mma_f16(acc, pa, b0v[h2], b1v[h2]);
          }
        }
      }
    }
    // after a timed-out wait, the copies this warp issued past it must still land (bounded)
    // before the ring is reused for the combine below; otherwise every issued step was consumed
    if (timed_out) {
      for (int m = n; m < n + kFp8Stages; ++m) {
        const int kbm = kstart + warp * kKeysPerStep + m * kStride;
        if (kbm < kend) mbar_wait(&fp8_full[warp][m % kFp8Stages], (m / kFp8Stages) & 1, a.timeout_ns, &no_abort);
      }
    }
  }

  // ---- combine the key groups' states in shared memory, write this split's partials (d = 256:
  // the two warps of a pair hold the same m and l and one half of the channels each)
  __shared__ float sm_m[kKG][kRowsPerGroup];
  __shared__ float sm_l[kKG][kRowsPerGroup];
  float (*sm_o)[kRowsPerGroup][D + 4];
  if constexpr (kFp8 || kTma16) {
    // the TMA ring is free now: every warp must be past its last read before it is reused
    __syncthreads();
    sm_o = reinterpret_cast<float (*)[kRowsPerGroup][D + 4]>(dsm);
  } else {
    __shared__ float sm_o_static[kKG][kRowsPerGroup][D + 4];
    sm_o = sm_o_static;
  }
  if constexpr (NH == 1) {
    // transposed: rows 2t, 2t+1; l summed over the 8 lanes (keys) of equal t
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float l = l_part[j];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      if (gr == 0 && hoff == 0) {
        sm_m[kg][2 * t + j] = m_run[j];
        sm_l[kg][2 * t + j] = l;
      }
    }
    // tile mu: c0, c1 -> channel A (rows 2t, 2t+1), c2, c3 -> channel B
    const float* vsc = kFp8 ? a.v_scale + hkv * D : nullptr;
#pragma unroll
    for (int mu = 0; mu < DW / 16; ++mu) {
      const int chA = kFp8 ? 16 * gr + mu : hoff + chA_of<DW>(gr, mu);
      const int chB = kFp8 ? 16 * gr + 8 + mu : hoff + chB_of<DW>(gr, mu);
      const float sA = kFp8 ? vsc[chA] : 1.f, sB = kFp8 ? vsc[chB] : 1.f;
      sm_o[kg][2 * t][chA] = oacc[2 * mu][0] * sA;
      sm_o[kg][2 * t + 1][chA] = oacc[2 * mu][1] * sA;
      sm_o[kg][2 * t][chB] = oacc[2 * mu + 1][0] * sB;
      sm_o[kg][2 * t + 1][chB] = oacc[2 * mu + 1][1] * sB;
    }
  } else {
#pragma unroll
    for (int rr = 0; rr < NH; ++rr) {
      float l = l_part[rr];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      if (t == 0 && hoff == 0) {
        sm_m[kg][gr + 8 * rr] = m_run[rr];
        sm_l[kg][gr + 8 * rr] = l;
      }
    }
    if constexpr (!kFp8) {
#pragma unroll
      for (int nu = 0; nu < kNT; ++nu) {
        sm_o[kg][gr][hoff + dv_of(nu, 2 * t)] = oacc[nu][0];
        sm_o[kg][gr][hoff + dv_of(nu, 2 * t + 1)] = oacc[nu][1];
        sm_o[kg][gr + 8][hoff + dv_of(nu, 2 * t)] = oacc[nu][2];
        sm_o[kg][gr + 8][hoff + dv_of(nu, 2 * t + 1)] = oacc[nu][3];
      }
    } else {
      // this thread's channels are 32t .. 32t + 31: apply the V scale there
      const float* vsc = a.v_scale + hkv * D;
#pragma unroll
      for (int nu = 0; nu < 16; ++nu) {
        const int c0 = dv8_of(nu, 2 * t), c1 = dv8_of(nu, 2 * t + 1);
        const float s0 = vsc[c0], s1 = vsc[c1];
        sm_o[kg][gr][c0] = oacc[nu][0] * s0;
        sm_o[kg][gr][c1] = oacc[nu][1] * s1;
        sm_o[kg][gr + 8][c0] = oacc[nu][2] * s0;
        sm_o[kg][gr + 8][c1] = oacc[nu][3] * s1;
      }
    }
  }
  __syncthreads();
  const int unit = seq * a.Hkv + hkv;
  const int nrows = min(8 * NH, R - row0);
  float* ws_o = a.ws + a.ws_o_offset;
  // thread -> (row, channel quad)
  for (int it = threadIdx.x; it < 8 * NH * (D / 4); it += kThreads) {
    const int r = it / (D / 4);
    const int c4 = it % (D / 4);
    if (r >= nrows) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kKG; ++w)
      if (sm_l[w][r] > 0.f) M = fmaxf(M, sm_m[w][r]);
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kKG; ++w) {
      if (!(sm_l[w][r] > 0.f)) continue;
      const float f = ex2(sm_m[w][r] - M);
      L += f * sm_l[w][r];
      o.x += f * sm_o[w][r][4 * c4 + 0];
      o.y += f * sm_o[w][r][4 * c4 + 1];
      o.z += f * sm_o[w][r][4 * c4 + 2];
      o.w += f * sm_o[w][r][4 * c4 + 3];
    }
    const size_t mi = ws_ml_index(a, unit, split, row0 + r);
    *reinterpret_cast<float4*>(ws_o + (mi / 2) * D + 4 * c4) = o;
    if (c4 == 0) {
      a.ws[mi] = (L > 0.f) ? M : -INFINITY;
      a.ws[mi + 1] = L;
    }
  }
  if (!a.tickets) return;  // the separate merge kernel combines the splits

  // ---- the last CTA of this (unit, row group) to finish merges all its splits' partials
  // (the two-state merge rule over the splits), then resets the ticket for the next call
  __shared__ unsigned int sm_last;
  __syncthreads();
  unsigned int* ticket = a.tickets + static_cast<size_t>(unit) * a.row_groups + grp;
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's partials are visible before its ticket is counted
    sm_last = (atomicAdd(ticket, 1u) == static_cast<unsigned int>(a.num_splits - 1)) ? 1u : 0u;
  }
  __syncthreads();
  if (!sm_last) return;
  __threadfence();  // every other split's partials are visible from here on
  const size_t ml_stride = static_cast<size_t>(a.rows_max) * 2;
  const size_t o_stride = static_cast<size_t>(a.rows_max) * D;
  for (int it = threadIdx.x; it < 8 * NH * (D / 4); it += kThreads) {
    const int r = it / (D / 4);
    const int c4 = it % (D / 4);
    if (r >= nrows) continue;
    const float* ml = a.ws + ws_ml_index(a, unit, 0, row0 + r);
    const float* wo = ws_o + (ws_ml_index(a, unit, 0, row0 + r) / 2) * D + 4 * c4;
    float M = -INFINITY;
    for (int sp = 0; sp < a.num_splits; ++sp) {
      const float2 v = __ldcg(reinterpret_cast<const float2*>(ml + sp * ml_stride));
      if (v.y > 0.f) M = fmaxf(M, v.x);
    }
    // empty partials hold l = 0 and o = 0: their weight is taken as 0, and their loads are
    // issued with the others (four splits at a time) rather than behind a branch
    float L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp0 = 0; sp0 < a.num_splits; sp0 += 4) {
      float2 v[4];
      float4 x[4];
#pragma unroll
      for (int u4 = 0; u4 < 4; ++u4) {
        const int sp = min(sp0 + u4, a.num_splits - 1);
        v[u4] = __ldcg(reinterpret_cast<const float2*>(ml + sp * ml_stride));
        x[u4] = __ldcg(reinterpret_cast<const float4*>(wo + sp * o_stride));
      }
#pragma unroll
      for (int u4 = 0; u4 < 4; ++u4) {
        const float f = (sp0 + u4 < a.num_splits && v[u4].y > 0.f) ? ex2(v[u4].x - M) : 0.f;
        L += f * v[u4].y;
        o.x += f * x[u4].x;
        o.y += f * x[u4].y;
        o.z += f * x[u4].z;
        o.w += f * x[u4].w;
      }
    }
    const int rr = row0 + r;
    const int i = rr / a.g, hh = rr % a.g;
    const int64_t orow = static_cast<int64_t>(u.tok0 + i) * a.Hq + hkv * a.g + hh;
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    uint2 packed;
    packed.x = pack_bf16x2(o.x * inv, o.y * inv);
    packed.y = pack_bf16x2(o.z * inv, o.w * inv);
    *reinterpret_cast<uint2*>(a.o + orow * D + 4 * c4) = packed;
    if (a.lse && c4 == 0) a.lse[orow] = (L > 0.f) ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
  if (threadIdx.x == 0) *ticket = 0u;  // no other CTA touches this ticket in this call
}

// One CTA per output row: merge the num_splits partials of (unit, row). The global max comes
// first; each warp then sums its share of the splits with weights e^{m_s - M}, and the warps'
// sums are added in shared memory.
template <int D>
__global__ void __launch_bounds__(kMergeThreads, 1) merge_kernel(MergeArgs a) {
  // the split-K pass (the grid this launch depends on) has completed from here on
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int unit = blockIdx.x / a.rows_max;
  const int r = blockIdx.x % a.rows_max;
  const int seq = unit / a.Hkv, hkv = unit % a.Hkv;
  int tok0, nq;
  if (a.cu_q) {
    tok0 = min(max(a.cu_q[seq], 0), a.total_q);
    nq = min(max(a.cu_q[seq + 1] - tok0, 0), a.total_q - tok0);
    if (nq <= 0 || nq * a.g > a.small_rows_limit) return;
  } else {
    tok0 = seq;
    nq = 1;
  }
  if (r >= nq * a.g) return;
  const int i = r / a.g, hh = r % a.g;
  const int S = a.num_splits;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kMW = kMergeThreads / 32;
  const float* ml = a.ws + (static_cast<size_t>(unit) * S * a.rows_max + r) * 2;
  const float* wo = a.ws + a.ws_o_offset + (static_cast<size_t>(unit) * S * a.rows_max + r) * D;
  const size_t ml_stride = static_cast<size_t>(a.rows_max) * 2;
  const size_t o_stride = static_cast<size_t>(a.rows_max) * D;
  __shared__ float sh_f[kMergeMaxSplits];  // weight 2^(m_s - M) of split s (0 for an empty split)
  __shared__ float sh_red[kMW];
  __shared__ float4 sh_o[kMW][D / 4];
  __shared__ float sh_l[kMW];

  // this warp's splits: s = warp, warp + kMW, ...; lane owns the channel quads lane + 32 j
  // (d = 64: lanes 16..31 hold none and read quad 0 again, their sums unused; d = 256: two each).
  // Every split's o row is written by the split-K pass (zeros for an empty split, whose weight
  // is 0), so the first kUnroll rows of this warp are loaded before the weights are known: their
  // loads overlap the (m, l) round below.
  constexpr int kC4 = D / 4;
  constexpr int kPL = (kC4 + 31) / 32;
  constexpr int kUnroll = D == 256 ? 8 : 16;
  auto load_rows = [&](int s0, float4 (&x)[kUnroll][kPL]) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int s = min(s0 + u * kMW, S - 1);
#pragma unroll
      for (int j = 0; j < kPL; ++j) {
        const int c4 = lane + 32 * j < kC4 ? lane + 32 * j : 0;
        x[u][j] = *reinterpret_cast<const float4*>(wo + s * o_stride + 4 * c4);
      }
    }
  };
  float4 x[kUnroll][kPL];
  load_rows(warp, x);

  // every split's (m, l) in one round of loads (a thread holds up to four), then the global max
  // over the non-empty partials
  constexpr int kPT = kMergeMaxSplits / kMergeThreads;
  float2 v[kPT];
  float M = -INFINITY;
#pragma unroll
  for (int u = 0; u < kPT; ++u) {
    const int s = threadIdx.x + u * kMergeThreads;
    v[u] = s < S ? *reinterpret_cast<const float2*>(ml + s * ml_stride) : make_float2(-INFINITY, 0.f);
    if (v[u].y > 0.f) M = fmaxf(M, v[u].x);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) sh_red[warp] = M;
  __syncthreads();
  M = sh_red[0];
#pragma unroll
  for (int w = 1; w < kMW; ++w) M = fmaxf(M, sh_red[w]);
  // the weights and the merged sum l
  float L = 0.f;
#pragma unroll
  for (int u = 0; u < kPT; ++u) {
    const int s = threadIdx.x + u * kMergeThreads;
    const float f = v[u].y > 0.f ? ex2(v[u].x - M) : 0.f;
    L += f * v[u].y;
    if (s < S) sh_f[s] = f;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  if (lane == 0) sh_l[warp] = L;
  __syncthreads();

  float4 o[kPL];
#pragma unroll
  for (int j = 0; j < kPL; ++j) o[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = warp;;) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int s = s0 + u * kMW;
      const float f = s < S ? sh_f[s] : 0.f;
#pragma unroll
      for (int j = 0; j < kPL; ++j) {
        o[j].x += f * x[u][j].x;
        o[j].y += f * x[u][j].y;
        o[j].z += f * x[u][j].z;
        o[j].w += f * x[u][j].w;
      }
    }
    s0 += kUnroll * kMW;
    if (s0 >= S) break;
    load_rows(s0, x);
  }
#pragma unroll
  for (int j = 0; j < kPL; ++j)
    if (lane + 32 * j < kC4) sh_o[warp][lane + 32 * j] = o[j];
  __syncthreads();
  if (warp != 0 || lane >= kC4) return;
  L = 0.f;
#pragma unroll
  for (int w = 0; w < kMW; ++w) L += sh_l[w];
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  const int64_t orow = (static_cast<int64_t>(tok0 + i) * a.Hq + hkv * a.g + hh);
#pragma unroll
  for (int j = 0; j < kPL; ++j) {
    const int c4 = lane + 32 * j;
    if (c4 >= kC4) break;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kMW; ++w) {
      const float4 y = sh_o[w][c4];
      acc.x += y.x;
      acc.y += y.y;
      acc.z += y.z;
      acc.w += y.w;
    }
    uint2 packed;
    packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(a.o + orow * D + 4 * c4) = packed;
  }
  if (a.lse && lane == 0) a.lse[orow] = (L > 0.f) ? (M + log2f(L)) * kLn2 : -INFINITY;
}

// Merge for many splits: the channels of an output row are shared by kMergeGroups CTAs (one
// per (unit, row, channel group)), so four times as many CTAs each read a quarter of the row's
// o partials. Every CTA takes the global max and the merged l from all splits' (m, l); its warp
// lanes are laid out as (split, channel quad), and the lanes of one quad add their splits' sums
// by shuffles, the warps theirs in shared memory.
constexpr int kMergeGroups = 4;
constexpr int kMergeGroupsMinSplits = 64;
template <int D>
__global__ void __launch_bounds__(kMergeThreads, 1) merge_cg_kernel(MergeArgs a) {
  // the split-K pass (the grid this launch depends on) has completed from here on
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int cg = blockIdx.x % kMergeGroups;
  const int row_id = blockIdx.x / kMergeGroups;
  const int unit = row_id / a.rows_max;
  const int r = row_id % a.rows_max;
  const int seq = unit / a.Hkv, hkv = unit % a.Hkv;
  int tok0, nq;
  if (a.cu_q) {
    tok0 = min(max(a.cu_q[seq], 0), a.total_q);
    nq = min(max(a.cu_q[seq + 1] - tok0, 0), a.total_q - tok0);
    if (nq <= 0 || nq * a.g > a.small_rows_limit) return;
  } else {
    tok0 = seq;
    nq = 1;
  }
  if (r >= nq * a.g) return;
  const int i = r / a.g, hh = r % a.g;
  const int S = a.num_splits;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kMW = kMergeThreads / 32;
  constexpr int kQ = (D / 4) / kMergeGroups;  // channel quads of this CTA
  constexpr int kSL = 32 / kQ;                 // splits side by side in a warp
  constexpr int kSP = kMW * kSL;               // splits per pass of the CTA
  constexpr int kUnroll = 8;
  const int q = lane % kQ, ssub = lane / kQ;
  const int c4 = cg * kQ + q;
  const float* ml = a.ws + (static_cast<size_t>(unit) * S * a.rows_max + r) * 2;
  const float* wo = a.ws + a.ws_o_offset + (static_cast<size_t>(unit) * S * a.rows_max + r) * D + 4 * c4;
  const size_t ml_stride = static_cast<size_t>(a.rows_max) * 2;
  const size_t o_stride = static_cast<size_t>(a.rows_max) * D;
  __shared__ float sh_f[kMergeMaxSplits];
  __shared__ float sh_red[kMW];
  __shared__ float4 sh_o[kMW][kQ];
  __shared__ float sh_l[kMW];

  // this lane's splits: warp * kSL + ssub + p * kSP; the first kUnroll of them are loaded before
  // the weights are known (every split's o row is written, zeros for an empty split)
  const int s_lane = warp * kSL + ssub;
  auto load_rows = [&](int p0, float4 (&x)[kUnroll]) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int s = min(s_lane + (p0 + u) * kSP, S - 1);
      x[u] = *reinterpret_cast<const float4*>(wo + s * o_stride);
    }
  };
  float4 x[kUnroll];
  load_rows(0, x);

  constexpr int kPT = kMergeMaxSplits / kMergeThreads;
  float2 v[kPT];
  float M = -INFINITY;
#pragma unroll
  for (int u = 0; u < kPT; ++u) {
    const int s = threadIdx.x + u * kMergeThreads;
    v[u] = s < S ? *reinterpret_cast<const float2*>(ml + s * ml_stride) : make_float2(-INFINITY, 0.f);
    if (v[u].y > 0.f) M = fmaxf(M, v[u].x);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) sh_red[warp] = M;
  __syncthreads();
  M = sh_red[0];
#pragma unroll
  for (int w = 1; w < kMW; ++w) M = fmaxf(M, sh_red[w]);
  float L = 0.f;
#pragma unroll
  for (int u = 0; u < kPT; ++u) {
    const int s = threadIdx.x + u * kMergeThreads;
    const float f = v[u].y > 0.f ? ex2(v[u].x - M) : 0.f;
    L += f * v[u].y;
    if (s < S) sh_f[s] = f;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
  if (lane == 0) sh_l[warp] = L;
  __syncthreads();

  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int p0 = 0;;) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int s = s_lane + (p0 + u) * kSP;
      const float f = s < S ? sh_f[s] : 0.f;
      o.x += f * x[u].x;
      o.y += f * x[u].y;
      o.z += f * x[u].z;
      o.w += f * x[u].w;
    }
    p0 += kUnroll;
    if (p0 * kSP >= S) break;
    load_rows(p0, x);
  }
  // the lanes of one quad: ssub = 0 .. kSL - 1, kQ lanes apart
#pragma unroll
  for (int off = kQ; off < 32; off <<= 1) {
    o.x += __shfl_xor_sync(0xffffffffu, o.x, off);
    o.y += __shfl_xor_sync(0xffffffffu, o.y, off);
    o.z += __shfl_xor_sync(0xffffffffu, o.z, off);
    o.w += __shfl_xor_sync(0xffffffffu, o.w, off);
  }
  if (lane < kQ) sh_o[warp][lane] = o;
  __syncthreads();
  if (warp != 0 || lane >= kQ) return;
  L = 0.f;
#pragma unroll
  for (int w = 0; w < kMW; ++w) L += sh_l[w];
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  const int64_t orow = (static_cast<int64_t>(tok0 + i) * a.Hq + hkv * a.g + hh);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int w = 0; w < kMW; ++w) {
    const float4 y = sh_o[w][lane];
    acc.x += y.x;
    acc.y += y.y;
    acc.z += y.z;
    acc.w += y.w;
  }
  uint2 packed;
  packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(a.o + orow * D + 4 * c4) = packed;
  if (a.lse && cg == 0 && lane == 0) a.lse[orow] = (L > 0.f) ? (M + log2f(L)) * kLn2 : -INFINITY;
}

// One split-K launch; after a prefill launch (varlen) a programmatic dependent one.
template <typename Kernel>
cudaError_t launch_one(Kernel kernel, dim3 grid, unsigned smem, cudaStream_t stream, const SplitKArgs& a) {
  if (!a.after_prefill) {
    kernel<<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <int D>
cudaError_t launch_splitk_d(const SplitKArgs& a, cudaStream_t stream) {
  // 8-row groups take the transposed form
  const bool half = a.group_rows == 8;
  const bool paged = a.block_table != nullptr;
  const dim3 grid = paged ? dim3(a.Hkv * a.row_groups, a.num_splits, a.num_seqs)
                          : dim3(a.num_splits, a.Hkv * a.row_groups, a.num_seqs);
  const bool window = a.causal && a.window > 0;
  const bool fp8 = a.k8 != nullptr;
  if ((paged || fp8) && window) return cudaErrorInvalidValue;  // no entry point pairs them
  if constexpr (D == 128) {
    if (fp8) {
      static_assert(kFp8SmemBytes >= sizeof(float) * kWarps * kRowsPerGroup * (D + 4), "combine buffer");
      auto k = half ? (paged ? splitk_kernel<D, 1, true, false, true> : splitk_kernel<D, 1, false, false, true>)
                    : (paged ? splitk_kernel<D, 2, true, false, true> : splitk_kernel<D, 2, false, false, true>);
      const cudaError_t e =
          cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kFp8SmemBytes));
      if (e != cudaSuccess) return e;
      return launch_one(k, grid, kFp8SmemBytes, stream, a);
    }
  } else if (fp8) {
    return cudaErrorInvalidValue;  // the FP8 cache is d = 128 only
  }
  if (window)
    return half ? launch_one(splitk_kernel<D, 1, false, true, false>, grid, 0, stream, a)
                : launch_one(splitk_kernel<D, 2, false, true, false>, grid, 0, stream, a);
  if (half)
    return paged ? launch_one(splitk_kernel<D, 1, true, false, false>, grid, 0, stream, a)
                 : launch_one(splitk_kernel<D, 1, false, false, false>, grid, 0, stream, a);
  if (D == 128 && !paged && a.tma16) {
    static_assert(kT16SmemBytes >= sizeof(float) * kWarps * kRowsPerGroup * (128 + 4), "combine buffer");
    auto k = splitk_kernel<D, 2, false, false, false, D == 128>;
    const cudaError_t e =
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kT16SmemBytes));
    if (e != cudaSuccess) return e;
    return launch_one(k, grid, kT16SmemBytes, stream, a);
  }
  return paged ? launch_one(splitk_kernel<D, 2, true, false, false>, grid, 0, stream, a)
               : launch_one(splitk_kernel<D, 2, false, false, false>, grid, 0, stream, a);
}

}  // namespace

cudaError_t launch_splitk(const SplitKArgs& a, cudaStream_t stream) {
  if (a.d == 64) return launch_splitk_d<64>(a, stream);
  if (a.d == 128) return launch_splitk_d<128>(a, stream);
  if (a.d == 256) return launch_splitk_d<256>(a, stream);
  return cudaErrorInvalidValue;
}

// The merge is a programmatic dependent launch: its CTAs may be scheduled while the split-K
// pass finishes (the split kernel signals this at its start) and wait for that grid to complete,
// with its writes visible, before reading any partial.
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  const bool groups = a.num_splits >= kMergeGroupsMinSplits;  // channels over kMergeGroups CTAs
  const long blocks = static_cast<long>(a.num_seqs) * a.Hkv * a.rows_max * (groups ? kMergeGroups : 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.d == 64) return cudaLaunchKernelEx(&cfg, groups ? merge_cg_kernel<64> : merge_kernel<64>, a);
  if (a.d == 128) return cudaLaunchKernelEx(&cfg, groups ? merge_cg_kernel<128> : merge_kernel<128>, a);
  if (a.d == 256) return cudaLaunchKernelEx(&cfg, groups ? merge_cg_kernel<256> : merge_kernel<256>, a);
  return cudaErrorInvalidValue;
}

}  // namespace bw
