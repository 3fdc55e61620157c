// Causal / non-causal bf16 prefill at head dim 256 on the 5th-generation tensor cores.
//
// Same method as the d <= 128 kernel ("Attention from the kernel's side", FlashAttention: what
// never touches memory; "Quantized kernels", 03 The structure): a query tile stays on chip, K
// and V tiles stream past it, S = Q K^T and P exist only on chip, each row keeps a running max
// m and sum l, o is rescaled when the reference max moves, O = o / l is written once. Head dim
// 256 is one of the fast kernels' head dims ("Production implications").
//
// GB300 mapping at d = 256. Tensor memory has 512 columns of 128 lanes; an fp32 O tile of 128
// rows x 256 channels takes 256 of them, so one query tile is in flight per CTA (not two as at
// d <= 128). Q itself sits in tensor memory as the S MMAs' A operand: read from shared memory,
// an M128 K16 A operand costs the same 4 KB per MMA whatever N is, and with N = 64 (64-key
// tiles) that made each S MMA take about 72 cycles instead of 32 (clock64 trace of the issuing
// warp). From tensor memory only K's 2 KB per MMA are read (about 37 cycles per MMA traced).
//   TMEM columns   0..255  O (fp32)   256..383  Q (bf16 pairs)   384 + 64 b .. 447 + 64 b  S buffer b
// Shared memory is one ring of seven 32 KB slots (224 KB): an item's Q arrives in two slots (two
// 128-row atoms each), then its K/V tiles of 64 keys x 256 channels (four 128-byte swizzle
// atoms) follow in the order the MMA warp consumes them. A work item is one 128-row query tile
// of a (sequence, head), taken from the same banded list as the d <= 128 kernel (persistent
// CTAs, atomic counter, longest tiles of a band first). 6 warps per CTA:
//   warp 4      TMA producer: per item the two Q slots, then the K and V tiles.
//   warp 5      MMA issuer, in the order S(0), S(1), PV(0), S(2), PV(1), S(3), ...: S of the
//               next K tile is computed into the other S buffer while the softmax works on
//               S(j), and S(j+2) reuses S(j)'s buffer only after PV(j) (the tensor pipe runs in
//               issue order). An item's Q slots go back to the producer once the softmax threads
//               have copied Q into tensor memory.
//   warps 0-3   softmax, thread = row = TMEM lane: S row (64 scores) from TMEM, mask on tiles
//               that cross the causal limit or the window start, row max, lazy rescale (the
//               reference max moves only when the max grows by more than 2^8), P as bf16 into
//               the first 32 columns of the S buffer. After an item's last step every S MMA of
//               it has completed, so the threads copy the next item's Q rows from its ring
//               slots into tensor memory first (the MMA warp starts that item's S MMAs while
//               they write this item's epilogue O = o / l, LSE).
// Ordering of a rescale: o may be rescaled in TMEM at step j only after PV(j-1) has completed.
// PV n commits to pv_done[n % 2]. When the softmax sees S(j), PV(j-2) and every PV before it have
// completed (S(j) was issued after PV(j-2), and a commit tracks every earlier MMA), and PV(j+1)
// cannot have been issued (P(j+1) does not exist yet); on pv_done[(j-1) % 2] the only phase that
// can still be open is PV(j-1)'s own, so a rescale waits for that parity without ambiguity and the
// common step waits for no PV at all.
// Every wait is bounded; a timed-out wait sets the device status word, the CTA stops producing
// output, waits for its own copies and MMAs and frees its TMEM.
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bw {

namespace {

constexpr int kD = 256;
constexpr int kBM = 128;   // rows per query tile
constexpr int kBN = 64;    // keys per K/V tile
constexpr int kAtoms = kD / 64;  // 128-byte swizzle atoms across the head dim
constexpr int kThreads = 192;
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kStages = 7;
constexpr int kLook = 2;  // S buffers: S(j+1) .. S(j+kLook-1) are issued before PV(j)
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kItemSlots = 2;
constexpr int kItemConsumers = 1 + 4;  // one lane of the MMA warp and of each softmax warp
constexpr uint32_t kTileBytes = kBN * kD * 2;  // 32 KB
constexpr uint32_t kBarOffset = kStages * kTileBytes;
constexpr uint32_t kSmemBytes = kBarOffset + 256 + 1024;  // + barriers, + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0, kColQ = 256, kColS = 384;  // S buffer b: columns kColS + 64 b

struct Bars {
  uint64_t qt_full;          // Q is in tensor memory
  uint64_t s_full[kLook];
  uint64_t p_full[kLook];
  uint64_t pv_done[kLook];  // PV n completes a phase of pv_done[n % kLook]
  uint64_t o_full, o_empty;
  uint64_t mma_done;
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t item_full[kItemSlots];
  uint64_t item_empty[kItemSlots];
  int item_q[kItemSlots];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct Item {
  bool active;
  int nq, nk;
  int q_lo;  // first row (within the sequence) of the query tile
  int j0;    // first K/V tile (64 keys) the tile needs
  int nt;    // K/V tiles it needs
  int q_c1, q_c2, kv_c1, kv_c2;  // TMA coordinates (dense {d, rows, seq*heads}, packed {d, heads, tokens})
  bool packed;
  int64_t out_row0;
  int64_t out_row_stride;
};

// Item numbering: bands of a.band_units (sequence, head) units; a.max_pairs holds the query tiles
// per unit here. Inside a band all units' last tiles come first (with a causal mask they see the
// most keys), then the tiles before them.
template <bool kWindow>
__device__ __forceinline__ Item make_item(const TcFwdArgs& a, int idx) {
  Item w;
  const int units = a.num_seqs * a.Hq;
  const int bu = a.band_units;
  const int per_band = bu * a.max_pairs;
  const int band = idx / per_band;
  const int within = idx % per_band;
  const int band_units = min(bu, units - band * bu);
  const int tile = a.max_pairs - 1 - within / band_units;
  const int unit = band * bu + within % band_units;
  const int s = unit / a.Hq;
  const int h = unit % a.Hq;
  const int g = a.Hq / a.Hkv;
  const int hkv = h / g;
  w.packed = a.cu_q != nullptr;
  int tok_q0 = 0, tok_k0 = 0;
  if (w.packed) {
    tok_q0 = min(max(a.cu_q[s], 0), a.Nq);
    w.nq = min(max(a.cu_q[s + 1] - tok_q0, 0), a.Nq - tok_q0);
    tok_k0 = min(max(a.cu_k[s], 0), a.Nk);
    w.nk = min(max(a.cu_k[s + 1] - tok_k0, 0), a.Nk - tok_k0);
  } else {
    w.nq = a.Nq;
    w.nk = a.Nk;
  }
  w.active = w.nq > 0 && tile * kBM < w.nq;
  if (w.packed && w.nq * g <= a.small_rows_limit) w.active = false;
  const int shift = w.nk - w.nq;
  w.q_lo = tile * kBM;
  int j0 = 0, j1 = 0;
  if (w.active) {
    const int q_hi = min(w.q_lo + kBM - 1, w.nq - 1);
    const int kend = a.causal ? max(min(w.nk, q_hi + shift + 1), 0) : w.nk;
    // with a window the tile's first row sees nothing below this key
    const int kbeg = kWindow ? min(max(0, w.q_lo + shift + 1 - a.window), kend) : 0;
    j0 = kbeg / kBN;
    j1 = (kend > kbeg) ? (kend + kBN - 1) / kBN : j0;
  }
  w.j0 = j0;
  w.nt = j1 - j0;
  if (w.packed) {
    w.q_c1 = h;
    w.q_c2 = tok_q0;
    w.kv_c1 = hkv;
    w.kv_c2 = tok_k0;
    w.out_row0 = static_cast<int64_t>(tok_q0) * a.Hq + h;
    w.out_row_stride = a.Hq;
  } else {
    w.q_c1 = 0;
    w.q_c2 = s * a.Hq + h;
    w.kv_c1 = 0;
    w.kv_c2 = s * a.Hkv + hkv;
    w.out_row0 = (static_cast<int64_t>(s) * a.Hq + h) * a.Nq;
    w.out_row_stride = 1;
  }
  return w;
}

__device__ __forceinline__ int next_item(Bars* bar, int k, uint64_t tmo, const volatile int* abort, bool* ok) {
  const int slot = k % kItemSlots;
  *ok = mbar_wait(&bar->item_full[slot], (k / kItemSlots) & 1, tmo, abort);
  return *ok ? *reinterpret_cast<volatile int*>(&bar->item_q[slot]) : -1;
}

__device__ __forceinline__ void tma_tile(const CUtensorMap* map, const Item& w, uint8_t* dst, uint64_t* bar,
                                         int atom, int row0, bool is_q) {
  const int c0 = atom * 64;
  if (w.packed)
    tma_load_3d(dst, map, bar, c0, is_q ? w.q_c1 : w.kv_c1, (is_q ? w.q_c2 : w.kv_c2) + row0);
  else
    tma_load_3d(dst, map, bar, c0, (is_q ? w.q_c1 : w.kv_c1) + row0, is_q ? w.q_c2 : w.kv_c2);
}

// One MMA D[tmem] (+)= A[tmem] B[smem].
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t blo, uint32_t bhi, uint32_t idesc,
                                        uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p, pe;\n\t.reg .b64 db;\n\telect.sync _|pe, 0xffffffff;\n\t"
      "setp.ne.b32 p, %5, 0;\n\tmov.b64 db, {%2, %3};\n\t"
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "r"(blo), "r"(bhi), "r"(idesc), "r"(acc)
      : "memory");
}

// S = Q K^T over the 256 channels: 16 K=16 steps, Q from tensor memory (8 columns = 16 channels
// per step), K from shared memory 4 steps per swizzle atom (the start address moves 32 B within
// an atom; the next atom is 64 rows x 128 B further).
__device__ __forceinline__ void mma_s(uint32_t d_tmem, uint32_t q_tmem, uint32_t k_lo, uint32_t hi, uint32_t idesc) {
#pragma unroll
  for (int at = 0; at < kAtoms; ++at)
#pragma unroll
    for (int s = 0; s < 4; ++s)
      umma_ts(d_tmem, q_tmem + at * 32 + 8 * s, k_lo + at * (kBN * 128 / 16) + 2 * s, hi, idesc, (at | s) ? 1u : 0u);
}

// O (+)= P V over the tile's 64 keys: 4 K=16 steps; P advances 8 TMEM columns (16 bf16) per
// step, V (MN-major, 128-byte rows of channels) 16 keys = 2048 B; N = 256 channels span the
// four atoms, one leading-dimension offset (64 keys x 128 B) apart.
__device__ __forceinline__ void mma_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_lo, uint32_t hi, uint32_t idesc,
                                       bool accumulate) {
#pragma unroll
  for (int s = 0; s < 4; ++s) umma_ts(d_tmem, p_tmem + 8 * s, v_lo + 128 * s, hi, idesc, (accumulate || s) ? 1u : 0u);
}

template <bool kWindow>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc256_kernel(const __grid_constant__ TcFwdArgs a,
                                                                    unsigned int* status, unsigned int* sched) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sRing = smem;  // [stages][32 KB]: a K or V tile [atoms][64 rows][128 B], or half of Q [2 atoms][128 rows][128 B]
  Bars* bar = reinterpret_cast<Bars*>(smem + kBarOffset);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int total_items = a.max_pairs * a.num_seqs * a.Hq;

  if (threadIdx.x == 0) {
    // packed (varlen) calls: the call's short-query pass, queued after this grid as a
    // programmatic dependent launch, may be scheduled from now on; its CTAs take the SMs that
    // these persistent CTAs leave once the item list runs out
    if (a.cu_q) asm volatile("griddepcontrol.launch_dependents;");
    mbar_init(&bar->qt_full, kBM);
    for (int i = 0; i < kLook; ++i) {
      mbar_init(&bar->s_full[i], 1);
      mbar_init(&bar->p_full[i], kBM);
      mbar_init(&bar->pv_done[i], 1);
    }
    mbar_init(&bar->o_full, 1);
    mbar_init(&bar->o_empty, kBM);
    mbar_init(&bar->mma_done, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar->kv_full[i], 1);
      mbar_init(&bar->kv_empty[i], 1);
    }
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(&bar->item_full[i], 1);
      mbar_init(&bar->item_empty[i], kItemConsumers);
    }
    bar->abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bar->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bar->tmem_base;
  volatile int* abort = &bar->abort;
  const uint64_t tmo = a.timeout_ns;
  auto vote = [](bool x) { return __all_sync(0xffffffffu, x); };

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
    }
    int nload = 0;  // ring loads (Q halves and K/V tiles) issued by this CTA, over all items
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int idx;
      Item w;
      do {
        int got = 0;
        if (lane == 0) got = static_cast<int>(atomicAdd(&sched[0], 1u));
        idx = __shfl_sync(0xffffffffu, got, 0);
        if (idx < total_items) w = make_item<kWindow>(a, idx);
      } while (idx < total_items && !w.active);
      if (idx >= total_items) idx = -1;
      const int qs = k % kItemSlots;
      if (k >= kItemSlots && !(ok = vote(mbar_wait(&bar->item_empty[qs], ((k / kItemSlots) - 1) & 1, tmo, abort))))
        break;
      if (lane == 0) {
        bar->item_q[qs] = idx;
        mbar_arrive(&bar->item_full[qs]);
      }
      if (idx < 0) break;
      // the item's Q in two ring slots (two atoms each), then its K/V tiles
      int kn = 0, vn = 0;  // K and V tiles of the item loaded so far, in the MMA warp's order
      for (int i = 0; i < 2 + 2 * w.nt; ++i, ++nload) {
        const int slot = nload % kStages;
        const int round = nload / kStages;
        if (round > 0 && !(ok = vote(mbar_wait(&bar->kv_empty[slot], (round - 1) & 1, tmo, abort)))) break;
        mbar_arrive_expect_tx(&bar->kv_full[slot], kTileBytes);
        if (i < 2) {
          for (int h = 0; h < 2; ++h)
            tma_tile(&a.tm_q, w, sRing + slot * kTileBytes + h * (kBM * 128), &bar->kv_full[slot], 2 * i + h, w.q_lo,
                     true);
          continue;
        }
        const bool is_k = kn < w.nt && kn < vn + kLook;
        for (int at = 0; at < kAtoms; ++at)
          tma_tile(is_k ? &a.tm_k : &a.tm_v, w, sRing + slot * kTileBytes + at * (kBN * 128), &bar->kv_full[slot],
                   at, (w.j0 + (is_k ? kn : vn)) * kBN, false);
        if (is_k)
          ++kn;
        else
          ++vn;
      }
    }
    if (!ok && lane == 0) raise_timeout(abort, status);
    // every copy this CTA issued lands before the CTA exits (bounded, not cut short by abort)
    const int no_abort = 0;
    for (int i = max(0, nload - kStages); i < nload; ++i)
      mbar_wait(&bar->kv_full[i % kStages], (i / kStages) & 1, tmo, &no_abort);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, 0, 0);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, kD, 0, 1);
    const uint32_t hi = sdesc_hi(1024);
    const uint32_t k_lo = sdesc_lo(smem_u32(sRing), 16);
    const uint32_t v_lo = sdesc_lo(smem_u32(sRing), kBN * 128);
    const uint32_t slot_step = kTileBytes >> 4;
    const uint32_t tO = tbase + kColO;
    int nload = 0;   // ring loads consumed (Q halves and K/V tiles), over all items
    int items = 0;   // items with K/V tiles started (tensor-memory Q copies consumed)
    int ns = 0;      // S MMAs issued, over all items (S buffer ns % kLook)
    int npv = 0;     // PV groups issued, over all items (P of PV n is in S buffer n % kLook)
    int ou = 0;      // items whose O accumulator was used
    bool ok = true;
    auto wait_load = [&](int i) -> bool {
      const bool r = vote(mbar_wait(&bar->kv_full[i % kStages], (i / kStages) & 1, tmo, abort));
      tc_fence_after();
      return r;
    };
    auto issue_s = [&](int i) {  // S into buffer ns % kLook from K in the slot of load i
      mma_s(tbase + kColS + 64 * (ns % kLook), tbase + kColQ, k_lo + (i % kStages) * slot_step, hi, idesc_qk);
      umma_commit(&bar->s_full[ns % kLook]);
      ++ns;
      umma_commit(&bar->kv_empty[i % kStages]);
    };
    for (int k = 0; ok; ++k) {
      const int idx = next_item(bar, k, tmo, abort, &ok);
      ok = vote(ok);
      __syncwarp();
      if (lane == 0 && ok) mbar_arrive(&bar->item_empty[k % kItemSlots]);
      if (!ok || idx < 0) break;
      const Item w = make_item<kWindow>(a, idx);
      const int nt = w.nt;
      // the item's two Q slots go back to the producer once their loads have landed and (items
      // with tiles) the softmax threads have copied Q into tensor memory
      if (!(ok = wait_load(nload) && wait_load(nload + 1))) break;
      if (nt > 0) {
        if (!(ok = vote(mbar_wait(&bar->qt_full, items & 1, tmo, abort)))) break;
        tc_fence_after();
        ++items;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bar->kv_empty[nload % kStages]);
        mbar_arrive(&bar->kv_empty[(nload + 1) % kStages]);
      }
      const int base = nload + 2;
      // the item's 2 nt loads in the order the producer issued them: K tile kn while
      // kn < vn + kLook (S of the next kLook - 1 tiles ahead of each PV), else V tile vn
      int kn = 0, vn = 0;
      for (int p = 0; p < 2 * nt; ++p) {
        const int i = base + p;
        if (!(ok = wait_load(i))) break;
        if (kn < nt && kn < vn + kLook) {
          issue_s(i);  // into the buffer whose P the PV kLook steps back read (in-order tensor pipe)
          ++kn;
          continue;
        }
        // the item's first PV overwrites O: the previous item's epilogue must have read it
        if (vn == 0 && ou > 0 && !(ok = vote(mbar_wait(&bar->o_empty, (ou - 1) & 1, tmo, abort)))) break;
        if (!(ok = vote(mbar_wait(&bar->p_full[npv % kLook], (npv / kLook) & 1, tmo, abort)))) break;
        tc_fence_after();
        mma_pv(tO, tbase + kColS + 64 * (npv % kLook), v_lo + (i % kStages) * slot_step, hi, idesc_pv, vn > 0);
        umma_commit(&bar->pv_done[npv % kLook]);
        ++npv;
        umma_commit(&bar->kv_empty[i % kStages]);
        if (vn == nt - 1) {
          umma_commit(&bar->o_full);
          ++ou;
        }
        ++vn;
      }
      if (!ok) break;
      nload += 2 + 2 * nt;
    }
    if (!ok && lane == 0) raise_timeout(abort, status);
    // all MMAs issued by this warp complete before TMEM is released
    const int no_abort = 0;
    umma_commit(&bar->mma_done);
    mbar_wait(&bar->mma_done, 0, tmo, &no_abort);
  } else {
    // ------------------------------------------------------------ softmax warps 0-3
    const int row = warp * 32 + lane;  // = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tO = tbase + lane_base + kColO;
    const float sl2 = a.scale_log2;
    int gs = 0;     // key steps done by this CTA, over all items: S buffer gs % kLook, PV index gs
    int oused = 0;  // items whose O accumulator was used
    bool ok = true;
    // the k-th item's index from the queue (-1: no more), the slot released
    auto fetch = [&](int k) -> int {
      const int idx = next_item(bar, k, tmo, abort, &ok);
      ok = vote(ok);
      __syncwarp();
      if (lane == 0 && ok) mbar_arrive(&bar->item_empty[k % kItemSlots]);
      return ok ? idx : -1;
    };
    // Item k's Q row of this thread goes from the shared-memory landing buffer (128-byte
    // swizzle: 16-byte chunk c of row r at chunk c ^ (r & 7)) into tensor memory, columns kColQ
    // on (bf16 pairs, the layout of an A operand read from tensor memory). Called once every S
    // MMA of the previous item has completed; it frees the landing buffer for the next Q.
    // Item k's Q row of this thread goes from its two ring slots (loads qb, qb + 1; 128-byte
    // swizzle: 16-byte chunk c of row r at chunk c ^ (r & 7)) into tensor memory, columns kColQ
    // on (bf16 pairs, the layout of an A operand read from tensor memory). Called once every S
    // MMA of the previous item has completed. An item without K/V tiles has no S MMA: its Q is
    // not copied, and the MMA warp hands its slots back without waiting for a copy.
    auto q_to_tmem = [&](int qb, bool used) -> bool {
      if (!used) return true;
      for (int h = 0; h < 2; ++h)
        if (!vote(mbar_wait(&bar->kv_full[(qb + h) % kStages], ((qb + h) / kStages) & 1, tmo, abort))) return false;
      const uint32_t tq = tbase + lane_base + kColQ;
#pragma unroll 1
      for (int at = 0; at < kAtoms; ++at) {
        uint32_t qv[32];
        const uint8_t* src = sRing + ((qb + (at >> 1)) % kStages) * kTileBytes + (at & 1) * (kBM * 128) + row * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 x = *reinterpret_cast<const uint4*>(src + ((c ^ (row & 7)) << 4));
          qv[4 * c] = x.x;
          qv[4 * c + 1] = x.y;
          qv[4 * c + 2] = x.z;
          qv[4 * c + 3] = x.w;
        }
        tmem_st32(tq + at * 32, qv);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar->qt_full);
      return true;
    };
    int nl = 0;  // load index of the current item's first Q slot (2 + 2 nt loads per item)
    int idx = fetch(0);
    Item w_next;
    if (ok && idx >= 0) {
      w_next = make_item<kWindow>(a, idx);
      ok = q_to_tmem(0, w_next.nt > 0);
    }
    for (int k = 0; ok && idx >= 0; ++k) {
      const Item w = w_next;
      const int q_row = w.q_lo + row;
      const bool row_ok = q_row < w.nq;
      const int lim = a.causal ? min(w.nk, q_row + (w.nk - w.nq) + 1) : w.nk;
      const int lo = kWindow ? q_row + (w.nk - w.nq) + 1 - a.window : 0;  // first key in the window
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < w.nt; ++j) {
        const int b = gs % kLook;
        const uint32_t tS = tbase + lane_base + kColS + 64 * b;
        if (!(ok = vote(mbar_wait(&bar->s_full[b], (gs / kLook) & 1, tmo, abort)))) break;
        tc_fence_after();
        uint32_t s0[32], s1[32];
        tmem_ld32(tS, s0);
        tmem_ld32(tS + 32, s1);
        tmem_wait_ld();
        tmem_reg_fence(s0);
        tmem_reg_fence(s1);
        const int kv0 = (w.j0 + j) * kBN;
        const uint32_t ninf = __float_as_uint(-INFINITY);
        if (kv0 + kBN > lim) {  // keys at or past the row's causal limit / the sequence end
          const int n = lim - kv0;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            if (e >= n) s0[e] = ninf;
            if (32 + e >= n) s1[e] = ninf;
          }
        }
        if (kWindow && kv0 < lo) {  // keys below the row's window
          const int n = lo - kv0;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            if (e < n) s0[e] = ninf;
            if (32 + e < n) s1[e] = ninf;
          }
        }
        float mx0 = __uint_as_float(s0[0]), mx1 = __uint_as_float(s1[0]);
#pragma unroll
        for (int e = 1; e < 31; e += 2) {
          mx0 = max3f(mx0, __uint_as_float(s0[e]), __uint_as_float(s0[e + 1]));
          mx1 = max3f(mx1, __uint_as_float(s1[e]), __uint_as_float(s1[e + 1]));
        }
        const float mt = max3f(mx0, mx1, fmaxf(__uint_as_float(s0[31]), __uint_as_float(s1[31])));
        const float m_new = fmaxf(m_ref, mt * sl2);
        float alpha_o = 1.f;
        if (m_new > m_ref + kRescaleThreshold) {
          const float alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
          l *= alpha;
          if (j > 0) alpha_o = alpha;
          m_ref = m_new;
        }
        const float nm = (m_ref == -INFINITY) ? 0.f : -m_ref;
        // p = 2^(s * scale * log2e - m) as bf16 pairs: keys 0-31 -> P columns 0-15, 32-63 -> 16-31
        float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        auto exp_half = [&](const uint32_t (&sc)[32], uint32_t col) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float x0, x1;
            ffma2(x0, x1, __uint_as_float(sc[2 * e]), __uint_as_float(sc[2 * e + 1]), sl2, nm);
            const float p0 = ex2(x0);
            const float p1 = ex2(x1);
            fadd2(ls[(2 * e) & 7], ls[(2 * e + 1) & 7], p0, p1);
            pk[e] = pack_bf16x2(p0, p1);
          }
          tmem_st16(tS + col, pk);
        };
        exp_half(s0, 0);
        exp_half(s1, 16);
        // o takes the new reference max before PV(j) adds to it (rare); PV(j-1) must be done
        if (__any_sync(0xffffffffu, alpha_o != 1.f)) {
          if (!(ok = vote(mbar_wait(&bar->pv_done[(gs - 1) % kLook], ((gs - 1) / kLook) & 1, tmo, abort))))
            break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < kD / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tO + c * 32, ov);
            tmem_wait_ld();
            tmem_reg_fence(ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha_o);
            tmem_st32(tO + c * 32, ov);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar->p_full[b]);
        l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        ++gs;
      }
      if (!ok) break;
      // every S MMA of this item has completed: the next item's Q may replace this one in tensor
      // memory, and the MMA warp starts its first S while this item's epilogue runs
      const int idx_next = fetch(k + 1);
      if (!ok) break;
      nl += 2 + 2 * w.nt;
      if (idx_next >= 0) {
        w_next = make_item<kWindow>(a, idx_next);
        if (!(ok = q_to_tmem(nl, w_next.nt > 0))) break;
      }
      // ---- epilogue: O = o / l (bf16), LSE = (m + log2 l) * ln 2
      if (w.nt > 0) {
        if (!(ok = vote(mbar_wait(&bar->o_full, oused & 1, tmo, abort)))) break;
        ++oused;
        tc_fence_after();
      }
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      uint16_t* orow = a.o + (w.out_row0 + static_cast<int64_t>(q_row) * w.out_row_stride) * kD;
#pragma unroll 1
      for (int c = 0; c < kD / 32; ++c) {
        uint32_t ov[32];
        if (w.nt > 0) {
          tmem_ld32(tO + c * 32, ov);
          tmem_wait_ld();
          tmem_reg_fence(ov);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = 0u;
        }
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint4 pkt;
            pkt.x = pack_bf16x2(__uint_as_float(ov[8 * v4 + 0]) * inv, __uint_as_float(ov[8 * v4 + 1]) * inv);
            pkt.y = pack_bf16x2(__uint_as_float(ov[8 * v4 + 2]) * inv, __uint_as_float(ov[8 * v4 + 3]) * inv);
            pkt.z = pack_bf16x2(__uint_as_float(ov[8 * v4 + 4]) * inv, __uint_as_float(ov[8 * v4 + 5]) * inv);
            pkt.w = pack_bf16x2(__uint_as_float(ov[8 * v4 + 6]) * inv, __uint_as_float(ov[8 * v4 + 7]) * inv);
            dst[v4] = pkt;
          }
        }
      }
      if (w.nt > 0) {
        // O has been read: the next item's first PV may overwrite it
        tc_fence_before();
        mbar_arrive(&bar->o_empty);
      }
      if (row_ok && a.lse)
        a.lse[w.out_row0 + static_cast<int64_t>(q_row) * w.out_row_stride] =
            (l > 0.f) ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
      idx = idx_next;
    }
    if (!ok && lane == 0) raise_timeout(abort, status);
    tc_fence_before();
  }
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
  // the last CTA to leave resets the item counter for the next launch that uses this slot
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&sched[1], 1u) == gridDim.x - 1) {
      atomicExch(&sched[0], 0u);
      atomicExch(&sched[1], 0u);
    }
  }
}

int g_num_sms[64] = {};

template <bool kWindow>
cudaError_t launch_w(const TcFwdArgs& a, unsigned int* status, unsigned int* sched, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(prefill_tc256_kernel<kWindow>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  int sms = (dev >= 0 && dev < 64) ? g_num_sms[dev] : 0;
  if (sms == 0) {
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) g_num_sms[dev] = sms;
  }
  const long items = static_cast<long>(a.max_pairs) * a.num_seqs * a.Hq;
  const int grid = static_cast<int>(items < sms ? items : sms);
  if (grid <= 0) return cudaSuccess;
  prefill_tc256_kernel<kWindow><<<grid, kThreads, kSmemBytes, stream>>>(a, status, sched);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc256(const TcFwdArgs& a, unsigned int* status, unsigned int* sched, cudaStream_t stream) {
  if (a.d != kD) return cudaErrorInvalidValue;
  const bool window = a.causal && a.window > 0;
  return window ? launch_w<true>(a, status, sched, stream) : launch_w<false>(a, status, sched, stream);
}

}  // namespace bw
