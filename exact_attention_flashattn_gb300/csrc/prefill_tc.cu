// Causal / non-causal bf16 prefill on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// The method is FlashAttention's tiled online softmax ("Attention from the kernel's side",
// FlashAttention: what never touches memory; "Quantized kernels", 03 The structure): a tile
// of queries stays on chip, K and V tiles stream past it, scores S = Q K^T and weights P
// exist only on chip, each row keeps a running max m and sum l, the unnormalised output o is
// rescaled by exp(m - m_new) when the max grows, and O = o / l is written once.
//
// GB300 mapping. A work item is two 128-row query tiles of one (sequence, head), or (kHeadPair:
// d = 128 with an even number of query heads per KV head) one query tile of two heads that share
// a KV head, whose K/V ranges are then identical, so no step runs one tile alone. The kernel is
// persistent: one CTA per SM takes items from a list in order through an atomic counter
// (dynamic, so long and short items balance); the producer warp publishes each item with the
// fields its consumers need already worked out. The list is cut into bands of (sequence, head)
// units and, inside a band, ordered longest first: the items in flight at any time then belong
// to one or two bands, whose K/V stay in L2 while every query tile of those heads reads them.
// The host sizes the band from the K/V bytes of a unit (16 to 64 units). 11 warps per CTA:
//   warp 8      TMA producer: takes the next item and hands it to the other roles through a
//               small shared-memory queue; per item, each Q tile once (its buffer is free when
//               that tile's last S MMA of the previous item completed: each tile has its own
//               full/empty pair), then K_j, V_j tiles (128 keys x d, 128-byte swizzle) into a
//               ring of shared-memory slots guarded by full/empty mbarriers; the ring runs on
//               across items.
//   warps 9,10  MMA issuers, one per query tile w: S_w = Q_w K_j^T into TMEM (fp32, 128 columns
//               per tile), then O_w += P_w V_j with P read from TMEM (bf16, aliased onto S_w)
//               and V from shared memory, S_w(j+1) after P_w V_j. A tcgen05.mma issue blocks at
//               about the tensor pipe's own rate (one M128 N128 K16 MMA per ~70 cycles, even
//               with the pipe idle), so an issuer that waits for P leaves the pipe without work;
//               with one issuer per tile the other tile's MMAs fill that time. The issuers take
//               P.V turns in step order (PV0(j), PV1(j), PV0(j+1), ...), which keeps the two
//               tiles' softmaxes alternating; their S MMAs and waits are not ordered. At d = 64
//               the O accumulators leave 128 TMEM columns free and each tile's P gets its own 64:
//               S(j + 1) is then issued as soon as the softmax has read S(j), so the softmax of
//               one tile never waits for that tile's own MMAs, and the P.V turns are dropped
//               (the softmax, not the MMA order, is the limit there). Warps 8-10
//               each run their loop converged (waits voted across the warp) and one elected lane
//               issues each copy, MMA and commit, which keeps their address arithmetic
//               warp-uniform.
//   warps 0-3,  softmax warpgroups, one per query tile, thread = row = TMEM lane: read the S
//   4-7         row, apply the causal mask on diagonal tiles only ("Attention Computation in
//               Practice", Masking variants: skip / full / diagonal), update m and l in
//               registers (exp2 with log2(e) folded into the scale), write P as bf16 into TMEM,
//               rescale O in TMEM when the running max grew by more than 2^8 (a lazily updated
//               reference max: l and o always share it, so the final o / l is unchanged), and
//               at the end of the item write O = o / l and the LSE; O goes out through 4 KB of
//               shared memory per warp so that the global stores write whole 128-byte rows.
//               Tiles entirely above the diagonal are never loaded.
// Every wait is bounded; a timed-out wait sets the device status word, the CTA stops
// producing output, waits for its own copies and MMAs and frees its TMEM.
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bw {

namespace {

constexpr int kBM = 128;  // rows per query tile
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kThreads = 352;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;  // warps 9 (query tile 0) and 10 (query tile 1)
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8
constexpr int kItemSlots = 2;              // depth of the item queue from producer to consumers
constexpr int kEarlyLoads = 2;             // K/V loads of an item issued before its Q

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;  // 128-byte swizzle atoms across the head dim
  static constexpr uint32_t kQBytes = kBM * D * 2;
  static constexpr uint32_t kTileBytes = kBN * D * 2;
  static constexpr int kStages = (D == 128) ? 4 : 6;
  // epilogue staging: 4 KB per softmax warp (32 rows x 64 columns of bf16)
  static constexpr uint32_t kStageOffset = 2 * kQBytes + kStages * kTileBytes;
  static constexpr uint32_t kStageBytes = 8 * 4096;
  static constexpr uint32_t kBarOffset = kStageOffset + kStageBytes;
  static constexpr uint32_t kSmemBytes = kBarOffset + 512 + 1024;  // + barriers, + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
  // d = 64 leaves 128 columns free: each tile's P gets its own 64 (bf16 pairs) instead of
  // overwriting its S, so S(j + 1) can be computed while the softmax of tile j runs
  static constexpr bool kSplitP = D == 64;
  static constexpr uint32_t kColP0 = 256 + 2 * D, kColP1 = 256 + 2 * D + 64;
  static_assert(!kSplitP || kColP1 + 64 <= kTmemCols, "P columns exceed tensor memory");
};

// What the consumers of an item need, computed once by the producer warp and published in the
// item queue. Each consumer warp would otherwise redo the list arithmetic (integer divisions)
// on a code path it runs once per item, where it delays the item's first MMA or softmax.
struct ItemRec {
  int idx;           // item index, -1: the list is exhausted
  int nq, nk;        // the sequence's query and key counts
  int q_lo[2];       // first row (within the sequence) of each query tile
  int j0[2], j1[2];  // each query tile's K/V tiles: [j0, j1)
  int nt[2];         // j1 - j0
  int jmin, nt_all;  // K/V tiles the item loads: jmin .. jmin + nt_all - 1
  int out_row_stride;
  int out_head_step;  // output rows between the two tiles' heads (head pairs; else 0)
  int64_t out_row0;  // output row index of the sequence's first query for tile 0's head
};

struct Barriers {
  uint64_t q_full[2], q_empty[2];  // per query tile
  uint64_t s_full[2];
  uint64_t p_full[2];  // P of the current K tile stored in TMEM
  uint64_t s_free[2];  // d = 64: the softmax has read S (the next S may overwrite it)
  uint64_t pv_done[2];  // d = 64: a P.V has completed (its P columns may be overwritten)
  uint64_t o_full[2];
  uint64_t o_empty[2];
  uint64_t mma_done[2];
  uint64_t tok[2];  // PV turn tokens: tok[0] issuer 0 -> 1, tok[1] issuer 1 -> 0
  uint64_t kv_full[6];
  uint64_t kv_empty[6];
  uint64_t item_full[kItemSlots];
  uint64_t item_empty[kItemSlots];
  ItemRec rec[kItemSlots];  // the item queue
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Barriers) <= 512, "barriers exceed the shared memory reserved for them");

struct Item {
  bool active;
  int nq, nk;
  int q_lo[2];  // first row (within the sequence) of each query tile
  int j0[2];    // first K/V tile each query tile needs
  int j1[2];    // one past its last K/V tile
  int nt[2];    // j1 - j0
  int jmin;     // first K/V tile of the item (over both query tiles)
  int nt_all;   // K/V tiles the item loads: jmin .. jmin + nt_all - 1
  // TMA coordinates: dense maps are {d, rows, seq*heads}, packed maps {d, heads, tokens}
  int q_c1, q_c2, kv_c1, kv_c2;
  bool packed;
  int q_dh;          // head pairs: the tiles' Q (and O) heads differ by this (else 0)
  int64_t out_row0;  // output row index of the sequence's first query for tile 0's head
  int64_t out_row_stride;
  int64_t out_head_step;
};

// Item numbering: bands of a.band_units (sequence, head) units; inside a band all units of the
// last query-tile pair come first, then those of the pair before, and so on (with a causal
// mask later pairs see more keys).
template <bool kWindow, bool kHeadPair>
__device__ __forceinline__ Item make_item(const TcFwdArgs& a, int idx) {
  Item w;
  // a unit is a (sequence, head), or with head pairs a (sequence, head pair)
  const int hpu = kHeadPair ? a.Hq / 2 : a.Hq;  // units per sequence
  const int units = a.num_seqs * hpu;
  const int bu = a.band_units;
  const int per_band = bu * a.max_pairs;
  const int band = idx / per_band;
  const int within = idx % per_band;
  const int band_units = min(bu, units - band * bu);
  const int pair = a.max_pairs - 1 - within / band_units;  // query-tile pair, or the query tile
  const int unit = band * bu + within % band_units;
  const int s = unit / hpu;
  const int h = (unit % hpu) * (kHeadPair ? 2 : 1);  // tile 0's head
  const int g = a.Hq / a.Hkv;
  const int hkv = h / g;
  w.packed = a.cu_q != nullptr;
  int tok_q0 = 0, tok_k0 = 0;
  if (w.packed) {
    // lengths come from device arrays: clamp them to the packed tensors (Nq, Nk = total rows)
    tok_q0 = min(max(a.cu_q[s], 0), a.Nq);
    w.nq = min(max(a.cu_q[s + 1] - tok_q0, 0), a.Nq - tok_q0);
    tok_k0 = min(max(a.cu_k[s], 0), a.Nk);
    w.nk = min(max(a.cu_k[s + 1] - tok_k0, 0), a.Nk - tok_k0);
  } else {
    w.nq = a.Nq;
    w.nk = a.Nk;
  }
  w.active = w.nq > 0 && pair * (kHeadPair ? 1 : 2) * kBM < w.nq;
  if (w.packed && w.nq * g <= a.small_rows_limit) w.active = false;
  const int shift = w.nk - w.nq;
  if constexpr (!kWindow) {
    // every query tile starts at K/V tile 0
    w.jmin = 0;
    w.nt_all = 0;
    for (int t = 0; t < 2; ++t) {
      w.q_lo[t] = kHeadPair ? pair * kBM : pair * 2 * kBM + t * kBM;
      int nt = 0;
      if (w.active && w.q_lo[t] < w.nq) {
        const int q_hi = min(w.q_lo[t] + kBM - 1, w.nq - 1);
        int kend = a.causal ? min(w.nk, q_hi + shift + 1) : w.nk;
        kend = max(kend, 0);
        nt = (kend + kBN - 1) / kBN;
      }
      w.j0[t] = 0;
      w.j1[t] = nt;
      w.nt[t] = nt;
      w.nt_all = max(w.nt_all, nt);
    }
  } else {
    int jmax = 0;
    w.jmin = 0x7fffffff;
    for (int t = 0; t < 2; ++t) {
      w.q_lo[t] = kHeadPair ? pair * kBM : pair * 2 * kBM + t * kBM;
      int j0 = 0, j1 = 0;
      if (w.active && w.q_lo[t] < w.nq) {
        const int q_hi = min(w.q_lo[t] + kBM - 1, w.nq - 1);
        const int kend = max(min(w.nk, q_hi + shift + 1), 0);
        // the tile's first row sees nothing below this key
        const int kbeg = min(max(0, w.q_lo[t] + shift + 1 - a.window), kend);
        j0 = kbeg / kBN;
        j1 = (kend > kbeg) ? (kend + kBN - 1) / kBN : j0;
      }
      w.j0[t] = j0;
      w.j1[t] = j1;
      w.nt[t] = j1 - j0;
      if (j1 > j0) {
        w.jmin = min(w.jmin, j0);
        jmax = max(jmax, j1);
      }
    }
    if (w.jmin > jmax) w.jmin = 0;
    w.nt_all = jmax - w.jmin;
  }
  w.q_dh = kHeadPair ? 1 : 0;
  if (w.packed) {
    w.q_c1 = h;
    w.q_c2 = tok_q0;  // + row
    w.kv_c1 = hkv;
    w.kv_c2 = tok_k0;  // + key
    w.out_row0 = static_cast<int64_t>(tok_q0) * a.Hq + h;
    w.out_row_stride = a.Hq;
    w.out_head_step = w.q_dh;
  } else {
    w.q_c1 = 0;  // + row
    w.q_c2 = s * a.Hq + h;
    w.kv_c1 = 0;  // + key
    w.kv_c2 = s * a.Hkv + hkv;
    w.out_row0 = (static_cast<int64_t>(s) * a.Hq + h) * a.Nq;
    w.out_row_stride = 1;
    w.out_head_step = static_cast<int64_t>(w.q_dh) * a.Nq;
  }
  return w;
}

// Consumer side of the item queue, called by a converged warp: wait for the k-th item this CTA
// runs (null: a wait gave up); the warp copies what it needs, then releases the slot.
__device__ __forceinline__ const ItemRec* wait_item(Barriers* bar, int k, uint64_t tmo, const volatile int* abort) {
  const int slot = k % kItemSlots;
  const bool ok = __all_sync(0xffffffffu, mbar_wait(&bar->item_full[slot], (k / kItemSlots) & 1, tmo, abort));
  return ok ? &bar->rec[slot] : nullptr;
}
__device__ __forceinline__ void release_item(Barriers* bar, int k) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&bar->item_empty[k % kItemSlots]);
}

__device__ __forceinline__ void tma_tile(const CUtensorMap* map, const Item& w, uint8_t* dst, uint64_t* bar,
                                         int half, int row0, bool is_q, int dh = 0) {
  const int c0 = half * 64;
  if (w.packed) {
    tma_load_3d(dst, map, bar, c0, (is_q ? w.q_c1 : w.kv_c1) + dh, (is_q ? w.q_c2 : w.kv_c2) + row0);
  } else {
    tma_load_3d(dst, map, bar, c0, (is_q ? w.q_c1 : w.kv_c1) + row0, (is_q ? w.q_c2 : w.kv_c2) + dh);
  }
}

// kWindow: causal sliding window (its own instance; the plain path keeps K/V tile 0 as start)
template <int D, bool kWindow, bool kHeadPair>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ TcFwdArgs a,
                                                                 unsigned int* status, unsigned int* sched) {
  using C = Cfg<D>;
  constexpr int kItemConsumers = 2 + 8;  // one lane of each MMA warp and of each softmax warp
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                      // [2][halves][128 rows][128 B]
  uint8_t* sRing = smem + 2 * C::kQBytes;  // [stages][halves][128 rows][128 B]
  Barriers* bar = reinterpret_cast<Barriers*>(smem + C::kBarOffset);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int total_items = a.max_pairs * a.num_seqs * (kHeadPair ? a.Hq / 2 : a.Hq);

  if (threadIdx.x == 0) {
    // packed (varlen) calls: the call's short-query pass, queued after this grid as a
    // programmatic dependent launch, may be scheduled from now on; its CTAs take the SMs that
    // these persistent CTAs leave once the item list runs out
    if (a.cu_q) asm volatile("griddepcontrol.launch_dependents;");
    mbar_init(&bar->q_full[0], 1);
    mbar_init(&bar->q_full[1], 1);
    mbar_init(&bar->q_empty[0], 1);  // the tile's MMA warp
    mbar_init(&bar->q_empty[1], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar->s_full[i], 1);
      mbar_init(&bar->p_full[i], kBM);
      mbar_init(&bar->s_free[i], kBM);
      mbar_init(&bar->pv_done[i], 1);
      mbar_init(&bar->o_full[i], 1);
      mbar_init(&bar->o_empty[i], kBM);
    }
    mbar_init(&bar->tok[0], 1);
    mbar_init(&bar->tok[1], 1);
    mbar_init(&bar->mma_done[0], 1);
    mbar_init(&bar->mma_done[1], 1);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&bar->kv_full[i], 1);
      mbar_init(&bar->kv_empty[i], 2);  // one commit per MMA warp
    }
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(&bar->item_full[i], 1);
      mbar_init(&bar->item_empty[i], kItemConsumers);
    }
    bar->abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bar->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bar->tmem_base;
  volatile int* abort = &bar->abort;
  const uint64_t tmo = a.timeout_ns;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    // Like the MMA warp, the whole warp runs the loop with identical values; lane 0 takes items
    // from the counter and publishes them, one elected lane issues each copy.
    {
      if (lane == 0) {
        prefetch_tmap(&a.tm_q);
        prefetch_tmap(&a.tm_k);
        prefetch_tmap(&a.tm_v);
      }
      auto vote = [](bool x) { return __all_sync(0xffffffffu, x); };
      int nload = 0;  // K/V tiles issued by this CTA, over all items
      int items = 0;  // active items started by this CTA
      bool ok = true;
      // query tile t of the item: its buffer is free once the tile's last S MMA of the previous
      // item completed
      auto load_q = [&](const Item& w, int t) -> bool {
        if (items > 0 && !vote(mbar_wait(&bar->q_empty[t], (items - 1) & 1, tmo, abort))) return false;
        mbar_arrive_expect_tx(&bar->q_full[t], C::kQBytes);
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_tile(&a.tm_q, w, sQ + t * C::kQBytes + hf * (kBM * 128), &bar->q_full[t], hf, w.q_lo[t], true,
                   kHeadPair ? t : 0);
        return true;
      };
      for (int k = 0; ok; ++k) {
        // take the next active item from the list and hand it to the consumers
        int idx;
        Item w;
        do {
          int got = 0;
          if (lane == 0) got = static_cast<int>(atomicAdd(&sched[0], 1u));
          idx = __shfl_sync(0xffffffffu, got, 0);
          if (idx < total_items) w = make_item<kWindow, kHeadPair>(a, idx);
        } while (idx < total_items && !w.active);
        if (idx >= total_items) idx = -1;
        const int qs = k % kItemSlots;
        if (k >= kItemSlots && !(ok = vote(mbar_wait(&bar->item_empty[qs], ((k / kItemSlots) - 1) & 1, tmo, abort))))
          break;
        if (lane == 0) {
          ItemRec& r = bar->rec[qs];
          r.idx = idx;
          if (idx >= 0) {
            r.nq = w.nq;
            r.nk = w.nk;
            r.q_lo[0] = w.q_lo[0];
            r.q_lo[1] = w.q_lo[1];
            r.j0[0] = w.j0[0];
            r.j0[1] = w.j0[1];
            r.j1[0] = w.j1[0];
            r.j1[1] = w.j1[1];
            r.nt[0] = w.nt[0];
            r.nt[1] = w.nt[1];
            r.jmin = w.jmin;
            r.nt_all = w.nt_all;
            r.out_row_stride = static_cast<int>(w.out_row_stride);
            r.out_row0 = w.out_row0;
            if (kHeadPair) r.out_head_step = static_cast<int>(w.out_head_step);
          }
          mbar_arrive(&bar->item_full[qs]);
        }
        if (idx < 0) break;
        // K/V loads need only ring slots: the first ones go out before the Q wait, whose
        // buffers are free only once every S MMA of the previous item has completed
        const int n_early = min(2 * w.nt_all, kEarlyLoads);
        for (int i = 0; i < 2 * w.nt_all; ++i, ++nload) {
          if (i == n_early) {
            if (!(ok = load_q(w, 0) && load_q(w, 1))) break;
            ++items;
          }
          const int slot = nload % C::kStages;
          const int round = nload / C::kStages;
          if (round > 0 && !(ok = vote(mbar_wait(&bar->kv_empty[slot], (round - 1) & 1, tmo, abort)))) break;
          mbar_arrive_expect_tx(&bar->kv_full[slot], C::kTileBytes);
          for (int hf = 0; hf < C::kHalves; ++hf)
            tma_tile((i & 1) ? &a.tm_v : &a.tm_k, w, sRing + slot * C::kTileBytes + hf * (kBN * 128),
                     &bar->kv_full[slot], hf, (w.jmin + (i >> 1)) * kBN, false);
        }
        if (ok && n_early == 2 * w.nt_all) {  // items with no more than kEarlyLoads loads
          if (!(ok = load_q(w, 0) && load_q(w, 1))) break;
          ++items;
        }
      }
      if (!ok && lane == 0) raise_timeout(abort, status);
      // every copy this CTA issued must have landed before the CTA may exit (bounded, and
      // not cut short by the abort flag)
      const int no_abort = 0;
      if (items > 0) {
        mbar_wait(&bar->q_full[0], (items - 1) & 1, tmo, &no_abort);
        mbar_wait(&bar->q_full[1], (items - 1) & 1, tmo, &no_abort);
      }
      for (int i = max(0, nload - C::kStages); i < nload; ++i)
        mbar_wait(&bar->kv_full[i % C::kStages], (i / C::kStages) & 1, tmo, &no_abort);
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ------------------------------------------------------------ MMA issuers, one per query tile
    // tcgen05.mma issue blocks at about the tensor pipe's own rate, so a single issuing warp that
    // waits (for P, a K/V tile or Q) leaves the pipe with nothing queued; with one issuer per
    // query tile the other tile's MMAs keep it fed. The two warps take P.V turns in step order
    // (PV0(j), PV1(j), PV0(j + 1), ...: a token barrier each way, arrived once per step whether
    // or not the tile has a P.V there), which keeps the two tiles' softmaxes alternating on the
    // SM's sub-partitions; their S MMAs and their waits are not ordered. Each warp runs its loop
    // converged (waits are voted); the MMA and commit wrappers let one elected lane issue. Both
    // warps release every K/V slot (two-arrival barriers), each only after the slot's load has
    // landed, so neither can arrive for a phase before the previous one has completed; each warp
    // releases its own tile's Q buffer. The token barriers cannot run two phases ahead either (a
    // warp's next arrival waits for the other's).
    {
      const int tt = warp - kMmaWarp;  // this warp's query tile
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, D, 0, 1);
      // descriptor halves: K-major Q and K tiles (8-row groups 1024 B apart), MN-major V tiles
      // (8-key groups 1024 B apart, the two 64-column halves kBN * 128 B apart)
      const uint32_t hi = sdesc_hi(1024);
      const uint32_t q_lo = sdesc_lo(smem_u32(sQ) + tt * C::kQBytes, 16);
      const uint32_t k_lo = sdesc_lo(smem_u32(sRing), 16);
      const uint32_t v_lo = sdesc_lo(smem_u32(sRing), kBN * 128);
      const uint32_t slot_step = C::kTileBytes >> 4;
      const uint32_t tS = tbase + (tt ? C::kColS1 : C::kColS0);
      const uint32_t tO = tbase + (tt ? C::kColO1 : C::kColO0);
      const uint32_t tP = C::kSplitP ? tbase + (tt ? C::kColP1 : C::kColP0) : tS;
      int nload = 0;  // K/V tiles consumed, over all items
      int items = 0;  // active items
      int pt = 0;     // p_full completions consumed
      int ou = 0;     // items whose O accumulator was used
      int gs = 0;     // steps of all items so far (both issuers count alike)
      int sf = 0;     // S MMAs issued by this warp, over all items
      bool ok = true;

      auto vote = [](bool x) { return __all_sync(0xffffffffu, x); };
      auto wait_load = [&](int i) -> bool {
        const bool r =
            __all_sync(0xffffffffu, mbar_wait(&bar->kv_full[i % C::kStages], (i / C::kStages) & 1, tmo, abort));
        tc_fence_after();
        return r;
      };
      // S = Q K^T, K in the load slot of load i
      auto issue_s = [&](int i) {
        const uint32_t kl = k_lo + (i % C::kStages) * slot_step;
        if constexpr (D == 128)
          umma_ss_k128(tS, q_lo, hi, kl, hi, idesc_qk, 0);
        else
          umma_ss_k64(tS, q_lo, hi, kl, hi, idesc_qk, 0);
        umma_commit(&bar->s_full[tt]);
      };
      // O += P V with V in the load slot of load i: 8 MMAs of K = 16 over the tile's keys
      auto issue_pv = [&](int i, bool accumulate) {
        umma_ts_k128(tO, tP, v_lo + (i % C::kStages) * slot_step, hi, idesc_pv, accumulate ? 1u : 0u);
        if constexpr (C::kSplitP) umma_commit(&bar->pv_done[tt]);
      };
      // S of load i; with P in its own columns it waits only until the softmax has read the
      // previous S out of the buffer
      auto start_s = [&](int i) -> bool {
        if (C::kSplitP && sf > 0) {
          if (!vote(mbar_wait(&bar->s_free[tt], (sf - 1) & 1, tmo, abort))) return false;
          tc_fence_after();
        }
        issue_s(i);
        ++sf;
        return true;
      };

      for (int k = 0; ok; ++k) {
        const ItemRec* rp = wait_item(bar, k, tmo, abort);
        if (!(ok = rp != nullptr)) break;
        if (rp->idx < 0) {
          release_item(bar, k);
          break;
        }
        const int nt = rp->nt_all;
        // this tile uses the item's K/V tiles [ta, te)
        const int ta = rp->j0[tt] - rp->jmin;
        const int te = ta + rp->nt[tt];
        release_item(bar, k);
        if (!(ok = vote(mbar_wait(&bar->q_full[tt], items & 1, tmo, abort)))) break;
        tc_fence_after();
        ++items;
        const int base = nload;
        if (te == ta) umma_commit(&bar->q_empty[tt]);  // no S MMA reads this tile's Q
        if (te > ta) {
          if (!(ok = wait_load(base + 2 * ta))) break;
          if (!(ok = start_s(base + 2 * ta))) break;
          if (te == ta + 1) umma_commit(&bar->q_empty[tt]);
        }
        for (int j = 0; j < nt; ++j) {
          const int ik = base + 2 * j, iv = ik + 1;
          // K_j: read by S(j), issued already, or not read by this tile at all
          if ((j < ta || j >= te) && !(ok = wait_load(ik))) break;
          umma_commit(&bar->kv_empty[ik % C::kStages]);
          if (!(ok = wait_load(iv))) break;
          if (C::kSplitP && j >= ta && j + 1 < te) {
            // S(j + 1) goes ahead of P(j).V(j): the softmax of tile j runs beside it
            if (!(ok = wait_load(ik + 2))) break;
            if (!(ok = start_s(ik + 2))) break;
            if (j + 2 == te) umma_commit(&bar->q_empty[tt]);  // the tile's last S
          }
          // P.V turns alternate: PV0(gs), PV1(gs), PV0(gs + 1), ... (not at d = 64, where each
          // tile's S runs ahead of its P.V and the two softmaxes overlap anyway: 3 % faster free)
          if constexpr (!C::kSplitP) {
            if (tt == 1) {
              if (!(ok = vote(mbar_wait(&bar->tok[0], gs & 1, tmo, abort)))) break;
            } else if (gs > 0) {
              if (!(ok = vote(mbar_wait(&bar->tok[1], (gs - 1) & 1, tmo, abort)))) break;
            }
          }
          bool passed = false;
          if (j >= ta && j < te) {
            // the first P.V of an item overwrites O: the previous item's epilogue must be done
            if (j == ta && ou > 0 && !(ok = vote(mbar_wait(&bar->o_empty[tt], (ou - 1) & 1, tmo, abort)))) break;
            if (!(ok = vote(mbar_wait(&bar->p_full[tt], pt & 1, tmo, abort)))) break;
            ++pt;
            tc_fence_after();
            issue_pv(iv, j > ta);
            __syncwarp();
            if (!C::kSplitP && lane == 0) mbar_arrive(&bar->tok[tt]);
            passed = true;
            if (j == te - 1) {
              umma_commit(&bar->o_full[tt]);
              ++ou;
            } else if (!C::kSplitP) {
              // S(j + 1) overwrites P(j): it follows this P.V in the warp's (in-order) stream
              if (!(ok = wait_load(ik + 2))) break;
              issue_s(ik + 2);
              if (j + 2 == te) umma_commit(&bar->q_empty[tt]);  // the tile's last S
            }
          }
          if (!ok) break;
          if (!passed && !C::kSplitP) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar->tok[tt]);
          }
          ++gs;
          umma_commit(&bar->kv_empty[iv % C::kStages]);
        }
        if (!ok) break;
        nload += 2 * nt;
      }
      if (!ok && lane == 0) raise_timeout(abort, status);
      // all MMAs issued by this warp complete before TMEM is released
      const int no_abort = 0;
      umma_commit(&bar->mma_done[tt]);
      mbar_wait(&bar->mma_done[tt], 0, tmo, &no_abort);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax warpgroups
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int row = (warp & 3) * 32 + lane;  // = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + lane_base + (t ? C::kColS1 : C::kColS0);
    const uint32_t tP = C::kSplitP ? tbase + lane_base + (t ? C::kColP1 : C::kColP0) : tS;
    const uint32_t tO = tbase + lane_base + (t ? C::kColO1 : C::kColO0);
    const float sl2 = a.scale_log2;
    int stiles = 0;  // s_full completions consumed, over all items
    int pw = 0;      // P tiles written, over all items
    int oused = 0;   // items whose O accumulator was used
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const ItemRec* rp = wait_item(bar, k, tmo, abort);
      if (!(ok = rp != nullptr)) break;
      if (rp->idx < 0) {
        release_item(bar, k);
        break;
      }
      // this warpgroup's query tile: the record's per-tile fields, read from shared memory
      const int q_row = rp->q_lo[t] + row;
      const int wnq = rp->nq, wnk = rp->nk;
      const bool row_ok = q_row < wnq;
      const int lim = a.causal ? min(wnk, q_row + (wnk - wnq) + 1) : wnk;
      // sliding window: keys below lo are outside this row's window
      const int lo = kWindow ? q_row + (wnk - wnq) + 1 - a.window : 0;
      const int ntile = rp->nt[t];
      const int jfirst = rp->j0[t];
      const int64_t out_row0 = kHeadPair ? rp->out_row0 + static_cast<int64_t>(t) * rp->out_head_step : rp->out_row0;
      const int out_stride = rp->out_row_stride;
      const int row_w = rp->q_lo[t] + (warp & 3) * 32;  // this warp's first row
      release_item(bar, k);
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < ntile; ++j) {
        ok = mbar_wait(&bar->s_full[t], stiles & 1, tmo, abort);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ++stiles;
        tc_fence_after();
        uint32_t s0[32], s1[32], s2[32], s3[32];
        tmem_ld32(tS, s0);
        tmem_ld32(tS + 32, s1);
        tmem_ld32(tS + 64, s2);
        tmem_ld32(tS + 96, s3);
        tmem_wait_ld();
        tmem_reg_fence(s0);
        tmem_reg_fence(s1);
        tmem_reg_fence(s2);
        tmem_reg_fence(s3);
        if constexpr (C::kSplitP) {
          // S is in registers: the MMA warp may compute the next S into the buffer
          tc_fence_before();
          mbar_arrive(&bar->s_free[t]);
        }
        const int kv0 = (jfirst + j) * kBN;
        // masks: keys at or past the causal limit (diagonal tiles), and with a window keys below
        // its start (window-edge tiles); each kind of tile tests its own bound only
        const uint32_t ninf = __float_as_uint(-INFINITY);
        if (kv0 + kBN > lim) {
          const int n = lim - kv0;  // keys of this tile the row sees from below
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            if (e >= n) s0[e] = ninf;
            if (32 + e >= n) s1[e] = ninf;
            if (64 + e >= n) s2[e] = ninf;
            if (96 + e >= n) s3[e] = ninf;
          }
        }
        if (kWindow && kv0 < lo) {
          const int n = lo - kv0;  // keys of this tile below the window
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            if (e < n) s0[e] = ninf;
            if (32 + e < n) s1[e] = ninf;
            if (64 + e < n) s2[e] = ninf;
            if (96 + e < n) s3[e] = ninf;
          }
        }
        // row max: four chains of 3-input max (a single 128-long chain is pure latency)
        float mx0 = __uint_as_float(s0[0]), mx1 = __uint_as_float(s1[0]);
        float mx2 = __uint_as_float(s2[0]), mx3 = __uint_as_float(s3[0]);
#pragma unroll
        for (int e = 1; e < 31; e += 2) {
          mx0 = max3f(mx0, __uint_as_float(s0[e]), __uint_as_float(s0[e + 1]));
          mx1 = max3f(mx1, __uint_as_float(s1[e]), __uint_as_float(s1[e + 1]));
          mx2 = max3f(mx2, __uint_as_float(s2[e]), __uint_as_float(s2[e + 1]));
          mx3 = max3f(mx3, __uint_as_float(s3[e]), __uint_as_float(s3[e + 1]));
        }
        mx0 = max3f(mx0, __uint_as_float(s0[31]), __uint_as_float(s1[31]));
        mx2 = max3f(mx2, __uint_as_float(s2[31]), __uint_as_float(s3[31]));
        const float mt = max3f(mx0, mx1, fmaxf(mx2, mx3));
        const float m_new = fmaxf(m_ref, mt * sl2);
        float alpha_o = 1.f;
        if (m_new > m_ref + kRescaleThreshold) {
          const float alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
          l *= alpha;
          if (j > 0) alpha_o = alpha;
          m_ref = m_new;
        }
        const float nm = (m_ref == -INFINITY) ? 0.f : -m_ref;
        if constexpr (C::kSplitP) {
          // the previous P.V (also the previous item's last) has read the P columns, and O
          // holds every earlier P.V before a rescale below
          if (pw > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&bar->pv_done[t], (pw - 1) & 1, tmo, abort));
            if (!ok) break;
            tc_fence_after();
          }
        }
        // p = 2^(s * scale * log2e - m) as bf16 pairs; keys 32c..32c+31 -> P columns 16c..16c+15,
        // stored a quarter at a time; fp32 pairs go through packed FMA / ADD; the sum runs as
        // 4 independent pair chains
        float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        auto exp_quarter = [&](const uint32_t (&sc)[32], uint32_t col) {
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
          tmem_st16(tP + col, pk);
        };
        exp_quarter(s0, 0);
        exp_quarter(s1, 16);
        // O must carry the new reference max before this tile's P.V starts (rare)
        if (__any_sync(0xffffffffu, alpha_o != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tO + c * 32, ov);
            tmem_wait_ld();
            tmem_reg_fence(ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha_o);
            tmem_st32(tO + c * 32, ov);
          }
        }
        exp_quarter(s2, 32);
        exp_quarter(s3, 48);
        // all of P is in TMEM: the MMA warp may start P.V
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar->p_full[t]);
        ++pw;
        l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      }
      if (!ok) break;
      // ---- epilogue: O = o / l (bf16), LSE = (m + log2 l) * ln 2
      if (ntile > 0) {
        ok = mbar_wait(&bar->o_full[t], oused & 1, tmo, abort);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        ++oused;
        tc_fence_after();
      }
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      // O leaves through this warp's 4 KB of shared memory, 64 columns at a time: each thread
      // writes its row's 128 bytes (16-byte chunk c of row r at chunk c ^ (r & 7), so a warp's
      // writes and reads spread over all banks), then each store instruction writes four rows'
      // 128 contiguous bytes to global memory instead of 16 bytes of 32 rows
      uint8_t* stg = smem + C::kStageOffset + warp * 4096;
      // all of O's columns are requested before one wait
      uint32_t ov[D / 32][32];
      if (ntile > 0) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32(tO + c * 32, ov[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_reg_fence(ov[c]);
      } else {
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[c][e] = 0u;
      }
#pragma unroll
      for (int hh = 0; hh < D / 64; ++hh) {
        const uint32_t (&oa)[32] = ov[2 * hh];
        const uint32_t (&ob)[32] = ov[2 * hh + 1];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t* src = (c < 4) ? oa + 8 * c : ob + 8 * (c - 4);
          uint4 pkt;
          pkt.x = pack_bf16x2(__uint_as_float(src[0]) * inv, __uint_as_float(src[1]) * inv);
          pkt.y = pack_bf16x2(__uint_as_float(src[2]) * inv, __uint_as_float(src[3]) * inv);
          pkt.z = pack_bf16x2(__uint_as_float(src[4]) * inv, __uint_as_float(src[5]) * inv);
          pkt.w = pack_bf16x2(__uint_as_float(src[6]) * inv, __uint_as_float(src[7]) * inv);
          *reinterpret_cast<uint4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) = pkt;
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rr = i * 4 + (lane >> 3);  // row within the warp's 32
          const int cc = lane & 7;             // 16-byte chunk of the row's 128 bytes
          const uint4 v = *reinterpret_cast<const uint4*>(stg + rr * 128 + ((cc ^ (rr & 7)) << 4));
          const int r = row_w + rr;
          if (r < wnq) {
            uint16_t* dst = a.o + (out_row0 + static_cast<int64_t>(r) * out_stride) * D + hh * 64 + cc * 8;
            *reinterpret_cast<uint4*>(dst) = v;
          }
        }
        __syncwarp();
      }
      if (ntile > 0) {
        // O has been read: the next item's first P.V may overwrite it
        tc_fence_before();
        mbar_arrive(&bar->o_empty[t]);
      }
      if (row_ok && a.lse)
        a.lse[out_row0 + static_cast<int64_t>(q_row) * out_stride] = (l > 0.f) ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
    }
    if (!ok && lane == 0) raise_timeout(abort, status);
    tc_fence_before();
  }
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, C::kTmemCols);
  }
  // The last CTA to leave resets the item counter for the next launch that uses this slot:
  // every CTA has made its final fetch before it counts itself out.
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(&sched[1], 1u) == gridDim.x - 1) {
      atomicExch(&sched[0], 0u);
      atomicExch(&sched[1], 0u);
    }
  }
}

// A CTA that waits on a barrier nobody arrives at, to exercise the bounded-wait path.
__global__ void wait_timeout_probe_kernel(uint64_t timeout_ns, unsigned int* status) {
  __shared__ uint64_t never;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(&never, 1);
    abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait(&never, 0, timeout_ns, &abort)) raise_timeout(&abort, status);
  }
  __syncthreads();
}

int g_num_sms[64] = {};

template <int D, bool kWindow, bool kHeadPair>
cudaError_t launch_d(const TcFwdArgs& a, unsigned int* status, unsigned int* sched, cudaStream_t stream) {
  using C = Cfg<D>;
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D, kWindow, kHeadPair>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::kSmemBytes));
  if (e != cudaSuccess) return e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  int sms = (dev >= 0 && dev < 64) ? g_num_sms[dev] : 0;
  if (sms == 0) {
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) g_num_sms[dev] = sms;
  }
  const long items = static_cast<long>(a.max_pairs) * a.num_seqs * (kHeadPair ? a.Hq / 2 : a.Hq);
  const int grid = static_cast<int>(items < sms ? items : sms);
  if (grid <= 0) return cudaSuccess;
  prefill_tc_kernel<D, kWindow, kHeadPair><<<grid, kThreads, C::kSmemBytes, stream>>>(a, status, sched);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const TcFwdArgs& a, unsigned int* status, unsigned int* sched, cudaStream_t stream) {
  const bool window = a.causal && a.window > 0;
  if (a.d == 64)
    return window ? launch_d<64, true, false>(a, status, sched, stream) : launch_d<64, false, false>(a, status, sched, stream);
  if (a.head_pair)  // two heads of one KV group per item (the host sets it at d = 128 for even g only)
    return window ? launch_d<128, true, true>(a, status, sched, stream) : launch_d<128, false, true>(a, status, sched, stream);
  return window ? launch_d<128, true, false>(a, status, sched, stream) : launch_d<128, false, false>(a, status, sched, stream);
}

cudaError_t launch_wait_timeout_probe(uint64_t timeout_ns, unsigned int* status, cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(timeout_ns, status);
  return cudaGetLastError();
}

}  // namespace bw
