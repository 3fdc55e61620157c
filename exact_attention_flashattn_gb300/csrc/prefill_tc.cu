// Causal / non-causal bf16 prefill on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// The method is FlashAttention's tiled online softmax ("Attention from the kernel's side",
// FlashAttention: what never touches memory; "Quantized kernels", 03 The structure): a tile
// of queries stays on chip, K and V tiles stream past it, scores S = Q K^T and weights P
// exist only on chip, each row keeps a running max m and sum l, the unnormalised output o is
// rescaled by exp(m - m_new) when the max grows, and O = o / l is written once.
//
// GB300 mapping (one CTA = two 128-row query tiles of one (sequence, head); 10 warps):
//   warp 8      TMA producer: loads both Q tiles once, then K_j, V_j tiles (128 keys x d,
//               128-byte swizzle) into a ring of shared-memory slots guarded by mbarriers.
//   warp 9      MMA issuer (one thread): S_w = Q_w K_j^T into TMEM (fp32, 128 columns per
//               tile), then O_w += P_w V_j with P read from TMEM (bf16, aliased onto S_w)
//               and V from shared memory. Issue order S0(j+1) after PV0(j), S1(j+1) after
//               PV1(j) lets softmax of one tile overlap the tensor core work of the other.
//   warps 0-3,  softmax warpgroups, one per query tile, thread = row = TMEM lane: read the
//   4-7         S row, apply the causal mask on diagonal tiles only ("Attention Computation
//               in Practice", Masking variants: skip / full / diagonal), update m and l in
//               registers (exp2 with log2(e) folded into the scale), write P as bf16 into
//               TMEM, and rescale O in TMEM when the running max grew by more than 2^8
//               (a lazily updated reference max: l and o always share it, so the final o / l
//               is unchanged). Tiles entirely above the diagonal are never loaded.
// Every wait is bounded; a timed-out wait sets the device status word, the CTA stops
// producing output, waits for its own copies and MMAs and frees its TMEM.
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"

namespace bw {

namespace {

constexpr int kBM = 128;  // rows per query tile
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kThreads = 320;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;  // 128-byte swizzle atoms across the head dim
  static constexpr uint32_t kQBytes = kBM * D * 2;
  static constexpr uint32_t kTileBytes = kBN * D * 2;
  static constexpr int kStages = (D == 128) ? 4 : 6;
  static constexpr uint32_t kBarOffset = 2 * kQBytes + kStages * kTileBytes;
  static constexpr uint32_t kSmemBytes = kBarOffset + 256 + 1024;  // + barriers, + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
};

struct Barriers {
  uint64_t q_full;
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full[2];
  uint64_t mma_done;
  uint64_t kv_full[6];
  uint64_t kv_empty[6];
  uint32_t tmem_base;
  int abort;
};

struct Work {
  bool active;
  int nq, nk;
  int q_lo[2];  // first row (within the sequence) of each query tile
  int nt[2];    // K/V tiles each query tile needs
  int nt_all;
  // TMA coordinates: dense maps are {d, rows, seq*heads}, packed maps {d, heads, tokens}
  int q_c1, q_c2, kv_c1, kv_c2;
  bool packed;
  int64_t out_row0;  // output row index of the sequence's first query for this head
  int64_t out_row_stride;
};

__device__ __forceinline__ Work make_work(const TcFwdArgs& a) {
  Work w;
  const int pair = static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);  // long tiles first
  const int h = blockIdx.y;
  const int s = blockIdx.z;
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
  w.active = w.nq > 0 && pair * 2 * kBM < w.nq;
  if (w.packed && w.nq * g <= a.small_rows_limit) w.active = false;
  const int shift = w.nk - w.nq;
  w.nt_all = 0;
  for (int t = 0; t < 2; ++t) {
    w.q_lo[t] = pair * 2 * kBM + t * kBM;
    int nt = 0;
    if (w.active && w.q_lo[t] < w.nq) {
      const int q_hi = min(w.q_lo[t] + kBM - 1, w.nq - 1);
      int kend = a.causal ? min(w.nk, q_hi + shift + 1) : w.nk;
      kend = max(kend, 0);
      nt = (kend + kBN - 1) / kBN;
    }
    w.nt[t] = nt;
    w.nt_all = max(w.nt_all, nt);
  }
  if (w.packed) {
    w.q_c1 = h;
    w.q_c2 = tok_q0;  // + row
    w.kv_c1 = hkv;
    w.kv_c2 = tok_k0;  // + key
    w.out_row0 = static_cast<int64_t>(tok_q0) * a.Hq + h;
    w.out_row_stride = a.Hq;
  } else {
    w.q_c1 = 0;  // + row
    w.q_c2 = s * a.Hq + h;
    w.kv_c1 = 0;  // + key
    w.kv_c2 = s * a.Hkv + hkv;
    w.out_row0 = (static_cast<int64_t>(s) * a.Hq + h) * a.Nq;
    w.out_row_stride = 1;
  }
  return w;
}

__device__ __forceinline__ void tma_tile(const CUtensorMap* map, const Work& w, uint8_t* dst, uint64_t* bar,
                                         int half, int row0, bool is_q) {
  const int c0 = half * 64;
  if (w.packed) {
    tma_load_3d(dst, map, bar, c0, is_q ? w.q_c1 : w.kv_c1, (is_q ? w.q_c2 : w.kv_c2) + row0);
  } else {
    tma_load_3d(dst, map, bar, c0, (is_q ? w.q_c1 : w.kv_c1) + row0, is_q ? w.q_c2 : w.kv_c2);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ TcFwdArgs a,
                                                                 unsigned int* status) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                         // [2][halves][128 rows][128 B]
  uint8_t* sRing = smem + 2 * C::kQBytes;     // [stages][halves][128 rows][128 B]
  Barriers* bar = reinterpret_cast<Barriers*>(smem + C::kBarOffset);

  const Work w = make_work(a);
  if (!w.active) return;  // uniform over the CTA, before any barrier or TMEM use

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bar->q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar->s_full[i], 1);
      mbar_init(&bar->p_full[i], kBM);
      mbar_init(&bar->o_full[i], 1);
    }
    mbar_init(&bar->mma_done, 1);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&bar->kv_full[i], 1);
      mbar_init(&bar->kv_empty[i], 1);
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
    if (lane == 0) {
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      mbar_arrive_expect_tx(&bar->q_full, 2 * C::kQBytes);
      for (int t = 0; t < 2; ++t)
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_tile(&a.tm_q, w, sQ + t * C::kQBytes + hf * (kBM * 128), &bar->q_full, hf, w.q_lo[t], true);
      const int nloads = 2 * w.nt_all;
      int issued = 0;
      for (int i = 0; i < nloads; ++i) {
        const int slot = i % C::kStages;
        const int round = i / C::kStages;
        if (round > 0 && !mbar_wait(&bar->kv_empty[slot], (round - 1) & 1, tmo, abort)) {
          raise_timeout(abort, status);
          break;
        }
        const bool is_v = i & 1;
        const int j = i >> 1;
        mbar_arrive_expect_tx(&bar->kv_full[slot], C::kTileBytes);
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_tile(is_v ? &a.tm_v : &a.tm_k, w, sRing + slot * C::kTileBytes + hf * (kBN * 128),
                   &bar->kv_full[slot], hf, j * kBN, false);
        issued = i + 1;
      }
      // every copy this CTA issued must have landed before the CTA may exit (bounded, and
      // not cut short by the abort flag)
      const int no_abort = 0;
      mbar_wait(&bar->q_full, 0, tmo, &no_abort);
      for (int i = max(0, issued - C::kStages); i < issued; ++i)
        mbar_wait(&bar->kv_full[i % C::kStages], (i / C::kStages) & 1, tmo, &no_abort);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, D, 0, 1);
      const uint32_t sQ_addr = smem_u32(sQ);
      const uint32_t sRing_addr = smem_u32(sRing);
      const uint32_t colS[2] = {C::kColS0, C::kColS1};
      const uint32_t colO[2] = {C::kColO0, C::kColO1};
      bool ok = mbar_wait(&bar->q_full, 0, tmo, abort);
      tc_fence_after();

      auto wait_load = [&](int i) -> bool {
        const bool r = mbar_wait(&bar->kv_full[i % C::kStages], (i / C::kStages) & 1, tmo, abort);
        tc_fence_after();
        return r;
      };
      auto issue_s = [&](int t, int j) {
        const uint32_t kslot = sRing_addr + ((2 * j) % C::kStages) * C::kTileBytes;
        const uint32_t qaddr = sQ_addr + t * C::kQBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
          umma_ss(tbase + colS[t], sdesc_sw128(qaddr + off, 16, 1024), sdesc_sw128(kslot + off, 16, 1024),
                  idesc_qk, kk > 0);
        }
        umma_commit(&bar->s_full[t]);
      };
      auto issue_pv = [&](int t, int j) {
        const uint32_t vslot = sRing_addr + ((2 * j + 1) % C::kStages) * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          umma_ts(tbase + colO[t], tbase + colS[t] + kk * 8, sdesc_sw128(vslot + kk * 16 * 128, kBN * 128, 1024),
                  idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        }
      };

      const int nt = w.nt_all;
      if (ok && nt > 0) {
        ok = wait_load(0);
        if (ok) {
          if (w.nt[0] > 0) issue_s(0, 0);
          if (w.nt[1] > 0) issue_s(1, 0);
          umma_commit(&bar->kv_empty[0]);
        }
      }
      for (int j = 0; ok && j < nt; ++j) {
        if (!(ok = wait_load(2 * j + 1))) break;
        for (int t = 0; t < 2; ++t) {
          if (j < w.nt[t]) {
            if (!(ok = mbar_wait(&bar->p_full[t], j & 1, tmo, abort))) break;
            tc_fence_after();
            issue_pv(t, j);
            if (j == w.nt[t] - 1) umma_commit(&bar->o_full[t]);
          }
          if (t == 0 && j + 1 < nt && !(ok = wait_load(2 * (j + 1)))) break;
          if (j + 1 < w.nt[t]) issue_s(t, j + 1);
        }
        if (!ok) break;
        if (j + 1 < nt) umma_commit(&bar->kv_empty[(2 * (j + 1)) % C::kStages]);
        umma_commit(&bar->kv_empty[(2 * j + 1) % C::kStages]);
      }
      if (!ok) raise_timeout(abort, status);
      // all MMAs issued by this thread complete before TMEM is released
      const int no_abort = 0;
      umma_commit(&bar->mma_done);
      mbar_wait(&bar->mma_done, 0, tmo, &no_abort);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int t = warp >> 2;          // query tile of this warpgroup
    const int row = (warp & 3) * 32 + lane;  // = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + lane_base + (t ? C::kColS1 : C::kColS0);
    const uint32_t tO = tbase + lane_base + (t ? C::kColO1 : C::kColO0);
    const int q_row = w.q_lo[t] + row;
    const bool row_ok = q_row < w.nq;
    int lim = a.causal ? min(w.nk, q_row + (w.nk - w.nq) + 1) : w.nk;
    const float sl2 = a.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    const int ntile = w.nt[t];
    for (int j = 0; j < ntile; ++j) {
      ok = mbar_wait(&bar->s_full[t], j & 1, tmo, abort);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_reg_fence(sr[c]);
      const int kv0 = j * kBN;
      if (kv0 + kBN > lim) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (kv0 + c * 32 + e >= lim) sr[c][e] = __float_as_uint(-INFINITY);
      }
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) mt = fmaxf(mt, __uint_as_float(sr[c][e]));
      const float m_new = fmaxf(m_ref, mt * sl2);
      float alpha_o = 1.f;
      if (m_new > m_ref + kRescaleThreshold) {
        const float alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_new);
        l *= alpha;
        if (j > 0) alpha_o = alpha;
        m_ref = m_new;
      }
      const float muse = (m_ref == -INFINITY) ? 0.f : m_ref;
      float lsum = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float p0 = ex2(fmaf(__uint_as_float(sr[c][2 * e]), sl2, -muse));
          const float p1 = ex2(fmaf(__uint_as_float(sr[c][2 * e + 1]), sl2, -muse));
          lsum += p0 + p1;
          pk[e] = pack_bf16x2(p0, p1);
        }
        // P chunk c (32 keys) -> 16 columns of the S region
#pragma unroll
        for (int e = 0; e < 16; ++e) sr[c][e] = pk[e];
      }
      l += lsum;
      {
        uint32_t p01[32], p23[32];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          p01[e] = sr[0][e];
          p01[16 + e] = sr[1][e];
          p23[e] = sr[2][e];
          p23[16 + e] = sr[3][e];
        }
        tmem_st32(tS, p01);
        tmem_st32(tS + 32, p23);
      }
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
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bar->p_full[t]);
    }
    // ---- epilogue: O = o / l (bf16), LSE = (m + log2 l) * ln 2
    if (ok && ntile > 0) {
      ok = mbar_wait(&bar->o_full[t], 0, tmo, abort);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    if (!ok) {
      if (lane == 0) raise_timeout(abort, status);
    } else {
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      uint16_t* orow = a.o + (w.out_row0 + static_cast<int64_t>(q_row) * w.out_row_stride) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        if (ntile > 0) {
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
      if (row_ok && a.lse)
        a.lse[w.out_row0 + static_cast<int64_t>(q_row) * w.out_row_stride] =
            (l > 0.f) ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, C::kTmemCols);
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

template <int D>
cudaError_t launch_d(const TcFwdArgs& a, unsigned int* status, cudaStream_t stream) {
  using C = Cfg<D>;
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::kSmemBytes));
  if (e != cudaSuccess) return e;
  dim3 grid(a.max_pairs, a.Hq, a.cu_q ? a.num_seqs : a.B);
  prefill_tc_kernel<D><<<grid, kThreads, C::kSmemBytes, stream>>>(a, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_tc(const TcFwdArgs& a, unsigned int* status, cudaStream_t stream) {
  if (a.d == 64) return launch_d<64>(a, status, stream);
  return launch_d<128>(a, status, stream);
}

cudaError_t launch_wait_timeout_probe(uint64_t timeout_ns, unsigned int* status, cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(timeout_ns, status);
  return cudaGetLastError();
}

}  // namespace bw
