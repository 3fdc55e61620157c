// fp32-input prefill with true fp32 FMA arithmetic (no tensor cores: TF32 would round the
// inputs to a 10-bit mantissa). Each query row is owned by 4 threads that split the head
// dimension; K and V tiles are staged in shared memory and shared by the CTA's 64 rows.
// The per-row state is the online-softmax triple (m, l, o) of "Attention from the kernel's
// side", The online softmax, updated every 8 keys; scores carry log2(e) in the scale so the
// exponentials are exp2. Causal masking ("Attention Computation in Practice", Masking
// variants) stops each CTA at the last key its last row sees and masks per key inside that
// range.
#include <math.h>

#include "kernels.h"

namespace bw {

namespace {

constexpr int kRows = 64;      // query rows per CTA
constexpr int kThreads = 256;  // 4 threads per row

template <int D>
struct Fp32Cfg {
  static constexpr int KT = (D == 64) ? 128 : 64;  // keys per shared-memory tile
  static constexpr int CPT = D / 16;               // float4 chunks of the head dim per thread
  static constexpr size_t kSmem = 2ull * KT * D * sizeof(float);
};

__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

template <int D>
__global__ void __launch_bounds__(kThreads) prefill_fp32_kernel(Fp32FwdArgs a) {
  using C = Fp32Cfg<D>;
  constexpr int KT = C::KT;
  constexpr int CPT = C::CPT;
  constexpr int C4 = D / 4;  // float4 per row
  extern __shared__ float4 smem4[];
  float4* Ks = smem4;
  float4* Vs = smem4 + KT * C4;

  const int tid = threadIdx.x;
  const int rloc = tid >> 2;
  const int t = tid & 3;
  const int b = blockIdx.z, h = blockIdx.y;
  const int q0 = blockIdx.x * kRows;
  const int row = q0 + rloc;
  const int hk = h / (a.Hq / a.Hkv);
  const bool row_ok = row < a.Nq;
  const int shift = a.Nk - a.Nq;

  const float4* qrow = reinterpret_cast<const float4*>(a.q + ((static_cast<size_t>(b) * a.Hq + h) * a.Nq + row) * D);
  const float4* kb = reinterpret_cast<const float4*>(a.k + (static_cast<size_t>(b) * a.Hkv + hk) * a.Nk * D);
  const float4* vb = reinterpret_cast<const float4*>(a.v + (static_cast<size_t>(b) * a.Hkv + hk) * a.Nk * D);

  float4 qr[CPT], acc[CPT];
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    qr[i] = row_ok ? qrow[t + 4 * i] : make_float4(0.f, 0.f, 0.f, 0.f);
    acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // keys [lo, lim) are visible to this row (lo > 0 only with a sliding window)
  int lim = a.causal ? min(a.Nk, row + shift + 1) : a.Nk;
  if (!row_ok) lim = 0;
  const bool windowed = a.causal && a.window > 0;
  const int lo = windowed ? max(0, row + shift + 1 - a.window) : 0;
  const int last_row = min(q0 + kRows - 1, a.Nq - 1);
  int kend = a.causal ? min(a.Nk, last_row + shift + 1) : a.Nk;
  kend = max(kend, 0);
  // the CTA's first row has the lowest window start; tiles below it are skipped
  const int kbeg = windowed ? max(0, q0 + shift + 1 - a.window) / KT * KT : 0;

  const unsigned quad = 0xFu << (threadIdx.x & 28);
  float m = -INFINITY, l = 0.f;
  for (int j0 = kbeg; j0 < kend; j0 += KT) {
    __syncthreads();
    for (int idx = tid; idx < KT * C4; idx += kThreads) {
      const int key = j0 + idx / C4;
      const int c = idx % C4;
      float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
      if (key < a.Nk) {
        kv = kb[static_cast<size_t>(key) * C4 + c];
        vv = vb[static_cast<size_t>(key) * C4 + c];
      }
      Ks[idx] = kv;
      Vs[idx] = vv;
    }
    __syncthreads();
    const int nvis = min(KT, lim - j0);  // same for the 4 threads of a row
    const int jlo = lo - j0;              // keys of this tile below jlo are outside the window
    for (int jj = max(0, jlo) & ~7; jj < nvis; jj += 8) {
      float s[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4* kr = Ks + (jj + u) * C4 + t;
        float acc_s = 0.f;
#pragma unroll
        for (int i = 0; i < CPT; ++i) acc_s += dot4(qr[i], kr[4 * i]);
        s[u] = acc_s;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        s[u] += __shfl_xor_sync(quad, s[u], 1);
        s[u] += __shfl_xor_sync(quad, s[u], 2);
      }
      float mt = -INFINITY;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        s[u] = (jj + u < nvis && jj + u >= jlo) ? s[u] * a.scale_log2 : -INFINITY;
        mt = fmaxf(mt, s[u]);
      }
      const float mn = fmaxf(m, mt);
      if (mn == -INFINITY) continue;
      const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - mn);
      l *= alpha;
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        acc[i].x *= alpha;
        acc[i].y *= alpha;
        acc[i].z *= alpha;
        acc[i].w *= alpha;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float p = exp2f(s[u] - mn);
        l += p;
        const float4* vr = Vs + (jj + u) * C4 + t;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
          const float4 vv = vr[4 * i];
          acc[i].x = fmaf(p, vv.x, acc[i].x);
          acc[i].y = fmaf(p, vv.y, acc[i].y);
          acc[i].z = fmaf(p, vv.z, acc[i].z);
          acc[i].w = fmaf(p, vv.w, acc[i].w);
        }
      }
      m = mn;
    }
  }
  if (!row_ok) return;
  const float inv = (l > 0.f) ? 1.f / l : 0.f;
  float4* orow = reinterpret_cast<float4*>(a.o + ((static_cast<size_t>(b) * a.Hq + h) * a.Nq + row) * D);
#pragma unroll
  for (int i = 0; i < CPT; ++i)
    orow[t + 4 * i] = make_float4(acc[i].x * inv, acc[i].y * inv, acc[i].z * inv, acc[i].w * inv);
  if (a.lse && t == 0) {
    a.lse[(static_cast<size_t>(b) * a.Hq + h) * a.Nq + row] = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
  }
}

template <int D>
cudaError_t launch_d(const Fp32FwdArgs& a, cudaStream_t stream) {
  const size_t smem = Fp32Cfg<D>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(prefill_fp32_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((a.Nq + kRows - 1) / kRows, a.Hq, a.B);
  prefill_fp32_kernel<D><<<grid, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_fp32(const Fp32FwdArgs& a, cudaStream_t stream) {
  if (a.d == 64) return launch_d<64>(a, stream);
  return launch_d<128>(a, stream);
}

}  // namespace bw
