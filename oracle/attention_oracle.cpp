// Exact-attention oracle: plain, slow, obviously correct fp64 CPU code.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product path (the CUDA library and its
// Python binding) may include, link, load or call this file. Only the test suite,
// the smoke check and the benchmark's CPU-baseline leg use it.
//
// What it computes (all in IEEE double, std::exp / std::log, no fast-math):
//   s_ij = scale * sum_c q_ic k_jc                       (scores, one row per query)
//   P_ij = exp(s_ij - max_j s_ij) / sum_j exp(...)       (safe softmax over visible j)
//   O_i  = sum_j P_ij v_j
//   LSE_i = max_j s_ij + ln sum_j exp(s_ij - max_j s_ij)
// Sources for each routine are given beside it, as the page title and section:
//   [P1] "Attention from the kernel's side: FlashAttention, online softmax and fused
//        dequant" (trefon.com notes), sections "The online softmax", "Prefill and decode
//        are different problems".
//   [P2] "Quantized kernels" (baselanaya.com lab, day 25), sections 02 and 03.
//   [P3] "Attention Computation in Practice" (inference-engineering learning materials),
//        section 4 "Tiny example", section 5 "GQA in the kernel", "Masking variants",
//        "The four attention kernels you actually use".
//   [P4] "Attention kernels" (llm-inference-explained), sections "Concept" and "Maths".
//
// Three ways of computing the same numbers are kept deliberately separate:
//   method 0  naive: the whole visible score row is materialised (Algorithm 0, [P4] Concept;
//             [P3] section 4), then a safe softmax ([P1] The online softmax) and a weighted sum.
//   method 1  tiled(block): the online-softmax recurrence over key tiles of `block` keys,
//             starting from m = -inf, l = 0, o = 0 ([P1] The online softmax; [P4] Maths,
//             first display; [P2] section 03).
//   method 2  split-K(W): the visible keys are cut into W contiguous slices, each slice is
//             folded into its own partial (m, l, o), and the partials are merged left to right
//             with the two-state merge rule ([P4] Maths, second display; [P1] Flash-decoding).
//
// Readings where the pages are silent (each one is listed in the design notes):
//   * -inf - (-inf): the rescale factor of a state whose max is still -inf is taken as 0
//     (the guard in [P4] Code), and a partial with l == 0 contributes nothing to a merge.
//     A row with no visible key returns O = 0 and LSE = -inf.
//   * causal with Nq != Nk is aligned to the end: query i sees key j iff j <= i + (Nk - Nq).
//   * sliding window W ([P3] Masking variants, i - W < j <= i) is applied on top of the causal
//     mask with the same end alignment: query i sees keys i' - W < j <= i', i' = i + (Nk - Nq);
//     W <= 0 means no window.
//   * split-K slice w covers keys [w*c, min((w+1)*c, n)) with c = ceil(n / W) over the n
//     visible keys of the row; slices past the end are empty.
//   * GQA: query head h reads KV head floor(h / (Hq / Hkv)) ([P3] GQA in the kernel).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <limits>
#include <thread>
#include <vector>

namespace {

const double kNegInf = -std::numeric_limits<double>::infinity();

// One query row against a contiguous run of keys: everything the three methods need.
struct RowJob {
  const double* q;    // [d]
  const double* k;    // first key row; row j at k + j * kv_stride
  const double* v;    // first value row; row j at v + j * kv_stride
  int64_t kv_stride;  // elements between consecutive key (and value) rows
  int n_vis;          // keys [k_begin, n_vis) are visible to this query
  double* o;          // [d] output
  double* lse;        // nullable
  int k_begin;        // first visible key (a sliding window starts past 0)
};

// Running state of the online softmax: max m, sum l, unnormalised output o.
struct State {
  double m = kNegInf;
  double l = 0.0;
  std::vector<double> o;
  explicit State(int d) : o(d, 0.0) {}
};

double dot(const double* a, const double* b, int d) {
  double s = 0.0;
  for (int c = 0; c < d; ++c) s += a[c] * b[c];
  return s;
}

// Fold keys [j0, j1) into the state: one step of the online-softmax recurrence.
// [P1] The online softmax; [P4] Maths, first display; [P2] section 03.
void fold_tile(State& st, const RowJob& r, int j0, int j1, int d, double scale) {
  if (j1 <= j0) return;
  std::vector<double> s(j1 - j0);
  double m_tile = kNegInf;
  for (int j = j0; j < j1; ++j) {
    s[j - j0] = scale * dot(r.q, r.k + j * r.kv_stride, d);
    m_tile = std::max(m_tile, s[j - j0]);
  }
  const double m_new = std::max(st.m, m_tile);
  // Rescale what was accumulated under the old max; a state that has seen nothing has
  // m = -inf and nothing to rescale ([P4] Code guard).
  const double alpha = (st.m == kNegInf) ? 0.0 : std::exp(st.m - m_new);
  st.l *= alpha;
  for (int c = 0; c < d; ++c) st.o[c] *= alpha;
  for (int j = j0; j < j1; ++j) {
    const double p = std::exp(s[j - j0] - m_new);
    st.l += p;
    const double* vj = r.v + j * r.kv_stride;
    for (int c = 0; c < d; ++c) st.o[c] += p * vj[c];
  }
  st.m = m_new;
}

// Merge partial state b into a. [P4] Maths, second display: m = max(m_a, m_b),
// l = l_a e^{m_a-m} + l_b e^{m_b-m}, o likewise. An empty partial (l == 0) contributes
// nothing, which also avoids -inf - (-inf).
void merge_into(State& a, const State& b, int d) {
  if (b.l == 0.0) return;
  if (a.l == 0.0) {
    a = b;
    return;
  }
  const double m = std::max(a.m, b.m);
  const double fa = std::exp(a.m - m);
  const double fb = std::exp(b.m - m);
  a.l = a.l * fa + b.l * fb;
  for (int c = 0; c < d; ++c) a.o[c] = a.o[c] * fa + b.o[c] * fb;
  a.m = m;
}

// After the last tile: O = o / l, LSE = m + ln l. No visible key: O = 0, LSE = -inf.
void finish(const State& st, const RowJob& r, int d) {
  if (st.l == 0.0) {
    for (int c = 0; c < d; ++c) r.o[c] = 0.0;
    if (r.lse) *r.lse = kNegInf;
    return;
  }
  for (int c = 0; c < d; ++c) r.o[c] = st.o[c] / st.l;
  if (r.lse) *r.lse = st.m + std::log(st.l);
}

// Algorithm 0 for one row: the score row is materialised, then softmax, then P.V.
// [P4] Concept (three steps); [P3] section 4, naive; safe softmax from [P1].
void naive_row(const RowJob& r, int d, double scale) {
  const int j0 = r.k_begin;
  const int n = r.n_vis - j0;
  if (n <= 0) {
    for (int c = 0; c < d; ++c) r.o[c] = 0.0;
    if (r.lse) *r.lse = kNegInf;
    return;
  }
  std::vector<double> s(n);
  double mx = kNegInf;
  for (int j = 0; j < n; ++j) {
    s[j] = scale * dot(r.q, r.k + (j0 + j) * r.kv_stride, d);
    mx = std::max(mx, s[j]);
  }
  double sum = 0.0;
  for (int j = 0; j < n; ++j) {
    s[j] = std::exp(s[j] - mx);
    sum += s[j];
  }
  for (int c = 0; c < d; ++c) r.o[c] = 0.0;
  for (int j = 0; j < n; ++j) {
    const double p = s[j] / sum;
    const double* vj = r.v + (j0 + j) * r.kv_stride;
    for (int c = 0; c < d; ++c) r.o[c] += p * vj[c];
  }
  if (r.lse) *r.lse = mx + std::log(sum);
}

// Tiled: key tiles [t*block, (t+1)*block) clipped to the visible range, in key order.
void tiled_row(const RowJob& r, int d, double scale, int block) {
  State st(d);
  for (int j0 = r.k_begin / block * block; j0 < r.n_vis; j0 += block)
    fold_tile(st, r, std::max(j0, r.k_begin), std::min(j0 + block, r.n_vis), d, scale);
  finish(st, r, d);
}

// Split-K: W slices of c = ceil(n/W) keys, each folded as one tile into its own partial,
// merged left to right.
void splitk_partials(const RowJob& r, int d, double scale, int workers, std::vector<State>& parts) {
  const int n = r.n_vis - r.k_begin;
  parts.assign(workers, State(d));
  if (n <= 0) return;
  const int chunk = (n + workers - 1) / workers;
  for (int w = 0; w < workers; ++w) {
    const int j0 = std::min(n, w * chunk);
    const int j1 = std::min(n, j0 + chunk);
    fold_tile(parts[w], r, r.k_begin + j0, r.k_begin + j1, d, scale);
  }
}

void splitk_row(const RowJob& r, int d, double scale, int workers) {
  std::vector<State> parts;
  splitk_partials(r, d, scale, workers, parts);
  State acc(d);
  for (const State& p : parts) merge_into(acc, p, d);
  finish(acc, r, d);
}

int run_rows(const std::vector<RowJob>& jobs, int d, double scale, int method, int param, int nthreads) {
  if (method == 1 && param < 1) return 1;
  if (method == 2 && param < 1) return 1;
  if (method < 0 || method > 2) return 1;
  unsigned hw = std::thread::hardware_concurrency();
  int nt = nthreads > 0 ? nthreads : (hw ? static_cast<int>(hw) : 1);
  nt = std::max(1, std::min<int>(nt, static_cast<int>(jobs.size())));
  std::atomic<size_t> next(0);
  auto worker = [&]() {
    for (;;) {
      const size_t i = next.fetch_add(1);
      if (i >= jobs.size()) return;
      const RowJob& r = jobs[i];
      if (method == 0) naive_row(r, d, scale);
      else if (method == 1) tiled_row(r, d, scale, param);
      else splitk_row(r, d, scale, param);
    }
  };
  if (nt == 1) {
    worker();
  } else {
    std::vector<std::thread> pool;
    for (int t = 0; t < nt; ++t) pool.emplace_back(worker);
    for (auto& th : pool) th.join();
  }
  return 0;
}

// Visible keys for query i: causal aligned to the end of the key sequence ([P3] Masking
// variants, "j <= i", extended to Nq != Nk by aligning the last query with the last key).
int visible_keys(int i, int nq, int nk, int causal) {
  if (!causal) return nk;
  const long lim = static_cast<long>(i) + (nk - nq) + 1;
  return static_cast<int>(std::max(0L, std::min<long>(lim, nk)));
}

// First visible key under a sliding window of W keys ending at the causal limit (W <= 0: none).
int first_visible_key(int i, int nq, int nk, int causal, int window) {
  if (!causal || window <= 0) return 0;
  const long lo = static_cast<long>(i) + (nk - nq) + 1 - window;
  return static_cast<int>(std::max(0L, std::min<long>(lo, nk)));
}

}  // namespace

extern "C" {

// Dense layout: q, o [B, Hq, Nq, d]; k, v [B, Hkv, Nk, d]; lse [B, Hq, Nq] (nullable).
// method 0 naive, 1 tiled(param = block), 2 split-K(param = workers). nthreads 0 = all cores.
// window > 0 (with causal): sliding window of that many keys.
int oracle_attention(const double* q, const double* k, const double* v, double* o, double* lse,
                     int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal, double scale,
                     int method, int param, int nthreads, int window) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0 || d <= 0 || Hq % Hkv) return 1;
  const int g = Hq / Hkv;
  std::vector<RowJob> jobs;
  jobs.reserve(static_cast<size_t>(B) * Hq * Nq);
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < Hq; ++h) {
      const int hk = h / g;  // [P3] GQA in the kernel: head h reads KV head h / (Hq/Hkv)
      const double* kb = k + (static_cast<int64_t>(b) * Hkv + hk) * Nk * d;
      const double* vb = v + (static_cast<int64_t>(b) * Hkv + hk) * Nk * d;
      for (int i = 0; i < Nq; ++i) {
        const int64_t row = (static_cast<int64_t>(b) * Hq + h) * Nq + i;
        jobs.push_back(RowJob{q + row * d, kb, vb, d, visible_keys(i, Nq, Nk, causal), o + row * d,
                              lse ? lse + row : nullptr, first_visible_key(i, Nq, Nk, causal, window)});
      }
    }
  return run_rows(jobs, d, scale, method, param, nthreads);
}

// Single-query decode against a cache: q, o [B, Hq, d]; kc, vc [B, Hkv, cap, d];
// nk[b] valid keys per sequence (host array), all visible (the new token's K/V are already
// in the cache). lse [B, Hq] nullable.
int oracle_decode(const double* q, const double* kc, const double* vc, const int32_t* nk, double* o,
                  double* lse, int B, int Hq, int Hkv, int cap, int d, double scale, int method,
                  int param, int nthreads) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || cap < 0 || d <= 0 || Hq % Hkv) return 1;
  const int g = Hq / Hkv;
  std::vector<RowJob> jobs;
  for (int b = 0; b < B; ++b) {
    if (nk[b] < 0 || nk[b] > cap) return 1;
    for (int h = 0; h < Hq; ++h) {
      const int hk = h / g;
      const int64_t row = static_cast<int64_t>(b) * Hq + h;
      jobs.push_back(RowJob{q + row * d, kc + (static_cast<int64_t>(b) * Hkv + hk) * cap * d,
                            vc + (static_cast<int64_t>(b) * Hkv + hk) * cap * d, d, nk[b], o + row * d,
                            lse ? lse + row : nullptr, 0});
    }
  }
  return run_rows(jobs, d, scale, method, param, nthreads);
}

// Packed variable-length batch ([P3] APPEND / MIXED, cu_seqlens): q, o [total_q, Hq, d];
// k, v [total_k, Hkv, d]; cu_q, cu_k host prefix sums of length num_seqs + 1 with [0] = 0;
// lse [total_q, Hq] nullable. Causal is aligned to each sequence's end.
int oracle_varlen(const double* q, const double* k, const double* v, const int32_t* cu_q,
                  const int32_t* cu_k, double* o, double* lse, int num_seqs, int Hq, int Hkv, int d,
                  int causal, double scale, int method, int param, int nthreads, int window) {
  if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv) return 1;
  if (num_seqs > 0 && (cu_q[0] != 0 || cu_k[0] != 0)) return 1;
  const int g = Hq / Hkv;
  std::vector<RowJob> jobs;
  for (int s = 0; s < num_seqs; ++s) {
    const int nq = cu_q[s + 1] - cu_q[s];
    const int nk = cu_k[s + 1] - cu_k[s];
    if (nq < 0 || nk < 0) return 1;
    for (int i = 0; i < nq; ++i)
      for (int h = 0; h < Hq; ++h) {
        const int hk = h / g;
        const int64_t row = static_cast<int64_t>(cu_q[s] + i) * Hq + h;
        const int64_t k0 = static_cast<int64_t>(cu_k[s]) * Hkv + hk;
        jobs.push_back(RowJob{q + row * d, k + k0 * d, v + k0 * d, static_cast<int64_t>(Hkv) * d,
                              visible_keys(i, nq, nk, causal), o + row * d, lse ? lse + row : nullptr,
                              first_visible_key(i, nq, nk, causal, window)});
      }
  }
  return run_rows(jobs, d, scale, method, param, nthreads);
}

// The naive path's softmax matrix for one head (P, [Nq, Nk], zeros where masked), so that
// tests can check its rows against the softmax definition. q [Nq, d], k [Nk, d].
int oracle_probs(const double* q, const double* k, double* p, int Nq, int Nk, int d, int causal,
                 double scale) {
  if (Nq < 0 || Nk < 0 || d <= 0) return 1;
  for (int i = 0; i < Nq; ++i) {
    double* pr = p + static_cast<int64_t>(i) * Nk;
    for (int j = 0; j < Nk; ++j) pr[j] = 0.0;
    const int n = visible_keys(i, Nq, Nk, causal);
    if (n == 0) continue;
    double mx = kNegInf;
    for (int j = 0; j < n; ++j) {
      pr[j] = scale * dot(q + static_cast<int64_t>(i) * d, k + static_cast<int64_t>(j) * d, d);
      mx = std::max(mx, pr[j]);
    }
    double sum = 0.0;
    for (int j = 0; j < n; ++j) {
      pr[j] = std::exp(pr[j] - mx);
      sum += pr[j];
    }
    for (int j = 0; j < n; ++j) pr[j] /= sum;
  }
  return 0;
}

// The split-K partial states of one query over n keys (no mask): m[W], l[W], o[W, d].
// Empty slices report m = -inf, l = 0, o = 0.
int oracle_partials(const double* q, const double* k, const double* v, int n, int d, double scale,
                    int workers, double* m, double* l, double* o) {
  if (n < 0 || d <= 0 || workers < 1) return 1;
  RowJob r{q, k, v, d, n, nullptr, nullptr, 0};
  std::vector<State> parts;
  splitk_partials(r, d, scale, workers, parts);
  for (int w = 0; w < workers; ++w) {
    m[w] = parts[w].m;
    l[w] = parts[w].l;
    for (int c = 0; c < d; ++c) o[static_cast<int64_t>(w) * d + c] = parts[w].o[c];
  }
  return 0;
}

// Merge two partial states (m, l, o[d]) with the two-state merge rule; result in (m, l, o).
int oracle_merge(double ma, double la, const double* oa, double mb, double lb, const double* ob, int d,
                 double* m, double* l, double* o) {
  if (d <= 0) return 1;
  State a(d), b(d);
  a.m = ma;
  a.l = la;
  b.m = mb;
  b.l = lb;
  for (int c = 0; c < d; ++c) {
    a.o[c] = oa[c];
    b.o[c] = ob[c];
  }
  merge_into(a, b, d);
  *m = a.m;
  *l = a.l;
  for (int c = 0; c < d; ++c) o[c] = a.o[c];
  return 0;
}

// FP8 E4M3 code -> value (the 8-bit float of the OCP FP8 formats: 1 sign bit, 4 exponent bits
// with bias 7, 3 mantissa bits; exponent field 0 is subnormal (m/8 * 2^-6); no infinities, the
// codes S.1111.111 are NaN; largest finite 448). Used for the FP8 KV cache, whose value is this
// decoded code times a per-(KV head, channel) scale ("Attention from the kernel's side", Why a
// quantised cache needs a fused kernel: the cache stores a narrow code plus a scale, and the
// kernel turns the codes into values as it reads them).
int oracle_e4m3_decode(const uint8_t* x, int64_t n, double* out) {
  if (n < 0 || (n > 0 && (!x || !out))) return 1;
  for (int64_t i = 0; i < n; ++i) {
    const int b = x[i];
    const double sign = (b & 0x80) ? -1.0 : 1.0;
    const int e = (b >> 3) & 0xF;
    const int m = b & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) {
      mag = std::numeric_limits<double>::quiet_NaN();
    } else if (e == 0) {
      mag = std::ldexp(static_cast<double>(m) / 8.0, -6);
    } else {
      mag = std::ldexp(1.0 + static_cast<double>(m) / 8.0, e - 7);
    }
    out[i] = sign * mag;
  }
  return 0;
}

int oracle_hardware_threads(void) {
  unsigned hw = std::thread::hardware_concurrency();
  return hw ? static_cast<int>(hw) : 1;
}

}  // extern "C"
