// kvp_oracle.cpp - the oracle of the pruned-KV decode path in plain C++.
//
// TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
// benchmark's CPU legs load this library (through oracle/cpp.py). The GPU
// library shares no code with it and never loads it.
//
// Plain, slow and obviously correct: double precision throughout (bf16
// inputs are widened exactly), every step in the pages' order, no blocking
// or fusion. Independent (batch, kv head) units, and rows of the scorer,
// are spread over std::thread workers; the arithmetic of a unit does not
// depend on the thread count.
//
// Pages the steps come from (title and section):
//   [KVzap]  "NVIDIA가 AI 메모리 압축 신기술 KVzap 오픈소스 공개!": "KVzap의 구조"
//            (a linear layer or a 2-layer MLP maps a token's hidden state to a
//            score per KV head), "실제 적용" (low scores removed, the last 128
//            tokens always kept), "메모리 및 계산 효율" (overheads),
//            "이게 뭔데?" (335 GB for Llama1-65B at 128k tokens).
//   [DMS]    "Nvidia의 새로운 기술, 정확도 손실 없이 LLM 추론 비용을 8배 절감":
//            "DMS 작동 방식" (keep/evict decision per token, standard
//            attention over what is kept), "지연 삭제 (Delayed Eviction)",
//            "주요 요점" / "앞으로의 전망" (MLA).
//   [DeInfer] gist.science summary of arXiv 2604.17709, "2. 제안 방법 -> 나.
//            페이지드 KV 캐시 및 CUDA Graph 통합" (remapping index list, copy
//            into a compact fixed-address buffer).
//   [BeaconKV] "LLM 추론 비용 혁신: '비콘KV'가 KV 캐시 메모리 4배 절감하며
//            성능까지 잡는 비결" (important entries full precision, the others
//            compressed lossily).
// Readings where the pages are silent are those of the numpy oracle
// (oracle/kvp_oracle.py), which this file restates independently.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

namespace {

constexpr int64_t kNever = 2147483647;  // expire value of an entry kept for good
constexpr int kPage = 16;               // rows per page of the compacted cache

int g_threads = 0;  // 0: the machine's hardware threads

int n_threads() {
  if (g_threads > 0) return g_threads;
  const unsigned h = std::thread::hardware_concurrency();
  return h > 0 ? static_cast<int>(h) : 1;
}

// f(i) for i in [0, n), spread over the worker threads in contiguous blocks.
void parallel_for(int64_t n, const std::function<void(int64_t)>& f) {
  const int nt = static_cast<int>(std::min<int64_t>(n_threads(), std::max<int64_t>(n, 1)));
  if (nt <= 1) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  std::vector<std::thread> pool;
  pool.reserve(nt);
  for (int t = 0; t < nt; ++t) {
    const int64_t a = n * t / nt, b = n * (t + 1) / nt;
    pool.emplace_back([a, b, &f] {
      for (int64_t i = a; i < b; ++i) f(i);
    });
  }
  for (auto& th : pool) th.join();
}

// bf16 bit pattern -> its value (the top 16 bits of an IEEE binary32).
double widen(uint16_t bits) {
  const uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return static_cast<double>(f);
}

// ---------------------------------------------------------------- 2. rules
// [KVzap] "실제 적용": a score at or above tau keeps the entry for good;
// otherwise it lives while it is one of the last `window` positions, i.e.
// until step pos + window. A NaN score compares false: low.
int64_t expire_kvzap_one(double score, double tau, int64_t pos, int64_t window) {
  return (score >= tau) ? kNever : pos + window;
}

// [DMS] "지연 삭제": never flagged (f < 0) -> kept; flagged at step f -> gone
// at f + delay, but not before it leaves the window.
int64_t expire_dms_one(int64_t f, int64_t pos, int64_t delay, int64_t window) {
  return (f < 0) ? kNever : std::max(f + delay, pos + window);
}

// ---------------------------------------------------------------- fp8 E4M3
// Value of the positive code c (0..127): exponent bias 7, 3 mantissa bits,
// subnormals at exponent field 0, code 127 NaN.
double e4m3_value(int c) {
  const int e = c >> 3, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) return (m / 8.0) * std::ldexp(1.0, -6);
  return (1.0 + m / 8.0) * std::ldexp(1.0, e - 7);
}

// The 127 finite non-negative E4M3 values, ascending (codes 0..126).
const std::vector<double>& e4m3_grid() {
  static const std::vector<double> g = [] {
    std::vector<double> v(127);
    for (int c = 0; c < 127; ++c) v[c] = e4m3_value(c);
    return v;
  }();
  return g;
}

// Nearest E4M3 value, ties to the code with an even last mantissa bit,
// magnitudes of 448 and above saturate to 448 (code 126), NaN -> 0x7F; the
// sign is kept, also for a zero result.
uint8_t e4m3_encode_one(double v) {
  if (std::isnan(v)) return 0x7F;
  const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  const double a = std::fabs(v);
  const std::vector<double>& g = e4m3_grid();
  int code;
  if (a >= 448.0) {
    code = 126;
  } else {
    // lo: the largest code whose value is <= a; hi: the next one
    const int lo = static_cast<int>(std::upper_bound(g.begin(), g.end(), a) - g.begin()) - 1;
    const int hi = std::min(lo + 1, 126);
    const double dlo = a - g[lo], dhi = g[hi] - a;
    if (hi == lo || dlo < dhi) code = lo;
    else if (dhi < dlo) code = hi;
    else code = (hi % 2 == 0) ? hi : lo;
  }
  return static_cast<uint8_t>(code | sign);
}

double e4m3_decode_one(uint8_t c) {
  const double v = e4m3_value(c & 0x7F);
  return (c & 0x80) ? -v : v;
}

// One bf16 row of d values -> E4M3 codes and its float32 scale:
// scale = amax / 448 and inv = 448 / amax (binary32, round to nearest), each
// element x * inv rounded to E4M3; an all-zero row: scale 0, codes 0.
void quantize_row(const uint16_t* row, int d, uint8_t* codes, float* scale) {
  float amax = 0.f;
  for (int e = 0; e < d; ++e) amax = std::max(amax, std::fabs(static_cast<float>(widen(row[e]))));
  const float s = amax / 448.0f;
  *scale = s;
  if (!(amax > 0.f)) {
    for (int e = 0; e < d; ++e) codes[e] = 0;
    return;
  }
  const float inv = 448.0f / amax;
  for (int e = 0; e < d; ++e) {
    const float y = static_cast<float>(widen(row[e])) * inv;
    codes[e] = e4m3_encode_one(static_cast<double>(y));
  }
}

// ---------------------------------------------------------------- softmax
// One query over n rows: logits l_i = scale * q . k_i; two-pass softmax
// (maximum, then exp(l_i - m)); out = sum_i w_i v_i / sum_i w_i. n = 0 gives
// zeros.
void softmax_attend(const double* q, int dk, const std::vector<const double*>& K,
                    const std::vector<const double*>& V, int dv, double scale, double* out) {
  for (int e = 0; e < dv; ++e) out[e] = 0.0;
  const size_t n = K.size();
  if (n == 0) return;
  std::vector<double> l(n);
  double m = -INFINITY;
  for (size_t i = 0; i < n; ++i) {
    double s = 0.0;
    for (int e = 0; e < dk; ++e) s += K[i][e] * q[e];
    l[i] = s * scale;
    m = std::max(m, l[i]);
  }
  double den = 0.0;
  for (size_t i = 0; i < n; ++i) {
    const double w = std::exp(l[i] - m);
    den += w;
    for (int e = 0; e < dv; ++e) out[e] += w * V[i][e];
  }
  for (int e = 0; e < dv; ++e) out[e] /= den;
}

}  // namespace

extern "C" {

// Worker threads (0 = the machine's hardware threads).
void kvpo_set_threads(int n) { g_threads = n > 0 ? n : 0; }
int kvpo_threads() { return n_threads(); }

void kvpo_widen_bf16(const uint16_t* x, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = widen(x[i]);
}

// ---------------------------------------------------------------- 1. score
// [KVzap] "KVzap의 구조". Linear: s[t, h] = sum_k x[t, k] w[h, k] + b[h].
void kvpo_score_linear(const uint16_t* x, int64_t n_tok, int D, const double* w, int H, const double* bias,
                       double* s) {
  parallel_for(n_tok, [&](int64_t t) {
    std::vector<double> xr(D);
    for (int k = 0; k < D; ++k) xr[k] = widen(x[t * D + k]);
    for (int h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int k = 0; k < D; ++k) acc += xr[k] * w[static_cast<int64_t>(h) * D + k];
      s[t * H + h] = acc + (bias ? bias[h] : 0.0);
    }
  });
}

// Exact GELU: u * Phi(u) = u / 2 * (1 + erf(u / sqrt 2)).
void kvpo_gelu(const double* u, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = 0.5 * u[i] * (1.0 + std::erf(u[i] / std::sqrt(2.0)));
}

// MLP: u_j = sum_k x_k w1[j, k] + b1_j; z_j = GELU(u_j); s_h = sum_j z_j w2[h, j] + b2_h.
void kvpo_score_mlp(const uint16_t* x, int64_t n_tok, int D, const uint16_t* w1, int hidden, const uint16_t* w2,
                    int H, const double* b1, const double* b2, double* s) {
  std::vector<double> w1f(static_cast<size_t>(hidden) * D), w2f(static_cast<size_t>(H) * hidden);
  for (size_t i = 0; i < w1f.size(); ++i) w1f[i] = widen(w1[i]);
  for (size_t i = 0; i < w2f.size(); ++i) w2f[i] = widen(w2[i]);
  parallel_for(n_tok, [&](int64_t t) {
    std::vector<double> xr(D), z(hidden);
    for (int k = 0; k < D; ++k) xr[k] = widen(x[t * D + k]);
    for (int j = 0; j < hidden; ++j) {
      double u = 0.0;
      const double* wr = &w1f[static_cast<size_t>(j) * D];
      for (int k = 0; k < D; ++k) u += xr[k] * wr[k];
      u += b1 ? b1[j] : 0.0;
      kvpo_gelu(&u, 1, &z[j]);
    }
    for (int h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int j = 0; j < hidden; ++j) acc += z[j] * w2f[static_cast<size_t>(h) * hidden + j];
      s[t * H + h] = acc + (b2 ? b2[h] : 0.0);
    }
  });
}

// ---------------------------------------------------------------- 2. mask
// Element-wise rules on broadcast (flattened) operands.
void kvpo_expire_kvzap(const double* score, const double* tau, const int64_t* pos, int64_t n, int64_t window,
                       int64_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = expire_kvzap_one(score[i], tau[i], pos[i], window);
}

void kvpo_expire_dms(const int64_t* flag, const int64_t* pos, int64_t n, int64_t delay, int64_t window,
                     int64_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = expire_dms_one(flag[i], pos[i], delay, window);
}

// Present at step `now` iff now < expire.
void kvpo_present(const int64_t* expire, int64_t n, int64_t now, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = now < expire[i];
}

// expire [BH, T] -> keep [BH, T] (present at `now`: now < expire), keep bits
// [BH, ceil(T / 32)] (bit i of word w = position 32 w + i), count [BH].
void kvpo_mask(const int64_t* expire, int64_t BH, int64_t T, int64_t now, uint8_t* keep, uint32_t* bits,
               int64_t* count) {
  const int64_t nw = (T + 31) / 32;
  parallel_for(BH, [&](int64_t u) {
    int64_t c = 0;
    for (int64_t w = 0; w < nw; ++w) bits[u * nw + w] = 0;
    for (int64_t t = 0; t < T; ++t) {
      const bool k = now < expire[u * T + t];
      keep[u * T + t] = k ? 1 : 0;
      if (k) {
        bits[u * nw + t / 32] |= 1u << (t % 32);
        ++c;
      }
    }
    count[u] = c;
  });
}

// The lower order statistic at index k_h of the T scores of each (b, h)
// (scores [B, T, H]; NaN ranks above every number), rounded to float32.
void kvpo_threshold(const double* s, int64_t B, int64_t T, int64_t H, const int64_t* k_per_head, float* tau) {
  parallel_for(B * H, [&](int64_t u) {
    const int64_t b = u / H, h = u % H;
    std::vector<double> col(T);
    for (int64_t t = 0; t < T; ++t) col[t] = s[(b * T + t) * H + h];
    std::sort(col.begin(), col.end(), [](double a, double c) {
      if (std::isnan(a)) return false;
      if (std::isnan(c)) return true;
      return a < c;
    });
    tau[u] = static_cast<float>(col[k_per_head[h]]);
  });
}

// ---------------------------------------------------------------- 3. compaction
// [DeInfer] 나.: for every (b, h) in b-major / h-minor order, the positions
// present at `now` in ascending order (the remapping index list); (b, h)
// gets ceil((n + reserve) / 16) consecutive pages after the previous one's;
// slot j is row j % 16 of page base + j / 16. The pages of one (b, h) are
// filled by one worker.
//
// Dense source: K/V [B, T, H, d] bf16 bits, expire [B, H, T]. Outputs as the
// cache's arrays (pools [cap, 16, d], expire_pool [cap, 16], page_table [B,
// H, max_pages], remap [B, H, max_pages * 16], count [B, H]), already set to
// their empty values by the caller. Returns the pages used, or -1 - (b*H+h)
// of the first (b, h) that does not fit.
int64_t kvpo_compact_dense(const uint16_t* k, const uint16_t* v, const int64_t* expire, int64_t B, int64_t T,
                           int64_t H, int64_t d, int64_t now, int64_t reserve, int64_t n_pages_cap,
                           int64_t max_pages, uint16_t* k_pool, uint16_t* v_pool, int64_t* expire_pool,
                           int64_t* page_table, int64_t* remap, int64_t* count) {
  const int64_t BH = B * H;
  std::vector<int64_t> n(BH), base(BH);
  parallel_for(BH, [&](int64_t u) {
    int64_t c = 0;
    for (int64_t t = 0; t < T; ++t) c += now < expire[u * T + t];
    n[u] = c;
  });
  int64_t used = 0;
  for (int64_t u = 0; u < BH; ++u) {
    const int64_t npg = (n[u] + reserve + kPage - 1) / kPage;
    if (npg > max_pages || used + npg > n_pages_cap) return -1 - u;
    base[u] = used;
    used += npg;
  }
  parallel_for(BH, [&](int64_t u) {
    const int64_t b = u / H, h = u % H;
    const int64_t npg = (n[u] + reserve + kPage - 1) / kPage;
    for (int64_t p = 0; p < npg; ++p) page_table[u * max_pages + p] = base[u] + p;
    int64_t j = 0;
    for (int64_t t = 0; t < T; ++t) {
      if (!(now < expire[u * T + t])) continue;
      const int64_t row = (base[u] + j / kPage) * kPage + j % kPage;
      const int64_t src = ((b * T + t) * H + h) * d;
      std::memcpy(k_pool + row * d, k + src, d * 2);
      std::memcpy(v_pool + row * d, v + src, d * 2);
      expire_pool[row] = expire[u * T + t];
      remap[u * max_pages * kPage + j] = t;
      ++j;
    }
    count[u] = j;
  });
  return used;
}

// Recompaction of a paged cache: the slots j < count of every (b, h) whose
// expire is present at `now`, in slot order, carrying remap and expire.
int64_t kvpo_compact_paged(const uint16_t* sk, const uint16_t* sv, const int64_t* sexp, const int64_t* spt,
                           int64_t smax_pages, const int64_t* sremap, const int64_t* scount, int64_t BH, int64_t d,
                           int64_t now, int64_t reserve, int64_t n_pages_cap, int64_t max_pages, uint16_t* k_pool,
                           uint16_t* v_pool, int64_t* expire_pool, int64_t* page_table, int64_t* remap,
                           int64_t* count) {
  std::vector<int64_t> n(BH), base(BH);
  auto src_row = [&](int64_t u, int64_t j) { return spt[u * smax_pages + j / kPage] * kPage + j % kPage; };
  parallel_for(BH, [&](int64_t u) {
    int64_t c = 0;
    for (int64_t j = 0; j < scount[u]; ++j) c += now < sexp[src_row(u, j)];
    n[u] = c;
  });
  int64_t used = 0;
  for (int64_t u = 0; u < BH; ++u) {
    const int64_t npg = (n[u] + reserve + kPage - 1) / kPage;
    if (npg > max_pages || used + npg > n_pages_cap) return -1 - u;
    base[u] = used;
    used += npg;
  }
  parallel_for(BH, [&](int64_t u) {
    const int64_t npg = (n[u] + reserve + kPage - 1) / kPage;
    for (int64_t p = 0; p < npg; ++p) page_table[u * max_pages + p] = base[u] + p;
    int64_t j = 0;
    for (int64_t i = 0; i < scount[u]; ++i) {
      const int64_t r = src_row(u, i);
      if (!(now < sexp[r])) continue;
      const int64_t row = (base[u] + j / kPage) * kPage + j % kPage;
      std::memcpy(k_pool + row * d, sk + r * d, d * 2);
      std::memcpy(v_pool + row * d, sv + r * d, d * 2);
      expire_pool[row] = sexp[r];
      remap[u * max_pages * kPage + j] = sremap[u * smax_pages * kPage + i];
      ++j;
    }
    count[u] = j;
  });
  return used;
}

// Decode-time append: the new token's k/v [B, H, d] into slot count[b, h] of
// its own pages with its expire value. Returns -1 on success, else the first
// (b, h) without a free slot (nothing written for it or after it).
int64_t kvpo_append(uint16_t* k_pool, uint16_t* v_pool, int64_t* expire_pool, const int64_t* page_table,
                    int64_t max_pages, int64_t* remap, int64_t* count, int64_t BH, int64_t d, const uint16_t* k_new,
                    const uint16_t* v_new, int64_t pos, const int64_t* expire_new) {
  for (int64_t u = 0; u < BH; ++u) {
    const int64_t j = count[u], p = j / kPage;
    if (p >= max_pages || page_table[u * max_pages + p] < 0) return u;
    const int64_t row = page_table[u * max_pages + p] * kPage + j % kPage;
    std::memcpy(k_pool + row * d, k_new + u * d, d * 2);
    std::memcpy(v_pool + row * d, v_new + u * d, d * 2);
    expire_pool[row] = expire_new[u];
    remap[u * max_pages * kPage + j] = pos;
    count[u] = j + 1;
  }
  return -1;
}

// ---------------------------------------------------------------- 4. attention
// [DMS] "DMS 작동 방식" step 5: o[b, j] = softmax_i(scale q[b, j] . k_i) v_i
// over the slots i of (b, h = j / g) present at `now`. q [B, Hq, d] bf16
// bits; out [B, Hq, d] float32.
void kvpo_decode_attention(const uint16_t* q, int64_t B, int64_t Hq, int64_t H, int64_t d, const uint16_t* k_pool,
                           const uint16_t* v_pool, const int64_t* expire_pool, const int64_t* page_table,
                           int64_t max_pages, const int64_t* count, int64_t now, double scale, float* out) {
  const int64_t g = Hq / H;
  parallel_for(B * H, [&](int64_t u) {
    const int64_t b = u / H, h = u % H;
    std::vector<double> Kf, Vf;
    Kf.reserve(static_cast<size_t>(count[u]) * d);
    Vf.reserve(static_cast<size_t>(count[u]) * d);
    for (int64_t j = 0; j < count[u]; ++j) {
      const int64_t row = page_table[u * max_pages + j / kPage] * kPage + j % kPage;
      if (!(now < expire_pool[row])) continue;
      for (int64_t e = 0; e < d; ++e) {
        Kf.push_back(widen(k_pool[row * d + e]));
        Vf.push_back(widen(v_pool[row * d + e]));
      }
    }
    const size_t n = Kf.size() / d;
    std::vector<const double*> K(n), V(n);
    for (size_t i = 0; i < n; ++i) {
      K[i] = &Kf[i * d];
      V[i] = &Vf[i * d];
    }
    std::vector<double> qf(d), o(d);
    for (int64_t jq = h * g; jq < (h + 1) * g; ++jq) {
      for (int64_t e = 0; e < d; ++e) qf[e] = widen(q[(b * Hq + jq) * d + e]);
      softmax_attend(qf.data(), static_cast<int>(d), K, V, static_cast<int>(d), scale, o.data());
      for (int64_t e = 0; e < d; ++e) out[(b * Hq + jq) * d + e] = static_cast<float>(o[e]);
    }
  });
}

// The same attention with each row's softmax normaliser on the log scale:
// lse[b, j] = ln sum_i exp(scale q[b, j] . k_i) over the present slots
// (-inf, with a zero row, when there are none). lse [B, Hq] double.
void kvpo_decode_attention_lse(const uint16_t* q, int64_t B, int64_t Hq, int64_t H, int64_t d,
                               const uint16_t* k_pool, const uint16_t* v_pool, const int64_t* expire_pool,
                               const int64_t* page_table, int64_t max_pages, const int64_t* count, int64_t now,
                               double scale, float* out, double* lse) {
  const int64_t g = Hq / H;
  parallel_for(B * H, [&](int64_t u) {
    const int64_t b = u / H, h = u % H;
    std::vector<int64_t> rows;
    for (int64_t j = 0; j < count[u]; ++j) {
      const int64_t row = page_table[u * max_pages + j / kPage] * kPage + j % kPage;
      if (now < expire_pool[row]) rows.push_back(row);
    }
    std::vector<double> qf(d), logit(rows.size()), o(d);
    for (int64_t jq = h * g; jq < (h + 1) * g; ++jq) {
      for (int64_t e = 0; e < d; ++e) qf[e] = widen(q[(b * Hq + jq) * d + e]);
      double m = -INFINITY;
      for (size_t i = 0; i < rows.size(); ++i) {
        double dot = 0.0;
        for (int64_t e = 0; e < d; ++e) dot += widen(k_pool[rows[i] * d + e]) * qf[e];
        logit[i] = dot * scale;
        m = std::max(m, logit[i]);
      }
      double den = 0.0;
      for (int64_t e = 0; e < d; ++e) o[e] = 0.0;
      for (size_t i = 0; i < rows.size(); ++i) {
        const double w = std::exp(logit[i] - m);
        den += w;
        for (int64_t e = 0; e < d; ++e) o[e] += w * widen(v_pool[rows[i] * d + e]);
      }
      for (int64_t e = 0; e < d; ++e) out[(b * Hq + jq) * d + e] = rows.empty() ? 0.f : static_cast<float>(o[e] / den);
      lse[b * Hq + jq] = rows.empty() ? -INFINITY : m + std::log(den);
    }
  });
}

// Attention over the union of disjoint parts from each part's rows
// (normalised over the part) and lse: lse = ln sum_p exp(lse_p), out = sum_p
// exp(lse_p - lse) out_p; parts with lse -inf weigh nothing, a row with none
// is zero with lse -inf. outs [P, rows, d], lses [P, rows] double.
void kvpo_merge_attention(const double* outs, const double* lses, int64_t P, int64_t rows, int64_t d, double* out,
                          double* lse) {
  for (int64_t r = 0; r < rows; ++r) {
    double m = -INFINITY;
    for (int64_t p = 0; p < P; ++p) m = std::max(m, lses[p * rows + r]);
    for (int64_t e = 0; e < d; ++e) out[r * d + e] = 0.0;
    if (m == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double total = 0.0;
    for (int64_t p = 0; p < P; ++p) total += std::exp(lses[p * rows + r] - m);
    for (int64_t p = 0; p < P; ++p) {
      const double w = std::exp(lses[p * rows + r] - m) / total;
      for (int64_t e = 0; e < d; ++e) out[r * d + e] += w * outs[(p * rows + r) * d + e];
    }
    lse[r] = m + std::log(total);
  }
}

// Brute force over the dense cache K/V [B, T, H, d]: every position in
// [lo, now] (no pages, no masks).
void kvpo_dense_attention(const uint16_t* q, int64_t B, int64_t Hq, const uint16_t* k, const uint16_t* v, int64_t T,
                          int64_t H, int64_t d, int64_t lo, int64_t now, double scale, float* out) {
  const int64_t g = Hq / H;
  parallel_for(B * Hq, [&](int64_t u) {
    const int64_t b = u / Hq, jq = u % Hq, h = jq / g;
    std::vector<double> Kf, Vf;
    Kf.reserve(static_cast<size_t>(std::max<int64_t>(0, std::min(now + 1, T) - std::max<int64_t>(lo, 0))) * d);
    Vf.reserve(Kf.capacity());
    for (int64_t t = std::max<int64_t>(lo, 0); t <= now && t < T; ++t) {
      for (int64_t e = 0; e < d; ++e) {
        Kf.push_back(widen(k[((b * T + t) * H + h) * d + e]));
        Vf.push_back(widen(v[((b * T + t) * H + h) * d + e]));
      }
    }
    const size_t n = Kf.size() / d;
    std::vector<const double*> K(n), V(n);
    for (size_t i = 0; i < n; ++i) {
      K[i] = &Kf[i * d];
      V[i] = &Vf[i * d];
    }
    std::vector<double> qf(d), o(d);
    for (int64_t e = 0; e < d; ++e) qf[e] = widen(q[u * d + e]);
    softmax_attend(qf.data(), static_cast<int>(d), K, V, static_cast<int>(d), scale, o.data());
    for (int64_t e = 0; e < d; ++e) out[u * d + e] = static_cast<float>(o[e]);
  });
}

// ---------------------------------------------------------------- 5. fp8 tier
// [BeaconKV]: entries with tau_q <= s < tau (or, with DMS flags, the flagged
// ones) are kept once more as E4M3 codes with one float32 scale per row.
// Selection of the fp8 tier on broadcast (flattened) operands: tau_q <= s < tau
// (NaN never).
void kvpo_quant_select(const double* s, const double* tau, const double* tau_q, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (s[i] >= tau_q[i]) && (s[i] < tau[i]);
}

void kvpo_e4m3_encode(const double* v, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_encode_one(v[i]);
}

void kvpo_e4m3_decode(const uint8_t* c, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_decode_one(c[i]);
}

void kvpo_quantize_rows(const uint16_t* rows, int64_t n_rows, int64_t d, uint8_t* codes, float* scale) {
  for (int64_t r = 0; r < n_rows; ++r) quantize_row(rows + r * d, static_cast<int>(d), codes + r * d, scale + r);
}

// The fp8 tier of a dense source: sel [B, H, T] (1 = goes to the tier),
// start [B, H, T] (its first visible step); pages as kvpo_compact_dense.
int64_t kvpo_compact_quant_dense(const uint16_t* k, const uint16_t* v, const uint8_t* sel, const int64_t* start,
                                 int64_t B, int64_t T, int64_t H, int64_t d, int64_t reserve, int64_t n_pages_cap,
                                 int64_t max_pages, uint8_t* kq_pool, uint8_t* vq_pool, float* kscale,
                                 float* vscale, int64_t* start_pool, int64_t* page_table, int64_t* remap,
                                 int64_t* count) {
  const int64_t BH = B * H;
  std::vector<int64_t> n(BH), base(BH);
  parallel_for(BH, [&](int64_t u) {
    int64_t c = 0;
    for (int64_t t = 0; t < T; ++t) c += sel[u * T + t] != 0;
    n[u] = c;
  });
  int64_t used = 0;
  for (int64_t u = 0; u < BH; ++u) {
    const int64_t npg = (n[u] + reserve + kPage - 1) / kPage;
    if (npg > max_pages || used + npg > n_pages_cap) return -1 - u;
    base[u] = used;
    used += npg;
  }
  parallel_for(BH, [&](int64_t u) {
    const int64_t b = u / H, h = u % H;
    const int64_t npg = (n[u] + reserve + kPage - 1) / kPage;
    for (int64_t p = 0; p < npg; ++p) page_table[u * max_pages + p] = base[u] + p;
    int64_t j = 0;
    for (int64_t t = 0; t < T; ++t) {
      if (!sel[u * T + t]) continue;
      const int64_t row = (base[u] + j / kPage) * kPage + j % kPage;
      const int64_t src = ((b * T + t) * H + h) * d;
      quantize_row(k + src, static_cast<int>(d), kq_pool + row * d, kscale + row);
      quantize_row(v + src, static_cast<int>(d), vq_pool + row * d, vscale + row);
      start_pool[row] = start[u * T + t];
      remap[u * max_pages * kPage + j] = t;
      ++j;
    }
    count[u] = j;
  });
  return used;
}

// Decode-time append into the fp8 tier of the (b, h) with sel[u] set.
int64_t kvpo_append_quant(uint8_t* kq_pool, uint8_t* vq_pool, float* kscale, float* vscale, int64_t* start_pool,
                          const int64_t* page_table, int64_t max_pages, int64_t* remap, int64_t* count, int64_t BH,
                          int64_t d, const uint16_t* k_new, const uint16_t* v_new, int64_t pos, const uint8_t* sel,
                          const int64_t* start_new) {
  for (int64_t u = 0; u < BH; ++u) {
    if (!sel[u]) continue;
    const int64_t j = count[u], p = j / kPage;
    if (p >= max_pages || page_table[u * max_pages + p] < 0) return u;
    const int64_t row = page_table[u * max_pages + p] * kPage + j % kPage;
    quantize_row(k_new + u * d, static_cast<int>(d), kq_pool + row * d, kscale + row);
    quantize_row(v_new + u * d, static_cast<int>(d), vq_pool + row * d, vscale + row);
    start_pool[row] = start_new[u];
    remap[u * max_pages * kPage + j] = pos;
    count[u] = j + 1;
  }
  return -1;
}

// Attention over the bf16 tier's slots present at `now` and the fp8 tier's
// slots visible at `now` (now >= start), the latter dequantized exactly
// (code value times the row's scale).
void kvpo_decode_attention_two_tier(const uint16_t* q, int64_t B, int64_t Hq, int64_t H, int64_t d,
                                    const uint16_t* k_pool, const uint16_t* v_pool, const int64_t* expire_pool,
                                    const int64_t* page_table, int64_t max_pages, const int64_t* count,
                                    const uint8_t* kq_pool, const uint8_t* vq_pool, const float* kscale,
                                    const float* vscale, const int64_t* start_pool, const int64_t* page_table_q,
                                    int64_t max_pages_q, const int64_t* count_q, int64_t now, double scale,
                                    float* out) {
  const int64_t g = Hq / H;
  parallel_for(B * H, [&](int64_t u) {
    const int64_t b = u / H, h = u % H;
    std::vector<double> Kf, Vf;
    Kf.reserve(static_cast<size_t>(count[u]) * d);
    Vf.reserve(static_cast<size_t>(count[u]) * d);
    for (int64_t j = 0; j < count[u]; ++j) {
      const int64_t row = page_table[u * max_pages + j / kPage] * kPage + j % kPage;
      if (!(now < expire_pool[row])) continue;
      for (int64_t e = 0; e < d; ++e) {
        Kf.push_back(widen(k_pool[row * d + e]));
        Vf.push_back(widen(v_pool[row * d + e]));
      }
    }
    for (int64_t j = 0; j < count_q[u]; ++j) {
      const int64_t row = page_table_q[u * max_pages_q + j / kPage] * kPage + j % kPage;
      if (!(now >= start_pool[row])) continue;
      for (int64_t e = 0; e < d; ++e) {
        Kf.push_back(e4m3_decode_one(kq_pool[row * d + e]) * static_cast<double>(kscale[row]));
        Vf.push_back(e4m3_decode_one(vq_pool[row * d + e]) * static_cast<double>(vscale[row]));
      }
    }
    const size_t n = Kf.size() / d;
    std::vector<const double*> K(n), V(n);
    for (size_t i = 0; i < n; ++i) {
      K[i] = &Kf[i * d];
      V[i] = &Vf[i * d];
    }
    std::vector<double> qf(d), o(d);
    for (int64_t jq = h * g; jq < (h + 1) * g; ++jq) {
      for (int64_t e = 0; e < d; ++e) qf[e] = widen(q[(b * Hq + jq) * d + e]);
      softmax_attend(qf.data(), static_cast<int>(d), K, V, static_cast<int>(d), scale, o.data());
      for (int64_t e = 0; e < d; ++e) out[(b * Hq + jq) * d + e] = static_cast<float>(o[e]);
    }
  });
}

// ---------------------------------------------------------------- 6. MLA latent cache
// [DMS] "주요 요점" / "앞으로의 전망": one latent row [c_t, k_rope_t] per token
// kept or dropped whole; absorbed decode attention: query head j's logit
// against slot t is scale q_j . row_t and its output the weighted sum of the
// rows' first dc values. The latent cache is the paged cache with one kv
// head (rows in the K pool).
void kvpo_decode_attention_mla(const uint16_t* q, int64_t B, int64_t Hq, int64_t R, int64_t dc,
                               const uint16_t* pool, const int64_t* expire_pool, const int64_t* page_table,
                               int64_t max_pages, const int64_t* count, int64_t now, double scale, float* out) {
  parallel_for(B, [&](int64_t b) {
    std::vector<double> C;
    C.reserve(static_cast<size_t>(count[b]) * R);
    for (int64_t j = 0; j < count[b]; ++j) {
      const int64_t row = page_table[b * max_pages + j / kPage] * kPage + j % kPage;
      if (!(now < expire_pool[row])) continue;
      for (int64_t e = 0; e < R; ++e) C.push_back(widen(pool[row * R + e]));
    }
    const size_t n = C.size() / R;
    std::vector<const double*> K(n);
    for (size_t i = 0; i < n; ++i) K[i] = &C[i * R];
    std::vector<double> qf(R), o(dc);
    for (int64_t jq = 0; jq < Hq; ++jq) {
      for (int64_t e = 0; e < R; ++e) qf[e] = widen(q[(b * Hq + jq) * R + e]);
      softmax_attend(qf.data(), static_cast<int>(R), K, K, static_cast<int>(dc), scale, o.data());
      for (int64_t e = 0; e < dc; ++e) out[(b * Hq + jq) * dc + e] = static_cast<float>(o[e]);
    }
  });
}

// ---------------------------------------------------------------- closed forms
// [KVzap] "이게 뭔데?": K and V, one d_model-wide row each per token per layer.
int64_t kvpo_kv_cache_bytes(int64_t n_layers, int64_t d_model, int64_t n_tokens, int64_t elem_bytes) {
  return 2 * n_layers * d_model * n_tokens * elem_bytes;
}

// Per-token multiply-adds of a decoder layer's Q, K, V, O and feed-forward projections.
int64_t kvpo_linear_projection_macs(int64_t d_model, int64_t n_q_heads, int64_t n_kv_heads, int64_t head_dim,
                                    int64_t ffn_hidden, int gated) {
  return 2 * d_model * n_q_heads * head_dim + 2 * d_model * n_kv_heads * head_dim +
         (gated ? 3 : 2) * d_model * ffn_hidden;
}

// [KVzap] "메모리 및 계산 효율": per-token multiply-adds of the surrogate
// (hidden <= 0: the linear one).
int64_t kvpo_scorer_macs(int64_t d_model, int64_t n_kv_heads, int64_t hidden) {
  return hidden <= 0 ? d_model * n_kv_heads : d_model * hidden + hidden * n_kv_heads;
}

}  // extern "C"
