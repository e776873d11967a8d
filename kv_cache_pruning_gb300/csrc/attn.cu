// kvp_decode_attn: split-KV single-query GQA attention over the compacted
// pages (DMS article, "DMS 작동 방식" step 5: standard attention over the kept
// cache).
//
// Grid (split, kv head, batch); each CTA reads up to `pps` pages of one
// (b, h). Its 4 warps take every 4th page; each warp owns a ring of NST
// stages that its lane 0 fills with 1-D bulk copies (K page, V page, the
// page's 16 expire values) completing on an mbarrier.
//
// Lane layout per warp: LPR = D/8 lanes cover one row (8 bf16 = 16 bytes
// each), RPS = 32/LPR rows are processed per step, RS = 16/RPS steps per page.
// q . k partial sums of all G heads and RS steps are reduced across the LPR
// lanes with a transposing butterfly (each exchange halves the values a lane
// holds), then masked (slot < count and now < expire), and an fp32 online
// softmax in base 2 (q is pre-scaled by scale*log2 e) updates the running
// max, sum and the G x 8 output accumulators of the lane. The 4 warps' states
// are merged in shared memory, one partial (acc, m, l) per (b, q head, split)
// goes to the workspace, and a second kernel merges the splits.
#include "kvp_common.cuh"

namespace kvp {
namespace {

constexpr int kWarps = 4;
constexpr int kNst = 3;

template <int D, int G>
struct AttnCfg {
  static constexpr int LPR = D / 8;
  static constexpr int RPS = 32 / LPR;
  static constexpr int RS = kPage / RPS;
  static constexpr int V = RS * G;
  static constexpr int VL = V >= LPR ? V / LPR : 1;
  static constexpr int DUP = V >= LPR ? 1 : LPR / V;
  static constexpr int GL = LPR / G;
  static constexpr int PAGE_BYTES = kPage * D * 2;
  static constexpr int STAGE_BYTES = 2 * PAGE_BYTES + kPage * 4;
  static constexpr int STAGES_BYTES = kWarps * kNst * STAGE_BYTES;
  static constexpr int PS_FLOATS = RPS * G * RS;  // per warp
  static constexpr int PS_BYTES = kWarps * PS_FLOATS * 4;
  static constexpr int BAR_BYTES = kWarps * kNst * 8;
  static constexpr int MERGE_BYTES = kWarps * G * (D + 2) * 4;
  static constexpr int SMEM = STAGES_BYTES + PS_BYTES + BAR_BYTES + MERGE_BYTES;
  static_assert(G <= LPR, "group larger than lanes per row");
  static_assert(STAGE_BYTES % 16 == 0 && PS_BYTES % 16 == 0, "16-byte layout");
};

struct AttnParams {
  const uint16_t* q;
  const uint16_t* k_pool;
  const uint16_t* v_pool;
  const int32_t* expire_pool;
  const int32_t* page_table;
  const int32_t* count;
  int H, Hq, max_pages, n_pages_cap, now, pps, n_splits;
  float qscale;
  float* part_acc;  // [B, Hq, n_splits, D]
  float* part_ml;   // [B, Hq, n_splits, 2]
  int32_t* status;
};

// Transposing butterfly: N values per lane, exchange partner lane ^ O. After
// each exchange a lane keeps the half of the index range selected by bit O of
// its lane id, summed with its partner's copy of that half.
template <int N, int O>
struct TransposeReduce {
  static KVP_DEV void run(float* v, int lane) {
    if constexpr (O == 0) {
      return;
    } else if constexpr (N == 1) {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
      TransposeReduce<1, O / 2>::run(v, lane);
    } else {
      const bool up = (lane & O) != 0;
#pragma unroll
      for (int k = 0; k < N / 2; ++k) {
        const float send = up ? v[k] : v[k + N / 2];
        const float keep = up ? v[k + N / 2] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      TransposeReduce<N / 2, O / 2>::run(v, lane);
    }
  }
};

KVP_DEV void unpack8(const uint4& w, float (&f)[8]) {
  f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x);
  f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
  f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z);
  f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
}

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32) attn_split_kernel(const AttnParams p) {
  using C = AttnCfg<D, G>;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int bh = b * p.H + h;
  const int cnt = min(max(p.count[bh], 0), p.max_pages * kPage);
  const int npages = (cnt + kPage - 1) / kPage;
  const int pg0 = split * p.pps;
  if (pg0 >= npages) return;  // whole CTA: nothing of this (b, h) falls in this split
  const int pg1 = min(npages, pg0 + p.pps);

  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = smem + warp * kNst * C::STAGE_BYTES;
  float* p_s = reinterpret_cast<float*>(smem + C::STAGES_BYTES) + warp * C::PS_FLOATS;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::STAGES_BYTES + C::PS_BYTES) + warp * kNst;
  float* merge = reinterpret_cast<float*>(smem + C::STAGES_BYTES + C::PS_BYTES + C::BAR_BYTES);

  const int rowsel = lane / C::LPR;
  const int s = lane % C::LPR;

  float qf[G][8];
#pragma unroll
  for (int i = 0; i < G; ++i) {
    const uint4 w =
        __ldg(reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(b) * p.Hq + h * G + i) * D) + s);
    unpack8(w, qf[i]);
#pragma unroll
    for (int e = 0; e < 8; ++e) qf[i][e] *= p.qscale;
  }

  const int first = pg0 + warp;
  const int nk = first < pg1 ? (pg1 - first + kWarps - 1) / kWarps : 0;
  const int32_t* ptab = p.page_table + static_cast<int64_t>(bh) * p.max_pages;

  auto issue = [&](int k) {
    const int st = k % kNst;
    const int64_t phys = ptab[first + k * kWarps];
    uint8_t* dst = ring + st * C::STAGE_BYTES;
    if (phys < 0 || phys >= p.n_pages_cap) {
      // inconsistent page table: no copy; the stage reads as an empty page
      record_error(p.status, KVP_ERR_BOUNDS);
      uint4* z = reinterpret_cast<uint4*>(dst);
      for (int i = 0; i < C::STAGE_BYTES / 16; ++i) z[i] = make_uint4(0, 0, 0, 0);
      mbar_arrive(&bars[st]);
      return;
    }
    mbar_arrive_expect_tx(&bars[st], C::STAGE_BYTES);
    bulk_g2s(dst, p.k_pool + phys * kPage * D, C::PAGE_BYTES, &bars[st]);
    bulk_g2s(dst + C::PAGE_BYTES, p.v_pool + phys * kPage * D, C::PAGE_BYTES, &bars[st]);
    bulk_g2s(dst + 2 * C::PAGE_BYTES, p.expire_pool + phys * kPage, kPage * 4, &bars[st]);
  };

  if (lane == 0) {
    for (int st = 0; st < kNst; ++st) mbar_init(&bars[st], 1);
    fence_mbar_init();
    for (int k = 0; k < nk && k < kNst; ++k) issue(k);
  }
  __syncwarp();

  float m_run[G], l_run[G], acc[G][8];
#pragma unroll
  for (int i = 0; i < G; ++i) {
    m_run[i] = -1e30f;
    l_run[i] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
  }

  const int idx_base = (C::V >= C::LPR) ? s * C::VL : s / C::DUP;
  const int my_head = idx_base / C::RS;

  for (int k = 0; k < nk; ++k) {
    const int st = k % kNst;
    const bool ok = mbar_wait(&bars[st], static_cast<uint32_t>((k / kNst) & 1), nullptr, p.status);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) record_error(p.status, KVP_ERR_TIMEOUT);
      break;
    }
    const uint8_t* stage = ring + st * C::STAGE_BYTES;
    const uint16_t* Ks = reinterpret_cast<const uint16_t*>(stage);
    const uint16_t* Vs = reinterpret_cast<const uint16_t*>(stage + C::PAGE_BYTES);
    const int32_t* Es = reinterpret_cast<const int32_t*>(stage + 2 * C::PAGE_BYTES);
    const int page = first + k * kWarps;

    // ---- logits: partial dot products, then reduce across the row's lanes
    float part[C::V];
#pragma unroll
    for (int t = 0; t < C::RS; ++t) {
      const int r = t * C::RPS + rowsel;
      float kf[8];
      unpack8(reinterpret_cast<const uint4*>(Ks + r * D)[s], kf);
#pragma unroll
      for (int i = 0; i < G; ++i) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) a = fmaf(qf[i][e], kf[e], a);
        part[i * C::RS + t] = a;
      }
    }
    TransposeReduce<C::V, C::LPR / 2>::run(part, lane);

    float x[C::VL];
    float mloc = -INFINITY;
#pragma unroll
    for (int u = 0; u < C::VL; ++u) {
      const int idx = idx_base + u;
      const int r = (idx % C::RS) * C::RPS + rowsel;
      const bool valid = (page * kPage + r < cnt) && (p.now < Es[r]);
      x[u] = valid ? part[u] : -INFINITY;
      mloc = fmaxf(mloc, x[u]);
    }
#pragma unroll
    for (int o = 1; o < C::GL; o <<= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
#pragma unroll
    for (int o = C::LPR; o < 32; o <<= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));

    float alpha[G];
#pragma unroll
    for (int i = 0; i < G; ++i) {
      const float mi = __shfl_sync(0xffffffffu, mloc, i * C::GL);
      const float mnew = fmaxf(m_run[i], mi);
      alpha[i] = exp2f(m_run[i] - mnew);
      m_run[i] = mnew;
    }
    float mh = m_run[0];
#pragma unroll
    for (int i = 1; i < G; ++i)
      if (my_head == i) mh = m_run[i];
#pragma unroll
    for (int u = 0; u < C::VL; ++u) {
      const float pv = exp2f(x[u] - mh);
      if (s % C::DUP == 0) p_s[rowsel * G * C::RS + idx_base + u] = pv;
    }
    __syncwarp();

    // ---- rescale and accumulate P . V for this lane's rows and columns
#pragma unroll
    for (int i = 0; i < G; ++i) {
      l_run[i] *= alpha[i];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[i][e] *= alpha[i];
    }
#pragma unroll
    for (int t = 0; t < C::RS; ++t) {
      const int r = t * C::RPS + rowsel;
      float vf[8];
      unpack8(reinterpret_cast<const uint4*>(Vs + r * D)[s], vf);
#pragma unroll
      for (int i = 0; i < G; ++i) {
        const float pr = p_s[rowsel * G * C::RS + i * C::RS + t];
        l_run[i] += pr;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(pr, vf[e], acc[i][e]);
      }
    }
    __syncwarp();
    if (lane == 0 && k + kNst < nk) {
      fence_proxy_async();
      issue(k + kNst);
    }
  }

  // ---- combine the RPS row groups of the warp
#pragma unroll
  for (int o = C::LPR; o < 32; o <<= 1) {
#pragma unroll
    for (int i = 0; i < G; ++i) {
      l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], o);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[i][e] += __shfl_xor_sync(0xffffffffu, acc[i][e], o);
    }
  }
  if (rowsel == 0) {
#pragma unroll
    for (int i = 0; i < G; ++i) {
      float* mrow = merge + (warp * G + i) * (D + 2);
#pragma unroll
      for (int e = 0; e < 8; ++e) mrow[8 * s + e] = acc[i][e];
      if (s == 0) {
        mrow[D] = m_run[i];
        mrow[D + 1] = l_run[i];
      }
    }
  }
  __syncthreads();

  // ---- merge the warps into this split's partial
  for (int idx = threadIdx.x; idx < G * D; idx += kWarps * 32) {
    const int i = idx / D, e = idx - i * D;
    float M = -1e30f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, merge[(w * G + i) * (D + 2) + D]);
    float L = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float* mrow = merge + (w * G + i) * (D + 2);
      const float sc = exp2f(mrow[D] - M);
      L = fmaf(sc, mrow[D + 1], L);
      A = fmaf(sc, mrow[e], A);
    }
    const size_t o = (static_cast<size_t>(b) * p.Hq + h * G + i) * p.n_splits + split;
    p.part_acc[o * D + e] = A;
    if (e == 0) {
      p.part_ml[o * 2] = M;
      p.part_ml[o * 2 + 1] = L;
    }
  }
}

// out[b, j] = sum_s 2^(m_s - M) acc_s / sum_s 2^(m_s - M) l_s over the splits
// that hold pages of (b, h = j / G); zero when nothing is present.
__global__ void attn_merge_kernel(int H, int Hq, int G, int D, int pps, int n_splits, int max_pages,
                                  const int32_t* __restrict__ count,
                                  const float* __restrict__ part_acc, const float* __restrict__ part_ml,
                                  float* __restrict__ out) {
  const int j = blockIdx.x, b = blockIdx.y;
  const int h = j / G;
  const int cnt = min(max(count[b * H + h], 0), max_pages * kPage);
  const int npages = (cnt + kPage - 1) / kPage;
  const int ns = min(n_splits, (npages + pps - 1) / pps);
  const size_t base = (static_cast<size_t>(b) * Hq + j) * n_splits;
  float M = -1e30f;
  for (int sp = 0; sp < ns; ++sp) M = fmaxf(M, part_ml[(base + sp) * 2]);
  for (int e = threadIdx.x; e < D; e += blockDim.x) {
    float L = 0.f, A = 0.f;
    for (int sp = 0; sp < ns; ++sp) {
      const float sc = exp2f(part_ml[(base + sp) * 2] - M);
      L = fmaf(sc, part_ml[(base + sp) * 2 + 1], L);
      A = fmaf(sc, part_acc[(base + sp) * D + e], A);
    }
    out[(static_cast<size_t>(b) * Hq + j) * D + e] = L > 0.f ? A / L : 0.f;
  }
}

template <int D, int G>
kvp_status launch_attn(const AttnParams& p, int B, cudaStream_t st) {
  using C = AttnCfg<D, G>;
  auto kern = attn_split_kernel<D, G>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
    return KVP_ERR_CUDA;
  kern<<<dim3(p.n_splits, p.H, B), kWarps * 32, C::SMEM, st>>>(p);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

template <int D>
kvp_status dispatch_g(const AttnParams& p, int B, int G, cudaStream_t st) {
  switch (G) {
    case 1: return launch_attn<D, 1>(p, B, st);
    case 2: return launch_attn<D, 2>(p, B, st);
    case 4: return launch_attn<D, 4>(p, B, st);
    case 8: return launch_attn<D, 8>(p, B, st);
    default: return KVP_ERR_UNSUPPORTED;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int pps_or_default(int pps) { return pps > 0 ? pps : 16; }

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" size_t kvp_decode_attn_workspace_bytes(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                                  int max_pages, int pages_per_split) {
  if (batch <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || max_pages < 0) return 0;
  const int pps = pps_or_default(pages_per_split);
  const size_t ns = max_pages > 0 ? (max_pages + pps - 1) / pps : 1;
  return static_cast<size_t>(batch) * n_q_heads * ns * (head_dim + 2) * sizeof(float);
}

extern "C" kvp_status kvp_decode_attn(int batch, int n_q_heads, int n_kv_heads, int head_dim, const void* q,
                                      const void* k_pool, const void* v_pool, const int32_t* expire_pool,
                                      int n_pages_cap, const int32_t* page_table, int max_pages,
                                      const int32_t* count, int now, float scale, float* out, int pages_per_split,
                                      void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
  if (batch <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || max_pages < 0 || pages_per_split < 0 || n_pages_cap < 0)
    return KVP_ERR_INVALID;
  if (static_cast<int64_t>(max_pages) * kPage > 0x7fffffff) return KVP_ERR_UNSUPPORTED;
  if (n_q_heads % n_kv_heads != 0) return KVP_ERR_INVALID;
  const int G = n_q_heads / n_kv_heads;
  if (head_dim != 64 && head_dim != 128) return KVP_ERR_UNSUPPORTED;
  if (G != 1 && G != 2 && G != 4 && G != 8) return KVP_ERR_UNSUPPORTED;
  if (!(scale >= 0.f)) return KVP_ERR_INVALID;
  if (q == nullptr || k_pool == nullptr || v_pool == nullptr || expire_pool == nullptr || page_table == nullptr ||
      count == nullptr || out == nullptr)
    return KVP_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(expire_pool)) return KVP_ERR_ALIGN;
  const size_t need =
      kvp_decode_attn_workspace_bytes(batch, n_q_heads, n_kv_heads, head_dim, max_pages, pages_per_split);
  if (workspace == nullptr || workspace_bytes < need) return KVP_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KVP_ERR_ALIGN;
  if (static_cast<int64_t>(batch) * n_kv_heads > 65535 * 65535LL || n_kv_heads > 65535 || batch > 65535)
    return KVP_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int pps = pps_or_default(pages_per_split);
  const int ns = max_pages > 0 ? (max_pages + pps - 1) / pps : 1;
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(head_dim));
  float* part_acc = static_cast<float*>(workspace);
  float* part_ml = part_acc + static_cast<size_t>(batch) * n_q_heads * ns * head_dim;
  AttnParams p{static_cast<const uint16_t*>(q),
               static_cast<const uint16_t*>(k_pool),
               static_cast<const uint16_t*>(v_pool),
               expire_pool,
               page_table,
               count,
               n_kv_heads,
               n_q_heads,
               max_pages,
               n_pages_cap,
               now,
               pps,
               ns,
               sc * 1.4426950408889634f,
               part_acc,
               part_ml,
               status};
  if (max_pages > 0) {
    const kvp_status s = head_dim == 128 ? dispatch_g<128>(p, batch, G, st) : dispatch_g<64>(p, batch, G, st);
    if (s != KVP_OK) return s;
  }
  attn_merge_kernel<<<dim3(n_q_heads, batch), head_dim, 0, st>>>(n_kv_heads, n_q_heads, G, head_dim, pps, ns, max_pages, count,
                                                                 part_acc, part_ml, out);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}
