// kvp_mask, kvp_compact, kvp_compact_paged, kvp_append.
//
// Rules (KVzap summary "실제 적용"; DMS article "지연 삭제 (Delayed Eviction)"):
// an entry gets the first step at which it is gone,
//   KVZAP  expire = score >= tau ? never : pos + window
//   DMS    expire = flag < 0 ? never : max(flag + delay, pos + window)
// and is present at step `now` iff now < expire.
//
// Compaction (DeInfer summary, "나. 페이지드 KV 캐시 및 CUDA Graph 통합"):
// a preparation pass counts the present entries of each 1024-entry chunk of
// every (b, h) (warp ballots), a single-CTA scan turns the counts into the
// remapping offsets and the page base of every (b, h), and a copy pass
// re-derives each entry's slot from a block-wide prefix sum of ballots and
// moves its K and V rows with 16-byte vector loads and stores.
#include "kvp_common.cuh"

namespace kvp {
namespace {

constexpr int kChunk = 1024;        // entries per counting / copying CTA
constexpr int kCopyThreads = 256;   // 8 warps; 256 entries per round

KVP_DEV int32_t expire_kvzap(float s, float tau, int pos, int window) {
  return (s >= tau) ? kNever : pos + window;  // NaN compares false: treated as low
}
KVP_DEV int32_t expire_dms(int flag, int pos, int delay, int window) {
  return flag < 0 ? kNever : max(flag + delay, pos + window);
}

// ------------------------------------------------------------------ mask
__global__ void __launch_bounds__(1024) mask_kernel(int mode, int H, int n_pos, int pos0,
                                                    const float* __restrict__ scores, const float* __restrict__ tau,
                                                    const int32_t* __restrict__ flag, int window, int delay, int now,
                                                    int32_t* __restrict__ expire, uint32_t* __restrict__ keep_bits,
                                                    int32_t* __restrict__ count) {
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh - b * H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float th = (mode == KVP_MASK_KVZAP) ? tau[bh] : 0.f;
  const int n_words = (n_pos + 31) >> 5;
  int kept = 0;
  for (int t0 = 0; t0 < n_pos; t0 += blockDim.x) {
    const int t = t0 + threadIdx.x;
    bool keep = false;
    if (t < n_pos) {
      int32_t e;
      if (mode == KVP_MASK_KVZAP) {
        e = expire_kvzap(scores[(static_cast<int64_t>(b) * n_pos + t) * H + h], th, pos0 + t, window);
      } else {
        e = expire_dms(flag[static_cast<int64_t>(bh) * n_pos + t], pos0 + t, delay, window);
      }
      expire[static_cast<int64_t>(bh) * n_pos + t] = e;
      keep = now < e;
    }
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    const int word = (t0 >> 5) + warp;
    if (lane == 0 && word < n_words) {
      if (keep_bits) keep_bits[static_cast<int64_t>(bh) * n_words + word] = bal;
      kept += __popc(bal);
    }
  }
  __shared__ int sums[32];
  if (lane == 0) sums[warp] = kept;
  __syncthreads();
  if (threadIdx.x == 0) {
    int total = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) total += sums[w];
    if (count) count[bh] = total;
  }
}

// ------------------------------------------------------------------ sources
// Dense source: entry t of (b, h) is row (b, t, h) of K/V, present iff
// now < expire[b, h, t].
struct DenseSrc {
  const uint16_t* k;
  const uint16_t* v;
  int64_t sb, st, sh;
  const int32_t* expire;  // [B, H, n]
  int H;
  int n;                  // entries per (b, h)
  KVP_DEV int length(int) const { return n; }
  KVP_DEV int32_t expire_of(int bh, int t) const { return expire[static_cast<int64_t>(bh) * n + t]; }
  KVP_DEV int position_of(int, int t) const { return t; }
  KVP_DEV const uint16_t* k_row(int bh, int t) const {
    const int b = bh / H, h = bh - b * H;
    return k + b * sb + t * st + h * sh;
  }
  KVP_DEV const uint16_t* v_row(int bh, int t) const {
    const int b = bh / H, h = bh - b * H;
    return v + b * sb + t * st + h * sh;
  }
};

// Paged source: entry j of (b, h) is slot j (< count, clamped to the page
// table) of its pages. A page id outside the pool is recorded and its slots
// read as absent; no row of it is ever touched.
struct PagedSrc {
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* expire_pool;
  const int32_t* page_table;
  const int32_t* remap;
  const int32_t* count;
  int max_pages;
  int n_pages_cap;
  int d;
  int32_t* status;
  KVP_DEV int length(int bh) const { return min(max(count[bh], 0), max_pages * kPage); }
  KVP_DEV int64_t row_index(int bh, int j) const {
    const int pg = page_table[static_cast<int64_t>(bh) * max_pages + (j >> 4)];
    if (pg < 0 || pg >= n_pages_cap) return -1;
    return static_cast<int64_t>(pg) * kPage + (j & 15);
  }
  KVP_DEV int32_t expire_of(int bh, int j) const {
    const int64_t r = row_index(bh, j);
    if (r < 0) {
      record_error(status, KVP_ERR_BOUNDS);
      return 0;
    }
    return expire_pool[r];
  }
  KVP_DEV int position_of(int bh, int j) const {
    return remap[static_cast<int64_t>(bh) * max_pages * kPage + j];
  }
  KVP_DEV const uint16_t* k_row(int bh, int j) const { return k + row_index(bh, j) * d; }
  KVP_DEV const uint16_t* v_row(int bh, int j) const { return v + row_index(bh, j) * d; }
};

// Workspace layout (int32): chunk counts [BH*NC], chunk offsets [BH*NC],
// page base [BH], flag [1] (1 = budget ok).
struct CompactWs {
  int32_t* chunk_cnt;
  int32_t* chunk_off;
  int32_t* base;
  int32_t* ok;
};
size_t compact_ws_bytes(int BH, int NC) { return (static_cast<size_t>(2) * BH * NC + BH + 1) * sizeof(int32_t); }
CompactWs carve(void* ws, int BH, int NC) {
  int32_t* p = static_cast<int32_t*>(ws);
  return CompactWs{p, p + static_cast<size_t>(BH) * NC, p + static_cast<size_t>(2) * BH * NC,
                   p + static_cast<size_t>(2) * BH * NC + BH};
}

// Preparation, part 1: present entries per chunk.
template <class Src>
__global__ void __launch_bounds__(256) count_kernel(Src src, int now, int NC, int32_t* __restrict__ chunk_cnt) {
  const int bh = blockIdx.y, c = blockIdx.x;
  const int n = src.length(bh);
  const int lo = c * kChunk;
  int kept = 0;
  for (int t = lo + threadIdx.x; t < lo + kChunk && t < n; t += blockDim.x) kept += (now < src.expire_of(bh, t));
  kept = __reduce_add_sync(0xffffffffu, kept);
  __shared__ int sums[8];
  if ((threadIdx.x & 31) == 0) sums[threadIdx.x >> 5] = kept;
  __syncthreads();
  if (threadIdx.x == 0) {
    int total = 0;
    for (int w = 0; w < 8; ++w) total += sums[w];
    chunk_cnt[static_cast<int64_t>(bh) * NC + c] = total;
  }
}

// Preparation, part 2 (one CTA): per-(b, h) counts, chunk offsets, page bases
// in (b-major, h-minor) order, budget checks.
__global__ void __launch_bounds__(1024) scan_kernel(int BH, int NC, int reserve, int max_pages, int n_pages_cap,
                                                    CompactWs ws, int32_t* __restrict__ count,
                                                    int32_t* __restrict__ status) {
  __shared__ int warp_tot[32];
  __shared__ int carry_s;
  __shared__ int bad_s;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    carry_s = 0;
    bad_s = 0;
  }
  __syncthreads();
  for (int b0 = 0; b0 < BH; b0 += 1024) {
    const int bh = b0 + tid;
    int pages = 0;
    if (bh < BH) {
      int cnt = 0;
      for (int c = 0; c < NC; ++c) {
        ws.chunk_off[static_cast<int64_t>(bh) * NC + c] = cnt;
        cnt += ws.chunk_cnt[static_cast<int64_t>(bh) * NC + c];
      }
      count[bh] = cnt;
      pages = (cnt + reserve + kPage - 1) / kPage;
      if (pages > max_pages) atomicExch(&bad_s, 1);
    }
    // block-wide exclusive scan of pages
    int incl = pages;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int wt = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wt, o);
        if (lane >= o) wt += y;
      }
      warp_tot[lane] = wt;  // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_tot[warp - 1] : 0) + incl - pages;
    const int carry = carry_s;
    if (bh < BH) ws.base[bh] = carry + before;
    __syncthreads();
    if (tid == 0) carry_s = carry + warp_tot[31];
    __syncthreads();
  }
  if (tid == 0) {
    const bool ok = !bad_s && carry_s <= n_pages_cap;
    ws.ok[0] = ok ? 1 : 0;
    if (!ok) record_error(status, KVP_ERR_CAPACITY);
  }
}

// Copy pass: one CTA per (chunk, b*H + h).
template <int D, class Src>
__global__ void __launch_bounds__(kCopyThreads) scatter_kernel(Src src, int now, int NC, int reserve, int max_pages,
                                                               CompactWs ws, const int32_t* __restrict__ count,
                                                               uint16_t* __restrict__ k_pool,
                                                               uint16_t* __restrict__ v_pool,
                                                               int32_t* __restrict__ expire_pool,
                                                               int32_t* __restrict__ page_table,
                                                               int32_t* __restrict__ remap) {
  constexpr int VPR = D / 8;            // 16-byte vectors per row
  constexpr int EPP = 32 / (2 * VPR);   // entries copied per warp pass (K and V rows)
  if (ws.ok[0] == 0) return;
  const int bh = blockIdx.y, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = src.length(bh);
  const int cnt = count[bh];
  const int base = ws.base[bh];
  const int pages = (cnt + reserve + kPage - 1) / kPage;
  const int64_t cap = static_cast<int64_t>(max_pages) * kPage;

  // page table row and remap tail, split across this (b, h)'s chunk CTAs
  {
    const int seg = (max_pages + NC - 1) / NC;
    for (int p = c * seg + threadIdx.x; p < min(max_pages, (c + 1) * seg); p += blockDim.x)
      page_table[static_cast<int64_t>(bh) * max_pages + p] = p < pages ? base + p : -1;
    const int64_t rseg = (cap + NC - 1) / NC;
    for (int64_t j = c * rseg + threadIdx.x; j < min(cap, (c + 1) * rseg); j += blockDim.x)
      if (j >= cnt) remap[bh * cap + j] = -1;
  }
  // zero the unused rows of this (b, h)'s pages
  if (c == 0) {
    for (int j = cnt + warp; j < pages * kPage; j += kCopyThreads / 32) {
      const int64_t row = static_cast<int64_t>(base + (j >> 4)) * kPage + (j & 15);
      if (lane < VPR) {
        reinterpret_cast<uint4*>(k_pool + row * D)[lane] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4*>(v_pool + row * D)[lane] = make_uint4(0, 0, 0, 0);
      }
      if (lane == 0) expire_pool[row] = 0;
    }
  }

  __shared__ int warp_cnt[kCopyThreads / 32];
  int running = ws.chunk_off[static_cast<int64_t>(bh) * NC + c];
  const int lo = c * kChunk, hi = min(lo + kChunk, n);
  for (int r0 = lo; r0 < hi; r0 += kCopyThreads) {
    const int t = r0 + threadIdx.x;
    int32_t e = 0;
    bool keep = false;
    if (t < hi) {
      e = src.expire_of(bh, t);
      keep = now < e;
    }
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) warp_cnt[warp] = __popc(bal);
    __syncthreads();
    int woff = 0, rtot = 0;
#pragma unroll
    for (int w = 0; w < kCopyThreads / 32; ++w) {
      const int x = warp_cnt[w];
      woff += (w < warp) ? x : 0;
      rtot += x;
    }
    __syncthreads();
    const int slot0 = running + woff;  // slot of this warp's first kept entry
    if (keep) {
      const int j = slot0 + __popc(bal & ((1u << lane) - 1u));
      const int64_t row = static_cast<int64_t>(base + (j >> 4)) * kPage + (j & 15);
      expire_pool[row] = e;
      remap[bh * cap + j] = src.position_of(bh, t);
    }
    // move the K and V rows: EPP entries per pass, one 16-byte vector per
    // lane; up to kBatch passes are loaded before any is stored
    constexpr int kBatch = 8;
    const int sub = lane / (2 * VPR);
    const int vec = lane % (2 * VPR);
    const bool is_v = vec >= VPR;
    const int vi = is_v ? vec - VPR : vec;
    unsigned m = bal;
    int done = 0;
    while (m) {
      uint4 val[kBatch];
      int js[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        unsigned mm = m;
        for (int q = 0; q < sub; ++q) mm &= mm - 1u;  // the sub-th remaining entry
        js[u] = -1;
        if (mm) {
          const int ts = r0 + warp * 32 + (__ffs(mm) - 1);
          const uint16_t* srow = is_v ? src.v_row(bh, ts) : src.k_row(bh, ts);
          val[u] = __ldg(reinterpret_cast<const uint4*>(srow) + vi);
          js[u] = slot0 + done + sub;
        }
#pragma unroll
        for (int q = 0; q < EPP; ++q) m &= (m ? m - 1u : 0u);
        done += EPP;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (js[u] >= 0) {
          const int64_t row = static_cast<int64_t>(base + (js[u] >> 4)) * kPage + (js[u] & 15);
          reinterpret_cast<uint4*>((is_v ? v_pool : k_pool) + row * D)[vi] = val[u];
        }
      }
    }
    running += rtot;
  }
}

// ------------------------------------------------------------------ append
template <int D>
__global__ void __launch_bounds__(256) append_kernel(int mode, int BH, int pos, const uint16_t* __restrict__ k_new,
                                                     const uint16_t* __restrict__ v_new,
                                                     const float* __restrict__ score, const float* __restrict__ tau,
                                                     const int32_t* __restrict__ flag, int window, int delay,
                                                     uint16_t* __restrict__ k_pool, uint16_t* __restrict__ v_pool,
                                                     int32_t* __restrict__ expire_pool, int n_pages_cap,
                                                     const int32_t* __restrict__ page_table, int max_pages,
                                                     int32_t* __restrict__ remap, int32_t* __restrict__ count,
                                                     int32_t* __restrict__ status) {
  constexpr int VPR = D / 8;
  const int bh = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (bh >= BH) return;
  const int j = count[bh];
  if (j < 0) {
    if (lane == 0) record_error(status, KVP_ERR_BOUNDS);
    return;
  }
  const int p = j >> 4;
  const int page = (p < max_pages) ? page_table[static_cast<int64_t>(bh) * max_pages + p] : -1;
  if (page < 0) {
    if (lane == 0) record_error(status, KVP_ERR_CAPACITY);
    return;
  }
  if (page >= n_pages_cap) {
    if (lane == 0) record_error(status, KVP_ERR_BOUNDS);
    return;
  }
  const int64_t row = static_cast<int64_t>(page) * kPage + (j & 15);
  if (lane < 2 * VPR) {
    const bool is_v = lane >= VPR;
    const int vi = is_v ? lane - VPR : lane;
    const uint4 val = reinterpret_cast<const uint4*>((is_v ? v_new : k_new) + static_cast<int64_t>(bh) * D)[vi];
    reinterpret_cast<uint4*>((is_v ? v_pool : k_pool) + row * D)[vi] = val;
  }
  if (lane == 0) {
    const int32_t e = (mode == KVP_MASK_KVZAP) ? expire_kvzap(score[bh], tau[bh], pos, window)
                                               : expire_dms(flag[bh], pos, delay, window);
    expire_pool[row] = e;
    remap[static_cast<int64_t>(bh) * max_pages * kPage + j] = pos;
    count[bh] = j + 1;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <class Src>
kvp_status run_compact(const Src& src, int BH, int NC, int head_dim, int now, int reserve, void* k_pool,
                       void* v_pool, int32_t* expire_pool, int n_pages_cap, int32_t* page_table, int max_pages,
                       int32_t* remap, int32_t* count, void* workspace, int32_t* status, cudaStream_t st) {
  CompactWs ws = carve(workspace, BH, NC);
  const dim3 grid(NC, BH);
  count_kernel<Src><<<grid, 256, 0, st>>>(src, now, NC, ws.chunk_cnt);
  scan_kernel<<<1, 1024, 0, st>>>(BH, NC, reserve, max_pages, n_pages_cap, ws, count, status);
  auto* kp = static_cast<uint16_t*>(k_pool);
  auto* vp = static_cast<uint16_t*>(v_pool);
  if (head_dim == 128)
    scatter_kernel<128, Src><<<grid, kCopyThreads, 0, st>>>(src, now, NC, reserve, max_pages, ws, count, kp, vp,
                                                            expire_pool, page_table, remap);
  else
    scatter_kernel<64, Src><<<grid, kCopyThreads, 0, st>>>(src, now, NC, reserve, max_pages, ws, count, kp, vp,
                                                           expire_pool, page_table, remap);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" kvp_status kvp_mask(int mode, int batch, int n_kv_heads, int n_pos, int pos0, const float* scores,
                               const float* tau, const int32_t* flag_step, int window, int delay, int now,
                               int32_t* expire, uint32_t* keep_bits, int32_t* count, void* stream) {
  if (batch < 0 || n_kv_heads <= 0 || n_pos < 0 || pos0 < 0 || window < 0 || delay < 0) return KVP_ERR_INVALID;
  if (mode == KVP_MASK_KVZAP) {
    if (scores == nullptr || tau == nullptr || flag_step != nullptr) return KVP_ERR_INVALID;
  } else if (mode == KVP_MASK_DMS) {
    if (flag_step == nullptr || scores != nullptr || tau != nullptr) return KVP_ERR_INVALID;
  } else {
    return KVP_ERR_INVALID;
  }
  if (expire == nullptr) return KVP_ERR_INVALID;
  if (static_cast<int64_t>(pos0) + n_pos + window + delay >= kNever) return KVP_ERR_INVALID;
  if (static_cast<int64_t>(batch) * n_kv_heads > 0x7fffffff) return KVP_ERR_UNSUPPORTED;
  if (batch == 0 || n_pos == 0) {
    if (count != nullptr && batch > 0)
      return cudaMemsetAsync(count, 0, sizeof(int32_t) * batch * n_kv_heads, static_cast<cudaStream_t>(stream)) ==
                     cudaSuccess
                 ? KVP_OK
                 : KVP_ERR_CUDA;
    return KVP_OK;
  }
  const int threads = n_pos >= 1024 ? 1024 : ((n_pos + 31) / 32) * 32;
  mask_kernel<<<batch * n_kv_heads, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      mode, n_kv_heads, n_pos, pos0, scores, tau, flag_step, window, delay, now, expire, keep_bits, count);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

extern "C" size_t kvp_compact_workspace_bytes(int batch, int n_kv_heads, int n_pos) {
  if (batch <= 0 || n_kv_heads <= 0 || n_pos < 0) return 0;
  const int NC = n_pos > 0 ? (n_pos + kChunk - 1) / kChunk : 1;
  return compact_ws_bytes(batch * n_kv_heads, NC);
}

extern "C" size_t kvp_compact_paged_workspace_bytes(int batch, int n_kv_heads, int src_max_pages) {
  if (batch <= 0 || n_kv_heads <= 0 || src_max_pages < 0) return 0;
  return kvp_compact_workspace_bytes(batch, n_kv_heads, src_max_pages * kPage);
}

static kvp_status check_dst(int head_dim, int reserve, void* k_pool, void* v_pool, int32_t* expire_pool,
                            int n_pages_cap, int32_t* page_table, int max_pages, int32_t* remap, int32_t* count,
                            int32_t* status) {
  if (head_dim != 64 && head_dim != 128) return KVP_ERR_UNSUPPORTED;
  if (reserve < 0 || n_pages_cap < 0 || max_pages < 0) return KVP_ERR_INVALID;
  if (k_pool == nullptr || v_pool == nullptr || expire_pool == nullptr || page_table == nullptr ||
      remap == nullptr || count == nullptr || status == nullptr)
    return KVP_ERR_INVALID;
  if (!aligned16(k_pool) || !aligned16(v_pool)) return KVP_ERR_ALIGN;
  if (static_cast<int64_t>(max_pages) * kPage > 0x7fffffff) return KVP_ERR_UNSUPPORTED;
  return KVP_OK;
}

extern "C" kvp_status kvp_compact(int batch, int n_kv_heads, int head_dim, int n_pos, const void* k_src,
                                  const void* v_src, int64_t stride_b, int64_t stride_t, int64_t stride_h,
                                  const int32_t* expire, int now, int reserve, void* k_pool, void* v_pool,
                                  int32_t* expire_pool, int n_pages_cap, int32_t* page_table, int max_pages,
                                  int32_t* remap, int32_t* count, void* workspace, size_t workspace_bytes,
                                  int32_t* status, void* stream) {
  if (batch <= 0 || n_kv_heads <= 0 || n_pos < 0) return KVP_ERR_INVALID;
  kvp_status s = check_dst(head_dim, reserve, k_pool, v_pool, expire_pool, n_pages_cap, page_table, max_pages,
                           remap, count, status);
  if (s != KVP_OK) return s;
  if (n_pos > 0 && (k_src == nullptr || v_src == nullptr || expire == nullptr)) return KVP_ERR_INVALID;
  if (!aligned16(k_src) || !aligned16(v_src) || stride_b % 8 || stride_t % 8 || stride_h % 8) return KVP_ERR_ALIGN;
  if (stride_b < 0 || stride_t < 0 || stride_h < 0) return KVP_ERR_INVALID;
  if (workspace == nullptr || workspace_bytes < kvp_compact_workspace_bytes(batch, n_kv_heads, n_pos))
    return KVP_ERR_WORKSPACE;
  const int NC = n_pos > 0 ? (n_pos + kChunk - 1) / kChunk : 1;
  DenseSrc src{static_cast<const uint16_t*>(k_src), static_cast<const uint16_t*>(v_src), stride_b, stride_t,
               stride_h, expire, n_kv_heads, n_pos};
  return run_compact(src, batch * n_kv_heads, NC, head_dim, now, reserve, k_pool, v_pool, expire_pool, n_pages_cap,
                     page_table, max_pages, remap, count, workspace, status, static_cast<cudaStream_t>(stream));
}

extern "C" kvp_status kvp_compact_paged(int batch, int n_kv_heads, int head_dim, const void* src_k_pool,
                                        const void* src_v_pool, const int32_t* src_expire_pool,
                                        int src_n_pages_cap, const int32_t* src_page_table, int src_max_pages, const int32_t* src_remap,
                                        const int32_t* src_count, int now, int reserve, void* k_pool, void* v_pool,
                                        int32_t* expire_pool, int n_pages_cap, int32_t* page_table, int max_pages,
                                        int32_t* remap, int32_t* count, void* workspace, size_t workspace_bytes,
                                        int32_t* status, void* stream) {
  if (batch <= 0 || n_kv_heads <= 0 || src_max_pages < 0 || src_n_pages_cap < 0) return KVP_ERR_INVALID;
  if (static_cast<int64_t>(src_max_pages) * kPage > 0x7fffffff) return KVP_ERR_UNSUPPORTED;
  kvp_status s = check_dst(head_dim, reserve, k_pool, v_pool, expire_pool, n_pages_cap, page_table, max_pages,
                           remap, count, status);
  if (s != KVP_OK) return s;
  if (src_k_pool == nullptr || src_v_pool == nullptr || src_expire_pool == nullptr || src_page_table == nullptr ||
      src_remap == nullptr || src_count == nullptr)
    return KVP_ERR_INVALID;
  if (!aligned16(src_k_pool) || !aligned16(src_v_pool)) return KVP_ERR_ALIGN;
  if (src_k_pool == k_pool || src_v_pool == v_pool || src_count == count || src_page_table == page_table ||
      src_remap == remap || src_expire_pool == expire_pool)
    return KVP_ERR_INVALID;
  if (workspace == nullptr ||
      workspace_bytes < kvp_compact_paged_workspace_bytes(batch, n_kv_heads, src_max_pages))
    return KVP_ERR_WORKSPACE;
  const int n_slots = src_max_pages * kPage;
  const int NC = n_slots > 0 ? (n_slots + kChunk - 1) / kChunk : 1;
  PagedSrc src{static_cast<const uint16_t*>(src_k_pool),
               static_cast<const uint16_t*>(src_v_pool),
               src_expire_pool,
               src_page_table,
               src_remap,
               src_count,
               src_max_pages,
               src_n_pages_cap,
               head_dim,
               status};
  return run_compact(src, batch * n_kv_heads, NC, head_dim, now, reserve, k_pool, v_pool, expire_pool, n_pages_cap,
                     page_table, max_pages, remap, count, workspace, status, static_cast<cudaStream_t>(stream));
}

extern "C" kvp_status kvp_append(int mode, int batch, int n_kv_heads, int head_dim, int pos, const void* k_new,
                                 const void* v_new, const float* score, const float* tau, const int32_t* flag_step,
                                 int window, int delay, void* k_pool, void* v_pool, int32_t* expire_pool,
                                 int n_pages_cap, const int32_t* page_table, int max_pages, int32_t* remap,
                                 int32_t* count, int32_t* status, void* stream) {
  if (batch <= 0 || n_kv_heads <= 0 || pos < 0 || window < 0 || delay < 0 || max_pages < 0 || n_pages_cap < 0)
    return KVP_ERR_INVALID;
  if (head_dim != 64 && head_dim != 128) return KVP_ERR_UNSUPPORTED;
  if (mode == KVP_MASK_KVZAP) {
    if (score == nullptr || tau == nullptr || flag_step != nullptr) return KVP_ERR_INVALID;
  } else if (mode == KVP_MASK_DMS) {
    if (flag_step == nullptr || score != nullptr || tau != nullptr) return KVP_ERR_INVALID;
  } else {
    return KVP_ERR_INVALID;
  }
  if (k_new == nullptr || v_new == nullptr || k_pool == nullptr || v_pool == nullptr || expire_pool == nullptr ||
      page_table == nullptr || remap == nullptr || count == nullptr || status == nullptr)
    return KVP_ERR_INVALID;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool)) return KVP_ERR_ALIGN;
  if (static_cast<int64_t>(pos) + window + delay >= kNever) return KVP_ERR_INVALID;
  const int BH = batch * n_kv_heads;
  const int blocks = (BH + 7) / 8;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto* kp = static_cast<uint16_t*>(k_pool);
  auto* vp = static_cast<uint16_t*>(v_pool);
  auto* kn = static_cast<const uint16_t*>(k_new);
  auto* vn = static_cast<const uint16_t*>(v_new);
  if (head_dim == 128)
    append_kernel<128><<<blocks, 256, 0, st>>>(mode, BH, pos, kn, vn, score, tau, flag_step, window, delay, kp, vp,
                                               expire_pool, n_pages_cap, page_table, max_pages, remap, count,
                                               status);
  else
    append_kernel<64><<<blocks, 256, 0, st>>>(mode, BH, pos, kn, vn, score, tau, flag_step, window, delay, kp, vp,
                                              expire_pool, n_pages_cap, page_table, max_pages, remap, count,
                                              status);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}
