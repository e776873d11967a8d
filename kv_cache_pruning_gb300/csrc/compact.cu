// kvp_mask, kvp_compact, kvp_compact_masked, kvp_compact_quant, kvp_compact_paged, kvp_append,
// kvp_append_quant, and the MLA latent cache's kvp_compact_latent, kvp_compact_latent_paged,
// kvp_append_latent.
//
// Rules (KVzap summary "실제 적용"; DMS article "지연 삭제 (Delayed Eviction)"):
// an entry gets the first step at which it is gone,
//   KVZAP  expire = score >= tau ? never : pos + window
//   DMS    expire = flag < 0 ? never : max(flag + delay, pos + window)
// and is present at step `now` iff now < expire.
//
// Compaction (DeInfer summary, "나. 페이지드 KV 캐시 및 CUDA Graph 통합"):
// a preparation pass counts the present entries of each 128-entry segment of
// every (b, h) (one warp per segment) and adds each CTA's total to the
// (b, h)'s count with one atomic; a copy pass (again one warp per segment)
// derives its segment's first slot from the counts of the segments before it
// and, up to 1,024 (b, h), its page base and the budget check from all
// counts (above that a one-CTA pass computes the bases), lists the segment's
// present entries with ballots (the remapping index list) and moves their K
// and V rows through a shared-memory stage with 16-byte asynchronous copies.
// Where an entry's presence comes from is a "source" view: a precomputed
// expire array, the mask rule applied to scores or flag steps on the fly, a
// paged cache, or the fp8 tier's selection (whose copy pass quantizes).
#include <mutex>
#include <type_traits>


#include "kvp_common.cuh"

namespace kvp {
namespace {

constexpr int kSeg = 128;           // entries per warp segment
constexpr int kQuantMetaWords = 3 * KVP_PAGE_TOKENS;  // fp8 tier page record: start, K scale, V scale
constexpr int kWarpsPerCta = 4;     // segments per CTA in the count and copy passes
constexpr int kLatentRow = KVP_MLA_LATENT_DIM + KVP_MLA_ROPE_DIM;  // MLA latent row: compressed KV, rotary key

KVP_DEV int32_t expire_kvzap(float s, float tau, int pos, int window) {
  return (s >= tau) ? kNever : pos + window;  // NaN compares false: treated as low
}
KVP_DEV int32_t expire_dms(int flag, int pos, int delay, int window) {
  return flag < 0 ? kNever : max(flag + delay, pos + window);
}

// ------------------------------------------------------------------ mask
// One CTA per (b, h). Each thread takes kMaskUnroll positions per round, all
// of whose score (or flag) loads are issued before any is used, so a round
// costs one memory latency rather than kMaskUnroll of them.
constexpr int kMaskUnroll = 8;

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
  const int step = blockDim.x;
  int kept = 0;
  for (int t0 = 0; t0 < n_pos; t0 += step * kMaskUnroll) {
    float sc[kMaskUnroll];
    int32_t fl[kMaskUnroll];
#pragma unroll
    for (int u = 0; u < kMaskUnroll; ++u) {
      const int t = t0 + u * step + threadIdx.x;
      sc[u] = 0.f;
      fl[u] = 0;
      if (t < n_pos) {
        if (mode == KVP_MASK_KVZAP) {
          sc[u] = scores[(static_cast<int64_t>(b) * n_pos + t) * H + h];
        } else {
          fl[u] = flag[static_cast<int64_t>(bh) * n_pos + t];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kMaskUnroll; ++u) {
      const int tb = t0 + u * step;  // first position of this sub-round
      if (tb >= n_pos) break;        // uniform across the CTA
      const int t = tb + threadIdx.x;
      bool keep = false;
      if (t < n_pos) {
        const int32_t e = (mode == KVP_MASK_KVZAP) ? expire_kvzap(sc[u], th, pos0 + t, window)
                                                   : expire_dms(fl[u], pos0 + t, delay, window);
        expire[static_cast<int64_t>(bh) * n_pos + t] = e;
        keep = now < e;
      }
      const unsigned bal = __ballot_sync(0xffffffffu, keep);
      const int word = (tb >> 5) + warp;
      if (lane == 0 && word < n_words) {
        if (keep_bits) keep_bits[static_cast<int64_t>(bh) * n_words + word] = bal;
        kept += __popc(bal);
      }
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
// A source yields, for entry t of one (b, h): its expire value, the index of
// its K/V row (row address = base + row * stride elements) and its position.
//
// Dense source: entry t is row (b, t, h) of K/V, present iff now < expire[b, h, t].
struct DenseSrc {
  const uint16_t* k;
  const uint16_t* v;
  int64_t sb, st, sh;
  const int32_t* expire;  // [B, H, n]
  int H;
  int n;                  // entries per (b, h)
  struct View {
    const uint16_t* kb;
    const uint16_t* vb;
    int64_t stride;
    const int32_t* exp;
    int n;
    KVP_DEV int length() const { return n; }
    KVP_DEV int32_t expire_row(int t, int64_t& row) const {
      row = t;
      return exp[t];
    }
    KVP_DEV int position_of(int t) const { return t; }
    KVP_DEV bool keep(int32_t e, int now) const { return now < e; }
  };
  KVP_DEV View view(int bh) const {
    const int b = bh / H, h = bh - b * H;
    const int64_t off = b * sb + h * sh;
    return View{k + off, v + off, st, expire + static_cast<int64_t>(bh) * n, n};
  }
};

// Masked dense source: the same rows as DenseSrc, but each entry's expire is
// derived where it is needed from its score and the (b, h)'s threshold (KVzap)
// or its flag step (DMS), with the mask kernel's rule and position t, so that
// no [B, H, n] expire array is written or read.
struct MaskedSrc {
  const uint16_t* k;
  const uint16_t* v;
  int64_t sb, st, sh;
  int mode;
  const float* scores;     // KVzap: [B, n, H]
  const float* tau;        // KVzap: [B, H]
  const int32_t* flag;     // DMS: [B, H, n]
  int window, delay;
  int H;
  int n;
  struct View {
    const uint16_t* kb;
    const uint16_t* vb;
    int64_t stride;
    int mode;
    const float* sc;       // this (b, h)'s scores, entry t at sc[t * H]
    const int32_t* fl;     // this (b, h)'s flag steps, entry t at fl[t]
    float th;
    int H, window, delay, n;
    KVP_DEV int length() const { return n; }
    KVP_DEV int32_t expire_row(int t, int64_t& row) const {
      row = t;
      return mode == KVP_MASK_KVZAP ? expire_kvzap(sc[static_cast<int64_t>(t) * H], th, t, window)
                                    : expire_dms(fl[t], t, delay, window);
    }
    KVP_DEV int position_of(int t) const { return t; }
    KVP_DEV bool keep(int32_t e, int now) const { return now < e; }
  };
  KVP_DEV View view(int bh) const {
    const int b = bh / H, h = bh - b * H;
    const int64_t off = b * sb + h * sh;
    const bool kvz = mode == KVP_MASK_KVZAP;
    return View{k + off,
                v + off,
                st,
                mode,
                kvz ? scores + static_cast<int64_t>(b) * n * H + h : nullptr,
                kvz ? nullptr : flag + static_cast<int64_t>(bh) * n,
                kvz ? tau[bh] : 0.f,
                H,
                window,
                delay,
                n};
  }
};

// Selection for the fp8 tier (quantize instead of drop; BeaconKV article):
// KVzap: entry t of the dense source goes to the tier iff tau_q <= score <
// tau (NaN never); DMS: iff it is flagged (flag step >= 0). Its value is the
// step from which it is visible there, the step its full-precision copy is
// gone: t + window (KVzap), max(flag + delay, t + window) (DMS). `now` plays
// no part in the choice.
constexpr int32_t kNotSelected = INT32_MIN;

struct QuantSrc {
  const uint16_t* k;
  const uint16_t* v;
  int64_t sb, st, sh;
  int mode;
  const float* scores;     // KVzap: [B, n, H]
  const float* tau;        // KVzap: [B, H]
  const float* tau_q;      // KVzap: [B, H]
  const int32_t* flag;     // DMS: [B, H, n]
  int window, delay;
  int H;
  int n;
  struct View {
    const uint16_t* kb;
    const uint16_t* vb;
    int64_t stride;
    int mode;
    const float* sc;
    const int32_t* fl;
    float th, tq;
    int H, window, delay, n;
    KVP_DEV int length() const { return n; }
    KVP_DEV int32_t expire_row(int t, int64_t& row) const {
      row = t;
      if (mode == KVP_MASK_DMS) {
        const int32_t f = fl[t];
        return f >= 0 ? expire_dms(f, t, delay, window) : kNotSelected;
      }
      const float x = sc[static_cast<int64_t>(t) * H];
      return (x >= tq && x < th) ? t + window : kNotSelected;
    }
    KVP_DEV int position_of(int t) const { return t; }
    KVP_DEV bool keep(int32_t e, int) const { return e != kNotSelected; }
  };
  KVP_DEV View view(int bh) const {
    const int b = bh / H, h = bh - b * H;
    const int64_t off = b * sb + h * sh;
    const bool kvz = mode == KVP_MASK_KVZAP;
    return View{k + off,
                v + off,
                st,
                mode,
                kvz ? scores + static_cast<int64_t>(b) * n * H + h : nullptr,
                kvz ? nullptr : flag + static_cast<int64_t>(bh) * n,
                kvz ? tau[bh] : 0.f,
                kvz ? tau_q[bh] : 0.f,
                H,
                window,
                delay,
                n};
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
  struct View {
    const uint16_t* kb;
    const uint16_t* vb;
    int64_t stride;
    const int32_t* expire_pool;
    const int32_t* ptab;
    const int32_t* remap;
    int n, n_pages_cap;
    int32_t* status;
    KVP_DEV int length() const { return n; }
    KVP_DEV int32_t expire_row(int j, int64_t& row) const {
      const int pg = ptab[j >> 4];
      if (pg < 0 || pg >= n_pages_cap) {
        record_error(status, KVP_ERR_BOUNDS);
        row = -1;
        return 0;
      }
      row = static_cast<int64_t>(pg) * kPage + (j & 15);
      return expire_pool[row];
    }
    KVP_DEV int position_of(int j) const { return remap[j]; }
    KVP_DEV bool keep(int32_t e, int now) const { return now < e; }
  };
  KVP_DEV View view(int bh) const {
    const int n = min(max(count[bh], 0), max_pages * kPage);
    return View{k, v, d, expire_pool, page_table + static_cast<int64_t>(bh) * max_pages,
                remap + static_cast<int64_t>(bh) * max_pages * kPage, n, n_pages_cap, status};
  }
};

// Workspace layout (int32): segment counts [BH*NS], a second [BH*NS] block
// kept for the layout's stability, page base [BH], flag [1] (1 = budget ok);
// base and flag are used only above kFusedBH pairs.
struct CompactWs {
  int32_t* seg_cnt;
  int32_t* seg_off;
  int32_t* base;
  int32_t* ok;
};
size_t compact_ws_bytes(int64_t BH, int NS) { return (static_cast<size_t>(2) * BH * NS + BH + 1) * sizeof(int32_t); }
// (b, h) pairs a compaction takes: the count pass puts them on the grid's y
// dimension.
constexpr int64_t kMaxCompactBH = 65535;
CompactWs carve(void* ws, int BH, int NS) {
  int32_t* p = static_cast<int32_t*>(ws);
  const size_t n = static_cast<size_t>(BH) * NS;
  return CompactWs{p, p + n, p + 2 * n, p + 2 * n + BH};
}
int n_segments(int n) { return n > 0 ? (n + kSeg - 1) / kSeg : 1; }

// Preparation: present entries per segment (one warp each); the CTA's
// segments (all of one (b, h)) are summed and added to the (b, h)'s count
// with one atomic.
template <class Src>
__global__ void __launch_bounds__(kWarpsPerCta * 32) count_kernel(Src src, int now, int NS,
                                                                   int32_t* __restrict__ seg_cnt,
                                                                   int32_t* __restrict__ count) {
  __shared__ int cta_kept[kWarpsPerCta];
  pdl_launch_dependents();  // the copy pass may be scheduled now; it waits for this grid's end
  const int bh = blockIdx.y;
  const int warp = threadIdx.x >> 5;
  const int sg = blockIdx.x * kWarpsPerCta + warp;
  const int lane = threadIdx.x & 31;
  int kept = 0;
  if (sg < NS) {
    const auto sv = src.view(bh);
    const int lo = sg * kSeg, hi = min(lo + kSeg, sv.length());
#pragma unroll
    for (int u = 0; u < kSeg / 32; ++u) {  // independent loads, all in flight together
      const int t = lo + u * 32 + lane;
      if (t < hi) {
        int64_t row;
        const int32_t e = sv.expire_row(t, row);
        kept += (row >= 0 && sv.keep(e, now));
      }
    }
    kept = __reduce_add_sync(0xffffffffu, kept);
    if (lane == 0) seg_cnt[static_cast<int64_t>(bh) * NS + sg] = kept;
  }
  if (lane == 0) cta_kept[warp] = kept;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
#pragma unroll
    for (int w = 0; w < kWarpsPerCta; ++w) t += cta_kept[w];
    if (t) atomicAdd(&count[bh], t);  // count was zeroed before this kernel
  }
}

// Page bases for B*H above kFusedBH (one CTA): bases in (b-major, h-minor)
// order and the budget checks. Up to kFusedBH pairs every copy-pass CTA
// derives its own base and the checks from the counts instead.
constexpr int kFusedBH = 1024;

__global__ void __launch_bounds__(1024) base_kernel(int BH, int reserve, int max_pages, int n_pages_cap,
                                                    CompactWs ws, const int32_t* __restrict__ count,
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
      pages = (count[bh] + reserve + kPage - 1) / kPage;
      if (pages > max_pages) atomicExch(&bad_s, 1);
    }
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

// 16-byte asynchronous global -> shared copy (no register staging).
KVP_DEV void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
KVP_DEV void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
// Closes the group of this thread's copies issued so far; waits until at most
// one group (the newest) is still in flight.
KVP_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
KVP_DEV void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
KVP_DEV void cp_async_wait_two() { asm volatile("cp.async.wait_group 2;" ::: "memory"); }

// Copy pass: one warp per 128-entry segment of one (b, h); grid
// (B*H, ceil(NS / 4)). The warp lists the segment's present entries (source
// row indices, in order) in shared memory and writes their expire and remap
// entries, then moves their K and V rows through a shared-memory stage of
// kStage entries: every row of a batch is requested with 16-byte async
// copies before the first one is stored, so a warp keeps up to
// kStage * 2 * D * 2 bytes in flight without spending registers on them.
// The segment's expire values, the counts of the segments before it and
// (up to kFusedBH pairs) the counts of all pairs are requested together
// before any of them is used.
// Entries per warp batch: 20 (45 KB of stage per CTA, 5 CTAs and 20 warps per
// SM) measured best on a GB300 at 16 x 8192 tokens, 26 % kept: 51.7 us against
// 53.6 / 54.7 / 54.9 us for 16 / 24 / 32.
constexpr int kStage = 20;

// An entry is NPOOL rows of D bf16 values: a K and a V row (NPOOL = 2), or
// one latent row of an MLA cache (NPOOL = 1, D = 576: 72 pieces of 16 bytes,
// moved kStageWide at a time through three stage buffers, so that two batches
// are loading while a third is stored). The quantizing copy (kQ) splits the
// same bytes into two buffers of kStage / 2 entries, so that its arithmetic
// on one batch overlaps the next batch's loads.
constexpr int kStageWide = 8;
template <int D, int NPOOL>
constexpr int entry_pieces() {
  return NPOOL * D * 2 / 16;
}
template <int D, int NPOOL, bool kQ>
constexpr int stage_entries() {
  return entry_pieces<D, NPOOL>() > 32 ? kStageWide : (kQ ? kStage / 2 : kStage);
}
template <int D, int NPOOL, bool kQ>
constexpr int stage_buffers() {
  return entry_pieces<D, NPOOL>() > 32 ? 3 : (kQ ? 2 : 1);
}
template <int D, int NPOOL, bool kQ>
constexpr int scatter_smem_bytes() {
  return kWarpsPerCta *
         (stage_buffers<D, NPOOL, kQ>() * stage_entries<D, NPOOL, kQ>() * entry_pieces<D, NPOOL>() * 16 + kSeg * 8);
}

template <int D, int NPOOL, class Src, bool kFused>
__global__ void __launch_bounds__(kWarpsPerCta * 32) scatter_kernel(Src src, int now, int NS, int reserve,
                                                                     int max_pages, int n_pages_cap, int BH,
                                                                     CompactWs ws,
                                                                     const int32_t* __restrict__ count,
                                                                     int32_t* __restrict__ status,
                                                                     uint16_t* __restrict__ k_pool,
                                                                     uint16_t* __restrict__ v_pool,
                                                                     int32_t* __restrict__ expire_pool,
                                                                     int32_t* __restrict__ page_table,
                                                                     int32_t* __restrict__ remap) {
  constexpr int E16 = entry_pieces<D, NPOOL>();  // 16-byte pieces per entry (K row then V row, or the latent row)
  constexpr bool kNarrow = E16 <= 32 && 32 % E16 == 0;  // whole entries per warp instruction
  constexpr int EPI = kNarrow ? 32 / E16 : 1;    // entries per warp instruction (1 for D = 128, 2 for D = 64)
  // fp8 tier: k_pool / v_pool hold E4M3 codes (D bytes a row) and expire_pool
  // is the per-page record [start x 16, K scale x 16, V scale x 16]
  constexpr bool kQuant = std::is_same<Src, QuantSrc>::value;
  constexpr int kSt = stage_entries<D, NPOOL, kQuant>();
  static_assert(NPOOL == 2 || (!kQuant && !kNarrow), "one-pool entries are the wide latent rows");
  constexpr int kMetaStride = kQuant ? kQuantMetaWords : kPage;
  extern __shared__ __align__(16) uint8_t sm_raw[];
  pdl_launch_dependents();
  pdl_wait();  // segment counts and (b, h) counts come from the passes before this one
  const int bh = blockIdx.x;  // pairs vary fastest: CTAs resident together read the same positions of all heads
  const int warp = threadIdx.x >> 5;
  const int sg = blockIdx.y * kWarpsPerCta + warp;
  const int lane = threadIdx.x & 31;
  constexpr int kBufs = stage_buffers<D, NPOOL, kQuant>();
  uint4* stage = reinterpret_cast<uint4*>(sm_raw) + warp * kBufs * kSt * E16;
  int64_t* lst = reinterpret_cast<int64_t*>(sm_raw + kWarpsPerCta * kBufs * kSt * E16 * 16) + warp * kSeg;
  const bool live = sg < NS;

  // ---- loads that do not depend on one another, all issued first
  const auto sv = src.view(bh);
  const int n = sv.length();
  const int lo = sg * kSeg, hi = min(lo + kSeg, n);
  int64_t rows[kSeg / 32];
  int32_t exps[kSeg / 32];
#pragma unroll
  for (int u = 0; u < kSeg / 32; ++u) {
    const int t = lo + u * 32 + lane;
    rows[u] = -1;
    exps[u] = 0;
    if (live && t < hi) exps[u] = sv.expire_row(t, rows[u]);
  }
  int slot0 = 0;  // first slot of this segment: the present entries of the segments before it
  if (live)
    for (int c0 = 0; c0 < sg; c0 += 32)
      slot0 += c0 + lane < sg ? ws.seg_cnt[static_cast<int64_t>(bh) * NS + c0 + lane] : 0;
  int base;
  if constexpr (kFused) {
    // this (b, h)'s first page and the budget, from the counts of all pairs
    __shared__ int64_t red_s[3][kWarpsPerCta];
    int64_t before = 0, total = 0, bad = 0;
    for (int i = threadIdx.x; i < BH; i += kWarpsPerCta * 32) {
      const int pg = (count[i] + reserve + kPage - 1) / kPage;
      before += i < bh ? pg : 0;
      total += pg;
      bad |= pg > max_pages;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      before += __shfl_xor_sync(0xffffffffu, before, o);
      total += __shfl_xor_sync(0xffffffffu, total, o);
      bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    }
    if (lane == 0) {
      red_s[0][warp] = before;
      red_s[1][warp] = total;
      red_s[2][warp] = bad;
    }
    __syncthreads();
    before = total = bad = 0;
#pragma unroll
    for (int w = 0; w < kWarpsPerCta; ++w) {
      before += red_s[0][w];
      total += red_s[1][w];
      bad |= red_s[2][w];
    }
    if (bad || total > n_pages_cap) {
      if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) record_error(status, KVP_ERR_CAPACITY);
      return;
    }
    base = static_cast<int>(before);
  } else {
    if (ws.ok[0] == 0) return;
    base = ws.base[bh];
  }
  // a warp past the last segment has nothing to list; with wide rows it stays for the CTA's shared copy below
  if (kNarrow && !live) return;
  slot0 = __reduce_add_sync(0xffffffffu, slot0);
  const int cnt = count[bh];
  const int pages = (cnt + reserve + kPage - 1) / kPage;
  const int64_t cap = static_cast<int64_t>(max_pages) * kPage;
  int32_t* remap_bh = remap + bh * cap;

  // ---- this segment's share of the page-table row, the remap tail and the
  // zeroing of unused rows in the (b, h)'s last pages
  {
    constexpr int VPR = D / 8;
    const int seg = (max_pages + NS - 1) / NS;
    for (int p = sg * seg + lane; p < min(max_pages, (sg + 1) * seg); p += 32)
      page_table[static_cast<int64_t>(bh) * max_pages + p] = p < pages ? base + p : -1;
    const int64_t rseg = (cap + NS - 1) / NS;
    const int64_t rlo = sg * rseg > cnt ? sg * rseg : static_cast<int64_t>(cnt);
    for (int64_t j = rlo + lane; j < min(cap, (sg + 1) * rseg); j += 32) remap_bh[j] = -1;
    const int zseg = (pages * kPage - cnt + NS - 1) / NS;
    for (int j = cnt + sg * zseg; j < min(pages * kPage, cnt + (sg + 1) * zseg); ++j) {
      const int64_t row = static_cast<int64_t>(base + (j >> 4)) * kPage + (j & 15);
      if constexpr (kQuant) {
        if (lane < D / 16) {
          reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(k_pool) + row * D)[lane] = make_uint4(0, 0, 0, 0);
          reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(v_pool) + row * D)[lane] = make_uint4(0, 0, 0, 0);
        }
        if (lane < 3) expire_pool[static_cast<int64_t>(base + (j >> 4)) * kMetaStride + lane * kPage + (j & 15)] = 0;
      } else {
        for (int x = lane; x < VPR; x += 32) {
          reinterpret_cast<uint4*>(k_pool + row * D)[x] = make_uint4(0, 0, 0, 0);
          if constexpr (NPOOL == 2) reinterpret_cast<uint4*>(v_pool + row * D)[x] = make_uint4(0, 0, 0, 0);
        }
        if (lane == 0) expire_pool[row] = 0;
      }
    }
  }

  // ---- list the present entries; write their expire and remap entries
  int nk = 0;
#pragma unroll
  for (int u = 0; u < kSeg / 32; ++u) {
    const int t = lo + u * 32 + lane;
    const int64_t row = rows[u];
    const int32_t e = exps[u];
    const bool keep = (t < hi) && (row >= 0) && sv.keep(e, now);
    const unsigned bal = __ballot_sync(0xffffffffu, keep);
    if (keep) {
      const int i = nk + __popc(bal & ((1u << lane) - 1u));
      const int j = slot0 + i;
      lst[i] = row;
      expire_pool[static_cast<int64_t>(base + (j >> 4)) * kMetaStride + (j & 15)] = e;
      remap_bh[j] = sv.position_of(t);
    }
    nk += __popc(bal);
  }
  __syncwarp();

  // ---- move the rows through the stage
  if constexpr (!kNarrow) {
    // wide rows: the CTA's kept rows (its warps' lists one after another, all
    // of the same (b, h)) are shared out evenly over its warps, so that a
    // segment kept whole (the recent window) does not fall to one warp alone;
    // each warp's share goes through its three stage buffers, batches b + 1
    // and b + 2 requested before batch b is stored
    static_assert(kBufs == 3, "wide rows use three stage buffers");
    __shared__ int s_nk[kWarpsPerCta], s_slot0[kWarpsPerCta];
    if (lane == 0) {
      s_nk[warp] = nk;
      s_slot0[warp] = slot0;
    }
    __syncthreads();
    int pre[kWarpsPerCta + 1];
    pre[0] = 0;
#pragma unroll
    for (int w = 0; w < kWarpsPerCta; ++w) pre[w + 1] = pre[w] + s_nk[w];
    const int tot = pre[kWarpsPerCta];
    const int c_lo = warp * tot / kWarpsPerCta, c_hi = (warp + 1) * tot / kWarpsPerCta;
    const int64_t* lst_cta = reinterpret_cast<const int64_t*>(sm_raw + kWarpsPerCta * kBufs * kSt * E16 * 16);
    // the source row of entry c of the CTA's list (its warp's list holds it at c - pre[w]); the same in every lane
    auto src_row_of = [&](int c) {
      int w = 0;
#pragma unroll
      for (int u = 1; u < kWarpsPerCta; ++u) w += c >= pre[u] ? 1 : 0;
      return lst_cta[w * kSeg + (c - pre[w])];
    };
    // the CTA's entries take consecutive slots from its first warp's on, so a batch lands in consecutive rows
    const int64_t row_cta = static_cast<int64_t>(base) * kPage + s_slot0[0];
    auto load = [&](int c0, uint4* buf) {
      const int nb = min(kSt, c_hi - c0);
      for (int i = 0; i < nb; ++i) {
        const uint4* src = reinterpret_cast<const uint4*>(sv.kb + src_row_of(c0 + i) * sv.stride);
        for (int pc = lane; pc < E16; pc += 32) cp_async16(buf + i * E16 + pc, src + pc);
      }
      cp_async_commit();
    };
    if (c_lo < c_hi) load(c_lo, stage);
    if (c_lo + kSt < c_hi) load(c_lo + kSt, stage + kSt * E16);
    for (int b = 0, c0 = c_lo; c0 < c_hi; ++b, c0 += kSt) {
      uint4* cur = stage + (b % 3) * kSt * E16;
      // batch b + 2 goes into the buffer batch b - 1 was stored from; then this lane's copies of batch b have landed
      if (c0 + 2 * kSt < c_hi) {
        load(c0 + 2 * kSt, stage + ((b + 2) % 3) * kSt * E16);
        cp_async_wait_two();
      } else if (c0 + kSt < c_hi) {
        cp_async_wait_one();
      } else {
        cp_async_wait_all();
      }
      __syncwarp();  // and every lane's
      const int nb = min(kSt, c_hi - c0);
      uint4* dst = reinterpret_cast<uint4*>(k_pool + (row_cta + c0) * D);
      for (int x = lane; x < nb * E16; x += 32) dst[x] = cur[x];
      __syncwarp();  // every lane is done with this buffer before it is refilled
    }
    return;
  }
  const int piece = lane % E16;          // 16-byte piece of an entry this lane moves
  const int sub = lane / E16;            // entry of a warp instruction this lane serves
  const bool is_v = piece >= E16 / 2;
  const int vi = is_v ? piece - E16 / 2 : piece;
  const uint16_t* sbase = is_v ? sv.vb : sv.kb;
  uint16_t* dbase = is_v ? v_pool : k_pool;
  // the entries of batch i0 .. into buf, as one group of async copies
  auto load_batch = [&](int i0, uint4* buf) {
    const int nb = min(kSt, nk - i0);
    for (int i = sub; i < nb; i += EPI)
      cp_async16(buf + i * E16 + piece, reinterpret_cast<const uint4*>(sbase + lst[i0 + i] * sv.stride) + vi);
    cp_async_commit();
  };
  if (kBufs == 2 && nk > 0) load_batch(0, stage);
  for (int i0 = 0, bt = 0; i0 < nk; i0 += kSt, ++bt) {
    const int nb = min(kSt, nk - i0);
    uint4* cur = stage + (bt & (kBufs - 1)) * kSt * E16;
    if constexpr (kBufs == 2) {  // the next batch is requested into the other buffer before this one is used
      if (i0 + kSt < nk) {
        load_batch(i0 + kSt, stage + ((bt + 1) & 1) * kSt * E16);
        cp_async_wait_one();
      } else {
        cp_async_wait_all();
      }
    } else {
      load_batch(i0, cur);
      cp_async_wait_all();
    }
    __syncwarp();
    if constexpr (kQuant) {
      // Three steps per batch. (1) Each row's amax, reduced over its E16 / 2
      // lanes and gathered so that lane i holds entry i's K and V maxima.
      // (2) Lane i takes entry i's scales amax / 448 and inverses 448 / amax
      // (IEEE divisions) and stores the scales: the divisions run once per
      // batch rather than once per warp instruction. (3) Every element times
      // its row's inverse, rounded to E4M3 (saturating), 8 codes per lane; a
      // row whose amax is 0 stores zero codes.
      static_assert(kSt <= 32, "one entry per lane in the scale step");
      constexpr int kRowLanes = E16 / 2;
      uint8_t* qbase = reinterpret_cast<uint8_t*>(dbase);
      float amk = 0.f, amv = 0.f;  // lane i: entry i's K and V row maxima
#pragma unroll 4
      for (int ib = 0; ib < nb; ib += EPI) {
        const int i = ib + sub;
        const uint4 w = i < nb ? cur[i * E16 + piece] : make_uint4(0, 0, 0, 0);
        const float f[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                            bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
#pragma unroll
        for (int o = 1; o < kRowLanes; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
#pragma unroll
        for (int e = 0; e < EPI; ++e) {
          const float ak = __shfl_sync(0xffffffffu, amax, e * E16);
          const float av = __shfl_sync(0xffffffffu, amax, e * E16 + kRowLanes);
          if (lane == ib + e) {
            amk = ak;
            amv = av;
          }
        }
      }
      float ik = -1.f, iv = -1.f;  // the inverses; -1: amax 0, zero codes
      if (lane < nb) {
        const int j = slot0 + i0 + lane;
        float* meta = reinterpret_cast<float*>(expire_pool) + static_cast<int64_t>(base + (j >> 4)) * kMetaStride +
                      (j & 15);
        meta[kPage] = __fdiv_rn(amk, 448.f);
        meta[2 * kPage] = __fdiv_rn(amv, 448.f);
        if (amk > 0.f) ik = __fdiv_rn(448.f, amk);
        if (amv > 0.f) iv = __fdiv_rn(448.f, amv);
      }
#pragma unroll 4
      for (int ib = 0; ib < nb; ib += EPI) {
        const int i = ib + sub;
        const float ink = __shfl_sync(0xffffffffu, ik, i & 31);
        const float inv_v = __shfl_sync(0xffffffffu, iv, i & 31);
        if (i < nb) {
          const float inv = is_v ? inv_v : ink;
          const uint4 w = cur[i * E16 + piece];
          const float f[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                              bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
          uint32_t packed[2] = {0u, 0u};
          if (inv >= 0.f) {
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const uint32_t c2 = cvt_f32x2_to_e4m3x2(__fmul_rn(f[e], inv), __fmul_rn(f[e + 1], inv));
              packed[e >> 2] |= c2 << (16 * ((e >> 1) & 1));
            }
          }
          const int j = slot0 + i0 + i;
          const int64_t row = static_cast<int64_t>(base + (j >> 4)) * kPage + (j & 15);
          reinterpret_cast<uint2*>(qbase + row * D)[vi] = make_uint2(packed[0], packed[1]);
        }
      }
    } else {
      for (int i = sub; i < nb; i += EPI) {
        const int j = slot0 + i0 + i;
        const int64_t row = static_cast<int64_t>(base + (j >> 4)) * kPage + (j & 15);
        reinterpret_cast<uint4*>(dbase + row * D)[vi] = cur[i * E16 + piece];
      }
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ append
template <int D>
__global__ void __launch_bounds__(256) append_kernel(int mode, int BH, int pos_arg, const int32_t* __restrict__ pos_dev,
                                                     const uint16_t* __restrict__ k_new,
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
  // the position from device memory (one captured step replayed for every
  // position) or the argument
  const int pos = pos_dev != nullptr ? *pos_dev : pos_arg;
  if (pos < 0 || static_cast<int64_t>(pos) + window + delay >= kNever) {
    if (lane == 0) record_error(status, KVP_ERR_INVALID);
    return;
  }
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

// Decode-time append into the fp8 tier: one warp per (b, h); the token goes
// in iff tau_q <= score < tau, its K and V rows quantized like the copy
// pass's (each lane takes D / 32 elements, the row's amax is reduced over the
// warp), start = pos + window.
template <int D>
__global__ void __launch_bounds__(256) append_quant_kernel(int mode, int BH, int pos,
                                                           const uint16_t* __restrict__ k_new,
                                                           const uint16_t* __restrict__ v_new,
                                                           const float* __restrict__ score,
                                                           const float* __restrict__ tau,
                                                           const float* __restrict__ tau_q,
                                                           const int32_t* __restrict__ flag, int window, int delay,
                                                           uint8_t* __restrict__ kq_pool, uint8_t* __restrict__ vq_pool,
                                                           int32_t* __restrict__ meta_pool, int n_pages_cap,
                                                           const int32_t* __restrict__ page_table, int max_pages,
                                                           int32_t* __restrict__ remap, int32_t* __restrict__ count,
                                                           int32_t* __restrict__ status) {
  constexpr int EPL = D / 32;  // elements a lane quantizes (4 or 2)
  const int bh = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (bh >= BH) return;
  int32_t start;
  if (mode == KVP_MASK_DMS) {
    const int32_t f = flag[bh];
    if (f < 0) return;  // not flagged: stays bf16 (the same for the whole warp)
    start = expire_dms(f, pos, delay, window);
  } else {
    const float sc = score[bh];
    if (!(sc >= tau_q[bh] && sc < tau[bh])) return;  // not in the fp8 tier (the same for the whole warp)
    start = pos + window;
  }
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
  int32_t* meta = meta_pool + static_cast<int64_t>(page) * kQuantMetaWords;
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    const uint16_t* src = (w ? v_new : k_new) + static_cast<int64_t>(bh) * D + lane * EPL;
    float f[EPL];
    if constexpr (EPL == 4) {
      const uint2 x = *reinterpret_cast<const uint2*>(src);
      f[0] = bf16_lo(x.x); f[1] = bf16_hi(x.x); f[2] = bf16_lo(x.y); f[3] = bf16_hi(x.y);
    } else {
      const uint32_t x = *reinterpret_cast<const uint32_t*>(src);
      f[0] = bf16_lo(x); f[1] = bf16_hi(x);
    }
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(f[e]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = __fdiv_rn(amax, 448.f);
    uint32_t packed = 0u;
    if (amax > 0.f) {
      const float inv = __fdiv_rn(448.f, amax);
#pragma unroll
      for (int e = 0; e < EPL; e += 2) {
        packed |= cvt_f32x2_to_e4m3x2(__fmul_rn(f[e], inv), __fmul_rn(f[e + 1], inv)) << (8 * e);
      }
    }
    uint8_t* dst = (w ? vq_pool : kq_pool) + row * D + lane * EPL;
    if constexpr (EPL == 4) *reinterpret_cast<uint32_t*>(dst) = packed;
    else *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(packed);
    if (lane == 0) reinterpret_cast<float*>(meta)[(1 + w) * kPage + (j & 15)] = scale;
  }
  if (lane == 0) {
    meta[j & 15] = start;
    remap[static_cast<int64_t>(bh) * max_pages * kPage + j] = pos;
    count[bh] = j + 1;
  }
}

// Decode-time append of MLA latent rows: one warp per batch element (one
// latent "head"), the row's 72 pieces of 16 bytes spread over the lanes; the
// expire value follows the same rules as append_kernel's.
__global__ void __launch_bounds__(256) append_latent_kernel(int mode, int B, int pos,
                                                            const uint16_t* __restrict__ lat_new,
                                                            const float* __restrict__ score,
                                                            const float* __restrict__ tau,
                                                            const int32_t* __restrict__ flag, int window, int delay,
                                                            uint16_t* __restrict__ pool,
                                                            int32_t* __restrict__ expire_pool, int n_pages_cap,
                                                            const int32_t* __restrict__ page_table, int max_pages,
                                                            int32_t* __restrict__ remap, int32_t* __restrict__ count,
                                                            int32_t* __restrict__ status) {
  constexpr int VPR = kLatentRow / 8;
  const int b = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  const int j = count[b];
  if (j < 0) {
    if (lane == 0) record_error(status, KVP_ERR_BOUNDS);
    return;
  }
  const int p = j >> 4;
  const int page = (p < max_pages) ? page_table[static_cast<int64_t>(b) * max_pages + p] : -1;
  if (page < 0) {
    if (lane == 0) record_error(status, KVP_ERR_CAPACITY);
    return;
  }
  if (page >= n_pages_cap) {
    if (lane == 0) record_error(status, KVP_ERR_BOUNDS);
    return;
  }
  const int64_t row = static_cast<int64_t>(page) * kPage + (j & 15);
  const uint4* src = reinterpret_cast<const uint4*>(lat_new + static_cast<int64_t>(b) * kLatentRow);
  uint4* dst = reinterpret_cast<uint4*>(pool + row * kLatentRow);
  for (int x = lane; x < VPR; x += 32) dst[x] = src[x];
  if (lane == 0) {
    const int32_t e = (mode == KVP_MASK_KVZAP) ? expire_kvzap(score[b], tau[b], pos, window)
                                               : expire_dms(flag[b], pos, delay, window);
    expire_pool[row] = e;
    remap[static_cast<int64_t>(b) * max_pages * kPage + j] = pos;
    count[b] = j + 1;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <class Src>
kvp_status run_compact(const Src& src, int BH, int NS, int head_dim, int now, int reserve, void* k_pool,
                       void* v_pool, int32_t* expire_pool, int n_pages_cap, int32_t* page_table, int max_pages,
                       int32_t* remap, int32_t* count, void* workspace, int32_t* status, cudaStream_t st) {
  CompactWs ws = carve(workspace, BH, NS);
  const dim3 grid((NS + kWarpsPerCta - 1) / kWarpsPerCta, BH);
  const dim3 grid_t(BH, (NS + kWarpsPerCta - 1) / kWarpsPerCta);
  if (cudaMemsetAsync(count, 0, static_cast<size_t>(BH) * sizeof(int32_t), st) != cudaSuccess) return KVP_ERR_CUDA;
  count_kernel<Src><<<grid, kWarpsPerCta * 32, 0, st>>>(src, now, NS, ws.seg_cnt, count);
  const bool fused = BH <= kFusedBH;
  if (!fused) base_kernel<<<1, 1024, 0, st>>>(BH, reserve, max_pages, n_pages_cap, ws, count, status);
  auto* kp = static_cast<uint16_t*>(k_pool);
  auto* vp = static_cast<uint16_t*>(v_pool);
  constexpr bool kQ = std::is_same<Src, QuantSrc>::value;
#define KVP_SCATTER(DIM, NP, FUSED)                                                                          \
  do {                                                                                                        \
    static const bool attr_ok = cudaFuncSetAttribute(scatter_kernel<DIM, NP, Src, FUSED>,                    \
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize,            \
                                                     scatter_smem_bytes<DIM, NP, kQ>()) == cudaSuccess;       \
    if (!attr_ok) return KVP_ERR_CUDA;                                                                        \
    if (launch_pdl(scatter_kernel<DIM, NP, Src, FUSED>, grid_t, dim3(kWarpsPerCta * 32),                     \
                   scatter_smem_bytes<DIM, NP, kQ>(), st, src, now, NS, reserve, max_pages, n_pages_cap, BH, ws, \
                   static_cast<const int32_t*>(count), status, kp, vp, expire_pool, page_table,                \
                   remap) != cudaSuccess)                                                                     \
      return KVP_ERR_CUDA;                                                                                    \
  } while (0)
  if (head_dim == kLatentRow) {  // one pool: the MLA latent rows
    if constexpr (!std::is_same<Src, QuantSrc>::value) {
      if (fused) KVP_SCATTER(kLatentRow, 1, true); else KVP_SCATTER(kLatentRow, 1, false);
    } else {
      return KVP_ERR_UNSUPPORTED;
    }
  } else if (head_dim == 128) {
    if (fused) KVP_SCATTER(128, 2, true); else KVP_SCATTER(128, 2, false);
  } else {
    if (fused) KVP_SCATTER(64, 2, true); else KVP_SCATTER(64, 2, false);
  }
#undef KVP_SCATTER
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
  return compact_ws_bytes(static_cast<int64_t>(batch) * n_kv_heads, n_segments(n_pos));
}

extern "C" size_t kvp_compact_paged_workspace_bytes(int batch, int n_kv_heads, int src_max_pages) {
  if (batch <= 0 || n_kv_heads <= 0 || src_max_pages < 0) return 0;
  if (static_cast<int64_t>(src_max_pages) * kPage > 0x7fffffff) return 0;
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
  if (static_cast<int64_t>(batch) * n_kv_heads > kMaxCompactBH) return KVP_ERR_UNSUPPORTED;
  kvp_status s = check_dst(head_dim, reserve, k_pool, v_pool, expire_pool, n_pages_cap, page_table, max_pages,
                           remap, count, status);
  if (s != KVP_OK) return s;
  if (n_pos > 0 && (k_src == nullptr || v_src == nullptr || expire == nullptr)) return KVP_ERR_INVALID;
  if (!aligned16(k_src) || !aligned16(v_src) || stride_b % 8 || stride_t % 8 || stride_h % 8) return KVP_ERR_ALIGN;
  if (stride_b < 0 || stride_t < 0 || stride_h < 0) return KVP_ERR_INVALID;
  if (workspace == nullptr || workspace_bytes < kvp_compact_workspace_bytes(batch, n_kv_heads, n_pos))
    return KVP_ERR_WORKSPACE;
  const int NS = n_segments(n_pos);
  DenseSrc src{static_cast<const uint16_t*>(k_src), static_cast<const uint16_t*>(v_src), stride_b, stride_t,
               stride_h, expire, n_kv_heads, n_pos};
  return run_compact(src, batch * n_kv_heads, NS, head_dim, now, reserve, k_pool, v_pool, expire_pool, n_pages_cap,
                     page_table, max_pages, remap, count, workspace, status, static_cast<cudaStream_t>(stream));
}

extern "C" kvp_status kvp_compact_masked(int mode, int batch, int n_kv_heads, int head_dim, int n_pos,
                                         const void* k_src, const void* v_src, int64_t stride_b, int64_t stride_t,
                                         int64_t stride_h, const float* scores, const float* tau,
                                         const int32_t* flag_step, int window, int delay, int now, int reserve,
                                         void* k_pool, void* v_pool, int32_t* expire_pool, int n_pages_cap,
                                         int32_t* page_table, int max_pages, int32_t* remap, int32_t* count,
                                         void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
  if (batch <= 0 || n_kv_heads <= 0 || n_pos < 0 || window < 0 || delay < 0) return KVP_ERR_INVALID;
  if (static_cast<int64_t>(batch) * n_kv_heads > kMaxCompactBH) return KVP_ERR_UNSUPPORTED;
  // the per-position inputs may be NULL when there are no positions; tau is read per (b, h)
  if (mode == KVP_MASK_KVZAP) {
    if (flag_step != nullptr || tau == nullptr || (n_pos > 0 && scores == nullptr)) return KVP_ERR_INVALID;
  } else if (mode == KVP_MASK_DMS) {
    if (scores != nullptr || tau != nullptr || (n_pos > 0 && flag_step == nullptr)) return KVP_ERR_INVALID;
  } else {
    return KVP_ERR_INVALID;
  }
  if (static_cast<int64_t>(n_pos) + window + delay >= kNever) return KVP_ERR_INVALID;
  kvp_status s = check_dst(head_dim, reserve, k_pool, v_pool, expire_pool, n_pages_cap, page_table, max_pages,
                           remap, count, status);
  if (s != KVP_OK) return s;
  if (n_pos > 0 && (k_src == nullptr || v_src == nullptr)) return KVP_ERR_INVALID;
  if (!aligned16(k_src) || !aligned16(v_src) || stride_b % 8 || stride_t % 8 || stride_h % 8) return KVP_ERR_ALIGN;
  if (stride_b < 0 || stride_t < 0 || stride_h < 0) return KVP_ERR_INVALID;
  if (workspace == nullptr || workspace_bytes < kvp_compact_workspace_bytes(batch, n_kv_heads, n_pos))
    return KVP_ERR_WORKSPACE;
  const int NS = n_segments(n_pos);
  MaskedSrc src{static_cast<const uint16_t*>(k_src),
                static_cast<const uint16_t*>(v_src),
                stride_b,
                stride_t,
                stride_h,
                mode,
                scores,
                tau,
                flag_step,
                window,
                delay,
                n_kv_heads,
                n_pos};
  return run_compact(src, batch * n_kv_heads, NS, head_dim, now, reserve, k_pool, v_pool, expire_pool, n_pages_cap,
                     page_table, max_pages, remap, count, workspace, status, static_cast<cudaStream_t>(stream));
}

extern "C" kvp_status kvp_compact_quant(int mode, int batch, int n_kv_heads, int head_dim, int n_pos,
                                        const void* k_src, const void* v_src, int64_t stride_b, int64_t stride_t,
                                        int64_t stride_h, const float* scores, const float* tau, const float* tau_q,
                                        const int32_t* flag_step, int window, int delay, int reserve, void* kq_pool,
                                        void* vq_pool, int32_t* meta_pool, int n_pages_cap, int32_t* page_table,
                                        int max_pages, int32_t* remap, int32_t* count, void* workspace,
                                        size_t workspace_bytes, int32_t* status, void* stream) {
  if (batch <= 0 || n_kv_heads <= 0 || n_pos < 0 || window < 0 || delay < 0) return KVP_ERR_INVALID;
  if (static_cast<int64_t>(batch) * n_kv_heads > kMaxCompactBH) return KVP_ERR_UNSUPPORTED;
  if (mode == KVP_MASK_KVZAP) {
    if (flag_step != nullptr || tau == nullptr || tau_q == nullptr || (n_pos > 0 && scores == nullptr))
      return KVP_ERR_INVALID;
  } else if (mode == KVP_MASK_DMS) {
    if (scores != nullptr || tau != nullptr || tau_q != nullptr || (n_pos > 0 && flag_step == nullptr))
      return KVP_ERR_INVALID;
  } else {
    return KVP_ERR_INVALID;
  }
  if (static_cast<int64_t>(n_pos) + window + delay >= kNever) return KVP_ERR_INVALID;
  kvp_status s = check_dst(head_dim, reserve, kq_pool, vq_pool, meta_pool, n_pages_cap, page_table, max_pages,
                           remap, count, status);
  if (s != KVP_OK) return s;
  if (n_pos > 0 && (k_src == nullptr || v_src == nullptr)) return KVP_ERR_INVALID;
  if (!aligned16(k_src) || !aligned16(v_src) || stride_b % 8 || stride_t % 8 || stride_h % 8) return KVP_ERR_ALIGN;
  if (stride_b < 0 || stride_t < 0 || stride_h < 0) return KVP_ERR_INVALID;
  if (workspace == nullptr || workspace_bytes < kvp_compact_workspace_bytes(batch, n_kv_heads, n_pos))
    return KVP_ERR_WORKSPACE;
  const int NS = n_segments(n_pos);
  QuantSrc src{static_cast<const uint16_t*>(k_src),
               static_cast<const uint16_t*>(v_src),
               stride_b,
               stride_t,
               stride_h,
               mode,
               scores,
               tau,
               tau_q,
               flag_step,
               window,
               delay,
               n_kv_heads,
               n_pos};
  return run_compact(src, batch * n_kv_heads, NS, head_dim, 0, reserve, kq_pool, vq_pool, meta_pool, n_pages_cap,
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
  if (static_cast<int64_t>(batch) * n_kv_heads > kMaxCompactBH) return KVP_ERR_UNSUPPORTED;
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
  const int NS = n_segments(src_max_pages * kPage);
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
  return run_compact(src, batch * n_kv_heads, NS, head_dim, now, reserve, k_pool, v_pool, expire_pool, n_pages_cap,
                     page_table, max_pages, remap, count, workspace, status, static_cast<cudaStream_t>(stream));
}

namespace {
kvp_status append_impl(int mode, int batch, int n_kv_heads, int head_dim, int pos, const int32_t* pos_dev,
                       const void* k_new, const void* v_new, const float* score, const float* tau,
                       const int32_t* flag_step, int window, int delay, void* k_pool, void* v_pool,
                       int32_t* expire_pool, int n_pages_cap, const int32_t* page_table, int max_pages,
                       int32_t* remap, int32_t* count, int32_t* status, void* stream) {
  if (batch <= 0 || n_kv_heads <= 0 || pos < 0 || window < 0 || delay < 0 || max_pages < 0 || n_pages_cap < 0)
    return KVP_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(pos_dev) & 3u) != 0) return KVP_ERR_ALIGN;
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
  if (static_cast<int64_t>(batch) * n_kv_heads > 0x7ffffff0) return KVP_ERR_UNSUPPORTED;
  const int BH = batch * n_kv_heads;
  const int blocks = (BH + 7) / 8;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto* kp = static_cast<uint16_t*>(k_pool);
  auto* vp = static_cast<uint16_t*>(v_pool);
  auto* kn = static_cast<const uint16_t*>(k_new);
  auto* vn = static_cast<const uint16_t*>(v_new);
  if (head_dim == 128)
    append_kernel<128><<<blocks, 256, 0, st>>>(mode, BH, pos, pos_dev, kn, vn, score, tau, flag_step, window, delay,
                                               kp, vp, expire_pool, n_pages_cap, page_table, max_pages, remap, count,
                                               status);
  else
    append_kernel<64><<<blocks, 256, 0, st>>>(mode, BH, pos, pos_dev, kn, vn, score, tau, flag_step, window, delay,
                                              kp, vp, expire_pool, n_pages_cap, page_table, max_pages, remap, count,
                                              status);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}
}  // namespace

extern "C" kvp_status kvp_append(int mode, int batch, int n_kv_heads, int head_dim, int pos, const void* k_new,
                                 const void* v_new, const float* score, const float* tau, const int32_t* flag_step,
                                 int window, int delay, void* k_pool, void* v_pool, int32_t* expire_pool,
                                 int n_pages_cap, const int32_t* page_table, int max_pages, int32_t* remap,
                                 int32_t* count, int32_t* status, void* stream) {
  return append_impl(mode, batch, n_kv_heads, head_dim, pos, nullptr, k_new, v_new, score, tau, flag_step, window,
                     delay, k_pool, v_pool, expire_pool, n_pages_cap, page_table, max_pages, remap, count, status,
                     stream);
}

extern "C" kvp_status kvp_append_devpos(int mode, int batch, int n_kv_heads, int head_dim, const int32_t* pos_dev,
                                        const void* k_new, const void* v_new, const float* score, const float* tau,
                                        const int32_t* flag_step, int window, int delay, void* k_pool, void* v_pool,
                                        int32_t* expire_pool, int n_pages_cap, const int32_t* page_table,
                                        int max_pages, int32_t* remap, int32_t* count, int32_t* status,
                                        void* stream) {
  if (pos_dev == nullptr) return KVP_ERR_INVALID;
  return append_impl(mode, batch, n_kv_heads, head_dim, 0, pos_dev, k_new, v_new, score, tau, flag_step, window,
                     delay, k_pool, v_pool, expire_pool, n_pages_cap, page_table, max_pages, remap, count, status,
                     stream);
}

extern "C" kvp_status kvp_append_quant(int mode, int batch, int n_kv_heads, int head_dim, int pos, const void* k_new,
                                       const void* v_new, const float* score, const float* tau, const float* tau_q,
                                       const int32_t* flag_step, int window, int delay, void* kq_pool, void* vq_pool,
                                       int32_t* meta_pool, int n_pages_cap, const int32_t* page_table, int max_pages,
                                       int32_t* remap, int32_t* count, int32_t* status, void* stream) {
  if (batch <= 0 || n_kv_heads <= 0 || pos < 0 || window < 0 || delay < 0 || max_pages < 0 || n_pages_cap < 0)
    return KVP_ERR_INVALID;
  if (head_dim != 64 && head_dim != 128) return KVP_ERR_UNSUPPORTED;
  if (mode == KVP_MASK_KVZAP) {
    if (score == nullptr || tau == nullptr || tau_q == nullptr || flag_step != nullptr) return KVP_ERR_INVALID;
  } else if (mode == KVP_MASK_DMS) {
    if (flag_step == nullptr || score != nullptr || tau != nullptr || tau_q != nullptr) return KVP_ERR_INVALID;
  } else {
    return KVP_ERR_INVALID;
  }
  if (k_new == nullptr || v_new == nullptr || kq_pool == nullptr || vq_pool == nullptr || meta_pool == nullptr ||
      page_table == nullptr || remap == nullptr || count == nullptr || status == nullptr)
    return KVP_ERR_INVALID;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(kq_pool) || !aligned16(vq_pool) || !aligned16(meta_pool))
    return KVP_ERR_ALIGN;
  if (static_cast<int64_t>(pos) + window + delay >= kNever) return KVP_ERR_INVALID;
  if (static_cast<int64_t>(batch) * n_kv_heads > 0x7ffffff0) return KVP_ERR_UNSUPPORTED;
  const int BH = batch * n_kv_heads;
  const int blocks = (BH + 7) / 8;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto* kn = static_cast<const uint16_t*>(k_new);
  auto* vn = static_cast<const uint16_t*>(v_new);
  auto* kq = static_cast<uint8_t*>(kq_pool);
  auto* vq = static_cast<uint8_t*>(vq_pool);
  if (head_dim == 128)
    append_quant_kernel<128><<<blocks, 256, 0, st>>>(mode, BH, pos, kn, vn, score, tau, tau_q, flag_step, window,
                                                     delay, kq, vq, meta_pool, n_pages_cap, page_table, max_pages,
                                                     remap, count, status);
  else
    append_quant_kernel<64><<<blocks, 256, 0, st>>>(mode, BH, pos, kn, vn, score, tau, tau_q, flag_step, window,
                                                    delay, kq, vq, meta_pool, n_pages_cap, page_table, max_pages,
                                                    remap, count, status);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

// ------------------------------------------------------------------ MLA latent cache
// One "kv head" whose entries are latent rows of kLatentRow bf16 values in a
// single pool; the count, base and copy passes are those of the K/V cache.

static kvp_status check_dst_latent(int row_dim, int reserve, void* pool, int32_t* expire_pool, int n_pages_cap,
                                   int32_t* page_table, int max_pages, int32_t* remap, int32_t* count,
                                   int32_t* status) {
  if (row_dim != kLatentRow) return KVP_ERR_UNSUPPORTED;
  if (reserve < 0 || n_pages_cap < 0 || max_pages < 0) return KVP_ERR_INVALID;
  if (pool == nullptr || expire_pool == nullptr || page_table == nullptr || remap == nullptr || count == nullptr ||
      status == nullptr)
    return KVP_ERR_INVALID;
  if (!aligned16(pool)) return KVP_ERR_ALIGN;
  if (static_cast<int64_t>(max_pages) * kPage > 0x7fffffff) return KVP_ERR_UNSUPPORTED;
  return KVP_OK;
}

extern "C" kvp_status kvp_compact_latent(int mode, int batch, int row_dim, int n_pos, const void* lat_src,
                                         int64_t stride_b, int64_t stride_t, const float* scores, const float* tau,
                                         const int32_t* flag_step, int window, int delay, int now, int reserve,
                                         void* pool, int32_t* expire_pool, int n_pages_cap, int32_t* page_table,
                                         int max_pages, int32_t* remap, int32_t* count, void* workspace,
                                         size_t workspace_bytes, int32_t* status, void* stream) {
  if (batch <= 0 || n_pos < 0 || window < 0 || delay < 0) return KVP_ERR_INVALID;
  if (static_cast<int64_t>(batch) > kMaxCompactBH) return KVP_ERR_UNSUPPORTED;
  if (mode == KVP_MASK_KVZAP) {
    if (flag_step != nullptr || tau == nullptr || (n_pos > 0 && scores == nullptr)) return KVP_ERR_INVALID;
  } else if (mode == KVP_MASK_DMS) {
    if (scores != nullptr || tau != nullptr || (n_pos > 0 && flag_step == nullptr)) return KVP_ERR_INVALID;
  } else {
    return KVP_ERR_INVALID;
  }
  if (static_cast<int64_t>(n_pos) + window + delay >= kNever) return KVP_ERR_INVALID;
  kvp_status s = check_dst_latent(row_dim, reserve, pool, expire_pool, n_pages_cap, page_table, max_pages, remap,
                                  count, status);
  if (s != KVP_OK) return s;
  if (n_pos > 0 && lat_src == nullptr) return KVP_ERR_INVALID;
  if (!aligned16(lat_src) || stride_b % 8 || stride_t % 8) return KVP_ERR_ALIGN;
  if (stride_b < 0 || stride_t < 0) return KVP_ERR_INVALID;
  if (workspace == nullptr || workspace_bytes < kvp_compact_workspace_bytes(batch, 1, n_pos))
    return KVP_ERR_WORKSPACE;
  const int NS = n_segments(n_pos);
  const auto* l = static_cast<const uint16_t*>(lat_src);
  MaskedSrc src{l, l, stride_b, stride_t, 0, mode, scores, tau, flag_step, window, delay, 1, n_pos};
  return run_compact(src, batch, NS, kLatentRow, now, reserve, pool, nullptr, expire_pool, n_pages_cap, page_table,
                     max_pages, remap, count, workspace, status, static_cast<cudaStream_t>(stream));
}

extern "C" kvp_status kvp_compact_latent_paged(int batch, int row_dim, const void* src_pool,
                                               const int32_t* src_expire_pool, int src_n_pages_cap,
                                               const int32_t* src_page_table, int src_max_pages,
                                               const int32_t* src_remap, const int32_t* src_count, int now,
                                               int reserve, void* pool, int32_t* expire_pool, int n_pages_cap,
                                               int32_t* page_table, int max_pages, int32_t* remap, int32_t* count,
                                               void* workspace, size_t workspace_bytes, int32_t* status,
                                               void* stream) {
  if (batch <= 0 || src_max_pages < 0 || src_n_pages_cap < 0) return KVP_ERR_INVALID;
  if (static_cast<int64_t>(batch) > kMaxCompactBH) return KVP_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(src_max_pages) * kPage > 0x7fffffff) return KVP_ERR_UNSUPPORTED;
  kvp_status s = check_dst_latent(row_dim, reserve, pool, expire_pool, n_pages_cap, page_table, max_pages, remap,
                                  count, status);
  if (s != KVP_OK) return s;
  if (src_pool == nullptr || src_expire_pool == nullptr || src_page_table == nullptr || src_remap == nullptr ||
      src_count == nullptr)
    return KVP_ERR_INVALID;
  if (!aligned16(src_pool)) return KVP_ERR_ALIGN;
  if (src_pool == pool || src_count == count || src_page_table == page_table || src_remap == remap ||
      src_expire_pool == expire_pool)
    return KVP_ERR_INVALID;
  if (workspace == nullptr || workspace_bytes < kvp_compact_paged_workspace_bytes(batch, 1, src_max_pages))
    return KVP_ERR_WORKSPACE;
  const int NS = n_segments(src_max_pages * kPage);
  const auto* sp = static_cast<const uint16_t*>(src_pool);
  PagedSrc src{sp, sp, src_expire_pool, src_page_table, src_remap, src_count, src_max_pages, src_n_pages_cap,
               kLatentRow, status};
  return run_compact(src, batch, NS, kLatentRow, now, reserve, pool, nullptr, expire_pool, n_pages_cap, page_table,
                     max_pages, remap, count, workspace, status, static_cast<cudaStream_t>(stream));
}

extern "C" kvp_status kvp_append_latent(int mode, int batch, int row_dim, int pos, const void* lat_new,
                                        const float* score, const float* tau, const int32_t* flag_step, int window,
                                        int delay, void* pool, int32_t* expire_pool, int n_pages_cap,
                                        const int32_t* page_table, int max_pages, int32_t* remap, int32_t* count,
                                        int32_t* status, void* stream) {
  if (batch <= 0 || pos < 0 || window < 0 || delay < 0 || max_pages < 0 || n_pages_cap < 0) return KVP_ERR_INVALID;
  if (row_dim != kLatentRow) return KVP_ERR_UNSUPPORTED;
  if (mode == KVP_MASK_KVZAP) {
    if (score == nullptr || tau == nullptr || flag_step != nullptr) return KVP_ERR_INVALID;
  } else if (mode == KVP_MASK_DMS) {
    if (flag_step == nullptr || score != nullptr || tau != nullptr) return KVP_ERR_INVALID;
  } else {
    return KVP_ERR_INVALID;
  }
  if (lat_new == nullptr || pool == nullptr || expire_pool == nullptr || page_table == nullptr || remap == nullptr ||
      count == nullptr || status == nullptr)
    return KVP_ERR_INVALID;
  if (!aligned16(lat_new) || !aligned16(pool)) return KVP_ERR_ALIGN;
  if (static_cast<int64_t>(pos) + window + delay >= kNever) return KVP_ERR_INVALID;
  append_latent_kernel<<<(batch + 7) / 8, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      mode, batch, pos, static_cast<const uint16_t*>(lat_new), score, tau, flag_step, window, delay,
      static_cast<uint16_t*>(pool), expire_pool, n_pages_cap, page_table, max_pages, remap, count, status);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

// ------------------------------------------------------------------ no-allocation variant
// Scratch of kvp_compact_noalloc: a fixed array in device memory, present on
// every GPU that loads this library until the process exits. Host code only
// sees a stand-in symbol for it; its device address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
static __device__ __align__(256) int32_t g_compact_scratch[KVP_COMPACT_NOALLOC_SCRATCH_BYTES / sizeof(int32_t)];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};
}  // namespace

extern "C" kvp_status kvp_compact_noalloc(int batch, int n_kv_heads, int head_dim, int n_pos, const void* k_src,
                                          const void* v_src, int64_t stride_b, int64_t stride_t, int64_t stride_h,
                                          const int32_t* expire, int now, int reserve, void* k_pool, void* v_pool,
                                          int32_t* expire_pool, int n_pages_cap, int32_t* page_table, int max_pages,
                                          int32_t* remap, int32_t* count, int32_t* status, void* stream) {
  if (batch <= 0 || n_kv_heads <= 0 || n_pos < 0) return KVP_ERR_INVALID;
  if (static_cast<int64_t>(batch) * n_kv_heads > kMaxCompactBH) return KVP_ERR_UNSUPPORTED;
  const size_t need = kvp_compact_workspace_bytes(batch, n_kv_heads, n_pos);
  if (need > KVP_COMPACT_NOALLOC_SCRATCH_BYTES) return KVP_ERR_WORKSPACE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KVP_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_compact_scratch) != cudaSuccess || addr == nullptr) return KVP_ERR_CUDA;
      g_scratch_addr[dev] = addr;
    }
    scratch = g_scratch_addr[dev];
  }
  // every word of the scratch that the compaction reads is written earlier in
  // the same call, so nothing needs clearing between calls
  return kvp_compact(batch, n_kv_heads, head_dim, n_pos, k_src, v_src, stride_b, stride_t, stride_h, expire, now,
                     reserve, k_pool, v_pool, expire_pool, n_pages_cap, page_table, max_pages, remap, count, scratch,
                     KVP_COMPACT_NOALLOC_SCRATCH_BYTES, status, stream);
}
