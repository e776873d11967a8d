// kvp_decode_attn: single-query GQA attention over the compacted pages (DMS
// article, "DMS 작동 방식" step 5: standard attention over the kept cache).
//
// Persistent, page-balanced split-KV decode. All pages of all (b, h) form one
// global list (b-major, h-minor, page order); every warp of the grid takes one
// contiguous slice of it, so every warp streams the same number of pages
// (+-1) whatever the per-head survivor counts are. A warp's lane 0 keeps
// NST pages in flight with 1-D bulk copies (K page, V page, the page's 16
// expire values) completing on per-stage mbarriers; all lanes compute.
//
// Per page (LPR = D/8 lanes cover a row, 16 bytes each; RPS = 32/LPR rows per
// step; RS = 16/RPS steps): q.k partial sums of the G query heads of the kv
// head are reduced across the row's lanes with a transposing butterfly, masked
// (slot < count and now < expire), and an fp32 base-2 online softmax updates
// the running max, sum and G x 8 accumulators of each lane.
//
// When a warp's slice ends a (b, h) segment it either owns the whole (b, h)
// (writes the output) or writes its partial (acc, m, l) to the workspace and
// bumps the (b, h)'s counter; the warp that brings the counter to the number
// of pieces merges them (log-sum-exp in fp32) and resets the counter. Nothing
// ever waits on another warp.
#include <cuda_fp16.h>

#include "kvp_common.cuh"

namespace kvp {
namespace {

constexpr int kWarps = 8;       // warps per CTA
// Pages in flight per warp. Two beat three on a GB300 (Llama-3-8B-shaped cache,
// G = 4: 88.1 / 32.4 / 16.4 us against 89.9 / 33.9 / 16.0 us at 0 / 75 /
// 93.75 % pruned): 1,216 warps x 2 pages already keep about 20 MB in flight.
constexpr int kNst = 2;
constexpr int kMaxBH = 4096;    // (b, h) pairs whose page prefix fits in shared memory
constexpr int kMaxCtas = 512;   // grid bound used to size the workspace
// Fewest pages a warp's slice gets when there are not enough pages for every
// warp of the grid: 8 when the average (b, h) has 64 pages or more (fewer
// pieces to merge), else 4 (more warps streaming). Measured on a GB300: 4 x
// 8192 tokens at 75 % pruned 20.7 us with 8 against 21.9 us with 4; 16 x 8192
// at 93.75 % pruned 24.8 us with 8 against 20.7 us with 4.
constexpr int kMinPagesLong = 8, kMinPagesShort = 4;
constexpr int kThreads = kWarps * 32;

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
  static constexpr int QPAGE_BYTES = kPage * D;         // fp8 tier: E4M3 codes of one page's K (or V) rows
  static constexpr int QMETA_BYTES = 3 * kPage * 4;     // fp8 tier: start, K scale, V scale per slot
  static constexpr int RING_BYTES = kWarps * kNst * STAGE_BYTES;
  static constexpr int PS_FLOATS = RPS * G * RS;  // per warp
  static constexpr int PS_BYTES = kWarps * PS_FLOATS * 4;
  static constexpr int BAR_BYTES = kWarps * (kNst + 1) * 8;  // per warp: ring stages, then its merge
  static constexpr int PREF_BYTES = (kMaxBH + 1) * 4;
  static constexpr int SMEM = RING_BYTES + PS_BYTES + BAR_BYTES + PREF_BYTES;
  static_assert(G <= LPR, "group larger than lanes per row");
  static_assert(STAGE_BYTES % 16 == 0 && PS_BYTES % 16 == 0, "16-byte layout");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(2 * QPAGE_BYTES + QMETA_BYTES <= STAGE_BYTES, "an fp8 page fits a stage");
};

struct AttnParams {
  const uint16_t* q;
  const uint16_t* k_pool;
  const uint16_t* v_pool;
  const int32_t* expire_pool;
  const int32_t* page_table;
  const int32_t* count;
  int B, H, Hq, max_pages, n_pages_cap, now;
  float qscale;
  float* out;        // [B, Hq, D]
  float* part_acc;   // [slots, G, D]
  float* part_ml;    // [slots, G, 2]
  int32_t* pieces;   // [B*H] arrival counters, zero at entry and exit
  int32_t* status;
  // fp8 tier (two-tier kernels only)
  const uint8_t* kq_pool;      // [n_pages_cap_q, 16, D] E4M3 codes
  const uint8_t* vq_pool;
  const int32_t* meta_pool;    // [n_pages_cap_q, 3, 16]: start, K scale, V scale
  const int32_t* page_table_q;
  const int32_t* count_q;
  int max_pages_q, n_pages_cap_q;
  const int32_t* now_dev;  // device int32 holding the decode position, or null: `now` is used
  float* lse;              // [B, Hq]: ln of the sum of exp(scaled logits) of each row, or null
};

// A row's natural log-sum-exp from its base-2 reference m2 and its sum
// l = sum 2^(x - m2) of the base-2 logits x (-inf when the row is empty).
KVP_DEV float row_lse(float m2, float l) { return l > 0.f ? (m2 + log2f(l)) * 0.69314718055994531f : -INFINITY; }

// Eight E4M3 codes (bytes of x then y, element 0 in the lowest byte) to fp32,
// exactly (every E4M3 value is an fp16 value).
KVP_DEV void unpack_e4m3_8(uint32_t x, uint32_t y, float (&f)[8]) {
  const uint32_t w[2] = {x, y};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t h2 = cvt_e4m3x2_to_f16x2(w[h] >> (16 * q));
      const float2 ff = __half22float2(*reinterpret_cast<const __half2*>(&h2));
      f[4 * h + 2 * q] = ff.x;
      f[4 * h + 2 * q + 1] = ff.y;
    }
  }
}

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

// d += a * b on two fp32 lanes at once: the packed f32x2 FMA of sm_100 and later.
KVP_DEV void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%0, %1};\n\t"
      "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rc;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// A logit may exceed the running max by this much (base 2) before the running
// state is rescaled: p then stays below 2^8, far inside fp32 range, and most
// pages skip the cross-lane max reduction altogether.
constexpr float kLazyRescale = 8.0f;


KVP_DEV int clamp_count(const int32_t* count, int bh, int max_pages) {
  return min(max(count[bh], 0), max_pages * kPage);
}

// Slices are cut evenly in a cost coordinate rather than in pages: page g of
// (b, h) number bh costs c(g) = 2g + kBoundaryCost * bh, i.e. every (b, h)
// start counts as kBoundaryCost / 2 extra pages. A slice that holds a (b, h)
// boundary stops its page stream to reduce and publish a partial state, so it
// gets fewer pages and the warps finish closer together (measured on a GB300
// at 16 x 8192 tokens: 3 extra pages per boundary, among 1.5 / 3 / 4.5 / 6,
// took the kernel from 36.0 to 34.7 us). c is strictly increasing, so slices
// are contiguous; a slice can be empty only between two (b, h) with empty ones
// in between, never inside one.
constexpr int kBoundaryCost = 6;

// Slice holding page g of (b, h) bh, for nw slices and total cost c_end.
KVP_DEV int slice_of(int g, int bh, int nw, int64_t c_end) {
  return static_cast<int>((2 * static_cast<int64_t>(g) + static_cast<int64_t>(kBoundaryCost) * bh) * nw / c_end);
}

// Merge of the npc partial states (acc, m, l) of (b, h) cbh, held in
// consecutive workspace slots from s0, by the warp whose arrival completed
// them: writes the output rows and resets the (b, h)'s counter. With `staged`
// (the warp's page ring is idle, at the end of its slice) two bulk copies
// bring every piece into the ring in one round trip; otherwise the lanes load
// them from L2 (the staged path holds one piece per lane: npc <= 32). Returns
// false if a bounded wait gave up.
template <int D, int G>
KVP_DEV bool merge_pieces(const AttnParams& p, int cbh, int npc, size_t s0, bool staged, uint8_t* ring,
                          uint64_t* mbar, uint32_t& merge_par, int lane) {
  // every piece of this (b, h) is written: merge them. Lanes take
  // pieces for the maxima and weights (one round of loads for up to
  // 32 pieces); then lanes take float4 columns of all G heads and the
  // pieces go by in batches of 8 whose loads are all in flight at once.
  fence_acq_rel_gpu();
  constexpr int F4 = G * D / 4;           // float4 of one piece's acc
  constexpr int FPL = (F4 + 31) / 32;     // ... per lane
  constexpr int JB = 16 / FPL < 8 ? (16 / FPL > 0 ? 16 / FPL : 1) : 8;  // pieces per batch of loads
  constexpr int kAccB = G * D * 4, kMlB = G * 2 * 4;  // bytes of a piece's acc and (m, l)
  if (staged) {
    // End of the slice: this warp's ring is idle. The pieces sit in
    // consecutive slots, so two bulk copies bring every acc and every
    // (m, l) into it in one round trip.
    float* sacc = reinterpret_cast<float*>(ring);
    uint8_t* sml_raw = ring + static_cast<size_t>(npc) * kAccB;
    const size_t ml0 = s0 * kMlB, ml_a = ml0 & ~size_t(15);
    const size_t ml_b = (ml0 + static_cast<size_t>(npc) * kMlB + 15) & ~size_t(15);
    const float* sml = reinterpret_cast<const float*>(sml_raw + (ml0 - ml_a));
    if (lane == 0) {
      fence_proxy_async();
      mbar_arrive_expect_tx(mbar, static_cast<uint32_t>(npc * kAccB + (ml_b - ml_a)));
      bulk_g2s(sacc, p.part_acc + s0 * G * D, static_cast<uint32_t>(npc * kAccB), mbar);
      bulk_g2s(sml_raw, reinterpret_cast<const uint8_t*>(p.part_ml) + ml_a, static_cast<uint32_t>(ml_b - ml_a),
               mbar);
    }
    const bool okm = mbar_wait(mbar, merge_par, nullptr, p.status);
    merge_par ^= 1u;
    if (!__all_sync(0xffffffffu, okm)) {
      if (lane == 0) {
        record_error(p.status, KVP_ERR_TIMEOUT);
        (void)mbar_wait(mbar, merge_par ^ 1u);  // the two copies land before the ring is released (bounded)
      }
      __syncwarp();
      return false;
    }
    float M[G], wr[G], L[G];
#pragma unroll
    for (int i = 0; i < G; ++i) {
      const float m = lane < npc ? sml[lane * G * 2 + 2 * i] : -1e30f;
      float mx = m;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      M[i] = mx;
      wr[i] = lane < npc ? exp2f(m - mx) : 0.f;
      float l = wr[i] * (lane < npc ? sml[lane * G * 2 + 2 * i + 1] : 0.f);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      L[i] = l;
    }
    if (p.lse != nullptr && lane < G) {
      float mm = M[0], ll = L[0];
#pragma unroll
      for (int i = 1; i < G; ++i)
        if (lane == i) {
          mm = M[i];
          ll = L[i];
        }
      p.lse[static_cast<size_t>(cbh) * G + lane] = row_lse(mm, ll);
    }
    float4 A[FPL];
#pragma unroll
    for (int k2 = 0; k2 < FPL; ++k2) A[k2] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < npc; ++j) {
#pragma unroll
      for (int k2 = 0; k2 < FPL; ++k2) {
        constexpr int kHeadF4 = D / 4;
        const int h0 = (32 * k2) / kHeadF4 < G ? (32 * k2) / kHeadF4 : G - 1;
        float w = __shfl_sync(0xffffffffu, wr[h0], j);
        if constexpr (kHeadF4 < 32) {
          const int h1 = (32 * k2 + 16) / kHeadF4 < G ? (32 * k2 + 16) / kHeadF4 : G - 1;
          const float w1 = __shfl_sync(0xffffffffu, wr[h1], j);
          if (lane >= 16) w = w1;
        }
        const int f = lane + 32 * k2;
        if (f < F4) {
          const float4 v = reinterpret_cast<const float4*>(sacc + static_cast<size_t>(j) * G * D)[f];
          A[k2].x = fmaf(w, v.x, A[k2].x);
          A[k2].y = fmaf(w, v.y, A[k2].y);
          A[k2].z = fmaf(w, v.z, A[k2].z);
          A[k2].w = fmaf(w, v.w, A[k2].w);
        }
      }
    }
#pragma unroll
    for (int k2 = 0; k2 < FPL; ++k2) {
      const int f = lane + 32 * k2;
      if (f < F4) {
        const int hd = f / (D / 4);
        float Lh = L[0];
#pragma unroll
        for (int i = 1; i < G; ++i)
          if (hd == i) Lh = L[i];
        const float inv = Lh > 0.f ? 1.f / Lh : 0.f;
        reinterpret_cast<float4*>(p.out + static_cast<size_t>(cbh) * G * D)[f] =
            make_float4(A[k2].x * inv, A[k2].y * inv, A[k2].z * inv, A[k2].w * inv);
      }
    }
    if (lane == 0) p.pieces[cbh] = 0;
    return true;
  }
  float M[G], mr[G], lr[G];
#pragma unroll
  for (int i = 0; i < G; ++i) M[i] = -1e30f;
  for (int b0 = 0; b0 < npc; b0 += 32) {
    const int pc = b0 + lane;
#pragma unroll
    for (int i = 0; i < G; ++i) {
      mr[i] = pc < npc ? __ldcg(p.part_ml + ((s0 + pc) * G + i) * 2) : -1e30f;
      lr[i] = pc < npc ? __ldcg(p.part_ml + ((s0 + pc) * G + i) * 2 + 1) : 0.f;
      M[i] = fmaxf(M[i], mr[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < G; ++i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M[i] = fmaxf(M[i], __shfl_xor_sync(0xffffffffu, M[i], o));
  }
  float L[G];
  float4 A[FPL];
#pragma unroll
  for (int i = 0; i < G; ++i) L[i] = 0.f;
#pragma unroll
  for (int k = 0; k < FPL; ++k) A[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int b0 = 0; b0 < npc; b0 += 32) {
    const int pc = b0 + lane;
    if (npc > 32) {  // the registers hold the last chunk of the first pass
#pragma unroll
      for (int i = 0; i < G; ++i) {
        mr[i] = pc < npc ? __ldcg(p.part_ml + ((s0 + pc) * G + i) * 2) : -1e30f;
        lr[i] = pc < npc ? __ldcg(p.part_ml + ((s0 + pc) * G + i) * 2 + 1) : 0.f;
      }
    }
    float wr[G];
#pragma unroll
    for (int i = 0; i < G; ++i) {
      wr[i] = pc < npc ? exp2f(mr[i] - M[i]) : 0.f;
      L[i] = fmaf(wr[i], lr[i], L[i]);
    }
    const int nb = min(32, npc - b0);
    for (int j0 = 0; j0 < nb; j0 += JB) {
      float4 v[JB][FPL];
#pragma unroll
      for (int jj = 0; jj < JB; ++jj) {
#pragma unroll
        for (int k = 0; k < FPL; ++k) {
          const int f = lane + 32 * k;
          v[jj][k] = (j0 + jj < nb && f < F4)
                         ? __ldcg(reinterpret_cast<const float4*>(p.part_acc + (s0 + b0 + j0 + jj) * G * D) + f)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int jj = 0; jj < JB; ++jj) {
        const int src = (j0 + jj) & 31;  // the lane that holds this piece's weights
#pragma unroll
        for (int k = 0; k < FPL; ++k) {
          constexpr int kHeadF4 = D / 4;  // float4 per head row
          const int h0 = (32 * k) / kHeadF4 < G ? (32 * k) / kHeadF4 : G - 1;
          float w = __shfl_sync(0xffffffffu, wr[h0], src);
          if constexpr (kHeadF4 < 32) {  // lanes 16-31 are on the next head
            const int h1 = (32 * k + 16) / kHeadF4 < G ? (32 * k + 16) / kHeadF4 : G - 1;
            const float w1 = __shfl_sync(0xffffffffu, wr[h1], src);
            if (lane >= 16) w = w1;
          }
          A[k].x = fmaf(w, v[jj][k].x, A[k].x);
          A[k].y = fmaf(w, v[jj][k].y, A[k].y);
          A[k].z = fmaf(w, v[jj][k].z, A[k].z);
          A[k].w = fmaf(w, v[jj][k].w, A[k].w);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < G; ++i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L[i] += __shfl_xor_sync(0xffffffffu, L[i], o);
  }
  if (p.lse != nullptr && lane < G) {
    float mm = M[0], ll = L[0];
#pragma unroll
    for (int i = 1; i < G; ++i)
      if (lane == i) {
        mm = M[i];
        ll = L[i];
      }
    p.lse[static_cast<size_t>(cbh) * G + lane] = row_lse(mm, ll);
  }
#pragma unroll
  for (int k = 0; k < FPL; ++k) {
    const int f = lane + 32 * k;
    if (f < F4) {
      const int hd = f / (D / 4);
      float Lh = L[0];
#pragma unroll
      for (int i = 1; i < G; ++i)
        if (hd == i) Lh = L[i];
      const float inv = Lh > 0.f ? 1.f / Lh : 0.f;
      reinterpret_cast<float4*>(p.out + static_cast<size_t>(cbh) * G * D)[f] =
          make_float4(A[k].x * inv, A[k].y * inv, A[k].z * inv, A[k].w * inv);
    }
  }
  if (lane == 0) p.pieces[cbh] = 0;
  return true;
}

// kQ: the two-tier kernel. Each (b, h) then lists its bf16 pages and after
// them its fp8-tier pages (quantize instead of drop): a fp8 page stages its K
// and V codes and its per-slot record; a lane reads the 8 codes of the same 8
// columns it covers in a bf16 row, the K row scale multiplies the lane's
// partial dot product and the V row scale multiplies p in the P.V update (the
// softmax sum takes p itself); a slot of that tier counts once now >= start.
template <int D, int G, bool kQ>
__global__ void __launch_bounds__(kThreads, 1) attn_decode_kernel(const AttnParams p) {
  using C = AttnCfg<D, G>;
  extern __shared__ __align__(128) uint8_t smem[];
  pdl_launch_dependents();
  pdl_wait();  // inputs (counts, pages, workspace counters) come from the kernels before this one
  const int now = p.now_dev != nullptr ? *p.now_dev : p.now;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = p.B * p.H;
  uint8_t* ring = smem + warp * kNst * C::STAGE_BYTES;
  float* p_s = reinterpret_cast<float*>(smem + C::RING_BYTES) + warp * C::PS_FLOATS;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::RING_BYTES + C::PS_BYTES) + warp * (kNst + 1);
  int* pref = reinterpret_cast<int*>(smem + C::RING_BYTES + C::PS_BYTES + C::BAR_BYTES);

  // ---- page prefix over (b, h), identical in every CTA, and the last (b, h) with pages
  __shared__ int s_last_bh;
  {
    __shared__ int wsum[kWarps];
    __shared__ int wlast[kWarps];
    __shared__ int carry;
    if (tid == 0) {
      carry = 0;
      s_last_bh = 0;
    }
    __syncthreads();
    for (int base = 0; base < BH; base += kThreads) {
      const int bh = base + tid;
      int np = bh < BH ? (clamp_count(p.count, bh, p.max_pages) + kPage - 1) / kPage : 0;
      if constexpr (kQ) np += bh < BH ? (clamp_count(p.count_q, bh, p.max_pages_q) + kPage - 1) / kPage : 0;
      int incl = np;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int wl = __reduce_max_sync(0xffffffffu, np > 0 ? bh : -1);
      if (lane == 31) wsum[warp] = incl;
      if (lane == 0) wlast[warp] = wl;
      __syncthreads();
      int before = carry;
      for (int w = 0; w < warp; ++w) before += wsum[w];
      if (bh < BH) pref[bh] = before + incl - np;
      __syncthreads();
      if (tid == 0) {
        int t = 0, lb = s_last_bh;
        for (int w = 0; w < kWarps; ++w) {
          t += wsum[w];
          lb = max(lb, wlast[w]);
        }
        carry += t;
        s_last_bh = lb;
      }
      __syncthreads();
    }
    if (tid == 0) pref[BH] = carry;
    __syncthreads();
  }
  const int NP = pref[BH];

  // ---- (b, h) without pages: zero output rows
  for (int bh = blockIdx.x; bh < BH; bh += gridDim.x) {
    if (pref[bh + 1] == pref[bh]) {
      for (int i = tid; i < G * D; i += kThreads) p.out[static_cast<size_t>(bh) * G * D + i] = 0.f;
      if (p.lse != nullptr && tid < G) p.lse[static_cast<size_t>(bh) * G + tid] = -INFINITY;
    }
  }
  if (NP == 0) return;

  // ---- this warp's slice of the global page list
  // slices of at least min_pages pages (fewer pieces to merge on small
  // problems); every one of the first NW slices is non-empty
  const int nw_all = gridDim.x * kWarps;
  const int min_pages = NP >= 64 * BH ? kMinPagesLong : kMinPagesShort;
  const int NW = max(1, min(nw_all, NP / min_pages));
  const int gw = warp * gridDim.x + blockIdx.x;  // slices go round-robin over the CTAs (all SMs busy)
  if (gw >= NW) return;
  const int last_bh = s_last_bh;  // (b, h) of the last page
  const int64_t c_end = 2 * static_cast<int64_t>(NP - 1) + static_cast<int64_t>(kBoundaryCost) * last_bh + 1;
  // first page of slice w: the first page whose cost reaches ceil(w * c_end / NW); a_out: the (b, h) searched
  // to (that page's, or one before it with no pages)
  auto slice_start = [&](int w, int& a_out) {
    const int64_t T = (static_cast<int64_t>(w) * c_end + NW - 1) / NW;
    auto maxc = [&](int k) {
      return 2 * static_cast<int64_t>(pref[k + 1] - 1) + static_cast<int64_t>(kBoundaryCost) * k;
    };
    if (maxc(BH - 1) < T) return NP;
    int a = 0, b = BH - 1;
    while (a < b) {
      const int mid = (a + b) >> 1;
      if (maxc(mid) >= T) b = mid; else a = mid + 1;
    }
    const int64_t g = (T - static_cast<int64_t>(kBoundaryCost) * a + 1) / 2;
    a_out = a;
    return static_cast<int>(min(static_cast<int64_t>(NP), max(static_cast<int64_t>(pref[a]), g)));
  };
  // the slice's two ends on two lanes at once (a serial chain of integer work each)
  int a_s = 0, r_s = NP;
  if (lane == 0) r_s = slice_start(gw, a_s);
  if (lane == 1 && gw + 1 < NW) r_s = slice_start(gw + 1, a_s);
  const int r0 = __shfl_sync(0xffffffffu, r_s, 0);
  const int r1 = __shfl_sync(0xffffffffu, r_s, 1);
  if (r1 <= r0) return;  // an empty slice (between two (b, h) with empty ones in between)
  const int n_my = r1 - r0;

  // first (b, h) of the slice: the one whose page range holds page r0 (the start's search ended at it or at
  // a (b, h) with no pages before it)
  int cbh = __shfl_sync(0xffffffffu, a_s, 0);  // consumer cursor
  while (pref[cbh + 1] <= r0) ++cbh;

  // Page ids of the slice, 32 per register: lane j of block b holds the id of
  // slice page 32*b + j. Block b+1 is loaded when issuing enters block b, so
  // every id is in a register about 32 pages before lane 0 needs it.
  // bit j of qb0 / qb1: slice page 32 * blk + j (blk even / odd) is a fp8-tier page
  uint32_t qb0 = 0, qb1 = 0;
  auto load_ids = [&](int blk, uint32_t& qbits) {  // all lanes call this
    const int kk = blk * 32 + lane;
    int id = -1;
    bool isq = false;
    if (kk < n_my) {
      const int g = r0 + kk;
      int a = 0, b = BH - 1;
      while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (pref[mid] <= g) a = mid; else b = mid - 1;
      }
      const int li = g - pref[a];
      if constexpr (kQ) {
        const int na = (clamp_count(p.count, a, p.max_pages) + kPage - 1) / kPage;
        isq = li >= na;
        id = isq ? static_cast<int>(p.page_table_q[static_cast<int64_t>(a) * p.max_pages_q + (li - na)])
                 : static_cast<int>(p.page_table[static_cast<int64_t>(a) * p.max_pages + li]);
      } else {
        id = static_cast<int>(p.page_table[static_cast<int64_t>(a) * p.max_pages + li]);
      }
    }
    if constexpr (kQ) qbits = __ballot_sync(0xffffffffu, isq);
    return id;
  };
  int ids0 = load_ids(0, qb0), ids1 = load_ids(1, qb1);
  auto page_id = [&](int k, bool& isq) {  // all lanes call this
    const int blk = k >> 5;
    const int v = __shfl_sync(0xffffffffu, (blk & 1) ? ids1 : ids0, k & 31);
    isq = kQ && ((((blk & 1) ? qb1 : qb0) >> (k & 31)) & 1u);
    if ((k & 31) == 0 && k > 0) {  // block blk - 1 is done: its register takes block blk + 1
      if (blk & 1) ids0 = load_ids(blk + 1, qb0); else ids1 = load_ids(blk + 1, qb1);
    }
    return v;
  };
  auto issue = [&](int k, int64_t phys, bool isq) {  // lane 0
    const int st = k % kNst;
    uint8_t* dst = ring + st * C::STAGE_BYTES;
    if (phys < 0 || phys >= (isq ? p.n_pages_cap_q : p.n_pages_cap)) {
      // inconsistent page table: no copy; the stage reads as an empty page
      record_error(p.status, KVP_ERR_BOUNDS);
      uint4* z = reinterpret_cast<uint4*>(dst);
      for (int i = 0; i < C::STAGE_BYTES / 16; ++i) z[i] = make_uint4(0, 0, 0, 0);
      if (isq) {  // a fp8 slot counts once now >= start: make every start unreachable
        int32_t* starts = reinterpret_cast<int32_t*>(dst + 2 * C::QPAGE_BYTES);
        for (int i = 0; i < kPage; ++i) starts[i] = kNever;
      }
      mbar_arrive(&bars[st]);
      return;
    }
    if (kQ && isq) {
      mbar_arrive_expect_tx(&bars[st], 2 * C::QPAGE_BYTES + C::QMETA_BYTES);
      bulk_g2s(dst, p.kq_pool + phys * C::QPAGE_BYTES, C::QPAGE_BYTES, &bars[st]);
      bulk_g2s(dst + C::QPAGE_BYTES, p.vq_pool + phys * C::QPAGE_BYTES, C::QPAGE_BYTES, &bars[st]);
      bulk_g2s(dst + 2 * C::QPAGE_BYTES, p.meta_pool + phys * 3 * kPage, C::QMETA_BYTES, &bars[st]);
      return;
    }
    mbar_arrive_expect_tx(&bars[st], C::STAGE_BYTES);
    bulk_g2s(dst, p.k_pool + phys * kPage * D, C::PAGE_BYTES, &bars[st]);
    bulk_g2s(dst + C::PAGE_BYTES, p.v_pool + phys * kPage * D, C::PAGE_BYTES, &bars[st]);
    bulk_g2s(dst + 2 * C::PAGE_BYTES, p.expire_pool + phys * kPage, kPage * 4, &bars[st]);
  };
  if (lane == 0) {
    for (int st = 0; st <= kNst; ++st) mbar_init(&bars[st], 1);
    fence_mbar_init();
  }
  __syncwarp();
  for (int k = 0; k < n_my && k < kNst; ++k) {
    bool isq;
    const int pid = page_id(k, isq);
    if (lane == 0) issue(k, pid, isq);
  }
  __syncwarp();

  const int rowsel = lane / C::LPR;
  const int s = lane % C::LPR;
  const int idx_base = (C::V >= C::LPR) ? s * C::VL : s / C::DUP;
  const int my_head = idx_base / C::RS;

  auto load_q = [&](int bh, uint4 (&raw)[G]) {
#pragma unroll
    for (int i = 0; i < G; ++i)
      raw[i] = __ldg(reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(bh) * G + i) * D) + s);
  };
  auto next_bh = [&](int bh) {  // next (b, h) that has pages
    int n = bh + 1;
    while (n < BH && pref[n + 1] == pref[n]) ++n;
    return n;
  };

  float qf[G][8];
  uint4 qn[G];
  {
    uint4 qc[G];
    load_q(cbh, qc);
#pragma unroll
    for (int i = 0; i < G; ++i) {
      unpack8(qc[i], qf[i]);
#pragma unroll
      for (int e = 0; e < 8; ++e) qf[i][e] *= p.qscale;
    }
  }
  int seg_end = min(pref[cbh + 1], r1);
  int cnt = clamp_count(p.count, cbh, p.max_pages);
  int cnt_next = 0;
  int cnt_q = kQ ? clamp_count(p.count_q, cbh, p.max_pages_q) : 0;  // fp8-tier slots of this (b, h)
  int cnt_q_next = 0;
  if (seg_end < r1) {
    if constexpr (G < 8) load_q(next_bh(cbh), qn);  // G = 8 loads the next query rows at the switch
    cnt_next = clamp_count(p.count, next_bh(cbh), p.max_pages);
    if constexpr (kQ) cnt_q_next = clamp_count(p.count_q, next_bh(cbh), p.max_pages_q);
  }

  float m_run[G], l_run[G], acc[G][8];
#pragma unroll
  for (int i = 0; i < G; ++i) {
    m_run[i] = -1e30f;
    l_run[i] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
  }

  uint32_t merge_par = 0;  // phase of this warp's merge barrier
  for (int k = 0; k < n_my; ++k) {
    const int g = r0 + k;
    const int st = k % kNst;
    const bool ok = mbar_wait(&bars[st], static_cast<uint32_t>((k / kNst) & 1), nullptr, p.status);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) {
        record_error(p.status, KVP_ERR_TIMEOUT);
        // let the copies this warp issued land before its shared memory can
        // go to another CTA (each wait bounded again)
        for (int kk = k; kk < n_my && kk < k + kNst; ++kk) (void)mbar_wait(&bars[kk % kNst], (kk / kNst) & 1u);
      }
      __syncwarp();
      return;  // outputs of this call are unspecified after a timeout
    }
    const uint8_t* stage = ring + st * C::STAGE_BYTES;
    const uint16_t* Ks = reinterpret_cast<const uint16_t*>(stage);
    const uint16_t* Vs = reinterpret_cast<const uint16_t*>(stage + C::PAGE_BYTES);
    const int32_t* Es = reinterpret_cast<const int32_t*>(stage + 2 * C::PAGE_BYTES);
    const int li = g - pref[cbh];
    const int na_cur = (cnt + kPage - 1) / kPage;  // bf16 pages of this (b, h)
    const bool isq = kQ && li >= na_cur;           // a fp8-tier page (uniform in the warp)
    const int slot0 = (isq ? li - na_cur : li) * kPage;

    // For G <= 4 this lane's share of the page goes to registers and the
    // stage is handed straight back to the copy engine, so every stage of the
    // ring stays in flight while the warp computes. For G = 8 the query rows
    // and accumulators take those registers: K and V are read from the stage
    // where they are used and the stage goes back after the page.
    constexpr bool kRegStage = G < 8;
    const uint8_t* Kq = stage;
    const uint8_t* Vq = stage + C::QPAGE_BYTES;
    const int32_t* Mq = reinterpret_cast<const int32_t*>(stage + 2 * C::QPAGE_BYTES);
    // the lane's 16 bytes of K (or V) row t * RPS + rowsel; fp8 page: the 8
    // codes in .x/.y and, for V, the row's scale in .z
    auto k_word = [&](int t) {
      const int row = t * C::RPS + rowsel;
      if (isq) {
        const uint2 kc = reinterpret_cast<const uint2*>(Kq + row * D)[s];
        return make_uint4(kc.x, kc.y, 0u, 0u);
      }
      return reinterpret_cast<const uint4*>(Ks + row * D)[s];
    };
    auto v_word = [&](int t) {
      const int row = t * C::RPS + rowsel;
      if (isq) {
        const uint2 vc = reinterpret_cast<const uint2*>(Vq + row * D)[s];
        return make_uint4(vc.x, vc.y, static_cast<uint32_t>(Mq[2 * kPage + row]), 0u);
      }
      return reinterpret_cast<const uint4*>(Vs + row * D)[s];
    };
    auto issue_next = [&]() {
      __syncwarp();
      if (k + kNst < n_my) {
        bool isq_n;
        const int pid = page_id(k + kNst, isq_n);
        if (lane == 0) {
          fence_proxy_async();
          issue(k + kNst, pid, isq_n);
        }
      }
    };
    uint4 kr[kRegStage ? C::RS : 1], vr[kRegStage ? C::RS : 1];
    int32_t er[C::VL];
    float ksu[C::VL];  // fp8 page: K scale of the row of each logit this lane holds after the reduction
    if constexpr (kRegStage) {
#pragma unroll
      for (int t = 0; t < C::RS; ++t) {
        kr[t] = k_word(t);
        vr[t] = v_word(t);
      }
    }
    if (isq) {
#pragma unroll
      for (int u = 0; u < C::VL; ++u) {
        const int r = ((idx_base + u) % C::RS) * C::RPS + rowsel;
        er[u] = Mq[r];
        ksu[u] = __int_as_float(Mq[kPage + r]);
      }
    } else {
#pragma unroll
      for (int u = 0; u < C::VL; ++u) er[u] = Es[((idx_base + u) % C::RS) * C::RPS + rowsel];
    }
    if constexpr (kRegStage) issue_next();

    // ---- logits
    float part[C::V];
#pragma unroll
    for (int t = 0; t < C::RS; ++t) {
      float kf[8];
      uint4 kw;
      if constexpr (kRegStage) kw = kr[t]; else kw = k_word(t);
      if (isq) unpack_e4m3_8(kw.x, kw.y, kf); else unpack8(kw, kf);
#pragma unroll
      for (int i = 0; i < G; ++i) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int e = 0; e < 8; e += 2) fma2(a0, a1, qf[i][e], qf[i][e + 1], kf[e], kf[e + 1]);
        part[i * C::RS + t] = a0 + a1;
      }
    }
    TransposeReduce<C::V, C::LPR / 2>::run(part, lane);

    float mh = m_run[0];
#pragma unroll
    for (int i = 1; i < G; ++i)
      if (my_head == i) mh = m_run[i];
    float x[C::VL];
    bool grow = false;
#pragma unroll
    for (int u = 0; u < C::VL; ++u) {
      const int r = ((idx_base + u) % C::RS) * C::RPS + rowsel;
      const bool valid = isq ? (slot0 + r < cnt_q) && (now >= er[u]) : (slot0 + r < cnt) && (now < er[u]);
      x[u] = valid ? (isq ? part[u] * ksu[u] : part[u]) : -INFINITY;
      grow |= x[u] > mh + kLazyRescale;
    }
    if (__any_sync(0xffffffffu, grow)) {
      // a logit outgrew the running max: exact page max per head, rescale
      float mloc = -INFINITY;
#pragma unroll
      for (int u = 0; u < C::VL; ++u) mloc = fmaxf(mloc, x[u]);
#pragma unroll
      for (int o = 1; o < C::GL; o <<= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
#pragma unroll
      for (int o = C::LPR; o < 32; o <<= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
#pragma unroll
      for (int i = 0; i < G; ++i) {
        const float mi = __shfl_sync(0xffffffffu, mloc, i * C::GL);
        const float mnew = fmaxf(m_run[i], mi);
        const float alpha = exp2f(m_run[i] - mnew);
        m_run[i] = mnew;
        l_run[i] *= alpha;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] *= alpha;
      }
      mh = m_run[0];
#pragma unroll
      for (int i = 1; i < G; ++i)
        if (my_head == i) mh = m_run[i];
    }
#pragma unroll
    for (int u = 0; u < C::VL; ++u) {
      const float pv = exp2f(x[u] - mh);
      if (s % C::DUP == 0) p_s[rowsel * G * C::RS + idx_base + u] = pv;
    }
    __syncwarp();

    // ---- accumulate P . V
#pragma unroll
    for (int t = 0; t < C::RS; ++t) {
      float vf[8];
      uint4 vw;
      if constexpr (kRegStage) vw = vr[t]; else vw = v_word(t);
      if (isq) unpack_e4m3_8(vw.x, vw.y, vf); else unpack8(vw, vf);
#pragma unroll
      for (int i = 0; i < G; ++i) {
        const float pr = p_s[rowsel * G * C::RS + i * C::RS + t];
        l_run[i] += pr;
        const float pw = isq ? pr * __uint_as_float(vw.z) : pr;
#pragma unroll
        for (int e = 0; e < 8; e += 2) fma2(acc[i][e], acc[i][e + 1], pw, pw, vf[e], vf[e + 1]);
      }
    }
    if constexpr (!kRegStage) issue_next();  // the stage is read for the last time above

    // ---- end of a (b, h) segment of this slice
    if (g + 1 == seg_end) {
      // the running state is reset after this segment: combine the row groups in place
      float (&lt)[G] = l_run;
      float (&at)[G][8] = acc;
#pragma unroll
      for (int o = C::LPR; o < 32; o <<= 1) {
#pragma unroll
        for (int i = 0; i < G; ++i) {
          lt[i] += __shfl_xor_sync(0xffffffffu, lt[i], o);
#pragma unroll
          for (int e = 0; e < 8; ++e) at[i][e] += __shfl_xor_sync(0xffffffffu, at[i][e], o);
        }
      }
      const bool whole = pref[cbh] >= r0 && pref[cbh + 1] <= r1;
      if (whole) {
        if (p.lse != nullptr && lane < G) {
          float mm = m_run[0], ll = lt[0];
#pragma unroll
          for (int i = 1; i < G; ++i)
            if (lane == i) {
              mm = m_run[i];
              ll = lt[i];
            }
          p.lse[static_cast<size_t>(cbh) * G + lane] = row_lse(mm, ll);
        }
        if (rowsel == 0) {
#pragma unroll
          for (int i = 0; i < G; ++i) {
            float4* o = reinterpret_cast<float4*>(p.out + (static_cast<size_t>(cbh) * G + i) * D + 8 * s);
            const float inv = lt[i] > 0.f ? 1.f / lt[i] : 0.f;
            o[0] = make_float4(at[i][0] * inv, at[i][1] * inv, at[i][2] * inv, at[i][3] * inv);
            o[1] = make_float4(at[i][4] * inv, at[i][5] * inv, at[i][6] * inv, at[i][7] * inv);
          }
        }
      } else {
        const int w_first = slice_of(pref[cbh], cbh, NW, c_end);
        const int w_last = slice_of(pref[cbh + 1] - 1, cbh, NW, c_end);
        const size_t slot = static_cast<size_t>(gw) + cbh;
        if (rowsel == 0) {
#pragma unroll
          for (int i = 0; i < G; ++i) {
            float4* o = reinterpret_cast<float4*>(p.part_acc + (slot * G + i) * D + 8 * s);
            o[0] = make_float4(at[i][0], at[i][1], at[i][2], at[i][3]);
            o[1] = make_float4(at[i][4], at[i][5], at[i][6], at[i][7]);
          }
        }
        if (lane < G) {
          float mm = m_run[0], ll = lt[0];
#pragma unroll
          for (int i = 1; i < G; ++i)
            if (lane == i) {
              mm = m_run[i];
              ll = lt[i];
            }
          p.part_ml[(slot * G + lane) * 2] = mm;
          p.part_ml[(slot * G + lane) * 2 + 1] = ll;
        }
        fence_acq_rel_gpu();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(&p.pieces[cbh], 1) == (w_last - w_first);
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          constexpr int kAccB = G * D * 4, kMlB = G * 2 * 4;  // bytes of a piece's acc and (m, l)
          // pieces the staged merge takes: as many as the idle ring holds, and at
          // most one per lane (its maxima and weights are held one piece per lane)
          constexpr int kRingPieces = (kNst * C::STAGE_BYTES - 32) / (kAccB + kMlB);
          constexpr int kStaged = kRingPieces < 32 ? kRingPieces : 32;
          const int npc = w_last - w_first + 1;
          if (!merge_pieces<D, G>(p, cbh, npc, static_cast<size_t>(w_first) + cbh, g + 1 == r1 && npc <= kStaged,
                                  ring, &bars[kNst], merge_par, lane))
            return;
        }
      }
      // next segment
      if (g + 1 < r1) {
        cbh = next_bh(cbh);
        seg_end = min(pref[cbh + 1], r1);
        cnt = cnt_next;
        cnt_q = cnt_q_next;
        if constexpr (G >= 8) load_q(cbh, qn);
#pragma unroll
        for (int i = 0; i < G; ++i) {
          unpack8(qn[i], qf[i]);
#pragma unroll
          for (int e = 0; e < 8; ++e) qf[i][e] *= p.qscale;
        }
        if (seg_end < r1) {
          if constexpr (G < 8) load_q(next_bh(cbh), qn);
          cnt_next = clamp_count(p.count, next_bh(cbh), p.max_pages);
          if constexpr (kQ) cnt_q_next = clamp_count(p.count_q, next_bh(cbh), p.max_pages_q);
        }
#pragma unroll
        for (int i = 0; i < G; ++i) {
          m_run[i] = -1e30f;
          l_run[i] = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- tensor-core page math
// The same persistent split-KV decode, with each page's two products on the
// tensor cores (mma.sync m16n8k16, bf16 operands, fp32 accumulate):
//   S   = K Q^T    M = 16 tokens, N = 8 query heads of the kv head (G <= 8,
//                  the rest zero), K = head_dim in steps of 16
//   O^T = V^T P^T  M = 16 dims per step, N = 8 heads, K = the page's 16 tokens
// K and V arrive as 16-row x 64-column boxes with the 128-byte swizzle, so the
// ldmatrix reads (V transposed by the load itself) are free of bank
// conflicts; P goes through 512 bytes of shared memory per warp, as a bf16
// hi + lo pair (two products, about 16 bits of p), to become the second
// product's B operand. A thread owns heads 2t and 2t+1 of both
// results, so its softmax state and its output columns coincide.
template <int D>
struct MmaCfg {
  static constexpr int NBOX = D / 64;                    // 64-column boxes per page of K (or V)
  static constexpr int BOX_BYTES = kPage * 128;          // 16 rows x 128 bytes
  static constexpr int PAGE_BYTES = NBOX * BOX_BYTES;
  static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;     // K boxes, then V boxes
  static constexpr int RING_BYTES = kWarps * kNst * STAGE_BYTES;
  static constexpr int REC_WORDS = 3 * kPage;            // per stage: the page's 16 expire values
  static constexpr int REC_BYTES = kWarps * kNst * REC_WORDS * 4;
  // per warp: P^T hi and lo, 8 heads x 16 tokens, bf16; a head's row padded to kPtRow halves so that the
  // stores (lanes 4 apart in heads) and the 32-bit reads (8 heads x 4 token pairs) fall on distinct banks
  static constexpr int kPtRow = 24;
  static constexpr int PT_BYTES = kWarps * 2 * 8 * kPtRow * 2;
  static constexpr int BAR_BYTES = kWarps * (kNst + 1) * 8;
  static constexpr int PREF_BYTES = (kMaxBH + 1) * 4;
  static constexpr int SMEM = 1024 + RING_BYTES + REC_BYTES + PT_BYTES + BAR_BYTES + PREF_BYTES;
  static constexpr int QPAGE_BYTES = kPage * D;         // fp8 tier: E4M3 codes of a page's K (or V) rows
  // where the codes land (swizzled tensor copies, read in place): K's in the room of the K boxes, V's in the
  // room of the V boxes, each on a 1024-byte boundary
  static constexpr int QK_OFF = 0;
  static constexpr int QV_OFF = PAGE_BYTES;
  static_assert(D == 64 || D == 128, "a code row is one 64- or 128-byte swizzle span");
  static_assert(QV_OFF % 1024 == 0 && QV_OFF + QPAGE_BYTES <= STAGE_BYTES, "code tiles");
  static_assert(PAGE_BYTES == kPage * D * 2, "a page is its boxes");
  static_assert(STAGE_BYTES % 1024 == 0, "swizzled boxes start on 1024 bytes");
  static_assert(SMEM <= 232448, "shared memory budget");
};

KVP_DEV uint32_t bf16x2_to_f16x2(uint32_t w) {
  const __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// kQ: the two-tier kernel. A fp8-tier page arrives as its E4M3 codes and its
// record (start steps, K and V row scales). The codes come by tensor copies
// with the swizzle of their row width and are read by ldmatrix as they are;
// each pair of codes becomes fp16 in registers (exactly: every E4M3 value is
// an fp16 value). K: a thread holds dims 4t .. 4t + 3 of its rows where the
// fp16 product expects 2t, 2t + 1, 2t + 8, 2t + 9, so the query fragments take
// the same order (a dot product does not depend on the order of its terms),
// converted to fp16 once per (b, h). V, read transposed as 16-bit words: a
// thread holds dims 2g, 2g + 1 of tokens 2t, 2t + 1, so its output rows g and
// g + 8 are dims 2g and 2g + 1 of each 16 (the accumulators are moved to that
// order by shuffles at the (b, h)'s first fp8 page, and stored from it). The
// K row scale applies to S; the V row scale is folded into p, which enters
// the product as one fp16 value (11 bits; the bf16 pages take p as a bf16
// hi + lo pair).
template <int D, int G, bool kQ>
__global__ void __launch_bounds__(kThreads, 1) attn_mma_kernel(const AttnParams p,
                                                               const __grid_constant__ CUtensorMap tmK,
                                                               const __grid_constant__ CUtensorMap tmV,
                                                               const __grid_constant__ CUtensorMap tmKq,
                                                               const __grid_constant__ CUtensorMap tmVq) {
  using C = MmaCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  pdl_launch_dependents();
  pdl_wait();  // inputs (counts, pages, workspace counters) come from the kernels before this one
  const int now = p.now_dev != nullptr ? *p.now_dev : p.now;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = p.B * p.H;
  uint8_t* ring = smem + warp * kNst * C::STAGE_BYTES;
  int32_t* exp_s = reinterpret_cast<int32_t*>(smem + C::RING_BYTES) + warp * kNst * C::REC_WORDS;
  uint16_t* pt_s = reinterpret_cast<uint16_t*>(smem + C::RING_BYTES + C::REC_BYTES) + warp * 2 * 8 * C::kPtRow;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::RING_BYTES + C::REC_BYTES + C::PT_BYTES) + warp * (kNst + 1);
  int* pref = reinterpret_cast<int*>(smem + C::RING_BYTES + C::REC_BYTES + C::PT_BYTES + C::BAR_BYTES);
  if (tid == 0) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    if constexpr (kQ) {
      prefetch_tmap(&tmKq);
      prefetch_tmap(&tmVq);
    }
  }

  // ---- page prefix over (b, h), identical in every CTA, and the last (b, h) with pages
  __shared__ int s_last_bh;
  {
    __shared__ int wsum[kWarps];
    __shared__ int wlast[kWarps];
    __shared__ int carry;
    if (tid == 0) {
      carry = 0;
      s_last_bh = 0;
    }
    __syncthreads();
    for (int base = 0; base < BH; base += kThreads) {
      const int bh = base + tid;
      int np = bh < BH ? (clamp_count(p.count, bh, p.max_pages) + kPage - 1) / kPage : 0;
      if constexpr (kQ) np += bh < BH ? (clamp_count(p.count_q, bh, p.max_pages_q) + kPage - 1) / kPage : 0;
      int incl = np;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int wl = __reduce_max_sync(0xffffffffu, np > 0 ? bh : -1);
      if (lane == 31) wsum[warp] = incl;
      if (lane == 0) wlast[warp] = wl;
      __syncthreads();
      int before = carry;
      for (int w = 0; w < warp; ++w) before += wsum[w];
      if (bh < BH) pref[bh] = before + incl - np;
      __syncthreads();
      if (tid == 0) {
        int t = 0, lb = s_last_bh;
        for (int w = 0; w < kWarps; ++w) {
          t += wsum[w];
          lb = max(lb, wlast[w]);
        }
        carry += t;
        s_last_bh = lb;
      }
      __syncthreads();
    }
    if (tid == 0) pref[BH] = carry;
    __syncthreads();
  }
  const int NP = pref[BH];

  // ---- (b, h) without pages: zero output rows
  for (int bh = blockIdx.x; bh < BH; bh += gridDim.x) {
    if (pref[bh + 1] == pref[bh]) {
      for (int i = tid; i < G * D; i += kThreads) p.out[static_cast<size_t>(bh) * G * D + i] = 0.f;
      if (p.lse != nullptr && tid < G) p.lse[static_cast<size_t>(bh) * G + tid] = -INFINITY;
    }
  }
  if (NP == 0) return;

  // ---- this warp's slice of the global page list
  // slices of at least min_pages pages (fewer pieces to merge on small
  // problems); every one of the first NW slices is non-empty
  const int nw_all = gridDim.x * kWarps;
  const int min_pages = NP >= 64 * BH ? kMinPagesLong : kMinPagesShort;
  const int NW = max(1, min(nw_all, NP / min_pages));
  const int gw = warp * gridDim.x + blockIdx.x;  // slices go round-robin over the CTAs (all SMs busy)
  if (gw >= NW) return;
  const int last_bh = s_last_bh;  // (b, h) of the last page
  const int64_t c_end = 2 * static_cast<int64_t>(NP - 1) + static_cast<int64_t>(kBoundaryCost) * last_bh + 1;
  // first page of slice w: the first page whose cost reaches ceil(w * c_end / NW); a_out: the (b, h) searched
  // to (that page's, or one before it with no pages)
  auto slice_start = [&](int w, int& a_out) {
    const int64_t T = (static_cast<int64_t>(w) * c_end + NW - 1) / NW;
    auto maxc = [&](int k) {
      return 2 * static_cast<int64_t>(pref[k + 1] - 1) + static_cast<int64_t>(kBoundaryCost) * k;
    };
    if (maxc(BH - 1) < T) return NP;
    int a = 0, b = BH - 1;
    while (a < b) {
      const int mid = (a + b) >> 1;
      if (maxc(mid) >= T) b = mid; else a = mid + 1;
    }
    const int64_t g = (T - static_cast<int64_t>(kBoundaryCost) * a + 1) / 2;
    a_out = a;
    return static_cast<int>(min(static_cast<int64_t>(NP), max(static_cast<int64_t>(pref[a]), g)));
  };
  // the slice's two ends on two lanes at once (a serial chain of integer work each)
  int a_s = 0, r_s = NP;
  if (lane == 0) r_s = slice_start(gw, a_s);
  if (lane == 1 && gw + 1 < NW) r_s = slice_start(gw + 1, a_s);
  const int r0 = __shfl_sync(0xffffffffu, r_s, 0);
  const int r1 = __shfl_sync(0xffffffffu, r_s, 1);
  if (r1 <= r0) return;  // an empty slice (between two (b, h) with empty ones in between)
  const int n_my = r1 - r0;

  // first (b, h) of the slice: the one whose page range holds page r0 (the start's search ended at it or at
  // a (b, h) with no pages before it)
  int cbh = __shfl_sync(0xffffffffu, a_s, 0);  // consumer cursor
  while (pref[cbh + 1] <= r0) ++cbh;

  // Page ids of the slice, 32 per register: lane j of block b holds the id of
  // slice page 32*b + j. Block b+1 is loaded when issuing enters block b, so
  // every id is in a register about 32 pages before lane 0 needs it.
  // bit j of qb0 / qb1: slice page 32 * blk + j (blk even / odd) is a fp8-tier page
  uint32_t qb0 = 0, qb1 = 0;
  auto load_ids = [&](int blk, uint32_t& qbits) {  // all lanes call this
    const int kk = blk * 32 + lane;
    int id = -1;
    bool isq = false;
    if (kk < n_my) {
      const int g = r0 + kk;
      int a = 0, b = BH - 1;
      while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (pref[mid] <= g) a = mid; else b = mid - 1;
      }
      const int li = g - pref[a];
      if constexpr (kQ) {
        const int na = (clamp_count(p.count, a, p.max_pages) + kPage - 1) / kPage;
        isq = li >= na;
        id = isq ? static_cast<int>(p.page_table_q[static_cast<int64_t>(a) * p.max_pages_q + (li - na)])
                 : static_cast<int>(p.page_table[static_cast<int64_t>(a) * p.max_pages + li]);
      } else {
        id = static_cast<int>(p.page_table[static_cast<int64_t>(a) * p.max_pages + li]);
      }
    }
    if constexpr (kQ) qbits = __ballot_sync(0xffffffffu, isq);
    return id;
  };
  int ids0 = load_ids(0, qb0), ids1 = load_ids(1, qb1);
  auto page_id = [&](int k, bool& isq) {  // all lanes call this
    const int blk = k >> 5;
    const int v = __shfl_sync(0xffffffffu, (blk & 1) ? ids1 : ids0, k & 31);
    isq = kQ && ((((blk & 1) ? qb1 : qb0) >> (k & 31)) & 1u);
    if ((k & 31) == 0 && k > 0) {  // block blk - 1 is done: its register takes block blk + 1
      if (blk & 1) ids0 = load_ids(blk + 1, qb0); else ids1 = load_ids(blk + 1, qb1);
    }
    return v;
  };
  // A page's K and V rows arrive as 16-row x 64-column boxes with the
  // 128-byte swizzle (tensor copies of the pools viewed as [pages x 16, D]);
  // its 16 expire values go to the stage's record with a 1-D bulk copy.
  auto issue = [&](int k, int64_t phys, bool isq) {  // lane 0
    const int st = k % kNst;
    uint8_t* dst = ring + st * C::STAGE_BYTES;
    int32_t* rec = exp_s + st * C::REC_WORDS;
    if (phys < 0 || phys >= (isq ? p.n_pages_cap_q : p.n_pages_cap)) {
      // inconsistent page table: no copy; every slot of the page reads as gone
      record_error(p.status, KVP_ERR_BOUNDS);
      uint4* z = reinterpret_cast<uint4*>(dst);
      for (int i = 0; i < C::STAGE_BYTES / 16; ++i) z[i] = make_uint4(0, 0, 0, 0);
      for (int i = 0; i < C::REC_WORDS; ++i) rec[i] = (isq && i < kPage) ? kNever : 0;
      mbar_arrive(&bars[st]);
      return;
    }
    if (kQ && isq) {
      mbar_arrive_expect_tx(&bars[st], 2 * C::QPAGE_BYTES + C::REC_WORDS * 4);
      tma_load_2d(dst + C::QK_OFF, &tmKq, 0, static_cast<int>(phys) * kPage, &bars[st]);
      tma_load_2d(dst + C::QV_OFF, &tmVq, 0, static_cast<int>(phys) * kPage, &bars[st]);
      bulk_g2s(rec, p.meta_pool + phys * C::REC_WORDS, C::REC_WORDS * 4, &bars[st]);
      return;
    }
    mbar_arrive_expect_tx(&bars[st], C::STAGE_BYTES + kPage * 4);
    const int y = static_cast<int>(phys) * kPage;
#pragma unroll
    for (int j = 0; j < C::NBOX; ++j) {
      tma_load_2d(dst + j * C::BOX_BYTES, &tmK, 64 * j, y, &bars[st]);
      tma_load_2d(dst + C::PAGE_BYTES + j * C::BOX_BYTES, &tmV, 64 * j, y, &bars[st]);
    }
    bulk_g2s(rec, p.expire_pool + phys * kPage, kPage * 4, &bars[st]);
  };
  if (lane == 0) {
    for (int st = 0; st <= kNst; ++st) mbar_init(&bars[st], 1);
    fence_mbar_init();
  }
  __syncwarp();
  for (int k = 0; k < n_my && k < kNst; ++k) {
    bool isq;
    const int pid = page_id(k, isq);
    if (lane == 0) issue(k, pid, isq);
  }
  __syncwarp();

  // ---- query rows of the kv head as mma B fragments (bf16, unscaled): thread
  // (g, t) = (lane / 4, lane % 4) holds head g's dims 16 ks + 2t, +1 and
  // 16 ks + 8 + 2t, +1; heads g >= G are zero
  const int gq = lane >> 2, tq = lane & 3;
  constexpr int KS = D / 16;  // k-steps of the logits, m-tiles of the output
  auto load_qf = [&](int bh, uint32_t (&f)[KS][2]) {
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      f[ks][0] = 0u;
      f[ks][1] = 0u;
    }
    if (gq < G) {
      const uint16_t* qr = p.q + (static_cast<size_t>(bh) * G + gq) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        f[ks][0] = __ldg(reinterpret_cast<const uint32_t*>(qr + 16 * ks + 2 * tq));
        f[ks][1] = __ldg(reinterpret_cast<const uint32_t*>(qr + 16 * ks + 8 + 2 * tq));
      }
    }
  };
  auto next_bh = [&](int bh) {  // next (b, h) that has pages
    int n = bh + 1;
    while (n < BH && pref[n + 1] == pref[n]) ++n;
    return n;
  };
  uint32_t qf[KS][2], qn[KS][2];
  load_qf(cbh, qf);
  int seg_end = min(pref[cbh + 1], r1);
  int cnt = clamp_count(p.count, cbh, p.max_pages);
  int cnt_next = 0;
  int cnt_q = kQ ? clamp_count(p.count_q, cbh, p.max_pages_q) : 0;  // fp8-tier slots of this (b, h)
  int cnt_q_next = 0;
  if (seg_end < r1) {
    load_qf(next_bh(cbh), qn);
    cnt_next = clamp_count(p.count, next_bh(cbh), p.max_pages);
    if constexpr (kQ) cnt_q_next = clamp_count(p.count_q, next_bh(cbh), p.max_pages_q);
  }

  // running state of heads 2t and 2t+1 (this thread's columns of both mma
  // results): max, this thread's share of the sum (its tokens g and g+8),
  // and O^T[dim 16 mt + g (+8)][head 2t (+1)]
  float m2[2] = {-1e30f, -1e30f}, l2[2] = {0.f, 0.f};
  float o[KS][4];
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  const uint32_t ring_u32 = smem_u32(ring);
  const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: the lane's matrix and row within it
  uint32_t merge_par = 0;  // phase of this warp's merge barrier
  bool q_perm = false;     // qf holds this (b, h)'s query in the fp8 pages' order and fp16
  for (int k = 0; k < n_my; ++k) {
    const int g = r0 + k;
    const int st = k % kNst;
    const bool ok = mbar_wait(&bars[st], static_cast<uint32_t>((k / kNst) & 1), nullptr, p.status);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) {
        record_error(p.status, KVP_ERR_TIMEOUT);
        // let the copies this warp issued land before its shared memory can
        // go to another CTA (each wait bounded again)
        for (int kk = k; kk < n_my && kk < k + kNst; ++kk) (void)mbar_wait(&bars[kk % kNst], (kk / kNst) & 1u);
      }
      __syncwarp();
      return;  // outputs of this call are unspecified after a timeout
    }
    const uint32_t kbase = ring_u32 + st * C::STAGE_BYTES;
    const uint32_t vbase = kbase + C::PAGE_BYTES;
    const int32_t* rec = exp_s + st * C::REC_WORDS;
    const int li = g - pref[cbh];
    const int na_cur = (cnt + kPage - 1) / kPage;  // bf16 pages of this (b, h)
    const bool isq = kQ && li >= na_cur;           // a fp8-tier page (uniform in the warp)
    const int slot0 = (isq ? li - na_cur : li) * kPage;

    if (isq && !q_perm) {
      // the first fp8 page of this (b, h). The query fragments go to the K
      // codes' order, as fp16: thread (g, t) takes dims 4t, 4t + 1 (from
      // thread (g, 2t mod 4)) and 4t + 2, 4t + 3 (from (g, 2t + 1 mod 4)) of
      // each k-step, the first of its registers for t < 2, the second after.
      const int s0 = (lane & ~3) | ((2 * tq) & 3), s1 = (lane & ~3) | ((2 * tq + 1) & 3);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint32_t x0 = __shfl_sync(0xffffffffu, qf[ks][0], s0), x1 = __shfl_sync(0xffffffffu, qf[ks][1], s0);
        const uint32_t y0 = __shfl_sync(0xffffffffu, qf[ks][0], s1), y1 = __shfl_sync(0xffffffffu, qf[ks][1], s1);
        qf[ks][0] = bf16x2_to_f16x2(tq < 2 ? x0 : x1);
        qf[ks][1] = bf16x2_to_f16x2(tq < 2 ? y0 : y1);
      }
      // The accumulators go to the V codes' order: rows g and g + 8 of each
      // 16 output dims become dims 2g and 2g + 1, held before by thread
      // (2g mod 8, t) and (2g + 1 mod 8, t), in their first pair for g < 4
      // and their second after.
      const int sa = (((2 * gq) & 7) << 2) | tq, sb = (((2 * gq + 1) & 7) << 2) | tq;
      const bool upper = gq >= 4;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        float x[4], y[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          x[c] = __shfl_sync(0xffffffffu, o[mt][c], sa);
          y[c] = __shfl_sync(0xffffffffu, o[mt][c], sb);
        }
        o[mt][0] = upper ? x[2] : x[0];
        o[mt][1] = upper ? x[3] : x[1];
        o[mt][2] = upper ? y[2] : y[0];
        o[mt][3] = upper ? y[3] : y[1];
      }
      q_perm = true;
    }

    // ---- S = K Q^T: 16 tokens x 8 heads
    float sacc[4] = {0.f, 0.f, 0.f, 0.f};
    if (isq) {
      // A = the K codes in place: matrices 0 / 1 are rows 0-7 / 8-15 of
      // k-step 2 kp's 16 bytes, 2 / 3 of k-step 2 kp + 1's; thread (g, t)
      // receives 4 codes (dims 4t .. 4t + 3) of rows g and g + 8 of each
#pragma unroll
      for (int kp = 0; kp < KS / 2; ++kp) {
        const int r = (mi & 1) * 8 + ri;
        const int chunk = 2 * kp + (mi >> 1);
        const int sw = D == 128 ? (r & 7) : ((r >> 1) & 3);
        const uint32_t addr = kbase + C::QK_OFF + r * D + ((chunk ^ sw) << 4);
        uint32_t c0, c1, c2, c3;
        ldsm_x4(addr, c0, c1, c2, c3);
        mma_f16_16816(sacc, cvt_e4m3x2_to_f16x2(c0), cvt_e4m3x2_to_f16x2(c1), cvt_e4m3x2_to_f16x2(c0 >> 16),
                      cvt_e4m3x2_to_f16x2(c1 >> 16), qf[2 * kp][0], qf[2 * kp][1]);
        mma_f16_16816(sacc, cvt_e4m3x2_to_f16x2(c2), cvt_e4m3x2_to_f16x2(c3), cvt_e4m3x2_to_f16x2(c2 >> 16),
                      cvt_e4m3x2_to_f16x2(c3 >> 16), qf[2 * kp + 1][0], qf[2 * kp + 1][1]);
      }
    } else {
      // A = K from the swizzled boxes
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        // matrices: 0 rows 0-7 / 1 rows 8-15 of the k-step's first 8 dims, 2 / 3 of its second 8
        const int r = (mi & 1) * 8 + ri;
        const int chunk = (ks & 3) * 2 + (mi >> 1);
        const uint32_t addr = kbase + (ks >> 2) * C::BOX_BYTES + r * 128 + ((chunk ^ (r & 7)) << 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(addr, a0, a1, a2, a3);
        mma_bf16_16816(sacc, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
      }
    }

    // ---- V^T fragments: A of the second product, read transposed by ldmatrix
    // from the swizzled boxes. For G <= 4 all of them go to registers now and
    // the stage is handed back before the softmax, so the ring keeps kNst pages
    // in flight; G = 8 needs those registers and reads them after the softmax.
    constexpr bool kEarly = G <= 4;
    auto v_frag = [&](int mt, uint32_t (&a)[4]) {
      // matrices: 0 tokens 0-7 / dims +0, 1 tokens 0-7 / dims +8, 2 tokens 8-15 / +0, 3 tokens 8-15 / +8
      const int r = (mi >> 1) * 8 + ri;
      const int chunk = (mt & 3) * 2 + (mi & 1);
      const uint32_t addr = vbase + (mt >> 2) * C::BOX_BYTES + r * 128 + ((chunk ^ (r & 7)) << 4);
      ldsm_x4_trans(addr, a[0], a[1], a[2], a[3]);
    };
    // a fp8 page: the V fragments of output dims 16 mt .. 16 mt + 15, for mt = 2 mp and 2 mp + 1, from the codes.
    // Matrices: 0 / 1 tokens 0-7 / 8-15 of the 16 codes of dims 32 mp .., 2 / 3 of dims 32 mp + 16 ..; read
    // transposed as 16-bit words, thread (g, t) gets codes (2t, 2g), (2t, 2g + 1), (2t + 1, 2g), (2t + 1, 2g + 1)
    // (token, dim) of each, regrouped by dim into two fp16 pairs
    auto vq_frag2 = [&](int mp, uint32_t (&a0)[4], uint32_t (&a1)[4]) {
      const int r = (mi & 1) * 8 + ri;
      const int chunk = 2 * mp + (mi >> 1);
      const int sw = D == 128 ? (r & 7) : ((r >> 1) & 3);
      const uint32_t addr = kbase + C::QV_OFF + r * D + ((chunk ^ sw) << 4);
      uint32_t w[4];
      ldsm_x4_trans(addr, w[0], w[1], w[2], w[3]);
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = __byte_perm(w[j], 0u, 0x3120);  // [dim 2g: t0, t1 | dim 2g + 1: t0, t1]
      a0[0] = cvt_e4m3x2_to_f16x2(w[0]);
      a0[1] = cvt_e4m3x2_to_f16x2(w[0] >> 16);
      a0[2] = cvt_e4m3x2_to_f16x2(w[1]);
      a0[3] = cvt_e4m3x2_to_f16x2(w[1] >> 16);
      a1[0] = cvt_e4m3x2_to_f16x2(w[2]);
      a1[1] = cvt_e4m3x2_to_f16x2(w[2] >> 16);
      a1[2] = cvt_e4m3x2_to_f16x2(w[3]);
      a1[3] = cvt_e4m3x2_to_f16x2(w[3] >> 16);
    };
    uint32_t va[kEarly ? KS : 1][4];
    const int32_t e0 = rec[gq], e1 = rec[gq + 8];
    const float ks0 = isq ? __int_as_float(rec[kPage + gq]) : 1.f;
    const float ks1 = isq ? __int_as_float(rec[kPage + gq + 8]) : 1.f;
    const float vs0 = isq ? __int_as_float(rec[2 * kPage + gq]) : 1.f;
    const float vs1 = isq ? __int_as_float(rec[2 * kPage + gq + 8]) : 1.f;
    auto issue_next = [&]() {
      __syncwarp();  // every lane is done with the stage
      if (k + kNst < n_my) {
        bool isq_n;
        const int pid = page_id(k + kNst, isq_n);
        if (lane == 0) {
          fence_proxy_async();
          issue(k + kNst, pid, isq_n);
        }
      }
    };
    if constexpr (kEarly) {
      if (isq) {
#pragma unroll
        for (int mp = 0; mp < KS / 2; ++mp) vq_frag2(mp, va[2 * mp], va[2 * mp + 1]);
      } else {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) v_frag(mt, va[mt]);
      }
      issue_next();
    }

    // ---- mask and online softmax (base 2, lazy rescaling) for tokens g, g+8
    bool v0, v1;
    float sc0 = p.qscale, sc1 = p.qscale;
    if (isq) {  // fp8 slots count once now >= start; the K row scales apply to S
      v0 = (slot0 + gq < cnt_q) && (now >= e0);
      v1 = (slot0 + gq + 8 < cnt_q) && (now >= e1);
      sc0 *= ks0;
      sc1 *= ks1;
    } else {
      v0 = (slot0 + gq < cnt) && (now < e0);
      v1 = (slot0 + gq + 8 < cnt) && (now < e1);
    }
    float x[4];
    x[0] = v0 ? sacc[0] * sc0 : -INFINITY;
    x[1] = v0 ? sacc[1] * sc0 : -INFINITY;
    x[2] = v1 ? sacc[2] * sc1 : -INFINITY;
    x[3] = v1 ? sacc[3] * sc1 : -INFINITY;
    const bool grow = x[0] > m2[0] + kLazyRescale || x[2] > m2[0] + kLazyRescale || x[1] > m2[1] + kLazyRescale ||
                      x[3] > m2[1] + kLazyRescale;
    if (__any_sync(0xffffffffu, grow)) {
      float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float n0 = fmaxf(m2[0], mx0), n1 = fmaxf(m2[1], mx1);
      const float al0 = exp2f(m2[0] - n0), al1 = exp2f(m2[1] - n1);
      m2[0] = n0;
      m2[1] = n1;
      l2[0] *= al0;
      l2[1] *= al1;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        o[mt][0] *= al0;
        o[mt][1] *= al1;
        o[mt][2] *= al0;
        o[mt][3] *= al1;
      }
    }
    // p on a bf16 page as a bf16 pair hi + lo (the P.V product keeps about
    // 16 bits of p), on a fp8 page as one fp16 value times the V row scale
    // (11 bits); the sum takes p itself.
    float pf[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) pf[i] = exp2f(x[i] - m2[i & 1]);
    l2[0] += pf[0] + pf[2];
    l2[1] += pf[1] + pf[3];
    // P^T through shared memory: pt_s[hi / lo][head][token]
    const int tok[4] = {gq, gq, gq + 8, gq + 8};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (isq) {
        const float pv = pf[i] * ((i < 2) ? vs0 : vs1);
        pt_s[(2 * tq + (i & 1)) * C::kPtRow + tok[i]] = __half_as_ushort(__float2half_rn(pv));
      } else {
        const __nv_bfloat16 hi = __float2bfloat16_rn(pf[i]);
        const __nv_bfloat16 lo = __float2bfloat16_rn(pf[i] - __bfloat162float(hi));
        pt_s[(2 * tq + (i & 1)) * C::kPtRow + tok[i]] = __bfloat16_as_ushort(hi);
        pt_s[8 * C::kPtRow + (2 * tq + (i & 1)) * C::kPtRow + tok[i]] = __bfloat16_as_ushort(lo);
      }
    }
    __syncwarp();
    const uint32_t pb0 = *reinterpret_cast<const uint32_t*>(pt_s + gq * C::kPtRow + 2 * tq);
    const uint32_t pb1 = *reinterpret_cast<const uint32_t*>(pt_s + gq * C::kPtRow + 8 + 2 * tq);
    uint32_t pl0 = 0u, pl1 = 0u;
    if (!isq) {
      pl0 = *reinterpret_cast<const uint32_t*>(pt_s + 8 * C::kPtRow + gq * C::kPtRow + 2 * tq);
      pl1 = *reinterpret_cast<const uint32_t*>(pt_s + 8 * C::kPtRow + gq * C::kPtRow + 8 + 2 * tq);
    }

    // ---- O^T += V^T P^T
    if (isq) {
#pragma unroll
      for (int mp = 0; mp < KS / 2; ++mp) {
        if constexpr (kEarly) {
          mma_f16_16816(o[2 * mp], va[2 * mp][0], va[2 * mp][1], va[2 * mp][2], va[2 * mp][3], pb0, pb1);
          mma_f16_16816(o[2 * mp + 1], va[2 * mp + 1][0], va[2 * mp + 1][1], va[2 * mp + 1][2], va[2 * mp + 1][3],
                        pb0, pb1);
        } else {
          uint32_t a0[4], a1[4];
          vq_frag2(mp, a0, a1);
          mma_f16_16816(o[2 * mp], a0[0], a0[1], a0[2], a0[3], pb0, pb1);
          mma_f16_16816(o[2 * mp + 1], a1[0], a1[1], a1[2], a1[3], pb0, pb1);
        }
      }
    } else {
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        uint32_t a[4];
        if constexpr (kEarly) {
          a[0] = va[mt][0];
          a[1] = va[mt][1];
          a[2] = va[mt][2];
          a[3] = va[mt][3];
        } else {
          v_frag(mt, a);
        }
        mma_bf16_16816(o[mt], a[0], a[1], a[2], a[3], pb0, pb1);
        mma_bf16_16816(o[mt], a[0], a[1], a[2], a[3], pl0, pl1);
      }
    }
    if constexpr (!kEarly) issue_next();
    __syncwarp();  // pt_s is rewritten by the next page

    // ---- end of a (b, h) segment of this slice
    if (g + 1 == seg_end) {
      float lt0 = l2[0], lt1 = l2[1];
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {  // the sum over this warp's tokens
        lt0 += __shfl_xor_sync(0xffffffffu, lt0, off);
        lt1 += __shfl_xor_sync(0xffffffffu, lt1, off);
      }
      const int h0 = 2 * tq, h1 = 2 * tq + 1;
      // output rows g and g + 8 of each 16 dims: dims g and g + 8, or 2g and 2g + 1 after a fp8 page
      const int da = q_perm ? 2 * gq : gq, db = q_perm ? 2 * gq + 1 : gq + 8;
      const bool whole = pref[cbh] >= r0 && pref[cbh + 1] <= r1;
      if (whole) {
        const float i0 = lt0 > 0.f ? 1.f / lt0 : 0.f, i1 = lt1 > 0.f ? 1.f / lt1 : 0.f;
        float* ob = p.out + static_cast<size_t>(cbh) * G * D;
        if (p.lse != nullptr && gq == 0) {
          if (h0 < G) p.lse[static_cast<size_t>(cbh) * G + h0] = row_lse(m2[0], lt0);
          if (h1 < G) p.lse[static_cast<size_t>(cbh) * G + h1] = row_lse(m2[1], lt1);
        }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          if (h0 < G) {
            ob[h0 * D + 16 * mt + da] = o[mt][0] * i0;
            ob[h0 * D + 16 * mt + db] = o[mt][2] * i0;
          }
          if (h1 < G) {
            ob[h1 * D + 16 * mt + da] = o[mt][1] * i1;
            ob[h1 * D + 16 * mt + db] = o[mt][3] * i1;
          }
        }
      } else {
        const int w_first = slice_of(pref[cbh], cbh, NW, c_end);
        const int w_last = slice_of(pref[cbh + 1] - 1, cbh, NW, c_end);
        const size_t slot = static_cast<size_t>(gw) + cbh;
        float* pa = p.part_acc + slot * G * D;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          if (h0 < G) {
            pa[h0 * D + 16 * mt + da] = o[mt][0];
            pa[h0 * D + 16 * mt + db] = o[mt][2];
          }
          if (h1 < G) {
            pa[h1 * D + 16 * mt + da] = o[mt][1];
            pa[h1 * D + 16 * mt + db] = o[mt][3];
          }
        }
        if (gq == 0) {
          if (h0 < G) {
            p.part_ml[(slot * G + h0) * 2] = m2[0];
            p.part_ml[(slot * G + h0) * 2 + 1] = lt0;
          }
          if (h1 < G) {
            p.part_ml[(slot * G + h1) * 2] = m2[1];
            p.part_ml[(slot * G + h1) * 2 + 1] = lt1;
          }
        }
        fence_acq_rel_gpu();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(&p.pieces[cbh], 1) == (w_last - w_first);
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          constexpr int kAccB = G * D * 4, kMlB = G * 2 * 4;  // bytes of a piece's acc and (m, l)
          // pieces the staged merge takes: as many as the idle ring holds, and at
          // most one per lane (its maxima and weights are held one piece per lane)
          constexpr int kRingPieces = (kNst * C::STAGE_BYTES - 32) / (kAccB + kMlB);
          constexpr int kStaged = kRingPieces < 32 ? kRingPieces : 32;
          const int npc = w_last - w_first + 1;
          if (!merge_pieces<D, G>(p, cbh, npc, static_cast<size_t>(w_first) + cbh, g + 1 == r1 && npc <= kStaged,
                                  ring, &bars[kNst], merge_par, lane))
            return;
        }
      }
      // next segment
      if (g + 1 < r1) {
        cbh = next_bh(cbh);
        seg_end = min(pref[cbh + 1], r1);
        cnt = cnt_next;
        cnt_q = cnt_q_next;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          qf[ks][0] = qn[ks][0];
          qf[ks][1] = qn[ks][1];
        }
        q_perm = false;
        if (seg_end < r1) {
          load_qf(next_bh(cbh), qn);
          cnt_next = clamp_count(p.count, next_bh(cbh), p.max_pages);
          if constexpr (kQ) cnt_q_next = clamp_count(p.count_q, next_bh(cbh), p.max_pages_q);
        }
        m2[0] = m2[1] = -1e30f;
        l2[0] = l2[1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      }
    }
  }
}

// Grid of the persistent kernel on this process's device: one CTA per SM
// times the CTAs an SM holds, computed once (with the shared-memory opt-in).
template <int D, int G, bool kQ>
int attn_grid() {
  static const int grid = [] {
    using C = AttnCfg<D, G>;
    auto kern = attn_decode_kernel<D, G, kQ>;
    int dev = 0, nsm = 0, occ = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess ||
        cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, C::SMEM) != cudaSuccess || occ <= 0)
      return 0;
    return nsm * occ < kMaxCtas ? nsm * occ : kMaxCtas;
  }();
  return grid;
}

template <int D, int G, bool kQ>
kvp_status launch_attn(const AttnParams& p, int grid_limit, cudaStream_t st) {
  using C = AttnCfg<D, G>;
  int grid = attn_grid<D, G, kQ>();
  if (grid <= 0) return KVP_ERR_CUDA;
  if (grid_limit > 0 && grid > grid_limit) grid = grid_limit;
  if (launch_pdl(attn_decode_kernel<D, G, kQ>, dim3(grid), dim3(kThreads), C::SMEM, st, p) != cudaSuccess)
    return KVP_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

template <int D, int G, bool kQ>
int attn_mma_grid() {
  static const int grid = [] {
    using C = MmaCfg<D>;
    auto kern = attn_mma_kernel<D, G, kQ>;
    int dev = 0, nsm = 0, occ = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess ||
        cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, C::SMEM) != cudaSuccess || occ <= 0)
      return 0;
    return nsm * occ < kMaxCtas ? nsm * occ : kMaxCtas;
  }();
  return grid;
}

template <int D, int G, bool kQ>
kvp_status launch_attn_mma(const AttnParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           const CUtensorMap& tmKq, const CUtensorMap& tmVq, int grid_limit, cudaStream_t st) {
  using C = MmaCfg<D>;
  int grid = attn_mma_grid<D, G, kQ>();
  if (grid <= 0) return KVP_ERR_CUDA;
  if (grid_limit > 0 && grid > grid_limit) grid = grid_limit;
  if (launch_pdl(attn_mma_kernel<D, G, kQ>, dim3(grid), dim3(kThreads), C::SMEM, st, p, tmK, tmV, tmKq, tmVq) !=
      cudaSuccess)
    return KVP_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

template <int D, bool kQ>
kvp_status dispatch_mma(const AttnParams& p, int G, int grid_limit, cudaStream_t st) {
  CUtensorMap tmK, tmV;
  const int64_t rows = static_cast<int64_t>(p.n_pages_cap) * kPage;
  if (!make_tmap_bf16(&tmK, p.k_pool, rows, D, D, kPage, 64) || !make_tmap_bf16(&tmV, p.v_pool, rows, D, D, kPage, 64))
    return KVP_ERR_CUDA;
  // the fp8 tier's K and V codes, 16 rows a box (a pool with no pages takes no copy: the bf16 maps stand in)
  CUtensorMap tmKq = tmK, tmVq = tmV;
  const int64_t rows_q = static_cast<int64_t>(p.n_pages_cap_q) * kPage;
  if (kQ && rows_q > 0 &&
      (!make_tmap_u8_rows(&tmKq, p.kq_pool, rows_q, D, kPage) || !make_tmap_u8_rows(&tmVq, p.vq_pool, rows_q, D, kPage)))
    return KVP_ERR_CUDA;
  if constexpr (kQ) {
    if (G == 1) return launch_attn_mma<D, 1, kQ>(p, tmK, tmV, tmKq, tmVq, grid_limit, st);
    if (G == 2) return launch_attn_mma<D, 2, kQ>(p, tmK, tmV, tmKq, tmVq, grid_limit, st);
  }
  if (G == 4) return launch_attn_mma<D, 4, kQ>(p, tmK, tmV, tmKq, tmVq, grid_limit, st);
  if (G != 8) return KVP_ERR_UNSUPPORTED;
  return launch_attn_mma<D, 8, kQ>(p, tmK, tmV, tmKq, tmVq, grid_limit, st);
}

template <int D, bool kQ>
kvp_status dispatch_g(const AttnParams& p, int G, int grid_limit, cudaStream_t st) {
  switch (G) {
    case 1: return launch_attn<D, 1, kQ>(p, grid_limit, st);
    case 2: return launch_attn<D, 2, kQ>(p, grid_limit, st);
    case 4: return launch_attn<D, 4, kQ>(p, grid_limit, st);
    case 8: return launch_attn<D, 8, kQ>(p, grid_limit, st);
    default: return KVP_ERR_UNSUPPORTED;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// workspace: arrival counters [BH], then part_ml [slots, G, 2], then
// part_acc [slots, G, D], each region starting on 16 bytes; slots = warps of
// the largest grid + BH (a slice's piece of (b, h) goes to slot warp + b*H + h).
size_t round16(size_t n) { return (n + 15) / 16 * 16; }
size_t ws_counter_bytes(int BH) { return round16(static_cast<size_t>(BH) * 4); }
size_t ws_slots(int BH) { return static_cast<size_t>(kMaxCtas) * kWarps + BH; }
size_t ws_ml_bytes(int BH, int G) { return round16(ws_slots(BH) * G * 2 * sizeof(float)); }

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" size_t kvp_decode_attn_workspace_bytes(int batch, int n_q_heads, int n_kv_heads, int head_dim) {
  if (batch <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || n_q_heads % n_kv_heads) return 0;
  const int BH = batch * n_kv_heads;
  const int G = n_q_heads / n_kv_heads;
  return ws_counter_bytes(BH) + ws_ml_bytes(BH, G) + ws_slots(BH) * G * head_dim * sizeof(float);
}

namespace {
struct QuantTier {
  const void* kq_pool;
  const void* vq_pool;
  const int32_t* meta_pool;
  int n_pages_cap;
  const int32_t* page_table;
  int max_pages;
  const int32_t* count;
};

// Two-tier calls from this many query heads per kv head on go to the tensor-core kernel (the CUDA-core kernel
// keeps any below it); 1: all of them.
#ifndef KVP_TWO_TIER_MMA_FROM
#define KVP_TWO_TIER_MMA_FROM 1
#endif
constexpr int kTwoTierMmaFrom = KVP_TWO_TIER_MMA_FROM;
// One-tier calls from this many query heads per kv head on go to the tensor-core kernel.
#ifndef KVP_ONE_TIER_MMA_FROM
#define KVP_ONE_TIER_MMA_FROM 4
#endif
constexpr int kOneTierMmaFrom = KVP_ONE_TIER_MMA_FROM;

kvp_status decode_attn_impl(int batch, int n_q_heads, int n_kv_heads, int head_dim, const void* q, const void* k_pool,
                            const void* v_pool, const int32_t* expire_pool, int n_pages_cap,
                            const int32_t* page_table, int max_pages, const int32_t* count, const QuantTier* qt,
                            int now, const int32_t* now_dev, float scale, float* out, float* lse, int grid_limit,
                            void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
  if (batch <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || max_pages < 0 || grid_limit < 0 || n_pages_cap < 0)
    return KVP_ERR_INVALID;
  if (n_q_heads % n_kv_heads != 0) return KVP_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(now_dev) & 3u) != 0) return KVP_ERR_ALIGN;
  if (static_cast<int64_t>(max_pages) * kPage > 0x7fffffff) return KVP_ERR_UNSUPPORTED;
  const int G = n_q_heads / n_kv_heads;
  if (head_dim != 64 && head_dim != 128) return KVP_ERR_UNSUPPORTED;
  if (G != 1 && G != 2 && G != 4 && G != 8) return KVP_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(batch) * n_kv_heads > kMaxBH) return KVP_ERR_UNSUPPORTED;
  if (!(scale >= 0.f)) return KVP_ERR_INVALID;
  if (q == nullptr || k_pool == nullptr || v_pool == nullptr || expire_pool == nullptr || page_table == nullptr ||
      count == nullptr || out == nullptr)
    return KVP_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(expire_pool) || !aligned16(out))
    return KVP_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return KVP_ERR_ALIGN;
  if (qt != nullptr) {
    if (qt->max_pages < 0 || qt->n_pages_cap < 0) return KVP_ERR_INVALID;
    if (static_cast<int64_t>(qt->max_pages) * kPage > 0x7fffffff) return KVP_ERR_UNSUPPORTED;
    if (qt->kq_pool == nullptr || qt->vq_pool == nullptr || qt->meta_pool == nullptr || qt->page_table == nullptr ||
        qt->count == nullptr)
      return KVP_ERR_INVALID;
    if (!aligned16(qt->kq_pool) || !aligned16(qt->vq_pool) || !aligned16(qt->meta_pool)) return KVP_ERR_ALIGN;
  }
  const size_t need = kvp_decode_attn_workspace_bytes(batch, n_q_heads, n_kv_heads, head_dim);
  if (workspace == nullptr || workspace_bytes < need) return KVP_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KVP_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int BH = batch * n_kv_heads;
  const float sc = scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(head_dim));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* pieces = reinterpret_cast<int32_t*>(ws);
  float* part_ml = reinterpret_cast<float*>(ws + ws_counter_bytes(BH));
  float* part_acc = reinterpret_cast<float*>(ws + ws_counter_bytes(BH) + ws_ml_bytes(BH, G));
  // the counters are zero on entry: zero-filled by the caller before the
  // workspace's first use, and reset by every merge of the previous call
  AttnParams p{static_cast<const uint16_t*>(q),
               static_cast<const uint16_t*>(k_pool),
               static_cast<const uint16_t*>(v_pool),
               expire_pool,
               page_table,
               count,
               batch,
               n_kv_heads,
               n_q_heads,
               max_pages,
               n_pages_cap,
               now,
               sc * 1.4426950408889634f,
               out,
               part_acc,
               part_ml,
               pieces,
               status,
               qt ? static_cast<const uint8_t*>(qt->kq_pool) : nullptr,
               qt ? static_cast<const uint8_t*>(qt->vq_pool) : nullptr,
               qt ? qt->meta_pool : nullptr,
               qt ? qt->page_table : nullptr,
               qt ? qt->count : nullptr,
               qt ? qt->max_pages : 0,
               qt ? qt->n_pages_cap : 0,
               now_dev,
               lse};
  // Eight query heads per kv head go to the tensor-core kernel: with the
  // CUDA-core page math a page takes twice the multiply-adds of G = 4 and the
  // kernel is bound by instruction issue (measured on a GB300, Llama-3-8B
  // cache, keep-all: 192 against 95 us). So do two-tier calls at every G,
  // where the tensor-core kernel reads a fp8 page's codes in place (Llama-3-8B
  // cache at G = 4, a quarter / half / three quarters of the entries in the
  // fp8 tier: 43.0 / 55.3 / 68.5 against 64.6 / 91.0 / 116.8 us; a 65B-shaped
  // MHA layer at G = 1: 249 / 347 / 458 against 301 / 446 / 588 us). And
  // one-tier calls from four on (the same cache at G = 4, kept whole / 75 /
  // 87.5 / 96.9 % pruned: 89.4 / 31.9 / 17.1 / 12.4 against 90.9 / 33.2 /
  // 22.8 / 14.8 us); below four the CUDA-core kernel is at the HBM rate kept
  // whole. The tensor-core kernel reads the pools through tensor maps, whose
  // row coordinates stay below 2^31.
  const bool mma = (G >= kOneTierMmaFrom || (qt != nullptr && G >= kTwoTierMmaFrom)) && n_pages_cap > 0 &&
                   static_cast<int64_t>(n_pages_cap) * kPage <= 0x7fffffff;
  if (qt != nullptr) {
    if (mma)
      return head_dim == 128 ? dispatch_mma<128, true>(p, G, grid_limit, st) : dispatch_mma<64, true>(p, G, grid_limit, st);
    return head_dim == 128 ? dispatch_g<128, true>(p, G, grid_limit, st) : dispatch_g<64, true>(p, G, grid_limit, st);
  }
  if (mma)
    return head_dim == 128 ? dispatch_mma<128, false>(p, G, grid_limit, st) : dispatch_mma<64, false>(p, G, grid_limit, st);
  return head_dim == 128 ? dispatch_g<128, false>(p, G, grid_limit, st) : dispatch_g<64, false>(p, G, grid_limit, st);
}
}  // namespace

extern "C" kvp_status kvp_decode_attn(int batch, int n_q_heads, int n_kv_heads, int head_dim, const void* q,
                                      const void* k_pool, const void* v_pool, const int32_t* expire_pool,
                                      int n_pages_cap, const int32_t* page_table, int max_pages,
                                      const int32_t* count, int now, float scale, float* out, int grid_limit,
                                      void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
  return decode_attn_impl(batch, n_q_heads, n_kv_heads, head_dim, q, k_pool, v_pool, expire_pool, n_pages_cap,
                          page_table, max_pages, count, nullptr, now, nullptr, scale, out, nullptr, grid_limit,
                          workspace, workspace_bytes, status, stream);
}

extern "C" kvp_status kvp_decode_attn_lse(int batch, int n_q_heads, int n_kv_heads, int head_dim, const void* q,
                                          const void* k_pool, const void* v_pool, const int32_t* expire_pool,
                                          int n_pages_cap, const int32_t* page_table, int max_pages,
                                          const int32_t* count, int now, float scale, float* out, float* lse,
                                          int grid_limit, void* workspace, size_t workspace_bytes, int32_t* status,
                                          void* stream) {
  if (lse == nullptr) return KVP_ERR_INVALID;
  return decode_attn_impl(batch, n_q_heads, n_kv_heads, head_dim, q, k_pool, v_pool, expire_pool, n_pages_cap,
                          page_table, max_pages, count, nullptr, now, nullptr, scale, out, lse, grid_limit,
                          workspace, workspace_bytes, status, stream);
}

extern "C" kvp_status kvp_decode_attn_devpos(int batch, int n_q_heads, int n_kv_heads, int head_dim, const void* q,
                                             const void* k_pool, const void* v_pool, const int32_t* expire_pool,
                                             int n_pages_cap, const int32_t* page_table, int max_pages,
                                             const int32_t* count, const int32_t* now_dev, float scale, float* out,
                                             int grid_limit, void* workspace, size_t workspace_bytes,
                                             int32_t* status, void* stream) {
  if (now_dev == nullptr) return KVP_ERR_INVALID;
  return decode_attn_impl(batch, n_q_heads, n_kv_heads, head_dim, q, k_pool, v_pool, expire_pool, n_pages_cap,
                          page_table, max_pages, count, nullptr, 0, now_dev, scale, out, nullptr, grid_limit,
                          workspace, workspace_bytes, status, stream);
}

extern "C" kvp_status kvp_decode_attn_two_tier(int batch, int n_q_heads, int n_kv_heads, int head_dim, const void* q,
                                               const void* k_pool, const void* v_pool, const int32_t* expire_pool,
                                               int n_pages_cap, const int32_t* page_table, int max_pages,
                                               const int32_t* count, const void* kq_pool, const void* vq_pool,
                                               const int32_t* meta_pool, int n_pages_cap_q,
                                               const int32_t* page_table_q, int max_pages_q, const int32_t* count_q,
                                               int now, float scale, float* out, int grid_limit, void* workspace,
                                               size_t workspace_bytes, int32_t* status, void* stream) {
  const QuantTier qt{kq_pool, vq_pool, meta_pool, n_pages_cap_q, page_table_q, max_pages_q, count_q};
  return decode_attn_impl(batch, n_q_heads, n_kv_heads, head_dim, q, k_pool, v_pool, expire_pool, n_pages_cap,
                          page_table, max_pages, count, &qt, now, nullptr, scale, out, nullptr, grid_limit,
                          workspace, workspace_bytes, status, stream);
}

// ---------------------------------------------------------------- merging partial attention
// Attention over a set of slots split into parts (each part's output row o_r
// normalised over its own slots, and its log-sum-exp lse_r) is the same
// attention over the union:
//   lse = ln sum_r exp(lse_r),   o = sum_r exp(lse_r - lse) o_r.
// One warp per row, lanes over float4 columns; a part with lse_r = -inf (no
// slots) weighs nothing, and a row with no slots in any part is zero with
// lse -inf.
namespace kvp {
namespace {

constexpr int kMergeWarps = 8;

__global__ void __launch_bounds__(kMergeWarps * 32) attn_merge_kernel(int n_parts, int64_t rows, int d,
                                                                      const float* __restrict__ outs,
                                                                      const float* __restrict__ lses,
                                                                      float* __restrict__ out,
                                                                      float* __restrict__ lse_out) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  float m = -INFINITY;
  for (int r = lane; r < n_parts; r += 32) m = fmaxf(m, lses[static_cast<int64_t>(r) * rows + row]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const int f4 = d / 4;
  float4* orow = reinterpret_cast<float4*>(out + row * d);
  if (m == -INFINITY) {
    for (int c = lane; c < f4; c += 32) orow[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lse_out != nullptr && lane == 0) lse_out[row] = -INFINITY;
    return;
  }
  float w_sum = 0.f;
  for (int r = lane; r < n_parts; r += 32) w_sum += expf(lses[static_cast<int64_t>(r) * rows + row] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) w_sum += __shfl_xor_sync(0xffffffffu, w_sum, o);
  const float inv = 1.f / w_sum;
  for (int c = lane; c < f4; c += 32) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r = 0; r < n_parts; ++r) {
      const float w = expf(lses[static_cast<int64_t>(r) * rows + row] - m) * inv;
      if (w == 0.f) continue;  // an empty part's row is not read
      const float4 v = reinterpret_cast<const float4*>(outs + (static_cast<int64_t>(r) * rows + row) * d)[c];
      a.x = fmaf(w, v.x, a.x);
      a.y = fmaf(w, v.y, a.y);
      a.z = fmaf(w, v.z, a.z);
      a.w = fmaf(w, v.w, a.w);
    }
    orow[c] = a;
  }
  if (lse_out != nullptr && lane == 0) lse_out[row] = m + logf(w_sum);
}

}  // namespace
}  // namespace kvp

extern "C" kvp_status kvp_attn_merge(int n_parts, int64_t rows, int head_dim, const float* outs, const float* lses,
                                     float* out, float* lse_out, void* stream) {
  if (n_parts <= 0 || rows < 0 || head_dim <= 0 || head_dim % 4 != 0) return KVP_ERR_INVALID;
  if (rows == 0) return KVP_OK;
  if (outs == nullptr || lses == nullptr || out == nullptr) return KVP_ERR_INVALID;
  if (!aligned16(outs) || !aligned16(out) || (reinterpret_cast<uintptr_t>(lses) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(lse_out) & 3u) != 0)
    return KVP_ERR_ALIGN;
  const int64_t blocks = (rows + kMergeWarps - 1) / kMergeWarps;
  if (blocks > 0x7fffffff) return KVP_ERR_UNSUPPORTED;
  if (launch_pdl(attn_merge_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kMergeWarps * 32), 0,
                 static_cast<cudaStream_t>(stream), n_parts, rows, head_dim, outs, lses, out, lse_out) != cudaSuccess)
    return KVP_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}
