// kvp_decode_attn_mla: MLA's absorbed decode attention over a pruned latent
// cache (DMS article, "주요 요점" and "앞으로의 전망": the method carries over
// to Multi-Head Latent Attention, whose cache is one latent row per token).
//
// Query head j of batch element b scores slot t with scale * q[b, j] . row_t
// over the whole 576-value row (512 compressed-KV values, then the 64-value
// rotary key) and takes the softmax-weighted sum of the rows' first 512
// values. Every query head reads the same rows, so a page is worth
// 16 tokens x (576 + 512) x 2 flops per head: on CUDA cores that outruns HBM
// from a few heads on, so both products run on the tensor cores. A page lands
// in shared memory as nine 16-row x 64-column boxes with the 128-byte swizzle
// (the mma.sync kernels copy it whole, the pool seen as [rows][9][64]; the
// tcgen05 kernel copies box by box, shared by a cluster) plus its 16 expire
// values. Three kernels, by the number of query heads:
//
//   mla_decode_kernel (up to 32 heads): a CTA of 4 warps per (batch element,
//     16-head tile, slice of its pages), mma.sync m16n8k16:
//       S   = C Q^T     M = 16 tokens, N = 16 heads, K = 576: warp w takes
//                       the 144 values 144w .. 144w + 143; the four partial
//                       products are summed through shared memory (one CTA
//                       barrier per page)
//       softmax         every warp computes the same weights (online, base 2,
//                       lazy rescaling)
//       O^T += Cv^T P^T M = 16 of the 512 compressed values at a time, N = 16
//                       heads, K = 16 tokens: warp w owns values 128w ..
//                       128w + 127 (its A operand read transposed by
//                       ldmatrix); P as a bf16 hi + lo pair
//   mla_tile_kernel (33 to 64 heads): a CTA of 8 warps per (batch element,
//     64-head tile, slice), warp w owning heads 8w .. 8w + 7 outright
//   mla_tc_kernel (65 heads and more): tcgen05 with the query, the logits and
//     an output quarter in tensor memory, four CTAs per (batch element,
//     128-head tile, slice) as a cluster sharing each page's copies
//
// Slices of a unit (batch element, head tile) write their partial states; a
// second kernel, launched right after as the first one's programmatic
// dependent, merges them in fp32 with one CTA per (unit, head), so the
// merge's reads of the partial accumulators are spread over the whole GPU.
#include "kvp_common.cuh"

namespace kvp {
namespace {

constexpr int kDc = KVP_MLA_LATENT_DIM;       // compressed-KV values (the output width)
constexpr int kDr = KVP_MLA_ROPE_DIM;         // rotary-key values
constexpr int kRow = kDc + kDr;               // latent row
constexpr int kHT = 16;                       // query heads per CTA (two n-tiles of 8)
constexpr int kMW = 4;                        // warps per CTA
constexpr int kMThreads = kMW * 32;
constexpr int kRingPages = 4;                 // pages in flight per CTA
constexpr int kMaxSplits = 64;
constexpr int kBoxes = kRow / 64;             // 64-column boxes per page
constexpr int kBoxBytes = kPage * 128;        // 16 rows x 128 bytes
constexpr int kStageBytes = kBoxes * kBoxBytes;
constexpr int kKsW = kRow / 16 / kMW;         // k-steps of the logits per warp
constexpr int kMtW = kDc / 16 / kMW;          // m-tiles of the output per warp
constexpr int kSpartFloats = 32 * 8;          // one warp's partial logits (8 per lane, as two planes of float4)
// A head's row of P^T in shared memory: 16 tokens and 8 halves of padding, so that the stores (lanes
// 4 apart in heads) and the 32-bit reads (8 heads x 4 token pairs) fall on distinct banks
constexpr int kPtRow = 24;
constexpr int kPtHalves = 2 * 2 * 8 * kPtRow;  // one warp's P^T: n-tile x (hi, lo) x 8 heads x kPtRow
// The running maximum is raised only when a logit exceeds it by more than
// this (base 2), so p stays below 2^8 and most pages skip the reduction.
constexpr float kLazyRescale = 8.0f;

constexpr int kRingOff = 0;
constexpr int kRecOff = kRingOff + kRingPages * kStageBytes;
constexpr int kSpartOff = kRecOff + kRingPages * kPage * 4;
constexpr int kPtOff = kSpartOff + 2 * kMW * kSpartFloats * 4;
constexpr int kBarOff = kPtOff + kMW * kPtHalves * 2;
constexpr int kSmemUsed = kBarOff + kRingPages * 8;
constexpr int kSmemBytes = 1024 + kSmemUsed;  // room to align the ring to 1024 bytes

static_assert(kRow % (16 * kMW) == 0 && kDc % (16 * kMW) == 0 && kRow % 64 == 0, "latent row tiling");
static_assert(kKsW == 9 && kMtW == 8, "per-warp shares of the two products");
static_assert(kStageBytes % 1024 == 0, "swizzled boxes start on 1024 bytes");
static_assert(kRecOff % 16 == 0 && kSpartOff % 16 == 0 && kPtOff % 16 == 0 && kBarOff % 8 == 0, "alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct MlaParams {
  const uint16_t* q;          // [B, Hq, kRow]
  const int32_t* expire_pool; // [n_pages_cap, 16]
  const int32_t* page_table;  // [B, max_pages]
  const int32_t* count;       // [B]
  int B, Hq, HT, NS;          // batch, query heads, head tiles, slices per unit
  int TH;                     // query heads per tile: 16, 64 (mla_tile_kernel) or 128 (mla_tc_kernel)
  int max_pages, n_pages_cap, now;
  float qscale;               // scale * log2(e)
  float* out;                 // [B, Hq, kDc]
  float* part_acc;            // [units, NS, TH, kDc]
  float* part_ml;             // [units, NS, TH, 2]
  int32_t* status;
};

// One page into a ring stage, issued by a whole warp with the same arguments
// in every lane: lane 0 copies the page's nine swizzled 16 x 64 boxes with
// one tensor copy (tmap_page views the pool as [rows][9][64], so the page's
// 16 rows land box after box), lane 1 its 16 expire values. A copy
// instruction takes about 100 ns of the SM's copy engine whatever its size,
// so one 18 KB copy per page rather than nine 2 KB ones. An id outside the
// pool (an inconsistent page table) makes no copy: the warp fills the stage
// with zeros and the page's expire values with 0 (every slot gone) and lane
// 0 arrives on the barrier.
__device__ __forceinline__ void issue_page_warp(const void* tmap_page, uint8_t* dst, int32_t* rec, uint64_t* bar,
                                                int phys, const MlaParams& p, int lane) {
  if (phys < 0 || phys >= p.n_pages_cap) {
    if (lane == 0) record_error(p.status, KVP_ERR_BOUNDS);
    uint4* z = reinterpret_cast<uint4*>(dst);
    for (int i = lane; i < kStageBytes / 16; i += 32) z[i] = make_uint4(0, 0, 0, 0);
    if (lane < kPage) rec[lane] = 0;
    fence_proxy_async();  // ordered before a later tensor copy into the stage
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
    return;
  }
  if (lane == 0) mbar_arrive_expect_tx(bar, kStageBytes + kPage * 4);
  __syncwarp();
  if (lane == 0)
    tma_load_3d(dst, tmap_page, 0, phys * kPage, 0, bar);
  else if (lane == 1)
    bulk_g2s(rec, p.expire_pool + static_cast<int64_t>(phys) * kPage, kPage * 4, bar);
}

// The page ids of a slice for a warp that issues its pages in order: lane l
// holds page 32 c + l of the current chunk c and of the next one, so an id
// is a shuffle away and its load was made a chunk earlier (-1 past the slice).
struct SlicePageIds {
  const int32_t* row;  // the batch element's page-table row from the slice's first page
  int n, lane, cur, nxt;
  __device__ int load(int c) const {
    const int k = 32 * c + lane;
    return k < n ? row[k] : -1;
  }
  __device__ void start() {
    cur = load(0);
    nxt = load(1);
  }
  // page k's id; every lane calls it, for k = 0, 1, 2, ... in turn
  __device__ int get(int k) {
    if (k > 0 && (k & 31) == 0) {
      cur = nxt;
      nxt = load((k >> 5) + 1);
    }
    return __shfl_sync(0xffffffffu, cur, k & 31);
  }
};

__global__ void __launch_bounds__(kMThreads, 1) mla_decode_kernel(const MlaParams p,
                                                                  const __grid_constant__ CUtensorMap tmPage) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  pdl_launch_dependents();
  pdl_wait();  // counts, pages and the workspace counters come from the kernels before this one
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // unit (b, ht) and slice s; head tiles vary fastest so that the CTAs that
  // read the same pages run side by side
  const int ht = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.HT));
  const int rest = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.HT));
  const int s = rest % p.NS;
  const int b = rest / p.NS;
  const int unit = b * p.HT + ht;
  const int h_base = ht * kHT;

  uint8_t* ring = smem + kRingOff;
  int32_t* rec_s = reinterpret_cast<int32_t*>(smem + kRecOff);
  float* spart = reinterpret_cast<float*>(smem + kSpartOff);
  uint16_t* pt_s = reinterpret_cast<uint16_t*>(smem + kPtOff) + warp * kPtHalves;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBarOff);

  const int cnt = min(max(p.count[b], 0), p.max_pages * kPage);
  const int np = (cnt + kPage - 1) / kPage;
  const int pg0 = static_cast<int>(static_cast<int64_t>(s) * np / p.NS);
  const int pg1 = static_cast<int>(static_cast<int64_t>(s + 1) * np / p.NS);
  const int n_my = pg1 - pg0;

  if (tid == 0) {
    prefetch_tmap(&tmPage);
    for (int st = 0; st < kRingPages; ++st) mbar_init(&bars[st], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Page k of the slice into stage k % kRingPages (warp 0, every lane).
  SlicePageIds ids{p.page_table + static_cast<int64_t>(b) * p.max_pages + pg0, n_my, lane, -1, -1};
  auto issue = [&](int k) {
    const int st = k % kRingPages;
    issue_page_warp(&tmPage, ring + st * kStageBytes, rec_s + st * kPage, &bars[st], ids.get(k), p, lane);
  };
  int issued = 0;  // pages issued so far (warp 0's count)
  if (warp == 0) {
    ids.start();
    for (; issued < n_my && issued < kRingPages; ++issued) issue(issued);
  }

  // ---- query rows of the tile as mma B fragments: thread (g, t) = (lane / 4,
  // lane % 4) holds, for k-step ks of this warp and n-tile nt, head
  // 8 nt + g's values 16 ks + 2t, +1 and 16 ks + 8 + 2t, +1 (zero past Hq)
  const int gq = lane >> 2, tq = lane & 3;
  uint32_t qf[kKsW][2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int h = h_base + 8 * nt + gq;
    const uint16_t* qr = p.q + (static_cast<int64_t>(b) * p.Hq + h) * kRow;
#pragma unroll
    for (int i = 0; i < kKsW; ++i) {
      const int ks = warp * kKsW + i;
      qf[i][nt][0] = h < p.Hq ? __ldg(reinterpret_cast<const uint32_t*>(qr + 16 * ks + 2 * tq)) : 0u;
      qf[i][nt][1] = h < p.Hq ? __ldg(reinterpret_cast<const uint32_t*>(qr + 16 * ks + 8 + 2 * tq)) : 0u;
    }
  }

  // running state of heads 8 nt + 2t and 8 nt + 2t + 1 (this thread's columns
  // of both products): max, this thread's share of the sum (tokens g, g + 8),
  // and O^T[value 16 mt + g (+8)][head 8 nt + 2t (+1)] for this warp's m-tiles
  float m2[2][2], l2[2][2];
  float o[kMtW][2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    m2[nt][0] = m2[nt][1] = -1e30f;
    l2[nt][0] = l2[nt][1] = 0.f;
#pragma unroll
    for (int j = 0; j < kMtW; ++j) o[j][nt][0] = o[j][nt][1] = o[j][nt][2] = o[j][nt][3] = 0.f;
  }

  const uint32_t ring_u32 = smem_u32(ring);
  const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: the lane's matrix and row within it
  for (int k = 0; k < n_my; ++k) {
    const int st = k % kRingPages;
    const bool ok = mbar_wait(&bars[st], static_cast<uint32_t>((k / kRingPages) & 1), nullptr, p.status);
    const uint32_t base = ring_u32 + st * kStageBytes;

    // ---- partial logits over this warp's 144 values
    // two independent partial sums per n-tile (even and odd k-steps), so the products do not form one chain
    float sacc2[2][2][4] = {};
#pragma unroll
    for (int i = 0; i < kKsW; ++i) {
      const int ks = warp * kKsW + i;
      // matrices: 0 rows 0-7 / 1 rows 8-15 of the k-step's first 8 values, 2 / 3 of its second 8
      const int r = (mi & 1) * 8 + ri;
      const int chunk = (ks & 3) * 2 + (mi >> 1);
      const uint32_t addr = base + (ks >> 2) * kBoxBytes + r * 128 + ((chunk ^ (r & 7)) << 4);
      uint32_t a0, a1, a2, a3;
      ldsm_x4(addr, a0, a1, a2, a3);
      mma_bf16_16816(sacc2[0][i & 1], a0, a1, a2, a3, qf[i][0][0], qf[i][0][1]);
      mma_bf16_16816(sacc2[1][i & 1], a0, a1, a2, a3, qf[i][1][0], qf[i][1][1]);
    }
    float sacc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[nt][e] = sacc2[nt][0][e] + sacc2[nt][1][e];
    float* sp = spart + (k & 1) * (kMW * kSpartFloats);  // two buffers: page k + 1 writes the other
    // plane nt holds every lane's float4 of n-tile nt side by side: a warp's access is 512 contiguous bytes
    *reinterpret_cast<float4*>(sp + warp * kSpartFloats + lane * 4) =
        make_float4(sacc[0][0], sacc[0][1], sacc[0][2], sacc[0][3]);
    *reinterpret_cast<float4*>(sp + warp * kSpartFloats + 128 + lane * 4) =
        make_float4(sacc[1][0], sacc[1][1], sacc[1][2], sacc[1][3]);
    // every partial is written; every warp is done with page k - 1's stage
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        record_error(p.status, KVP_ERR_TIMEOUT);
        // the copies already issued land before the CTA's shared memory is
        // released (each wait bounded again)
        for (int kk = k; kk < issued; ++kk) (void)mbar_wait(&bars[kk % kRingPages], (kk / kRingPages) & 1u);
      }
      return;  // outputs of this call are unspecified after a timeout
    }
    if (warp == 0 && k >= 1 && issued < n_my) {  // page k - 1's stage takes the next page
      if (lane == 0) fence_proxy_async();
      __syncwarp();
      issue(issued);
      ++issued;
    }

    // ---- full logits (the four partials in a fixed order, so every warp
    // holds the same values), mask, online softmax
    float sv[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int w = 0; w < kMW; ++w) {
      const float4 u0 = *reinterpret_cast<const float4*>(sp + w * kSpartFloats + lane * 4);
      const float4 u1 = *reinterpret_cast<const float4*>(sp + w * kSpartFloats + 128 + lane * 4);
      sv[0][0] += u0.x;
      sv[0][1] += u0.y;
      sv[0][2] += u0.z;
      sv[0][3] += u0.w;
      sv[1][0] += u1.x;
      sv[1][1] += u1.y;
      sv[1][2] += u1.z;
      sv[1][3] += u1.w;
    }
    const int32_t* rec = rec_s + st * kPage;
    const int slot0 = (pg0 + k) * kPage;
    const bool v0 = (slot0 + gq < cnt) && (p.now < rec[gq]);
    const bool v1 = (slot0 + gq + 8 < cnt) && (p.now < rec[gq + 8]);
    float x[2][4];
    bool grow = false;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      x[nt][0] = v0 ? sv[nt][0] * p.qscale : -INFINITY;
      x[nt][1] = v0 ? sv[nt][1] * p.qscale : -INFINITY;
      x[nt][2] = v1 ? sv[nt][2] * p.qscale : -INFINITY;
      x[nt][3] = v1 ? sv[nt][3] * p.qscale : -INFINITY;
      grow = grow || x[nt][0] > m2[nt][0] + kLazyRescale || x[nt][2] > m2[nt][0] + kLazyRescale ||
             x[nt][1] > m2[nt][1] + kLazyRescale || x[nt][3] > m2[nt][1] + kLazyRescale;
    }
    if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float mx0 = fmaxf(x[nt][0], x[nt][2]), mx1 = fmaxf(x[nt][1], x[nt][3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float n0 = fmaxf(m2[nt][0], mx0), n1 = fmaxf(m2[nt][1], mx1);
        const float al0 = exp2f(m2[nt][0] - n0), al1 = exp2f(m2[nt][1] - n1);
        m2[nt][0] = n0;
        m2[nt][1] = n1;
        l2[nt][0] *= al0;
        l2[nt][1] *= al1;
#pragma unroll
        for (int j = 0; j < kMtW; ++j) {
          o[j][nt][0] *= al0;
          o[j][nt][1] *= al1;
          o[j][nt][2] *= al0;
          o[j][nt][3] *= al1;
        }
      }
    }
    // p as a bf16 pair hi + lo (the product keeps about 16 bits of p; the
    // sum takes p itself); P^T through this warp's shared memory,
    // pt_s[n-tile][hi / lo][head][token]
    const int tok[4] = {gq, gq, gq + 8, gq + 8};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      float pf[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pf[i] = exp2f(x[nt][i] - m2[nt][i & 1]);
      l2[nt][0] += pf[0] + pf[2];
      l2[nt][1] += pf[1] + pf[3];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(pf[i]);
        const __nv_bfloat16 lo = __float2bfloat16_rn(pf[i] - __bfloat162float(hi));
        const int hrow = 2 * tq + (i & 1);
        pt_s[((nt * 2 + 0) * 8 + hrow) * kPtRow + tok[i]] = __bfloat16_as_ushort(hi);
        pt_s[((nt * 2 + 1) * 8 + hrow) * kPtRow + tok[i]] = __bfloat16_as_ushort(lo);
      }
    }
    __syncwarp();
    // B fragments of P^T (k = tokens, n = heads): head 8 nt + g, tokens 2t, +1 and 2t + 8, +9
    uint32_t pb[2][2], pl[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint16_t* hi_row = pt_s + ((nt * 2 + 0) * 8 + gq) * kPtRow;
      const uint16_t* lo_row = pt_s + ((nt * 2 + 1) * 8 + gq) * kPtRow;
      pb[nt][0] = *reinterpret_cast<const uint32_t*>(hi_row + 2 * tq);
      pb[nt][1] = *reinterpret_cast<const uint32_t*>(hi_row + 8 + 2 * tq);
      pl[nt][0] = *reinterpret_cast<const uint32_t*>(lo_row + 2 * tq);
      pl[nt][1] = *reinterpret_cast<const uint32_t*>(lo_row + 8 + 2 * tq);
    }

    // ---- O^T += Cv^T P^T over this warp's 128 compressed values
#pragma unroll
    for (int j = 0; j < kMtW; ++j) {
      const int mt = warp * kMtW + j;
      // matrices: 0 tokens 0-7 / values +0, 1 tokens 0-7 / +8, 2 tokens 8-15 / +0, 3 tokens 8-15 / +8
      const int r = (mi >> 1) * 8 + ri;
      const int chunk = (mt & 3) * 2 + (mi & 1);
      const uint32_t addr = base + (mt >> 2) * kBoxBytes + r * 128 + ((chunk ^ (r & 7)) << 4);
      uint32_t a0, a1, a2, a3;
      ldsm_x4_trans(addr, a0, a1, a2, a3);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        mma_bf16_16816(o[j][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
        mma_bf16_16816(o[j][nt], a0, a1, a2, a3, pl[nt][0], pl[nt][1]);
      }
    }
    __syncwarp();  // pt_s is rewritten by the next page
  }

  // ---- this slice's state: the sums over the tokens of all lanes
  float lt[2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float v = l2[nt][c];
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      lt[nt][c] = v;
    }
  }
  if (p.NS == 1) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int h = h_base + 8 * nt + 2 * tq + c;
        if (h >= p.Hq) continue;
        const float inv = lt[nt][c] > 0.f ? 1.f / lt[nt][c] : 0.f;
        float* orow = p.out + (static_cast<int64_t>(b) * p.Hq + h) * kDc;
#pragma unroll
        for (int j = 0; j < kMtW; ++j) {
          const int d0 = 16 * (warp * kMtW + j) + gq;
          orow[d0] = o[j][nt][c] * inv;
          orow[d0 + 8] = o[j][nt][2 + c] * inv;
        }
      }
    }
    return;
  }

  const int64_t slot = static_cast<int64_t>(unit) * p.NS + s;
  if (n_my > 0) {  // an empty slice leaves its accumulator unwritten: its sum is 0 and the merge skips it
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int hl = 8 * nt + 2 * tq + c;
        float* pa = p.part_acc + (slot * kHT + hl) * kDc;
#pragma unroll
        for (int j = 0; j < kMtW; ++j) {
          const int d0 = 16 * (warp * kMtW + j) + gq;
          pa[d0] = o[j][nt][c];
          pa[d0 + 8] = o[j][nt][2 + c];
        }
      }
    }
  }
  if (warp == 0 && gq == 0) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int hl = 8 * nt + 2 * tq + c;
        p.part_ml[(slot * kHT + hl) * 2] = m2[nt][c];
        p.part_ml[(slot * kHT + hl) * 2 + 1] = lt[nt][c];
      }
    }
  }
}

// Merge of the slices of every unit: CTA (unit, hl) takes head TH * tile + hl,
// thread c the float4 c of its 512 output values. The slices' (m, l) give
// the weights exp2(m - M) (an empty slice, l = 0, has none and its
// accumulator is not read), then the accumulators are summed with all of a
// batch of slices' loads in flight.
__global__ void __launch_bounds__(kDc / 4) mla_merge_kernel(const MlaParams p) {
  __shared__ float w_s[kMaxSplits];
  __shared__ float il_s;
  pdl_launch_dependents();
  pdl_wait();  // every slice's partial state is written
  const int unit = static_cast<int>(blockIdx.x / p.TH), hl = static_cast<int>(blockIdx.x % p.TH);
  const int b = unit / p.HT, h = (unit % p.HT) * p.TH + hl;
  if (h >= p.Hq) return;
  const int c4 = threadIdx.x;
  const float* ml = p.part_ml + static_cast<int64_t>(unit) * p.NS * p.TH * 2;
  if (c4 < 32) {
    float M = -INFINITY;
    for (int sl = c4; sl < p.NS; sl += 32) {
      const float l = __ldcg(ml + (sl * p.TH + hl) * 2 + 1);
      if (l > 0.f) M = fmaxf(M, __ldcg(ml + (sl * p.TH + hl) * 2));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int sl = c4; sl < p.NS; sl += 32) {
      const float l = __ldcg(ml + (sl * p.TH + hl) * 2 + 1);
      const float w = l > 0.f ? exp2f(__ldcg(ml + (sl * p.TH + hl) * 2) - M) : 0.f;
      w_s[sl] = w;
      L += w * l;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (c4 == 0) il_s = L > 0.f ? 1.f / L : 0.f;
  }
  __syncthreads();
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* acc = reinterpret_cast<const float4*>(p.part_acc + static_cast<int64_t>(unit) * p.NS * p.TH * kDc);
  constexpr int kBatch = 8;
  for (int s0 = 0; s0 < p.NS; s0 += kBatch) {
    float4 v[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int sl = s0 + j;
      v[j] = (sl < p.NS && w_s[sl] != 0.f) ? __ldcg(acc + (static_cast<int64_t>(sl) * p.TH + hl) * (kDc / 4) + c4)
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const float w = s0 + j < p.NS ? w_s[s0 + j] : 0.f;
      a.x = fmaf(w, v[j].x, a.x);
      a.y = fmaf(w, v[j].y, a.y);
      a.z = fmaf(w, v[j].z, a.z);
      a.w = fmaf(w, v[j].w, a.w);
    }
  }
  const float il = il_s;
  reinterpret_cast<float4*>(p.out + (static_cast<int64_t>(b) * p.Hq + h) * kDc)[c4] =
      make_float4(a.x * il, a.y * il, a.z * il, a.w * il);
}


// ---------------------------------------------------------------- 64-head tiles
// From 33 query heads on: a CTA takes 64 query heads of one batch element and
// one slice of its pages with eight warps, warp w owning query heads
// 8w .. 8w + 7 of the tile outright. The slice's pages stream through a ring
// of kTRing stages (the nine swizzled boxes and the 16 expire values of a
// page per stage); each stage has a full barrier (the copies' bytes) and an
// empty barrier (one arrival per warp with heads). Lane 0 of warp 0 fills the
// ring: the first kTRing pages up front, then, after its warp's page k, page
// k - 1 + kTRing into the stage of page k - 1, which the other warps have
// usually left by then. Warps meet only at the ring; the page loop has no CTA
// barrier. Per page, warp w computes
//   S   = C Q^T     M = 16 tokens, N = its 8 heads, K = all 576 values
//                   (the query rows from shared memory, ldmatrix), four
//                   independent partial sums over the k-steps
//   softmax         online, base 2, lazy rescaling, for heads 2t and 2t + 1
//                   of the thread (as in the one-tier tensor-core attention)
//   O^T += Cv^T P^T M = 16 of the 512 values at a time (32 m-tiles), N = 8
//                   heads, K = the page's 16 tokens; P as bf16 hi + lo
// One page load serves 64 heads. The SM's registers sit in four files of 16K,
// one per scheduler: eight warps (two per file) may use up to 255 registers
// each, and the 128 output accumulators of a thread need most of them; a
// ninth, copy-only warp would put three warps on one file and cap every
// thread at 168.
constexpr int kTHeads = 64;                          // query heads per CTA
constexpr int kTWarps = kTHeads / 8;                 // 8 heads each
constexpr int kTThreads = kTWarps * 32;
constexpr int kTRing = 6;                            // ring stages: up to 5 pages ahead of warp 0
constexpr int kQRowBytes = kRow * 2 + 16;            // a query row in shared memory, padded (conflict-free ldmatrix)
constexpr int kTRingOff = 0;
constexpr int kTRecOff = kTRingOff + kTRing * kStageBytes;
constexpr int kTQOff = kTRecOff + kTRing * kPage * 4;
constexpr int kTPtOff = kTQOff + kTHeads * kQRowBytes;
constexpr int kTBarOff = kTPtOff + kTWarps * 2 * 8 * kPtRow * 2;
constexpr int kTSmemUsed = kTBarOff + 2 * kTRing * 8 + 16;
constexpr int kTSmemBytes = 1024 + kTSmemUsed;
static_assert(kTRecOff % 16 == 0 && kTQOff % 16 == 0 && kTPtOff % 16 == 0 && kTBarOff % 8 == 0, "alignment");
static_assert(kTSmemBytes <= 232448, "shared memory budget");

__global__ void __launch_bounds__(kTThreads, 1) mla_tile_kernel(const MlaParams p,
                                                                const __grid_constant__ CUtensorMap tmPage) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  pdl_launch_dependents();
  pdl_wait();  // counts and pages come from the kernels before this one
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ht = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.HT));
  const int rest = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.HT));
  const int s = rest % p.NS;
  const int b = rest / p.NS;
  const int unit = b * p.HT + ht;
  const int h_base = ht * kTHeads;
  const int n_act = min(kTWarps, (p.Hq - h_base + 7) / 8);  // warps with heads (at least warp 0)

  uint8_t* ring = smem + kTRingOff;
  int32_t* rec_s = reinterpret_cast<int32_t*>(smem + kTRecOff);
  uint8_t* q_s = smem + kTQOff;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kTBarOff);
  uint64_t* empty = full + kTRing;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kTRing);

  const int cnt = min(max(p.count[b], 0), p.max_pages * kPage);
  const int np = (cnt + kPage - 1) / kPage;
  const int pg0 = static_cast<int>(static_cast<int64_t>(s) * np / p.NS);
  const int pg1 = static_cast<int>(static_cast<int64_t>(s + 1) * np / p.NS);
  const int n_my = pg1 - pg0;

  // ---- the tile's query rows into shared memory (zero past Hq)
  for (int i = tid; i < kTHeads * (kRow / 8); i += kTThreads) {
    const int hl = i / (kRow / 8), c = i - hl * (kRow / 8);
    const int h = h_base + hl;
    const uint4 v = h < p.Hq ? __ldg(reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(b) * p.Hq + h) * kRow) + c)
                             : make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(q_s + hl * kQRowBytes + c * 16) = v;
  }
  if (tid == 0) {
    prefetch_tmap(&tmPage);
    for (int st = 0; st < kTRing; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], n_act);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (warp >= n_act) return;

  // page k of the slice into stage k % kTRing (warp 0, every lane; the stage is free)
  const bool filler = warp == 0;
  SlicePageIds ids{p.page_table + static_cast<int64_t>(b) * p.max_pages + pg0, n_my, lane, -1, -1};
  auto issue = [&](int k) {
    const int st = k % kTRing;
    issue_page_warp(&tmPage, ring + st * kStageBytes, rec_s + st * kPage, &full[st], ids.get(k), p, lane);
  };
  int n_issued = 0;
  if (filler) {
    ids.start();
    for (; n_issued < min(kTRing, n_my); ++n_issued) issue(n_issued);
  }

  const int gq = lane >> 2, tq = lane & 3;
  const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: the lane's matrix and row within it
  // query B fragments of two k-steps per ldmatrix.x4: matrix m = (k-step ks + m / 2, values 8 (m & 1) ..),
  // row = head 8 warp + ri
  const uint32_t qaddr = smem_u32(q_s) + (8 * warp + ri) * kQRowBytes + (mi >> 1) * 32 + (mi & 1) * 16;
  uint16_t* pt_s = reinterpret_cast<uint16_t*>(smem + kTPtOff) + warp * 2 * 8 * kPtRow;
  const uint32_t ring_u32 = smem_u32(ring);

  float m2[2] = {-1e30f, -1e30f}, l2[2] = {0.f, 0.f};
  float o[kDc / 16][4];
#pragma unroll
  for (int mt = 0; mt < kDc / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  for (int k = 0; k < n_my; ++k) {
    const int st = k % kTRing;
    const bool ok = mbar_wait(&full[st], static_cast<uint32_t>((k / kTRing) & 1), abort_flag, p.status);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) {
        record_error(p.status, KVP_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      if (filler && lane == 0) {
        // the copies already issued land before the CTA's shared memory is released (each wait bounded again)
        for (int kk = k; kk < n_issued; ++kk) (void)mbar_wait(&full[kk % kTRing], (kk / kTRing) & 1u);
      }
      return;  // outputs of this call are unspecified after a timeout
    }
    const uint32_t base = ring_u32 + st * kStageBytes;

    // ---- S = C Q^T: 16 tokens x this warp's 8 heads, four partial sums
    float sacc[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) sacc[u][0] = sacc[u][1] = sacc[u][2] = sacc[u][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < kRow / 16; ks += 2) {
      uint32_t b00, b01, b10, b11;
      ldsm_x4(qaddr + ks * 32, b00, b01, b10, b11);
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int kk = ks + h2;
        // matrices: 0 rows 0-7 / 1 rows 8-15 of the k-step's first 8 values, 2 / 3 of its second 8
        const int r = (mi & 1) * 8 + ri;
        const int chunk = (kk & 3) * 2 + (mi >> 1);
        const uint32_t addr = base + (kk >> 2) * kBoxBytes + r * 128 + ((chunk ^ (r & 7)) << 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(addr, a0, a1, a2, a3);
        if (h2 == 0)
          mma_bf16_16816(sacc[kk & 3], a0, a1, a2, a3, b00, b01);
        else
          mma_bf16_16816(sacc[kk & 3], a0, a1, a2, a3, b10, b11);
      }
    }
    float sv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) sv[i] = (sacc[0][i] + sacc[1][i]) + (sacc[2][i] + sacc[3][i]);

    // ---- mask and online softmax (base 2, lazy rescaling) for tokens gq, gq + 8, heads 2tq, 2tq + 1
    const int32_t* rec = rec_s + st * kPage;
    const int slot0 = (pg0 + k) * kPage;
    const bool v0 = (slot0 + gq < cnt) && (p.now < rec[gq]);
    const bool v1 = (slot0 + gq + 8 < cnt) && (p.now < rec[gq + 8]);
    float x[4];
    x[0] = v0 ? sv[0] * p.qscale : -INFINITY;
    x[1] = v0 ? sv[1] * p.qscale : -INFINITY;
    x[2] = v1 ? sv[2] * p.qscale : -INFINITY;
    x[3] = v1 ? sv[3] * p.qscale : -INFINITY;
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
      for (int mt = 0; mt < kDc / 16; ++mt) {
        o[mt][0] *= al0;
        o[mt][1] *= al1;
        o[mt][2] *= al0;
        o[mt][3] *= al1;
      }
    }
    // p as a bf16 pair hi + lo (the product keeps about 16 bits of p; the sum takes p itself);
    // P^T through this warp's shared memory: pt_s[hi / lo][head][token]
    float pf[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) pf[i] = exp2f(x[i] - m2[i & 1]);
    l2[0] += pf[0] + pf[2];
    l2[1] += pf[1] + pf[3];
    const int tok[4] = {gq, gq, gq + 8, gq + 8};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(pf[i]);
      const __nv_bfloat16 lo = __float2bfloat16_rn(pf[i] - __bfloat162float(hi));
      pt_s[(2 * tq + (i & 1)) * kPtRow + tok[i]] = __bfloat16_as_ushort(hi);
      pt_s[8 * kPtRow + (2 * tq + (i & 1)) * kPtRow + tok[i]] = __bfloat16_as_ushort(lo);
    }
    __syncwarp();
    const uint32_t pb0 = *reinterpret_cast<const uint32_t*>(pt_s + gq * kPtRow + 2 * tq);
    const uint32_t pb1 = *reinterpret_cast<const uint32_t*>(pt_s + gq * kPtRow + 8 + 2 * tq);
    const uint32_t pl0 = *reinterpret_cast<const uint32_t*>(pt_s + 8 * kPtRow + gq * kPtRow + 2 * tq);
    const uint32_t pl1 = *reinterpret_cast<const uint32_t*>(pt_s + 8 * kPtRow + gq * kPtRow + 8 + 2 * tq);

    // ---- O^T += Cv^T P^T over all 512 compressed values
#pragma unroll
    for (int mt = 0; mt < kDc / 16; ++mt) {
      // matrices: 0 tokens 0-7 / values +0, 1 tokens 0-7 / +8, 2 tokens 8-15 / +0, 3 tokens 8-15 / +8
      const int r = (mi >> 1) * 8 + ri;
      const int chunk = (mt & 3) * 2 + (mi & 1);
      const uint32_t addr = base + (mt >> 2) * kBoxBytes + r * 128 + ((chunk ^ (r & 7)) << 4);
      uint32_t a0, a1, a2, a3;
      ldsm_x4_trans(addr, a0, a1, a2, a3);
      mma_bf16_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
      mma_bf16_16816(o[mt], a0, a1, a2, a3, pl0, pl1);
    }
    __syncwarp();  // every lane is done with the stage and with pt_s
    if (lane == 0) mbar_arrive(&empty[st]);
    if (filler && n_issued < n_my && k >= 1) {
      // refill the stage of page k - 1 once every warp has left it (lane 0 waits for the warp)
      const int kr = k - 1;
      bool freed = true;
      if (lane == 0)
        freed = mbar_wait(&empty[kr % kTRing], static_cast<uint32_t>((kr / kTRing) & 1), abort_flag, p.status);
      if (__shfl_sync(0xffffffffu, freed ? 1 : 0, 0)) {
        issue(n_issued);
        ++n_issued;
      } else if (lane == 0) {
        record_error(p.status, KVP_ERR_TIMEOUT);
        *abort_flag = 1;  // every warp leaves at its next wait; this one drains its copies there
      }
    }
  }

  // ---- this slice's state: the sums over the tokens of all lanes
  float lt[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    float v = l2[c];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    lt[c] = v;
  }
  const int hl0 = 8 * warp + 2 * tq;  // this thread's heads hl0, hl0 + 1 of the tile
  if (p.NS == 1) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int h = h_base + hl0 + c;
      if (h >= p.Hq) continue;
      const float inv = lt[c] > 0.f ? 1.f / lt[c] : 0.f;
      float* orow = p.out + (static_cast<int64_t>(b) * p.Hq + h) * kDc;
#pragma unroll
      for (int mt = 0; mt < kDc / 16; ++mt) {
        orow[16 * mt + gq] = o[mt][c] * inv;
        orow[16 * mt + gq + 8] = o[mt][2 + c] * inv;
      }
    }
    return;
  }
  const int64_t slot = static_cast<int64_t>(unit) * p.NS + s;
  if (n_my > 0) {  // an empty slice leaves its accumulator unwritten: its sum is 0 and the merge skips it
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float* pa = p.part_acc + (slot * kTHeads + hl0 + c) * kDc;
#pragma unroll
      for (int mt = 0; mt < kDc / 16; ++mt) {
        pa[16 * mt + gq] = o[mt][c];
        pa[16 * mt + gq + 8] = o[mt][2 + c];
      }
    }
  }
  if (gq == 0) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      p.part_ml[(slot * kTHeads + hl0 + c) * 2] = m2[c];
      p.part_ml[(slot * kTHeads + hl0 + c) * 2 + 1] = lt[c];
    }
  }
}

// ---------------------------------------------------------------- tcgen05 tiles
// From kTcFrom query heads on, both products run on the tcgen05 tensor cores
// with the query heads as M = 128 (rows past Hq are zero). Tensor memory has
// 512 columns of 128 lanes and the fp32 output of 128 heads x 512 values
// alone would fill it, so the output is split over a cluster of four CTAs:
// CTA (unit, slice, quarter v) owns output values 128v .. 128v + 127, and all
// four compute the same logits and weights. Per lane = head, tensor memory
// holds
//   columns   0..287  the query row, 576 bf16 (the A operand of S)
//   columns 288..383  S of a block of 96 tokens (6 pages), fp32; P of that
//                     block, 96 bf16, is written over columns 288..335 once
//                     both warps of the row pair have read S
//   columns 384..511  the output quarter, fp32
// Per block of 6 pages:
//   S  = Q C^T      M = 128 heads, N = 96 tokens, K = 576: 36 MMAs, A from
//                   tensor memory, B the block's rows (K-major, 128-byte
//                   swizzle; box j of the 6 pages lies in one 12 KB run)
//   softmax         online, base 2, lazy rescaling of the output in tensor
//                   memory; p rounded to bf16 for the product, the running
//                   sum takes p itself
//   O += P Cv       M = 128, N = 128 values, K = 16 tokens per page: B is the
//                   page's rows read MN-major (values contiguous)
// A tcgen05.mma with N <= 96 takes as long as one with N = 96 (about 48
// cycles, measured), so the logits take 96 tokens a block; that leaves room
// for one S buffer, and S of block i + 1 waits for block i's output product.
// Eight softmax warps: warps w and w + 4 share tensor-memory lane quadrant w
// (rows 32w ..), warp w taking tokens 0..47 of each block and output columns
// 0..63, w + 4 tokens 48..95 and columns 64..127; the pair exchanges its row
// maximum once per block through shared memory behind a 64-thread named
// barrier. Lane 0 of warp 8 issues the MMAs and lane 0 of warp 9 the copies,
// into a ring of two 6-page stages: each CTA of the cluster copies a quarter
// of every page's boxes into all four (TMA multicast), and a stage is reused
// once all four have released it (each CTA's release is a multicast commit).
constexpr int kCHeads = 128;                          // M of both products
constexpr int kCParts = 4;                            // CTAs per (unit, slice), one per output quarter
constexpr int kCVals = kDc / kCParts;                 // output values per CTA
constexpr int kCPages = 6;                            // pages per block
constexpr int kCTok = kCPages * kPage;                // tokens per block: the N of S
constexpr int kCHalf = kCTok / 2;                     // tokens per softmax thread
constexpr int kCBufs = 1;                             // S buffers in tensor memory
constexpr int kCBoxRun = kCPages * kBoxBytes;         // box j of a block's pages
constexpr int kCRing = 2;                             // ring stages (blocks)
constexpr int kCStageBytes = kBoxes * kCBoxRun;
constexpr uint16_t kCAllCtas = (1u << kCParts) - 1;   // the cluster: the four quarter CTAs of a (unit, slice)
constexpr int kCSoftWarps = 8;
constexpr int kCMmaWarp = kCSoftWarps, kCCopyWarp = kCSoftWarps + 1;
constexpr int kCThreads = (kCSoftWarps + 2) * 32;
constexpr uint32_t kTcQCol = 0;
constexpr uint32_t kTcBufCol = kTcQCol + kRow / 2;    // buffer b at kTcBufCol + b * kCTok
constexpr uint32_t kTcPOff = 0;                       // P at the start of its block's buffer
constexpr uint32_t kTcOCol = kTcBufCol + kCBufs * kCTok;
constexpr uint32_t kTcCols = 512;
static_assert(kTcOCol + kCVals <= kTcCols, "tensor-memory plan");
static_assert(kCHalf % 16 == 0 && kCTok % 16 == 0 && kCBoxRun % 1024 == 0 && kCVals % 64 == 0, "block tiling");
constexpr int kCRecOff = kCRing * kCStageBytes;                 // expire values of each stage's pages
constexpr int kCBiasOff = kCRecOff + kCRing * kCTok * 4;        // per softmax warp: its tokens' mask as 0 / -inf
constexpr int kCXchOff = kCBiasOff + kCSoftWarps * kCHalf * 4;  // [2][softmax warp][32]: row maxima, then sums
constexpr int kCBarOff = kCXchOff + 2 * kCSoftWarps * 32 * 4;
constexpr int kCNBars = 2 * kCRing + 7;               // full, empty, s_full[2], p_full[2], o_done[2], fin
constexpr int kCSmemUsed = kCBarOff + kCNBars * 8 + 16;
constexpr int kCSmemBytes = 1024 + kCSmemUsed;
static_assert(kCStageBytes % 1024 == 0 && kCRecOff % 16 == 0 && kCBiasOff % 16 == 0 &&
                  kCXchOff % 16 == 0 && kCBarOff % 8 == 0,
              "alignment");
static_assert(kCSmemBytes <= 232448, "shared memory budget");

__global__ void __launch_bounds__(kCThreads, 1) mla_tc_kernel(const MlaParams p,
                                                              const __grid_constant__ CUtensorMap tmL) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  pdl_launch_dependents();
  pdl_wait();  // counts and pages come from the kernels before this one
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // quarter fastest, then head tile: the CTAs that read the same pages run side by side
  const int vq = static_cast<int>(blockIdx.x % kCParts);
  const int r1 = static_cast<int>(blockIdx.x / kCParts);
  const int ht = r1 % p.HT;
  const int r2 = r1 / p.HT;
  const int s = r2 % p.NS;
  const int b = r2 / p.NS;
  const int unit = b * p.HT + ht;
  const int h_base = ht * kCHeads;

  uint8_t* ring = smem;
  int32_t* rec_s = reinterpret_cast<int32_t*>(smem + kCRecOff);
  float* bias_s = reinterpret_cast<float*>(smem + kCBiasOff);
  float* xch_s = reinterpret_cast<float*>(smem + kCXchOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kCBarOff);
  uint64_t* empty = full + kCRing;
  uint64_t* s_full = empty + kCRing;  // [2]
  uint64_t* p_full = s_full + 2;      // [2]
  uint64_t* o_done = p_full + 2;      // [2]
  uint64_t* fin = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fin + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int cnt = min(max(p.count[b], 0), p.max_pages * kPage);
  const int np = (cnt + kPage - 1) / kPage;
  const int pg0 = static_cast<int>(static_cast<int64_t>(s) * np / p.NS);
  const int pg1 = static_cast<int>(static_cast<int64_t>(s + 1) * np / p.NS);
  const int n_my = pg1 - pg0;
  const int nb = (n_my + kCPages - 1) / kCPages;
  const int slot_end = min(cnt, pg1 * kPage);  // this slice's slots end here

  if (tid == 0) {
    for (int st = 0; st < kCRing; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kCParts);  // every CTA of the cluster releases the stage in all four
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(&s_full[j], 1);
      mbar_init(&p_full[j], kCSoftWarps);
      mbar_init(&o_done[j], 1);
    }
    mbar_init(fin, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmL);
  }
  if (warp == kCMmaWarp) {
    tmem_alloc(tmem_slot, kTcCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // every CTA's barriers exist before any copy or release reaches them
  const uint32_t tmem = *tmem_slot;
  const uint32_t crank = cluster_ctarank();

  if (warp < 4) {
    // ---- the query rows into tensor memory (thread = head row; zero past Hq)
    const int row = warp * 32 + lane;
    const int h = h_base + row;
    const uint4* src =
        h < p.Hq ? reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(b) * p.Hq + h) * kRow) : nullptr;
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll 1
    for (int c = 0; c < kBoxes; ++c) {
      uint32_t v[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 u = src != nullptr ? __ldg(src + c * 8 + i) : make_uint4(0, 0, 0, 0);
        v[4 * i] = u.x;
        v[4 * i + 1] = u.y;
        v[4 * i + 2] = u.z;
        v[4 * i + 3] = u.w;
      }
      tmem_st32(trow + kTcQCol + c * 32, v);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == kCCopyWarp) {
    // ------------------------------------------------------------ copies
    // The whole warp issues, one copy per lane (a copy instruction holds its
    // thread for about 100 ns): lane 3 pp + jj (pp < 6, jj < 3) copies box
    // crank + 4 jj of page pp into all four CTAs, lane 18 + pp page pp's
    // expire values into this one. Lane pp < 6 holds page pp of the block
    // (-1: past the slice or a bad id), read a block ahead.
    auto page_id = [&](int i) {
      int ph = -1;
      const int k = i * kCPages + lane;
      if (lane < kCPages && i < nb && k < n_my) {
        ph = p.page_table[static_cast<int64_t>(b) * p.max_pages + pg0 + k];
        if (ph < 0 || ph >= p.n_pages_cap) {
          record_error(p.status, KVP_ERR_BOUNDS);  // inconsistent page table: the page reads as gone
          ph = -1;
        }
      }
      return ph;
    };
    int ph_cur = page_id(0);
    int i = 0;
    bool okp = true;
    for (; i < nb; ++i) {
      const int st = i % kCRing;
      bool okw = true;
      if (lane == 0 && i >= kCRing)
        okw = mbar_wait(&empty[st], static_cast<uint32_t>((i / kCRing - 1) & 1), abort_flag, p.status);
      if (!__shfl_sync(0xffffffffu, okw ? 1 : 0, 0)) {
        if (lane == 0) {
          record_error(p.status, KVP_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        okp = false;
        break;
      }
      const int ph_nxt = page_id(i + 1);
      uint8_t* stage = ring + st * kCStageBytes;
      int32_t* rec = rec_s + st * kCTok;
      if (lane < kCPages && ph_cur < 0) {
        for (int tt = 0; tt < kPage; ++tt) rec[lane * kPage + tt] = 0;
        fence_proxy_async();  // ordered before a later copy into the same place
      }
      const int valid = __popc(__ballot_sync(0xffffffffu, lane < kCPages && ph_cur >= 0));
      __syncwarp();
      if (lane == 0) {
        fence_proxy_async();
        mbar_arrive_expect_tx(&full[st], kCStageBytes + valid * kPage * 4);
      }
      __syncwarp();
      const int src = lane < 3 * kCPages ? lane / 3 : (lane < 4 * kCPages ? lane - 3 * kCPages : 0);
      const int ph = __shfl_sync(0xffffffffu, ph_cur, src);
      // a page past the slice (or a bad one) is read from past the pool's last row: zeros
      const int y = (ph >= 0 ? ph : p.n_pages_cap) * kPage;
      if (lane < 3 * kCPages) {
        const int pp = lane / 3, j = static_cast<int>(crank) + kCParts * (lane % 3);
        if (j < kBoxes)
          tma_load_2d_multicast(stage + j * kCBoxRun + pp * kBoxBytes, &tmL, 64 * j, y, &full[st], kCAllCtas);
      } else if (lane < 4 * kCPages && ph >= 0) {
        const int pp = lane - 3 * kCPages;
        bulk_g2s(rec + pp * kPage, p.expire_pool + static_cast<int64_t>(ph) * kPage, kPage * 4, &full[st]);
      }
      ph_cur = ph_nxt;
    }
    if (!okp && lane == 0) {
      // the copies already issued land before the CTA's shared memory is released (each wait bounded again)
      for (int kk = max(0, i - kCRing); kk < i; ++kk) (void)mbar_wait(&full[kk % kCRing], (kk / kCRing) & 1u);
    }
    __syncwarp();
  } else if (warp == kCMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nb > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kCHeads, kCTok);
      constexpr uint32_t idO = idesc_bf16_f32(kCHeads, kCVals) | kIdescBMnMajor;
      const uint32_t ring_u32 = smem_u32(ring);
      // S of block i into buffer i % kCBufs; the block's pages must have landed
      // and, from block kCBufs on, the products of block i - kCBufs (which read
      // P from that buffer) must be complete
      auto issue_s = [&](int i) -> bool {
        if (!mbar_wait(&full[i % kCRing], static_cast<uint32_t>((i / kCRing) & 1), abort_flag, p.status)) return false;
        if (i >= kCBufs && !mbar_wait(&o_done[i % kCBufs], static_cast<uint32_t>(((i - kCBufs) / kCBufs) & 1),
                                      abort_flag, p.status))
          return false;
        tc_fence_after();
        const uint32_t base = ring_u32 + (i % kCRing) * kCStageBytes;
        const uint32_t d = tmem + kTcBufCol + (i % kCBufs) * kCTok;
        // the descriptor once per block; each product adds its box's offset to the start-address field (in
        // 16-byte units; shared addresses stay below 256 KB, so the field cannot carry into the next)
        const uint64_t bdesc0 = sw128_kmajor_desc(base);
        umma_bf16_tmem_a(d, tmem + kTcQCol, bdesc0, idS, 0u);
#pragma unroll
        for (int kk = 1; kk < kRow / 16; ++kk)
          umma_bf16_tmem_a_acc(d, tmem + kTcQCol + kk * 8,
                               bdesc0 + static_cast<uint64_t>(((kk >> 2) * kCBoxRun + (kk & 3) * 32) >> 4), idS);
        umma_commit(&s_full[i % kCBufs]);
        return true;
      };
      bool ok = true;
      for (int i = 0; ok && i < min(kCBufs, nb); ++i) ok = issue_s(i);
      for (int i = 0; ok && i < nb; ++i) {
        const int st = i % kCRing;
        ok = mbar_wait(&p_full[i % kCBufs], static_cast<uint32_t>((i / kCBufs) & 1), abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t vbase = ring_u32 + st * kCStageBytes + (kCVals / 64) * vq * kCBoxRun;
        const uint32_t pa = tmem + kTcBufCol + (i % kCBufs) * kCTok + kTcPOff;
#pragma unroll
        for (int ks = 0; ks < kCPages; ++ks) {
          const uint64_t bdesc = sw128_mnmajor_desc(vbase + ks * kBoxBytes, kCBoxRun, 1024);
          umma_bf16_tmem_a(tmem + kTcOCol, pa + ks * 8, bdesc, idO, (i > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(&o_done[i % kCBufs]);
        umma_commit_multicast(&empty[st], kCAllCtas);  // the stage is free in this CTA: tell all four
        if (i + kCBufs < nb) ok = issue_s(i + kCBufs);
      }
      if (!ok) {
        record_error(p.status, KVP_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      umma_commit(fin);
      (void)mbar_wait(fin, 0u);  // every product issued has completed before tensor memory is freed
      // the other CTAs' releases of the last stages have reached this CTA's barriers before it exits
      for (int i = max(0, nb - kCRing); i < nb; ++i)
        (void)mbar_wait(&empty[i % kCRing], static_cast<uint32_t>((i / kCRing) & 1), abort_flag, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    // warp w: rows 32 (w & 3) .., tokens kCHalf (w >> 2) .. of each block; output columns (kCVals / 2) (w >> 2) ..
    const int quad = warp & 3, hs = warp >> 2;
    const int row = quad * 32 + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    const int bar_id = 1 + quad;  // named barrier of the pair (warps quad, quad + 4)
    float* bias = bias_s + warp * kCHalf;
    float m = -1e30f, l = 0.f;
    bool ok = true;
    for (int i = 0; i < nb; ++i) {
      const int st = i % kCRing;
      const uint32_t bcol = kTcBufCol + (i % kCBufs) * kCTok;
      ok = mbar_wait(&s_full[i % kCBufs], static_cast<uint32_t>((i / kCBufs) & 1), abort_flag, p.status);
      // the pair leaves together, so that neither waits at the barrier for a partner that has left
      if (named_bar_or(bar_id, 64, !ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[kCHalf];
      tmem_ld_cols(trow + bcol + hs * kCHalf, x);
      // this warp's tokens' mask as an additive bias
      {
        const int32_t* rec = rec_s + st * kCTok + hs * kCHalf;
        const int slot0 = (pg0 + i * kCPages) * kPage + hs * kCHalf;
#pragma unroll
        for (int j = lane; j < kCHalf; j += 32) bias[j] = (slot0 + j < slot_end && p.now < rec[j]) ? 0.f : -INFINITY;
        __syncwarp();
      }
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < kCHalf; j += 4) {
        const float4 bb = *reinterpret_cast<const float4*>(bias + j);
        x[j] = fmaf(x[j], p.qscale, bb.x);
        x[j + 1] = fmaf(x[j + 1], p.qscale, bb.y);
        x[j + 2] = fmaf(x[j + 2], p.qscale, bb.z);
        x[j + 3] = fmaf(x[j + 3], p.qscale, bb.w);
        mx = fmaxf(mx, fmaxf(fmaxf(x[j], x[j + 1]), fmaxf(x[j + 2], x[j + 3])));
      }
      // the row maximum over both halves (double-buffered by block parity); past this barrier both
      // warps of the pair have read their S, so either may write P over it
      float* xb = xch_s + (i & 1) * kCSoftWarps * 32;
      xb[warp * 32 + lane] = mx;
      tc_fence_before();
      named_bar_sync(bar_id, 64);
      tc_fence_after();
      mx = fmaxf(mx, xb[(warp ^ 4) * 32 + lane]);
      const bool grow = mx > m + kLazyRescale;  // the same in both warps of the pair
      if (i > 0 && __any_sync(0xffffffffu, grow)) {
        ok = mbar_wait(&o_done[(i - 1) % kCBufs], static_cast<uint32_t>(((i - 1) / kCBufs) & 1), abort_flag,
                       p.status);
        if (named_bar_or(bar_id, 64, !ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float al = grow ? exp2f(m - mx) : 1.f;
#pragma unroll 1
        for (int c = hs * (kCVals / 2); c < (hs + 1) * (kCVals / 2); c += 32) {
          float v[32];
          tmem_ld32(trow + kTcOCol + c, v);
          uint32_t w[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) w[j] = __float_as_uint(v[j] * al);
          tmem_st32(trow + kTcOCol + c, w);
        }
      }
      if (grow) {
        l *= exp2f(m - mx);
        m = mx;
      }
      // p = 2^(x - m) rounded to bf16 for the product; the sum takes p itself
      uint32_t pk[kCHalf / 2];
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int j = 0; j < kCHalf / 2; ++j) {
        const float p0 = ex2_approx(x[2 * j] - m);
        const float p1 = ex2_approx(x[2 * j + 1] - m);
        ls0 += p0;
        ls1 += p1;
        const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);  // p0 in the low half
        pk[j] = *reinterpret_cast<const uint32_t*>(&pb);
      }
      l += ls0 + ls1;
      // P of tokens kCHalf hs .. at columns bcol + kTcPOff + (kCHalf / 2) hs ..
      tmem_st_cols(trow + bcol + kTcPOff + hs * (kCHalf / 2), pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[i % kCBufs]);
    }
    if (ok && nb > 0) {
      ok = mbar_wait(&o_done[(nb - 1) % kCBufs], static_cast<uint32_t>(((nb - 1) / kCBufs) & 1), abort_flag,
                     p.status);
      ok = !named_bar_or(bar_id, 64, !ok);
      tc_fence_after();
    }
    if (!ok) {
      if (lane == 0) {
        record_error(p.status, KVP_ERR_TIMEOUT);
        *abort_flag = 1;
      }
    } else {
      // the row's sum over both halves
      float* xb = xch_s + (nb & 1) * kCSoftWarps * 32;
      xb[warp * 32 + lane] = l;
      named_bar_sync(bar_id, 64);
      const float lt = l + xb[(warp ^ 4) * 32 + lane];
      const int h = h_base + row;
      const int c0 = hs * (kCVals / 2);
      if (p.NS == 1) {
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        float* orow = p.out + (static_cast<int64_t>(b) * p.Hq + h) * kDc + vq * kCVals;
#pragma unroll 1
        for (int c = c0; c < c0 + kCVals / 2; c += 32) {
          float v[32];
          if (nb > 0) {
            tmem_ld32(trow + kTcOCol + c, v);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.f;
          }
          if (h < p.Hq) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(orow + c + j) =
                  make_float4(v[j] * inv, v[j + 1] * inv, v[j + 2] * inv, v[j + 3] * inv);
          }
        }
      } else {
        const int64_t slot = static_cast<int64_t>(unit) * p.NS + s;
        if (nb > 0) {  // an empty slice leaves its accumulator unwritten: its sum is 0 and the merge skips it
          float* pa = p.part_acc + (slot * kCHeads + row) * kDc + vq * kCVals;
#pragma unroll 1
          for (int c = c0; c < c0 + kCVals / 2; c += 32) {
            float v[32];
            tmem_ld32(trow + kTcOCol + c, v);
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(pa + c + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
          }
        }
        if (vq == 0 && hs == 0) {
          p.part_ml[(slot * kCHeads + row) * 2] = m;
          p.part_ml[(slot * kCHeads + row) * 2 + 1] = lt;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kCMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcCols);
  }
  cluster_sync();  // no CTA leaves while another may still signal it
}

int sm_count() {
  static const int n = [] {
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
      return 0;
    return nsm;
  }();
  return n;
}

// Which kernel takes a call (batch 16 x 8192 tokens): CTAs of
// mla_decode_kernel take 16-head tiles up to kTileFrom - 1 query heads (at 32
// heads two tiles of 16 ran 87 us where one 64-head tile with half its warps
// idle ran 90 us), mla_tile_kernel 64-head tiles up to kTcFrom - 1 (106 us at
// 40 heads, 121 us at 64, where mla_tc_kernel takes about 137 us at any head
// count up to 128), mla_tc_kernel 128-head tiles from kTcFrom on (137 us at
// 128 heads, where two 64-head tiles take 262 us).
#ifndef KVP_MLA_TC_FROM
#define KVP_MLA_TC_FROM 65
#endif
constexpr int kTileFrom = 33;
constexpr int kTcFrom = KVP_MLA_TC_FROM;
enum MlaPath { kPath16, kPath64, kPathTc };
MlaPath mla_path(int n_q_heads) {
  return n_q_heads >= kTcFrom ? kPathTc : (n_q_heads >= kTileFrom ? kPath64 : kPath16);
}
int tile_heads(int n_q_heads) {
  const MlaPath k = mla_path(n_q_heads);
  return k == kPathTc ? kCHeads : (k == kPath64 ? kTHeads : kHT);
}
int n_tiles(int n_q_heads) { return (n_q_heads + tile_heads(n_q_heads) - 1) / tile_heads(n_q_heads); }
int ctas_per_slice(int n_q_heads) { return mla_path(n_q_heads) == kPathTc ? kCParts : 1; }

// Slices per unit: as many as one wave of CTAs holds (two per SM for the
// 16-head kernel, one for the others), so no CTA waits for a second wave
// (128 units on 152 SMs: 2 slices, 256 CTAs, rather than 3 slices and 384
// CTAs in 1.26 waves); at least one.
int pick_splits(int batch, int n_q_heads) {
  const int nsm = sm_count();
  const int64_t units = static_cast<int64_t>(batch) * n_tiles(n_q_heads) * ctas_per_slice(n_q_heads);
  const int per_sm = mla_path(n_q_heads) == kPath16 ? 2 : 1;
  const int64_t want = per_sm * static_cast<int64_t>(nsm > 0 ? nsm : 1) / units;
  return static_cast<int>(want < 1 ? 1 : (want > kMaxSplits ? kMaxSplits : want));
}

size_t round16(size_t n) { return (n + 15) / 16 * 16; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// workspace: part_ml [units, NS, TH, 2], then part_acc [units, NS, TH, kDc],
// each region starting on 16 bytes; every call writes the (m, l) of every
// slice and the accumulator of every slice with pages before the merge reads
// them, so nothing carries over from one call to the next
size_t ws_ml_bytes(int64_t units, int ns, int th) { return round16(static_cast<size_t>(units) * ns * th * 2 * 4); }

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" size_t kvp_decode_attn_mla_workspace_bytes(int batch, int n_q_heads, int n_splits) {
  if (batch <= 0 || n_q_heads <= 0 || n_splits < 0 || n_splits > kMaxSplits) return 0;
  const int ns = n_splits > 0 ? n_splits : pick_splits(batch, n_q_heads);
  const int64_t units = static_cast<int64_t>(batch) * n_tiles(n_q_heads);
  const int th = tile_heads(n_q_heads);
  return ws_ml_bytes(units, ns, th) + static_cast<size_t>(units) * ns * th * kDc * 4;
}

extern "C" kvp_status kvp_decode_attn_mla(int batch, int n_q_heads, int latent_dim, int rope_dim, const void* q,
                                          const void* pool, const int32_t* expire_pool, int n_pages_cap,
                                          const int32_t* page_table, int max_pages, const int32_t* count, int now,
                                          float scale, float* out, int n_splits, void* workspace,
                                          size_t workspace_bytes, int32_t* status, void* stream) {
  if (batch <= 0 || n_q_heads <= 0 || max_pages < 0 || n_pages_cap < 0) return KVP_ERR_INVALID;
  if (n_splits < 0 || n_splits > kMaxSplits) return KVP_ERR_INVALID;
  if (latent_dim != kDc || rope_dim != kDr) return KVP_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_pages) * kPage > 0x7fffffff || static_cast<int64_t>(n_pages_cap) * kPage > 0x7fffffff)
    return KVP_ERR_UNSUPPORTED;
  if (!(scale >= 0.f)) return KVP_ERR_INVALID;
  if (q == nullptr || pool == nullptr || expire_pool == nullptr || page_table == nullptr || count == nullptr ||
      out == nullptr)
    return KVP_ERR_INVALID;
  if (!aligned16(q) || !aligned16(pool) || !aligned16(expire_pool) || !aligned16(out)) return KVP_ERR_ALIGN;
  const int ns = n_splits > 0 ? n_splits : pick_splits(batch, n_q_heads);
  const int HT = n_tiles(n_q_heads);
  const int th = tile_heads(n_q_heads);
  const int64_t units = static_cast<int64_t>(batch) * HT;
  const MlaPath path = mla_path(n_q_heads);
  const int64_t grid = units * ns * ctas_per_slice(n_q_heads);
  if (grid > 0x7fffffff || units * th > 0x7fffffff) return KVP_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < kvp_decode_attn_mla_workspace_bytes(batch, n_q_heads, ns))
    return KVP_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KVP_ERR_ALIGN;
  if (n_pages_cap == 0) {  // nothing can be read: every row is empty
    return cudaMemsetAsync(out, 0, static_cast<size_t>(batch) * n_q_heads * kDc * sizeof(float),
                           static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KVP_OK
               : KVP_ERR_CUDA;
  }
  // the tensor-core kernel copies 16 x 64 boxes; the others a page (16 rows x nine 64-column groups) at a time
  CUtensorMap tmL;
  const bool ok_map = path == kPathTc
                          ? make_tmap_bf16(&tmL, pool, static_cast<int64_t>(n_pages_cap) * kPage, kRow, kRow, kPage, 64)
                          : make_tmap_bf16_groups(&tmL, pool, static_cast<int64_t>(n_pages_cap) * kPage, kRow, kRow,
                                                  kPage);
  if (!ok_map) return KVP_ERR_CUDA;
  static const bool attr_ok =
      cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) ==
          cudaSuccess &&
      cudaFuncSetAttribute(mla_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTSmemBytes) ==
          cudaSuccess &&
      cudaFuncSetAttribute(mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCSmemBytes) == cudaSuccess;
  if (!attr_ok) return KVP_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  MlaParams p{static_cast<const uint16_t*>(q),
              expire_pool,
              page_table,
              count,
              batch,
              n_q_heads,
              HT,
              ns,
              th,
              max_pages,
              n_pages_cap,
              now,
              (scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(kRow))) * 1.4426950408889634f,
              out,
              reinterpret_cast<float*>(ws + ws_ml_bytes(units, ns, th)),
              reinterpret_cast<float*>(ws),
              status};
  const dim3 g(static_cast<unsigned>(grid));
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const cudaError_t le =
      path == kPathTc   ? launch_pdl_cluster(mla_tc_kernel, g, dim3(kCThreads), kCSmemBytes, cs, kCParts, p, tmL)
      : path == kPath64 ? launch_pdl(mla_tile_kernel, g, dim3(kTThreads), kTSmemBytes, cs, p, tmL)
                        : launch_pdl(mla_decode_kernel, g, dim3(kMThreads), kSmemBytes, cs, p, tmL);
  if (le != cudaSuccess) return KVP_ERR_CUDA;
  if (ns > 1 && launch_pdl(mla_merge_kernel, dim3(static_cast<unsigned>(units * th)), dim3(kDc / 4), 0,
                           static_cast<cudaStream_t>(stream), p) != cudaSuccess)
    return KVP_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}
