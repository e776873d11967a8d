// kvp_decode_attn_mla: MLA's absorbed decode attention over a pruned latent
// cache (DMS article, "주요 요점" and "앞으로의 전망": the method carries over
// to Multi-Head Latent Attention, whose cache is one latent row per token).
//
// Query head j of batch element b scores slot t with scale * q[b, j] . row_t
// over the whole 576-value row (512 compressed-KV values, then the 64-value
// rotary key) and takes the softmax-weighted sum of the rows' first 512
// values. Every query head reads the same rows, so a page is worth
// 16 tokens x (576 + 512) x 2 flops per head: on CUDA cores that outruns HBM
// from a few heads on; here both products run on the tensor cores
// (mma.sync m16n8k16, bf16 operands, fp32 accumulate).
//
// A CTA (4 warps) takes 16 query heads of one batch element and one slice of
// its pages. Its pages arrive through a ring of kRingPages stages as nine
// 16-row x 64-column boxes each (tensor copies of the pool viewed as
// [pages x 16, 576], with the 128-byte swizzle, so ldmatrix reads are free of
// bank conflicts), plus the page's 16 expire values. Per page:
//   S   = C Q^T     M = 16 tokens, N = 16 heads, K = 576: warp w takes the
//                   144 values 144w .. 144w + 143; the four partial products
//                   are summed through shared memory (one CTA barrier)
//   softmax         every warp computes the same weights from the same sums
//                   (online, base 2, lazy rescaling)
//   O^T += Cv^T P^T M = 16 of the 512 compressed values at a time, N = 16
//                   heads, K = 16 tokens: warp w owns values 128w .. 128w+127
//                   (8 m-tiles), its A operand read transposed by ldmatrix
// Slices of a unit (batch element, 16 heads) write their partial states; a
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
constexpr int kSpartFloats = 32 * 8;          // one warp's partial logits (8 per lane)
constexpr int kPtHalves = 2 * 2 * 8 * kPage;  // one warp's P^T: n-tile x (hi, lo) x 8 heads x 16 tokens
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
  int B, Hq, HT, NS;          // batch, query heads, 16-head tiles, slices per unit
  int max_pages, n_pages_cap, now;
  float qscale;               // scale * log2(e)
  float* out;                 // [B, Hq, kDc]
  float* part_acc;            // [units, NS, 16, kDc]
  float* part_ml;             // [units, NS, 16, 2]
  int32_t* status;
};

__global__ void __launch_bounds__(kMThreads, 1) mla_decode_kernel(const MlaParams p,
                                                                  const __grid_constant__ CUtensorMap tmL) {
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
    prefetch_tmap(&tmL);
    for (int st = 0; st < kRingPages; ++st) mbar_init(&bars[st], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // Page k of the slice into stage k % kRingPages (thread 0).
  auto issue = [&](int k) {
    const int st = k % kRingPages;
    uint8_t* dst = ring + st * kStageBytes;
    int32_t* rec = rec_s + st * kPage;
    const int phys = p.page_table[static_cast<int64_t>(b) * p.max_pages + pg0 + k];
    if (phys < 0 || phys >= p.n_pages_cap) {
      // inconsistent page table: no copy; the page reads as zeros and every
      // slot of it as gone
      record_error(p.status, KVP_ERR_BOUNDS);
      uint4* z = reinterpret_cast<uint4*>(dst);
      for (int i = 0; i < kStageBytes / 16; ++i) z[i] = make_uint4(0, 0, 0, 0);
      for (int i = 0; i < kPage; ++i) rec[i] = 0;
      mbar_arrive(&bars[st]);
      return;
    }
    mbar_arrive_expect_tx(&bars[st], kStageBytes + kPage * 4);
    const int y = phys * kPage;
#pragma unroll
    for (int j = 0; j < kBoxes; ++j) tma_load_2d(dst + j * kBoxBytes, &tmL, 64 * j, y, &bars[st]);
    bulk_g2s(rec, p.expire_pool + static_cast<int64_t>(phys) * kPage, kPage * 4, &bars[st]);
  };
  int issued = 0;  // pages issued so far (thread 0's count)
  if (tid == 0)
    for (; issued < n_my && issued < kRingPages; ++issued) issue(issued);

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
    float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int i = 0; i < kKsW; ++i) {
      const int ks = warp * kKsW + i;
      // matrices: 0 rows 0-7 / 1 rows 8-15 of the k-step's first 8 values, 2 / 3 of its second 8
      const int r = (mi & 1) * 8 + ri;
      const int chunk = (ks & 3) * 2 + (mi >> 1);
      const uint32_t addr = base + (ks >> 2) * kBoxBytes + r * 128 + ((chunk ^ (r & 7)) << 4);
      uint32_t a0, a1, a2, a3;
      ldsm_x4(addr, a0, a1, a2, a3);
      mma_bf16_16816(sacc[0], a0, a1, a2, a3, qf[i][0][0], qf[i][0][1]);
      mma_bf16_16816(sacc[1], a0, a1, a2, a3, qf[i][1][0], qf[i][1][1]);
    }
    float* sp = spart + (k & 1) * (kMW * kSpartFloats);  // two buffers: page k + 1 writes the other
    *reinterpret_cast<float4*>(sp + warp * kSpartFloats + lane * 8) =
        make_float4(sacc[0][0], sacc[0][1], sacc[0][2], sacc[0][3]);
    *reinterpret_cast<float4*>(sp + warp * kSpartFloats + lane * 8 + 4) =
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
    if (tid == 0 && k >= 1 && issued < n_my) {  // page k - 1's stage takes the next page
      fence_proxy_async();
      issue(issued);
      ++issued;
    }

    // ---- full logits (the four partials in a fixed order, so every warp
    // holds the same values), mask, online softmax
    float sv[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int w = 0; w < kMW; ++w) {
      const float4 u0 = *reinterpret_cast<const float4*>(sp + w * kSpartFloats + lane * 8);
      const float4 u1 = *reinterpret_cast<const float4*>(sp + w * kSpartFloats + lane * 8 + 4);
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
        pt_s[((nt * 2 + 0) * 8 + hrow) * kPage + tok[i]] = __bfloat16_as_ushort(hi);
        pt_s[((nt * 2 + 1) * 8 + hrow) * kPage + tok[i]] = __bfloat16_as_ushort(lo);
      }
    }
    __syncwarp();
    // B fragments of P^T (k = tokens, n = heads): head 8 nt + g, tokens 2t, +1 and 2t + 8, +9
    uint32_t pb[2][2], pl[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint16_t* hi_row = pt_s + ((nt * 2 + 0) * 8 + gq) * kPage;
      const uint16_t* lo_row = pt_s + ((nt * 2 + 1) * 8 + gq) * kPage;
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

// Merge of the slices of every unit: CTA (unit, hl) takes head h_base + hl,
// thread c the float4 c of its 512 output values. The slices' (m, l) give
// the weights exp2(m - M) (an empty slice, l = 0, has none and its
// accumulator is not read), then the accumulators are summed with all of a
// batch of slices' loads in flight.
__global__ void __launch_bounds__(kDc / 4) mla_merge_kernel(const MlaParams p) {
  __shared__ float w_s[kMaxSplits];
  __shared__ float il_s;
  pdl_launch_dependents();
  pdl_wait();  // every slice's partial state is written
  const int unit = static_cast<int>(blockIdx.x / kHT), hl = static_cast<int>(blockIdx.x % kHT);
  const int b = unit / p.HT, h = (unit % p.HT) * kHT + hl;
  if (h >= p.Hq) return;
  const int c4 = threadIdx.x;
  const float* ml = p.part_ml + static_cast<int64_t>(unit) * p.NS * kHT * 2;
  if (c4 < 32) {
    float M = -INFINITY;
    for (int sl = c4; sl < p.NS; sl += 32) {
      const float l = __ldcg(ml + (sl * kHT + hl) * 2 + 1);
      if (l > 0.f) M = fmaxf(M, __ldcg(ml + (sl * kHT + hl) * 2));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int sl = c4; sl < p.NS; sl += 32) {
      const float l = __ldcg(ml + (sl * kHT + hl) * 2 + 1);
      const float w = l > 0.f ? exp2f(__ldcg(ml + (sl * kHT + hl) * 2) - M) : 0.f;
      w_s[sl] = w;
      L += w * l;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (c4 == 0) il_s = L > 0.f ? 1.f / L : 0.f;
  }
  __syncthreads();
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* acc = reinterpret_cast<const float4*>(p.part_acc + static_cast<int64_t>(unit) * p.NS * kHT * kDc);
  constexpr int kBatch = 8;
  for (int s0 = 0; s0 < p.NS; s0 += kBatch) {
    float4 v[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int sl = s0 + j;
      v[j] = (sl < p.NS && w_s[sl] != 0.f) ? __ldcg(acc + (static_cast<int64_t>(sl) * kHT + hl) * (kDc / 4) + c4)
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

int n_tiles(int n_q_heads) { return (n_q_heads + kHT - 1) / kHT; }

// Slices per unit: as many as one wave of CTAs holds (two per SM), so no
// CTA waits for a second wave (128 units on 152 SMs: 2 slices, 256 CTAs,
// rather than 3 slices and 384 CTAs in 1.26 waves); at least one.
int pick_splits(int batch, int n_q_heads) {
  const int nsm = sm_count();
  const int64_t units = static_cast<int64_t>(batch) * n_tiles(n_q_heads);
  const int64_t want = 2 * static_cast<int64_t>(nsm > 0 ? nsm : 1) / units;
  return static_cast<int>(want < 1 ? 1 : (want > kMaxSplits ? kMaxSplits : want));
}

size_t round16(size_t n) { return (n + 15) / 16 * 16; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// workspace: part_ml [units, NS, 16, 2], then part_acc [units, NS, 16, kDc],
// each region starting on 16 bytes; every call writes the (m, l) of every
// slice and the accumulator of every slice with pages before the merge reads
// them, so nothing carries over from one call to the next
size_t ws_ml_bytes(int64_t units, int ns) { return round16(static_cast<size_t>(units) * ns * kHT * 2 * 4); }

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" size_t kvp_decode_attn_mla_workspace_bytes(int batch, int n_q_heads, int n_splits) {
  if (batch <= 0 || n_q_heads <= 0 || n_splits < 0 || n_splits > kMaxSplits) return 0;
  const int ns = n_splits > 0 ? n_splits : pick_splits(batch, n_q_heads);
  const int64_t units = static_cast<int64_t>(batch) * n_tiles(n_q_heads);
  return ws_ml_bytes(units, ns) + static_cast<size_t>(units) * ns * kHT * kDc * 4;
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
  const int64_t units = static_cast<int64_t>(batch) * HT;
  const int64_t grid = units * ns;
  if (grid > 0x7fffffff || units * kHT > 0x7fffffff) return KVP_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < kvp_decode_attn_mla_workspace_bytes(batch, n_q_heads, ns))
    return KVP_ERR_WORKSPACE;
  if (!aligned16(workspace)) return KVP_ERR_ALIGN;
  if (n_pages_cap == 0) {  // nothing can be read: every row is empty
    return cudaMemsetAsync(out, 0, static_cast<size_t>(batch) * n_q_heads * kDc * sizeof(float),
                           static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KVP_OK
               : KVP_ERR_CUDA;
  }
  CUtensorMap tmL;
  if (!make_tmap_bf16(&tmL, pool, static_cast<int64_t>(n_pages_cap) * kPage, kRow, kRow, kPage, 64))
    return KVP_ERR_CUDA;
  static const bool attr_ok = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   kSmemBytes) == cudaSuccess;
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
              max_pages,
              n_pages_cap,
              now,
              (scale > 0.f ? scale : 1.0f / sqrtf(static_cast<float>(kRow))) * 1.4426950408889634f,
              out,
              reinterpret_cast<float*>(ws + ws_ml_bytes(units, ns)),
              reinterpret_cast<float*>(ws),
              status};
  if (launch_pdl(mla_decode_kernel, dim3(static_cast<unsigned>(grid)), dim3(kMThreads), kSmemBytes,
                 static_cast<cudaStream_t>(stream), p, tmL) != cudaSuccess)
    return KVP_ERR_CUDA;
  if (ns > 1 && launch_pdl(mla_merge_kernel, dim3(static_cast<unsigned>(units * kHT)), dim3(kDc / 4), 0,
                           static_cast<cudaStream_t>(stream), p) != cudaSuccess)
    return KVP_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}
