// kvp_score: KVzap surrogate scores on the tcgen05 tensor cores.
//
// KVzap summary ("NVIDIA가 AI 메모리 압축 신기술 KVzap 오픈소스 공개!"),
// 핵심 내용 정리 -> "KVzap의 구조": one linear layer, or a 2-layer MLP, maps a
// token's hidden state to a score per KV head; "실제 적용": every cache entry is
// scored during inference.
//
// One persistent warp-specialised kernel serves both scorers:
//   warp 0      TMA producer: 128x64 tiles of x and BNx64 tiles of the weight
//               (both K-major, 128-byte swizzle) into a STAGES-deep ring
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma 128xBNx16, fp32
//               accumulators double-buffered in tensor memory
//   epilogue    tcgen05.ld of the accumulator rows, then
//               LINEAR (warps 2..5, one per TMEM lane quadrant):
//                       s_h = acc[2h] + acc[2h+1] + b_h (weight rows interleave
//                       the bf16 high and low halves of the fp32 weight)
//               MLP (warps 2..9, two per quadrant, each taking 128 of the 256
//                       hidden columns): GELU(acc + b1) dotted with W2; the
//                       upper half's partial scores are added to the lower
//                       half's through shared memory -> per-chunk partials
// A small reduction kernel then sums the MLP chunk partials in a fixed order.
//
// A decode step scores only the batch's new tokens (a few rows): one 128-row
// tile would leave the whole weight to a single CTA. Up to kGemvMaxRows rows
// the Linear scorer is instead a CUDA-core dot product over the same bf16
// hi/lo weight rows, spread over one CTA per (head, group of 8 rows); the
// MLP scorer likewise runs its few rows on the CUDA cores, one CTA per 8
// hidden units and group of 8 rows. The Linear path requests kGemvBatch
// chunks of each row per thread before the first product; the MLP path
// stages the rows' inputs in shared memory and requests a warp's weights a
// piece (kMlpXPiece values) ahead.
#include "kvp_common.cuh"

namespace kvp {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kMlpBN = 256;
constexpr int kMlpMaxH = 16;
constexpr int kGemvMaxRows = 64;  // Linear scorer: rows up to which the CUDA-core kernel runs
constexpr int kGemvRows = 8;      // rows per CTA of that kernel
constexpr int kGemvThreads = 256;
constexpr int kMlpGemvUnits = 8;   // MLP scorer, few rows: hidden units per CTA (one per warp)
constexpr int kGemvBatch = 4;      // 16-byte chunks of a row each thread requests before using any

enum { kEpiLinear = 0, kEpiMlp = 1 };
// TMA warp, MMA warp, then 4 epilogue warps (LINEAR) or 8 (MLP: its GELU and
// W2 epilogue is the long pole, so two warps share each lane quadrant).
template <int EPI>
constexpr int epi_threads() { return EPI == kEpiMlp ? 256 : 128; }
template <int EPI>
constexpr int score_threads() { return 64 + epi_threads<EPI>(); }

template <int BN>
struct ScoreCfg {
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = BN <= 32 ? 8 : (BN <= 128 ? 6 : 4);
  static constexpr int kTmemCols = (2 * BN < 32) ? 32 : 2 * BN;
  static constexpr int kBarBytes = 256;
  // MLP: W2 columns and b1 of the hidden chunk, then the upper half's partial
  // scores [2 accumulator buffers][128 rows][kMlpMaxH]
  static constexpr int kEpiBytes = (BN == kMlpBN) ? (kMlpBN * kMlpMaxH * 4 + kMlpBN * 4 + 2 * kBM * kMlpMaxH * 4) : 0;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kBarBytes + kEpiBytes;
  static_assert(kBBytes % 1024 == 0, "B tile must keep 1024-byte alignment");
  static_assert(kSmem <= 232448, "shared memory budget");
};

struct ScoreParams {
  int n_tok;
  int n_heads;
  int hidden;
  int m_tiles;
  int n_tiles;
  int k_blocks;
  const float* bias;        // LINEAR: b[H]; MLP: b1[hidden]; may be null
  const uint16_t* w2;       // MLP: bf16 [H, hidden]
  float* out;               // LINEAR: scores [n_tok, H]; MLP: partials [n_tiles, n_tok, H]
  int32_t* status;
};

template <int BN, int EPI>
__global__ void __launch_bounds__(score_threads<EPI>(), 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const ScoreParams p) {
  using C = ScoreCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(tiles + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* w2s = reinterpret_cast<float*>(tiles + C::kStages * C::kStageBytes + C::kBarBytes);
  float* b1s = w2s + kMlpBN * kMlpMaxH;
  float* comb = b1s + kMlpBN;  // MLP: upper-half partial scores [2][kBM][kMlpMaxH]
  constexpr int kEpi = epi_threads<EPI>();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpi);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int n_tiles_total = p.m_tiles * p.n_tiles;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const uint64_t pol_x = policy_evict_first();  // hidden states stream through once
      const uint64_t pol_w = policy_evict_last();   // weights are re-read by every tile
      uint32_t stage = 0, phase = 0;
      uint32_t issued = 0, issued_par = 0;  // per stage: loaded at least once, parity of its last load
      for (int t = blockIdx.x; t < n_tiles_total && !*abort_flag; t += gridDim.x) {
        const int mt = t / p.n_tiles, nt = t - mt * p.n_tiles;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) {
            record_error(p.status, KVP_ERR_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          uint8_t* a = tiles + stage * C::kStageBytes;
          issued |= 1u << stage;
          issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
          mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
          tma_load_2d_hint(a, &tmA, kb * kBK, mt * kBM, &full[stage], pol_x);
          tma_load_2d_hint(a + C::kABytes, &tmB, kb * kBK, nt * BN, &full[stage], pol_w);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort_flag) {
        // a wait gave up: the loads already issued land before the shared
        // memory is released (each wait bounded again)
        for (int s = 0; s < C::kStages; ++s)
          if ((issued >> s) & 1u) (void)mbar_wait(&full[s], (issued_par >> s) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      int last_stage = -1;     // stage and phase of the last commit, which tracks every MMA issued before it
      uint32_t last_par = 0;
      for (int t = blockIdx.x; t < n_tiles_total && !*abort_flag; t += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status)) {
          record_error(p.status, KVP_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) {
            record_error(p.status, KVP_ERR_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(tiles + stage * C::kStageBytes);
          const uint64_t adesc = sw128_kmajor_desc(a_addr);
          const uint64_t bdesc = sw128_kmajor_desc(a_addr + C::kABytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            umma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(&empty[stage]);  // frees this smem stage once the MMAs have read it
          last_stage = static_cast<int>(stage);
          last_par = phase;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        umma_commit(&tfull[acc]);  // accumulator ready for the epilogue
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // a wait gave up: the MMAs already issued finish before tensor memory is
      // freed (bounded)
      if (*abort_flag && last_stage >= 0) (void)mbar_wait(&empty[last_stage], last_par);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;          // TMEM lane quadrant this warp may access
    const int half = (warp - 2) >> 2;   // MLP: which 128 of the 256 hidden columns (LINEAR: 0)
    const int row = quad * 32 + lane;
    const int etid = threadIdx.x - 64;
    uint32_t acc = 0, acc_phase = 0;
    int cur_nt = -1;
    for (int t = blockIdx.x; t < n_tiles_total; t += gridDim.x) {
      const int mt = t / p.n_tiles, nt = t - mt * p.n_tiles;
      if constexpr (EPI == kEpiMlp) {
        if (nt != cur_nt) {  // stage this hidden chunk's W2 columns and b1 as fp32
          named_bar_sync(1, kEpi);
          const int H = p.n_heads;
          for (int i = etid; i < kMlpBN * H; i += kEpi) {
            const int c = i / H, h = i - c * H;
            const uint32_t w = p.w2[static_cast<size_t>(h) * p.hidden + nt * kMlpBN + c];
            w2s[c * H + h] = __uint_as_float(w << 16);
          }
          for (int c = etid; c < kMlpBN; c += kEpi) b1s[c] = p.bias ? p.bias[nt * kMlpBN + c] : 0.f;
          named_bar_sync(1, kEpi);
          cur_nt = nt;
        }
      }
      const bool ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, p.status);
      if (named_bar_or(3, kEpi, !ok)) {  // every epilogue thread leaves together
        if (etid == 0) {
          record_error(p.status, KVP_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN;
      const int grow = mt * kBM + row;
      if constexpr (EPI == kEpiLinear) {
        float v[BN];
#pragma unroll
        for (int c = 0; c < BN; c += 16) tmem_ld16(taddr + c, *reinterpret_cast<float(*)[16]>(&v[c]));
        tc_fence_before();
        mbar_arrive(&tempty[acc]);
        if (grow < p.n_tok) {
          const int H = p.n_heads;
          float* o = p.out + static_cast<size_t>(grow) * H;
#pragma unroll
          for (int h = 0; h < BN / 2; ++h) {
            if (h < H) o[h] = v[2 * h] + v[2 * h + 1] + (p.bias ? __ldg(p.bias + h) : 0.f);
          }
        }
      } else {
        const int H = p.n_heads;
        float part[kMlpMaxH];
#pragma unroll
        for (int h = 0; h < kMlpMaxH; ++h) part[h] = 0.f;
        constexpr int kCols = kMlpBN / 2;
#pragma unroll 1
        for (int cc = half * kCols; cc < (half + 1) * kCols; cc += 32) {
          float v[32];
          tmem_ld32(taddr + cc, v);
          if (cc == (half + 1) * kCols - 32) {
            tc_fence_before();
            mbar_arrive(&tempty[acc]);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float u = v[j] + b1s[cc + j];
            const float z = 0.5f * u * (1.0f + erff(u * 0.70710678118654752f));
            const float* wr = w2s + (cc + j) * H;
#pragma unroll
            for (int h = 0; h < kMlpMaxH; ++h)
              if (h < H) part[h] = fmaf(z, wr[h], part[h]);
          }
        }
        float* cb = comb + (acc * kBM + row) * kMlpMaxH;
        if (half == 1) {
#pragma unroll
          for (int h = 0; h < kMlpMaxH; ++h) cb[h] = part[h];
        }
        named_bar_sync(2, kEpi);  // the buffer of this accumulator is next written two tiles on
        if (half == 0 && grow < p.n_tok) {
          float* o = p.out + (static_cast<size_t>(nt) * p.n_tok + grow) * H;
#pragma unroll
          for (int h = 0; h < kMlpMaxH; ++h)
            if (h < H) o[h] = part[h] + cb[h];
        }
      }
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// W [H, D] fp32 -> Wt [n_rows, D] bf16 with row 2h = bf16(W[h]) and row 2h+1 =
// bf16(W[h] - bf16(W[h])); rows >= 2H are zero.
__global__ void split_weight_kernel(const float* __restrict__ w, int H, int D, int n_rows,
                                    __nv_bfloat16* __restrict__ wt) {
  const size_t n = static_cast<size_t>(n_rows) * D;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / D);
    const int k = static_cast<int>(i - static_cast<size_t>(r) * D);
    const int h = r >> 1;
    __nv_bfloat16 out = __float2bfloat16_rn(0.f);
    if (h < H) {
      const float x = w[static_cast<size_t>(h) * D + k];
      const __nv_bfloat16 hi = __float2bfloat16_rn(x);
      out = (r & 1) ? __float2bfloat16_rn(x - __bfloat162float(hi)) : hi;
    }
    wt[i] = out;
  }
}

// Linear scores of a few rows: CTA (h, g) computes scores[t, h] for the rows t
// of group g, sum_k x[t, k] * (hi[k] + lo[k]) with the two bf16 halves of
// weight row h (rows 2h and 2h + 1 of the split operand): each thread takes
// 8-value chunks k = 8c .. 8c + 7 (16-byte loads) in a strided loop, both
// products accumulated in fp32, then the CTA's partial sums are added
// through shared memory in a fixed order.
__global__ void __launch_bounds__(kGemvThreads) score_gemv_kernel(const uint16_t* __restrict__ x, int64_t ld_x,
                                                                  int n_tok, int D, const uint16_t* __restrict__ wt,
                                                                  int H, const float* __restrict__ bias,
                                                                  float* __restrict__ out) {
  __shared__ float red[kGemvThreads / 32][kGemvRows];
  const int h = blockIdx.x;
  const int r0 = blockIdx.y * kGemvRows;
  const int nr = min(kGemvRows, n_tok - r0);
  const uint4* hi = reinterpret_cast<const uint4*>(wt + static_cast<int64_t>(2 * h) * D);
  const uint4* lo = reinterpret_cast<const uint4*>(wt + static_cast<int64_t>(2 * h + 1) * D);
  float acc[kGemvRows];
#pragma unroll
  for (int r = 0; r < kGemvRows; ++r) acc[r] = 0.f;
  const int nch = D / 8;
  for (int c0 = threadIdx.x; c0 < nch; c0 += kGemvThreads * kGemvBatch) {
    uint4 a[kGemvBatch], bq[kGemvBatch];
#pragma unroll
    for (int u = 0; u < kGemvBatch; ++u) {
      const int c = c0 + u * kGemvThreads;
      a[u] = c < nch ? __ldg(hi + c) : make_uint4(0, 0, 0, 0);
      bq[u] = c < nch ? __ldg(lo + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int r = 0; r < kGemvRows; ++r) {
      if (r < nr) {
        uint4 xv[kGemvBatch];
#pragma unroll
        for (int u = 0; u < kGemvBatch; ++u) {
          const int c = c0 + u * kGemvThreads;
          xv[u] = c < nch ? __ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(r0 + r) * ld_x) + c)
                          : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kGemvBatch; ++u) {
          const uint32_t aw[4] = {a[u].x, a[u].y, a[u].z, a[u].w}, bw[4] = {bq[u].x, bq[u].y, bq[u].z, bq[u].w};
          const uint32_t xw[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float x0 = __uint_as_float(xw[i] << 16), x1 = __uint_as_float(xw[i] & 0xFFFF0000u);
            acc[r] = fmaf(x0, __uint_as_float(aw[i] << 16), acc[r]);
            acc[r] = fmaf(x0, __uint_as_float(bw[i] << 16), acc[r]);
            acc[r] = fmaf(x1, __uint_as_float(aw[i] & 0xFFFF0000u), acc[r]);
            acc[r] = fmaf(x1, __uint_as_float(bw[i] & 0xFFFF0000u), acc[r]);
          }
        }
      }
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int r = 0; r < kGemvRows; ++r) {
    float v = acc[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[warp][r] = v;
  }
  __syncthreads();
  if (threadIdx.x < nr) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kGemvThreads / 32; ++w) v += red[w][threadIdx.x];
    out[static_cast<int64_t>(r0 + threadIdx.x) * H + h] = v + (bias ? __ldg(bias + h) : 0.f);
  }
}

// KVzap-MLP scores of a few rows. CTA (g, r) takes hidden units 8g .. 8g + 7
// and rows 8r .. 8r + 7; warp w computes unit 8g + w (u[t, j] = sum_k x[t, k]
// w1[j, k] in fp32), the warp sums its lanes, and lane t applies the bias and
// the exact GELU. The CTA then writes part[g, t, h] = sum over its 8 units, in
// order, of z[t, j] * w2[h, j]; mlp_reduce_warp_kernel adds the groups'
// partials in order. The rows' x values pass through shared memory
// kMlpXPiece at a time (one cooperative load for the CTA's 8 warps), and a
// warp requests its w1 values for a piece in one go, the next piece's before
// it uses the current one: 16-byte chunk c of a piece goes to lane c % 32.
constexpr int kMlpXPiece = 2048;  // x values per row staged at a time
__global__ void __launch_bounds__(kGemvThreads) score_mlp_gemv_kernel(const uint16_t* __restrict__ x, int64_t ld_x,
                                                                      int n_tok, int D, const uint16_t* __restrict__ w1,
                                                                      const float* __restrict__ b1,
                                                                      const uint16_t* __restrict__ w2, int hidden, int H,
                                                                      float* __restrict__ part) {
  constexpr int kCh = kMlpXPiece / 8;  // 16-byte chunks of a row per piece
  constexpr int kPer = kCh / 32;       // a lane's chunks per piece
  __shared__ __align__(16) uint4 xs[kGemvRows][kCh];
  __shared__ float zs[kMlpGemvUnits][kGemvRows];
  const int g = blockIdx.x;
  const int r0 = blockIdx.y * kGemvRows;
  const int nr = min(kGemvRows, n_tok - r0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = g * kMlpGemvUnits + warp;
  const uint4* wr = reinterpret_cast<const uint4*>(w1 + static_cast<int64_t>(j) * D);
  float acc[kGemvRows];
#pragma unroll
  for (int r = 0; r < kGemvRows; ++r) acc[r] = 0.f;
  const int nch = D / 8;
  uint4 wa[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int c = lane + 32 * u;
    wa[u] = c < nch ? __ldg(wr + c) : make_uint4(0, 0, 0, 0);
  }
  for (int c0 = 0; c0 < nch; c0 += kCh) {
    __syncthreads();  // every warp is done with the previous piece
    for (int i = threadIdx.x; i < nr * kCh; i += kGemvThreads) {
      const int r = i / kCh, c = i - r * kCh;
      xs[r][c] = c0 + c < nch ? __ldg(reinterpret_cast<const uint4*>(x + static_cast<int64_t>(r0 + r) * ld_x) + c0 + c)
                              : make_uint4(0, 0, 0, 0);
    }
    uint4 wn[kPer];  // the next piece's weights, in flight while this piece is used
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int c = c0 + kCh + lane + 32 * u;
      wn[u] = c < nch ? __ldg(wr + c) : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kGemvRows; ++r) {
      if (r < nr) {
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const uint4 xv = xs[r][lane + 32 * u];
          const uint32_t aw[4] = {wa[u].x, wa[u].y, wa[u].z, wa[u].w};
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[r] = fmaf(__uint_as_float(xw[i] << 16), __uint_as_float(aw[i] << 16), acc[r]);
            acc[r] = fmaf(__uint_as_float(xw[i] & 0xFFFF0000u), __uint_as_float(aw[i] & 0xFFFF0000u), acc[r]);
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) wa[u] = wn[u];
  }
  float mine = 0.f;
#pragma unroll
  for (int r = 0; r < kGemvRows; ++r) {
    float v = acc[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == r) mine = v;
  }
  if (lane < nr) {
    const float u = mine + (b1 ? __ldg(b1 + j) : 0.f);
    zs[warp][lane] = 0.5f * u * (1.0f + erff(u * 0.70710678118654752f));
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < kGemvRows * H; idx += kGemvThreads) {
    const int t = idx / H, h = idx - t * H;
    if (t < nr) {
      float pv = 0.f;
#pragma unroll
      for (int jl = 0; jl < kMlpGemvUnits; ++jl) {
        const uint32_t wb = w2[static_cast<int64_t>(h) * hidden + g * kMlpGemvUnits + jl];
        pv = fmaf(zs[jl][t], __uint_as_float(wb << 16), pv);
      }
      part[(static_cast<int64_t>(g) * n_tok + r0 + t) * H + h] = pv;
    }
  }
}

// The few-row MLP path's partials: hidden / 8 groups per score. One warp per
// score: lane l loads groups l, l + 32, .. (all in flight), adds them in
// that order, then the warp adds its lanes' sums with a fixed butterfly.
__global__ void __launch_bounds__(256) mlp_reduce_warp_kernel(const float* __restrict__ part, int n_chunks, int64_t n,
                                                              int H, const float* __restrict__ b2,
                                                              float* __restrict__ scores) {
  const int64_t i = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (i >= n) return;  // uniform in the warp
  constexpr int kPer = 8;
  float v[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int c = lane + 32 * u;
    v[u] = c < n_chunks ? __ldg(part + c * n + i) : 0.f;
  }
  float s = 0.f;
  for (int c0 = 32 * kPer; c0 < n_chunks; c0 += 32) s += (c0 + lane < n_chunks) ? __ldg(part + (c0 + lane) * n + i) : 0.f;
#pragma unroll
  for (int u = 0; u < kPer; ++u) s += v[u];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) scores[i] = s + (b2 ? b2[i % H] : 0.f);
}

// scores[t, h] = sum_c part[c, t, h] + b2[h], chunks summed in order.
__global__ void mlp_reduce_kernel(const float* __restrict__ part, int n_chunks, int64_t n, int H,
                                  const float* __restrict__ b2, float* __restrict__ scores) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float s = b2 ? b2[i % H] : 0.f;
    for (int c = 0; c < n_chunks; ++c) s += part[c * n + i];
    scores[i] = s;
  }
}

bool make_tmap(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  return make_tmap_bf16(m, base, rows, cols, ld, box_rows, kBK);
}

int linear_bn(int H) {
  const int rows = 2 * H;
  return rows <= 16 ? 16 : rows <= 32 ? 32 : rows <= 64 ? 64 : 128;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// Per-instance launch set-up, done once per process: the shared-memory
// opt-in and the SM count of the device.
template <int BN, int EPI>
int score_grid_cap() {
  static const int nsm = [] {
    using C = ScoreCfg<BN>;
    if (cudaFuncSetAttribute(score_tc_kernel<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) !=
        cudaSuccess)
      return 0;
    return sm_count();
  }();
  return nsm;
}

template <int BN, int EPI>
kvp_status launch_score(const CUtensorMap& ta, const CUtensorMap& tb, const ScoreParams& p, cudaStream_t st) {
  using C = ScoreCfg<BN>;
  const int nsm = score_grid_cap<BN, EPI>();
  if (nsm <= 0) return KVP_ERR_CUDA;
  const int tiles = p.m_tiles * p.n_tiles;
  const int grid = tiles < nsm ? tiles : nsm;
  score_tc_kernel<BN, EPI><<<grid, score_threads<EPI>(), C::kSmem, st>>>(ta, tb, p);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" size_t kvp_score_split_weight_bytes(int d_model, int n_kv_heads) {
  if (d_model <= 0 || n_kv_heads <= 0) return 0;
  return static_cast<size_t>(linear_bn(n_kv_heads)) * d_model * 2;
}

extern "C" kvp_status kvp_score_split_weight(int d_model, int n_kv_heads, const float* w, void* w_split,
                                             size_t w_split_bytes, void* stream) {
  if (d_model <= 0 || n_kv_heads <= 0 || w == nullptr || w_split == nullptr) return KVP_ERR_INVALID;
  if (d_model % 8 != 0 || d_model > 65536 || n_kv_heads > 64) return KVP_ERR_UNSUPPORTED;
  if (w_split_bytes < kvp_score_split_weight_bytes(d_model, n_kv_heads)) return KVP_ERR_WORKSPACE;
  if (!aligned16(w_split)) return KVP_ERR_ALIGN;
  const int bn = linear_bn(n_kv_heads);
  const size_t nel = static_cast<size_t>(bn) * d_model;
  const int blocks = static_cast<int>((nel + 255) / 256 < 4096 ? (nel + 255) / 256 : 4096);
  split_weight_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      w, n_kv_heads, d_model, bn, static_cast<__nv_bfloat16*>(w_split));
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

extern "C" size_t kvp_score_workspace_bytes(int scorer, int64_t n_tok, int d_model, int n_kv_heads, int hidden) {
  if (n_tok < 0 || d_model <= 0 || n_kv_heads <= 0) return 0;
  if (scorer == KVP_SCORER_LINEAR) {
    return static_cast<size_t>(linear_bn(n_kv_heads)) * d_model * 2;
  }
  if (scorer == KVP_SCORER_LINEAR_SPLIT) return 0;
  if (scorer == KVP_SCORER_MLP) {
    if (hidden <= 0) return 0;
    const int chunks = n_tok <= kGemvMaxRows ? hidden / kMlpGemvUnits : hidden / kMlpBN;
    return static_cast<size_t>(chunks) * n_tok * n_kv_heads * sizeof(float);
  }
  return 0;
}

extern "C" kvp_status kvp_score(int scorer, int64_t n_tok, int d_model, int n_kv_heads, int hidden, const void* x,
                                int64_t ld_x, const void* w, const float* b, const void* w2, const float* b2,
                                float* scores, void* workspace, size_t workspace_bytes, int32_t* status,
                                void* stream) {
  if (scorer != KVP_SCORER_LINEAR && scorer != KVP_SCORER_MLP && scorer != KVP_SCORER_LINEAR_SPLIT)
    return KVP_ERR_INVALID;
  if (n_tok < 0 || d_model <= 0 || n_kv_heads <= 0) return KVP_ERR_INVALID;
  if (n_tok == 0) return KVP_OK;
  if (x == nullptr || w == nullptr || scores == nullptr) return KVP_ERR_INVALID;
  if (ld_x < d_model) return KVP_ERR_INVALID;
  if (d_model % 8 != 0 || d_model > 65536 || n_kv_heads > 64) return KVP_ERR_UNSUPPORTED;
  if (ld_x % 8 != 0 || !aligned16(x)) return KVP_ERR_ALIGN;
  if (scorer != KVP_SCORER_MLP && (w2 != nullptr || b2 != nullptr)) return KVP_ERR_INVALID;
  if (scorer == KVP_SCORER_LINEAR_SPLIT && !aligned16(w)) return KVP_ERR_ALIGN;
  if (n_tok > (int64_t(1) << 31) - 1) return KVP_ERR_UNSUPPORTED;
  const size_t need = kvp_score_workspace_bytes(scorer, n_tok, d_model, n_kv_heads, hidden);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return KVP_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KVP_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  ScoreParams p{};
  p.n_tok = static_cast<int>(n_tok);
  p.n_heads = n_kv_heads;
  p.m_tiles = static_cast<int>((n_tok + kBM - 1) / kBM);
  p.k_blocks = (d_model + kBK - 1) / kBK;
  p.status = status;

  CUtensorMap ta, tb;
  if (!make_tmap(&ta, x, n_tok, d_model, ld_x, kBM)) return KVP_ERR_CUDA;

  if (scorer == KVP_SCORER_LINEAR || scorer == KVP_SCORER_LINEAR_SPLIT) {
    const int bn = linear_bn(n_kv_heads);
    const void* wt = w;
    if (scorer == KVP_SCORER_LINEAR) {
      const kvp_status s = kvp_score_split_weight(d_model, n_kv_heads, static_cast<const float*>(w), workspace,
                                                  workspace_bytes, stream);
      if (s != KVP_OK) return s;
      wt = workspace;
    }
    if (n_tok <= kGemvMaxRows) {  // a decode step's few new tokens
      const dim3 grid(n_kv_heads, static_cast<unsigned>((n_tok + kGemvRows - 1) / kGemvRows));
      score_gemv_kernel<<<grid, kGemvThreads, 0, st>>>(static_cast<const uint16_t*>(x), ld_x, static_cast<int>(n_tok),
                                                       d_model, static_cast<const uint16_t*>(wt), n_kv_heads, b,
                                                       scores);
      return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
    }
    if (!make_tmap(&tb, wt, bn, d_model, d_model, bn)) return KVP_ERR_CUDA;
    p.n_tiles = 1;
    p.bias = b;
    p.out = scores;
    switch (bn) {
      case 16: return launch_score<16, kEpiLinear>(ta, tb, p, st);
      case 32: return launch_score<32, kEpiLinear>(ta, tb, p, st);
      case 64: return launch_score<64, kEpiLinear>(ta, tb, p, st);
      default: return launch_score<128, kEpiLinear>(ta, tb, p, st);
    }
  }

  // MLP
  if (w2 == nullptr) return KVP_ERR_INVALID;
  if (hidden <= 0 || hidden % kMlpBN != 0 || n_kv_heads > kMlpMaxH) return KVP_ERR_UNSUPPORTED;
  if (!aligned16(w)) return KVP_ERR_ALIGN;
  float* part = static_cast<float*>(workspace);
  const int64_t n = n_tok * n_kv_heads;
  const int blocks = static_cast<int>((n + 255) / 256 < 8192 ? (n + 255) / 256 : 8192);
  if (n_tok <= kGemvMaxRows) {  // a decode step's few new tokens
    const dim3 grid(hidden / kMlpGemvUnits, static_cast<unsigned>((n_tok + kGemvRows - 1) / kGemvRows));
    score_mlp_gemv_kernel<<<grid, kGemvThreads, 0, st>>>(static_cast<const uint16_t*>(x), ld_x,
                                                         static_cast<int>(n_tok), d_model,
                                                         static_cast<const uint16_t*>(w), b,
                                                         static_cast<const uint16_t*>(w2), hidden, n_kv_heads, part);
    if (cudaGetLastError() != cudaSuccess) return KVP_ERR_CUDA;
    const int64_t wblocks = (n * 32 + 255) / 256;
    mlp_reduce_warp_kernel<<<static_cast<unsigned>(wblocks), 256, 0, st>>>(part, hidden / kMlpGemvUnits, n,
                                                                           n_kv_heads, b2, scores);
    return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
  }
  if (!make_tmap(&tb, w, hidden, d_model, d_model, kMlpBN)) return KVP_ERR_CUDA;
  p.n_tiles = hidden / kMlpBN;
  p.hidden = hidden;
  p.bias = b;
  p.w2 = static_cast<const uint16_t*>(w2);
  p.out = part;
  kvp_status s = launch_score<kMlpBN, kEpiMlp>(ta, tb, p, st);
  if (s != KVP_OK) return s;
  mlp_reduce_kernel<<<blocks, 256, 0, st>>>(part, p.n_tiles, n, n_kv_heads, b2, scores);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}
