// kvp_threshold: each (b, h)'s threshold as an order statistic of its own
// scores, chosen on the device.
//
// KVzap summary, "실제 적용": entries with low scores are removed, but the
// pages leave open how "low" is set. This library's reading is a per-(b, h)
// quantile: tau[b, h] = the element of rank k = floor(q * (n - 1)) (from 0,
// ascending) of that head's n scores, NaN ranked above +inf.
//
// Radix select, most significant byte first. Every float maps to a 32-bit key
// whose unsigned order is the float order (NaN last). Pass p (0..3) histograms
// byte 3 - p of the keys that agree with the (b, h)'s prefix of the p bytes
// chosen so far; the last CTA of each (b, head group) to finish a pass picks
// the byte whose cumulative count passes the remaining rank and extends the
// prefix. After four passes the prefix is the key of the answer.
//
// A CTA takes a chunk of positions of one b and up to 32 heads, reads them as
// one contiguous run of the [B, n, H] score array, counts into a shared
// histogram per head and adds its non-zero bins to the global histogram with
// atomics. The pass's last CTA is found with a counter, no waiting: every CTA
// fences its histogram atomics and bumps the counter; the one that sees the
// final count does the selection.
#include <algorithm>
#include <cmath>

#include "kvp_common.cuh"

namespace kvp {
namespace {

constexpr int kHeadsPerCta = 32;
constexpr int kBins = 256;
constexpr int kPasses = 4;
constexpr int kThrThreads = 256;
constexpr int kThrUnroll = 8;      // loads in flight per thread
constexpr int kMinRows = 64;       // positions per CTA at least

KVP_DEV uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0xffffffffu;  // NaN ranks above +inf
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
KVP_DEV float key_value(uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k); }

// Workspace (uint32): histogram [B*H][256], prefix [B*H], remaining rank
// [B*H], pass counters [4][B][head groups]. Zeroed at the start of each call
// except prefix and rank, which are written before they are read; a pass's
// selecting CTA clears the histogram bins it has read.
struct ThrWs {
  uint32_t* hist;
  uint32_t* prefix;
  uint32_t* krem;
  uint32_t* done;
};
size_t thr_ws_words(int B, int H) {
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t G = (H + kHeadsPerCta - 1) / kHeadsPerCta;
  return BH * kBins + 2 * BH + kPasses * static_cast<size_t>(B) * G;
}
ThrWs thr_carve(void* ws, int B, int H) {
  uint32_t* p = static_cast<uint32_t*>(ws);
  const size_t BH = static_cast<size_t>(B) * H;
  return ThrWs{p, p + BH * kBins, p + BH * kBins + BH, p + BH * kBins + 2 * BH};
}

// VEC = 4 reads four adjacent heads of a row as one 16-byte load (H a
// multiple of 4, scores 16-byte aligned); VEC = 1 reads one score at a time.
// kFixed (VEC = 4, and the loads of a row divide the block): every thread
// keeps the same four heads for the whole chunk, with their prefixes in
// registers, and steps down the rows.
template <int VEC, bool kFixed>
__global__ void __launch_bounds__(kThrThreads, 4) select_pass(int pass, int H, int n, int rows, uint32_t k0,
                                                           const float* __restrict__ scores, ThrWs ws,
                                                           float* __restrict__ tau) {
  __shared__ uint32_t hist[kHeadsPerCta * kBins];
  __shared__ uint32_t pre_s[kHeadsPerCta];
  __shared__ int last_s;
  const int b = blockIdx.y, g = blockIdx.z;
  const int h0 = g * kHeadsPerCta;
  const int hn = min(kHeadsPerCta, H - h0);
  const int shift = 24 - 8 * pass;
  const int64_t bh0 = static_cast<int64_t>(b) * H + h0;
  for (int i = threadIdx.x; i < hn * kBins; i += kThrThreads) hist[i] = 0;
  if (threadIdx.x < hn) pre_s[threadIdx.x] = pass > 0 ? ws.prefix[bh0 + threadIdx.x] : 0u;
  __syncthreads();

  // ---- count this chunk's keys that agree with the prefix
  const int t0 = blockIdx.x * rows;
  const int t1 = min(n, t0 + rows);
  const int hv = hn / VEC;          // loads per row
  const int nv = (t1 - t0) * hv;    // loads in the chunk
  const float* base = scores + (static_cast<int64_t>(b) * n + t0) * H + h0;
  if constexpr (kFixed) {
    const int jc = threadIdx.x % hv;  // this thread's heads: 4 jc .. 4 jc + 3
    const int dr = kThrThreads / hv;  // rows between two of its loads
    const int nrows = t1 - t0;
    uint32_t pre[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) pre[c] = pre_s[4 * jc + c];
    uint32_t* hj = hist + 4 * jc * kBins;
    for (int r0 = threadIdx.x / hv; r0 < nrows; r0 += dr * kThrUnroll) {
      float4 x[kThrUnroll];
#pragma unroll
      for (int u = 0; u < kThrUnroll; ++u) {  // all loads first
        const int r = r0 + u * dr;
        x[u] = r < nrows ? __ldg(reinterpret_cast<const float4*>(base + static_cast<int64_t>(r) * H + 4 * jc))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kThrUnroll; ++u) {
        if (r0 + u * dr < nrows) {
          const float f[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t key = order_key(f[c]);
            if (pass == 0 || (key >> (shift + 8)) == pre[c]) atomicAdd(&hj[c * kBins + ((key >> shift) & 0xffu)], 1u);
          }
        }
      }
    }
  } else {
  // load e = r * hv + j (row t0 + r, heads h0 + VEC j ..); (r, j) of this
  // thread's next load is advanced by kThrThreads loads without a division
  const int dr = kThrThreads / hv, dj = kThrThreads - dr * hv;
  int r = threadIdx.x / hv, j = threadIdx.x - r * hv;
  for (int e0 = threadIdx.x; e0 < nv; e0 += kThrThreads * kThrUnroll) {
    float v[kThrUnroll][VEC];
    int jj[kThrUnroll];
#pragma unroll
    for (int u = 0; u < kThrUnroll; ++u) {  // all loads first
      jj[u] = j;
      if (e0 + u * kThrThreads < nv) {
        const float* src = base + static_cast<int64_t>(r) * H + VEC * j;
        if constexpr (VEC == 4) {
          const float4 x = __ldg(reinterpret_cast<const float4*>(src));
          v[u][0] = x.x;
          v[u][1] = x.y;
          v[u][2] = x.z;
          v[u][3] = x.w;
        } else {
          v[u][0] = __ldg(src);
        }
      }
      r += dr;
      j += dj;
      if (j >= hv) {
        j -= hv;
        ++r;
      }
    }
#pragma unroll
    for (int u = 0; u < kThrUnroll; ++u) {
      if (e0 + u * kThrThreads < nv) {
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
          const int hh = VEC * jj[u] + c;
          const uint32_t key = order_key(v[u][c]);
          if (pass == 0 || (key >> (shift + 8)) == pre_s[hh]) atomicAdd(&hist[hh * kBins + ((key >> shift) & 0xffu)], 1u);
        }
      }
    }
  }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < hn * kBins; i += kThrThreads) {
    const uint32_t c = hist[i];
    if (c) atomicAdd(&ws.hist[bh0 * kBins + i], c);
  }
  fence_acq_rel_gpu();  // this thread's histogram additions before the counter
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t prev = atomicAdd(&ws.done[(static_cast<int64_t>(pass) * gridDim.y + b) * gridDim.z + g], 1u);
    last_s = prev == gridDim.x - 1;
    if (last_s) fence_acq_rel_gpu();  // every CTA's additions before the reads below
  }
  __syncthreads();
  if (!last_s) return;

  // ---- the last CTA: warp w takes heads w, w + 8, .. and picks, per head,
  // the byte holding rank krem; all of a warp's bin loads are issued first
  constexpr int kHW = kHeadsPerCta / (kThrThreads / 32);  // heads per warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t c[kHW][8];
  uint32_t kr[kHW];
#pragma unroll
  for (int hw = 0; hw < kHW; ++hw) {
    const int jh = warp + hw * (kThrThreads / 32);
    if (jh < hn) {
      const uint32_t* hb = ws.hist + (bh0 + jh) * kBins + lane * 8;
#pragma unroll
      for (int i = 0; i < 8; ++i) c[hw][i] = __ldcg(hb + i);
      kr[hw] = pass > 0 ? ws.krem[bh0 + jh] : k0;
    }
  }
#pragma unroll
  for (int hw = 0; hw < kHW; ++hw) {
    const int jh = warp + hw * (kThrThreads / 32);
    if (jh >= hn) break;  // uniform in the warp
    const int64_t bh = bh0 + jh;
    // every CTA's counts for this pass are in: clear the bins for the next
    // pass (a later launch on the same stream)
    uint32_t* hb = ws.hist + bh * kBins + lane * 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) hb[i] = 0u;
    uint32_t sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) sum += c[hw][i];
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned m = __ballot_sync(0xffffffffu, incl > kr[hw]);
    if (m != 0 && lane == __ffs(m) - 1) {
      uint32_t before = incl - sum;
      int d = 0;
#pragma unroll
      for (int i = 0; i < 7; ++i)
        if (d == i && before + c[hw][i] <= kr[hw]) {
          before += c[hw][i];
          d = i + 1;
        }
      const uint32_t pre = (pre_s[jh] << 8) | static_cast<uint32_t>(lane * 8 + d);
      ws.prefix[bh] = pre;
      ws.krem[bh] = kr[hw] - before;
      if (pass == kPasses - 1) tau[bh] = key_value(pre);
    }
  }
}

}  // namespace
}  // namespace kvp

using namespace kvp;

extern "C" size_t kvp_threshold_workspace_bytes(int batch, int n_kv_heads) {
  if (batch <= 0 || n_kv_heads <= 0) return 0;
  return thr_ws_words(batch, n_kv_heads) * sizeof(uint32_t);
}

extern "C" kvp_status kvp_threshold(int batch, int n_kv_heads, int n_pos, const float* scores, double q, float* tau,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (batch <= 0 || n_kv_heads <= 0 || n_pos <= 0) return KVP_ERR_INVALID;
  if (scores == nullptr || tau == nullptr) return KVP_ERR_INVALID;
  if (!(q >= 0.0 && q <= 1.0)) return KVP_ERR_INVALID;  // NaN fails too
  const int G = (n_kv_heads + kHeadsPerCta - 1) / kHeadsPerCta;
  if (batch > 65535 || G > 65535) return KVP_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(n_pos) * kHeadsPerCta + kThrThreads * kThrUnroll > 0x7fffffff) return KVP_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < kvp_threshold_workspace_bytes(batch, n_kv_heads))
    return KVP_ERR_WORKSPACE;
  const uint32_t k0 = static_cast<uint32_t>(std::floor(q * static_cast<double>(n_pos - 1)));
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return KVP_ERR_CUDA;
  // about four CTAs per SM (what 60 registers a thread allow) over all
  // (b, head group) pairs, kMinRows positions each at least
  const int64_t units = static_cast<int64_t>(batch) * G;
  const int64_t want = std::max<int64_t>(1, (4 * static_cast<int64_t>(sms) + units - 1) / units);
  const int64_t chunks0 = std::min<int64_t>(want, (n_pos + kMinRows - 1) / kMinRows);
  const int rows = static_cast<int>((n_pos + chunks0 - 1) / chunks0);
  const int chunks = (n_pos + rows - 1) / rows;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ThrWs ws = thr_carve(workspace, batch, n_kv_heads);
  if (cudaMemsetAsync(workspace, 0, thr_ws_words(batch, n_kv_heads) * sizeof(uint32_t), st) != cudaSuccess)
    return KVP_ERR_CUDA;
  const dim3 grid(chunks, batch, G);
  const bool vec4 = n_kv_heads % 4 == 0 && (reinterpret_cast<uintptr_t>(scores) & 15u) == 0;
  // fixed heads per thread when every head group's row of float4 loads (8
  // for a full group, (H mod 32) / 4 for the last) divides the block
  const int hv_last = (n_kv_heads - (G - 1) * kHeadsPerCta) / 4;
  const bool fixed = vec4 && kThrThreads % (kHeadsPerCta / 4) == 0 && hv_last > 0 && kThrThreads % hv_last == 0;
  for (int p = 0; p < kPasses; ++p) {
    if (fixed)
      select_pass<4, true><<<grid, kThrThreads, 0, st>>>(p, n_kv_heads, n_pos, rows, k0, scores, ws, tau);
    else if (vec4)
      select_pass<4, false><<<grid, kThrThreads, 0, st>>>(p, n_kv_heads, n_pos, rows, k0, scores, ws, tau);
    else
      select_pass<1, false><<<grid, kThrThreads, 0, st>>>(p, n_kv_heads, n_pos, rows, k0, scores, ws, tau);
  }
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}
