/*
 * kvp.h - C ABI of libkvp, KV-cache pruning at decode time on one GB300
 * (sm_103a).
 *
 * The path, step by step, and the pages that define it:
 *
 *   kvp_score        "NVIDIA가 AI 메모리 압축 신기술 KVzap 오픈소스 공개!" (KVzap
 *                    summary), 핵심 내용 정리 -> "KVzap의 구조", "실제 적용": a
 *                    small surrogate (one linear layer, or a 2-layer MLP) maps
 *                    each token's hidden state to one score per KV head.
 *   kvp_mask         same page, "실제 적용": low-scoring entries are removed,
 *                    the most recent 128 tokens are always kept; and
 *                    "Nvidia의 새로운 기술, 정확도 손실 없이 LLM 추론 비용을 8배
 *                    절감" (DMS article), "지연 삭제 (Delayed Eviction)": a token
 *                    flagged for eviction stays for a delay window first.
 *   kvp_compact      DeInfer summary (gist.science, arXiv 2604.17709), "나.
 *                    페이지드 KV 캐시 및 CUDA Graph 통합": a preparation pass
 *                    builds a remapping index list, a copy pass gathers the
 *                    kept rows into a compact buffer with fixed addresses.
 *   kvp_append       the decode-time side of the same rules: the new token is
 *                    scored once and written into a reserved slot.
 *   kvp_decode_attn  DMS article, "DMS 작동 방식" step 5: standard attention
 *                    over what is kept; here split-KV single-query GQA decode.
 *   kvp_*_latent, kvp_decode_attn_mla
 *                    DMS article, "주요 요점" and "앞으로의 전망": the same
 *                    pruning over MLA's single latent cache.
 *
 * Conventions shared by every entry point:
 *   - Pointers named in a comment as "device" are CUDA device addresses
 *     (any allocator; torch tensors work). The library never allocates,
 *     frees or keeps a device buffer: the caller owns every buffer,
 *     including workspace (size from the matching *_workspace_bytes call).
 *     The one exception is kvp_compact_noalloc, whose scratch is a fixed
 *     array in the library's device memory (see its declaration).
 *   - Every call is asynchronous and ordered on `stream` (a cudaStream_t,
 *     NULL = legacy default stream). Nothing synchronises the host.
 *   - Host-side argument checks return a status at once and launch nothing.
 *   - Errors found on the device (page budget exhausted, a bounded wait that
 *     gave up) are recorded in `status`, a device int32 the caller zeroes:
 *     kernels only ever replace a 0 there with a nonzero kvp_status code, so
 *     it holds the first error. Outputs of a call that recorded an error are
 *     unspecified. `status` may be NULL where a call cannot fail on device.
 *   - bf16 means IEEE-754 binary32 truncated to its top 16 bits (the
 *     `__nv_bfloat16` / torch.bfloat16 format). Rows are 16-byte aligned.
 *   - Positions count tokens from 0; `now` is the position of the token being
 *     decoded, whose own K/V is already in the cache.
 */
#ifndef KVP_H
#define KVP_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVP_API __attribute__((visibility("default")))
#else
#define KVP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvp_status {
  KVP_OK = 0,
  KVP_ERR_INVALID = 1,      /* null pointer, negative size, inconsistent shapes */
  KVP_ERR_ALIGN = 2,        /* a pointer or stride breaks the 16-byte rule */
  KVP_ERR_CAPACITY = 3,     /* page pool, page table or reserve too small (device) */
  KVP_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  KVP_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up (device) */
  KVP_ERR_UNSUPPORTED = 6,  /* shape outside what the kernels handle */
  KVP_ERR_WORKSPACE = 7,    /* workspace pointer NULL or smaller than required */
  KVP_ERR_BOUNDS = 8        /* a page id or count read on the device is out of range (device);
                               the access is skipped, never performed */
} kvp_status;

enum { KVP_SCORER_LINEAR = 0, KVP_SCORER_MLP = 1, KVP_SCORER_LINEAR_SPLIT = 2 };
enum { KVP_MASK_KVZAP = 0, KVP_MASK_DMS = 1 };

#define KVP_PAGE_TOKENS 16            /* rows per page of the compacted cache */
#define KVP_WINDOW_DEFAULT 128        /* KVzap: the last 128 tokens are always kept */
#define KVP_EXPIRE_NEVER 2147483647   /* expire value of an entry kept for good */

/* Human-readable name of a status code (static string). */
KVP_API const char* kvp_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
KVP_API int kvp_version(void);

/* kvp_selftest_wait - exercises the bounded wait that every kernel of this
 * library puts on its mbarriers (no page describes it; it is the library's
 * failure handling). One warp waits on an mbarrier that nothing arrives on;
 * after limit_ns of wall time (the %globaltimer clock, checked every 1024
 * probes; 0 gives up at the second check) the wait gives up, KVP_ERR_TIMEOUT
 * is recorded in `status` and the kernel returns, leaving the context usable.
 *
 * limit_ns   at most 10 s (else KVP_ERR_INVALID)
 * status     device int32 (required), as in every other call
 * waited_us  device uint32 (or NULL): microseconds the wait lasted
 */
KVP_API kvp_status kvp_selftest_wait(uint64_t limit_ns, int32_t* status, uint32_t* waited_us, void* stream);

/* ------------------------------------------------------------------------ */
/* kvp_score - KVzap surrogate scores (KVzap summary, "KVzap의 구조",
 * "실제 적용").
 *
 *   LINEAR: scores[t, h] = sum_k x[t, k] * w[h, k] + b[h]
 *   MLP:    scores[t, h] = sum_j GELU(sum_k x[t, k] * w[j, k] + b[j]) * w2[h, j] + b2[h]
 *           with the exact (erf) GELU and the hidden activations in fp32.
 *
 * n_tok      rows of x (any >= 0; 0 is a no-op)
 * d_model    D, a multiple of 8, <= 65536
 * n_kv_heads H, 1..64
 * hidden     MLP hidden width, a multiple of 256 (ignored for LINEAR)
 * x          device bf16 [n_tok, D], row stride ld_x elements (multiple of 8,
 *            >= D), base 16-byte aligned
 * w          LINEAR: device fp32 [H, D] (a linear layer's weight layout)
 *            LINEAR_SPLIT: device bf16, the operand kvp_score_split_weight
 *                    wrote for this (D, H), 16-byte aligned
 *            MLP:    device bf16 W1 [hidden, D]
 * b          LINEAR: device fp32 [H] or NULL;  MLP: device fp32 b1 [hidden] or NULL
 * w2         MLP: device bf16 [H, hidden];  LINEAR: must be NULL
 * b2         MLP: device fp32 [H] or NULL;  LINEAR: must be NULL
 * scores     device fp32 [n_tok, H] (output, token-major)
 * workspace  device, >= kvp_score_workspace_bytes(...) bytes, 256-byte aligned
 *            (LINEAR_SPLIT needs none: NULL and 0 are accepted; MLP holds
 *            fp32 partial scores per chunk of the hidden layer: hidden / 256
 *            chunks, or hidden / 8 up to 64 rows)
 *
 * The dense contraction runs on the tcgen05 tensor cores: LINEAR splits the
 * fp32 weight into two bf16 halves (hi + lo) so that the products keep ~16
 * mantissa bits of w; accumulation is fp32 throughout. Up to 64 rows (the
 * new tokens of a decode step) the scorers run the same products on the CUDA
 * cores instead (a single 128-row tensor-core tile would leave the whole
 * weight to one CTA): LINEAR and LINEAR_SPLIT over one CTA per head and group
 * of 8 rows, MLP over one CTA per 8 hidden units and group of 8 rows, its
 * partial scores summed in a fixed order. LINEAR does that split
 * on every call (one small kernel); a caller whose weight does not change
 * between calls (a decode loop: the weight is the layer's) splits it once with
 * kvp_score_split_weight and passes LINEAR_SPLIT; the scores are identical.
 */
KVP_API size_t kvp_score_workspace_bytes(int scorer, int64_t n_tok, int d_model, int n_kv_heads, int hidden);
KVP_API kvp_status kvp_score(int scorer, int64_t n_tok, int d_model, int n_kv_heads, int hidden,
                     const void* x, int64_t ld_x, const void* w, const float* b,
                     const void* w2, const float* b2, float* scores,
                     void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/* kvp_score_split_weight - the KVzap-Linear weight in the form the scorer's
 * tensor cores take (no page describes this step; it is how this library
 * keeps fp32 weights on bf16 tensor cores): w_split is bf16
 * [rows, D] with rows = kvp_score_split_weight_bytes / (2 D), row 2h =
 * bf16(w[h]) (round to nearest even), row 2h+1 = bf16(w[h] - bf16(w[h])), and
 * rows >= 2H zero. w device fp32 [H, D]; w_split device, >= the size below,
 * 16-byte aligned. D a multiple of 8, H 1..64.
 */
KVP_API size_t kvp_score_split_weight_bytes(int d_model, int n_kv_heads);
KVP_API kvp_status kvp_score_split_weight(int d_model, int n_kv_heads, const float* w, void* w_split,
                                          size_t w_split_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* kvp_mask - keep/evict decision per (batch, kv head, position) (KVzap
 * summary "실제 적용"; DMS article "지연 삭제").
 *
 * Each entry gets expire = the first step at which it is no longer cached:
 *   KVZAP: expire = (score >= tau[b,h]) ? KVP_EXPIRE_NEVER : pos + window
 *          (NaN scores count as low)
 *   DMS:   expire = (flag_step < 0) ? KVP_EXPIRE_NEVER
 *                                   : max(flag_step + delay, pos + window)
 * and is present at step `now` iff now < expire. pos = pos0 + index.
 *
 * mode       KVP_MASK_KVZAP or KVP_MASK_DMS
 * scores     KVZAP: device fp32 [B, n_pos, H] (kvp_score output with
 *            n_tok = B*n_pos);  DMS: NULL
 * tau        KVZAP: device fp32 [B, H];  DMS: NULL
 * flag_step  DMS: device int32 [B, H, n_pos], -1 = never flagged; KVZAP: NULL
 * window     >= 0 (KVP_WINDOW_DEFAULT = 128);  delay >= 0 (DMS)
 * expire     device int32 [B, H, n_pos] (output, required)
 * keep_bits  device uint32 [B, H, ceil(n_pos/32)] (output or NULL); bit i of
 *            word w is position index 32*w + i; bits past n_pos are 0
 * count      device int32 [B, H] (output or NULL): present entries
 */
KVP_API kvp_status kvp_mask(int mode, int batch, int n_kv_heads, int n_pos, int pos0,
                    const float* scores, const float* tau, const int32_t* flag_step,
                    int window, int delay, int now,
                    int32_t* expire, uint32_t* keep_bits, int32_t* count, void* stream);

/* kvp_threshold - each (b, h)'s KVzap threshold chosen on the device as an
 * order statistic of its own scores. The KVzap summary ("실제 적용") removes
 * low-scoring entries but leaves open how "low" is set; this entry point
 * takes the plainest per-head reading, a quantile of the head's scores.
 *
 * tau[b, h] = the element of rank k = floor(q * (n_pos - 1)) (counted from 0,
 * ascending) among scores[b, t, h], t in [0, n_pos); NaN ranks above +inf, so
 * it is chosen only when fewer than n_pos - k scores are numbers. q = 0 gives
 * the minimum, q = 1 the maximum, q = 0.5 at odd n_pos the median. Exact:
 * the result is one of the inputs, bit for bit (-0.0 and +0.0 are one value).
 *
 * scores     device fp32 [B, n_pos, H] (kvp_score's output layout)
 * q          in [0, 1], else KVP_ERR_INVALID
 * tau        device fp32 [B, H] (output)
 * workspace  device, kvp_threshold_workspace_bytes(batch, n_kv_heads) bytes
 *            (1 KiB per (b, h) plus a little); zeroed by the call itself
 * Limits: batch <= 65535 and n_pos * 32 below 2^31, else KVP_ERR_UNSUPPORTED.
 * Radix select over the scores' order-preserving 32-bit keys: four passes of
 * 8 bits, each one read of the scores (the later ones mostly from L2).
 */
KVP_API size_t kvp_threshold_workspace_bytes(int batch, int n_kv_heads);
KVP_API kvp_status kvp_threshold(int batch, int n_kv_heads, int n_pos, const float* scores, double q,
                                 float* tau, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* kvp_compact - gather the entries present at `now` into 16-row pages
 * (DeInfer summary, "나. 페이지드 KV 캐시 및 CUDA Graph 통합": remapping index
 * list, then a copy into a compact fixed-address buffer).
 *
 * For every (b, h), in b-major then h-minor order, the present positions are
 * taken in ascending order; (b, h) receives n = ceil((count + reserve) / 16)
 * consecutive pages starting right after the previous (b, h)'s pages. Slot j
 * of (b, h) is row j % 16 of page page_table[b, h, j / 16].
 *
 * Source (dense): k_src, v_src device bf16, element (b, t, h, e) at
 *   b*stride_b + t*stride_t + h*stride_h + e (strides in elements, multiples
 *   of 8; e contiguous), t in [0, n_pos).
 * expire     device int32 [B, H, n_pos] (kvp_mask output)
 * reserve    free slots kept after the survivors of each (b, h) for kvp_append
 * Outputs (all device):
 *   k_pool, v_pool   bf16 [n_pages_cap, 16, head_dim]; rows past count in a
 *                    (b, h)'s last page are zero
 *   expire_pool      int32 [n_pages_cap, 16]; the entry's expire, 0 in unused rows
 *   page_table       int32 [B, H, max_pages]; page ids, -1 past the (b, h)'s pages
 *   remap            int32 [B, H, max_pages*16]; source position of slot j, -1
 *                    past count
 *   count            int32 [B, H]
 * A budget overflow records KVP_ERR_CAPACITY in `status` (required).
 * head_dim is 64 or 128.
 */
KVP_API size_t kvp_compact_workspace_bytes(int batch, int n_kv_heads, int n_pos);
KVP_API kvp_status kvp_compact(int batch, int n_kv_heads, int head_dim, int n_pos,
                       const void* k_src, const void* v_src,
                       int64_t stride_b, int64_t stride_t, int64_t stride_h,
                       const int32_t* expire, int now, int reserve,
                       void* k_pool, void* v_pool, int32_t* expire_pool, int n_pages_cap,
                       int32_t* page_table, int max_pages, int32_t* remap, int32_t* count,
                       void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/* kvp_compact_masked - kvp_mask and kvp_compact in one pass, with no expire
 * array in between (the mask is fused into the preparation and copy passes
 * of the DeInfer summary's compaction, "나. 페이지드 KV 캐시 및 CUDA Graph
 * 통합"; the keep rules are KVzap's "실제 적용" and the DMS article's "지연
 * 삭제 (Delayed Eviction)").
 *
 * Every output is bit-identical to kvp_mask(mode, batch, n_kv_heads, n_pos,
 * pos0 = 0, scores, tau, flag_step, window, delay, now, expire, ...) followed
 * by kvp_compact(..., expire, now, reserve, ...) on the same K/V: entry t of
 * the dense source is position t, its expire is derived from its score (or
 * flag step) where it is needed, and expire_pool receives it for the kept
 * entries. No dense expire, keep bits or per-position output is written.
 *
 * mode, scores, tau, flag_step, window, delay: as in kvp_mask (scores device
 *   fp32 [B, n_pos, H] and tau [B, H] for KVP_MASK_KVZAP; flag_step device
 *   int32 [B, H, n_pos] for KVP_MASK_DMS; the other mode's pointers NULL).
 * Every other argument, output, workspace size
 * (kvp_compact_workspace_bytes) and error is kvp_compact's.
 * n_pos + window + delay must stay below KVP_EXPIRE_NEVER (else
 * KVP_ERR_INVALID).
 */
KVP_API kvp_status kvp_compact_masked(int mode, int batch, int n_kv_heads, int head_dim, int n_pos,
                       const void* k_src, const void* v_src,
                       int64_t stride_b, int64_t stride_t, int64_t stride_h,
                       const float* scores, const float* tau, const int32_t* flag_step,
                       int window, int delay, int now, int reserve,
                       void* k_pool, void* v_pool, int32_t* expire_pool, int n_pages_cap,
                       int32_t* page_table, int max_pages, int32_t* remap, int32_t* count,
                       void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/* kvp_compact_quant - the fp8 tier of "quantize instead of drop" (BeaconKV
 * article "LLM 추론 비용 혁신: '비콘KV'가 ...", core idea and first FAQ answer:
 * important entries keep full precision, the others are compressed lossily,
 * for instance by low-precision quantization). The article fixes no format;
 * this library's reading is:
 *
 *   - entry t of the dense source goes to the fp8 tier iff
 *     tau_q[b,h] <= scores[b,t,h] < tau[b,h] (a NaN score never does); with
 *     tau_q <= tau this is the band that the bf16 tier (kvp_mask with tau)
 *     keeps only while it is in the window;
 *   - its K row and its V row are each stored as FP8 E4M3 codes with one fp32
 *     scale per row: scale = amax(|row|) / 448 and inv = 448 / amax(|row|)
 *     (IEEE divisions), code = E4M3(x * inv) (fp32 product, rounded to
 *     nearest even, saturating to +-448); an all-zero row has scale 0 and
 *     zero codes; value = code * scale;
 *   - it is visible to kvp_decode_attn_two_tier from step t + window on, the
 *     step its bf16 copy leaves the window, so at any step an entry is in one
 *     tier at most.
 *
 * With DMS flags (mode KVP_MASK_DMS) the entries quantized are the flagged
 * ones (flag_step >= 0: quantize instead of evict), visible from
 * max(flag + delay, t + window) on, the step their bf16 copy is gone.
 *
 * Selected entries are laid out like kvp_compact's survivors: ascending
 * position, (b, h) in b-major / h-minor order, ceil((count + reserve) / 16)
 * consecutive pages each.
 * Source, strides, reserve, workspace (kvp_compact_workspace_bytes) and
 * errors: as kvp_compact. KVP_MASK_KVZAP: scores device fp32 [B, n_pos, H]
 * (may be NULL when n_pos is 0), tau and tau_q device fp32 [B, H], flag_step
 * NULL. KVP_MASK_DMS: flag_step device int32 [B, H, n_pos] and delay as in
 * kvp_mask, scores / tau / tau_q NULL.
 * Outputs (all device):
 *   kq_pool, vq_pool  uint8 [n_pages_cap, 16, head_dim] E4M3 codes, 16-byte
 *                     aligned; rows past count in a (b, h)'s last page zero
 *   meta_pool         int32 [n_pages_cap, 3, 16]: per slot the start step, the
 *                     K scale and the V scale (fp32 bit patterns); 0 in unused rows
 *   page_table, remap, count: as kvp_compact (remap = source position)
 */
KVP_API kvp_status kvp_compact_quant(int mode, int batch, int n_kv_heads, int head_dim, int n_pos,
                       const void* k_src, const void* v_src,
                       int64_t stride_b, int64_t stride_t, int64_t stride_h,
                       const float* scores, const float* tau, const float* tau_q, const int32_t* flag_step,
                       int window, int delay, int reserve,
                       void* kq_pool, void* vq_pool, int32_t* meta_pool, int n_pages_cap,
                       int32_t* page_table, int max_pages, int32_t* remap, int32_t* count,
                       void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/* kvp_append_quant - the decode-time side of the fp8 tier: the token at
 * position `pos` (k_new, v_new device bf16 [B, H, head_dim], 16-byte aligned)
 * goes into slot count[b, h] of its (b, h)'s fp8 pages iff
 * tau_q[b, h] <= score[b, h] < tau[b, h] (KVP_MASK_KVZAP; device fp32 [B, H],
 * the score the token got for the bf16 tier's kvp_append), start = pos +
 * window; or iff flag_step[b, h] >= 0 (KVP_MASK_DMS; device int32 [B, H]),
 * start = max(flag + delay, pos + window). It is quantized exactly as
 * kvp_compact_quant does; remap and count grow by one. The slot must be one of the pages the compaction reserved, else
 * KVP_ERR_CAPACITY is recorded in `status` and that (b, h) is left as it is.
 * Pools and tables: as kvp_compact_quant writes them.
 */
KVP_API kvp_status kvp_append_quant(int mode, int batch, int n_kv_heads, int head_dim, int pos,
                       const void* k_new, const void* v_new,
                       const float* score, const float* tau, const float* tau_q, const int32_t* flag_step,
                       int window, int delay,
                       void* kq_pool, void* vq_pool, int32_t* meta_pool, int n_pages_cap,
                       const int32_t* page_table, int max_pages, int32_t* remap, int32_t* count,
                       int32_t* status, void* stream);

/* kvp_compact_noalloc - kvp_compact for callers that cannot allocate device
 * memory. No page describes this entry point; it is a convenience of this
 * library. Some hosts hand a library only the tensors of the operation and no
 * way to get more GPU memory: a runtime that owns every device allocation
 * through its own pool, or a plugin interface with no workspace hook, or a
 * latency-critical loop where cudaMalloc (which can synchronise the device)
 * is not allowed. This variant takes the same arguments as kvp_compact minus
 * the workspace and allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library call. Its scratch is a fixed array of
 * KVP_COMPACT_NOALLOC_SCRATCH_BYTES (1 MiB) in the library's device memory,
 * which every GPU that loads the library keeps until the process exits.
 *
 * Limits and rules:
 *   - kvp_compact_workspace_bytes(batch, n_kv_heads, n_pos) must not exceed
 *     KVP_COMPACT_NOALLOC_SCRATCH_BYTES, else KVP_ERR_WORKSPACE and nothing
 *     is launched (2*B*H*ceil(n_pos/128) + B*H + 1 words of 4 bytes, e.g.
 *     B*H = 128 at 8192 positions needs 66 KB).
 *   - The first call on a device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *   - All calls share the one array per device and it keeps the last call's
 *     contents; calls that overlap on the GPU (other streams, other host
 *     threads) race on it. Nothing in it needs clearing between calls.
 */
#define KVP_COMPACT_NOALLOC_SCRATCH_BYTES (1u << 20)
KVP_API kvp_status kvp_compact_noalloc(int batch, int n_kv_heads, int head_dim, int n_pos,
                                       const void* k_src, const void* v_src,
                                       int64_t stride_b, int64_t stride_t, int64_t stride_h,
                                       const int32_t* expire, int now, int reserve,
                                       void* k_pool, void* v_pool, int32_t* expire_pool, int n_pages_cap,
                                       int32_t* page_table, int max_pages, int32_t* remap, int32_t* count,
                                       int32_t* status, void* stream);

/* kvp_compact_paged - the same compaction with a paged cache (as written by
 * kvp_compact / kvp_append) as the source: slots j < src_count[b, h] whose
 * expire_pool entry is present at `now` are kept, in slot order, and carry
 * their remap position and expire value over. Source and destination must
 * not overlap (use two pools and swap them). A source page id outside
 * [0, src_n_pages_cap) records KVP_ERR_BOUNDS and its slots count as absent.
 */
KVP_API size_t kvp_compact_paged_workspace_bytes(int batch, int n_kv_heads, int src_max_pages);
KVP_API kvp_status kvp_compact_paged(int batch, int n_kv_heads, int head_dim,
                             const void* src_k_pool, const void* src_v_pool,
                             const int32_t* src_expire_pool, int src_n_pages_cap,
                             const int32_t* src_page_table,
                             int src_max_pages, const int32_t* src_remap, const int32_t* src_count,
                             int now, int reserve,
                             void* k_pool, void* v_pool, int32_t* expire_pool, int n_pages_cap,
                             int32_t* page_table, int max_pages, int32_t* remap, int32_t* count,
                             void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/* ------------------------------------------------------------------------ */
/* kvp_append - decode step: write the new token (position `pos`) of every
 * (b, h) into slot count[b, h], with its expire value from the same rules as
 * kvp_mask (KVZAP: score[b, h] vs tau[b, h]; DMS: flag_step[b, h]), then
 * increment count. A (b, h) with no free slot left records
 * KVP_ERR_CAPACITY in `status` (required) and is left unchanged.
 *
 * k_new, v_new  device bf16 [B, H, head_dim]
 * score, tau    KVZAP: device fp32 [B, H] each;  DMS: NULL
 * flag_step     DMS: device int32 [B, H];  KVZAP: NULL
 * pools (n_pages_cap pages), page_table, remap, count: as written by
 *               kvp_compact; a page id outside [0, n_pages_cap) records
 *               KVP_ERR_BOUNDS and nothing is written for that (b, h).
 */
KVP_API kvp_status kvp_append(int mode, int batch, int n_kv_heads, int head_dim, int pos,
                      const void* k_new, const void* v_new,
                      const float* score, const float* tau, const int32_t* flag_step,
                      int window, int delay,
                      void* k_pool, void* v_pool, int32_t* expire_pool, int n_pages_cap,
                      const int32_t* page_table, int max_pages, int32_t* remap, int32_t* count,
                      int32_t* status, void* stream);

/* kvp_append_devpos - kvp_append with the position read from device memory:
 * pos_dev is a device int32 (4-byte aligned) holding the position of the
 * token being appended when the call runs on the stream. Everything else is
 * kvp_append's. A decode step built from this call and
 * kvp_decode_attn_devpos takes no per-step host value, so it can be captured
 * once in a CUDA graph and replayed for every step, the caller advancing the
 * position in device memory between replays (the fixed-address replay of the
 * DeInfer summary, "나. 페이지드 KV 캐시 및 CUDA Graph 통합"). A position below 0
 * or with pos + window + delay >= KVP_EXPIRE_NEVER records KVP_ERR_INVALID in
 * `status` and nothing is written.
 */
KVP_API kvp_status kvp_append_devpos(int mode, int batch, int n_kv_heads, int head_dim, const int32_t* pos_dev,
                                     const void* k_new, const void* v_new,
                                     const float* score, const float* tau, const int32_t* flag_step,
                                     int window, int delay,
                                     void* k_pool, void* v_pool, int32_t* expire_pool, int n_pages_cap,
                                     const int32_t* page_table, int max_pages, int32_t* remap, int32_t* count,
                                     int32_t* status, void* stream);

/* ------------------------------------------------------------------------ */
/* kvp_decode_attn - single-query attention over the kept entries (DMS
 * article, "DMS 작동 방식" step 5: standard attention kernels on the pruned
 * cache).
 *
 *   out[b, j] = sum_i softmax_i(scale * q[b, j] . k_i) v_i
 *
 * over the slots i < count[b, h] of kv head h = j / (Hq / H) whose expire is
 * greater than `now`. An empty set gives a zero row.
 *
 * The pages of all (b, h) are split evenly over the warps of a persistent
 * grid (split-KV along pages, whatever the per-head survivor counts); partial
 * softmax states of a (b, h) that spans several warps are merged in fp32 by
 * the last of them to finish. At 1 and 2 query heads per kv head the page
 * math runs on the CUDA cores in fp32; at 4 and 8 it runs on the tensor
 * cores (bf16 products with fp32 accumulation, the softmax weights entering
 * the P.V product as a bf16 hi + lo pair, about 16 bits each).
 *
 * q          device bf16 [B, Hq, head_dim];  Hq a multiple of H, Hq/H in {1,2,4,8},
 *            B*H <= 4096
 * pools (n_pages_cap pages), expire_pool, page_table (width max_pages), count:
 *            as kvp_compact writes them. count is clamped to max_pages*16; a
 *            page id outside [0, n_pages_cap) records KVP_ERR_BOUNDS in
 *            `status` (may be NULL) and that page counts as empty.
 * scale      > 0, or 0 for 1/sqrt(head_dim)
 * out        device fp32 [B, Hq, head_dim], 16-byte aligned
 * grid_limit 0 = the default grid (one CTA per SM); > 0 caps the number of
 *            CTAs (so the same inputs can be split differently)
 * workspace  device, >= kvp_decode_attn_workspace_bytes(...), 16-byte aligned;
 *            holds the partial states and per-(b, h) arrival counters. It
 *            must be zero-filled before its first use (cudaMemset of the whole
 *            buffer); every call that records no error in `status` leaves it
 *            ready for the next call (each merge resets its counter), so no
 *            per-call clearing runs. After a call that recorded an error, zero
 *            it again. Calls that share a workspace must not overlap on the GPU.
 */
KVP_API size_t kvp_decode_attn_workspace_bytes(int batch, int n_q_heads, int n_kv_heads, int head_dim);
KVP_API kvp_status kvp_decode_attn(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                   const void* q, const void* k_pool, const void* v_pool,
                                   const int32_t* expire_pool, int n_pages_cap,
                                   const int32_t* page_table, int max_pages,
                                   const int32_t* count, int now, float scale, float* out,
                                   int grid_limit, void* workspace, size_t workspace_bytes,
                                   int32_t* status, void* stream);

/* kvp_decode_attn_devpos - kvp_decode_attn with the decode position read
 * from device memory: now_dev is a device int32 (4-byte aligned) read when
 * the call runs on the stream (see kvp_append_devpos). Everything else,
 * including the workspace, is kvp_decode_attn's.
 */
KVP_API kvp_status kvp_decode_attn_devpos(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                          const void* q, const void* k_pool, const void* v_pool,
                                          const int32_t* expire_pool, int n_pages_cap,
                                          const int32_t* page_table, int max_pages,
                                          const int32_t* count, const int32_t* now_dev, float scale, float* out,
                                          int grid_limit, void* workspace, size_t workspace_bytes,
                                          int32_t* status, void* stream);

/* kvp_decode_attn_lse - kvp_decode_attn that also returns each output row's
 * log-sum-exp (DMS article, "DMS 작동 방식": the standard attention over what is
 * kept, whose softmax normaliser this is):
 *
 *   lse[b, j] = ln sum_i exp(scale * q[b, j] . k_i)
 *
 * over the same present slots (-inf when there are none, with a zero output
 * row). Attention over a set of slots split into parts, each part's rows
 * with its lse, is recovered exactly by kvp_attn_merge: a long sequence's
 * pages can be attended in parts (separate caches, or separate devices whose
 * (out, lse) rows the caller gathers) and merged.
 *
 * lse        device fp32 [B, Hq] (output, required, 4-byte aligned). Every
 *            other argument, and the workspace rules: as kvp_decode_attn.
 */
KVP_API kvp_status kvp_decode_attn_lse(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                       const void* q, const void* k_pool, const void* v_pool,
                                       const int32_t* expire_pool, int n_pages_cap,
                                       const int32_t* page_table, int max_pages,
                                       const int32_t* count, int now, float scale, float* out, float* lse,
                                       int grid_limit, void* workspace, size_t workspace_bytes,
                                       int32_t* status, void* stream);

/* kvp_attn_merge - one attention output from n_parts partial ones over
 * disjoint parts of the same slots, each normalised over its own part
 * (kvp_decode_attn_lse's out and lse):
 *
 *   lse[r] = ln sum_p exp(lses[p, r]),   out[r] = sum_p exp(lses[p, r] - lse[r]) outs[p, r]
 *
 * A part with lse -inf (no slots) weighs nothing; a row with no slots in any
 * part comes out zero with lse -inf. lses must be finite or -inf.
 *
 * outs       device fp32 [n_parts, rows, head_dim], 16-byte aligned
 * lses       device fp32 [n_parts, rows]
 * out        device fp32 [rows, head_dim] (output), 16-byte aligned; it may
 *            not overlap outs
 * lse_out    device fp32 [rows] (output) or NULL
 * head_dim   a multiple of 4; rows >= 0 (0: nothing to do); n_parts >= 1
 */
KVP_API kvp_status kvp_attn_merge(int n_parts, int64_t rows, int head_dim, const float* outs, const float* lses,
                                  float* out, float* lse_out, void* stream);

/* kvp_decode_attn_two_tier - kvp_decode_attn over both tiers of "quantize
 * instead of drop" (BeaconKV article; the fp8 tier as kvp_compact_quant
 * writes it):
 *
 *   out[b, j] = sum_i softmax_i(scale * q[b, j] . k_i) v_i
 *
 * over the bf16 slots i < count[b, h] with expire > now, and the fp8 slots
 * i < count_q[b, h] with start <= now, whose k and v are their E4M3 codes
 * times the row's scale. Both tiers' pages of a (b, h) form one list, split
 * over the persistent grid like kvp_decode_attn's.
 *
 * Arguments up to `count` and from `now` on: as kvp_decode_attn (same
 * workspace size and rules). On the tensor cores (every G, unless the
 * pools pass 2^31 rows) a fp8 page's codes are turned into fp16 (exactly)
 * and multiplied by the query converted to fp16, which is exact for bf16
 * values of magnitude 2^-17 .. 65504; its softmax weights, times the V row
 * scale, enter the
 * P.V product as one fp16 value each (relative error <= 2^-11, subnormal
 * below 2^-14). kq_pool, vq_pool, meta_pool (16-byte aligned),
 * n_pages_cap_q, page_table_q (width max_pages_q), count_q: the fp8 tier as
 * kvp_compact_quant writes it. A fp8 page id outside [0, n_pages_cap_q)
 * records KVP_ERR_BOUNDS and the page counts as empty.
 */
KVP_API kvp_status kvp_decode_attn_two_tier(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                   const void* q, const void* k_pool, const void* v_pool,
                                   const int32_t* expire_pool, int n_pages_cap,
                                   const int32_t* page_table, int max_pages, const int32_t* count,
                                   const void* kq_pool, const void* vq_pool, const int32_t* meta_pool,
                                   int n_pages_cap_q, const int32_t* page_table_q, int max_pages_q,
                                   const int32_t* count_q, int now, float scale, float* out,
                                   int grid_limit, void* workspace, size_t workspace_bytes,
                                   int32_t* status, void* stream);

/* ------------------------------------------------------------------------ */
/* MLA latent cache. The DMS article ("주요 요점"; "앞으로의 전망") says the method
 * applies to Multi-Head Latent Attention, whose cache holds one latent row per
 * token, shared by every query head: c_t (KVP_MLA_LATENT_DIM values of
 * compressed KV) followed by the shared rotary key (KVP_MLA_ROPE_DIM values).
 * The article gives no further detail; this library's reading is that a
 * token's latent row is kept or dropped as a whole, by one score (or DMS
 * flag) per token, under the same rules as a kv head's entry (kvp_mask), and
 * that the pruned cache is read by MLA's absorbed decode attention.
 *
 * A latent cache is a paged cache with one "kv head" and one pool: pool bf16
 * [n_pages_cap, 16, row_dim], row_dim = KVP_MLA_LATENT_DIM + KVP_MLA_ROPE_DIM
 * (the only supported width; anything else is KVP_ERR_UNSUPPORTED);
 * expire_pool, page_table [B, max_pages], remap [B, max_pages*16] and count
 * [B] as kvp_compact writes them with n_kv_heads = 1.
 */
#define KVP_MLA_LATENT_DIM 512
#define KVP_MLA_ROPE_DIM 64

/* kvp_compact_latent - kvp_compact_masked for a latent cache: the present
 * latent rows of every batch element into 16-row pages.
 *
 * lat_src    device bf16, row (b, t) at b*stride_b + t*stride_t (elements,
 *            multiples of 8), row_dim contiguous values, t in [0, n_pos)
 * scores     KVZAP: device fp32 [B, n_pos] (kvp_score's output with one
 *            head); tau device fp32 [B];  DMS: NULL, NULL
 * flag_step  DMS: device int32 [B, n_pos];  KVZAP: NULL
 * Outputs, reserve, window, delay, now, status: kvp_compact_masked's with
 * n_kv_heads = 1 and the one pool; rows past count in a batch element's
 * last page are zero. Workspace: kvp_compact_workspace_bytes(batch, 1, n_pos).
 */
KVP_API kvp_status kvp_compact_latent(int mode, int batch, int row_dim, int n_pos, const void* lat_src,
                                      int64_t stride_b, int64_t stride_t,
                                      const float* scores, const float* tau, const int32_t* flag_step,
                                      int window, int delay, int now, int reserve,
                                      void* pool, int32_t* expire_pool, int n_pages_cap,
                                      int32_t* page_table, int max_pages, int32_t* remap, int32_t* count,
                                      void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/* kvp_compact_latent_paged - kvp_compact_paged for a latent cache (the
 * source and destination are latent caches; they share no buffer).
 * Workspace: kvp_compact_paged_workspace_bytes(batch, 1, src_max_pages).
 */
KVP_API kvp_status kvp_compact_latent_paged(int batch, int row_dim, const void* src_pool,
                                            const int32_t* src_expire_pool, int src_n_pages_cap,
                                            const int32_t* src_page_table, int src_max_pages,
                                            const int32_t* src_remap, const int32_t* src_count,
                                            int now, int reserve, void* pool, int32_t* expire_pool, int n_pages_cap,
                                            int32_t* page_table, int max_pages, int32_t* remap, int32_t* count,
                                            void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/* kvp_append_latent - kvp_append for a latent cache: the new token's latent
 * row of every batch element into slot count[b].
 *
 * lat_new       device bf16 [B, row_dim]
 * score, tau    KVZAP: device fp32 [B] each;  DMS: NULL
 * flag_step     DMS: device int32 [B];  KVZAP: NULL
 * Everything else, and the errors, as kvp_append.
 */
KVP_API kvp_status kvp_append_latent(int mode, int batch, int row_dim, int pos, const void* lat_new,
                                     const float* score, const float* tau, const int32_t* flag_step,
                                     int window, int delay, void* pool, int32_t* expire_pool, int n_pages_cap,
                                     const int32_t* page_table, int max_pages, int32_t* remap, int32_t* count,
                                     int32_t* status, void* stream);

/* kvp_decode_attn_mla - MLA's absorbed decode attention over a pruned latent
 * cache:
 *
 *   out[b, j] = sum_t softmax_t(scale * q[b, j] . row_t) row_t[0 : latent_dim]
 *
 * over the slots t < count[b] whose expire is greater than `now`. q[b, j] is
 * query head j's absorbed query: its no-position part multiplied by that
 * head's key up-projection (latent_dim values), then its rotary part
 * (rope_dim values). The result is the head's attention-weighted compressed
 * value, to which the caller applies the head's value up-projection. An
 * empty set gives a zero row.
 *
 * Work is cut into units (a tile of query heads of one batch element), and
 * each unit's pages into n_splits equal slices. Both products run on the
 * tensor cores with bf16 operands and fp32 accumulation:
 *   up to 32 query heads   tiles of 16 heads, one CTA per (unit, slice)
 *                          (mma.sync); the softmax weights enter the
 *                          weighted sum as a bf16 hi + lo pair
 *   33 to 64 query heads   one tile of 64 heads, one CTA per (unit, slice)
 *                          (mma.sync), weights as a hi + lo pair
 *   from 65 query heads    tiles of 128 heads on tcgen05 (tensor memory):
 *                          a cluster of four CTAs per (unit, slice), one
 *                          per quarter of the latent_dim output values,
 *                          sharing each page's copies; each weight is
 *                          rounded to bf16 once (relative error <= 2^-9 per
 *                          weight; the normaliser sums the unrounded
 *                          weights, so an output value is off by at most
 *                          about 2^-9 times the largest |row value|)
 * With more than one slice, a second kernel launched by the same call merges
 * the slices in fp32, one CTA per (unit, head).
 *
 * latent_dim, rope_dim  KVP_MLA_LATENT_DIM and KVP_MLA_ROPE_DIM (else
 *            KVP_ERR_UNSUPPORTED)
 * q          device bf16 [B, n_q_heads, latent_dim + rope_dim], n_q_heads >= 1
 * pool, expire_pool, page_table (width max_pages), count: a latent cache;
 *            count is clamped to max_pages*16, a page id outside
 *            [0, n_pages_cap) records KVP_ERR_BOUNDS in `status` (may be
 *            NULL) and the page counts as empty. n_pages_cap*16 < 2^31.
 * scale      > 0, or 0 for 1/sqrt(latent_dim + rope_dim)
 * out        device fp32 [B, n_q_heads, latent_dim], 16-byte aligned
 * n_splits   slices per unit, 1..64; 0 picks one from the current device's
 *            SM count (as many as fill one wave of CTAs: two per SM for
 *            16-head tiles, one for the others; at least 1)
 * workspace  device, >= kvp_decode_attn_mla_workspace_bytes(batch,
 *            n_q_heads, n_splits) (asked on the device that runs the call
 *            when n_splits = 0), 16-byte aligned; every call writes what it
 *            reads, so it needs no clearing. Calls that share a workspace
 *            must not overlap on the GPU.
 */
KVP_API size_t kvp_decode_attn_mla_workspace_bytes(int batch, int n_q_heads, int n_splits);
KVP_API kvp_status kvp_decode_attn_mla(int batch, int n_q_heads, int latent_dim, int rope_dim, const void* q,
                                       const void* pool, const int32_t* expire_pool, int n_pages_cap,
                                       const int32_t* page_table, int max_pages, const int32_t* count, int now,
                                       float scale, float* out, int n_splits, void* workspace,
                                       size_t workspace_bytes, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVP_H */
