"""Oracle for pruned-KV decode: a plain, slow, obviously correct CPU reference.

TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import this module. The library's GPU path
never calls it and shares no code with it.

Everything here is float64 numpy (bf16 inputs are widened exactly). The
method is taken step by step from these pages:

[DMS]     "Nvidia의 새로운 기술, 정확도 손실 없이 LLM 추론 비용을 8배 절감"
          (euno.news rendering of a VentureBeat article on Dynamic Memory
          Sparsification).
[KVzap]   "NVIDIA가 AI 메모리 압축 신기술 KVzap 오픈소스 공개!" (max5.ai summary
          of a MarkTechPost article).
[DeInfer] gist.science summary of arXiv 2604.17709 (DeInfer), section
          "2. 제안 방법 → 나. 페이지드 KV 캐시 및 CUDA Graph 통합".
[BeaconKV] "LLM 추론 비용 혁신: '비콘KV'가 KV 캐시 메모리 4배 절감하며 성능까지
          잡는 비결" (jiinsi.com paper briefing).

Steps and where they come from:

1. score   [KVzap, 핵심 내용 정리 → "KVzap의 구조", "실제 적용"]: a surrogate
           maps each token's hidden state to one score per KV head; either a
           single linear layer or a 2-layer MLP.
2. mask    [KVzap, "실제 적용"]: low-scoring entries are removed, the most
           recent 128 tokens are always kept.
           [DMS, "지연 삭제 (Delayed Eviction)"]: a token flagged for eviction
           stays for a delay window, then is removed.
3. compact [DeInfer, 나. → 준비 단계 / 그래프 재생 단계]: scan the logical
           blocks, produce a remapping index list, copy the kept rows into a
           compact buffer with fixed addresses (16-token pages here).
4. attend  [DMS, "DMS 작동 방식" step 5 and "메모리의 미래"]: standard
           attention over what is kept (single-query decode, GQA).
5. quantize [BeaconKV]: instead of dropping the less important entries,
           keep them in low precision (an fp8 tier, see section 5).
6. latent  [DMS, "주요 요점" / "앞으로의 전망"]: the same pruning over MLA's
           single latent cache (section 6).

Readings where the pages are silent (each is listed with its reason in the
repository's design notes): scores are raw surrogate outputs compared to a
per-(batch, kv-head) threshold tau, kept iff score >= tau; the window is the
last ``window`` positions counted from ``now`` inclusive; an entry flagged at
step f with delay d is present up to step f+d-1 and gone at f+d; GQA uses
contiguous query-head groups; softmax scale is 1/sqrt(head_dim); an empty kept
set gives a zero output; the MLP activation is the exact (erf) GELU and its
hidden activations stay in full precision.
"""
from __future__ import annotations

import math

import numpy as np
from scipy.special import erf

NEVER = 2**31 - 1     # expire value of an entry that is kept forever
PAGE = 16             # rows per page of the compacted cache
WINDOW = 128          # [KVzap, "실제 적용"]: the most recent 128 tokens are always kept


class CapacityError(RuntimeError):
    """The compacted cache does not fit the page budget the caller gave."""


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# 1. Scoring  [KVzap, 핵심 내용 정리 → "KVzap의 구조", "실제 적용"]
# ---------------------------------------------------------------------------

def score_linear(x_bits: np.ndarray, w: np.ndarray, bias: np.ndarray | None = None) -> np.ndarray:
    """KVzap-Linear: s[t, h] = sum_k x[t, k] * W[h, k] + b[h].

    x_bits: bf16 bits [n_tok, D]; w: float [H, D] (one row per KV head, the
    layout of a linear layer's weight); bias: [H] or None. Returns float64
    [n_tok, H].
    """
    x = widen_bf16(x_bits)
    s = x @ np.asarray(w, dtype=np.float64).T
    if bias is not None:
        s = s + np.asarray(bias, dtype=np.float64)[None, :]
    return s


def gelu(u: np.ndarray) -> np.ndarray:
    """Exact GELU: u * Phi(u) = u/2 * (1 + erf(u / sqrt 2))."""
    return 0.5 * u * (1.0 + erf(u / math.sqrt(2.0)))


def score_mlp(x_bits, w1_bits, w2_bits, b1=None, b2=None) -> np.ndarray:
    """KVzap-MLP: s = GELU(x W1^T + b1) W2^T + b2, hidden kept in float64.

    x_bits [n_tok, D], w1_bits [hidden, D], w2_bits [H, hidden], all bf16 bits.
    """
    x = widen_bf16(x_bits)
    u = x @ widen_bf16(w1_bits).T
    if b1 is not None:
        u = u + np.asarray(b1, dtype=np.float64)[None, :]
    z = gelu(u)
    s = z @ widen_bf16(w2_bits).T
    if b2 is not None:
        s = s + np.asarray(b2, dtype=np.float64)[None, :]
    return s


# ---------------------------------------------------------------------------
# 2. Masking  [KVzap, "실제 적용"]  [DMS, "지연 삭제 (Delayed Eviction)"]
#
# Each entry gets an "expire" step: the first decode step at which it is no
# longer in the cache. At step `now` an entry is present iff now < expire.
# ---------------------------------------------------------------------------

def expire_kvzap(score, tau, pos, window: int = WINDOW):
    """KVzap rule: an entry whose score is at least tau is kept for good;
    otherwise it survives only while it is one of the last `window` positions,
    i.e. while now < pos + window. NaN scores are treated as low."""
    score = np.asarray(score)
    pos = np.asarray(pos, dtype=np.int64)
    keep_forever = score >= tau
    return np.where(keep_forever, NEVER, pos + window).astype(np.int64)


def expire_dms(flag_step, pos, delay: int, window: int = WINDOW):
    """DMS rule with delayed eviction: an entry never flagged (flag_step < 0)
    is kept; one flagged at step f is gone at step f + delay, but not before it
    leaves the recent window (pos + window)."""
    f = np.asarray(flag_step, dtype=np.int64)
    pos = np.asarray(pos, dtype=np.int64)
    return np.where(f < 0, NEVER, np.maximum(f + delay, pos + window)).astype(np.int64)


def present(expire, now: int):
    return np.asarray(now) < np.asarray(expire)


def mask(expire_bht: np.ndarray, now: int):
    """From expire [B, H, T] -> (keep bool [B,H,T], keep_bits uint32 [B,H,ceil(T/32)],
    count int [B,H]). Bit i of word w stands for position 32*w + i."""
    keep = present(expire_bht, now)
    B, H, T = keep.shape
    nw = (T + 31) // 32
    bits = np.zeros((B, H, nw), dtype=np.uint64)
    for i in range(32):
        col = keep[:, :, i::32]
        bits[:, :, : col.shape[2]] |= col.astype(np.uint64) << np.uint64(i)
    return keep, bits.astype(np.uint32), keep.sum(axis=2).astype(np.int64)


def mask_kvzap(scores_bth, tau_bh, now: int, window: int = WINDOW, pos0: int = 0):
    """Scores laid out [B, T, H] (token-major, as the scorer emits them)."""
    s = np.asarray(scores_bth)
    B, T, H = s.shape
    pos = pos0 + np.arange(T)
    exp = expire_kvzap(s.transpose(0, 2, 1), np.asarray(tau_bh)[:, :, None], pos[None, None, :], window)
    return (exp,) + mask(exp, now)


def mask_dms(flag_step_bht, now: int, delay: int, window: int = WINDOW, pos0: int = 0):
    f = np.asarray(flag_step_bht)
    B, H, T = f.shape
    pos = pos0 + np.arange(T)
    exp = expire_dms(f, pos[None, None, :], delay, window)
    return (exp,) + mask(exp, now)


def threshold_at_quantile(scores_bth: np.ndarray, q) -> np.ndarray:
    """Per-(b, h) threshold: the lower order statistic at index floor(q*(T-1))
    of that head's T scores, rounded to float32 (the threshold is a float32
    input of the masking step). A harness choice, not part of the method.
    q is one quantile for every head, or one per kv head (shape [H]), as for
    heads with their own keep rates."""
    s = np.sort(np.asarray(scores_bth, dtype=np.float64), axis=1)
    B, T, H = s.shape
    if np.ndim(q) == 0:
        return s[:, int(math.floor(q * (T - 1))), :].astype(np.float32)
    k = np.floor(np.asarray(q, dtype=np.float64) * (T - 1)).astype(np.int64)
    assert k.shape == (H,)
    return s[:, k, np.arange(H)].astype(np.float32)


# ---------------------------------------------------------------------------
# 3. Compaction  [DeInfer, 나. 페이지드 KV 캐시 및 CUDA Graph 통합]
#
# Preparation: list the kept rows of every (b, h) in ascending position (the
# remapping index list). Copy: gather those rows into 16-row pages of a
# compact pool. Pages are handed out in (b-major, h-minor) order, each (b, h)
# getting ceil((count + reserve) / 16) contiguous pages; `reserve` free slots
# per (b, h) take later appends without moving anything.
# ---------------------------------------------------------------------------

class PagedCache:
    """The compacted cache: pools [n_pages, 16, d] (bf16 bits), expire_pool
    [n_pages, 16], page_table [B, H, max_pages] (-1 = unused), remap
    [B, H, max_pages*16] (source position of slot j, -1 = unused), count [B, H]."""

    def __init__(self, batch, n_kv_heads, head_dim, n_pages_cap, max_pages):
        self.k_pool = np.zeros((n_pages_cap, PAGE, head_dim), dtype=np.uint16)
        self.v_pool = np.zeros((n_pages_cap, PAGE, head_dim), dtype=np.uint16)
        self.expire_pool = np.zeros((n_pages_cap, PAGE), dtype=np.int64)
        self.page_table = np.full((batch, n_kv_heads, max_pages), -1, dtype=np.int64)
        self.remap = np.full((batch, n_kv_heads, max_pages * PAGE), -1, dtype=np.int64)
        self.count = np.zeros((batch, n_kv_heads), dtype=np.int64)
        self.pages_used = 0

    def slot_rows(self, b, h, slots):
        """(page, row) of slots j of (b, h)."""
        slots = np.asarray(slots, dtype=np.int64)
        return self.page_table[b, h, slots // PAGE], slots % PAGE


def _pages_for(n: int, reserve: int) -> int:
    return (n + reserve + PAGE - 1) // PAGE


def _fill(out: PagedCache, b, h, k_rows, v_rows, expire, positions, reserve):
    n = len(positions)
    npg = _pages_for(n, reserve)
    if npg > out.page_table.shape[2] or out.pages_used + npg > out.k_pool.shape[0]:
        raise CapacityError(f"(b={b}, h={h}) needs {npg} pages")
    base = out.pages_used
    out.page_table[b, h, :npg] = base + np.arange(npg)
    j = np.arange(n)
    out.k_pool[base + j // PAGE, j % PAGE] = k_rows
    out.v_pool[base + j // PAGE, j % PAGE] = v_rows
    out.expire_pool[base + j // PAGE, j % PAGE] = expire
    out.remap[b, h, :n] = positions
    out.count[b, h] = n
    out.pages_used += npg


def compact_dense(k_bits, v_bits, expire_bht, now, reserve, n_pages_cap, max_pages) -> PagedCache:
    """Dense K/V [B, T, H, d] + expire [B, H, T] -> PagedCache of the entries
    present at step `now`."""
    B, T, H, d = k_bits.shape
    out = PagedCache(B, H, d, n_pages_cap, max_pages)
    for b in range(B):
        for h in range(H):
            pos = np.nonzero(present(expire_bht[b, h], now))[0]
            _fill(out, b, h, k_bits[b, pos, h], v_bits[b, pos, h], expire_bht[b, h, pos], pos, reserve)
    return out


def compact_paged(src: PagedCache, now, reserve, n_pages_cap, max_pages) -> PagedCache:
    """Re-compaction of an existing paged cache: keep the slots present at
    `now`, in slot order, into a fresh set of pages."""
    B, H, _ = src.page_table.shape
    d = src.k_pool.shape[2]
    out = PagedCache(B, H, d, n_pages_cap, max_pages)
    for b in range(B):
        for h in range(H):
            slots = np.arange(src.count[b, h])
            pg, row = src.slot_rows(b, h, slots)
            e = src.expire_pool[pg, row]
            sel = present(e, now)
            pg, row = pg[sel], row[sel]
            _fill(out, b, h, src.k_pool[pg, row], src.v_pool[pg, row], e[sel],
                  src.remap[b, h, slots[sel]], reserve)
    return out


def append(cache: PagedCache, k_new_bits, v_new_bits, pos: int, expire_new):
    """Decode step: the new token's k/v [B, H, d] go into slot count[b, h] of
    its own (b, h) pages, with its expire step; raises if the reserve is used
    up."""
    B, H = cache.count.shape
    for b in range(B):
        for h in range(H):
            j = int(cache.count[b, h])
            p = j // PAGE
            if p >= cache.page_table.shape[2] or cache.page_table[b, h, p] < 0:
                raise CapacityError(f"(b={b}, h={h}) has no free slot")
            page = cache.page_table[b, h, p]
            cache.k_pool[page, j % PAGE] = k_new_bits[b, h]
            cache.v_pool[page, j % PAGE] = v_new_bits[b, h]
            cache.expire_pool[page, j % PAGE] = expire_new[b, h]
            cache.remap[b, h, j] = pos
            cache.count[b, h] = j + 1


# ---------------------------------------------------------------------------
# 4. Attention over the kept entries  [DMS, "DMS 작동 방식" step 5]
# ---------------------------------------------------------------------------

def _softmax_attend(q, K, V, scale):
    """One query q [dk] over rows K [n, dk], V [n, dv] (float64). Two-pass
    softmax; an empty set gives a zero row of V's width."""
    if K.shape[0] == 0:
        return np.zeros(V.shape[1])
    logits = (K @ q) * scale
    m = logits.max()
    w = np.exp(logits - m)
    return (w @ V) / w.sum()


def decode_attention(q_bits, cache: PagedCache, now: int, scale: float | None = None) -> np.ndarray:
    """o[b, j] = softmax_i(q[b, j] . k_i * scale) v_i over the slots i of
    (b, h = j // g) present at `now`; g = Hq / H. Returns float32 [B, Hq, d]."""
    B, Hq, d = q_bits.shape
    H = cache.count.shape[1]
    g = Hq // H
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    q = widen_bf16(q_bits)
    out = np.zeros((B, Hq, d))
    for b in range(B):
        for h in range(H):
            slots = np.arange(cache.count[b, h])
            pg, row = cache.slot_rows(b, h, slots)
            sel = present(cache.expire_pool[pg, row], now)
            K = widen_bf16(cache.k_pool[pg[sel], row[sel]])
            V = widen_bf16(cache.v_pool[pg[sel], row[sel]])
            for j in range(h * g, (h + 1) * g):
                out[b, j] = _softmax_attend(q[b, j], K, V, scale)
    return out.astype(np.float32)


def decode_attention_lse(q_bits, cache: PagedCache, now: int, scale: float | None = None):
    """decode_attention's rows and, for each, the natural log of the softmax's
    normaliser: lse[b, j] = ln sum_i exp(q[b, j] . k_i * scale) over the same
    present slots (-inf and a zero row for an empty set). Returns (float32
    [B, Hq, d], float64 [B, Hq])."""
    B, Hq, d = q_bits.shape
    H = cache.count.shape[1]
    g = Hq // H
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    q = widen_bf16(q_bits)
    out = np.zeros((B, Hq, d))
    lse = np.full((B, Hq), -np.inf)
    for b in range(B):
        for h in range(H):
            slots = np.arange(cache.count[b, h])
            pg, row = cache.slot_rows(b, h, slots)
            sel = present(cache.expire_pool[pg, row], now)
            K = widen_bf16(cache.k_pool[pg[sel], row[sel]])
            V = widen_bf16(cache.v_pool[pg[sel], row[sel]])
            if K.shape[0] == 0:
                continue
            for j in range(h * g, (h + 1) * g):
                logits = (K @ q[b, j]) * scale
                m = logits.max()
                w = np.exp(logits - m)
                out[b, j] = (w @ V) / w.sum()
                lse[b, j] = m + math.log(w.sum())
    return out.astype(np.float32), lse


def merge_attention(outs, lses):
    """Attention over the union of disjoint parts of a row's slots, from each
    part's attention row o_p (normalised over its own part) and its lse_p:
    lse = ln sum_p exp(lse_p), o = sum_p exp(lse_p - lse) o_p. A part with
    lse_p = -inf has no slots and weighs nothing; a row with no slots in any
    part is zero with lse -inf. outs [P, ..., d], lses [P, ...]. Returns
    (float64 [..., d], float64 [...])."""
    outs = np.asarray(outs, np.float64)
    lses = np.asarray(lses, np.float64)
    m = lses.max(axis=0)
    has = m > -np.inf
    m_safe = np.where(has, m, 0.0)
    w = np.where(has[None], np.exp(lses - m_safe[None]), 0.0)
    total = w.sum(axis=0)
    lse = np.where(has, m_safe + np.log(np.where(has, total, 1.0)), -np.inf)
    wn = np.where(has[None], w / np.where(has, total, 1.0)[None], 0.0)
    out = (wn[..., None] * outs).sum(axis=0)
    return out, lse


def dense_attention(q_bits, k_bits, v_bits, now: int, scale=None, lo=None):
    """Brute force over the dense cache [B, T, H, d]: every position in
    [lo, now] (lo = 0 by default). No pages, no masks."""
    B, Hq, d = q_bits.shape
    H = k_bits.shape[2]
    g = Hq // H
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    lo = 0 if lo is None else max(0, lo)
    q = widen_bf16(q_bits)
    out = np.zeros((B, Hq, d))
    for b in range(B):
        for j in range(Hq):
            h = j // g
            out[b, j] = _softmax_attend(q[b, j], widen_bf16(k_bits[b, lo:now + 1, h]),
                                        widen_bf16(v_bits[b, lo:now + 1, h]), scale)
    return out.astype(np.float32)


def window_attention(q_bits, k_bits, v_bits, now: int, window: int = WINDOW, scale=None):
    """Sliding-window attention over the last `window` positions ending at now
    ([DMS, "문제 완화를 위한 이전 시도" table, first row])."""
    return dense_attention(q_bits, k_bits, v_bits, now, scale, lo=now - window + 1)


# ---------------------------------------------------------------------------
# 5. Quantize instead of drop  [BeaconKV: the important entries keep full
#    precision, the others are compressed lossily by low-precision
#    quantization or pruning ("비콘KV" article, core-idea paragraph and its
#    first FAQ answer)]
#
# Reading (the article names no format): a second, fp8 tier. An entry whose
# score s has tau_q <= s < tau (NaN never) is stored once more, its K and V
# rows each as FP8 E4M3 codes with one float32 scale per row; it is visible
# in that tier from step pos + window on, i.e. from the step its full
# precision copy leaves the window. Entries with s >= tau stay bf16 for good
# (section 2); entries below tau_q are dropped after the window as before.
# With DMS flags instead of scores, every flagged entry (flag_step >= 0) is
# the one quantized instead of evicted: it enters the fp8 tier at the step
# its bf16 copy is gone, max(flag + delay, pos + window).
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_positive_values() -> np.ndarray:
    """Value of codes 0..127 of FP8 E4M3 (sign bit clear): exponent bias 7,
    three mantissa bits, subnormals at exponent field 0, no infinities, code
    127 (all ones) is NaN. Codes 128..255 are the negatives."""
    vals = np.empty(128)
    for code in range(128):
        e, m = code >> 3, code & 7
        if e == 15 and m == 7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = (m / 8.0) * 2.0 ** -6
        else:
            vals[code] = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


def e4m3_decode(codes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.int64)
    v = e4m3_positive_values()[codes & 0x7F]
    return np.where(codes & 0x80, -v, v)


def e4m3_encode(v) -> np.ndarray:
    """Round to the nearest E4M3 value, ties to the even code (the one whose
    mantissa's last bit is 0); magnitudes above 448 saturate to 448; NaN gives
    code 0x7F. The sign is kept, also for a result of zero (-0 -> 0x80)."""
    v = np.asarray(v, dtype=np.float64)
    grid = e4m3_positive_values()[:127]          # finite magnitudes, ascending
    a = np.abs(v)
    hi = np.clip(np.searchsorted(grid, a), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    dlo, dhi = a - grid[lo], grid[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(a >= E4M3_MAX, 126, np.where(a <= grid[lo], lo, np.where(pick_hi, hi, lo)))
    code = np.where(np.isnan(v), 0x7F, code)
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def quantize_rows(bits: np.ndarray):
    """bf16 rows [..., d] -> (codes uint8 [..., d], scale float32 [...]).
    In float32 with round to nearest: scale = amax(|row|) / 448 (the
    dequantization factor) and inv = 448 / amax(|row|); each element is
    multiplied by inv and rounded to E4M3. An all-zero row has scale 0 and
    codes 0."""
    x = widen_bf16(bits).astype(np.float32)
    amax = np.abs(x).max(axis=-1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    nz = amax > 0
    inv = (np.float32(E4M3_MAX) / np.where(nz, amax, np.float32(1.0))).astype(np.float32)
    y = (x * inv[..., None]).astype(np.float32)
    codes = np.where(nz[..., None], e4m3_encode(y), 0).astype(np.uint8)
    return codes, scale


def dequantize_rows(codes, scale) -> np.ndarray:
    return e4m3_decode(codes) * np.asarray(scale, dtype=np.float64)[..., None]


def quant_tier_select(scores_bth, tau_bh, tau_q_bh):
    """Entries that go to the fp8 tier: tau_q <= s < tau. [B, H, T] bool."""
    s = np.asarray(scores_bth).transpose(0, 2, 1)
    t = np.asarray(tau_bh)[:, :, None]
    tq = np.asarray(tau_q_bh)[:, :, None]
    return (s >= tq) & (s < t)


class QuantPagedCache:
    """The fp8 tier: code pools [n_pages, 16, d] uint8 for K and V, per-slot
    scales [n_pages, 16] float32, per-slot start step [n_pages, 16], page
    table [B, H, max_pages] (-1 = unused), remap [B, H, max_pages*16], count."""

    def __init__(self, batch, n_kv_heads, head_dim, n_pages_cap, max_pages):
        self.kq_pool = np.zeros((n_pages_cap, PAGE, head_dim), dtype=np.uint8)
        self.vq_pool = np.zeros((n_pages_cap, PAGE, head_dim), dtype=np.uint8)
        self.kscale = np.zeros((n_pages_cap, PAGE), dtype=np.float32)
        self.vscale = np.zeros((n_pages_cap, PAGE), dtype=np.float32)
        self.start_pool = np.zeros((n_pages_cap, PAGE), dtype=np.int64)
        self.page_table = np.full((batch, n_kv_heads, max_pages), -1, dtype=np.int64)
        self.remap = np.full((batch, n_kv_heads, max_pages * PAGE), -1, dtype=np.int64)
        self.count = np.zeros((batch, n_kv_heads), dtype=np.int64)
        self.pages_used = 0

    def slot_rows(self, b, h, slots):
        slots = np.asarray(slots, dtype=np.int64)
        return self.page_table[b, h, slots // PAGE], slots % PAGE


def quant_tier_select_dms(flag_step_bht):
    """DMS: the entries flagged for eviction go to the fp8 tier. [B, H, T] bool."""
    return np.asarray(flag_step_bht) >= 0


def compact_quant_dense(k_bits, v_bits, scores_bth, tau_bh, tau_q_bh, reserve, n_pages_cap, max_pages,
                        window: int = WINDOW, flag_step_bht=None, delay: int = 0) -> QuantPagedCache:
    """Dense K/V [B, T, H, d] -> the fp8 tier of the entries with
    tau_q <= s < tau (or, given DMS flag steps instead of scores, the flagged
    ones), in ascending position, pages handed out in (b-major, h-minor)
    order exactly as in section 3; start = position + window (DMS:
    max(flag + delay, position + window))."""
    B, T, H, d = k_bits.shape
    out = QuantPagedCache(B, H, d, n_pages_cap, max_pages)
    dms = flag_step_bht is not None
    sel = quant_tier_select_dms(flag_step_bht) if dms else quant_tier_select(scores_bth, tau_bh, tau_q_bh)
    for b in range(B):
        for h in range(H):
            pos = np.nonzero(sel[b, h])[0]
            n = len(pos)
            npg = _pages_for(n, reserve)
            if npg > max_pages or out.pages_used + npg > n_pages_cap:
                raise CapacityError(f"(b={b}, h={h}) needs {npg} fp8 pages")
            base = out.pages_used
            out.page_table[b, h, :npg] = base + np.arange(npg)
            j = np.arange(n)
            kc, ks = quantize_rows(k_bits[b, pos, h])
            vc, vs = quantize_rows(v_bits[b, pos, h])
            out.kq_pool[base + j // PAGE, j % PAGE] = kc
            out.vq_pool[base + j // PAGE, j % PAGE] = vc
            out.kscale[base + j // PAGE, j % PAGE] = ks
            out.vscale[base + j // PAGE, j % PAGE] = vs
            out.start_pool[base + j // PAGE, j % PAGE] = (
                expire_dms(np.asarray(flag_step_bht)[b, h, pos], pos, delay, window) if dms else pos + window)
            out.remap[b, h, :n] = pos
            out.count[b, h] = n
            out.pages_used += npg
    return out


def append_quant(qcache: QuantPagedCache, k_new_bits, v_new_bits, pos: int, score_bh, tau_bh, tau_q_bh,
                 window: int = WINDOW, flag_bh=None, delay: int = 0):
    """Decode step for the fp8 tier: the token at `pos` (k/v [B, H, d]) goes
    into slot count[b, h] of its (b, h)'s fp8 pages iff tau_q <= score < tau
    (DMS: iff flagged, flag_bh >= 0), quantized like the compaction's rows,
    with start = pos + window (DMS: max(flag + delay, pos + window)); raises
    if the reserved slots are used up."""
    B, H = qcache.count.shape
    if flag_bh is not None:
        sel = np.asarray(flag_bh) >= 0
    else:
        sel = (np.asarray(score_bh) >= np.asarray(tau_q_bh)) & (np.asarray(score_bh) < np.asarray(tau_bh))
    for b in range(B):
        for h in range(H):
            if not sel[b, h]:
                continue
            j = int(qcache.count[b, h])
            p = j // PAGE
            if p >= qcache.page_table.shape[2] or qcache.page_table[b, h, p] < 0:
                raise CapacityError(f"(b={b}, h={h}) has no free fp8 slot")
            page = qcache.page_table[b, h, p]
            kc, ks = quantize_rows(k_new_bits[b, h][None])
            vc, vs = quantize_rows(v_new_bits[b, h][None])
            qcache.kq_pool[page, j % PAGE] = kc[0]
            qcache.vq_pool[page, j % PAGE] = vc[0]
            qcache.kscale[page, j % PAGE] = ks[0]
            qcache.vscale[page, j % PAGE] = vs[0]
            qcache.start_pool[page, j % PAGE] = (
                expire_dms(np.asarray(flag_bh)[b, h], pos, delay, window) if flag_bh is not None else pos + window)
            qcache.remap[b, h, j] = pos
            qcache.count[b, h] = j + 1


def decode_attention_two_tier(q_bits, cache: PagedCache, qcache: QuantPagedCache, now: int,
                              scale: float | None = None) -> np.ndarray:
    """Attention over the union of the bf16 tier's slots present at `now`
    (now < expire) and the fp8 tier's slots visible at `now` (now >= start),
    the latter dequantized exactly (code value x row scale, float64)."""
    B, Hq, d = q_bits.shape
    H = cache.count.shape[1]
    g = Hq // H
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    q = widen_bf16(q_bits)
    out = np.zeros((B, Hq, d))
    for b in range(B):
        for h in range(H):
            pg, row = cache.slot_rows(b, h, np.arange(cache.count[b, h]))
            sel = present(cache.expire_pool[pg, row], now)
            Ka = widen_bf16(cache.k_pool[pg[sel], row[sel]])
            Va = widen_bf16(cache.v_pool[pg[sel], row[sel]])
            pq, rq = qcache.slot_rows(b, h, np.arange(qcache.count[b, h]))
            vis = now >= qcache.start_pool[pq, rq]
            pq, rq = pq[vis], rq[vis]
            Kb = dequantize_rows(qcache.kq_pool[pq, rq], qcache.kscale[pq, rq])
            Vb = dequantize_rows(qcache.vq_pool[pq, rq], qcache.vscale[pq, rq])
            K = np.concatenate([Ka, Kb.reshape(-1, d)])
            V = np.concatenate([Va, Vb.reshape(-1, d)])
            for j in range(h * g, (h + 1) * g):
                out[b, j] = _softmax_attend(q[b, j], K, V, scale)
    return out.astype(np.float32)


# ---------------------------------------------------------------------------
# 6. Latent-cache (MLA) pruning  [DMS, "주요 요점" (compatible with Multi-Head
#    Latent Attention as used by DeepSeek models) and "앞으로의 전망" (DMS
#    combined with MLA)]
#
# Reading: with MLA every token caches one latent row shared by all query
# heads, c_t (the compressed KV, dc values) followed by the shared rotary key
# (dr values). Pruning keeps or drops that row as a whole: one score (or DMS
# flag) per token, the rules of section 2 with a single "kv head", and the
# compaction of section 3 over rows of dc + dr values. Attention is MLA's
# absorbed decode form: query head j brings q_j = [q_nope_j W_UK_j^T, q_rope_j]
# (dc + dr values), its logit against slot t is scale * q_j . row_t, and its
# output is the softmax-weighted sum of the rows' first dc values (the
# compressed value, to which the caller applies W_UV_j).
# ---------------------------------------------------------------------------

def compact_latent_dense(lat_bits, expire_bt, now: int, reserve: int, n_pages_cap: int, max_pages: int) -> PagedCache:
    """Latent rows [B, T, dc + dr] + expire [B, T] -> PagedCache with one
    "kv head" (H = 1) whose K pool holds the latent rows (its V pool holds the
    same rows: one pool is enough for MLA, the cache format is section 3's)."""
    lat = np.asarray(lat_bits)[:, :, None, :]
    return compact_dense(lat, lat, np.asarray(expire_bt)[:, None, :], now, reserve, n_pages_cap, max_pages)


def decode_attention_mla(q_bits, cache: PagedCache, dc: int, now: int, scale: float | None = None) -> np.ndarray:
    """o[b, j] = sum_t softmax_t(scale * q[b, j] . row_t) row_t[:dc] over the
    latent slots present at `now`; q [B, Hq, dc + dr] bf16 bits, rows from the
    K pool; scale defaults to 1 / sqrt(dc + dr). Returns float32 [B, Hq, dc]."""
    B, Hq, Dl = q_bits.shape
    scale = 1.0 / math.sqrt(Dl) if scale is None else scale
    q = widen_bf16(q_bits)
    out = np.zeros((B, Hq, dc))
    for b in range(B):
        pg, row = cache.slot_rows(b, 0, np.arange(cache.count[b, 0]))
        sel = present(cache.expire_pool[pg, row], now)
        C = widen_bf16(cache.k_pool[pg[sel], row[sel]])
        for j in range(Hq):
            out[b, j] = _softmax_attend(q[b, j], C, C[:, :dc], scale)
    return out.astype(np.float32)


# ---------------------------------------------------------------------------
# Closed forms the pages quote
# ---------------------------------------------------------------------------

def kv_cache_bytes(n_layers: int, d_model: int, n_tokens: int, elem_bytes: int = 2) -> int:
    """K and V, one d_model-wide row each per token per layer
    ([KVzap, 이게 뭔데? / 핵심 내용 정리: Llama1-65B at 128k tokens])."""
    return 2 * n_layers * d_model * n_tokens * elem_bytes


def linear_projection_macs(d_model, n_q_heads, n_kv_heads, head_dim, ffn_hidden, gated=True) -> int:
    """Per-token multiply-adds of a decoder layer's linear projections
    (Q, K, V, O and the feed-forward block)."""
    qo = 2 * d_model * n_q_heads * head_dim
    kv = 2 * d_model * n_kv_heads * head_dim
    ffn = (3 if gated else 2) * d_model * ffn_hidden
    return qo + kv + ffn


def scorer_macs(d_model, n_kv_heads, hidden=None) -> int:
    """Per-token multiply-adds of the KVzap surrogate ([KVzap, "메모리 및 계산 효율"])."""
    if hidden is None:
        return d_model * n_kv_heads
    return d_model * hidden + hidden * n_kv_heads
