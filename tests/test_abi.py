"""CPU checks of the C ABI: the library builds, loads, exports every entry
point include/kvp.h declares, and rejects bad arguments on the host (no call
here reaches a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "kvp.h")) as f:
        text = f.read()
    return re.findall(r"^KVP_API[^;(]*?\b(kvp_\w+)\s*\(", text, flags=re.M | re.S)


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._builder().build()
    return ctypes.CDLL(path)


def test_header_declares_the_path():
    names = set(_declared())
    for n in ["kvp_score", "kvp_mask", "kvp_compact", "kvp_compact_masked", "kvp_compact_quant", "kvp_append_quant", "kvp_compact_paged",
              "kvp_threshold", "kvp_append", "kvp_decode_attn",
              "kvp_score_workspace_bytes", "kvp_compact_workspace_bytes", "kvp_decode_attn_workspace_bytes",
              "kvp_compact_latent", "kvp_compact_latent_paged", "kvp_append_latent", "kvp_decode_attn_mla",
              "kvp_decode_attn_mla_workspace_bytes", "kvp_status_string", "kvp_version"]:
        assert n in names, n


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), f"{n} declared in kvp.h but not exported"


def test_status_strings_and_version(lib):
    lib.kvp_status_string.restype = ctypes.c_char_p
    assert lib.kvp_status_string(0) == b"ok"
    assert b"aligned" in lib.kvp_status_string(2)
    assert lib.kvp_status_string(99) == b"unknown status"
    assert lib.kvp_version() >= 100


def test_workspace_sizes(lib):
    lib.kvp_score_workspace_bytes.restype = ctypes.c_size_t
    lib.kvp_score_split_weight_bytes.restype = ctypes.c_size_t
    assert lib.kvp_score_split_weight_bytes(4096, 8) == 16 * 4096 * 2   # 2H rows padded to 16
    assert lib.kvp_score_split_weight_bytes(256, 20) == 64 * 256 * 2
    assert lib.kvp_score_workspace_bytes(2, 1000, 4096, 8, 0) == 0      # LINEAR_SPLIT needs none
    lib.kvp_score_workspace_bytes.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int]
    # LINEAR: bf16 hi/lo weight rows, padded to 16 rows for 8 heads
    assert lib.kvp_score_workspace_bytes(0, 131072, 4096, 8, 0) == 16 * 4096 * 2
    # MLP: one fp32 partial per 256-wide hidden chunk, token and head
    assert lib.kvp_score_workspace_bytes(1, 1000, 4096, 8, 1024) == 4 * 1000 * 8 * 4
    lib.kvp_decode_attn_workspace_bytes.restype = ctypes.c_size_t
    # counters (B*H, 16-byte rounded) + (512 CTAs x 8 warps + B*H) * G * (d + 2) floats
    assert lib.kvp_decode_attn_workspace_bytes(2, 8, 2, 128) == 16 + (4096 + 4) * 4 * 130 * 4


def test_host_validation_without_gpu(lib):
    import kv_cache_pruning_gb300 as k
    L = k.library()
    # null x -> invalid; unsupported head count; unaligned x
    assert L.kvp_score(0, 10, 64, 2, 0, None, 64, None, None, None, None, None, None, 0, None, None) == k.KVP_ERR_INVALID
    assert L.kvp_score(0, 10, 64, 65, 0, 16, 64, 16, None, None, None, 16, 16, 1 << 20, None, None) == k.KVP_ERR_UNSUPPORTED
    assert L.kvp_score(0, 10, 64, 2, 0, 18, 64, 16, None, None, None, 16, 16, 1 << 20, None, None) == k.KVP_ERR_ALIGN
    assert L.kvp_score(0, 10, 64, 2, 0, 16, 64, 16, None, None, None, 16, 16, 8, None, None) == k.KVP_ERR_WORKSPACE
    # weight split: bad sizes, short output, unaligned output
    assert L.kvp_score_split_weight(0, 8, 16, 16, 1 << 20, None) == k.KVP_ERR_INVALID
    assert L.kvp_score_split_weight(4100, 8, 16, 16, 1 << 20, None) == k.KVP_ERR_UNSUPPORTED
    assert L.kvp_score_split_weight(4096, 8, 16, 16, 16 * 4096 * 2 - 1, None) == k.KVP_ERR_WORKSPACE
    assert L.kvp_score_split_weight(4096, 8, 16, 24, 1 << 20, None) == k.KVP_ERR_ALIGN
    # scorer on a pre-split weight: unaligned weight, MLP-only arguments
    assert L.kvp_score(2, 10, 64, 2, 0, 16, 64, 24, None, None, None, 16, None, 0, None, None) == k.KVP_ERR_ALIGN
    assert L.kvp_score(2, 10, 64, 2, 0, 16, 64, 16, None, 16, None, 16, None, 0, None, None) == k.KVP_ERR_INVALID
    # mask: both inputs given / unknown mode
    assert L.kvp_mask(0, 1, 1, 8, 0, 16, 16, 16, 128, 0, 7, 16, None, None, None) == k.KVP_ERR_INVALID
    assert L.kvp_mask(5, 1, 1, 8, 0, 16, 16, None, 128, 0, 7, 16, None, None, None) == k.KVP_ERR_INVALID
    # attention: head ratio not in {1,2,4,8}, bad head_dim
    assert L.kvp_decode_attn(1, 6, 2, 128, 16, 16, 16, 16, 1, 16, 1, 16, 0, 0.0, 16, 0, 16, 1 << 20, None,
                             None) == k.KVP_ERR_UNSUPPORTED
    assert L.kvp_decode_attn(1, 4, 2, 96, 16, 16, 16, 16, 1, 16, 1, 16, 0, 0.0, 16, 0, 16, 1 << 20, None,
                             None) == k.KVP_ERR_UNSUPPORTED
    # compaction: status word is required
    assert L.kvp_compact(1, 1, 128, 16, 16, 16, 0, 0, 0, 16, 15, 0, 16, 16, 16, 1, 16, 1, 16, 16, 16, 1 << 20,
                         None, None) == k.KVP_ERR_INVALID


def test_compact_masked_host_checks():
    """The fused mask + compaction entry point rejects bad arguments on the
    host before any CUDA call."""
    import kv_cache_pruning_gb300 as k
    L = k.library()

    def call(mode=0, hd=128, n_pos=16, kp=16, scores=16, tau=16, flag=None, window=128, delay=0, status=16):
        return L.kvp_compact_masked(mode, 1, 1, hd, n_pos, kp, 16, 0, 0, 0, scores, tau, flag, window, delay, 15, 0,
                                    16, 16, 16, 1, 16, 1, 16, 16, 16, 1 << 20, status, None)

    assert call(flag=16) == k.KVP_ERR_INVALID                        # KVzap with a flag array too
    assert call(tau=None) == k.KVP_ERR_INVALID                       # KVzap without a threshold
    assert call(mode=1, flag=16) == k.KVP_ERR_INVALID                # DMS with scores too
    assert call(mode=1, scores=None, tau=None) == k.KVP_ERR_INVALID  # DMS without flags
    assert call(mode=7) == k.KVP_ERR_INVALID
    assert call(window=-1) == k.KVP_ERR_INVALID
    assert call(n_pos=2**31 - 200, window=128, delay=100) == k.KVP_ERR_INVALID  # expire would overflow
    assert call(hd=96) == k.KVP_ERR_UNSUPPORTED
    assert call(status=None) == k.KVP_ERR_INVALID
    assert call(kp=8) == k.KVP_ERR_ALIGN


def test_compact_quant_host_checks():
    import kv_cache_pruning_gb300 as k
    L = k.library()

    def call(mode=0, hd=128, scores=16, tau=16, tau_q=16, flag=None, window=128, delay=0, kq=16, meta=16, status=16):
        return L.kvp_compact_quant(mode, 1, 1, hd, 16, 16, 16, 0, 0, 0, scores, tau, tau_q, flag, window, delay, 0,
                                   kq, 16, meta, 1, 16, 1, 16, 16, 16, 1 << 20, status, None)

    assert call(tau_q=None) == k.KVP_ERR_INVALID
    assert call(flag=16) == k.KVP_ERR_INVALID                                   # KVzap with flags too
    assert call(mode=1, flag=16) == k.KVP_ERR_INVALID                           # DMS with scores too
    assert call(mode=1, scores=None, tau=None, tau_q=None) == k.KVP_ERR_INVALID  # DMS without flags
    assert call(mode=1, scores=None, tau=None, tau_q=None, flag=16, delay=-1) == k.KVP_ERR_INVALID
    assert call(mode=3) == k.KVP_ERR_INVALID
    assert call(scores=None) == k.KVP_ERR_INVALID
    assert call(window=-1) == k.KVP_ERR_INVALID
    assert call(meta=None) == k.KVP_ERR_INVALID
    assert call(status=None) == k.KVP_ERR_INVALID
    assert call(hd=96) == k.KVP_ERR_UNSUPPORTED
    assert call(kq=8) == k.KVP_ERR_ALIGN


def test_append_quant_host_checks():
    import kv_cache_pruning_gb300 as k
    L = k.library()

    def call(mode=0, hd=128, pos=5, kn=16, score=16, tau=16, tau_q=16, flag=None, window=128, delay=0, status=16):
        return L.kvp_append_quant(mode, 1, 1, hd, pos, kn, 16, score, tau, tau_q, flag, window, delay, 16, 16, 16, 1,
                                  16, 1, 16, 16, status, None)

    assert call(tau_q=None) == k.KVP_ERR_INVALID
    assert call(mode=1, flag=16) == k.KVP_ERR_INVALID                          # DMS with scores too
    assert call(mode=1, score=None, tau=None, tau_q=None) == k.KVP_ERR_INVALID  # DMS without flags
    assert call(pos=-1) == k.KVP_ERR_INVALID
    assert call(window=-2) == k.KVP_ERR_INVALID
    assert call(status=None) == k.KVP_ERR_INVALID
    assert call(hd=32) == k.KVP_ERR_UNSUPPORTED
    assert call(kn=8) == k.KVP_ERR_ALIGN
    assert call(pos=2**31 - 100) == k.KVP_ERR_INVALID       # start would overflow


def test_threshold_host_checks():
    import kv_cache_pruning_gb300 as k
    L = k.library()
    # histogram 1 KiB per (b, h), prefix and rank, 4 pass counters per (b, head group of 32)
    assert L.kvp_threshold_workspace_bytes(16, 8) == (128 * 256 + 2 * 128 + 4 * 16) * 4
    assert L.kvp_threshold_workspace_bytes(1, 64) == (64 * 256 + 2 * 64 + 4 * 2) * 4
    assert L.kvp_threshold_workspace_bytes(0, 8) == 0
    ws = L.kvp_threshold_workspace_bytes(2, 3)

    def call(B=2, H=3, n=100, scores=16, q=0.5, tau=16, wsp=16, wsb=ws):
        return L.kvp_threshold(B, H, n, scores, q, tau, wsp, wsb, None)

    for q in (-0.01, 1.01, float("nan")):
        assert call(q=q) == k.KVP_ERR_INVALID
    assert call(n=0) == k.KVP_ERR_INVALID
    assert call(scores=None) == k.KVP_ERR_INVALID
    assert call(tau=None) == k.KVP_ERR_INVALID
    assert call(wsb=ws - 4) == k.KVP_ERR_WORKSPACE
    assert call(wsp=None) == k.KVP_ERR_WORKSPACE
    assert call(B=70000, wsb=1 << 40) == k.KVP_ERR_UNSUPPORTED


def test_latent_host_checks():
    """The latent-cache entry points reject bad arguments on the host before
    any CUDA call: row width other than 512 + 64, mode/input mismatches,
    missing status, unaligned pools, short workspace, aliased source and
    destination."""
    import kv_cache_pruning_gb300 as k
    L = k.library()
    ws = L.kvp_compact_workspace_bytes(1, 1, 16)

    def compact(mode=0, row=576, scores=16, tau=16, flag=None, window=128, lat=16, pool=16, status=16, wsb=ws):
        return L.kvp_compact_latent(mode, 1, row, 16, lat, 0, 576, scores, tau, flag, window, 0, 15, 0, pool, 16, 1,
                                    16, 1, 16, 16, 16, wsb, status, None)

    assert compact(row=512) == k.KVP_ERR_UNSUPPORTED
    assert compact(flag=16) == k.KVP_ERR_INVALID                         # KVzap with flags too
    assert compact(mode=1, flag=16) == k.KVP_ERR_INVALID                 # DMS with scores too
    assert compact(mode=1, scores=None, tau=None) == k.KVP_ERR_INVALID   # DMS without flags
    assert compact(tau=None) == k.KVP_ERR_INVALID
    assert compact(window=-1) == k.KVP_ERR_INVALID
    assert compact(status=None) == k.KVP_ERR_INVALID
    assert compact(pool=8) == k.KVP_ERR_ALIGN
    assert compact(lat=8) == k.KVP_ERR_ALIGN
    assert compact(wsb=ws - 4) == k.KVP_ERR_WORKSPACE
    pws = L.kvp_compact_paged_workspace_bytes(1, 1, 2)

    def paged(row=576, src=16, pool=32, cnt_src=16, cnt=48, wsb=pws):
        return L.kvp_compact_latent_paged(1, row, src, 16, 4, 16, 2, 16, cnt_src, 15, 0, pool, 64, 4, 80, 2, 96, cnt,
                                          16, wsb, 16, None)

    assert paged(row=640) == k.KVP_ERR_UNSUPPORTED
    assert paged(pool=16) == k.KVP_ERR_INVALID        # source and destination share the pool
    assert paged(cnt=16) == k.KVP_ERR_INVALID         # ... or the count
    assert paged(src=8) == k.KVP_ERR_ALIGN
    assert paged(wsb=pws - 1) == k.KVP_ERR_WORKSPACE

    def append(mode=0, row=576, pos=5, lat=16, score=16, tau=16, flag=None, status=16):
        return L.kvp_append_latent(mode, 1, row, pos, lat, score, tau, flag, 128, 0, 16, 16, 1, 16, 1, 16, 16, status,
                                   None)

    assert append(row=128) == k.KVP_ERR_UNSUPPORTED
    assert append(pos=-1) == k.KVP_ERR_INVALID
    assert append(mode=1, flag=16) == k.KVP_ERR_INVALID
    assert append(mode=1, score=None, tau=None) == k.KVP_ERR_INVALID
    assert append(status=None) == k.KVP_ERR_INVALID
    assert append(lat=8) == k.KVP_ERR_ALIGN
    assert append(pos=2**31 - 100) == k.KVP_ERR_INVALID    # expire would overflow


def test_mla_attention_host_checks_and_workspace():
    import kv_cache_pruning_gb300 as k
    L = k.library()
    # (m, l) and accumulators per unit, slice and head of the tile: 16-head tiles up to 32 heads, 64-head
    # tiles up to 64, 128-head tiles above
    assert L.kvp_decode_attn_mla_workspace_bytes(2, 20, 3) == 4 * 3 * 16 * 2 * 4 + 4 * 3 * 16 * 512 * 4
    assert L.kvp_decode_attn_mla_workspace_bytes(2, 33, 3) == 2 * 3 * 64 * 2 * 4 + 2 * 3 * 64 * 512 * 4
    assert L.kvp_decode_attn_mla_workspace_bytes(2, 65, 3) == 2 * 3 * 128 * 2 * 4 + 2 * 3 * 128 * 512 * 4
    assert L.kvp_decode_attn_mla_workspace_bytes(2, 130, 3) == 4 * 3 * 128 * 2 * 4 + 4 * 3 * 128 * 512 * 4
    assert L.kvp_decode_attn_mla_workspace_bytes(3, 16, 2) == 3 * 2 * 16 * 2 * 4 + 3 * 2 * 16 * 512 * 4
    assert L.kvp_decode_attn_mla_workspace_bytes(1, 1, 1) == 16 * 2 * 4 + 16 * 512 * 4
    assert L.kvp_decode_attn_mla_workspace_bytes(2, 16, 65) == 0
    assert L.kvp_decode_attn_mla_workspace_bytes(0, 16, 1) == 0
    ws = L.kvp_decode_attn_mla_workspace_bytes(2, 20, 3)

    def call(hq=20, dc=512, dr=64, q=16, out=16, ns=3, scale=0.0, wsp=16, wsb=ws, cap=4):
        return L.kvp_decode_attn_mla(2, hq, dc, dr, q, 16, 16, cap, 16, 2, 16, 30, scale, out, ns, wsp, wsb, None,
                                     None)

    assert call(dc=256) == k.KVP_ERR_UNSUPPORTED
    assert call(dr=32) == k.KVP_ERR_UNSUPPORTED
    assert call(hq=0) == k.KVP_ERR_INVALID
    assert call(ns=65) == k.KVP_ERR_INVALID
    assert call(scale=-1.0) == k.KVP_ERR_INVALID
    assert call(q=None) == k.KVP_ERR_INVALID
    assert call(q=8) == k.KVP_ERR_ALIGN
    assert call(out=24) == k.KVP_ERR_ALIGN
    assert call(wsb=ws - 16) == k.KVP_ERR_WORKSPACE
    assert call(wsp=None) == k.KVP_ERR_WORKSPACE
    assert call(cap=2**27) == k.KVP_ERR_UNSUPPORTED   # page rows past 2^31


def test_missing_library_fails_loudly(monkeypatch):
    import kv_cache_pruning_gb300 as k
    monkeypatch.setattr(k, "LIB_PATH", os.path.join(ROOT, "no_such_libkvp.so"))
    with pytest.raises(ImportError):
        k._load()


def _prototypes():
    """name -> (return type text, [parameter type texts]) for every KVP_API prototype of kvp.h."""
    with open(os.path.join(ROOT, "include", "kvp.h")) as f:
        text = re.sub(r"/\*.*?\*/", " ", f.read(), flags=re.S)
    out = {}
    for m in re.finditer(r"KVP_API\s+([^;(]*?)\b(kvp_\w+)\s*\(([^;]*?)\)\s*;", text, flags=re.S):
        ret, name, params = m.group(1).strip(), m.group(2), m.group(3).strip()
        plist = [] if params in ("", "void") else [" ".join(p.split()) for p in params.split(",")]
        # drop the parameter name: the last identifier (a pointer star stays with the type)
        types = [re.sub(r"\s*\b\w+$", "", p).strip() for p in plist]
        out[name] = (ret, types)
    return out


def _ctype_of(c_type: str):
    if "*" in c_type:
        return ctypes.c_char_p if c_type.replace(" ", "") == "constchar*" else ctypes.c_void_p
    base = c_type.replace("const ", "").strip()
    return {"int": ctypes.c_int, "int64_t": ctypes.c_int64, "uint64_t": ctypes.c_uint64, "size_t": ctypes.c_size_t,
            "float": ctypes.c_float, "double": ctypes.c_double, "kvp_status": ctypes.c_int}[base]


def test_binding_signatures_match_the_header():
    """Every entry point of kvp.h is bound in the Python package with the
    ctypes argument and return types its C prototype implies (a wrong width,
    say int for int64_t, would pass silently through ctypes otherwise)."""
    import kv_cache_pruning_gb300 as k
    protos = _prototypes()
    assert set(protos) == set(_declared())
    for name, (ret, params) in protos.items():
        assert name in k._SIGS, f"{name} has no binding"
        res, args = k._SIGS[name]
        assert res == _ctype_of(ret), f"{name}: return {ret} bound as {res}"
        assert len(args) == len(params), f"{name}: {len(params)} parameters, {len(args)} bound"
        for i, (c, a) in enumerate(zip(params, args)):
            assert a == _ctype_of(c), f"{name} parameter {i} ({c}) bound as {a}"


def test_header_constants_match_the_binding():
    import kv_cache_pruning_gb300 as k
    with open(os.path.join(ROOT, "include", "kvp.h")) as f:
        text = f.read()
    defines = {m.group(1): int(m.group(2)) for m in re.finditer(r"^#define\s+(KVP_\w+)\s+(\d+)", text, flags=re.M)}
    assert defines["KVP_PAGE_TOKENS"] == k.PAGE
    assert defines["KVP_WINDOW_DEFAULT"] == k.WINDOW
    assert defines["KVP_EXPIRE_NEVER"] == k.EXPIRE_NEVER
    assert defines["KVP_MLA_LATENT_DIM"] == k.KVP_MLA_LATENT_DIM
    assert defines["KVP_MLA_ROPE_DIM"] == k.KVP_MLA_ROPE_DIM
    enums = {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(KVP_(?:ERR|OK|SCORER|MASK)\w*)\s*=\s*(\d+)", text)}
    for name, value in enums.items():
        assert getattr(k, name) == value, name


def test_selftest_wait_host_checks():
    import kv_cache_pruning_gb300 as k
    L = k.library()
    assert L.kvp_selftest_wait(1000, None, None, None) == k.KVP_ERR_INVALID            # status is required
    assert L.kvp_selftest_wait(10**10 + 1, 16, None, None) == k.KVP_ERR_INVALID        # more than 10 s
