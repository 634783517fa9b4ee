"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, and rejects malformed or unsupported arguments on the host before
any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fattn():
    from paged_kv_cache_tiled_gb300 import build
    build.build()
    from paged_kv_cache_tiled_gb300 import fattn as F
    return F


def header_symbols():
    text = open(os.path.join(ROOT, "include", "fattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_header_symbol(fattn):
    syms = header_symbols()
    assert len(syms) >= 12
    lib = ctypes.CDLL(fattn.LIB_PATH)
    for s in syms:
        assert hasattr(lib, s), s
    assert sorted(fattn.EXPORTS) == syms


def test_status_strings(fattn):
    assert fattn.status_string(0) == "FA_OK"
    assert fattn.status_string(fattn.FA_ERR_BOUNDS) == "FA_ERR_BOUNDS"
    assert fattn.status_string(99) == "FA_ERR_UNKNOWN"


def test_host_validation(fattn):
    lib = fattn.library()
    P = ctypes.c_void_p
    dummy = P(4096)  # never dereferenced: validation fails first
    # negative sizes
    assert lib.fa_prefill(dummy, dummy, dummy, dummy, -1, 16, 4, 2, 64, 1, 0.1, None, None) == fattn.FA_ERR_INVALID_ARG
    # unsupported head dim / GQA ratio
    assert lib.fa_prefill(dummy, dummy, dummy, dummy, 1, 16, 4, 2, 96, 1, 0.1, None, None) == fattn.FA_ERR_UNSUPPORTED
    assert lib.fa_prefill(dummy, dummy, dummy, dummy, 1, 16, 5, 2, 64, 1, 0.1, None, None) == fattn.FA_ERR_UNSUPPORTED
    # empty problems are no-ops
    assert lib.fa_prefill(None, None, None, None, 0, 16, 4, 2, 64, 1, 0.1, None, None) == fattn.FA_OK
    # null pointers / misalignment
    assert lib.fa_prefill(None, dummy, dummy, dummy, 1, 16, 4, 2, 64, 1, 0.1, None, None) == fattn.FA_ERR_INVALID_ARG
    assert lib.fa_prefill(P(4097), dummy, dummy, dummy, 1, 16, 4, 2, 64, 1, 0.1, None, None) == fattn.FA_ERR_INVALID_ARG
    # outputs must be 32-byte aligned; non-positive scale is rejected
    assert lib.fa_prefill(dummy, dummy, dummy, P(4096 + 16), 1, 16, 4, 2, 64, 1, 0.1, None, None) == fattn.FA_ERR_INVALID_ARG
    assert lib.fa_prefill(dummy, dummy, dummy, dummy, 1, 16, 4, 2, 64, 1, 0.0, None, None) == fattn.FA_ERR_INVALID_ARG
    # host-buffer prefill: the same rules, plus every host pointer must be given
    H = lambda *a: lib.fa_prefill_host(*a)
    d8 = [dummy] * 8
    assert H(*d8, -1, 16, 4, 2, 64, 1, 0.1, None) == fattn.FA_ERR_INVALID_ARG
    assert H(*d8, 1, 16, 4, 2, 96, 1, 0.1, None) == fattn.FA_ERR_UNSUPPORTED
    assert H(*([None] * 8), 0, 16, 4, 2, 64, 1, 0.1, None) == fattn.FA_OK
    assert H(None, *d8[1:], 1, 16, 4, 2, 64, 1, 0.1, None) == fattn.FA_ERR_INVALID_ARG
    assert H(*d8[:3], None, *d8[4:], 1, 16, 4, 2, 64, 1, 0.1, None) == fattn.FA_ERR_INVALID_ARG
    assert H(*d8[:4], P(4097), *d8[5:], 1, 16, 4, 2, 64, 1, 0.1, None) == fattn.FA_ERR_INVALID_ARG
    assert H(*d8[:7], P(4096 + 16), 1, 16, 4, 2, 64, 1, 0.1, None) == fattn.FA_ERR_INVALID_ARG
    assert H(*d8, 1, 16, 4, 2, 64, 1, float("inf"), None) == fattn.FA_ERR_INVALID_ARG
    # paged: block size other than 16 is unsupported
    assert lib.fa_paged_attn(dummy, dummy, dummy, dummy, dummy, dummy, dummy, 2, 4, 8, 4, 2, 64, 32, 1, 0.1, 2, 1,
                             dummy, 1 << 20, None) == fattn.FA_ERR_UNSUPPORTED
    # paged: missing / short workspace
    need = lib.fa_paged_attn_workspace_size(2, 4, 4, 2, 64, 2)
    assert need > 0
    assert lib.fa_paged_attn(dummy, dummy, dummy, dummy, dummy, dummy, dummy, 2, 4, 8, 4, 2, 64, 16, 1, 0.1, 2, 1,
                             dummy, need - 1, None) == fattn.FA_ERR_WORKSPACE
    assert lib.fa_paged_attn(dummy, dummy, dummy, dummy, dummy, dummy, dummy, 2, 4, 8, 4, 2, 64, 16, 1, 0.1, 2, 1,
                             None, need, None) == fattn.FA_ERR_WORKSPACE
    # append: bad dtype code, head dim
    assert lib.fa_cache_append(dummy, dummy, dummy, dummy, dummy, 4, 2, 64, 8, 7, None) == fattn.FA_ERR_INVALID_ARG
    assert lib.fa_cache_append(dummy, dummy, dummy, dummy, dummy, 4, 2, 80, 8, 0, None) == fattn.FA_ERR_UNSUPPORTED
    assert lib.fa_cache_append(None, None, None, None, None, 0, 2, 64, 8, 0, None) == fattn.FA_OK
    # fused rotary append: bad sizes, dtype code, head dim, table, alignment
    args = lambda **kw: [kw.get(n, dummy) for n in ("q", "k", "v", "pos", "cs")] + [kw.get("max_pos", 8)] + \
        [kw.get(n, dummy) for n in ("qo", "kc", "vc", "sm")] + [kw.get("N", 4), 4, 2, kw.get("d", 64), 8,
                                                                 kw.get("dt", 0), None]
    assert lib.fa_cache_append_rope(*args(N=-1)) == fattn.FA_ERR_INVALID_ARG
    assert lib.fa_cache_append_rope(*args(dt=7)) == fattn.FA_ERR_INVALID_ARG
    assert lib.fa_cache_append_rope(*args(max_pos=0)) == fattn.FA_ERR_INVALID_ARG
    assert lib.fa_cache_append_rope(*args(d=80)) == fattn.FA_ERR_UNSUPPORTED
    assert lib.fa_cache_append_rope(*args(cs=None)) == fattn.FA_ERR_INVALID_ARG
    assert lib.fa_cache_append_rope(*args(qo=P(4096 + 8))) == fattn.FA_ERR_INVALID_ARG
    assert lib.fa_cache_append_rope(*args(N=0, q=None, k=None)) == fattn.FA_OK
    # decode graph: missing handle slot, negative token count, null handle
    gargs = [None] * 3 + [0, 0] + [None] * 7 + [1, 4, 8, 4, 2, 64, 1, 0.1, 1, 1, None, 0]
    assert lib.fa_decode_graph_create(None, *gargs) == fattn.FA_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    gargs[3] = -1
    assert lib.fa_decode_graph_create(ctypes.byref(h), *gargs) == fattn.FA_ERR_INVALID_ARG
    assert h.value is None
    assert lib.fa_decode_graph_launch(None, None) == fattn.FA_ERR_INVALID_ARG
    assert lib.fa_decode_graph_kernel_count(None) == 0
    lib.fa_decode_graph_destroy(None)
    # 8-bit cache: head dim, scales, chunks too long for the decode kernel
    assert lib.fa_cache_append_fp8(dummy, dummy, dummy, dummy, dummy, 4, 2, 64, 8, 1.0, 1.0, 0,
                                   None) == fattn.FA_ERR_UNSUPPORTED
    assert lib.fa_cache_append_fp8(dummy, dummy, dummy, dummy, dummy, 4, 2, 128, 8, 0.0, 1.0, 0,
                                   None) == fattn.FA_ERR_INVALID_ARG
    need8 = lib.fa_paged_attn_workspace_size(2, 4, 8, 2, 128, 8)
    assert lib.fa_paged_attn_fp8(dummy, dummy, dummy, 1.0, 1.0, dummy, dummy, dummy, dummy, 2, 4, 8, 8, 2, 128, 16,
                                 1, 0.1, 8, 5, dummy, need8, None) == fattn.FA_ERR_UNSUPPORTED   # 4 * 5 > 16 rows
    assert lib.fa_paged_attn_fp8(dummy, dummy, dummy, 1.0, -1.0, dummy, dummy, dummy, dummy, 2, 4, 8, 8, 2, 128, 16,
                                 1, 0.1, 2, 1, dummy, need8, None) == fattn.FA_ERR_INVALID_ARG
    assert lib.fa_paged_attn_fp8(dummy, dummy, dummy, 1.0, 1.0, dummy, dummy, dummy, dummy, 2, 4, 8, 8, 2, 64, 16,
                                 1, 0.1, 2, 1, dummy, need8, None) == fattn.FA_ERR_UNSUPPORTED
    # masked prefill workspace
    assert lib.fa_prefill_masked_workspace_size(16384) >= 128 * 128 + 128 * 4
    assert lib.fa_prefill_masked(dummy, dummy, dummy, dummy, dummy, 1, 300, 4, 2, 64, 0, 0.1, None, dummy, 10,
                                 None) == fattn.FA_ERR_WORKSPACE


def test_workspace_sizes_grow(fattn):
    a = fattn.fa_paged_attn_workspace_size(64, 256, 12, 2, 128, 64)
    b = fattn.fa_paged_attn_workspace_size(128, 256, 12, 2, 128, 128)
    assert 0 < a < b
    assert a % 256 == 0
