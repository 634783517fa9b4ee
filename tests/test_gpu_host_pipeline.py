"""Prefill from and to host memory (fa_prefill_host): the copies and the
attention are pipelined over row chunks of the batch (last rows first), and the result is
exactly fa_prefill's output (bit for bit: each chunk's launch meets the same
query tiles with the same key tiles in the same order), which is itself
checked against the fp64 oracle here too; pinned and pageable host memory, d
in {64, 128}, causal and not, ragged T, several chunks per sequence, a
non-default stream, and buffers reused across calls."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from fa_testutil import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    from paged_kv_cache_tiled_gb300 import build
    build.build()
    from paged_kv_cache_tiled_gb300 import fattn
    return fattn


def host_copies(case, pinned):
    hs = [t.contiguous() for t in (case.q, case.k, case.v)]
    hout = torch.empty_like(case.q)
    if pinned:
        hs = [t.pin_memory() for t in hs]
        hout = hout.pin_memory()
    return hs, hout


@pytest.mark.parametrize("B,T,Hq,Hkv,d,causal,pinned", [
    (3, 300, 4, 2, 128, True, True),     # ragged final tile, GQA 2
    (2, 129, 6, 2, 64, False, False),    # d = 64, non-causal, pageable host memory
    (4, 256, 12, 2, 128, True, True),    # GQA 6 (odd pairs), whole tiles
    (1, 77, 2, 2, 128, True, True),      # a single sequence, a single chunk
    (2, 2048, 12, 2, 128, True, True),   # four 512-row chunks (config 2's row split)
    (2, 1100, 4, 1, 64, False, True),    # non-causal, several chunks
])
def test_host_pipeline_matches_device_path(F, B, T, Hq, Hkv, d, causal, pinned):
    case = W.prefill_case(31 + B, B, T, Hq, Hkv, d, causal)
    (hq, hk, hv), hout = host_copies(case, pinned)
    q, k, v = (torch.empty(t.shape, dtype=t.dtype, device="cuda") for t in (hq, hk, hv))
    out = torch.full(hq.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    F.fa_prefill_host(hq, hk, hv, hout, q, k, v, out, causal=causal, scale=case.scale)
    torch.cuda.synchronize()
    assert F.fa_get_error() == F.FA_OK
    rows = max(128, (T // 4 + 127) // 128 * 128)
    assert F.fa_last_launch_count() == (T + rows - 1) // rows  # one launch per row chunk
    # the device buffers hold the inputs and the output afterwards
    for dev, host in ((q, hq), (k, hk), (v, hv), (out, hout)):
        assert torch.equal(dev.cpu(), host)
    ref_dev = F.fa_prefill(case.q.cuda(), case.k.cuda(), case.v.cuda(), causal=causal, scale=case.scale)
    assert torch.equal(hout, ref_dev.cpu())
    ref, _ = oracle.attention(case.q, case.k, case.v, causal, case.scale)
    assert_parity(hout, ref, f"host pipeline B={B} T={T} d={d}")


def test_host_pipeline_stream_order_and_reuse(F):
    """Two calls on a side stream reuse the same device buffers; the second
    must not overwrite inputs the first is still reading, and each host output
    is complete once that stream is synchronised."""
    c1 = W.prefill_case(41, 4, 384, 4, 2, 128, True)
    c2 = W.prefill_case(42, 4, 384, 4, 2, 128, True)
    (h1q, h1k, h1v), o1 = host_copies(c1, True)
    (h2q, h2k, h2v), o2 = host_copies(c2, True)
    q, k, v = (torch.empty(t.shape, dtype=t.dtype, device="cuda") for t in (h1q, h1k, h1v))
    out = torch.empty_like(q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        F.fa_prefill_host(h1q, h1k, h1v, o1, q, k, v, out, causal=True, scale=c1.scale, stream=s)
        F.fa_prefill_host(h2q, h2k, h2v, o2, q, k, v, out, causal=True, scale=c2.scale, stream=s)
    s.synchronize()
    assert F.fa_get_error() == F.FA_OK
    for c, o in ((c1, o1), (c2, o2)):
        ref = F.fa_prefill(c.q.cuda(), c.k.cuda(), c.v.cuda(), causal=True, scale=c.scale)
        assert torch.equal(o, ref.cpu())
