"""The allocation-free paged attention entry point.

fa_paged_attn_noalloc serves callers that cannot call cudaMalloc (device
memory reserved up front by another runtime's pool, or a plugin interface that
passes inputs and outputs but no scratch space): it runs fa_paged_attn on the
library's fixed per-device scratch array instead of a caller workspace.  Here it
is called through the C ABI and its output must equal, bit for bit, that of
fa_paged_attn with a caller-allocated workspace (both run the same
deterministic kernels on the same inputs), on several calls in a row (so later
calls start from the scratch contents an earlier call left behind); the mixed
batch is also checked against the fp64 oracle within the parity tolerance.  This file sorts last so that a run
stopping at the first failure has already run every other test."""
import ctypes

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


def _prepare(F, p):
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    F.fa_cache_append(p.k_new.cuda(), p.v_new.cuda(), kc, vc, p.slot_mapping.cuda())
    return dict(q=p.q.cuda(), kc=kc, vc=vc, bt=p.block_table.cuda(), ctx=p.ctx_lens.cuda(), ql=p.q_lens.cuda())


def _noalloc(F, p, t):
    """Raw C-ABI call; returns (status, out)."""
    out = torch.full_like(t["q"], 5.0)
    P = ctypes.c_void_p
    st = F.library().fa_paged_attn_noalloc(
        P(t["q"].data_ptr()), P(t["kc"].data_ptr()), P(t["vc"].data_ptr()), P(t["bt"].data_ptr()),
        P(t["ctx"].data_ptr()), P(t["ql"].data_ptr()), P(out.data_ptr()), p.num_seqs, p.max_blocks_per_seq,
        p.num_blocks, p.Hq, p.Hkv, p.d, 16, int(p.causal), float(p.scale), p.total_q, int(p.q_lens.max()),
        P(torch.cuda.current_stream().cuda_stream))
    return st, out


def _reference(F, p, t):
    return F.fa_paged_attn(t["q"], t["kc"], t["vc"], t["bt"], t["ctx"], t["ql"], causal=p.causal, scale=p.scale,
                           max_q_len=int(p.q_lens.max()))


def _same(got, ref, what):
    assert torch.isfinite(got.float()).all(), what
    assert torch.equal(got, ref), f"{what}: {(got != ref).sum().item()} elements differ from the workspace entry point"


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls(F):
    decode = W.paged_case(61, list(W.uniform_int(61, W.S_CTX, 127, 4095, 48)), [1] * 48, 12, 2, 128,
                          num_blocks=14000, max_blocks_per_seq=256)   # many splits -> merge partials in scratch
    mixed = W.paged_case(62, [0, 700, 31, 3000, 5], [300, 2, 129, 4, 40], 8, 2, 128, num_blocks=400)
    order = [decode, mixed, decode]
    for i, p in enumerate(order):
        assert F.fa_paged_attn_workspace_size(p.num_seqs, p.max_blocks_per_seq, p.Hq, p.Hkv, p.d,
                                              p.total_q) <= F.NOALLOC_SCRATCH_BYTES
        t = _prepare(F, p)
        ref = _reference(F, p, t)
        st, got = _noalloc(F, p, t)
        assert st == F.FA_OK, F.status_string(st)
        assert F.fa_get_error() == F.FA_OK
        _same(got, ref, f"call {i} ({p.name})")
        if p is mixed:
            kb, vb = oracle.cache_append(p.k_new, p.v_new, p.slot_mapping, oracle.to_bits(p.k_cache),
                                         oracle.to_bits(p.v_cache))
            want, _ = oracle.paged_attention(p.q, kb, vb, p.block_table, p.ctx_lens, p.q_lens, True, p.scale)
            assert_parity(got, want, f"call {i} against the oracle")


def test_noalloc_rejects_problems_beyond_the_scratch_size(F):
    # the scheduling lists grow with the number of sequences and query rows
    num_seqs, mbps, Hq, Hkv, d = 4_000_000, 64, 32, 8, 128
    assert F.fa_paged_attn_workspace_size(num_seqs, mbps, Hq, Hkv, d, num_seqs) > F.NOALLOC_SCRATCH_BYTES
    P = ctypes.c_void_p
    dummy = P(1 << 20)  # never dereferenced: the size check comes first
    st = F.library().fa_paged_attn_noalloc(dummy, dummy, dummy, dummy, dummy, dummy, dummy, num_seqs, mbps, 1 << 16,
                                           Hq, Hkv, d, 16, 1, 0.088, num_seqs, 1, None)
    assert st == F.FA_ERR_WORKSPACE
