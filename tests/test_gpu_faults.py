"""Failure detection without faulting the GPU: every pipeline wait in the
kernels is bounded.  With the time-out hook on, each kernel role first waits
on a barrier that nothing arrives on (bounded at 1 ms here); the kernels record
FA_ERR_TIMEOUT, drain their copies, free tensor memory and exit, and the
context stays usable for the next call."""
import pytest
import torch

import oracle
import workloads as W
from fa_testutil import assert_parity

pytestmark = pytest.mark.gpu
DEFAULT_LIMIT_NS = 4_000_000_000


@pytest.fixture(scope="module")
def F():
    from paged_kv_cache_tiled_gb300 import build
    build.build()
    from paged_kv_cache_tiled_gb300 import fattn
    yield fattn
    fattn.fa_debug_force_timeout(False)
    fattn.fa_debug_set_wait_limit(DEFAULT_LIMIT_NS)


class forced_timeout:
    def __init__(self, F):
        self.F = F

    def __enter__(self):
        self.F.fa_debug_set_wait_limit(1_000_000)
        self.F.fa_debug_force_timeout(True)

    def __exit__(self, *exc):
        self.F.fa_debug_force_timeout(False)
        self.F.fa_debug_set_wait_limit(DEFAULT_LIMIT_NS)


def test_prefill_wait_timeout_is_reported_and_recoverable(F):
    case = W.prefill_case(51, 2, 1024, 4, 2, 128)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    assert F.fa_get_error() == F.FA_OK
    with forced_timeout(F):
        F.fa_prefill(q, k, v, causal=True, scale=case.scale)
        st = F.fa_get_error()
    assert st == F.FA_ERR_TIMEOUT
    out = F.fa_prefill(q, k, v, causal=True, scale=case.scale)
    assert F.fa_get_error() == F.FA_OK
    ref, _ = oracle.attention(case.q, case.k, case.v, True, case.scale)
    assert_parity(out, ref, "after timeout")


def test_decode_wait_timeout_is_reported_and_recoverable(F):
    p = W.paged_case(52, [3000, 2000], [1, 1], 8, 2, 128, num_blocks=400)
    args = (p.q.cuda(), p.k_cache.cuda(), p.v_cache.cuda(), p.block_table.cuda(), p.ctx_lens.cuda(),
            p.q_lens.cuda())
    with forced_timeout(F):
        F.fa_paged_attn(*args, scale=p.scale, max_q_len=1)
        st = F.fa_get_error()
    assert st == F.FA_ERR_TIMEOUT
    out = F.fa_paged_attn(*args, scale=p.scale, max_q_len=1)
    assert F.fa_get_error() == F.FA_OK
    ref, _ = oracle.paged_attention(p.q, p.k_cache, p.v_cache, p.block_table, p.ctx_lens, p.q_lens, True, p.scale)
    assert_parity(out, ref, "decode after timeout")


def test_chunked_prefill_wait_timeout(F):
    p = W.paged_case(53, [500, 40], [300, 200], 8, 2, 128, num_blocks=100)
    args = (p.q.cuda(), p.k_cache.cuda(), p.v_cache.cuda(), p.block_table.cuda(), p.ctx_lens.cuda(),
            p.q_lens.cuda())
    with forced_timeout(F):
        F.fa_paged_attn(*args, scale=p.scale)
        st = F.fa_get_error()
    assert st == F.FA_ERR_TIMEOUT
    out = F.fa_paged_attn(*args, scale=p.scale)
    assert F.fa_get_error() == F.FA_OK
    ref, _ = oracle.paged_attention(p.q, p.k_cache, p.v_cache, p.block_table, p.ctx_lens, p.q_lens, True, p.scale)
    assert_parity(out, ref, "chunked prefill after timeout")
