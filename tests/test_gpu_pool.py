"""Paged attention over blocks shared between sequences ("Paged Attention
Kernels": blocks are shared when sequences have a common prefix).  A parent
sequence is forked three times through the block pool (on a block boundary and
inside a block, the latter copied on write with fa_copy_blocks); every
sequence then appends its own tokens.  The GPU result must match the oracle on
the same block tables and, independently, dense attention over each
sequence's logical tokens (prefix of the parent + its own)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from fa_testutil import assert_parity, bits

pytestmark = pytest.mark.gpu
Hq, Hkv, D = 8, 2, 128


@pytest.fixture(scope="module")
def F():
    from paged_kv_cache_tiled_gb300 import build
    build.build()
    from paged_kv_cache_tiled_gb300 import fattn
    return fattn


def test_shared_prefix_blocks(F):
    pool = F.BlockPool(600, 64)
    kc = torch.zeros(600, Hkv, 16, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    logical = {}
    drawn = [0]

    def write(seq, n):
        k = W.normal_tensor(81, W.S_KNEW, (n, Hkv, D), offset=drawn[0] * Hkv * D)
        v = W.normal_tensor(81, W.S_VNEW, (n, Hkv, D), offset=drawn[0] * Hkv * D)
        drawn[0] += n
        slots = torch.from_numpy(pool.append(seq, n))
        F.fa_cache_append(k.cuda(), v.cuda(), kc, vc, slots.cuda())
        ok, ov = logical.get(seq, (k[:0], v[:0]))
        logical[seq] = (torch.cat([ok, k]), torch.cat([ov, v]))

    par = pool.add_seq()
    write(par, 100)
    kids = []
    for prefix in (100, 96, 37):
        child, (src, dst) = pool.fork(par, prefix)
        if src >= 0:
            F.fa_copy_blocks(kc, vc, torch.tensor([[src, dst]], dtype=torch.int32, device="cuda"))
        pk, pv = logical[par]
        logical[child] = (pk[:prefix].clone(), pv[:prefix].clone())
        kids.append((child, prefix))
    for (child, _), n in zip(kids, (30, 5, 200)):
        write(child, n)
    write(par, 10)
    assert F.fa_get_error() == F.FA_OK

    seqs = [par] + [c for c, _ in kids]
    table, lens = pool.tables(seqs)
    ptab = table[0]
    for (child, prefix), row in zip(kids, table[1:]):   # the full prefix blocks really are shared
        assert np.array_equal(row[:prefix // 16], ptab[:prefix // 16])
        assert all(pool.refcount(int(b)) >= 2 for b in row[:prefix // 16])

    # decode for every sequence, and a 30-token chunk (the tensor-core path) for the first child
    for q_lens in ([1, 1, 1, 1], [1, 30, 1, 1]):
        ql = torch.tensor(q_lens, dtype=torch.int32)
        q = W.normal_tensor(82, W.S_Q, (int(ql.sum()), Hq, D))
        scale = 1.0 / np.sqrt(D)
        out = F.fa_paged_attn(q.cuda(), kc, vc, torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda(),
                              ql.cuda(), causal=True, scale=scale, max_q_len=max(q_lens))
        assert F.fa_get_error() == F.FA_OK
        ref, _ = oracle.paged_attention(q, bits(kc), bits(vc), table, lens, ql, True, scale)
        assert_parity(out, ref, f"paged over shared blocks, q_lens {q_lens}")
        r0 = 0
        for s, n in zip(seqs, q_lens):          # the logical sequences, contiguous, dense causal attention
            k, v = logical[s]
            dense, _ = oracle.attention(q[r0:r0 + n][None], k[None], v[None], True, scale)
            assert_parity(out[r0:r0 + n], dense[0], f"logical sequence {s}")
            r0 += n
