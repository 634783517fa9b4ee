"""Paged attention on the GPU against the fp64 oracle: decode (split-KV +
log-sum-exp merge) and chunked prefill (tensor-core kernel), both reading K/V
only through the block table; plus the page's invariance (paging does not
change the result) and corrupted-table handling."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from fa_testutil import assert_parity, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    from paged_kv_cache_tiled_gb300 import build
    build.build()
    from paged_kv_cache_tiled_gb300 import fattn
    return fattn


def run_paged(F, p, append=True, max_q_len=None, out_guard=False):
    """Append the chunk through fa_cache_append, then fa_paged_attn."""
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    if append and p.total_q:
        F.fa_cache_append(p.k_new.cuda(), p.v_new.cuda(), kc, vc, p.slot_mapping.cuda())
    q = p.q.cuda()
    pad = 64
    buf = torch.full((p.total_q + 2 * pad, p.Hq, p.d), 3.0, dtype=torch.bfloat16, device="cuda")
    out = buf[pad:pad + p.total_q]
    F.fa_paged_attn(q, kc, vc, p.block_table.cuda(), p.ctx_lens.cuda(), p.q_lens.cuda(), causal=p.causal,
                    scale=p.scale, out=out, max_q_len=max_q_len)
    st = F.fa_get_error()
    if out_guard:
        assert torch.all(buf[:pad] == 3.0) and torch.all(buf[pad + p.total_q:] == 3.0)
    return out, kc, vc, st


def oracle_paged(p, kc_bits=None, vc_bits=None, rows=None):
    if kc_bits is None:
        kc_bits, vc_bits = oracle.cache_append(p.k_new, p.v_new, p.slot_mapping, oracle.to_bits(p.k_cache),
                                               oracle.to_bits(p.v_cache))
    if rows is None:
        return oracle.paged_attention(p.q, kc_bits, vc_bits, p.block_table, p.ctx_lens, p.q_lens, p.causal,
                                      p.scale)[0], kc_bits, vc_bits
    return oracle.paged_attention_rows(p.q, kc_bits, vc_bits, p.block_table, p.ctx_lens, p.q_lens, p.causal,
                                       p.scale, rows)[0], kc_bits, vc_bits


def test_config1_paged_decode(F):
    """Config 1: fp32 K/V appended into a 12-block permuted cache, then each
    sequence decodes its last token (ctx 64)."""
    case, pg = W.config1()
    zeros = torch.zeros(12, 2, 16, 64, dtype=torch.bfloat16, device="cuda")
    kc, vc = zeros.clone(), zeros.clone()
    F.fa_cache_append(pg["k_tokens"].cuda(), pg["v_tokens"].cuda(), kc, vc, pg["slot_mapping"].cuda())
    qd = F.fa_stage_bf16(pg["q_decode"].cuda())
    out = F.fa_paged_attn(qd, kc, vc, pg["block_table"].cuda(), pg["ctx_lens"].cuda(), pg["q_lens"].cuda(),
                          causal=True, scale=case.scale, max_q_len=1)
    assert F.fa_get_error() == F.FA_OK
    z = np.zeros((12, 2, 16, 64), np.uint16)
    ek, ev = oracle.cache_append(pg["k_tokens"], pg["v_tokens"], pg["slot_mapping"], z, z)
    assert np.array_equal(bits(kc), ek) and np.array_equal(bits(vc), ev)
    ref, _ = oracle.paged_attention(pg["q_decode"], ek, ev, pg["block_table"], pg["ctx_lens"], pg["q_lens"], True,
                                    case.scale)
    assert_parity(out, ref, "c1 decode")
    dense, _ = oracle.attention(case.q, case.k, case.v, True, case.scale)
    assert_parity(out, dense[:, 63], "c1 decode vs prefill row 63")


def test_config3_full(F):
    """Config 3 at full size: 64 sequences, ctx U[128,4096], one query each."""
    p = W.config3()
    out, kc, vc, st = run_paged(F, p, max_q_len=1, out_guard=True)
    assert st == F.FA_OK
    ref, ek, ev = oracle_paged(p)
    assert np.array_equal(bits(kc), ek)
    assert_parity(out, ref, "c3")


def test_config5_full_size(F):
    """Config 5 in full: 16 sequences, cached ctx U[0,8192] plus a chunk
    U[1,512] appended first; causal within the chunk against its full context.
    Every (token, head) row is compared with the oracle -- the tensor-core
    chunks, the packed short chunks and the decode-routed sequences alike."""
    p = W.config5()
    out, kc, vc, st = run_paged(F, p, max_q_len=int(p.q_lens.max()), out_guard=True)
    assert st == F.FA_OK
    ref, ek, ev = oracle_paged(p)
    assert np.array_equal(bits(kc), ek) and np.array_equal(bits(vc), ev)
    assert_parity(out, ref, "c5 full")


MIXED = [
    # ctx_old, q_lens, Hq, Hkv, d
    ([0, 5, 100, 31, 700, 1000, 16], [1, 2, 4, 5, 16, 17, 300], 8, 2, 128),     # g = 4: decode up to q_len 4
    ([0, 200, 63, 1], [129, 130, 1, 2], 6, 2, 128),                              # g = 3 (odd): tile pairs
    ([10, 3000, 0, 257], [1, 1, 256, 33], 4, 4, 64),                             # MHA, d = 64
    ([4095, 1, 17], [1, 513, 127], 12, 2, 128),                                  # g = 6, long chunk
    # packed query slots (128/g tokens x the g heads of a group per 128-row tile)
    ([100, 0, 7], [200, 9, 64], 4, 2, 64),                                       # g = 2, d = 64
    ([2000, 17, 0], [129, 64, 31], 16, 2, 128),                                  # g = 8
    ([0, 900, 33, 5], [70, 5, 300, 2], 16, 1, 128),                              # g = 16: 8 tokens per slot
]


@pytest.mark.parametrize("cfg", MIXED, ids=lambda c: f"g{c[2] // c[3]}d{c[4]}n{len(c[0])}")
def test_mixed_batches_full(F, cfg):
    ctx_old, ql, Hq, Hkv, d = cfg
    p = W.paged_case(41, ctx_old, ql, Hq, Hkv, d, num_blocks=400)
    out, kc, vc, st = run_paged(F, p, out_guard=True)
    assert st == F.FA_OK
    ref, _, _ = oracle_paged(p, bits(kc), bits(vc))
    assert_parity(out, ref, f"mixed {cfg}")


def test_noncausal_paged(F):
    p = W.paged_case(42, [50, 300], [3, 200], 4, 2, 128, num_blocks=40, causal=False)
    out, kc, vc, st = run_paged(F, p)
    assert st == F.FA_OK
    ref, _, _ = oracle_paged(p, bits(kc), bits(vc))
    assert_parity(out, ref, "non-causal paged")


def test_paging_does_not_change_the_result(F):
    """Same logical K/V under two different physical placements: outputs are
    bit-identical ("paging does not reduce the number of logical KV elements")."""
    args = ([70, 1500, 0, 333], [1, 40, 200, 3], 8, 2, 128)
    p1 = W.paged_case(43, *args, num_blocks=300)
    p2 = W.paged_case(43, *args, num_blocks=300, perm_seed=99)
    assert not torch.equal(p1.block_table, p2.block_table)
    o1 = run_paged(F, p1)[0]
    o2 = run_paged(F, p2)[0]
    assert torch.equal(o1, o2)


def test_nonfinite_words_in_unused_slots_do_not_leak(F):
    """Slots past each context (and unused pool blocks) hold NaN: the result is
    unchanged because masked keys never contribute, even through zero weights."""
    args = ([37, 100, 5], [1, 50, 3], 8, 2, 128)
    clean = W.paged_case(44, *args, num_blocks=30)
    dirty = W.paged_case(44, *args, num_blocks=30, fill_unused=float("nan"))
    o1 = run_paged(F, clean)[0]
    o2 = run_paged(F, dirty)[0]
    assert torch.isfinite(o2.float()).all()
    assert torch.equal(o1, o2)


def test_corrupt_block_table_is_reported(F):
    p = W.paged_case(45, [100, 20], [1, 30], 8, 2, 128, num_blocks=20)
    p.block_table[0, 2] = 20 + 7    # outside the pool (decode path)
    p.block_table[1, 1] = -3        # negative (tensor-core path)
    out, kc, vc, st = run_paged(F, p, append=False, out_guard=True)
    assert st == F.FA_ERR_BOUNDS
    assert torch.isfinite(out.float()).all()


def test_decode_stream_range_boundaries(F):
    """Decode work is split into equal page ranges per warp: many tiny segments
    fall inside one range, and one long segment spans many ranges and CTAs (its
    pieces are combined inside each CTA, then across CTAs by the merge kernel);
    every row still matches the oracle."""
    ctx_old = [0, 1, 15, 16, 31, 12000, 2, 47, 63, 64, 300, 0, 9, 100, 4, 1]
    p = W.paged_case(46, ctx_old, [1] * len(ctx_old), 12, 2, 128, num_blocks=1200)
    out, kc, vc, st = run_paged(F, p, max_q_len=1, out_guard=True)
    assert st == F.FA_OK
    ref, _, _ = oracle_paged(p, bits(kc), bits(vc))
    assert_parity(out, ref, "stream boundaries")


def test_decode_workspace_needs_no_clearing(F):
    """The decode path's workspace (partials of segments cut by range
    boundaries, read back by the merge) needs no clearing: a workspace holding
    any bytes (all ones, random words, a previous call's contents) gives the
    same output as a zeroed one."""
    p = W.paged_case(47, [3000, 17, 900, 4000, 260], [1, 1, 1, 1, 1], 12, 2, 128, num_blocks=700)
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    F.fa_cache_append(p.k_new.cuda(), p.v_new.cuda(), kc, vc, p.slot_mapping.cuda())
    args = (p.q.cuda(), kc, vc, p.block_table.cuda(), p.ctx_lens.cuda(), p.q_lens.cuda())
    n = F.fa_paged_attn_workspace_size(p.num_seqs, p.max_blocks_per_seq, p.Hq, p.Hkv, p.d, p.total_q)
    gen = torch.Generator(device="cpu").manual_seed(5)
    fills = [torch.zeros(n, dtype=torch.uint8), torch.full((n,), 255, dtype=torch.uint8),
             torch.randint(0, 256, (n,), dtype=torch.uint8, generator=gen)]
    outs = []
    for fill in fills:
        ws = fill.cuda()
        for _ in range(2):  # the second call starts from the words the first one left
            outs.append(F.fa_paged_attn(*args, causal=True, scale=p.scale, max_q_len=1, ws=ws))
            assert F.fa_get_error() == F.FA_OK
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    ref, _, _ = oracle_paged(p, bits(kc), bits(vc))
    assert_parity(outs[0], ref, "decode, uncleared workspace")


@pytest.mark.parametrize("route", ["decode", "mixed"])
def test_empty_sequences_in_the_batch(F, route):
    """Sequences with q_len = 0 -- with cached context, and with ctx_len = 0 --
    sit between decode and chunk sequences: they produce no rows and read
    nothing, every other row matches the oracle, and nothing outside the output
    is written (guard bands).  A sequence with ctx_len = q_len = 1 (the first
    token of a prompt) decodes against itself alone."""
    if route == "decode":
        ctx_old, ql = [0, 300, 0, 45, 1000, 0, 7, 2999], [0, 1, 0, 0, 1, 1, 0, 1]
    else:
        ctx_old, ql = [0, 300, 0, 45, 1000, 0, 7, 200, 0], [0, 1, 0, 0, 130, 1, 0, 3, 0]
    p = W.paged_case(48, ctx_old, ql, 12, 2, 128, num_blocks=500)
    out, kc, vc, st = run_paged(F, p, max_q_len=max(ql), out_guard=True)
    assert st == F.FA_OK
    ref, _, _ = oracle_paged(p, bits(kc), bits(vc))
    assert_parity(out, ref, f"empty sequences ({route})")



def test_max_q_len_below_a_chunk_is_reported(F):
    """max_q_len is the caller's bound on every q_len; the decode CTAs keep the
    partials of cut segments in slots sized from it (6 rows here: Hq/Hkv = 6,
    max_q_len = 1).  A two-token chunk (12 rows) under that bound is reported as
    FA_ERR_BOUNDS instead of overflowing a slot, and the next call with the true
    bound matches the oracle."""
    p = W.paged_case(43, [3000, 2000], [1, 2], 12, 2, 128, num_blocks=400)
    _, _, _, st = run_paged(F, p, max_q_len=1, out_guard=True)
    assert st == F.FA_ERR_BOUNDS
    out, kc, vc, st = run_paged(F, p, max_q_len=2, out_guard=True)
    assert st == F.FA_OK
    ref, _, _ = oracle_paged(p, bits(kc), bits(vc))
    assert_parity(out, ref, "chunk of two tokens with the true bound")


def test_many_units_per_cta(F):
    """Chunked prefill with ~10 work units per CTA: units are handed out at run
    time through a ring of four shared-memory mailboxes per CTA, so each mailbox
    is reused several times within one launch; every row matches the oracle."""
    rng = np.random.default_rng(48)
    ctx_old = rng.integers(0, 200, 40).tolist()
    q_lens = rng.integers(257, 320, 40).tolist()   # Hq/Hkv = 4: 64 tokens per unit, 5 units per kv head
    p = W.paged_case(48, ctx_old, q_lens, 32, 8, 128, num_blocks=1200)
    out, kc, vc, st = run_paged(F, p, out_guard=True)
    assert st == F.FA_OK
    ref, _, _ = oracle_paged(p, bits(kc), bits(vc))
    assert_parity(out, ref, "many units per CTA")
