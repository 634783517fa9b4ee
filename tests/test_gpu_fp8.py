"""The 8-bit (E4M3) KV cache against the fp64 oracle: the quantising append is
bit-exact (codes and the channel-major V layout); the decode kernel over the
8-bit cache matches the oracle's paged attention over the same codes and
scales within the attention tolerance."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from fa_testutil import assert_parity, sample_rows

pytestmark = pytest.mark.gpu
K_SCALE, V_SCALE = 0.0625, 0.03125   # N(0,1) data / scale spans the E4M3 range without saturating much


@pytest.fixture(scope="module")
def F():
    from paged_kv_cache_tiled_gb300 import build
    build.build()
    from paged_kv_cache_tiled_gb300 import fattn
    return fattn


def _u8(t):
    return t.cpu().numpy()


def _caches(F, p, k_scale=K_SCALE, v_scale=V_SCALE, dtype=torch.bfloat16):
    """8-bit caches holding the old context (from the case's bf16 cache) plus the appended tokens."""
    nb, Hkv, _, d = p.k_cache.shape
    kc = torch.full((nb, Hkv, 16, d), 0x7F, dtype=torch.uint8, device="cuda")   # NaN codes where nothing is written
    vc = torch.full((nb, Hkv, d, 16), 0x7F, dtype=torch.uint8, device="cuda")
    # old context: every slot of the blocks the table uses
    used = np.unique(p.block_table.numpy()[p.block_table.numpy() >= 0])
    slots = torch.from_numpy((used[:, None] * 16 + np.arange(16)[None, :]).ravel().astype(np.int32))
    k_old = p.k_cache[torch.from_numpy(used).long()].permute(0, 2, 1, 3).reshape(-1, Hkv, d)
    v_old = p.v_cache[torch.from_numpy(used).long()].permute(0, 2, 1, 3).reshape(-1, Hkv, d)
    F.fa_cache_append_fp8(k_old.to(dtype).cuda(), v_old.to(dtype).cuda(), kc, vc, slots.cuda(), k_scale, v_scale)
    F.fa_cache_append_fp8(p.k_new.to(dtype).cuda(), p.v_new.to(dtype).cuda(), kc, vc, p.slot_mapping.cuda(),
                          k_scale, v_scale)
    ek, ev = oracle.cache_append_fp8(k_old.to(dtype), v_old.to(dtype), slots, np.full((nb, Hkv, 16, d), 0x7F, np.uint8),
                                     np.full((nb, Hkv, d, 16), 0x7F, np.uint8), k_scale, v_scale)
    ek, ev = oracle.cache_append_fp8(p.k_new.to(dtype), p.v_new.to(dtype), p.slot_mapping, ek, ev, k_scale, v_scale)
    return kc, vc, ek, ev


def _attn(F, p, kc, vc, k_scale=K_SCALE, v_scale=V_SCALE):
    out = F.fa_paged_attn_fp8(p.q.cuda(), kc, vc, k_scale, v_scale, p.block_table.cuda(), p.ctx_lens.cuda(),
                              p.q_lens.cuda(), causal=p.causal, scale=p.scale, max_q_len=int(p.q_lens.max()))
    return out, F.fa_get_error()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_fp8_append_is_bit_exact(F, dtype):
    p = W.paged_case(91, [33, 200, 0], [3, 17, 40], 8, 2, 128, num_blocks=64, dtype=dtype)
    kc, vc, ek, ev = _caches(F, p, dtype=dtype)
    assert F.fa_get_error() == F.FA_OK
    assert np.array_equal(_u8(kc), ek) and np.array_equal(_u8(vc), ev)


def test_fp8_decode_config3_shape(F):
    """Config 3's shape (64 sequences, ctx U[128, 4096], Hq=12, Hkv=2) on a
    smaller pool of contexts: every output row against the oracle."""
    ctx_old = list(W.uniform_int(92, W.S_CTX, 127, 1500, 64))
    p = W.paged_case(92, ctx_old, [1] * 64, 12, 2, 128, num_blocks=8000)
    kc, vc, ek, ev = _caches(F, p)
    assert np.array_equal(_u8(kc), ek) and np.array_equal(_u8(vc), ev)
    out, st = _attn(F, p, kc, vc)
    assert st == F.FA_OK
    ref, _ = oracle.paged_attention_fp8(p.q, ek, ev, K_SCALE, V_SCALE, p.block_table, p.ctx_lens, p.q_lens, True,
                                        p.scale)
    assert_parity(out, ref, "fp8 decode")


def test_fp8_decode_full_config3_sampled(F):
    p = W.config3()
    kc, vc, ek, ev = _caches(F, p)
    out, st = _attn(F, p, kc, vc)
    assert st == F.FA_OK
    idx = sample_rows(p.total_q * p.Hq, 300, 7)
    tok, head = idx // p.Hq, idx % p.Hq
    rows = np.stack([tok, np.zeros_like(tok), head], axis=1)      # one query per sequence: seq = token
    ref, _ = oracle.paged_attention_fp8(p.q, ek, ev, K_SCALE, V_SCALE, p.block_table, p.ctx_lens, p.q_lens, True,
                                        p.scale, rows=rows)
    assert_parity(out[tok, head], ref, "fp8 decode, config 3 sampled")


@pytest.mark.parametrize("g_qlen", [(6, 2), (4, 4), (1, 1)])
def test_fp8_decode_gqa_and_short_chunks(F, g_qlen):
    """Several query tokens per sequence (causal within the chunk) and other
    group sizes, with contexts that end inside a block and stream ranges cut
    inside sequences (merge partials)."""
    g, ql = g_qlen
    ctx_old = [0, 1, 15, 16, 31, 3000, 2, 47, 63, 64, 300, 9]
    p = W.paged_case(93, ctx_old, [ql] * len(ctx_old), 2 * g, 2, 128, num_blocks=800)
    kc, vc, ek, ev = _caches(F, p, 0.125, 0.25)
    out, st = _attn(F, p, kc, vc, 0.125, 0.25)
    assert st == F.FA_OK
    ref, _ = oracle.paged_attention_fp8(p.q, ek, ev, 0.125, 0.25, p.block_table, p.ctx_lens, p.q_lens, True, p.scale)
    assert_parity(out, ref, f"fp8 g={g} q_len={ql}")
