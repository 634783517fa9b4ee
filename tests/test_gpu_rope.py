"""Rotary position embedding fused with the cache append ("Operator Fusion",
fusion list: applying rotary position embeddings to queries and keys; updating
the KV cache while transforming key and value tensors) against the fp64
oracle.  Values are copied bit for bit; rotated values are computed in fp32 on
the GPU and in fp64 by the oracle, each rounded once to bf16, so they agree to
one bf16 unit in the last place."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu
CANARY = 0x7E7E  # bf16 pattern of about 8.4e37: no rotated or copied value here is that large


@pytest.fixture(scope="module")
def F():
    from paged_kv_cache_tiled_gb300 import build
    build.build()
    from paged_kv_cache_tiled_gb300 import fattn
    return fattn


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _check_rotated(got_bits, ref_bits, x_vals, pos, cos_sin, what):
    """|gpu - oracle| <= one bf16 ulp of the oracle value plus the fp32
    rounding error of the rotation, 2^-20 (|x_j c| + |x_partner s|) (the GPU
    rounds each product/sum to fp32 before the single bf16 rounding, which
    matters where the two terms nearly cancel).  Rows [..., d], one table row
    per leading index."""
    g = oracle.bits_to_f64(got_bits)
    r = oracle.bits_to_f64(ref_bits)
    x = np.abs(np.asarray(x_vals, dtype=np.float64))
    d = x.shape[-1]
    h = d // 2
    tab = np.abs(cos_sin.numpy().astype(np.float64))[np.asarray(pos)]
    tab = tab.reshape(tab.shape[0], *([1] * (x.ndim - 2)), d)
    c, s = tab[..., :h], tab[..., h:]
    mag = np.concatenate([x[..., :h] * c + x[..., h:] * s, x[..., h:] * c + x[..., :h] * s], axis=-1)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(r), 2.0 ** -126))) - 7)
    excess = np.abs(g - r) - (ulp + 2.0 ** -20 * mag)
    i = int(np.argmax(excess))
    assert excess.max() <= 0, f"{what}: gpu {g.flat[i]!r} oracle {r.flat[i]!r} bound {ulp.flat[i] + 2.0**-20 * mag.flat[i]:.3e}"
    assert (got_bits == ref_bits).mean() > 0.99, f"{what}: only {(got_bits == ref_bits).mean():.4f} bit-identical"


def _cache_rows(cache_bits, slots, Hkv):
    """Cache rows of the written tokens, in token order [n, Hkv, d]."""
    s = np.asarray(slots)
    return cache_bits[s // 16, :, s % 16]


def _run(F, c, dtype=torch.bfloat16):
    nb, Hkv, d = c.num_blocks, c.k.shape[1], c.q.shape[2]
    kc = torch.full((nb, Hkv, 16, d), CANARY - 0x10000 if CANARY > 0x7FFF else CANARY, dtype=torch.int16,
                    device="cuda").view(torch.bfloat16)
    vc = kc.clone()
    qo = torch.full(c.q.shape, CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    F.fa_cache_append_rope(c.q.to(dtype).cuda(), c.k.to(dtype).cuda(), c.v.to(dtype).cuda(), c.positions.cuda(),
                           c.cos_sin.cuda(), kc, vc, c.slot_mapping.cuda(), q_out=qo)
    st = F.fa_get_error()
    z = np.full((nb, Hkv, 16, d), CANARY, np.uint16)
    eq, ek, ev = oracle.rope_cache_append(c.q.to(dtype), c.k.to(dtype), c.v.to(dtype), c.positions, c.cos_sin,
                                          c.slot_mapping, z, z)
    return st, _bits(qo), _bits(kc), _bits(vc), eq, ek, ev


@pytest.mark.parametrize("d", [128, 64])
def test_rope_append_matches_oracle(F, d):
    """A chunk of new tokens the size of the mixed chunked-prefill workload
    (4096 tokens, Hq=32, Hkv=8), positions up to 8704, slots drawn from a
    20000-block pool, every 97th token unslotted."""
    c = W.rope_case(21, 4096, 32, 8, d, num_blocks=20000, max_pos=8704, skip_every=97)
    st, q, kc, vc, eq, ek, ev = _run(F, c)
    assert st == F.FA_OK
    assert np.array_equal(vc, ev)                      # values and untouched slots: exact
    assert np.array_equal(kc[ek == CANARY], ek[ek == CANARY])
    _check_rotated(q, eq, oracle.to_f64(c.q), c.positions, c.cos_sin, "q")
    w = c.slot_mapping.numpy() >= 0
    slots = c.slot_mapping.numpy()[w]
    _check_rotated(_cache_rows(kc, slots, 8), _cache_rows(ek, slots, 8), oracle.to_f64(c.k)[w],
                   c.positions.numpy()[w], c.cos_sin, "k")


def test_rope_append_fp32_inputs(F):
    c = W.rope_case(22, 300, 8, 2, 128, num_blocks=64, max_pos=4096, dtype=torch.float32)
    st, q, kc, vc, eq, ek, ev = _run(F, c, torch.float32)
    assert st == F.FA_OK
    assert np.array_equal(vc, ev)
    _check_rotated(q, eq, oracle.to_f64(c.q), c.positions, c.cos_sin, "q (fp32 in)")
    slots = c.slot_mapping.numpy()
    _check_rotated(_cache_rows(kc, slots, 2), _cache_rows(ek, slots, 2), oracle.to_f64(c.k),
                   c.positions, c.cos_sin, "k (fp32 in)")


def test_rope_append_position_out_of_range(F):
    c = W.rope_case(23, 64, 4, 2, 64, num_blocks=8, max_pos=100)
    c.positions[5] = 100
    c.positions[9] = -1
    nb, Hkv, d = c.num_blocks, 2, 64
    kc = torch.zeros(nb, Hkv, 16, d, dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    qo = torch.full(c.q.shape, 7.0, dtype=torch.bfloat16, device="cuda")
    F.fa_cache_append_rope(c.q.cuda(), c.k.cuda(), c.v.cuda(), c.positions.cuda(), c.cos_sin.cuda(), kc, vc,
                           c.slot_mapping.cuda(), q_out=qo)
    assert F.fa_get_error() == F.FA_ERR_BOUNDS
    for bad in (5, 9):
        assert torch.all(qo[bad] == 7.0)
        slot = int(c.slot_mapping[bad])
        assert torch.all(kc[slot // 16, :, slot % 16] == 0) and torch.all(vc[slot // 16, :, slot % 16] == 0)
    good = [i for i in range(64) if i not in (5, 9)]
    assert not torch.any(qo[good] == 7.0)
