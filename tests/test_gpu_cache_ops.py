"""Index and byte work on the GPU must match the oracle bit for bit:
the fused cache append, the block-table gather, the fp32->bf16 staging cast and
the mask-tile classes of the masked prefill."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from fa_testutil import bits

pytestmark = pytest.mark.gpu
CANARY = 0xA5A5
CANARY_I16 = CANARY - 0x10000  # same 16 bits as a signed value


@pytest.fixture(scope="module")
def F():
    from paged_kv_cache_tiled_gb300 import build
    build.build()
    from paged_kv_cache_tiled_gb300 import fattn
    return fattn


def canary_cache(nb, Hkv, d):
    return torch.full((nb, Hkv, 16, d), CANARY_I16, dtype=torch.int16).view(torch.bfloat16).cuda()


def test_stage_bf16_matches_oracle_rounding(F):
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100003).astype(np.float32),
                        np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 3.3895314e38, 1e-40],
                                 np.float32)])
    got = F.fa_stage_bf16(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(bits(got), oracle.bf16_rne(x))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("d", [64, 128])
def test_cache_append_bit_exact(F, dtype, d):
    nb, Hkv, N = 13, 3, 40
    rng = np.random.default_rng(d)
    slots = rng.choice(nb * 16, size=N, replace=False).astype(np.int32)
    slots[[3, 17]] = -1  # skipped tokens
    k = W.normal_tensor(1, W.S_KNEW, (N, Hkv, d), dtype)
    v = W.normal_tensor(1, W.S_VNEW, (N, Hkv, d), dtype)
    kc, vc = canary_cache(nb, Hkv, d), canary_cache(nb, Hkv, d)
    F.fa_cache_append(k.cuda(), v.cuda(), kc, vc, torch.from_numpy(slots).cuda())
    assert F.fa_get_error() == F.FA_OK
    zero = np.full((nb, Hkv, 16, d), CANARY, np.uint16)
    ek, ev = oracle.cache_append(k, v, slots, zero, zero)
    assert np.array_equal(bits(kc), ek) and np.array_equal(bits(vc), ev)


def test_cache_append_out_of_range_slot_is_reported(F):
    nb, Hkv, d = 4, 2, 64
    k = torch.randn(3, Hkv, d).to(torch.bfloat16)
    v = torch.randn(3, Hkv, d).to(torch.bfloat16)
    slots = torch.tensor([5, nb * 16, 63], dtype=torch.int32)
    kc, vc = canary_cache(nb, Hkv, d), canary_cache(nb, Hkv, d)
    F.fa_cache_append(k.cuda(), v.cuda(), kc, vc, slots.cuda())
    assert F.fa_get_error() == F.FA_ERR_BOUNDS
    assert F.fa_get_error() == F.FA_OK  # reading clears the word
    zero = np.full((nb, Hkv, 16, d), CANARY, np.uint16)
    ek, _ = oracle.cache_append(k[[0, 2]], v[[0, 2]], torch.tensor([5, 63], dtype=torch.int32), zero, zero)
    assert np.array_equal(bits(kc), ek)  # valid rows written, nothing else touched


def test_gather_page_block_table_example(F):
    """The page's block table: logical blocks 0 1 2 3 -> physical 17 4 29 8."""
    table = torch.tensor([[17, 4, 29, 8]], dtype=torch.int32)
    cache = W.normal_tensor(3, W.S_KC, (30, 2, 16, 128))
    out = F.fa_debug_gather_kv(cache.cuda(), table.cuda(), torch.tensor([64], dtype=torch.int32).cuda(), 64)
    assert F.fa_get_error() == F.FA_OK
    assert np.array_equal(bits(out)[0], oracle.gather_kv(cache, table, 0, 64))


def test_gather_random_tables(F):
    p = W.paged_case(5, [0, 37, 100, 16, 255], [1, 3, 1, 1, 1], 4, 2, 64, num_blocks=64, max_blocks_per_seq=20,
                     fill_unused=0.5)
    ctx = p.ctx_lens
    max_ctx = int(ctx.max())
    sentinel = torch.full((5, max_ctx, 2, 64), CANARY_I16, dtype=torch.int16).view(torch.bfloat16).cuda()
    out = F.fa_debug_gather_kv(p.k_cache.cuda(), p.block_table.cuda(), ctx.cuda(), max_ctx, out=sentinel)
    assert F.fa_get_error() == F.FA_OK
    got = bits(out)
    for s in range(5):
        c = int(ctx[s])
        assert np.array_equal(got[s, :c], oracle.gather_kv(p.k_cache, p.block_table, s, c))
        assert np.all(got[s, c:] == CANARY)


def test_gather_corrupt_table_is_reported(F):
    table = torch.tensor([[1, 2, 99]], dtype=torch.int32)  # 99 is outside a 10-block pool
    cache = torch.zeros(10, 1, 16, 64, dtype=torch.bfloat16)
    F.fa_debug_gather_kv(cache.cuda(), table.cuda(), torch.tensor([40], dtype=torch.int32).cuda(), 40)
    assert F.fa_get_error() == F.FA_ERR_BOUNDS


@pytest.mark.parametrize("T,kind", [(300, "random"), (512, "causal_inf"), (700, "band")])
def test_mask_tile_classes_match_oracle(F, T, kind):
    case = W.prefill_case(9, 1, T, 2, 1, 64, causal=False, mask_kind=kind)
    nbytes = F.fa_prefill_masked_workspace_size(T)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    F.fa_prefill_masked(case.q.cuda(), case.k.cuda(), case.v.cuda(), case.mask.cuda(), ws=ws)
    assert F.fa_get_error() == F.FA_OK
    nt = (T + 127) // 128
    got = ws[: nt * nt].cpu().numpy().reshape(nt, nt)
    assert np.array_equal(got, oracle.mask_tile_classes(case.mask))


@pytest.mark.parametrize("Tq,Tk", [(300, 300), (128, 640), (257, 129), (1, 3)])
@pytest.mark.parametrize("kind", ["random", "band", "causal_inf"])
def test_mask_tile_classes_entry_point(F, Tq, Tk, kind):
    """The standalone class pass equals the oracle on ragged and non-square masks, classes
    and the class-3 tiles' row runs."""
    mask = W.make_mask(kind, Tq, Tk, 11)
    if kind == "random":  # plant all-zero and all--inf tiles among the mixed ones
        mask[:128, :128] = 0.0
        if Tk > 128:
            mask[:, 128:256] = float("-inf")
    shape = ((Tq + 127) // 128, (Tk + 127) // 128)
    iv = torch.full(shape + (128, 2), 7, dtype=torch.uint8, device="cuda")  # 7: left untouched
    got = F.fa_mask_tile_classes(mask.cuda(), intervals=iv).cpu().numpy()
    assert F.fa_get_error() == F.FA_OK
    want, want_iv = oracle.mask_tile_classes(mask, intervals=True)
    assert np.array_equal(got, want)
    iv = iv.cpu().numpy()
    assert np.array_equal(iv[want == 3], want_iv[want == 3])  # each row's run of kept keys
    assert (iv[want != 3] == 7).all()
    if kind == "causal_inf" and Tq > 1:  # the diagonal tiles keep a run of keys per row
        assert (want == 3).any()

