"""Pins the fp64 CPU oracle to facts fixed outside itself.

Each check is chosen so that a plausible slip in the oracle (a dropped scale,
a transposed operand, a wrong GQA head map, a top-left instead of bottom-right
causal alignment, a wrong block-table index, a softmax over the wrong axis)
fails at least one of them.  No expected value here comes from the GPU path.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


# ----------------------------------------------------------------- bf16 ----
def test_bf16_rne_matches_library_conversion():
    # torch's float32 -> bfloat16 conversion is round-to-nearest-even
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),  # subnormals
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, -3.3895314e38], dtype=np.float32),
    ])
    # exact halfway cases: 1 + k*2^-8 + 2^-9 for several k (ties to even)
    ties = np.array([1 + k * 2.0 ** -7 + 2.0 ** -8 for k in range(8)], dtype=np.float32)
    x = np.concatenate([x, ties, -ties])
    got = oracle.bf16_rne(x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_bf16_rne_hand_cases():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: even neighbour is 1.0 (0x3F80)
    assert oracle.bf16_rne(np.array([1 + 2.0 ** -8], np.float32))[0] == 0x3F80
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd, 0x3F81) and 1+2^-6 (even, 0x3F82)
    assert oracle.bf16_rne(np.array([1 + 3 * 2.0 ** -8], np.float32))[0] == 0x3F82
    # just above halfway rounds up
    assert oracle.bf16_rne(np.array([np.float32(1 + 2.0 ** -8 + 2.0 ** -20)], np.float32))[0] == 0x3F81
    nan = oracle.bf16_rne(np.array([np.nan], np.float32))[0]
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x7F) != 0


# --------------------------------------------------------- closed forms ----
@pytest.mark.parametrize("n", [1, 2, 5, 9])
def test_geometric_weights_closed_form(n):
    """q = e0, k_j = j e0, scale = ln 2  =>  weights 2^j / (2^n - 1).

    With v_j[c] = (c + 1) * j:  O[c] = (c+1) * ((n-2) 2^n + 2) / (2^n - 1),
    LSE = ln(2^n - 1).  Batch 2 / heads 3 carry offsets so mixed-up indices fail.
    """
    B, Hq, d = 2, 3, 4
    q = torch.zeros(B, 1, Hq, d)
    k = torch.zeros(B, n, Hq, d)
    v = torch.zeros(B, n, Hq, d)
    for b in range(B):
        for h in range(Hq):
            q[b, 0, h, 0] = 1.0
            k[b, :, h, 0] = torch.arange(n, dtype=torch.float32)
            k[b, :, h, 1:] = 7.0  # ignored: q has no weight there
            for c in range(d):
                v[b, :, h, c] = (c + 1) * torch.arange(n, dtype=torch.float32) + 10 * b + 100 * h
    out, lse = oracle.attention(bf(q), bf(k), bf(v), causal=False, scale=math.log(2.0))
    mean_j = ((n - 2) * 2.0 ** n + 2) / (2.0 ** n - 1)
    for b in range(B):
        for h in range(Hq):
            for c in range(d):
                assert out[b, 0, h, c] == pytest.approx((c + 1) * mean_j + 10 * b + 100 * h, rel=1e-13, abs=1e-12)
            assert lse[b, h, 0] == pytest.approx(math.log(2.0 ** n - 1), rel=1e-13, abs=1e-13)


def test_two_key_sigmoid_form():
    """Two keys: O = sigma(s0 - s1) v0 + (1 - sigma(s0 - s1)) v1."""
    case = W.prefill_case(11, 1, 2, 1, 1, 8, causal=False)
    out, _ = oracle.attention(case.q, case.k, case.v, causal=False, scale=0.37)
    qd = case.q.float().double().numpy()[0, :, 0]
    kd = case.k.float().double().numpy()[0, :, 0]
    vd = case.v.float().double().numpy()[0, :, 0]
    for i in range(2):
        s = 0.37 * (kd @ qd[i])
        w0 = 1.0 / (1.0 + math.exp(-(s[0] - s[1])))
        np.testing.assert_allclose(out[0, i, 0], w0 * vd[0] + (1 - w0) * vd[1], rtol=1e-12, atol=1e-12)


def test_one_hot_values_expose_probability_rows():
    """v_j = e_j makes each output row the probability row: it sums to 1 and
    P_j / P_0 = exp(s_j - s_0) with s computed exactly from small integers."""
    Tq, Tk, d = 3, 5, 8
    rng = np.random.default_rng(3)
    qi = rng.integers(-3, 4, size=(Tq, d)).astype(np.float32)
    ki = rng.integers(-3, 4, size=(Tk, d)).astype(np.float32)
    v = np.zeros((Tk, d), np.float32)
    for j in range(Tk):
        v[j, j] = 1.0
    scale = 0.25
    out, lse = oracle.attention(bf(qi[None, :, None]), bf(ki[None, :, None]), bf(v[None, :, None]),
                                causal=False, scale=scale)
    P = out[0, :, 0, :Tk]
    assert np.all(out[0, :, 0, Tk:] == 0)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    S = (qi.astype(np.int64) @ ki.astype(np.int64).T) * scale  # exact integers times 1/4
    for i in range(Tq):
        for j in range(Tk):
            assert P[i, j] / P[i, 0] == pytest.approx(math.exp(S[i, j] - S[i, 0]), rel=1e-13)
        assert lse[0, 0, i] == pytest.approx(math.log(sum(math.exp(s) for s in S[i])), rel=1e-13)


# ---------------------------------------------------------- invariants ----
def test_zero_query_gives_masked_mean_bottom_right():
    """Q = 0: every visible key has equal weight.  With Tq < Tk (bottom-right
    causal) query i averages V[0 .. i + Tk - Tq] and LSE = ln(#visible)."""
    B, Tq, Tk, Hq, Hkv, d = 2, 5, 9, 4, 2, 16
    case = W.prefill_case(5, B, Tk, Hq, Hkv, d)
    q = torch.zeros(B, Tq, Hq, d, dtype=torch.bfloat16)
    out, lse = oracle.attention(q, case.k, case.v, causal=True, scale=0.1)
    vd = case.v.double().numpy()
    for b in range(B):
        for h in range(Hq):
            hk = h // (Hq // Hkv)
            for i in range(Tq):
                vis = i + Tk - Tq + 1
                np.testing.assert_allclose(out[b, i, h], vd[b, :vis, hk].mean(axis=0), rtol=1e-13, atol=1e-14)
                assert lse[b, h, i] == pytest.approx(math.log(vis), rel=1e-14)


def test_causal_row0_is_v0_and_constant_v():
    case = W.prefill_case(6, 2, 33, 4, 2, 16)
    out, _ = oracle.attention(case.q, case.k, case.v, causal=True, scale=0.2)
    vd = case.v.double().numpy()
    for h in range(4):
        assert np.array_equal(out[:, 0, h], vd[:, 0, h // 2])
    vconst = torch.full_like(case.v, 1.75)
    out2, _ = oracle.attention(case.q, case.k, vconst, causal=True, scale=0.2)
    np.testing.assert_allclose(out2, 1.75, rtol=0, atol=1e-14)


def test_linear_in_v_and_convex_hull():
    case = W.prefill_case(7, 1, 40, 2, 1, 8)
    rng = np.random.default_rng(1)
    v1 = torch.from_numpy(rng.integers(-8, 9, size=case.v.shape).astype(np.float32))
    v2 = torch.from_numpy(rng.integers(-8, 9, size=case.v.shape).astype(np.float32))
    o1, _ = oracle.attention(case.q, case.k, bf(v1), True, 0.3)
    o2, _ = oracle.attention(case.q, case.k, bf(v2), True, 0.3)
    o12, _ = oracle.attention(case.q, case.k, bf(v1 + 2 * v2), True, 0.3)
    np.testing.assert_allclose(o12, o1 + 2 * o2, rtol=1e-12, atol=1e-12)
    vd = v1.double().numpy()
    for i in range(40):
        lo = vd[0, :i + 1, 0].min(axis=0)
        hi = vd[0, :i + 1, 0].max(axis=0)
        assert np.all(o1[0, i, :, :] >= lo - 1e-12) and np.all(o1[0, i, :, :] <= hi + 1e-12)


def test_scale_is_applied_to_scores():
    """scale 2 with q equals scale 1 with 2q (exact in bf16); scale 1 differs."""
    case = W.prefill_case(8, 1, 24, 2, 2, 32)
    a, la = oracle.attention(case.q, case.k, case.v, True, 2.0)
    b, lb = oracle.attention((case.q.float() * 2).to(torch.bfloat16), case.k, case.v, True, 1.0)
    c, _ = oracle.attention(case.q, case.k, case.v, True, 1.0)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(la, lb, rtol=1e-12, atol=1e-12)
    assert np.abs(a - c).max() > 1e-3


def test_mask_equivalences():
    """-inf-above-diagonal mask == causal flag (bitwise); adding a constant to a
    mask row changes nothing; a fully masked row gives 0 and LSE -inf."""
    case = W.prefill_case(9, 2, 37, 4, 2, 16, causal=False)
    M = W.make_mask("causal_inf", 37, 37)
    a, la = oracle.attention(case.q, case.k, case.v, causal=False, scale=0.25, mask=M)
    b, lb = oracle.attention(case.q, case.k, case.v, causal=True, scale=0.25)
    assert np.array_equal(a, b) and np.array_equal(la, lb)
    R = W.make_mask("random", 37, 37, seed=2)
    R = torch.round(R * 8) / 8  # values on a 1/8 grid so that the row shifts below are exact
    r1, _ = oracle.attention(case.q, case.k, case.v, False, 0.25, mask=R)
    R2 = R.clone()
    R2[5] += 3.0
    R2[20] -= 6.5
    r2, _ = oracle.attention(case.q, case.k, case.v, False, 0.25, mask=R2)
    np.testing.assert_allclose(r1, r2, rtol=1e-12, atol=1e-13)
    F = torch.zeros(37, 37)
    F[11] = float("-inf")
    f, lf = oracle.attention(case.q, case.k, case.v, False, 0.25, mask=F)
    assert np.all(f[:, 11] == 0) and np.all(np.isneginf(lf[:, :, 11]))
    assert np.all(np.isfinite(lf[:, :, :11]))


def test_gqa_equals_mha_with_repeated_kv():
    """Reading: query head h uses kv head h // (Hq/Hkv) (contiguous groups)."""
    case = W.prefill_case(10, 2, 30, 6, 2, 16)
    a, la = oracle.attention(case.q, case.k, case.v, True, 0.2)
    k_rep = torch.repeat_interleave(case.k, 3, dim=2)
    v_rep = torch.repeat_interleave(case.v, 3, dim=2)
    b, lb = oracle.attention(case.q, k_rep, v_rep, True, 0.2)
    assert np.array_equal(a, b) and np.array_equal(la, lb)
    # a different head map (h % Hkv) gives a different answer
    k_alt = case.k[:, :, [0, 1, 0, 1, 0, 1]]
    v_alt = case.v[:, :, [0, 1, 0, 1, 0, 1]]
    c, _ = oracle.attention(case.q, k_alt, v_alt, True, 0.2)
    assert np.abs(a - c).max() > 1e-3


def test_lse_merge_over_key_splits_equals_unsplit():
    """Attention over disjoint key parts, merged by LSE weights, equals attention
    over all keys (the page's log-sum-exp statistics are a sufficient summary)."""
    case = W.prefill_case(12, 1, 50, 2, 1, 16, causal=False)
    q1 = case.q[:, 7:8]
    full, lfull = oracle.attention(q1, case.k, case.v, False, 0.3)
    cuts = [0, 13, 13, 31, 50]  # includes an empty part
    Os, ls = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        if b == a:
            Os.append(np.zeros((2, 16)))
            ls.append(np.full(2, -np.inf))
            continue
        o, l = oracle.attention(q1, case.k[:, a:b], case.v[:, a:b], False, 0.3)
        Os.append(o[0, 0])
        ls.append(l[0, :, 0])
    for h in range(2):
        O, L = oracle.lse_merge(np.stack([o[h] for o in Os]), np.array([l[h] for l in ls]))
        np.testing.assert_allclose(O, full[0, 0, h], rtol=1e-12, atol=1e-13)
        assert L == pytest.approx(lfull[0, h, 0], rel=1e-13)


# --------------------------------------------------------------- paging ----
def _read_golden_table():
    rows = {}
    with open(os.path.join(GOLDEN, "block_table_example.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *vals = line.split()
                rows[key] = [int(x) for x in vals]
    return rows


def test_page_block_table_example_gather():
    """The page's table (logical 0 1 2 3 -> physical 17 4 29 8): a 64-token
    sequence reads token t from physical block table[t // 16], offset t % 16."""
    g = _read_golden_table()
    bs = g["block_size"][0]
    table = np.array([g["physical"]], dtype=np.int32)
    assert g["logical"] == [0, 1, 2, 3] and bs == 16
    nb, Hkv, d = 30, 2, 4
    cache = np.zeros((nb, Hkv, bs, d), dtype=np.uint16)
    for blk in range(nb):
        for h in range(Hkv):
            for o in range(bs):
                cache[blk, h, o] = [blk, h, o, 0xBEEF]
    got = oracle.gather_kv(cache, table, 0, 64)
    for t in range(64):
        for h in range(Hkv):
            assert list(got[t, h]) == [g["physical"][t // 16], h, t % 16, 0xBEEF]
    with pytest.raises(RuntimeError):  # a table entry outside the pool is an error
        oracle.gather_kv(cache, np.array([[17, 4, 29, 30]], np.int32), 0, 64)


def test_paged_equals_contiguous_under_any_permutation():
    """Paging does not change the result: the same logical K/V under two
    different physical layouts give identical outputs, equal to dense attention
    on the logical sequence assembled directly from the generator."""
    ctx_old, qlen = [37, 0, 80], [1, 16, 5]
    p1 = W.paged_case(21, ctx_old, qlen, 4, 2, 16, num_blocks=40)
    p2 = W.paged_case(21, ctx_old, qlen, 4, 2, 16, num_blocks=40, perm_seed=22)  # other placement
    assert not np.array_equal(p1.block_table.numpy(), p2.block_table.numpy())
    outs = []
    for p in (p1, p2):
        kc, vc = oracle.cache_append(p.k_new, p.v_new, p.slot_mapping, oracle.to_bits(p.k_cache),
                                     oracle.to_bits(p.v_cache))
        o, _ = oracle.paged_attention(p1.q, kc, vc, p.block_table, p.ctx_lens, p.q_lens, True, p.scale)
        outs.append(o)
    assert np.array_equal(outs[0], outs[1])
    # dense reference from logical values: cached part + new chunk, per sequence
    q0 = 0
    for s, (co, ql) in enumerate(zip(ctx_old, qlen)):
        ctx = co + ql
        kl = torch.zeros(1, ctx, 2, 16)
        vl = torch.zeros(1, ctx, 2, 16)
        if co:
            off = s * max(c + l for c, l in zip(ctx_old, qlen)) * 2 * 16
            kl[0, :co] = torch.from_numpy(W.normal_f32(21, W.S_KC, co * 32, off)).reshape(co, 2, 16)
            vl[0, :co] = torch.from_numpy(W.normal_f32(21, W.S_VC, co * 32, off)).reshape(co, 2, 16)
        kl[0, co:] = p1.k_new[q0:q0 + ql].float()
        vl[0, co:] = p1.v_new[q0:q0 + ql].float()
        dense, _ = oracle.attention(p1.q[q0:q0 + ql].unsqueeze(0), bf(kl), bf(vl), True, p1.scale)
        assert np.array_equal(dense[0], outs[0][q0:q0 + ql])
        q0 += ql


def test_config1_decode_equals_prefill_last_row():
    case, pg = W.config1()
    dense, dl = oracle.attention(case.q, case.k, case.v, True, case.scale)
    nb = pg["num_blocks"]
    zeros = np.zeros((nb, 2, 16, 64), dtype=np.uint16)
    kc, vc = oracle.cache_append(pg["k_tokens"], pg["v_tokens"], pg["slot_mapping"], zeros, zeros)
    out, lse = oracle.paged_attention(pg["q_decode"], kc, vc, pg["block_table"], pg["ctx_lens"],
                                      pg["q_lens"], True, case.scale)
    assert np.array_equal(out, dense[:, 63])
    assert np.array_equal(lse, dl[:, :, 63])


def test_chunked_paged_equals_one_shot_prefill():
    """Append a chunk, then paged attention over the full context, equals a
    one-shot causal prefill of the whole sequence restricted to the chunk rows."""
    p = W.paged_case(23, [45], [19], 4, 2, 16, num_blocks=9)
    kc, vc = oracle.cache_append(p.k_new, p.v_new, p.slot_mapping, oracle.to_bits(p.k_cache),
                                 oracle.to_bits(p.v_cache))
    out, _ = oracle.paged_attention(p.q, kc, vc, p.block_table, p.ctx_lens, p.q_lens, True, p.scale)
    kfull = torch.cat([torch.from_numpy(W.normal_f32(23, W.S_KC, 45 * 32)).reshape(45, 2, 16),
                       p.k_new.float()])
    vfull = torch.cat([torch.from_numpy(W.normal_f32(23, W.S_VC, 45 * 32)).reshape(45, 2, 16),
                       p.v_new.float()])
    qfull = torch.cat([torch.zeros(45, 4, 16), p.q.float()])
    dense, _ = oracle.attention(bf(qfull[None]), bf(kfull[None]), bf(vfull[None]), True, p.scale)
    assert np.array_equal(out, dense[0, 45:])


def test_cache_append_exact_with_canaries():
    nb, Hkv, d = 6, 2, 8
    canary = 0xA5A5
    kc = np.full((nb, Hkv, 16, d), canary, np.uint16)
    vc = np.full((nb, Hkv, 16, d), canary, np.uint16)
    k = torch.randn(5, Hkv, d)
    v = torch.randn(5, Hkv, d)
    slots = torch.tensor([3, -1, 17, 95, 40], dtype=torch.int32)
    k2, v2 = oracle.cache_append(k, v, slots, kc, vc)
    kb, vb = oracle.bf16_rne(k), oracle.bf16_rne(v)
    touched = set()
    for i, s in enumerate(slots.tolist()):
        if s < 0:
            continue
        assert np.array_equal(k2[s // 16, :, s % 16], kb[i]) and np.array_equal(v2[s // 16, :, s % 16], vb[i])
        touched.add(s)
    for s in range(nb * 16):
        if s not in touched:
            assert np.all(k2[s // 16, :, s % 16] == canary) and np.all(v2[s // 16, :, s % 16] == canary)
    with pytest.raises(RuntimeError):
        oracle.cache_append(k[:1], v[:1], torch.tensor([96], dtype=torch.int32), kc, vc)


# --------------------------------------------------------- mask classes ----
def test_mask_tile_classes_recover_planted_map():
    """Classes and row intervals planted tile by tile are what the oracle reads back."""
    rng = np.random.default_rng(4)
    Tq, Tk, bm, bn = 70, 90, 16, 32  # ragged edges on both axes
    nti, ntj = -(-Tq // bm), -(-Tk // bn)
    planted = rng.integers(0, 4, size=(nti, ntj)).astype(np.uint8)
    planted[0, :3] = [0, 1, 3]  # every class at least once
    planted[1, :2] = [2, 2]
    want_iv = np.zeros((nti, ntj, bm, 2), np.uint8)
    M = np.zeros((Tq, Tk), np.float32)
    for ti in range(nti):
        for tj in range(ntj):
            blk = M[ti * bm:(ti + 1) * bm, tj * bn:(tj + 1) * bn]
            rows, cols = blk.shape
            if planted[ti, tj] == 0:
                blk[:] = -np.inf
            elif planted[ti, tj] == 2:
                blk[:] = -np.inf
                if (ti + tj) % 2 and cols >= 3:  # a row with two separate runs of zeros
                    r = rng.integers(0, rows)
                    blk[r, 0] = 0.0
                    blk[r, 2] = 0.0
                else:  # one finite non-zero element
                    blk[rng.integers(0, rows), rng.integers(0, cols)] = 0.5
            elif planted[ti, tj] == 3:
                blk[:] = -np.inf
                for r in range(rows):
                    lo = int(rng.integers(0, cols + 1))
                    hi = int(rng.integers(lo, cols + 1))
                    if r == 0:
                        lo, hi = 0, max(1, cols - 1)  # not empty, not the whole row
                    if r == 1 and rows > 2:
                        lo, hi = 0, 0  # an empty row
                    blk[r, lo:hi] = 0.0
                    want_iv[ti, tj, r] = (lo, hi) if hi > lo else (0, 0)
    got, iv = oracle.mask_tile_classes(M, bm, bn, intervals=True)
    assert np.array_equal(got, planted)
    assert np.array_equal(oracle.mask_tile_classes(M, bm, bn), planted)
    assert np.array_equal(iv[planted == 3], want_iv[planted == 3])
    assert not iv[planted != 3].any()
    # the causal mask: diagonal tiles restrict row r to keys [0, r + 1)
    cls, iv = oracle.mask_tile_classes(W.make_mask("causal_inf", 256, 256), intervals=True)
    assert np.array_equal(cls, np.array([[3, 0], [1, 3]], np.uint8))
    for d in (0, 1):
        assert np.array_equal(iv[d, d, :, 0], np.zeros(128, np.uint8))
        assert np.array_equal(iv[d, d, :, 1], np.arange(1, 129, dtype=np.uint8))


# ---------------------------------------------------- rotary + append -----
# The rotation is a reading (rotate-half pairing, caller-given cos/sin table);
# these pin the oracle's arithmetic to properties of that rotation that do
# not depend on its own code: a hand-worked case, the identity, norm
# preservation, the relative-position property and composition, plus the
# single rounding from fp64 to bf16.

def _bits(a):
    return oracle.bf16_rne(np.asarray(a, np.float32))


def test_rope_hand_case_quarter_and_half_turn():
    # d = 4: pairs (0, 2) and (1, 3); pair 0 turned by +90 degrees, pair 1 by 180
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    cs = np.array([[0.0, -1.0, 1.0, 0.0]], np.float32)  # cos0, cos1, sin0, sin1
    y = oracle.rope_f64(x, [0], cs)
    assert np.array_equal(y, [[-3.0, -2.0, 1.0, -4.0]])


def test_rope_zero_angle_is_the_plain_append():
    c = W.rope_case(11, 40, 4, 2, 64, num_blocks=8, max_pos=32, skip_every=7)
    ident = torch.cat([torch.ones(32, 32), torch.zeros(32, 32)], dim=1)
    z = np.zeros((8, 2, 16, 64), np.uint16)
    qo, kc, vc = oracle.rope_cache_append(c.q, c.k, c.v, c.positions, ident, c.slot_mapping, z, z)
    ek, ev = oracle.cache_append(c.k, c.v, c.slot_mapping, z, z)
    assert np.array_equal(qo, oracle.to_bits(c.q))
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 128))
    tab = W.rope_table(4096, 128)
    pos = rng.integers(0, 4096, 64)
    y = oracle.rope_f64(x, pos, tab)
    n0 = x[:, :64] ** 2 + x[:, 64:] ** 2
    n1 = y[:, :64] ** 2 + y[:, 64:] ** 2
    # the stored table is cos/sin rounded to fp32, so c^2 + s^2 = 1 within ~1e-7
    assert np.allclose(n1, n0, rtol=3e-7, atol=1e-12)


def test_rope_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((1, 128))
    k = rng.standard_normal((1, 128))
    tab = W.rope_table(4096, 128)

    def score(m, n):
        return float((oracle.rope_f64(q, [m], tab) @ oracle.rope_f64(k, [n], tab).T)[0, 0])

    for m, n, shift in [(10, 3, 100), (700, 650, 2000), (5, 5, 3000)]:
        assert abs(score(m, n) - score(m + shift, n + shift)) <= 1e-4 * (1.0 + abs(score(m, n)))
    assert abs(score(40, 3) - score(3, 40)) > 1e-3  # not symmetric: it is the signed offset that counts


def test_rope_rotations_compose():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((3, 64))
    tab = W.rope_table(2048, 64)
    a, b = [17, 400, 900], [5, 600, 1000]
    twice = oracle.rope_f64(oracle.rope_f64(x, a, tab), b, tab)
    once = oracle.rope_f64(x, np.add(a, b), tab)
    assert np.allclose(twice, once, rtol=0, atol=2e-5)


def test_rope_rounds_once_from_fp64():
    # y0 = 1 * (1 + 2^-8) - 2^-15 * (-2^-15) = 1 + 2^-8 + 2^-30: just above the
    # midpoint of bf16 1.0 and 1.0078125, so it rounds up.  Rounding through
    # fp32 first would lose the 2^-30 and round the tie to even (1.0).
    q = torch.tensor([[[1.0, 0.5, 2.0 ** -15, 0.25]]]).to(torch.bfloat16)
    kv = torch.zeros(1, 1, 4, dtype=torch.bfloat16)
    cs = np.array([[1 + 2.0 ** -8, 1.0, -2.0 ** -15, 0.0]], np.float32)
    z = np.zeros((1, 1, 16, 4), np.uint16)
    qo, _, _ = oracle.rope_cache_append(q, kv, kv, [0], cs, [0], z, z)
    assert qo[0, 0, 0] == 0x3F81           # 1.0078125
    assert qo[0, 0, 2] == _bits([2.0 ** -23])[0]
    assert qo[0, 0, 1] == _bits([0.5])[0] and qo[0, 0, 3] == _bits([0.25])[0]


# ------------------------------------------------------- 8-bit cache -------
# E4M3 codes are pinned to the format's definition (bias 7, 3 mantissa bits,
# largest finite 448, S.1111.111 NaN); the 8-bit paged oracle is pinned to the
# bf16 one on values both formats hold exactly.

def test_e4m3_codes_from_the_format_definition():
    cases = {0x00: 0.0, 0x38: 1.0, 0x30: 0.5, 0x7E: 448.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9,
             0x08: 2.0 ** -6, 0x39: 1.125, 0x40: 2.0, 0xB8: -1.0, 0xFE: -448.0}
    for code, val in cases.items():
        assert oracle.e4m3_value([code])[0] == val, hex(code)
    assert np.isnan(oracle.e4m3_value([0x7F, 0xFF])).all()


def test_e4m3_every_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF, 0x80)], np.uint8)
    vals = oracle.e4m3_value(codes).astype(np.float32)
    assert np.array_equal(oracle.quant_e4m3(vals, 1.0), codes)


def test_e4m3_bisection_equals_exhaustive_search():
    rng = np.random.default_rng(12)
    mids = (oracle.e4m3_value(np.arange(0, 0x7E)) + oracle.e4m3_value(np.arange(1, 0x7F))) / 2
    x = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(2000) * 1e-3, mids, -mids,
                        np.nextafter(mids.astype(np.float32), np.float32(0)), [447.9, 448.1, 500.0, 1e30]])
    x = x.astype(np.float32)
    assert np.array_equal(oracle.quant_e4m3(x, 1.0), oracle.e4m3_rne_exhaustive(x))


def test_e4m3_ties_to_even_and_saturation():
    x = np.array([1.0625, 1.1875, 2.0 ** -10, 2.0 ** -10 * 1.01, 464.0, 1e6, -1e6, 0.0, -2.0 ** -12], np.float32)
    assert list(oracle.quant_e4m3(x, 1.0)) == [0x38, 0x3A, 0x00, 0x01, 0x7E, 0x7E, 0xFE, 0x00, 0x80]
    # the division by the scale happens in binary32 before rounding
    assert oracle.quant_e4m3(np.array([3.0], np.float32), 1.5)[0] == 0x40


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.5, 4.0)])
def test_fp8_paged_oracle_equals_bf16_on_representable_values(k_scale, v_scale):
    p = W.paged_case(31, [40, 3, 130], [1, 2, 17], 4, 2, 64, num_blocks=64)
    rng = np.random.default_rng(9)

    def representable(shape, scale):
        codes = oracle.quant_e4m3(rng.standard_normal(shape).astype(np.float32), 1.0)
        return torch.from_numpy((oracle.e4m3_value(codes) * scale).astype(np.float32))

    k_all = representable((64 * 16, 2, 64), k_scale)      # one value per pool slot
    v_all = representable((64 * 16, 2, 64), v_scale)
    slots = torch.arange(64 * 16, dtype=torch.int32)
    z16 = np.zeros((64, 2, 16, 64), np.uint16)
    kb, vb = oracle.cache_append(k_all, v_all, slots, z16, z16)
    k8, v8 = oracle.cache_append_fp8(k_all, v_all, slots, np.zeros((64, 2, 16, 64), np.uint8),
                                     np.zeros((64, 2, 64, 16), np.uint8), k_scale, v_scale)
    assert np.array_equal(oracle.e4m3_value(k8) * k_scale, oracle.bits_to_f64(kb))
    assert np.array_equal(oracle.e4m3_value(v8).transpose(0, 1, 3, 2) * v_scale, oracle.bits_to_f64(vb))
    ref, lse_ref = oracle.paged_attention(p.q, kb, vb, p.block_table, p.ctx_lens, p.q_lens, True, p.scale)
    got, lse = oracle.paged_attention_fp8(p.q, k8, v8, k_scale, v_scale, p.block_table, p.ctx_lens, p.q_lens, True,
                                          p.scale)
    assert np.array_equal(got, ref) and np.array_equal(lse, lse_ref)


# ------------------------------------------------- sampled-row drivers ----
# The full-size parity checks (the 16384-token prefill, the chunked prefill
# over the paged cache, the sampled 8-bit decode) compare the GPU against the
# oracle's row-by-row entry points, which have their own indexing: they pick a
# (batch, head, row) or (sequence, row in chunk, head) triple, reuse the K/V of
# the previous row when the (batch or sequence, kv head) repeats, and place
# each row's output and LSE by its position in the request list.  These tests
# pin them to the full-matrix functions pinned above: every requested row must
# equal the corresponding row of the full result bit for bit (both evaluate the
# attention equation of "FlashAttention-Style Kernels" with the same fp64
# operations for that row).  The row lists revisit a (batch, kv head) out of
# order, switch between query heads of one group, and interleave sequences, so
# that a stale K/V reuse, a swapped head/row field or a misplaced LSE fails.

def _revisiting_rows(rng, n, dims):
    """n random index triples inside dims, plus runs that stay on one leading
    index while the other two change, in a shuffled order."""
    rows = [tuple(int(rng.integers(0, m)) for m in dims) for _ in range(n)]
    a = int(rng.integers(0, dims[0]))
    for x in range(dims[1]):
        rows.append((a, x, int(rng.integers(0, dims[2]))))
    rows += rows[:5]                      # repeated requests are answered again
    order = rng.permutation(len(rows))
    return np.array([rows[i] for i in order], dtype=np.int32)


@pytest.mark.parametrize("causal,mask_kind,nthreads", [(True, "random", 1), (True, None, 3),
                                                       (False, "band", 2), (False, None, 1)])
def test_attention_rows_equal_full_matrix_rows(causal, mask_kind, nthreads):
    B, Tq, Tk, Hq, Hkv, d = 2, 37, 53, 6, 2, 16          # Tq < Tk (bottom-right), g = 3
    q = W.normal_tensor(41, W.S_Q, (B, Tq, Hq, d))
    k = W.normal_tensor(41, W.S_K, (B, Tk, Hkv, d))
    v = W.normal_tensor(41, W.S_V, (B, Tk, Hkv, d))
    mask = None if mask_kind is None else W.make_mask(mask_kind, Tq, Tk, 41)
    full, lse_full = oracle.attention(q, k, v, causal, 0.3, mask=mask)
    rows = _revisiting_rows(np.random.default_rng(5), 60, (B, Hq, Tq))   # (b, h, i)
    got, lse = oracle.attention_rows(q, k, v, causal, 0.3, rows, mask=mask, nthreads=nthreads)
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    assert np.array_equal(got, full[b, i, h])
    assert np.array_equal(lse, lse_full[b, h, i])
    with pytest.raises(RuntimeError):      # a row outside the problem is an error, not a read
        oracle.attention_rows(q, k, v, causal, 0.3, np.array([[0, Hq, 0]], np.int32), mask=mask)


@pytest.mark.parametrize("nthreads", [1, 4])
def test_paged_attention_rows_equal_full_rows(nthreads):
    # mixed chunks: decode (1), a chunk longer than 16, a chunk spanning blocks, an empty context
    ctx_old, qlen = [37, 0, 80, 5, 130], [1, 17, 23, 1, 40]
    p = W.paged_case(43, ctx_old, qlen, 6, 2, 16, num_blocks=60, perm_seed=44)
    kc, vc = oracle.cache_append(p.k_new, p.v_new, p.slot_mapping, oracle.to_bits(p.k_cache),
                                 oracle.to_bits(p.v_cache))
    full, lse_full = oracle.paged_attention(p.q, kc, vc, p.block_table, p.ctx_lens, p.q_lens,
                                            True, p.scale)
    rng = np.random.default_rng(6)
    rows = [(s, int(rng.integers(0, qlen[s])), int(rng.integers(0, 6)))
            for s in rng.integers(0, len(qlen), 70)]
    rows += [(4, qi, h) for h in (5, 0, 3) for qi in (39, 0, 17)]          # one sequence, heads out of order
    rows = np.array([rows[i] for i in rng.permutation(len(rows))], dtype=np.int32)
    got, lse = oracle.paged_attention_rows(p.q, kc, vc, p.block_table, p.ctx_lens, p.q_lens, True,
                                           p.scale, rows, nthreads=nthreads)
    q_start = np.concatenate([[0], np.cumsum(qlen)])
    t = q_start[rows[:, 0]] + rows[:, 1]
    assert np.array_equal(got, full[t, rows[:, 2]])
    assert np.array_equal(lse, lse_full[t, rows[:, 2]])
    with pytest.raises(RuntimeError):      # a row past its sequence's chunk is an error
        oracle.paged_attention_rows(p.q, kc, vc, p.block_table, p.ctx_lens, p.q_lens, True, p.scale,
                                    np.array([[0, 1, 0]], np.int32))


def test_fp8_paged_attention_rows_equal_full_rows():
    ctx_old, qlen = [40, 3, 130, 0], [1, 2, 17, 9]
    p = W.paged_case(45, ctx_old, qlen, 8, 2, 32, num_blocks=40)
    rng = np.random.default_rng(7)
    k_all = torch.from_numpy(rng.standard_normal((40 * 16, 2, 32)).astype(np.float32))
    v_all = torch.from_numpy(rng.standard_normal((40 * 16, 2, 32)).astype(np.float32))
    k8, v8 = oracle.cache_append_fp8(k_all, v_all, torch.arange(40 * 16, dtype=torch.int32),
                                     np.zeros((40, 2, 16, 32), np.uint8), np.zeros((40, 2, 32, 16), np.uint8),
                                     0.5, 2.0)
    full, lse_full = oracle.paged_attention_fp8(p.q, k8, v8, 0.5, 2.0, p.block_table, p.ctx_lens, p.q_lens,
                                                True, p.scale)
    rows = np.array([(s, int(rng.integers(0, qlen[s])), int(rng.integers(0, 8)))
                     for s in rng.integers(0, 4, 50)] + [(2, 16, 7), (2, 0, 0), (2, 16, 1)], dtype=np.int32)
    got, lse = oracle.paged_attention_fp8(p.q, k8, v8, 0.5, 2.0, p.block_table, p.ctx_lens, p.q_lens, True,
                                          p.scale, rows=rows, nthreads=3)
    q_start = np.concatenate([[0], np.cumsum(qlen)])
    t = q_start[rows[:, 0]] + rows[:, 1]
    assert np.array_equal(got, full[t, rows[:, 2]])
    assert np.array_equal(lse, lse_full[t, rows[:, 2]])
