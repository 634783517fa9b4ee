"""Contiguous and masked prefill on the GPU against the fp64 oracle.

Small shapes are compared element by element (several tiles, ragged tails,
odd GQA ratios, MHA, non-causal, d in {64,128}); the full-size workloads are
compared on sampled rows in the same launch configuration the benchmark uses."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from fa_testutil import assert_parity, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    from paged_kv_cache_tiled_gb300 import build
    build.build()
    from paged_kv_cache_tiled_gb300 import fattn
    return fattn


def run_dense(F, case, with_lse=True):
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    lse = torch.full((case.B, case.Hq, case.T), 7.0, device="cuda") if with_lse else None
    out = F.fa_prefill(q, k, v, causal=case.causal, scale=case.scale, lse=lse)
    assert F.fa_get_error() == F.FA_OK
    return out, lse


def test_config1_tiny_fp32_staged(F):
    """Config 1: fp32 q/k/v staged to bf16 on the GPU, then causal GQA prefill."""
    case, _ = W.config1()
    staged = [F.fa_stage_bf16(t.cuda()) for t in (case.q, case.k, case.v)]
    lse = torch.empty(2, 4, 64, device="cuda")
    out = F.fa_prefill(*staged, causal=True, scale=case.scale, lse=lse)
    assert F.fa_get_error() == F.FA_OK
    ref, ref_lse = oracle.attention(case.q, case.k, case.v, True, case.scale)  # oracle rounds fp32 itself
    assert_parity(out, ref, "c1 out")
    assert_parity(lse, ref_lse, "c1 lse")


SHAPES = [
    # B, T, Hq, Hkv, d, causal
    (2, 512, 16, 16, 64, True),    # the page's SDPA example shape (2,16,512,64), causal, MHA
    (2, 300, 6, 2, 128, True),     # odd group size, ragged tail
    (1, 1000, 8, 2, 128, False),   # non-causal, ragged
    (3, 129, 4, 1, 128, True),     # one row past a tile
    (1, 1, 2, 1, 64, True),        # single token
    (2, 700, 12, 2, 128, True),    # Qwen-like heads, ragged
    (1, 384, 3, 3, 64, False),     # MHA, odd head count
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_dense_parity(F, shape):
    B, T, Hq, Hkv, d, causal = shape
    case = W.prefill_case(100 + T, B, T, Hq, Hkv, d, causal=causal)
    out, lse = run_dense(F, case)
    ref, ref_lse = oracle.attention(case.q, case.k, case.v, causal, case.scale)
    assert_parity(out, ref, f"out {shape}")
    assert_parity(lse, ref_lse, f"lse {shape}")


def growing_scores_case(B, T, Hq, Hkv, d, seed=5):
    """q = u for every row and k_j = (j / 8) u with |u|^2 = sqrt(d): the score of key
    j is j / 8 for every query, so each 128-key tile raises a row's running maximum
    by 16 (23 in log2 units), past the rescale threshold on every tile."""
    rng = np.random.default_rng(seed)
    u = rng.standard_normal(d)
    u *= np.sqrt(np.sqrt(d)) / np.linalg.norm(u)
    j = np.arange(T, dtype=np.float64) / 8.0
    q = np.broadcast_to(u, (B, T, Hq, d)).copy()
    k = np.broadcast_to((j[:, None] * u)[None, :, None, :], (B, T, Hkv, d)).copy()
    v = rng.standard_normal((B, T, Hkv, d))
    to = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    return to(q), to(k), to(v)


@pytest.mark.parametrize("causal", [True, False])
def test_running_max_rescale_on_every_tile(F, causal):
    """Scores that grow along the keys make every KV tile rescale the output
    accumulator in place (the softmax's rare path); the result still matches the
    oracle, densely and through the paged cache."""
    B, T, Hq, Hkv, d = 1, 1024, 4, 1, 128
    q, k, v = growing_scores_case(B, T, Hq, Hkv, d)
    scale = 1.0 / np.sqrt(d)
    out = F.fa_prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    assert F.fa_get_error() == F.FA_OK
    ref, _ = oracle.attention(q, k, v, causal, scale)
    assert_parity(out, ref, f"growing scores, dense, causal={causal}")
    # the same sequence through the paged cache (one sequence, table 0 1 2 ...)
    nb = T // 16
    kc = k[0].reshape(nb, 16, Hkv, d).permute(0, 2, 1, 3).contiguous().cuda()
    vc = v[0].reshape(nb, 16, Hkv, d).permute(0, 2, 1, 3).contiguous().cuda()
    bt = torch.arange(nb, dtype=torch.int32).reshape(1, nb).cuda()
    lens = torch.tensor([T], dtype=torch.int32).cuda()
    out_p = F.fa_paged_attn(q[0].contiguous().cuda(), kc, vc, bt, lens, lens, causal=causal, scale=scale, max_q_len=T)
    assert F.fa_get_error() == F.FA_OK
    assert_parity(out_p, ref[0], f"growing scores, paged, causal={causal}")


def test_config2_full_size(F):
    """Config 2 at full size (B=4, T=2048, Hq=12, Hkv=2, d=128), every element."""
    case = W.config2()
    out, lse = run_dense(F, case)
    ref, ref_lse = oracle.attention(case.q, case.k, case.v, True, case.scale)
    assert_parity(out, ref, "c2 out")
    assert_parity(lse, ref_lse, "c2 lse")


def test_repeat_calls_are_deterministic(F):
    case = W.prefill_case(77, 2, 640, 4, 2, 128)
    a, _ = run_dense(F, case)
    b, _ = run_dense(F, case)
    assert torch.equal(a, b)


@pytest.mark.parametrize("kind,causal,d", [("random", False, 128), ("band", False, 128), ("causal_inf", True, 128),
                                           ("band", True, 128), ("band", False, 64), ("causal_inf", False, 64)])
def test_masked_parity(F, kind, causal, d):
    """Band and causal masks give interval tiles (each row keeps one run of keys,
    not always starting at the tile's first column, some rows empty), the random
    mask general tiles; T = 520 leaves a ragged last tile row and column."""
    T = 520
    case = W.prefill_case(31, 2, T, 4, 2, d, causal=causal, mask_kind=kind)
    lse = torch.empty(2, 4, T, device="cuda")
    out = F.fa_prefill_masked(case.q.cuda(), case.k.cuda(), case.v.cuda(), case.mask.cuda(), causal=causal,
                              scale=case.scale, lse=lse)
    assert F.fa_get_error() == F.FA_OK
    ref, ref_lse = oracle.attention(case.q, case.k, case.v, causal, case.scale, mask=case.mask)
    assert_parity(out, ref, f"masked {kind}")
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse.cpu().numpy()), fin)
    assert_parity(lse.cpu()[torch.from_numpy(fin)], ref_lse[fin], f"masked lse {kind}")


def test_fully_masked_rows_give_zero(F):
    T = 200
    case = W.prefill_case(32, 1, T, 2, 1, 64, causal=False)
    M = torch.zeros(T, T)
    M[5] = float("-inf")
    M[150:] = float("-inf")  # rows 150.. see nothing: a whole query tile partly empty
    lse = torch.empty(1, 2, T, device="cuda")
    out = F.fa_prefill_masked(case.q.cuda(), case.k.cuda(), case.v.cuda(), M.cuda(), scale=case.scale, lse=lse)
    assert F.fa_get_error() == F.FA_OK
    ref, ref_lse = oracle.attention(case.q, case.k, case.v, False, case.scale, mask=M)
    assert_parity(out, ref, "fully masked")
    assert torch.all(out[0, 5] == 0) and torch.all(out[0, 150:] == 0)
    assert torch.all(torch.isneginf(lse[0, :, 5])) and torch.all(torch.isneginf(lse[0, :, 150:]))


def test_config4_full_size_sampled(F):
    """Config 4 (B=1, T=16384, Hq=32, Hkv=8, additive -inf-above-diagonal M)
    through the masked path, and the same problem through the causal flag;
    sampled rows against the oracle, and the two paths agree bit for bit."""
    case = W.config4()
    q, k, v, M = case.q.cuda(), case.k.cuda(), case.v.cuda(), case.mask.cuda()
    out_m = F.fa_prefill_masked(q, k, v, M, causal=False, scale=case.scale)
    out_c = F.fa_prefill(q, k, v, causal=True, scale=case.scale)
    assert F.fa_get_error() == F.FA_OK
    assert torch.equal(out_m, out_c)
    idx = sample_rows(case.T * case.Hq, 192, 4)
    rows = np.stack([np.zeros_like(idx), idx % case.Hq, idx // case.Hq], axis=1)
    rows[:8, 2] = [0, 1, 127, 128, 8191, 16254, 16382, 16383]
    ref, _ = oracle.attention_rows(case.q, case.k, case.v, False, case.scale, rows, mask=case.mask)
    got = out_m[0, rows[:, 2], rows[:, 1]]
    assert_parity(got, ref, "c4 sampled")


@pytest.mark.parametrize("q0,Tq,Tk,causal", [(0, 300, 300, True), (128, 200, 600, True), (256, 77, 333, True),
                                              (384, 216, 600, True), (128, 100, 250, False), (0, 600, 37, False)])
def test_prefill_rows_window(F, q0, Tq, Tk, causal):
    """A window of query rows against the first Tk keys: the oracle on the
    window (causal positions counted from the start of the sequence), the rows
    of the whole-problem call bit for bit, and nothing outside the window
    written."""
    case = W.prefill_case(51, 2, 600, 6, 2, 128, causal)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    out = torch.full_like(q, 3.0)
    F.fa_prefill_rows(q, k, v, q0, Tq, Tk, causal=causal, scale=case.scale, out=out)
    assert F.fa_get_error() == F.FA_OK
    assert torch.all(out[:, :q0] == 3.0) and torch.all(out[:, q0 + Tq:] == 3.0)
    win = out[:, q0:q0 + Tq]
    if causal:
        full = F.fa_prefill(q, k, v, causal=True, scale=case.scale)
        assert torch.equal(win, full[:, q0:q0 + Tq])
        kend = q0 + Tq  # keys past the last row are masked anyway; bottom-right alignment puts row i at q0 + i
    else:
        kend = Tk
    ref, _ = oracle.attention(case.q[:, q0:q0 + Tq].contiguous(), case.k[:, :kend].contiguous(),
                              case.v[:, :kend].contiguous(), causal, case.scale)
    assert_parity(win, ref, f"rows [{q0}, {q0 + Tq}) against {Tk} keys")


def test_prefill_rows_rejects_bad_windows(F):
    case = W.prefill_case(52, 1, 256, 2, 1, 64, True)
    q, k, v = case.q.cuda(), case.k.cuda(), case.v.cuda()
    for q0, Tq, Tk, causal in ((64, 10, 256, True),     # q0 not a multiple of 128
                               (128, 200, 256, True),   # past the sequence
                               (0, 200, 100, True)):    # causal rows that see keys past Tk
        with pytest.raises(F.FattnError):
            F.fa_prefill_rows(q, k, v, q0, Tq, Tk, causal=causal, scale=case.scale)
