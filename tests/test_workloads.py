"""The seeded input generators: published SplitMix64 outputs, determinism,
distribution sanity and the structure of the five workloads."""
import numpy as np
import torch

import workloads as W


def test_splitmix64_published_outputs():
    # SplitMix64 (Steele, Lea & Flood 2014; Vigna's reference C code): first
    # output for state 0 is 0xE220A8397B1DCDAF, for state 1234567 it is
    # 6457827717110365317.
    for state, first in [(0, 0xE220A8397B1DCDAF), (1234567, 6457827717110365317)]:
        z = np.array([state], dtype=np.uint64) + W._GAMMA
        assert int(W._mix64(z)[0]) == first


def test_counter_based_and_deterministic():
    a = W.normal_f32(5, W.S_Q, 1001)
    b = W.normal_f32(5, W.S_Q, 500, offset=501)
    assert np.array_equal(a[501:], b)
    assert np.array_equal(a, W.normal_f32(5, W.S_Q, 1001))
    assert not np.array_equal(a, W.normal_f32(5, W.S_K, 1001))
    x = W.normal_f32(1, W.S_V, 400000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    u = W.uniform_int(2, W.S_CTX, 128, 4096, 100000)
    assert u.min() == 128 and u.max() == 4096


def test_permutation_is_a_permutation():
    p = W.permutation(9, W.S_PERM, 20000)
    assert np.array_equal(np.sort(p), np.arange(20000))


def test_config_structures():
    c1, pg = W.config1()
    assert c1.q.dtype == torch.float32 and tuple(c1.q.shape) == (2, 64, 4, 64)
    assert len(set(pg["block_table"].reshape(-1).tolist())) == 8
    ctx = W.config3_lengths()
    assert ctx.min() >= 128 and ctx.max() <= 4096 and len(ctx) == 64
    co, ql = W.config5_lengths()
    assert co.min() >= 0 and co.max() <= 8192 and ql.min() >= 1 and ql.max() <= 512
    p = W.paged_case(3, [30, 0, 17], [2, 5, 16], 4, 2, 8, num_blocks=10, max_blocks_per_seq=4)
    bt = p.block_table.numpy()
    used = [b for s in range(3) for b in bt[s] if b >= 0]
    assert len(used) == len(set(used)) == 2 + 1 + 3  # ceil(32/16) + ceil(5/16) + ceil(33/16)
    assert p.slot_mapping.shape[0] == 23 and p.total_q == 23
    # slots land inside the owning sequence's blocks at positions ctx_old .. ctx-1
    sm = p.slot_mapping.tolist()
    assert sm[0] == bt[0, 30 // 16] * 16 + 30 % 16 and sm[1] == bt[0, 31 // 16] * 16 + 31 % 16


def test_flops_formula():
    assert W.attention_flops(2048, 2048, 128, 48, True) == 4 * 128 * 48 * (2048 * 2049 // 2)
    assert W.attention_flops(3, 10, 2, 1, True) == 4 * 2 * (8 + 9 + 10)
