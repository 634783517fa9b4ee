"""A decode step (cache append + paged attention) captured once as a CUDA
graph and replayed ("Fusion and CUDA Graphs with torch.compile": one CPU
submission for the recorded GPU work; replay needs stable addresses and
compatible shapes).  Replay must give exactly what the eager calls give, and
must follow buffer contents rewritten between replays."""
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


def _buffers(F, p):
    t = dict(q=p.q.cuda(), kn=p.k_new.cuda(), vn=p.v_new.cuda(), sm=p.slot_mapping.cuda(),
             kc=p.k_cache.cuda(), vc=p.v_cache.cuda(), bt=p.block_table.cuda(), ctx=p.ctx_lens.cuda(),
             ql=p.q_lens.cuda())
    t["out"] = torch.zeros_like(t["q"])
    t["ws"] = torch.empty(F.fa_paged_attn_workspace_size(p.num_seqs, p.max_blocks_per_seq, p.Hq, p.Hkv, p.d,
                                                         p.total_q), dtype=torch.uint8, device="cuda")
    return t


def _eager(F, p, t):
    F.fa_cache_append(t["kn"], t["vn"], t["kc"], t["vc"], t["sm"])
    F.fa_paged_attn(t["q"], t["kc"], t["vc"], t["bt"], t["ctx"], t["ql"], causal=True, scale=p.scale,
                    out=t["out"], max_q_len=int(p.q_lens.max()), ws=t["ws"])


def _graph(F, p, t):
    return F.DecodeGraph(t["q"], t["kc"], t["vc"], t["bt"], t["ctx"], t["ql"], t["out"], t["ws"], k_new=t["kn"],
                         v_new=t["vn"], slot_mapping=t["sm"], scale=p.scale, max_q_len=int(p.q_lens.max()))


def test_replay_equals_eager(F):
    p = W.paged_case(71, list(W.uniform_int(71, W.S_CTX, 100, 3000, 24)), [1] * 24, 12, 2, 128, num_blocks=6000)
    t = _buffers(F, p)
    _eager(F, p, t)                      # also the library's first-use setup, outside any capture
    assert F.fa_get_error() == F.FA_OK
    ref_out, ref_kc = t["out"].clone(), t["kc"].clone()
    t["kc"].copy_(p.k_cache.cuda())
    t["vc"].copy_(p.v_cache.cuda())
    t["out"].zero_()
    g = _graph(F, p, t)
    assert g.kernel_count == 3           # append, decode, merge
    assert torch.count_nonzero(t["out"]) == 0   # capture runs nothing
    g.replay()
    assert F.fa_get_error() == F.FA_OK
    assert torch.equal(t["out"], ref_out) and torch.equal(t["kc"], ref_kc)
    g.close()


def test_replay_follows_rewritten_inputs(F):
    """Two decode steps through one graph: before each replay the step's new
    token (q/k/v row, slot) and the context lengths are written into the
    captured buffers; each step matches the oracle on the cache as it stands."""
    n = 16
    ctx_old = list(W.uniform_int(72, W.S_CTX, 50, 2000, n))
    whole = W.paged_case(72, ctx_old, [2] * n, 8, 2, 128, num_blocks=4000, max_blocks_per_seq=130)  # both steps
    p = W.paged_case(72, ctx_old, [1] * n, 8, 2, 128, num_blocks=4000, max_blocks_per_seq=130)  # one step's shapes
    t = _buffers(F, p)
    t["bt"].copy_(whole.block_table.cuda())
    t["kc"].copy_(whole.k_cache.cuda())
    t["vc"].copy_(whole.v_cache.cuda())
    rows = lambda s: torch.arange(n) * 2 + s
    ctx0 = torch.tensor(ctx_old, dtype=torch.int32)

    def load_step(s):
        t["q"].copy_(whole.q[rows(s)].cuda())
        t["kn"].copy_(whole.k_new[rows(s)].cuda())
        t["vn"].copy_(whole.v_new[rows(s)].cuda())
        t["sm"].copy_(whole.slot_mapping[rows(s)].cuda())
        t["ctx"].copy_((ctx0 + s + 1).cuda())

    load_step(0)
    _eager(F, p, t)                      # first-use setup; also step 0 once
    t["kc"].copy_(whole.k_cache.cuda())
    t["vc"].copy_(whole.v_cache.cuda())
    g = _graph(F, p, t)
    kcb = oracle.to_bits(whole.k_cache)
    vcb = oracle.to_bits(whole.v_cache)
    ones = torch.ones(n, dtype=torch.int32)
    for s in range(2):
        load_step(s)
        g.replay()
        assert F.fa_get_error() == F.FA_OK
        kcb, vcb = oracle.cache_append(whole.k_new[rows(s)], whole.v_new[rows(s)], whole.slot_mapping[rows(s)], kcb,
                                       vcb)
        assert np.array_equal(bits(t["kc"]), kcb)
        ref, _ = oracle.paged_attention(whole.q[rows(s)], kcb, vcb, whole.block_table, ctx0 + s + 1, ones, True,
                                        p.scale)
        assert_parity(t["out"], ref, f"graph step {s}")
    g.close()


def test_replay_of_a_mixed_batch(F):
    """Decode rows and long chunks in one call: the graph holds the append, the
    decode kernel and merge, the work-list pass (captured on the library's side
    stream, forked from and joined back to the capture stream) and the
    tensor-core launch; replay equals the eager call bit for bit and the oracle."""
    ctx_old = [900, 40, 2000, 0, 310, 1500]
    q_lens = [1, 200, 2, 300, 1, 129]  # Hq/Hkv = 4: q_len <= 4 are decode rows
    p = W.paged_case(73, ctx_old, q_lens, 8, 2, 128, num_blocks=2000)
    t = _buffers(F, p)
    _eager(F, p, t)
    assert F.fa_get_error() == F.FA_OK
    ref_out, ref_kc = t["out"].clone(), t["kc"].clone()
    t["kc"].copy_(p.k_cache.cuda())
    t["vc"].copy_(p.v_cache.cuda())
    t["out"].zero_()
    g = _graph(F, p, t)
    assert g.kernel_count == 5           # append, decode, merge, work list, tensor-core prefill
    assert torch.count_nonzero(t["out"]) == 0
    g.replay()
    assert F.fa_get_error() == F.FA_OK
    assert torch.equal(t["out"], ref_out) and torch.equal(t["kc"], ref_kc)
    ref, _ = oracle.paged_attention(p.q, ref_kc.cpu(), t["vc"].cpu(), p.block_table, p.ctx_lens, p.q_lens, True,
                                    p.scale)
    assert_parity(t["out"], ref, "mixed batch, graph replay")
    # a second replay: the tensor-core kernel's unit tickets are zeroed again by
    # the captured work-list pass, so every unit is computed once more
    t["out"].zero_()
    g.replay()
    assert F.fa_get_error() == F.FA_OK
    assert torch.equal(t["out"], ref_out)
    g.close()
