"""Host-side block pool of the paged cache ("Paged Attention Kernels": blocks
allocated on demand, returned to a pool when a request ends, shared when
sequences have a common prefix).  Pure host logic through the C ABI; no GPU
needed.  The last test drives the pool with random operations and checks it
against a plain Python model of the same rules."""
import random

import numpy as np
import pytest


@pytest.fixture(scope="module")
def F():
    from paged_kv_cache_tiled_gb300 import build
    build.build()
    from paged_kv_cache_tiled_gb300 import fattn
    return fattn


def test_blocks_are_taken_on_demand(F):
    p = F.BlockPool(10, 8)
    s = p.add_seq()
    slots = p.append(s, 40)
    table, lens = p.tables([s])
    blocks = table[0, :3]
    assert len(set(blocks)) == 3 and (table[0, 3:] == -1).all() and lens[0] == 40
    assert np.array_equal(slots, [blocks[t // 16] * 16 + t % 16 for t in range(40)])
    assert p.num_free() == 7 and p.seq_len(s) == 40
    more = p.append(s, 8)           # fills block 2, no new block
    assert p.num_free() == 7 and np.array_equal(more, blocks[2] * 16 + np.arange(8, 16))
    assert p.append(s, 1)[0] // 16 not in blocks and p.num_free() == 6


def test_release_returns_blocks(F):
    p = F.BlockPool(4, 4)
    a = p.add_seq()
    p.append(a, 64)
    assert p.num_free() == 0
    with pytest.raises(F.FattnError):
        p.append(p.add_seq(), 1)
    p.release(a)
    assert p.num_free() == 4
    assert all(p.refcount(b) == 0 for b in range(4))


def test_fork_on_a_block_boundary_shares_without_copy(F):
    p = F.BlockPool(16, 8)
    par = p.add_seq()
    p.append(par, 32)
    (b0, b1), _ = p.tables([par])[0][0, :2], None
    child, cp = p.fork(par, 32)
    assert cp == (-1, -1)
    assert p.refcount(b0) == 2 and p.refcount(b1) == 2
    assert np.array_equal(p.tables([child])[0][0, :2], [b0, b1]) and p.seq_len(child) == 32
    c_slot = p.append(child, 1)[0]
    p_slot = p.append(par, 1)[0]
    assert c_slot // 16 not in (b0, b1) and p_slot // 16 not in (b0, b1, c_slot // 16)
    p.release(par)
    assert p.refcount(b0) == 1 and p.refcount(p_slot // 16) == 0
    p.release(child)
    assert p.num_free() == 16


@pytest.mark.parametrize("prefix", [40, 20, 1])
def test_fork_inside_a_block_copies_that_block(F, prefix):
    p = F.BlockPool(16, 8)
    par = p.add_seq()
    p.append(par, 40)
    pt = p.tables([par])[0][0]
    child, (src, dst) = p.fork(par, prefix)
    full = prefix // 16
    assert src == pt[full] and dst not in pt[:3] and p.refcount(dst) == 1
    ct = p.tables([child])[0][0]
    assert np.array_equal(ct[:full], pt[:full]) and ct[full] == dst and p.seq_len(child) == prefix
    assert all(p.refcount(b) == 2 for b in pt[:full]) and p.refcount(pt[full]) == 1
    assert p.append(child, 1)[0] == dst * 16 + prefix % 16   # the child writes into its own copy


def test_all_or_nothing_and_argument_errors(F):
    p = F.BlockPool(3, 8)
    s = p.add_seq()
    p.append(s, 40)
    with pytest.raises(F.FattnError) as e:
        p.append(s, 9)                       # needs a 4th block: none free
    assert e.value.status == F.FA_ERR_NO_BLOCKS and p.seq_len(s) == 40
    with pytest.raises(F.FattnError) as e:
        p.fork(s, 20)                        # partial prefix needs a fresh block
    assert e.value.status == F.FA_ERR_NO_BLOCKS
    big = F.BlockPool(100, 2)
    t = big.add_seq()
    with pytest.raises(F.FattnError) as e:
        big.append(t, 33)                    # beyond 2 blocks per sequence
    assert e.value.status == F.FA_ERR_INVALID_ARG and big.seq_len(t) == 0
    for bad in (lambda: p.release(77), lambda: p.fork(s, 41), lambda: p.tables([5])):
        with pytest.raises(F.FattnError):
            bad()
    assert p.seq_len(99) == -1 and p.refcount(-1) == -1


def test_random_operations_against_a_model(F):
    """Model: a sequence is a list of block ids and a length; a block's count
    is the number of live sequences listing it; free blocks are those with
    count 0.  Every table the pool reports must list exactly the model's
    blocks, every shared block must be full in every sequence that lists it,
    and every slot handed out must lie in the sequence's own blocks."""
    rng = random.Random(3)
    NB, MB = 64, 12
    p = F.BlockPool(NB, MB)
    model = {}                              # seq -> [blocks, len]
    for _ in range(3000):
        op = rng.random()
        live = list(model)
        if op < 0.15 or not live:
            s = p.add_seq()
            model[s] = [[], 0]
        elif op < 0.3:
            par = rng.choice(live)
            pre = rng.randint(0, model[par][1])
            need = 1 if pre % 16 else 0
            free = NB - len({b for bl, _ in model.values() for b in bl})
            if need > free:
                with pytest.raises(F.FattnError):
                    p.fork(par, pre)
                continue
            c, (src, dst) = p.fork(par, pre)
            blocks = model[par][0][:pre // 16]
            if pre % 16:
                assert src == model[par][0][pre // 16]
                blocks = blocks + [dst]
            else:
                assert (src, dst) == (-1, -1)
            model[c] = [blocks, pre]
        elif op < 0.8:
            s = rng.choice(live)
            n = rng.randint(0, 40)
            bl, ln = model[s]
            need = -(-(ln + n) // 16) - len(bl)
            free = NB - len({b for b2, _ in model.values() for b in b2})
            if -(-(ln + n) // 16) > MB or need > free:
                with pytest.raises(F.FattnError):
                    p.append(s, n)
                continue
            slots = p.append(s, n)
            table = p.tables([s])[0][0]
            bl = list(table[:-(-(ln + n) // 16)]) if ln + n else []
            assert bl[:len(model[s][0])] == model[s][0]
            assert all(sl // 16 == bl[(ln + i) // 16] and sl % 16 == (ln + i) % 16 for i, sl in enumerate(slots))
            model[s] = [bl, ln + n]
        else:
            s = rng.choice(live)
            p.release(s)
            del model[s]
        # invariants
        count = {}
        for bl, ln in model.values():
            for b in bl:
                count[b] = count.get(b, 0) + 1
        assert p.num_free() == NB - len(count)
        assert all(p.refcount(b) == count.get(b, 0) for b in range(NB))
        for s, (bl, ln) in model.items():
            table, lens = p.tables([s])
            assert lens[0] == ln and list(table[0, :len(bl)]) == bl and (table[0, len(bl):] == -1).all()
            for j, b in enumerate(bl):
                if count[b] > 1:
                    assert (j + 1) * 16 <= ln, "a shared block must be full"
