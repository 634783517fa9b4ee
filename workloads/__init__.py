"""Seeded synthetic inputs for the attention workloads.

This module is shared by the CPU oracle's tests and by the GPU path's tests and
benchmark.  It contains no attention arithmetic: it only draws numbers, rounds
them to the storage dtype and lays them out (dense tensors, block tables,
context lengths, slot mappings).

Random source
-------------
Every tensor has its own stream.  A stream is a SplitMix64 generator
(Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014) whose state starts at ``key = mix64((seed << 32) ^ stream_id)``.
Draw ``i`` of the stream is ``mix64(key + (i + 1) * 0x9E3779B97F4A7C15)``,
which is SplitMix64's i-th output, so any draw can be computed directly from
its index (counter based, vectorised here with numpy ``uint64`` arithmetic).

* uniform double in [0, 1):      ``(x >> 11) * 2**-53``
* uniform integer in [lo, hi]:   ``lo + x % (hi - lo + 1)``
* N(0, 1):                       Box-Muller on draws (2i, 2i+1):
  ``r = sqrt(-2 ln(1 - u1))``, value 2i = ``r cos(2 pi u2)``, value 2i+1 =
  ``r sin(2 pi u2)``, in float64, then rounded to float32 and (for bf16
  tensors) to bfloat16 with round-to-nearest-even.
* permutations: Fisher-Yates, swapping position ``i = n-1 .. 1`` with a
  uniform integer in ``[0, i]`` taken from draw ``n-1-i``.

Workload shapes follow the five configurations the attention library is
measured on (tiny GQA correctness case, Qwen2.5-1.5B-shaped causal prefill,
paged decode batch, long-context masked prefill, mixed chunked prefill over the
paged cache), with 16-token cache blocks as in the "Paged Attention Kernels"
section of "Fast Attention Kernels and Operator Fusion".
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

BLOCK_SIZE = 16

# stream ids (one per tensor role)
S_Q, S_K, S_V, S_CTX, S_QLEN, S_PERM, S_KC, S_VC, S_KNEW, S_VNEW, S_MISC, S_POS = range(1, 13)


def _mix64(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream_id: int) -> np.uint64:
    s = np.array([((int(seed) & 0xFFFFFFFF) << 32) ^ int(stream_id)], dtype=np.uint64)
    return _mix64(s)[0]


def draws_u64(seed: int, stream_id: int, start: int, n: int) -> np.ndarray:
    """Draws ``start .. start+n-1`` of a stream as uint64."""
    key = stream_key(seed, stream_id)
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + idx * _GAMMA)


def uniform01(seed: int, stream_id: int, n: int, start: int = 0) -> np.ndarray:
    x = draws_u64(seed, stream_id, start, n)
    return (x >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def uniform_int(seed: int, stream_id: int, lo: int, hi: int, n: int, start: int = 0) -> np.ndarray:
    x = draws_u64(seed, stream_id, start, n)
    span = np.uint64(hi - lo + 1)
    return (x % span).astype(np.int64) + lo


def normal_f32(seed: int, stream_id: int, n: int, offset: int = 0) -> np.ndarray:
    """``n`` N(0,1) values (float32), values ``offset .. offset+n-1`` of the stream."""
    out = np.empty(n, dtype=np.float32)
    pos = 0
    while pos < n:
        m = min(_CHUNK, n - pos)
        first = offset + pos
        p0 = first // 2
        p1 = (first + m - 1) // 2
        npairs = p1 - p0 + 1
        u = draws_u64(seed, stream_id, 2 * p0, 2 * npairs)
        u = (u >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        u1 = u[0::2]
        u2 = u[1::2]
        r = np.sqrt(-2.0 * np.log1p(-u1))
        z = np.empty(2 * npairs, dtype=np.float64)
        z[0::2] = r * np.cos(2.0 * math.pi * u2)
        z[1::2] = r * np.sin(2.0 * math.pi * u2)
        lo = first - 2 * p0
        out[pos:pos + m] = z[lo:lo + m].astype(np.float32)
        pos += m
    return out


def permutation(seed: int, stream_id: int, n: int) -> np.ndarray:
    """Fisher-Yates permutation of 0..n-1."""
    p = np.arange(n, dtype=np.int64)
    if n <= 1:
        return p
    x = draws_u64(seed, stream_id, 0, n - 1)
    for t, i in enumerate(range(n - 1, 0, -1)):
        j = int(x[t] % np.uint64(i + 1))
        p[i], p[j] = p[j], p[i]
    return p


def normal_tensor(seed: int, stream_id: int, shape, dtype=torch.bfloat16, offset: int = 0) -> torch.Tensor:
    n = int(np.prod(shape))
    t = torch.from_numpy(normal_f32(seed, stream_id, n, offset)).reshape(shape)
    return t if dtype == torch.float32 else t.to(dtype)


# --------------------------------------------------------------------------
# contiguous prefill inputs
# --------------------------------------------------------------------------
@dataclass
class PrefillCase:
    name: str
    q: torch.Tensor  # [B, T, Hq, d]
    k: torch.Tensor  # [B, T, Hkv, d]
    v: torch.Tensor  # [B, T, Hkv, d]
    causal: bool
    scale: float
    mask: torch.Tensor | None = None  # float32 [T, T] additive, broadcast over B and H

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def T(self):
        return self.q.shape[1]

    @property
    def Hq(self):
        return self.q.shape[2]

    @property
    def Hkv(self):
        return self.k.shape[2]

    @property
    def d(self):
        return self.q.shape[3]


def prefill_case(seed: int, B: int, T: int, Hq: int, Hkv: int, d: int, causal: bool = True,
                 dtype=torch.bfloat16, scale: float | None = None, name: str = "prefill",
                 mask_kind: str | None = None) -> PrefillCase:
    q = normal_tensor(seed, S_Q, (B, T, Hq, d), dtype)
    k = normal_tensor(seed, S_K, (B, T, Hkv, d), dtype)
    v = normal_tensor(seed, S_V, (B, T, Hkv, d), dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    mask = None
    if mask_kind is not None:
        mask = make_mask(mask_kind, T, T, seed)
    return PrefillCase(name, q, k, v, causal, scale, mask)


def make_mask(kind: str, Tq: int, Tk: int, seed: int = 0) -> torch.Tensor:
    """Additive float32 masks.

    ``causal_inf``: -inf above the diagonal (j > i + Tk - Tq), 0 elsewhere.
    ``random``:     mixed values: -inf with probability 1/4, else N(0,1)
                    (every row keeps its diagonal element finite).
    ``band``:       causal with a sliding window of 300 keys.
    """
    i = torch.arange(Tq).unsqueeze(1)
    j = torch.arange(Tk).unsqueeze(0)
    if kind == "causal_inf":
        m = torch.zeros(Tq, Tk, dtype=torch.float32)
        m.masked_fill_(j > i + (Tk - Tq), float("-inf"))
        return m
    if kind == "band":
        m = torch.zeros(Tq, Tk, dtype=torch.float32)
        pos = i + (Tk - Tq)
        m.masked_fill_((j > pos) | (j < pos - 300), float("-inf"))
        return m
    if kind == "random":
        vals = torch.from_numpy(normal_f32(seed, S_MISC, Tq * Tk)).reshape(Tq, Tk)
        u = torch.from_numpy(uniform01(seed, S_MISC + 100, Tq * Tk)).reshape(Tq, Tk)
        vals = vals.masked_fill(u < 0.25, float("-inf"))
        diag = (j == i + max(0, Tk - Tq)).expand(Tq, Tk)
        vals = torch.where(diag, torch.zeros_like(vals), vals)
        return vals.contiguous()
    raise ValueError(kind)


# --------------------------------------------------------------------------
# paged cache inputs
# --------------------------------------------------------------------------
@dataclass
class PagedCase:
    """A paged-attention batch.

    The cache pool holds ``num_blocks`` blocks of ``BLOCK_SIZE`` tokens laid out
    ``[num_blocks, Hkv, BLOCK_SIZE, d]``.  Sequence ``s`` has ``ctx_old[s]``
    tokens already in the cache and a new chunk of ``q_lens[s]`` tokens whose
    keys/values (``k_new``/``v_new``, packed token-major) are appended through
    ``slot_mapping`` before attention; ``ctx_lens = ctx_old + q_lens``.
    Queries are packed ``[sum(q_lens), Hq, d]`` in sequence order.
    """
    name: str
    k_cache: torch.Tensor  # [num_blocks, Hkv, 16, d]
    v_cache: torch.Tensor
    block_table: torch.Tensor  # int32 [num_seqs, max_blocks_per_seq]
    ctx_old: torch.Tensor  # int32 [num_seqs]
    q_lens: torch.Tensor  # int32 [num_seqs]
    q: torch.Tensor  # [total_q, Hq, d]
    k_new: torch.Tensor  # [total_q, Hkv, d]
    v_new: torch.Tensor
    slot_mapping: torch.Tensor  # int32 [total_q]
    causal: bool
    scale: float

    @property
    def ctx_lens(self):
        return (self.ctx_old + self.q_lens).to(torch.int32)

    @property
    def num_seqs(self):
        return self.block_table.shape[0]

    @property
    def max_blocks_per_seq(self):
        return self.block_table.shape[1]

    @property
    def num_blocks(self):
        return self.k_cache.shape[0]

    @property
    def Hq(self):
        return self.q.shape[1]

    @property
    def Hkv(self):
        return self.k_cache.shape[1]

    @property
    def d(self):
        return self.k_cache.shape[3]

    @property
    def total_q(self):
        return self.q.shape[0]


def paged_case(seed: int, ctx_old, q_lens, Hq: int, Hkv: int, d: int, num_blocks: int,
               max_blocks_per_seq: int | None = None, dtype=torch.bfloat16, causal: bool = True,
               scale: float | None = None, name: str = "paged", fill_unused: float = 0.0,
               table_fill: int = -1, perm_seed: int | None = None) -> PagedCase:
    """Builds a paged batch from explicit per-sequence lengths.

    Block ids are disjoint random draws from the pool (a Fisher-Yates
    permutation, consumed in sequence order).  Cached values are N(0,1) drawn
    by logical position (sequence, token, head, channel) so the content does
    not depend on where the blocks land (``perm_seed`` redraws only the block
    placement).  Unused table entries hold ``table_fill``; unused cache slots
    hold ``fill_unused``.
    """
    ctx_old = np.asarray(ctx_old, dtype=np.int64)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    ns = len(ctx_old)
    ctx = ctx_old + q_lens
    nblk = (ctx + BLOCK_SIZE - 1) // BLOCK_SIZE
    mbs = int(max_blocks_per_seq) if max_blocks_per_seq is not None else max(1, int(nblk.max()))
    assert nblk.max() <= mbs and int(nblk.sum()) <= num_blocks
    perm = permutation(seed if perm_seed is None else perm_seed, S_PERM, num_blocks)
    bt = np.full((ns, mbs), table_fill, dtype=np.int32)
    pos = 0
    for s in range(ns):
        bt[s, :nblk[s]] = perm[pos:pos + nblk[s]]
        pos += nblk[s]
    if scale is None:
        scale = 1.0 / math.sqrt(d)

    max_ctx = int(ctx.max()) if ns else 0
    kc = torch.full((num_blocks, Hkv, BLOCK_SIZE, d), fill_unused, dtype=torch.float32)
    vc = torch.full((num_blocks, Hkv, BLOCK_SIZE, d), fill_unused, dtype=torch.float32)
    for s in range(ns):
        n_old = int(ctx_old[s])
        if n_old == 0:
            continue
        off = s * max_ctx * Hkv * d
        ks = torch.from_numpy(normal_f32(seed, S_KC, n_old * Hkv * d, off)).reshape(n_old, Hkv, d)
        vs = torch.from_numpy(normal_f32(seed, S_VC, n_old * Hkv * d, off)).reshape(n_old, Hkv, d)
        t = torch.arange(n_old)
        blk = torch.from_numpy(bt[s]).long()[t // BLOCK_SIZE]
        kc[blk, :, t % BLOCK_SIZE, :] = ks
        vc[blk, :, t % BLOCK_SIZE, :] = vs
    total_q = int(q_lens.sum())
    q = normal_tensor(seed, S_Q, (total_q, Hq, d), torch.float32)
    k_new = normal_tensor(seed, S_KNEW, (total_q, Hkv, d), torch.float32)
    v_new = normal_tensor(seed, S_VNEW, (total_q, Hkv, d), torch.float32)
    slots = np.empty(total_q, dtype=np.int32)
    p = 0
    for s in range(ns):
        for t in range(int(ctx_old[s]), int(ctx[s])):
            slots[p] = bt[s, t // BLOCK_SIZE] * BLOCK_SIZE + t % BLOCK_SIZE
            p += 1
    cast = (lambda x: x) if dtype == torch.float32 else (lambda x: x.to(dtype))
    return PagedCase(name, kc.to(dtype) if dtype != torch.float32 else kc,
                     vc.to(dtype) if dtype != torch.float32 else vc,
                     torch.from_numpy(bt), torch.from_numpy(ctx_old.astype(np.int32)),
                     torch.from_numpy(q_lens.astype(np.int32)), cast(q), cast(k_new), cast(v_new),
                     torch.from_numpy(slots), causal, scale)


# --------------------------------------------------------------------------
# the five measured configurations
# --------------------------------------------------------------------------
def config1():
    """Tiny GQA case: B=2, T=64, Hq=4, Hkv=2, d=64, fp32 N(0,1), causal (seed 0).

    Returns the contiguous case plus the paged layout of the same keys/values:
    12 physical blocks, block table a Fisher-Yates permutation of 0..11,
    sequence 0 on perm[0:4], sequence 1 on perm[4:8]; slot_mapping writes every
    (sequence, token) of k/v; the decode query of sequence b is q[b, 63].
    """
    seed = 0
    case = prefill_case(seed, 2, 64, 4, 2, 64, causal=True, dtype=torch.float32, name="c1")
    perm = permutation(seed, S_PERM, 12)
    bt = np.stack([perm[0:4], perm[4:8]]).astype(np.int32)
    t = np.arange(64)
    slots = np.stack([bt[b, t // 16] * 16 + t % 16 for b in range(2)]).reshape(-1).astype(np.int32)
    paged = dict(
        block_table=torch.from_numpy(bt), num_blocks=12,
        slot_mapping=torch.from_numpy(slots),  # token order (b, t)
        k_tokens=case.k.reshape(2 * 64, 2, 64), v_tokens=case.v.reshape(2 * 64, 2, 64),
        q_decode=case.q[:, 63].contiguous(),  # [2, Hq, d]
        ctx_lens=torch.tensor([64, 64], dtype=torch.int32),
        q_lens=torch.tensor([1, 1], dtype=torch.int32),
    )
    return case, paged


def config2():
    """Causal prefill shaped like Qwen2.5-1.5B attention: B=4 T=2048 Hq=12 Hkv=2 d=128 bf16 (seed 1)."""
    return prefill_case(1, 4, 2048, 12, 2, 128, causal=True, name="c2")


def config3_lengths():
    return uniform_int(2, S_CTX, 128, 4096, 64)


def config3():
    """Paged decode: 64 sequences, ctx ~ U[128,4096] (seed 2), q_len 1, Hq=12 Hkv=2 d=128, pool 20000."""
    ctx = config3_lengths()
    return paged_case(2, ctx - 1, np.ones(64, dtype=np.int64), 12, 2, 128, 20000,
                      max_blocks_per_seq=4096 // 16, name="c3")


def config4():
    """Long prefill: B=1 T=16384 Hq=32 Hkv=8 d=128 bf16 plus additive M = -inf above the diagonal (seed 3)."""
    return prefill_case(3, 1, 16384, 32, 8, 128, causal=False, name="c4", mask_kind="causal_inf")


def config5_lengths():
    ctx_old = uniform_int(4, S_CTX, 0, 8192, 16)
    q_lens = uniform_int(4, S_QLEN, 1, 512, 16)
    return ctx_old, q_lens


def config5():
    """Chunked prefill over the paged cache: 16 seqs, ctx_old ~ U[0,8192], chunk ~ U[1,512], Hq=32 Hkv=8 (seed 4)."""
    ctx_old, q_lens = config5_lengths()
    return paged_case(4, ctx_old, q_lens, 32, 8, 128, 20000, max_blocks_per_seq=(8192 + 512) // 16,
                      name="c5")


def attention_flops(Tq: int, Tk: int, d: int, heads: int, causal: bool) -> float:
    """Algorithmic flops: 4*d per unmasked (query, key) pair.

    With bottom-right causal alignment (query i sits at position i + Tk - Tq,
    Tq <= Tk) the unmasked pairs number Tq*(Tk-Tq+1) + Tq*(Tq-1)/2.
    """
    if causal:
        pairs = Tq * (Tk - Tq + 1) + Tq * (Tq - 1) // 2
    else:
        pairs = Tq * Tk
    return 4.0 * d * heads * pairs


# ------------------------------------------------------ rotary + append ----
def rope_table(max_pos: int, d: int, theta: float = 1.0e6) -> torch.Tensor:
    """Caller-side table of the fused rotary append, float32 [max_pos, d]:
    row p holds cos(p * theta**(-2j/d)) at column j and the sine at column
    d/2 + j (j < d/2), angles in float64, stored as float32.  theta = 1e6 is
    the rotary base of the Qwen2.5 models the pages' example serves."""
    j = np.arange(d // 2, dtype=np.float64)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * theta ** (-2.0 * j / d)[None, :]
    return torch.from_numpy(np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32))


@dataclass
class RopeCase:
    name: str
    q: torch.Tensor          # [N, Hq, d]
    k: torch.Tensor          # [N, Hkv, d]
    v: torch.Tensor          # [N, Hkv, d]
    positions: torch.Tensor  # int32 [N]
    slot_mapping: torch.Tensor  # int32 [N]
    cos_sin: torch.Tensor    # float32 [max_pos, d]
    num_blocks: int

    @property
    def N(self) -> int:
        return self.q.shape[0]


def rope_case(seed: int, N: int, Hq: int, Hkv: int, d: int, num_blocks: int, max_pos: int,
              dtype=torch.bfloat16, skip_every: int = 0, name: str = "rope") -> RopeCase:
    """N new tokens: q, k, v ~ N(0,1) (streams S_Q, S_KNEW, S_VNEW); positions
    uniform in [0, max_pos) (stream S_POS); distinct cache slots drawn as a
    permutation of the pool (stream S_PERM); with skip_every > 0 every
    skip_every-th token gets slot -1 (not written)."""
    q = normal_tensor(seed, S_Q, (N, Hq, d), dtype)
    k = normal_tensor(seed, S_KNEW, (N, Hkv, d), dtype)
    v = normal_tensor(seed, S_VNEW, (N, Hkv, d), dtype)
    pos = uniform_int(seed, S_POS, 0, max_pos - 1, N).astype(np.int32)
    slots = permutation(seed, S_PERM, num_blocks * BLOCK_SIZE)[:N].astype(np.int32)
    if skip_every:
        slots[::skip_every] = -1
    return RopeCase(name, q, k, v, torch.from_numpy(pos), torch.from_numpy(slots), rope_table(max_pos, d),
                    num_blocks)
