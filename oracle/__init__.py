"""fp64 CPU oracle for tiled/paged attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package.  The product library never does, and this package
imports nothing from the product: it is a plain C implementation
(``oracle.c``, built with gcc on first use) of the definitions in
"Fast Attention Kernels and Operator Fusion":

* "FlashAttention-Style Kernels": softmax(Q K^T / sqrt(d) + M) V with the full
  score matrix materialised (fp64);
* "Paged Attention Kernels": logical token t of a sequence read from physical
  block ``block_table[t // 16]`` at offset ``t % 16``;
* "Operator Fusion" (fusion list): the KV-cache append.

Every function takes torch CPU tensors or numpy arrays.  bf16 inputs are passed
as their bit patterns; fp32 q/k/v inputs are first rounded to bf16 by the
oracle's own round-to-nearest-even (``bf16_rne``), which is what the
attention library is specified to compute on.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BLOCK_SIZE = 16


def build(force: bool = False) -> str:
    """Compiles ``liboracle.so`` with gcc (plain C11, -O2, IEEE semantics)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread",
                                   "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i, l, d = ctypes.c_int, ctypes.c_long, ctypes.c_double
        lib.ora_bf16_rne.restype = ctypes.c_uint16
        lib.ora_bf16_rne.argtypes = [ctypes.c_float]
        lib.ora_bf16_rne_array.argtypes = [P, P, l]
        lib.ora_bf16_to_double_array.argtypes = [P, P, l]
        lib.ora_attention.argtypes = [P, P, P, P, P, P, i, i, i, i, i, i, i, d, i]
        lib.ora_attention_rows.argtypes = [P, P, P, P, i, i, i, i, i, i, i, d, P, l, P, P, i]
        lib.ora_gather_kv.argtypes = [P, P, i, i, i, i, i, i, i, P]
        lib.ora_cache_append.argtypes = [P, P, P, i, i, i, i, i, P, P]
        lib.ora_rope_f64.argtypes = [P, P, P, i, l, i, P]
        lib.ora_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.ora_e4m3_value.restype = d
        lib.ora_quant_e4m3.argtypes = [P, l, ctypes.c_float, P]
        lib.ora_e4m3_rne_exhaustive.argtypes = [ctypes.c_float]
        lib.ora_e4m3_rne_exhaustive.restype = ctypes.c_uint8
        lib.ora_cache_append_fp8.argtypes = [P, P, P, i, i, i, i, ctypes.c_float, ctypes.c_float, P, P]
        lib.ora_paged_attention_fp8.argtypes = [P, P, P, d, d, P, P, P, i, i, i, i, i, i, i, d, P, l, P, P, i]
        lib.ora_rope_cache_append.argtypes = [P, P, P, P, P, i, P, i, i, i, i, i, i, P, P, P]
        lib.ora_paged_attention.argtypes = [P, P, P, P, P, P, i, i, i, i, i, i, i, i, d, P, P, i]
        lib.ora_paged_attention_rows.argtypes = [P, P, P, P, P, P, i, i, i, i, i, i, i, i, d,
                                                 P, l, P, P, i]
        lib.ora_lse_merge.argtypes = [i, i, P, P, P, P]
        lib.ora_lse_merge.restype = None
        lib.ora_mask_tile_classes.argtypes = [P, i, i, i, i, P, P]
        lib.ora_mask_tile_classes.restype = None
        _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _threads(n):
    return int(n) if n else (os.cpu_count() or 1)


def _check(st, what):
    if st != 0:
        raise RuntimeError(f"oracle {what} failed with status {st}")


# ---------------------------------------------------------------- bf16 ----
def bf16_rne(x) -> np.ndarray:
    """Round fp32 values to bf16 (RNE); returns uint16 bit patterns."""
    x = np.ascontiguousarray(x.numpy() if isinstance(x, torch.Tensor) else x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    _load().ora_bf16_rne_array(_ptr(x), _ptr(y), x.size)
    return y


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    y = np.empty(bits.shape, dtype=np.float64)
    _load().ora_bf16_to_double_array(_ptr(bits), _ptr(y), bits.size)
    return y


def to_bits(t) -> np.ndarray:
    """bf16 bit patterns of an input tensor (bf16 as is, fp32 via ``bf16_rne``)."""
    if isinstance(t, np.ndarray):
        if t.dtype == np.uint16:
            return np.ascontiguousarray(t)
        return bf16_rne(t)
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if t.dtype == torch.float32:
        return bf16_rne(t)
    raise TypeError(f"unsupported dtype {t.dtype}")


def to_f64(t) -> np.ndarray:
    """Exact float64 values of an input tensor (bf16 bit patterns decoded, fp32 widened)."""
    if isinstance(t, np.ndarray) and t.dtype == np.uint16:
        return bits_to_f64(t)
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return bits_to_f64(to_bits(t))
        return t.numpy().astype(np.float64)
    return np.ascontiguousarray(t, dtype=np.float64)


def _i32(t) -> np.ndarray:
    a = t.numpy() if isinstance(t, torch.Tensor) else np.asarray(t)
    return np.ascontiguousarray(a, dtype=np.int32)


def _f32(t) -> np.ndarray | None:
    if t is None:
        return None
    a = t.numpy() if isinstance(t, torch.Tensor) else np.asarray(t)
    return np.ascontiguousarray(a, dtype=np.float32)


# ------------------------------------------------------------ attention ---
def attention(q, k, v, causal: bool, scale: float, mask=None, nthreads=None):
    """Dense attention. q [B,Tq,Hq,d], k/v [B,Tk,Hkv,d] -> (out f64 [B,Tq,Hq,d], lse f64 [B,Hq,Tq])."""
    qb, kb, vb = to_bits(q), to_bits(k), to_bits(v)
    B, Tq, Hq, d = qb.shape
    Tk, Hkv = kb.shape[1], kb.shape[2]
    m = _f32(mask)
    out = np.zeros((B, Tq, Hq, d), dtype=np.float64)
    lse = np.zeros((B, Hq, Tq), dtype=np.float64)
    st = _load().ora_attention(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(m), _ptr(out), _ptr(lse),
                               B, Tq, Tk, Hq, Hkv, d, int(causal), float(scale), _threads(nthreads))
    _check(st, "attention")
    return out, lse


def attention_rows(q, k, v, causal: bool, scale: float, rows, mask=None, nthreads=None):
    """Selected rows (b, h, i) of dense attention -> (out f64 [n, d], lse f64 [n])."""
    qb, kb, vb = to_bits(q), to_bits(k), to_bits(v)
    B, Tq, Hq, d = qb.shape
    Tk, Hkv = kb.shape[1], kb.shape[2]
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    m = _f32(mask)
    out = np.zeros((len(r), d), dtype=np.float64)
    lse = np.zeros(len(r), dtype=np.float64)
    st = _load().ora_attention_rows(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(m), B, Tq, Tk, Hq, Hkv, d,
                                    int(causal), float(scale), _ptr(r), len(r), _ptr(out),
                                    _ptr(lse), _threads(nthreads))
    _check(st, "attention_rows")
    return out, lse


# ---------------------------------------------------------------- paged ---
def gather_kv(cache, block_table, seq: int, ctx_len: int, num_blocks: int | None = None):
    """Contiguous bf16 bits [ctx_len, Hkv, d] of one sequence read through its block table."""
    cb = to_bits(cache)
    bt = _i32(block_table)
    nb, Hkv, bs, d = cb.shape
    out = np.zeros((ctx_len, Hkv, d), dtype=np.uint16)
    st = _load().ora_gather_kv(_ptr(cb), _ptr(bt), bt.shape[1], nb if num_blocks is None else num_blocks,
                               seq, ctx_len, Hkv, d, bs, _ptr(out))
    _check(st, "gather_kv")
    return out


def cache_append(k, v, slot_mapping, k_cache_bits: np.ndarray, v_cache_bits: np.ndarray):
    """Writes new tokens into copies of the caches (bf16 bits); returns the new caches."""
    kb, vb = to_bits(k), to_bits(v)
    N, Hkv, d = kb.shape
    kc = np.ascontiguousarray(k_cache_bits, dtype=np.uint16).copy()
    vc = np.ascontiguousarray(v_cache_bits, dtype=np.uint16).copy()
    nb, _, bs, _ = kc.shape
    sm = _i32(slot_mapping)
    st = _load().ora_cache_append(_ptr(kb), _ptr(vb), _ptr(sm), N, Hkv, d, nb, bs, _ptr(kc), _ptr(vc))
    _check(st, "cache_append")
    return kc, vc


def rope_f64(x, positions, cos_sin) -> np.ndarray:
    """Rotate rows x f64 [nrows, d] (row i at table row positions[i]) with the
    rotate-half rotary embedding of table cos_sin f32 [max_pos, d]; fp64 result."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    nrows, d = x.shape
    pos = _i32(positions)
    cs = _f32(cos_sin)
    y = np.empty_like(x)
    _check(_load().ora_rope_f64(_ptr(x), _ptr(pos), _ptr(cs), cs.shape[0], nrows, d, _ptr(y)), "rope_f64")
    return y


def rope_cache_append(q, k, v, positions, cos_sin, slot_mapping, k_cache_bits: np.ndarray,
                      v_cache_bits: np.ndarray):
    """Rotary embedding fused with the append: returns (q_out bits [N,Hq,d], new k cache, new v cache).
    q and k are rotated from their exact values (bf16 or fp32); v is stored as bf16 (fp32 rounded, RNE)."""
    qb, kb, vb = to_f64(q), to_f64(k), to_bits(v)
    N, Hq, d = qb.shape
    Hkv = kb.shape[1]
    kc = np.ascontiguousarray(k_cache_bits, dtype=np.uint16).copy()
    vc = np.ascontiguousarray(v_cache_bits, dtype=np.uint16).copy()
    nb, _, bs, _ = kc.shape
    pos, sm, cs = _i32(positions), _i32(slot_mapping), _f32(cos_sin)
    qo = np.zeros(qb.shape, dtype=np.uint16)
    st = _load().ora_rope_cache_append(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(pos), _ptr(cs), cs.shape[0], _ptr(sm), N,
                                       Hq, Hkv, d, nb, bs, _ptr(qo), _ptr(kc), _ptr(vc))
    _check(st, "rope_cache_append")
    return qo, kc, vc


# ---------------------------------------------------------- fp8 cache ----
def e4m3_value(codes) -> np.ndarray:
    """Values (float64) of E4M3 codes."""
    codes = np.asarray(codes, dtype=np.uint8)
    lib = _load()
    return np.array([lib.ora_e4m3_value(int(c)) for c in codes.ravel()], dtype=np.float64).reshape(codes.shape)


def quant_e4m3(x, scale: float) -> np.ndarray:
    """E4M3 codes of float32(x) / float32(scale) (round to nearest even, saturating)."""
    x = np.ascontiguousarray(x.numpy() if isinstance(x, torch.Tensor) else x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().ora_quant_e4m3(_ptr(x), x.size, float(scale), _ptr(out))
    return out


def e4m3_rne_exhaustive(x) -> np.ndarray:
    """E4M3 codes of float32 values by exhaustive nearest-code search (cross-check of quant_e4m3)."""
    x = np.asarray(x, dtype=np.float32)
    lib = _load()
    return np.array([lib.ora_e4m3_rne_exhaustive(float(v)) for v in x.ravel()], np.uint8).reshape(x.shape)


def cache_append_fp8(k, v, slot_mapping, k_cache: np.ndarray, v_cache: np.ndarray, k_scale: float, v_scale: float):
    """Append into copies of the 8-bit caches (k [nb,Hkv,16,d], v [nb,Hkv,d,16]); returns them."""
    kf = to_f64(k).astype(np.float32)
    vf = to_f64(v).astype(np.float32)
    N, Hkv, d = kf.shape
    kc = np.ascontiguousarray(k_cache, dtype=np.uint8).copy()
    vc = np.ascontiguousarray(v_cache, dtype=np.uint8).copy()
    sm = _i32(slot_mapping)
    st = _load().ora_cache_append_fp8(_ptr(kf), _ptr(vf), _ptr(sm), N, Hkv, d, kc.shape[0], float(k_scale),
                                      float(v_scale), _ptr(kc), _ptr(vc))
    _check(st, "cache_append_fp8")
    return kc, vc


def paged_attention_fp8(q, k_cache, v_cache, k_scale: float, v_scale: float, block_table, ctx_lens, q_lens,
                        causal: bool, scale: float, rows=None, nthreads=None):
    """Paged attention over the 8-bit caches -> (out f64 [rows or sum q, Hq, d], lse)."""
    qb = to_bits(q)
    total_q, Hq, d = qb.shape
    kc = np.ascontiguousarray(k_cache, dtype=np.uint8)
    vc = np.ascontiguousarray(v_cache, dtype=np.uint8)
    nb, Hkv = kc.shape[0], kc.shape[1]
    bt, cl, ql = _i32(block_table), _i32(ctx_lens), _i32(q_lens)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n_out = total_q * Hq if r is None else len(r)
    out = np.empty((n_out, d), np.float64)
    lse = np.empty(n_out, np.float64)
    st = _load().ora_paged_attention_fp8(_ptr(qb), _ptr(kc), _ptr(vc), float(k_scale), float(v_scale), _ptr(bt),
                                         _ptr(cl), _ptr(ql), bt.shape[0], bt.shape[1], nb, Hq, Hkv, d, int(causal),
                                         float(scale), _ptr(r), 0 if r is None else len(r), _ptr(out), _ptr(lse),
                                         _threads(nthreads))
    _check(st, "paged_attention_fp8")
    if r is None:
        return out.reshape(total_q, Hq, d), lse.reshape(total_q, Hq)
    return out, lse


def paged_attention(q, k_cache, v_cache, block_table, ctx_lens, q_lens, causal: bool, scale: float,
                    nthreads=None):
    """Paged attention over packed queries -> (out f64 [sum q, Hq, d], lse f64 [sum q, Hq])."""
    qb, kc, vc = to_bits(q), to_bits(k_cache), to_bits(v_cache)
    bt, cl, ql = _i32(block_table), _i32(ctx_lens), _i32(q_lens)
    tq, Hq, d = qb.shape
    nb, Hkv, bs, _ = kc.shape
    out = np.zeros((tq, Hq, d), dtype=np.float64)
    lse = np.zeros((tq, Hq), dtype=np.float64)
    st = _load().ora_paged_attention(_ptr(qb), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl), _ptr(ql),
                                     len(cl), bt.shape[1], nb, Hq, Hkv, d, bs, int(causal),
                                     float(scale), _ptr(out), _ptr(lse), _threads(nthreads))
    _check(st, "paged_attention")
    return out, lse


def paged_attention_rows(q, k_cache, v_cache, block_table, ctx_lens, q_lens, causal: bool,
                         scale: float, rows, nthreads=None):
    """Selected rows (seq, query index in chunk, head) -> (out f64 [n, d], lse f64 [n])."""
    qb, kc, vc = to_bits(q), to_bits(k_cache), to_bits(v_cache)
    bt, cl, ql = _i32(block_table), _i32(ctx_lens), _i32(q_lens)
    tq, Hq, d = qb.shape
    nb, Hkv, bs, _ = kc.shape
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    out = np.zeros((len(r), d), dtype=np.float64)
    lse = np.zeros(len(r), dtype=np.float64)
    st = _load().ora_paged_attention_rows(_ptr(qb), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl),
                                          _ptr(ql), len(cl), bt.shape[1], nb, Hq, Hkv, d, bs,
                                          int(causal), float(scale), _ptr(r), len(r), _ptr(out),
                                          _ptr(lse), _threads(nthreads))
    _check(st, "paged_attention_rows")
    return out, lse


# ---------------------------------------------------------------- merge ---
def lse_merge(O_parts, lse_parts):
    """Merge normalised partial outputs over disjoint key sets -> (O [d], lse)."""
    Op = np.ascontiguousarray(O_parts, dtype=np.float64)
    lp = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, d = Op.shape
    O = np.zeros(d, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    _load().ora_lse_merge(n, d, _ptr(Op), _ptr(lp), _ptr(O), _ptr(lse))
    return O, float(lse[0])


def mask_tile_classes(mask, bm: int = 128, bn: int = 128, intervals: bool = False):
    """uint8 [ceil(Tq/bm), ceil(Tk/bn)]: 0 all -inf, 1 all zero, 3 every row's
    zeros one contiguous run among -inf, 2 otherwise.  With intervals=True also
    returns uint8 [ceil(Tq/bm), ceil(Tk/bn), bm, 2], each row's run [lo, hi) in
    the class-3 tiles (zeros elsewhere)."""
    m = _f32(mask)
    Tq, Tk = m.shape
    out = np.zeros(((Tq + bm - 1) // bm, (Tk + bn - 1) // bn), dtype=np.uint8)
    iv = np.zeros(out.shape + (bm, 2), dtype=np.uint8)
    _load().ora_mask_tile_classes(_ptr(m), Tq, Tk, bm, bn, _ptr(out), _ptr(iv))
    return (out, iv) if intervals else out
