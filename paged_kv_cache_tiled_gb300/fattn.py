"""ctypes binding of libfattn (include/fattn.h).

Argument marshalling only: every function here checks dtypes/shapes, passes
device pointers, sizes and the current CUDA stream to the C entry point of the
same name, and raises ``FattnError`` on a non-OK status.  All arithmetic runs
in the library's CUDA kernels; there is no CPU or PyTorch fallback, and
importing this module fails loudly when ``libfattn.so`` has not been built.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfattn.so")

(FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT, FA_ERR_BOUNDS, FA_ERR_WORKSPACE,
 FA_ERR_NO_BLOCKS) = range(8)
FA_BF16, FA_F32 = 0, 1

# every symbol declared in include/fattn.h
EXPORTS = [
    "fa_status_string", "fa_prefill", "fa_prefill_masked_workspace_size", "fa_prefill_masked", "fa_stage_bf16",
    "fa_cache_append", "fa_paged_attn_workspace_size", "fa_paged_attn", "fa_get_error", "fa_debug_gather_kv",
    "fa_debug_set_wait_limit", "fa_debug_force_timeout", "fa_last_launch_count", "fa_paged_attn_noalloc",
    "fa_cache_append_rope", "fa_decode_graph_create", "fa_decode_graph_launch", "fa_decode_graph_kernel_count",
    "fa_decode_graph_destroy", "fa_pool_create", "fa_pool_destroy", "fa_pool_add_seq", "fa_pool_fork",
    "fa_pool_append", "fa_pool_release", "fa_pool_tables", "fa_pool_num_free", "fa_pool_refcount", "fa_pool_seq_len",
    "fa_copy_blocks", "fa_cache_append_fp8", "fa_paged_attn_fp8", "fa_prefill_host", "fa_mask_tile_classes",
    "fa_prefill_rows",
]
NOALLOC_SCRATCH_BYTES = 32 << 20  # FA_NOALLOC_SCRATCH_BYTES


class FattnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with paged_kv_cache_tiled_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    Z = ctypes.c_size_t
    sig = {
        "fa_status_string": (ctypes.c_char_p, [I]),
        "fa_prefill": (I, [P, P, P, P, I, I, I, I, I, I, F, P, P]),
        "fa_prefill_host": (I, [P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P]),
        "fa_prefill_rows": (I, [P, P, P, P, I, I, I, I, I, I, F, I, I, I, P]),
        "fa_prefill_masked_workspace_size": (Z, [I]),
        "fa_prefill_masked": (I, [P, P, P, P, P, I, I, I, I, I, I, F, P, P, Z, P]),
        "fa_stage_bf16": (I, [P, P, Z, P]),
        "fa_mask_tile_classes": (I, [P, I, I, P, P, P]),
        "fa_cache_append": (I, [P, P, P, P, P, I, I, I, I, I, P]),
        "fa_paged_attn_workspace_size": (Z, [I, I, I, I, I, I]),
        "fa_paged_attn": (I, [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, I, P, Z, P]),
        "fa_get_error": (I, [P]),
        "fa_debug_gather_kv": (I, [P, P, P, P, I, I, I, I, I, I, P]),
        "fa_debug_set_wait_limit": (None, [ctypes.c_ulonglong]),
        "fa_cache_append_rope": (I, [P, P, P, P, P, I, P, P, P, P, I, I, I, I, I, I, P]),
        "fa_decode_graph_create": (I, [P, P, P, P, I, I, P, P, P, P, P, P, P, I, I, I, I, I, I, I,
                                       ctypes.c_float, I, I, P, ctypes.c_size_t]),
        "fa_decode_graph_launch": (I, [P, P]),
        "fa_decode_graph_kernel_count": (I, [P]),
        "fa_decode_graph_destroy": (None, [P]),
        "fa_pool_create": (I, [P, I, I]),
        "fa_pool_destroy": (None, [P]),
        "fa_pool_add_seq": (I, [P, P]),
        "fa_pool_fork": (I, [P, I, I, P, P, P]),
        "fa_pool_append": (I, [P, I, I, P]),
        "fa_pool_release": (I, [P, I]),
        "fa_pool_tables": (I, [P, P, I, P, P]),
        "fa_pool_num_free": (I, [P]),
        "fa_pool_refcount": (I, [P, I]),
        "fa_pool_seq_len": (I, [P, I]),
        "fa_copy_blocks": (I, [P, P, P, I, I, I, I, P]),
        "fa_cache_append_fp8": (I, [P, P, P, P, P, I, I, I, I, ctypes.c_float, ctypes.c_float, I, P]),
        "fa_paged_attn_fp8": (I, [P, P, P, ctypes.c_float, ctypes.c_float, P, P, P, P, I, I, I, I, I, I, I, I,
                                  ctypes.c_float, I, I, P, ctypes.c_size_t, P]),
        "fa_debug_force_timeout": (None, [I]),
        "fa_paged_attn_noalloc": (I, [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, I, P]),
        "fa_last_launch_count": (I, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def library() -> ctypes.CDLL:
    return _lib


def status_string(status: int) -> str:
    return _lib.fa_status_string(int(status)).decode()


fa_status_string = status_string


def _check(st: int, where: str):
    if st != FA_OK:
        raise FattnError(st, where)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype, ndim: int | None = None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


# ------------------------------------------------------------------ prefill
def fa_prefill(q, k, v, causal: bool = True, scale: float | None = None, out=None, lse=None, stream=None):
    """softmax(scale * Q K^T [+ causal mask]) V for q [B,T,Hq,d], k/v [B,T,Hkv,d] (bf16)."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _need(t, n, torch.bfloat16, 4)
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 4)
    if lse is not None:
        _need(lse, "lse", torch.float32)
    _check(_lib.fa_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, T, Hq, Hkv, d, int(causal), float(scale),
                           _ptr(lse), _stream(stream)), "fa_prefill")
    return out


def fa_prefill_rows(q, k, v, q0: int, Tq: int, Tk: int, causal: bool = True, scale: float | None = None, out=None,
                    stream=None):
    """Query rows [q0, q0+Tq) of every sequence against keys [0, Tk); q/k/v/out
    hold whole sequences [B, T, H, d] and only those rows of `out` are written."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _need(t, n, torch.bfloat16, 4)
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, 4)
    _check(_lib.fa_prefill_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, T, Hq, Hkv, d, int(causal), float(scale),
                                int(q0), int(Tq), int(Tk), _stream(stream)), "fa_prefill_rows")
    return out


def fa_prefill_host(q_host, k_host, v_host, out_host, q, k, v, out, causal: bool = True,
                    scale: float | None = None, stream=None):
    """fa_prefill from and to host memory: the host tensors (bf16, contiguous,
    ideally pinned) are copied into the caller's device buffers q/k/v and the
    result back into out_host, one sequence at a time, with the copies
    overlapping the kernels.  Ordered on `stream`; the host is not synchronised."""
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _need(t, n, torch.bfloat16, 4)
    for n, t, dev in (("q_host", q_host, q), ("k_host", k_host, k), ("v_host", v_host, v), ("out_host", out_host, out)):
        if not isinstance(t, torch.Tensor) or t.is_cuda:
            raise ValueError(f"{n} must be a host tensor")
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.shape != dev.shape:
            raise ValueError(f"{n} must be a contiguous bf16 tensor shaped like its device buffer")
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _check(_lib.fa_prefill_host(q_host.data_ptr(), k_host.data_ptr(), v_host.data_ptr(), out_host.data_ptr(),
                                _ptr(q), _ptr(k), _ptr(v), _ptr(out), B, T, Hq, Hkv, d, int(causal), float(scale),
                                _stream(stream)), "fa_prefill_host")
    return out_host


def fa_prefill_masked_workspace_size(T: int) -> int:
    return int(_lib.fa_prefill_masked_workspace_size(int(T)))


def fa_prefill_masked(q, k, v, mask, causal: bool = False, scale: float | None = None, out=None, lse=None, ws=None,
                      stream=None):
    """softmax(scale * Q K^T + M [+ causal]) V with an additive fp32 mask M [T, T]."""
    for n, t in (("q", q), ("k", k), ("v", v)):
        _need(t, n, torch.bfloat16, 4)
    _need(mask, "mask", torch.float32, 2)
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    nbytes = fa_prefill_masked_workspace_size(T)
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check(_lib.fa_prefill_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(mask), _ptr(out), B, T, Hq, Hkv, d, int(causal),
                                  float(scale), _ptr(lse), _ptr(ws), ws.numel() * ws.element_size(),
                                  _stream(stream)), "fa_prefill_masked")
    return out


def fa_mask_tile_classes(mask, out=None, intervals=None, stream=None):
    """uint8 [ceil(Tq/128), ceil(Tk/128)] classes of an fp32 mask [Tq, Tk]: 0 all -inf, 1 all zero,
    3 zeros forming one run per row among -inf, 2 otherwise.  `intervals` (optional, uint8
    [ceil(Tq/128), ceil(Tk/128), 128, 2]) receives each row's run [lo, hi) in class-3 tiles."""
    _need(mask, "mask", torch.float32, 2)
    Tq, Tk = mask.shape
    shape = ((Tq + 127) // 128, (Tk + 127) // 128)
    if out is None:
        out = torch.empty(shape, dtype=torch.uint8, device=mask.device)
    _need(out, "out", torch.uint8, 2)
    if tuple(out.shape) != shape:
        raise ValueError(f"out must have shape {shape}")
    if intervals is not None:
        _need(intervals, "intervals", torch.uint8, 4)
        if tuple(intervals.shape) != shape + (128, 2):
            raise ValueError(f"intervals must have shape {shape + (128, 2)}")
    _check(_lib.fa_mask_tile_classes(_ptr(mask), Tq, Tk, _ptr(out), _ptr(intervals) if intervals is not None else None,
                                     _stream(stream)), "fa_mask_tile_classes")
    return out


def fa_stage_bf16(src, dst=None, stream=None):
    """fp32 -> bf16 (round to nearest even)."""
    _need(src, "src", torch.float32)
    if dst is None:
        dst = torch.empty(src.shape, dtype=torch.bfloat16, device=src.device)
    _need(dst, "dst", torch.bfloat16)
    _check(_lib.fa_stage_bf16(_ptr(src), _ptr(dst), src.numel(), _stream(stream)), "fa_stage_bf16")
    return dst


# -------------------------------------------------------------------- paged
def fa_cache_append(k, v, k_cache, v_cache, slot_mapping, stream=None):
    """Writes k/v [N, Hkv, d] (bf16 or fp32) into the caches [num_blocks, Hkv, 16, d] at slot_mapping[N]."""
    if k.dtype not in (torch.bfloat16, torch.float32) or v.dtype != k.dtype:
        raise ValueError("k, v must both be bf16 or both fp32")
    _need(k, "k", k.dtype, 3)
    _need(v, "v", k.dtype, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    N, Hkv, d = k.shape
    dt = FA_F32 if k.dtype == torch.float32 else FA_BF16
    _check(_lib.fa_cache_append(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), N, Hkv, d,
                                k_cache.shape[0], dt, _stream(stream)), "fa_cache_append")


def fa_cache_append_rope(q, k, v, positions, cos_sin, k_cache, v_cache, slot_mapping, q_out=None, stream=None):
    """Rotary embedding of q [N,Hq,d] and k [N,Hkv,d] at table rows positions[N]
    (cos_sin fp32 [max_pos, d]: cosines then sines), fused with the cache
    append of the rotated k and of v; returns the rotated queries (bf16)."""
    if q.dtype not in (torch.bfloat16, torch.float32) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must all be bf16 or all fp32")
    _need(q, "q", q.dtype, 3)
    _need(k, "k", q.dtype, 3)
    _need(v, "v", q.dtype, 3)
    _need(positions, "positions", torch.int32, 1)
    _need(cos_sin, "cos_sin", torch.float32, 2)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    N, Hq, d = q.shape
    Hkv = k.shape[1]
    if q_out is None:
        q_out = torch.empty(N, Hq, d, dtype=torch.bfloat16, device=q.device)
    _need(q_out, "q_out", torch.bfloat16, 3)
    dt = FA_F32 if q.dtype == torch.float32 else FA_BF16
    _check(_lib.fa_cache_append_rope(_ptr(q), _ptr(k), _ptr(v), _ptr(positions), _ptr(cos_sin), cos_sin.shape[0],
                                     _ptr(q_out), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), N, Hq, Hkv, d,
                                     k_cache.shape[0], dt, _stream(stream)), "fa_cache_append_rope")
    return q_out


class BlockPool:
    """fa_pool_*: host-side block pool with reference counts and prefix
    sharing.  Methods mirror the C functions; arrays are numpy."""

    def __init__(self, num_blocks: int, max_blocks_per_seq: int):
        h = ctypes.c_void_p()
        _check(_lib.fa_pool_create(ctypes.byref(h), num_blocks, max_blocks_per_seq), "fa_pool_create")
        self._h, self.num_blocks, self.max_blocks_per_seq = h, num_blocks, max_blocks_per_seq

    def add_seq(self) -> int:
        s = ctypes.c_int()
        _check(_lib.fa_pool_add_seq(self._h, ctypes.byref(s)), "fa_pool_add_seq")
        return s.value

    def fork(self, parent: int, prefix_len: int):
        """Returns (child, (copy_src, copy_dst)) with (-1, -1) when no copy is needed."""
        c, a, b = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        _check(_lib.fa_pool_fork(self._h, parent, prefix_len, ctypes.byref(c), ctypes.byref(a), ctypes.byref(b)),
               "fa_pool_fork")
        return c.value, (a.value, b.value)

    def append(self, seq: int, n: int) -> np.ndarray:
        slots = np.zeros(max(n, 1), np.int32)
        _check(_lib.fa_pool_append(self._h, seq, n, slots.ctypes.data_as(ctypes.c_void_p)), "fa_pool_append")
        return slots[:n]

    def release(self, seq: int):
        _check(_lib.fa_pool_release(self._h, seq), "fa_pool_release")

    def tables(self, seqs):
        seqs = np.ascontiguousarray(seqs, dtype=np.int32)
        n = len(seqs)
        table = np.zeros((max(n, 1), self.max_blocks_per_seq), np.int32)
        lens = np.zeros(max(n, 1), np.int32)
        _check(_lib.fa_pool_tables(self._h, seqs.ctypes.data_as(ctypes.c_void_p), n,
                                   table.ctypes.data_as(ctypes.c_void_p), lens.ctypes.data_as(ctypes.c_void_p)),
               "fa_pool_tables")
        return table[:n], lens[:n]

    def num_free(self) -> int:
        return int(_lib.fa_pool_num_free(self._h))

    def refcount(self, block: int) -> int:
        return int(_lib.fa_pool_refcount(self._h, block))

    def seq_len(self, seq: int) -> int:
        return int(_lib.fa_pool_seq_len(self._h, seq))

    def close(self):
        if getattr(self, "_h", None):
            _lib.fa_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fa_copy_blocks(k_cache, v_cache, pairs, stream=None):
    """Copies cache block pairs[i, 0] onto pairs[i, 1] (pairs: int32 [n, 2] on the device)."""
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(pairs, "pairs", torch.int32, 2)
    num_blocks, Hkv, _, d = k_cache.shape
    _check(_lib.fa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pairs), pairs.shape[0], Hkv, d, num_blocks,
                               _stream(stream)), "fa_copy_blocks")


class DecodeGraph:
    """fa_decode_graph_*: the append of k_new/v_new (if given) plus paged
    attention, captured once with these tensors and replayed with one
    submission.  Keep every tensor alive and rewrite contents only."""

    def __init__(self, q, k_cache, v_cache, block_table, ctx_lens, q_lens, out, ws, *, k_new=None, v_new=None,
                 slot_mapping=None, causal: bool = True, scale: float | None = None, max_q_len: int | None = None):
        total_q, Hq, d = q.shape
        num_blocks, Hkv, _, _ = k_cache.shape
        num_seqs, mbps = block_table.shape
        n_new, dt = 0, FA_BF16
        if k_new is not None:
            n_new = k_new.shape[0]
            dt = FA_F32 if k_new.dtype == torch.float32 else FA_BF16
        self._keep = (q, k_cache, v_cache, block_table, ctx_lens, q_lens, out, ws, k_new, v_new, slot_mapping)
        h = ctypes.c_void_p()
        _check(_lib.fa_decode_graph_create(
            ctypes.byref(h), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), n_new, dt, _ptr(q), _ptr(k_cache),
            _ptr(v_cache), _ptr(block_table), _ptr(ctx_lens), _ptr(q_lens), _ptr(out), num_seqs, mbps, num_blocks,
            Hq, Hkv, d, int(causal), float(scale if scale is not None else 1.0 / math.sqrt(d)), total_q,
            int(max_q_len if max_q_len is not None else total_q), _ptr(ws), ws.numel() * ws.element_size()),
            "fa_decode_graph_create")
        self._h = h

    @property
    def kernel_count(self) -> int:
        return int(_lib.fa_decode_graph_kernel_count(self._h))

    def replay(self, stream=None):
        _check(_lib.fa_decode_graph_launch(self._h, _stream(stream)), "fa_decode_graph_launch")

    def close(self):
        if getattr(self, "_h", None):
            _lib.fa_decode_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fa_cache_append_fp8(k, v, k_cache, v_cache, slot_mapping, k_scale: float, v_scale: float, stream=None):
    """E4M3 codes of k/v [N, Hkv, d] (bf16 or fp32) / scale into k_cache uint8 [nb, Hkv, 16, d] and
    v_cache uint8 [nb, Hkv, d, 16] at slot_mapping[N]."""
    if k.dtype not in (torch.bfloat16, torch.float32) or v.dtype != k.dtype:
        raise ValueError("k, v must both be bf16 or both fp32")
    _need(k, "k", k.dtype, 3)
    _need(v, "v", k.dtype, 3)
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(v_cache, "v_cache", torch.uint8, 4)
    _need(slot_mapping, "slot_mapping", torch.int32, 1)
    N, Hkv, d = k.shape
    dt = FA_F32 if k.dtype == torch.float32 else FA_BF16
    _check(_lib.fa_cache_append_fp8(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping), N, Hkv, d,
                                    k_cache.shape[0], float(k_scale), float(v_scale), dt, _stream(stream)),
           "fa_cache_append_fp8")


def fa_paged_attn_fp8(q, k_cache, v_cache, k_scale: float, v_scale: float, block_table, ctx_lens, q_lens,
                      causal: bool = True, scale: float | None = None, out=None, max_q_len: int | None = None,
                      ws=None, stream=None):
    """Decode rows of q [total_q, Hq, d] against the 8-bit caches."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(v_cache, "v_cache", torch.uint8, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(ctx_lens, "ctx_lens", torch.int32, 1)
    _need(q_lens, "q_lens", torch.int32, 1)
    total_q, Hq, d = q.shape
    num_blocks, Hkv = k_cache.shape[0], k_cache.shape[1]
    num_seqs, mbps = block_table.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    max_q_len = total_q if max_q_len is None else max_q_len
    nbytes = fa_paged_attn_workspace_size(num_seqs, mbps, Hq, Hkv, d, total_q)
    if ws is None:
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    _check(_lib.fa_paged_attn_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), float(k_scale), float(v_scale),
                                  _ptr(block_table), _ptr(ctx_lens), _ptr(q_lens), _ptr(out), num_seqs, mbps,
                                  num_blocks, Hq, Hkv, d, 16, int(causal), float(scale), total_q, int(max_q_len),
                                  _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "fa_paged_attn_fp8")
    return out


def fa_paged_attn_workspace_size(num_seqs, max_blocks_per_seq, Hq, Hkv, d, total_q) -> int:
    return int(_lib.fa_paged_attn_workspace_size(num_seqs, max_blocks_per_seq, Hq, Hkv, d, total_q))


def fa_paged_attn(q, k_cache, v_cache, block_table, ctx_lens, q_lens, causal: bool = True,
                  scale: float | None = None, out=None, max_q_len: int | None = None, ws=None, stream=None):
    """Attention of packed queries q [total_q, Hq, d] against the paged cache."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(ctx_lens, "ctx_lens", torch.int32, 1)
    _need(q_lens, "q_lens", torch.int32, 1)
    total_q, Hq, d = q.shape
    num_blocks, Hkv, bs, _ = k_cache.shape
    num_seqs, mbps = block_table.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if max_q_len is None:
        max_q_len = total_q
    nbytes = fa_paged_attn_workspace_size(num_seqs, mbps, Hq, Hkv, d, total_q)
    if ws is None:
        ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    _check(_lib.fa_paged_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(ctx_lens),
                              _ptr(q_lens), _ptr(out), num_seqs, mbps, num_blocks, Hq, Hkv, d, bs, int(causal),
                              float(scale), total_q, int(max_q_len), _ptr(ws), ws.numel() * ws.element_size(),
                              _stream(stream)), "fa_paged_attn")
    return out


def fa_paged_attn_noalloc(q, k_cache, v_cache, block_table, ctx_lens, q_lens, causal: bool = True,
                          scale: float | None = None, out=None, max_q_len: int | None = None, stream=None):
    """fa_paged_attn without a workspace, for callers that cannot allocate device
    scratch: the library's fixed 32 MiB per-device array is used instead.  Calls
    must not overlap on the GPU (they share that array)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(ctx_lens, "ctx_lens", torch.int32, 1)
    _need(q_lens, "q_lens", torch.int32, 1)
    total_q, Hq, d = q.shape
    num_blocks, Hkv, bs, _ = k_cache.shape
    num_seqs, mbps = block_table.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if max_q_len is None:
        max_q_len = total_q
    _check(_lib.fa_paged_attn_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(ctx_lens),
                                      _ptr(q_lens), _ptr(out), num_seqs, mbps, num_blocks, Hq, Hkv, d, bs,
                                      int(causal), float(scale), total_q, int(max_q_len), _stream(stream)),
           "fa_paged_attn_noalloc")
    return out


# --------------------------------------------------------------- utilities
def fa_get_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error status."""
    return int(_lib.fa_get_error(_stream(stream)))


def fa_debug_gather_kv(cache, block_table, ctx_lens, max_ctx: int, out=None, stream=None):
    _need(cache, "cache", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(ctx_lens, "ctx_lens", torch.int32, 1)
    num_blocks, Hkv, _, d = cache.shape
    num_seqs, mbps = block_table.shape
    if out is None:
        out = torch.zeros(num_seqs, max_ctx, Hkv, d, dtype=torch.bfloat16, device=cache.device)
    _check(_lib.fa_debug_gather_kv(_ptr(cache), _ptr(block_table), _ptr(ctx_lens), _ptr(out), num_seqs, mbps,
                                   num_blocks, Hkv, d, max_ctx, _stream(stream)), "fa_debug_gather_kv")
    return out


def fa_debug_set_wait_limit(nanoseconds: int):
    _lib.fa_debug_set_wait_limit(int(nanoseconds))


def fa_debug_force_timeout(enable: bool):
    _lib.fa_debug_force_timeout(int(bool(enable)))


def fa_last_launch_count() -> int:
    return int(_lib.fa_last_launch_count())
