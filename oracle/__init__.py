"""fp64 CPU oracle for paged-KV attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The GPU library never calls it and shares
no code with it; the product path has no CPU fallback.

The arithmetic lives in ``pkv_oracle.c`` (plain C, double precision, loops in
the order of the definition). This module only compiles it with gcc when the
shared object is missing, and marshals numpy / torch CPU arrays into it.

Functions:
  append(...)   -- slot scatter of new K/V rows into the page pools
  decode(...)   -- one query row per request over its paged context (bf16 or float64 queries)
  rope_cache / rope_f64 / rope_bf16 -- rotary position embedding (rotate-half, theta 1e6 on the
                   pages), the step before decode attention for the new token's q and k rows
  prefill(...)  -- causal chunk attention, bottom-right aligned (row i of a
                   chunk after P cached tokens sees keys 0 .. P + i)

Passages followed: "FunASR vLLM Inference Engine Guide" section 2 (PagedAttention,
paged KV cache); "Fun-ASR-Nano Native Runtime Design", "Decoder And Prompt"
(16 query / 8 KV heads); "Optimizing ASR for 90-minute multi-speaker audio",
"Chunked prefill for long audio" (4096-token chunks). Pin status of each
function is recorded in its docstring.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_pkv_oracle.so")
_lock = threading.Lock()
_lib = None


class _Geom(ctypes.Structure):
    _fields_ = [
        ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int64),
    ]


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c into _pkv_oracle.so with gcc (-O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            vp, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
            gp = ctypes.POINTER(_Geom)
            lib.pkvo_append.argtypes = [gp, vp, vp, vp, i64, vp, vp]
            lib.pkvo_decode.argtypes = [gp, vp, vp, vp, vp, vp, i64, i64, dbl, vp, i32]
            lib.pkvo_prefill.argtypes = [gp, vp, vp, vp, vp, i64, vp, vp, i64, vp, i64, dbl, vp, i32]
            lib.pkvo_decode_q64.argtypes = [gp, vp, vp, vp, vp, vp, i64, i64, dbl, vp, i32]
            lib.pkvo_rope_cache.argtypes = [dbl, i32, i64, vp]
            lib.pkvo_rope_f64.argtypes = [vp, i64, i32, i32, vp, vp, i64, vp]
            lib.pkvo_rope_bf16.argtypes = [vp, i64, i32, i32, vp, vp, i64, vp]
            for f in (lib.pkvo_append, lib.pkvo_decode, lib.pkvo_prefill, lib.pkvo_decode_q64, lib.pkvo_rope_cache,
                      lib.pkvo_rope_f64, lib.pkvo_rope_bf16):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _bits(t) -> np.ndarray:
    """bf16 tensor (torch, CPU) or uint16 array -> contiguous uint16 numpy view of its bits."""
    if isinstance(t, np.ndarray):
        a = t
        if a.dtype != np.uint16:
            raise TypeError("expected the uint16 bit pattern of bf16 values")
    else:
        import torch

        if t.dtype != torch.bfloat16:
            raise TypeError(f"expected bfloat16, got {t.dtype}")
        a = t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return np.ascontiguousarray(a)


def _i32(a) -> np.ndarray:
    if isinstance(a, (list, tuple)):
        a = np.asarray(a)
    elif not isinstance(a, np.ndarray):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _geom(n_q_heads, n_kv_heads, head_dim, page_size, num_pages) -> _Geom:
    return _Geom(n_q_heads, n_kv_heads, head_dim, page_size, num_pages)


def _threads(n):
    if n is None:
        try:
            n = len(os.sched_getaffinity(0))
        except AttributeError:  # pragma: no cover
            n = os.cpu_count() or 1
    return max(1, int(n))


_ERR = {-1: "bad argument", -2: "index out of range (page id or length)", -3: "out of memory"}


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: {_ERR.get(rc, rc)}")


def append(k_new, v_new, slot_mapping, k_pages, v_pages):
    """Scatter new K/V rows into copies of the pools; returns (k_pages, v_pages) as uint16 bits.

    k_new, v_new: [n_tokens, n_kv_heads, head_dim] bf16.
    slot_mapping: [n_tokens] int; slot s -> page s // page_size, slot s % page_size; s < 0 skipped.
    k_pages, v_pages: [num_pages, n_kv_heads, page_size, head_dim] bf16.
    Pinned by tests/test_oracle.py (read-back through the block table, untouched slots, skips).
    """
    kp = _bits(k_pages).copy()
    vp = _bits(v_pages).copy()
    kn, vn = _bits(k_new), _bits(v_new)
    sm = _i32(slot_mapping)
    num_pages, n_kv, ps, d = kp.shape
    g = _geom(n_kv, n_kv, d, ps, num_pages)
    rc = _load().pkvo_append(ctypes.byref(g), _ptr(kn), _ptr(vn), _ptr(sm), int(sm.shape[0]), _ptr(kp), _ptr(vp))
    _check(rc, "append")
    return kp, vp


def decode(q, k_pages, v_pages, block_table, seq_lens, scale, n_threads=None) -> np.ndarray:
    """Decode attention in fp64: out[b, h] = softmax_j(scale * <q[b,h], k_j>) . v_j over j < seq_lens[b].

    q: [batch, n_q_heads, head_dim] bf16, or float64 (e.g. rope_f64's rotated rows);
    pools [num_pages, n_kv_heads, page_size, head_dim] bf16;
    block_table: [batch, max_pages] int32; seq_lens: [batch] int32. Returns float64 [batch, n_q_heads, head_dim].
    Pinned by tests/test_oracle.py (dense brute force through a different layout, torch SDPA,
    closed forms, head-map and page-map invariants).
    """
    q64 = isinstance(q, np.ndarray) and q.dtype == np.float64
    qb = np.ascontiguousarray(q) if q64 else _bits(q)
    kp, vp = _bits(k_pages), _bits(v_pages)
    bt, sl = _i32(block_table), _i32(seq_lens)
    batch, hq, d = qb.shape
    num_pages, n_kv, ps, d2 = kp.shape
    if d2 != d or vp.shape != kp.shape or bt.shape[0] != batch or sl.shape[0] != batch:
        raise ValueError("shape mismatch")
    out = np.zeros((batch, hq, d), dtype=np.float64)
    g = _geom(hq, n_kv, d, ps, num_pages)
    rc = (_load().pkvo_decode_q64 if q64 else _load().pkvo_decode)(
        ctypes.byref(g), _ptr(qb), _ptr(kp), _ptr(vp), _ptr(bt), _ptr(sl), batch, int(bt.shape[1]),
        float(scale), _ptr(out), _threads(n_threads),
    )
    _check(rc, "decode")
    return out


def prefill(q, k_pages, v_pages, block_table, prefix_lens, cu_q_lens, scale, rows=None, n_threads=None) -> np.ndarray:
    """Chunked-prefill attention in fp64 (causal, bottom-right aligned).

    q: [total_q, n_q_heads, head_dim] bf16, chunks packed by cu_q_lens [num_seqs + 1].
    Row i of request n attends keys 0 .. prefix_lens[n] + i of that request's pages.
    rows: optional iterable of global query rows to evaluate (default: all).
    Returns float64 [n_rows, n_q_heads, head_dim].
    Pinned by tests/test_oracle.py (torch SDPA with an explicit bottom-right mask,
    causality, equality with decode over the visible prefix).
    """
    qb = _bits(q)
    kp, vp = _bits(k_pages), _bits(v_pages)
    bt, pl, cu = _i32(block_table), _i32(prefix_lens), _i32(cu_q_lens)
    total_q, hq, d = qb.shape
    num_pages, n_kv, ps, _ = kp.shape
    num_seqs = int(pl.shape[0])
    if cu.shape[0] != num_seqs + 1 or int(cu[-1]) != total_q:
        raise ValueError("cu_q_lens must have num_seqs + 1 entries ending at total_q")
    if rows is None:
        r = None
        n_rows = total_q
    else:
        r = np.ascontiguousarray(np.asarray(list(rows) if not isinstance(rows, np.ndarray) else rows, dtype=np.int64))
        n_rows = int(r.shape[0])
    out = np.zeros((n_rows, hq, d), dtype=np.float64)
    g = _geom(hq, n_kv, d, ps, num_pages)
    rc = _load().pkvo_prefill(
        ctypes.byref(g), _ptr(qb), _ptr(kp), _ptr(vp), _ptr(bt), int(bt.shape[1]), _ptr(pl), _ptr(cu),
        num_seqs, None if r is None else _ptr(r), n_rows, float(scale), _ptr(out), _threads(n_threads),
    )
    _check(rc, "prefill")
    return out


def rope_cache(theta: float, head_dim: int, max_pos: int) -> np.ndarray:
    """cos/sin table [max_pos, head_dim] float32 of the rotate-half rotary embedding: row p holds
    cos(p w_i) for i < head_dim/2, then sin(p w_i), w_i = theta ** (-2 i / head_dim), evaluated in
    double and rounded to float once. ("Fun-ASR-Nano Native Runtime Design", "Decoder And Prompt":
    RoPE theta 1e6.) Pinned by tests/test_oracle.py (angle addition, theta from the smallest
    frequency, row 0)."""
    out = np.zeros((int(max_pos), int(head_dim)), dtype=np.float32)
    _check(_load().pkvo_rope_cache(float(theta), int(head_dim), int(max_pos), _ptr(out)), "rope_cache")
    return out


def _rope_args(x, positions, cache):
    xb = _bits(x)
    if xb.ndim != 3:
        raise ValueError("x must be [rows, heads, head_dim]")
    pos = _i32(positions)
    cs = np.ascontiguousarray(cache, dtype=np.float32)
    if pos.shape[0] != xb.shape[0] or cs.ndim != 2 or cs.shape[1] != xb.shape[2]:
        raise ValueError("shape mismatch")
    return xb, pos, cs


def rope_f64(x, positions, cache) -> np.ndarray:
    """Rotate rows x [rows, heads, head_dim] (bf16) at positions [rows] (negative: unrotated) in
    double: y1 = x1 c - x2 s, y2 = x2 c + x1 s over pairs (i, i + head_dim/2). Returns float64.
    Pinned by tests/test_oracle.py (unit vectors, position 0, pair norms, relative positions)."""
    xb, pos, cs = _rope_args(x, positions, cache)
    out = np.zeros(xb.shape, dtype=np.float64)
    rc = _load().pkvo_rope_f64(_ptr(xb), xb.shape[0], xb.shape[1], xb.shape[2], _ptr(pos), _ptr(cs),
                               cs.shape[0], _ptr(out))
    _check(rc, "rope_f64")
    return out


def rope_bf16(x, positions, cache) -> np.ndarray:
    """The same rotation evaluated in float (products rounded, then one fused multiply-add) and
    rounded to bf16 ties-to-even -- the form in which a rotated key row is stored. Returns uint16
    bits. Pinned by tests/test_oracle.py (within one bf16 step of rope_f64; exact at position 0)."""
    xb, pos, cs = _rope_args(x, positions, cache)
    out = np.zeros(xb.shape, dtype=np.uint16)
    rc = _load().pkvo_rope_bf16(_ptr(xb), xb.shape[0], xb.shape[1], xb.shape[2], _ptr(pos), _ptr(cs),
                                cs.shape[0], _ptr(out))
    _check(rc, "rope_bf16")
    return out
