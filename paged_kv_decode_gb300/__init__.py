"""paged_kv_decode_gb300 -- paged-KV attention for a GB300 (sm_103a), Python binding.

Thin marshalling over the C ABI of libpkv (include/pkv.h): every step of the
path (KV append, decode attention, chunked-prefill attention) runs in the
library's CUDA kernels. torch tensors supply device memory and the current
CUDA stream. There is no CPU fallback: without the compiled library every call
raises.

Layout (see include/pkv.h): pools bf16 [num_pages, Hkv, 16, D]; q / out bf16
[rows, Hq, D]; block tables int32 [rows, max_pages]; lengths int32. The Qwen3
decoder's 16/8/128 runs the tuned kernels; append, decode, the fused append +
decode call and chunked prefill also take head_dim 64 or 128 with 1 to 8 query
heads per KV head.
"""
from __future__ import annotations

import ctypes
from typing import Optional

from . import _lib

PKV_OK = 0
PKV_STATUS_BYTES = 256
ERRORS = {
    -1: "PKV_ERR_NULL_ARG",
    -2: "PKV_ERR_BAD_SHAPE",
    -3: "PKV_ERR_UNSUPPORTED",
    -4: "PKV_ERR_WORKSPACE_TOO_SMALL",
    -5: "PKV_ERR_CUDA",
    -6: "PKV_ERR_DEVICE_TIMEOUT",
    -7: "PKV_ERR_OUT_OF_BOUNDS",
    -8: "PKV_ERR_MISALIGNED",
}
ERR_CODES = {name: code for code, name in ERRORS.items()}

__all__ = [
    "PkvError", "desc", "Workspace", "append", "decode_attn", "prefill_chunk_attn",
    "decode_workspace_bytes", "prefill_workspace_bytes", "workspace_init", "read_status", "status_string",
    "decode_attn_noalloc", "decode_append_attn", "mixed_step_attn", "mixed_workspace_bytes", "rope_cos_sin",
]


class PkvError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {ERRORS.get(code, code)} ({status_string(code)})")


def status_string(code: int) -> str:
    return _lib.load().pkv_status_string(int(code)).decode()


def _check(code: int, what: str):
    if code != PKV_OK:
        raise PkvError(code, what)


def desc(num_pages: int, num_q_heads: int = 16, num_kv_heads: int = 8, head_dim: int = 128, page_size: int = 16):
    return _lib.CacheDesc(num_q_heads, num_kv_heads, head_dim, page_size, int(num_pages))


def _desc_of(k_pages, num_q_heads: Optional[int] = None) -> "_lib.CacheDesc":
    """Descriptor of a pool [num_pages, num_kv_heads, page_size, head_dim]; num_q_heads from the
    query tensor (default: as many as KV heads, which is all an append needs)."""
    if k_pages.dim() != 4:
        raise ValueError("pools are [num_pages, num_kv_heads, page_size, head_dim]")
    p, hkv, ps, d = k_pages.shape
    return desc(p, hkv if num_q_heads is None else int(num_q_heads), hkv, d, ps)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, name, device=None):
    import torch

    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


def workspace_init(ws, stream=None):
    _check(_lib.load().pkv_workspace_init(ctypes.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size(),
                                          _stream(stream)), "pkv_workspace_init")


def read_status(ws, stream=None) -> int:
    """Status word of a workspace (synchronises the stream; tests and debugging only)."""
    return int(_lib.load().pkv_read_status(ctypes.c_void_p(ws.data_ptr()), _stream(stream)))


def decode_workspace_bytes(batch: int, max_pages: int, num_pages: int = 1, num_q_heads: int = 16,
                           num_kv_heads: int = 8, head_dim: int = 128) -> int:
    """Workspace bytes of a decode call (default geometry: the Qwen3 decoder, 16/8/128)."""
    d = desc(num_pages, num_q_heads, num_kv_heads, head_dim)
    return int(_lib.load().pkv_decode_workspace_bytes(ctypes.byref(d), int(batch), int(max_pages)))


def prefill_workspace_bytes(num_seqs: int, max_q_len: int, num_pages: int = 1, num_q_heads: int = 16,
                            num_kv_heads: int = 8, head_dim: int = 128) -> int:
    """Workspace bytes of a prefill call (default geometry: the Qwen3 decoder, 16/8/128)."""
    d = desc(num_pages, num_q_heads, num_kv_heads, head_dim)
    return int(_lib.load().pkv_prefill_workspace_bytes(ctypes.byref(d), int(num_seqs), int(max_q_len)))


class Workspace:
    """A zero-initialised device workspace (uint8 tensor) for one stream's calls."""

    def __init__(self, nbytes: int, device=None):
        import torch

        nbytes = max(int(nbytes), PKV_STATUS_BYTES)
        self.tensor = torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
        workspace_init(self.tensor)

    @property
    def nbytes(self) -> int:
        return self.tensor.numel()

    def status(self) -> int:
        return read_status(self.tensor)

    def check(self, what: str = "device status"):
        """Read the status word (synchronises); on a device error, zero the workspace again before
        raising: a call that stopped early may have left split counters or tagged records behind,
        which the next call would take for its own."""
        code = self.status()
        if code != PKV_OK:
            workspace_init(self.tensor)
            raise PkvError(code, what)

    def ensure(self, nbytes: int):
        if nbytes > self.nbytes:
            self.__init__(nbytes, self.tensor.device)
        return self


def append(k_new, v_new, slot_mapping, k_pages, v_pages, workspace: Optional[Workspace] = None, stream=None):
    """Write rows k_new / v_new [n, 8, 128] into the pools at slot_mapping [n] (int32)."""
    import torch

    _need(k_pages, torch.bfloat16, "k_pages")
    dev = k_pages.device
    _need(v_pages, torch.bfloat16, "v_pages", dev)
    _need(k_new, torch.bfloat16, "k_new", dev)
    _need(v_new, torch.bfloat16, "v_new", dev)
    _need(slot_mapping, torch.int32, "slot_mapping", dev)
    n = slot_mapping.numel()
    if k_new.shape[0] != n or v_new.shape != k_new.shape or v_pages.shape != k_pages.shape:
        raise ValueError("shape mismatch")
    d = _desc_of(k_pages)
    ws = workspace.tensor if workspace is not None else None
    rc = _lib.load().pkv_append(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), n, _ptr(k_pages), _ptr(v_pages),
                                ctypes.byref(d), _stream(stream), _ptr(ws), 0 if ws is None else ws.numel())
    _check(rc, "pkv_append")


def decode_attn(q, k_pages, v_pages, block_table, seq_lens, out, scale: float, workspace: Workspace, stream=None):
    """Decode attention: out [B, Hq, D] from q [B, Hq, D] over the paged cache [P, Hkv, 16, D]
    (Hq / Hkv from 1 to 8 and D in 64, 128; 16/8/128 takes the tuned kernel)."""
    import torch

    _need(k_pages, torch.bfloat16, "k_pages")
    dev = k_pages.device
    _need(v_pages, torch.bfloat16, "v_pages", dev)
    _need(q, torch.bfloat16, "q", dev)
    _need(out, torch.bfloat16, "out", dev)
    _need(block_table, torch.int32, "block_table", dev)
    _need(seq_lens, torch.int32, "seq_lens", dev)
    B = q.shape[0]
    if out.shape != q.shape or block_table.dim() != 2 or block_table.shape[0] != B or seq_lens.numel() != B:
        raise ValueError("shape mismatch")
    d = _desc_of(k_pages, q.shape[1])
    ws = workspace.tensor
    rc = _lib.load().pkv_decode_attn(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seq_lens),
                                     _ptr(out), float(scale), _stream(stream), ctypes.byref(d), B,
                                     block_table.shape[1], _ptr(ws), ws.numel())
    _check(rc, "pkv_decode_attn")


EARLY_PREFETCH = 1  # PKV_DECODE_EARLY_PREFETCH


def rope_cos_sin(theta: float, max_pos: int, head_dim: int = 128, device=None, stream=None):
    """cos/sin table for decode_append_rope_attn, built on the device by pkv_rope_table: fp32
    [max_pos, head_dim], row p = cos(p w_i) for i < head_dim/2, then sin(p w_i), w_i = theta ** (-2 i /
    head_dim), angles in double rounded to float once. (RoPE theta 1e6 for the decoder on "Fun-ASR-Nano
    Native Runtime Design", "Decoder And Prompt".)"""
    import torch

    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if dev.type != "cuda":
        raise ValueError("the table is built on a CUDA device (the library has no CPU path)")
    table = torch.empty(int(max_pos), int(head_dim), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        rc = _lib.load().pkv_rope_table(_ptr(table), int(max_pos), int(head_dim), float(theta), _stream(stream))
    _check(rc, "pkv_rope_table")
    return table


def decode_append_rope_attn(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, cos_sin, out, scale: float,
                            workspace: Workspace, stream=None, early_prefetch: bool = False):
    """decode_append_attn with the rotary embedding of the new token: k_new and every q row are
    rotated at position seq_lens[b] - 1 (pairs i, i + head_dim/2; cos_sin from rope_cos_sin) before
    the append and the scores (any geometry decode_append_attn takes)."""
    import torch

    _need(cos_sin, torch.float32, "cos_sin", k_pages.device)
    if cos_sin.dim() != 2 or cos_sin.shape[1] != q.shape[-1]:
        raise ValueError("cos_sin must be [max_pos, head_dim]")
    _decode_append(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, out, scale, workspace, stream,
                   early_prefetch, cos_sin)


def decode_append_attn(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, out, scale: float,
                       workspace: Workspace, stream=None, early_prefetch: bool = False):
    """One decode step of one layer in one launch: write k_new / v_new [B, Hkv, D] at position
    seq_lens[b] - 1 of each request, then decode attention over seq_lens[b] positions (any geometry
    decode_attn takes).

    early_prefetch: the previous kernel on the stream writes neither the pools nor the block
    table nor the lengths, so they may be read while it finishes (PKV_DECODE_EARLY_PREFETCH)."""
    _decode_append(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, out, scale, workspace, stream,
                   early_prefetch, None)


def _decode_append(q, k_new, v_new, k_pages, v_pages, block_table, seq_lens, out, scale, workspace, stream,
                   early_prefetch, cos_sin):
    import torch

    _need(k_pages, torch.bfloat16, "k_pages")
    dev = k_pages.device
    _need(v_pages, torch.bfloat16, "v_pages", dev)
    _need(q, torch.bfloat16, "q", dev)
    _need(k_new, torch.bfloat16, "k_new", dev)
    _need(v_new, torch.bfloat16, "v_new", dev)
    _need(out, torch.bfloat16, "out", dev)
    _need(block_table, torch.int32, "block_table", dev)
    _need(seq_lens, torch.int32, "seq_lens", dev)
    B = q.shape[0]
    if (out.shape != q.shape or block_table.dim() != 2 or block_table.shape[0] != B or seq_lens.numel() != B
            or k_new.shape[0] != B or v_new.shape != k_new.shape):
        raise ValueError("shape mismatch")
    d = _desc_of(k_pages, q.shape[1])
    ws = workspace.tensor
    flags = EARLY_PREFETCH if early_prefetch else 0
    lib = _lib.load()
    if cos_sin is None:
        rc = lib.pkv_decode_append_attn(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pages), _ptr(v_pages),
                                        _ptr(block_table), _ptr(seq_lens), _ptr(out), float(scale), _stream(stream),
                                        ctypes.byref(d), B, block_table.shape[1], _ptr(ws), ws.numel(), flags)
        _check(rc, "pkv_decode_append_attn")
    else:
        rc = lib.pkv_decode_append_rope_attn(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pages), _ptr(v_pages),
                                             _ptr(block_table), _ptr(seq_lens), _ptr(cos_sin), cos_sin.shape[0],
                                             _ptr(out), float(scale), _stream(stream), ctypes.byref(d), B,
                                             block_table.shape[1], _ptr(ws), ws.numel(), flags)
        _check(rc, "pkv_decode_append_rope_attn")


def prefill_chunk_attn(q, k_pages, v_pages, block_table, prefix_lens, cu_q_lens, out, scale: float, max_q_len: int,
                       workspace: Workspace, stream=None):
    """Causal chunk attention: out [total_q, Hq, D] for chunks packed by cu_q_lens (Hq / Hkv from 1 to 8,
    D 64 or 128)."""
    import torch

    _need(k_pages, torch.bfloat16, "k_pages")
    dev = k_pages.device
    _need(v_pages, torch.bfloat16, "v_pages", dev)
    _need(q, torch.bfloat16, "q", dev)
    _need(out, torch.bfloat16, "out", dev)
    _need(block_table, torch.int32, "block_table", dev)
    _need(prefix_lens, torch.int32, "prefix_lens", dev)
    _need(cu_q_lens, torch.int32, "cu_q_lens", dev)
    S = prefix_lens.numel()
    if cu_q_lens.numel() != S + 1 or block_table.shape[0] != S or out.shape != q.shape:
        raise ValueError("shape mismatch")
    d = _desc_of(k_pages, q.shape[1])
    ws = workspace.tensor
    rc = _lib.load().pkv_prefill_chunk_attn(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                            _ptr(prefix_lens), _ptr(cu_q_lens), S, q.shape[0], _ptr(out),
                                            float(scale), _stream(stream), ctypes.byref(d), block_table.shape[1],
                                            int(max_q_len), _ptr(ws), ws.numel())
    _check(rc, "pkv_prefill_chunk_attn")


def mixed_workspace_bytes(num_seqs: int, max_q_len: int, dec_batch: int, dec_max_pages: int,
                          num_pages: int = 1) -> int:
    """Workspace bytes of a mixed-step call (16/8/128)."""
    d = desc(num_pages)
    return int(_lib.load().pkv_mixed_workspace_bytes(ctypes.byref(d), int(num_seqs), int(max_q_len), int(dec_batch),
                                                     int(dec_max_pages)))


def mixed_step_attn(q, k_pages, v_pages, block_table, prefix_lens, cu_q_lens, out, max_q_len: int, dec_q,
                    dec_block_table, dec_seq_lens, dec_out, scale: float, workspace: Workspace, stream=None):
    """One scheduler step of chunked prefill interleaved with decode, in one launch (16/8/128): out as
    prefill_chunk_attn gives it for the chunks (q, block_table, prefix_lens, cu_q_lens; may be empty) and
    dec_out as decode_attn gives it for the decode requests (dec_q, dec_block_table, dec_seq_lens), over
    the same pools. The workspace is sized by mixed_workspace_bytes."""
    import torch

    _need(k_pages, torch.bfloat16, "k_pages")
    dev = k_pages.device
    _need(v_pages, torch.bfloat16, "v_pages", dev)
    _need(dec_q, torch.bfloat16, "dec_q", dev)
    _need(dec_out, torch.bfloat16, "dec_out", dev)
    _need(dec_block_table, torch.int32, "dec_block_table", dev)
    _need(dec_seq_lens, torch.int32, "dec_seq_lens", dev)
    B = dec_q.shape[0]
    if dec_out.shape != dec_q.shape or dec_block_table.dim() != 2 or dec_block_table.shape[0] != B \
            or dec_seq_lens.numel() != B:
        raise ValueError("shape mismatch (decode part)")
    S = 0 if prefix_lens is None else prefix_lens.numel()
    if S:
        _need(q, torch.bfloat16, "q", dev)
        _need(out, torch.bfloat16, "out", dev)
        _need(block_table, torch.int32, "block_table", dev)
        _need(prefix_lens, torch.int32, "prefix_lens", dev)
        _need(cu_q_lens, torch.int32, "cu_q_lens", dev)
        if cu_q_lens.numel() != S + 1 or block_table.shape[0] != S or out.shape != q.shape:
            raise ValueError("shape mismatch (chunk part)")
    d = _desc_of(k_pages, dec_q.shape[1])
    ws = workspace.tensor
    rc = _lib.load().pkv_mixed_step_attn(
        _ptr(q) if S else None, _ptr(k_pages), _ptr(v_pages), _ptr(block_table) if S else None,
        _ptr(prefix_lens) if S else None, _ptr(cu_q_lens) if S else None, S, q.shape[0] if S else 0,
        _ptr(out) if S else None, block_table.shape[1] if S else 1, int(max_q_len) if S else 0, _ptr(dec_q),
        _ptr(dec_block_table), _ptr(dec_seq_lens), _ptr(dec_out), B, dec_block_table.shape[1], float(scale),
        _stream(stream), ctypes.byref(d), _ptr(ws), ws.numel())
    _check(rc, "pkv_mixed_step_attn")


def decode_attn_noalloc(q, k_pages, v_pages, block_table, seq_lens, out, scale: float, stream=None):
    """decode_attn without a workspace, for callers that may not allocate device memory.

    The split-KV scratch is a fixed 2 MiB array inside the library (batch <= 256).
    Calls share that array: run them in order on one stream, never overlapping on
    the GPU. Make the first call on a device before any CUDA-graph capture.
    """
    import torch

    _need(k_pages, torch.bfloat16, "k_pages")
    dev = k_pages.device
    _need(v_pages, torch.bfloat16, "v_pages", dev)
    _need(q, torch.bfloat16, "q", dev)
    _need(out, torch.bfloat16, "out", dev)
    _need(block_table, torch.int32, "block_table", dev)
    _need(seq_lens, torch.int32, "seq_lens", dev)
    B = q.shape[0]
    if out.shape != q.shape or block_table.dim() != 2 or block_table.shape[0] != B or seq_lens.numel() != B:
        raise ValueError("shape mismatch")
    d = _desc_of(k_pages, q.shape[1])
    rc = _lib.load().pkv_decode_attn_noalloc(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                             _ptr(seq_lens), _ptr(out), float(scale), _stream(stream),
                                             ctypes.byref(d), B, block_table.shape[1])
    _check(rc, "pkv_decode_attn_noalloc")
