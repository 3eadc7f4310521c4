"""Seeded synthetic inputs for paged-KV attention, shared by tests and the benchmark.

This module draws random numbers and builds index structures (page placement,
block tables, slot indices). It holds none of the attention arithmetic, and it
imports neither the GPU library nor the oracle.

Recipe (the same for every caller):
  * request lengths and page placement: ``numpy.random.default_rng(seed)``;
  * values: fp32 N(0, 1) from a seeded ``torch.Generator`` on the requested
    device, rounded to bf16 (round-to-nearest-even);
  * pool layout ``[layers][num_pages][n_kv_heads][page_size][head_dim]``; logical
    position j of a request is page ``block_table[b][j // page_size]``, slot
    ``j % page_size``; slot index ``s`` names page ``s // page_size``, slot
    ``s % page_size``;
  * physical pages are a random permutation of the pool (``permute=True``);
  * ``poison=True`` fills every slot that no request may read (the tail of a
    request's last page, the pending slots that this step appends, a spare
    "poison" page that unused block-table entries point at) with bf16 NaN.

Workload shapes follow the source pages: Qwen3-0.6B-class decoder with 28 layers
and 16 query / 8 KV heads ("Fun-ASR-Nano Native Runtime Design", "Decoder And
Prompt"); 4096-token prefill chunks ("Optimizing ASR for 90-minute multi-speaker
audio", "Chunked prefill for long audio"); ~12 s clips and ~38 min meetings at
up to 16 concurrent requests (same page, "Benchmark results"); CFG pairs of a
conditional request and a null-prompt companion that mirrors its generated
tokens ("An Efficient vLLM-Based Inference Pipeline for Unified Audio
Understanding and Generation", "Method"). head_dim 128 and page size 16 are
readings: no page states them.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

N_Q_HEADS = 16
N_KV_HEADS = 8
HEAD_DIM = 128
PAGE_SIZE = 16
N_LAYERS = 28
PREFILL_CHUNK = 4096
BF16_NAN_BITS = 0x7FC0


@dataclass(frozen=True)
class Geometry:
    n_q_heads: int = N_Q_HEADS
    n_kv_heads: int = N_KV_HEADS
    head_dim: int = HEAD_DIM
    page_size: int = PAGE_SIZE

    @property
    def scale(self) -> float:
        return float(self.head_dim) ** -0.5


QWEN3 = Geometry()


# ----------------------------------------------------------------------------
# request lengths of the five workloads
# ----------------------------------------------------------------------------

def config_seq_lens(config: int, seed: Optional[int] = None, context: int = 40000) -> np.ndarray:
    """Visible tokens per request (after this step's append) for a workload.

    1: tiny, batch 2, {37, 200}
    2: Qwen3-0.6B decode at batch 16, U{300..3000} (short clips plus prompt)
    3: long-audio decode, batch 1, ``context`` tokens (40,000; sweep 4096/16384/65536)
    5: CFG pairs, batch 32 interleaved (conditional, companion): g ~ U{16..512},
       conditional ~ U{1000..8000} (includes g), companion = U{8..64} + g
    The decode part of workload 4 is :func:`mixed_decode_lens`.
    """
    rng = np.random.default_rng(config if seed is None else seed)
    if config == 1:
        return np.array([37, 200], dtype=np.int32)
    if config == 2:
        return rng.integers(300, 3000, size=16, endpoint=True).astype(np.int32)
    if config == 3:
        return np.array([context], dtype=np.int32)
    if config == 5:
        g = rng.integers(16, 512, size=16, endpoint=True)
        cond = rng.integers(1000, 8000, size=16, endpoint=True)
        comp = rng.integers(8, 64, size=16, endpoint=True) + g
        out = np.empty(32, dtype=np.int32)
        out[0::2] = cond
        out[1::2] = comp
        return out
    raise ValueError(f"no decode lengths for workload {config}")


def mixed_decode_lens(seed: int = 4, n: int = 15) -> np.ndarray:
    """Workload 4: the concurrent decode requests, U{500..5000}."""
    rng = np.random.default_rng(seed)
    return rng.integers(500, 5000, size=n, endpoint=True).astype(np.int32)


# ----------------------------------------------------------------------------
# page placement
# ----------------------------------------------------------------------------

def place_pages(rng: np.random.Generator, lens, page_size: int, permute: bool = True,
                spare_pages: int = 0, max_pages: Optional[int] = None):
    """Give each request ceil(len / page_size) physical pages.

    Returns (block_table [B, max_pages] int32, num_pages, poison_page). The pool
    holds the requests' pages, ``spare_pages`` unused pages and one last page
    (``poison_page``) that every unused block-table entry points at.
    """
    lens = np.asarray(lens, dtype=np.int64)
    need = (lens + page_size - 1) // page_size
    used = int(need.sum())
    if max_pages is None:
        max_pages = max(1, int(need.max()) if len(need) else 1)
    if len(need) and int(need.max()) > max_pages:
        raise ValueError("max_pages smaller than a request's page count")
    n_assignable = used + spare_pages
    ids = rng.permutation(n_assignable) if permute else np.arange(n_assignable)
    poison_page = n_assignable
    bt = np.full((len(lens), max_pages), poison_page, dtype=np.int32)
    cur = 0
    for b, n in enumerate(need):
        bt[b, :n] = ids[cur:cur + n]
        cur += n
    return bt, n_assignable + 1, poison_page


def slots_of(block_table: np.ndarray, b: int, positions: np.ndarray, page_size: int) -> np.ndarray:
    """Slot indices of logical positions of request b (slot = page * page_size + offset)."""
    positions = np.asarray(positions, dtype=np.int64)
    pages = block_table[b, positions // page_size].astype(np.int64)
    return (pages * page_size + positions % page_size).astype(np.int32)


# ----------------------------------------------------------------------------
# value draws
# ----------------------------------------------------------------------------

def _generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, gen: torch.Generator, device, chunk_elems: int = 1 << 26) -> torch.Tensor:
    """fp32 N(0, 1) draws rounded to bf16, drawn in chunks to bound fp32 temporaries."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk_elems):
        e = min(n, s + chunk_elems)
        flat[s:e] = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    return out


def _nan_like_bf16(device) -> torch.Tensor:
    return torch.tensor([BF16_NAN_BITS], dtype=torch.int16).view(torch.bfloat16).to(device)


def _poison_slots(k_pages, v_pages, block_table, valid_lens, page_size, poison_page):
    """NaN every slot that no read may touch: tails past valid_lens and the poison page."""
    nan = _nan_like_bf16(k_pages.device)
    pages, offs = [], []
    for b, n in enumerate(valid_lens):
        total_pages_b = int((block_table[b] != poison_page).sum())
        # from position n to the end of the request's last allocated page
        for j in range(int(n), total_pages_b * page_size):
            pages.append(int(block_table[b, j // page_size]))
            offs.append(j % page_size)
    if pages:
        pi = torch.tensor(pages, dtype=torch.long, device=k_pages.device)
        oi = torch.tensor(offs, dtype=torch.long, device=k_pages.device)
        k_pages[:, pi, :, oi, :] = nan
        v_pages[:, pi, :, oi, :] = nan
    k_pages[:, poison_page] = nan
    v_pages[:, poison_page] = nan


# ----------------------------------------------------------------------------
# cases
# ----------------------------------------------------------------------------

@dataclass
class DecodeCase:
    """A decode step: request b sees seq_lens[b] tokens, the last one appended this step."""
    geom: Geometry
    seq_lens: np.ndarray          # [B] int32
    block_table: np.ndarray       # [B, max_pages] int32
    num_pages: int
    poison_page: int
    q: torch.Tensor               # [L, B, Hq, D] bf16
    k_pages: torch.Tensor         # [L, P, Hkv, ps, D] bf16
    v_pages: torch.Tensor
    k_new: Optional[torch.Tensor]  # [L, B, Hkv, D] bf16 (None when nothing is pending)
    v_new: Optional[torch.Tensor]
    slot_mapping: np.ndarray      # [B] int32, -1 for rows with seq_len 0
    seed: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def layers(self) -> int:
        return int(self.q.shape[0])

    def kv_bytes_per_layer(self) -> int:
        """Bytes of K and V a decode pass must read at least once (each cached row once)."""
        g = self.geom
        return int(self.seq_lens.astype(np.int64).sum()) * g.n_kv_heads * g.head_dim * 2 * 2


def decode_case(seed: int, seq_lens, *, geom: Geometry = QWEN3, layers: int = 1, device="cpu",
                pending_append: bool = True, permute: bool = True, poison: bool = True,
                spare_pages: int = 0, max_pages: Optional[int] = None) -> DecodeCase:
    """Build a decode step. With ``pending_append`` the token at position seq_len - 1
    is not yet in the pool (its slot holds poison) and comes as k_new / v_new."""
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    rng = np.random.default_rng(seed)
    bt, num_pages, poison_page = place_pages(rng, seq_lens, geom.page_size, permute, spare_pages, max_pages)
    gen = _generator(seed, device)
    B = len(seq_lens)
    L = layers
    kp = normal_bf16((L, num_pages, geom.n_kv_heads, geom.page_size, geom.head_dim), gen, device)
    vp = normal_bf16((L, num_pages, geom.n_kv_heads, geom.page_size, geom.head_dim), gen, device)
    q = normal_bf16((L, B, geom.n_q_heads, geom.head_dim), gen, device)
    slot = np.full(B, -1, dtype=np.int32)
    for b in range(B):
        if seq_lens[b] > 0:
            slot[b] = slots_of(bt, b, np.array([seq_lens[b] - 1]), geom.page_size)[0]
    k_new = v_new = None
    if pending_append:
        k_new = normal_bf16((L, B, geom.n_kv_heads, geom.head_dim), gen, device)
        v_new = normal_bf16((L, B, geom.n_kv_heads, geom.head_dim), gen, device)
    if poison:
        cached = seq_lens - 1 if pending_append else seq_lens
        _poison_slots(kp, vp, bt, np.maximum(cached, 0), geom.page_size, poison_page)
    return DecodeCase(geom, seq_lens, bt, num_pages, poison_page, q, kp, vp, k_new, v_new, slot, seed)


@dataclass
class PrefillCase:
    """Chunked prefill of num_seqs requests plus optional concurrent decode requests (one pool)."""
    geom: Geometry
    prefix_lens: np.ndarray       # [S] int32
    q_lens: np.ndarray            # [S] int32
    cu_q_lens: np.ndarray         # [S + 1] int32
    block_table: np.ndarray       # [S, max_pages] int32 (chunk requests)
    num_pages: int
    poison_page: int
    q: torch.Tensor               # [L, total_q, Hq, D]
    k_new: torch.Tensor           # [L, total_q, Hkv, D] (the chunks' own K/V, pending)
    v_new: torch.Tensor
    slot_mapping: np.ndarray      # [total_q]
    k_pages: torch.Tensor         # [L, P, Hkv, ps, D]
    v_pages: torch.Tensor
    dec_seq_lens: np.ndarray      # [Bd] (decode requests; may be empty)
    dec_block_table: np.ndarray   # [Bd, max_pages_dec]
    dec_q: Optional[torch.Tensor]  # [L, Bd, Hq, D]
    dec_k_new: Optional[torch.Tensor]
    dec_v_new: Optional[torch.Tensor]
    dec_slot_mapping: np.ndarray
    seed: int = 0

    @property
    def total_q(self) -> int:
        return int(self.cu_q_lens[-1])


def prefill_case(seed: int, prefix_lens, q_lens, *, dec_seq_lens=(), geom: Geometry = QWEN3,
                 layers: int = 1, device="cpu", permute: bool = True, poison: bool = True,
                 max_pages: Optional[int] = None) -> PrefillCase:
    prefix_lens = np.asarray(prefix_lens, dtype=np.int32)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    dec_seq_lens = np.asarray(dec_seq_lens, dtype=np.int32)
    S, Bd = len(prefix_lens), len(dec_seq_lens)
    totals = np.concatenate([prefix_lens.astype(np.int64) + q_lens, dec_seq_lens.astype(np.int64)])
    rng = np.random.default_rng(seed)
    bt_all, num_pages, poison_page = place_pages(rng, totals, geom.page_size, permute, 0, max_pages)
    ps = geom.page_size
    bt = bt_all[:S]
    dec_bt = bt_all[S:]
    if Bd:
        dec_w = max(1, int(((dec_seq_lens.astype(np.int64) + ps - 1) // ps).max()))
        dec_bt = np.ascontiguousarray(dec_bt[:, :dec_w])
    gen = _generator(seed, device)
    L = layers
    kp = normal_bf16((L, num_pages, geom.n_kv_heads, ps, geom.head_dim), gen, device)
    vp = normal_bf16((L, num_pages, geom.n_kv_heads, ps, geom.head_dim), gen, device)
    cu = np.zeros(S + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    total_q = int(cu[-1])
    q = normal_bf16((L, total_q, geom.n_q_heads, geom.head_dim), gen, device)
    k_new = normal_bf16((L, total_q, geom.n_kv_heads, geom.head_dim), gen, device)
    v_new = normal_bf16((L, total_q, geom.n_kv_heads, geom.head_dim), gen, device)
    slot = np.empty(total_q, dtype=np.int32)
    for n in range(S):
        pos = np.arange(prefix_lens[n], prefix_lens[n] + q_lens[n])
        slot[cu[n]:cu[n + 1]] = slots_of(bt, n, pos, ps)
    dec_q = dec_k = dec_v = None
    dec_slot = np.full(Bd, -1, dtype=np.int32)
    if Bd:
        dec_q = normal_bf16((L, Bd, geom.n_q_heads, geom.head_dim), gen, device)
        dec_k = normal_bf16((L, Bd, geom.n_kv_heads, geom.head_dim), gen, device)
        dec_v = normal_bf16((L, Bd, geom.n_kv_heads, geom.head_dim), gen, device)
        for b in range(Bd):
            if dec_seq_lens[b] > 0:
                dec_slot[b] = slots_of(dec_bt, b, np.array([dec_seq_lens[b] - 1]), ps)[0]
    if poison:
        cached = np.concatenate([prefix_lens, np.maximum(dec_seq_lens - 1, 0)])
        _poison_slots(kp, vp, bt_all, cached, ps, poison_page)
    return PrefillCase(geom, prefix_lens, q_lens, cu, np.ascontiguousarray(bt), num_pages, poison_page,
                       q, k_new, v_new, slot, kp, vp, dec_seq_lens, dec_bt, dec_q, dec_k, dec_v, dec_slot, seed)
