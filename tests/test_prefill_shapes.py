"""Chunked-prefill attention for cache geometries other than the Qwen3 decoder's
16/8/128, against the fp64 oracle.

The pages name further decoder backbones for the same slot (a Llama-style 2B
model, Qwen3-8B, OLMo-2-7B, SmolLM2-1.7B) without head counts, so these are the
geometries of the decode shape tests: 1 to 8 query heads per KV head, head_dim
64 and 128, several KV-head counts. The kernel pairs the query heads of a KV
head (an odd group's last pair repeats its head in the second slot and writes
only the first), so odd groups, G = 1 among them, are covered too. Small
chunks compare every row; longer ones every 13th row (coprime to the 128-row
query tile, so every row offset is reached) plus every row of the query tiles
whose key range the split schedule divides between CTAs. Same bar as the
tuned path (tests/parity.py).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_gb300 as pkv
from gpu_util import bits, ensure_built, i32
from parity import assert_close, bf16_to_f64
from paged_kv_decode_gb300 import workloads as W
from test_decode_shapes import SHAPES
from test_prefill import SAMPLE_STRIDE, split_cut_tiles

pytestmark = pytest.mark.gpu


def _run(case, dev, rows=None, what=""):
    ensure_built()
    g = case.geom
    kp, vp = case.k_pages[0].to(dev), case.v_pages[0].to(dev)
    q = case.q[0].to(dev)
    out = torch.full_like(q, float("nan"))
    max_q = int(case.q_lens.max())
    ws = pkv.Workspace(pkv.prefill_workspace_bytes(len(case.prefix_lens), max_q, case.num_pages, g.n_q_heads,
                                                   g.n_kv_heads, g.head_dim), dev)
    pkv.append(case.k_new[0].to(dev), case.v_new[0].to(dev), i32(case.slot_mapping, dev), kp, vp, ws)
    pkv.prefill_chunk_attn(q, kp, vp, i32(case.block_table, dev), i32(case.prefix_lens, dev),
                           i32(case.cu_q_lens, dev), out, g.scale, max_q, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0, what
    want_k, want_v = oracle.append(case.k_new[0], case.v_new[0], case.slot_mapping, case.k_pages[0], case.v_pages[0])
    assert np.array_equal(bits(kp), want_k) and np.array_equal(bits(vp), want_v), what
    want = oracle.prefill(case.q[0], want_k, want_v, case.block_table, case.prefix_lens, case.cu_q_lens, g.scale,
                          rows=rows)
    got = bf16_to_f64(out)
    assert_close(got if rows is None else got[np.asarray(rows)], want, what)
    return out


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_small_chunks_all_rows(cuda_device, shape):
    # two requests: a chunk of 300 rows after 130 cached tokens (a ragged last query tile, a prefix that is
    # not a multiple of the page) and one of 77 rows after none
    case = W.prefill_case(61, [130, 0], [300, 77], geom=SHAPES[shape], poison=True)
    _run(case, cuda_device, what=f"{shape} small chunks")


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_split_schedule(cuda_device, shape):
    # long cached prefixes: CTAs take equal shares of key tiles that cut through (request, head pair,
    # query tile) items, and the cut items' partial records are merged. Geometries with few head pairs
    # need more query tiles before whole items stop balancing over the SMs: four 2048-row chunks.
    geom = SHAPES[shape]
    pairs = geom.n_kv_heads * ((geom.n_q_heads // geom.n_kv_heads + 1) // 2)
    sms = torch.cuda.get_device_properties(cuda_device).multi_processor_count
    prefix, qlen, stride = [3000, 5000], [700, 1024], SAMPLE_STRIDE
    if not split_cut_tiles(prefix, qlen, sms, kv_heads=pairs):
        prefix, qlen, stride = [9000] * 4, [2048] * 4, 37  # 37 is coprime to 128 as well
    cut = split_cut_tiles(prefix, qlen, sms, kv_heads=pairs)
    assert cut, "expected the split schedule"
    case = W.prefill_case(62, prefix, qlen, geom=geom, poison=True)
    rows = set()
    for n in range(len(prefix)):
        lo, hi = int(case.cu_q_lens[n]), int(case.cu_q_lens[n + 1])
        rows |= set(range(lo, hi, stride)) | set(range(max(lo, hi - 16), hi))
    for n, t in cut[:: max(1, len(cut) // 2)][:2]:
        lo = int(case.cu_q_lens[n]) + 128 * t
        rows |= set(range(lo, min(lo + 128, int(case.cu_q_lens[n + 1]))))
    _run(case, cuda_device, rows=sorted(rows), what=f"{shape} split schedule")


@pytest.mark.parametrize("shape", ["g4_d128_32q8kv", "g2_d64_16q8kv", "g1_d128_32q32kv"])
def test_full_chunk_after_prefix(cuda_device, shape):
    # a 4096-row chunk after 8192 cached tokens, sampled rows
    case = W.prefill_case(63, [8192], [W.PREFILL_CHUNK], geom=SHAPES[shape], poison=True)
    rows = sorted(set(range(0, W.PREFILL_CHUNK, SAMPLE_STRIDE)) | set(range(W.PREFILL_CHUNK - 64, W.PREFILL_CHUNK)))
    _run(case, cuda_device, rows=rows, what=f"{shape} chunk 4096 after 8192")
