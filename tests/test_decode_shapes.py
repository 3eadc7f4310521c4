"""Decode attention, KV append and the fused append + decode call for cache
geometries other than the Qwen3 decoder's 16/8/128 (the decode kernel with
run-time head counts), against the fp64 oracle.

The pages name further decoder backbones for the same slot (a Llama-style 2B
model, Qwen3-8B, OLMo-2-7B, SmolLM2-1.7B) but give no head counts, so the
geometries here span the supported range instead: 1 to 8 query heads per KV
head (3, 5, 6 and 7 padded inside the kernel), head_dim 64 and 128, several
KV-head counts. Same bar as the
tuned path (tests/parity.py); exact cases bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_gb300 as pkv
from gpu_util import DecodeOnDevice, bits, i32
from parity import MEAN_ABS, REL_L2, assert_close, bf16_to_f64, stats
from paged_kv_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SHAPES = {
    "g4_d128_32q8kv": W.Geometry(32, 8, 128),
    "g1_d128_32q32kv": W.Geometry(32, 32, 128),
    "g1_d64_32q32kv": W.Geometry(32, 32, 64),
    "g2_d64_16q8kv": W.Geometry(16, 8, 64),
    "g8_d128_64q8kv": W.Geometry(64, 8, 128),
    "g8_d64_8q1kv": W.Geometry(8, 1, 64),
    "g2_d128_12q6kv": W.Geometry(12, 6, 128),
    "g4_d64_16q4kv": W.Geometry(16, 4, 64),
    # groups of 3, 5, 6 and 7 run padded to 4 or 8 heads
    "g3_d128_12q4kv": W.Geometry(12, 4, 128),
    "g5_d128_40q8kv": W.Geometry(40, 8, 128),
    "g6_d64_12q2kv": W.Geometry(12, 2, 64),
    "g7_d128_28q4kv": W.Geometry(28, 4, 128),
    "g7_d64_14q2kv": W.Geometry(14, 2, 64),
}


def _check(case, dev, what):
    run = DecodeOnDevice(case, 0, dev)
    out = run.step()
    torch.cuda.synchronize()
    kp, vp = run.pools_cpu()
    if case.k_new is not None:  # the append is bit-exact
        want_k, want_v = oracle.append(case.k_new[0], case.v_new[0], case.slot_mapping, case.k_pages[0],
                                       case.v_pages[0])
        assert np.array_equal(bits(kp), want_k) and np.array_equal(bits(vp), want_v), what
    want = oracle.decode(case.q[0], bits(kp), bits(vp), case.block_table, case.seq_lens, case.geom.scale)
    assert_close(bf16_to_f64(out), want, what)
    assert run.ws.status() == 0
    return run


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_batch16_mixed_lengths(cuda_device, shape):
    geom = SHAPES[shape]
    case = W.decode_case(21, W.config_seq_lens(2), geom=geom, pending_append=True, poison=True)
    _check(case, cuda_device, f"{shape} bs16")


@pytest.mark.parametrize("shape", ["g4_d128_32q8kv", "g1_d64_32q32kv", "g8_d128_64q8kv"])
def test_long_context_one_request(cuda_device, shape):
    case = W.decode_case(22, [40000], geom=SHAPES[shape], pending_append=True, poison=True)
    _check(case, cuda_device, f"{shape} 40k")


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_ragged_and_empty_rows(cuda_device, shape):
    lens = [1, 0, 17, 15, 16, 33, 0, 250, 4095, 3, 30000, 5]
    case = W.decode_case(23, lens, geom=SHAPES[shape], pending_append=True, poison=True)
    run = _check(case, cuda_device, f"{shape} ragged")
    out = run.out.cpu()
    for b in np.flatnonzero(np.asarray(lens) == 0):
        assert torch.count_nonzero(out[b].view(torch.int16)).item() == 0


@pytest.mark.parametrize("shape", ["g1_d64_32q32kv", "g8_d128_64q8kv"])
def test_single_cached_token_is_exact(cuda_device, shape):
    # softmax over one key is 1 and 1 * v rounds back to the same bf16
    case = W.decode_case(24, [1, 1, 1], geom=SHAPES[shape], pending_append=False, poison=True)
    run = DecodeOnDevice(case, 0, cuda_device)
    out = run.step()
    torch.cuda.synchronize()
    g = case.geom
    G = g.n_q_heads // g.n_kv_heads
    vp = bits(run.v_pages.cpu())
    for b in range(3):
        page = int(case.block_table[b, 0])
        for hq in range(g.n_q_heads):
            assert np.array_equal(bits(out[b, hq].cpu()), vp[page, hq // G, 0])


@pytest.mark.parametrize("shape", ["g4_d128_32q8kv", "g1_d64_32q32kv"])
def test_graph_replay_and_workspace_reuse(cuda_device, shape):
    # the split counters return to zero, so replays and repeated calls give the same bits
    case = W.decode_case(25, [40000, 300, 7000, 1], geom=SHAPES[shape], pending_append=False, poison=True)
    run = DecodeOnDevice(case, 0, cuda_device)
    eager = run.step().clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run.step()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run.step()
    for _ in range(3):
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(run.out.view(torch.int16), eager.view(torch.int16))
    counters = run.ws.tensor[pkv.PKV_STATUS_BYTES:pkv.PKV_STATUS_BYTES + 4 * case.batch * case.geom.n_kv_heads]
    assert torch.count_nonzero(counters).item() == 0
    assert run.ws.status() == 0


def test_page_id_outside_pool_is_reported(cuda_device):
    geom = SHAPES["g4_d128_32q8kv"]
    case = W.decode_case(26, [100, 40], geom=geom, pending_append=False, poison=True)
    run = DecodeOnDevice(case, 0, cuda_device)
    bt = case.block_table.copy()
    bt[1, 0] = case.num_pages + 5
    run.block_table = i32(bt, cuda_device)
    run.step()
    torch.cuda.synchronize()
    assert run.ws.status() == -7  # PKV_ERR_OUT_OF_BOUNDS


def _fused(case, layer, dev, early=False):
    run = DecodeOnDevice(case, layer, dev)
    pkv.decode_append_attn(run.q, run.k_new, run.v_new, run.k_pages, run.v_pages, run.block_table, run.seq_lens,
                           run.out, case.geom.scale, run.ws, early_prefetch=early)
    torch.cuda.synchronize()
    return run


FUSED_LENS = [700, 0, 33, 1, 16, 17, 2900, 5000]  # padding row, page boundaries, one-token and long rows


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_fused_append_decode_matches_oracle(cuda_device, shape):
    # one launch appends each request's new K/V rows and attends over the cache with them
    case = W.decode_case(28, FUSED_LENS, geom=SHAPES[shape], pending_append=True, poison=True)
    run = _fused(case, 0, cuda_device)
    want_k, want_v = oracle.append(case.k_new[0], case.v_new[0], case.slot_mapping, case.k_pages[0], case.v_pages[0])
    assert np.array_equal(bits(run.k_pages.cpu()), want_k) and np.array_equal(bits(run.v_pages.cpu()), want_v)
    want = oracle.decode(case.q[0], want_k, want_v, case.block_table, case.seq_lens, case.geom.scale)
    assert_close(bf16_to_f64(run.out), want, f"{shape} fused")
    for b, n in enumerate(case.seq_lens):
        if n == 0:
            assert torch.count_nonzero(run.out[b].view(torch.int16)).item() == 0
    assert run.ws.status() == 0


@pytest.mark.parametrize("shape", ["g4_d128_32q8kv", "g8_d64_8q1kv", "g1_d64_32q32kv", "g6_d64_12q2kv"])
def test_fused_equals_separate_calls_bitwise(cuda_device, shape):
    case = W.decode_case(29, FUSED_LENS, geom=SHAPES[shape], pending_append=True, poison=True)
    sep = DecodeOnDevice(case, 0, cuda_device)
    out_sep = sep.step().clone()
    fused = _fused(case, 0, cuda_device)
    assert torch.equal(out_sep.view(torch.int16), fused.out.view(torch.int16))
    assert torch.equal(sep.k_pages.view(torch.int16), fused.k_pages.view(torch.int16))
    assert torch.equal(sep.v_pages.view(torch.int16), fused.v_pages.view(torch.int16))


@pytest.mark.parametrize("shape", ["g4_d128_32q8kv", "g2_d64_16q8kv"])
@pytest.mark.parametrize("early", [False, True])
def test_fused_layer_chain_in_a_graph(cuda_device, shape, early):
    # two layers, each its own pool, replayed from a CUDA graph; with early prefetch each layer's
    # kernel may read its pool while the previous layer's kernel finishes
    case = W.decode_case(30, W.config_seq_lens(2), geom=SHAPES[shape], layers=2, pending_append=True, poison=True)
    runs = [DecodeOnDevice(case, layer, cuda_device) for layer in range(2)]

    def step():
        for r in runs:
            pkv.decode_append_attn(r.q, r.k_new, r.v_new, r.k_pages, r.v_pages, r.block_table, r.seq_lens, r.out,
                                   case.geom.scale, r.ws, early_prefetch=early)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for layer, r in enumerate(runs):  # the graph's replay appends again at the same slots: same bits
        r.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    for layer, r in enumerate(runs):
        want_k, want_v = oracle.append(case.k_new[layer], case.v_new[layer], case.slot_mapping,
                                       case.k_pages[layer], case.v_pages[layer])
        assert np.array_equal(bits(r.k_pages.cpu()), want_k) and np.array_equal(bits(r.v_pages.cpu()), want_v)
        want = oracle.decode(case.q[layer], want_k, want_v, case.block_table, case.seq_lens, case.geom.scale)
        assert_close(bf16_to_f64(r.out), want, f"{shape} graph layer {layer} early={early}")
        assert r.ws.status() == 0


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_rope_call_matches_oracle(cuda_device, shape):
    # the fused append + decode with the rotary embedding of the new token (theta 1e6, the table from
    # the oracle): rotated key rows bit-exact, outputs against decode over the double-rotated queries
    geom = SHAPES[shape]
    lens = [1, 0, 17, 300, 33, 2000, 16]
    case = W.decode_case(27, lens, geom=geom, pending_append=True, poison=True)
    cs = oracle.rope_cache(1e6, geom.head_dim, int(max(lens)) + 1)
    run = DecodeOnDevice(case, 0, cuda_device)
    pkv.decode_append_rope_attn(run.q, run.k_new, run.v_new, run.k_pages, run.v_pages, run.block_table,
                                run.seq_lens, torch.from_numpy(cs).to(cuda_device), run.out, geom.scale, run.ws,
                                early_prefetch=True)
    torch.cuda.synchronize()
    assert run.ws.status() == 0
    pos = np.asarray(case.seq_lens, dtype=np.int64) - 1  # -1 for the empty request: nothing appended
    k_rot = oracle.rope_bf16(case.k_new[0], pos, cs)
    want_k, want_v = oracle.append(k_rot, case.v_new[0], case.slot_mapping, case.k_pages[0], case.v_pages[0])
    assert np.array_equal(bits(run.k_pages), want_k) and np.array_equal(bits(run.v_pages), want_v)
    # The call rotates each query row in fp32 and rounds it to bf16, the score product's operand (the
    # header's definition). Element by element the oracle gets the query rotated by its bf16 form
    # (rope_bf16: the same formula and rounding decision, pinned against the double rotation); against
    # the double rotation itself the mean and relative-L2 bars hold as well.
    got = bf16_to_f64(run.out)
    want = oracle.decode(oracle.rope_bf16(case.q[0], pos, cs), want_k, want_v, case.block_table, case.seq_lens,
                         geom.scale)
    assert_close(got, want, f"{shape} rope")
    exact = stats(got, oracle.decode(oracle.rope_f64(case.q[0], pos, cs), want_k, want_v, case.block_table,
                                     case.seq_lens, geom.scale))
    assert exact["mean_abs"] <= MEAN_ABS and exact["rel_l2"] <= REL_L2, exact


def test_rope_position_beyond_table_is_reported(cuda_device):
    geom = SHAPES["g4_d64_16q4kv"]
    case = W.decode_case(28, [300, 40], geom=geom, pending_append=True, poison=False)
    cs = oracle.rope_cache(1e6, geom.head_dim, 100)  # 300 - 1 is past the last row
    run = DecodeOnDevice(case, 0, cuda_device)
    pkv.decode_append_rope_attn(run.q, run.k_new, run.v_new, run.k_pages, run.v_pages, run.block_table,
                                run.seq_lens, torch.from_numpy(cs).to(cuda_device), run.out, geom.scale, run.ws)
    torch.cuda.synchronize()
    assert run.ws.status() == pkv.ERR_CODES["PKV_ERR_OUT_OF_BOUNDS"]


@pytest.mark.parametrize("ranks", [2, 4, 8])
def test_kv_head_shards_reproduce_the_full_decode(cuda_device, ranks):
    # KV-head sharding (what a rank would hold when the KV cache is split across GPUs by KV head): shard r
    # keeps KV heads [r 8/N, (r+1) 8/N) of every page and their query heads, and is a geometry of its own
    # (16/N query, 8/N KV heads); each shard is an independent decode call here, on one GPU. The shards'
    # outputs, put side by side along the heads, equal the unsharded call's and the oracle's.
    case = W.decode_case(29, W.config_seq_lens(2), pending_append=False, poison=True)
    full = DecodeOnDevice(case, 0, cuda_device)
    ref = full.step().clone()
    torch.cuda.synchronize()
    kv_per, q_per = 8 // ranks, 16 // ranks
    parts = []
    for r in range(ranks):
        kp = full.k_pages[:, r * kv_per:(r + 1) * kv_per].contiguous()
        vp = full.v_pages[:, r * kv_per:(r + 1) * kv_per].contiguous()
        q = full.q[:, r * q_per:(r + 1) * q_per].contiguous()
        out = torch.full_like(q, float("nan"))
        ws = pkv.Workspace(pkv.decode_workspace_bytes(case.batch, case.max_pages, case.num_pages, q_per, kv_per,
                                                      128), cuda_device)
        pkv.decode_attn(q, kp, vp, full.block_table, full.seq_lens, out, case.geom.scale, ws)
        torch.cuda.synchronize()
        assert ws.status() == 0
        parts.append(out)
    sharded = torch.cat(parts, dim=1)
    want = oracle.decode(case.q[0], case.k_pages[0], case.v_pages[0], case.block_table, case.seq_lens,
                         case.geom.scale)
    assert_close(bf16_to_f64(sharded), want, f"{ranks} KV-head shards")
    assert_close(bf16_to_f64(sharded), bf16_to_f64(ref), f"{ranks} KV-head shards vs the unsharded call")
