"""Chunked-prefill attention on the GPU (tcgen05 kernel) against the fp64 oracle.

Small cases compare every output row. Full-size chunks (4096 rows after 0,
8192 or 32768 cached tokens) compare sampled rows, all heads, which the oracle
computes one by one: every 13th row (13 is coprime to the 128-row query tile,
so every row offset of a tile is hit), the last 64 rows, and every row of the
query tiles whose key range the split schedule divides between CTAs (there
the partial records and their merge produce the rows). The mixed step of
workload 4 (the chunk plus 15 decode requests in one pool, as one CUDA graph
with two branches) is compared with the oracle too. Bar as elsewhere:
max |diff| <= 1e-2, mean |diff| <= 1e-3, relative L2 <= 1e-2.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_gb300 as pkv
from gpu_util import bits, ensure_built, i32
from parity import assert_close, bf16_to_f64
from paged_kv_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu


class PrefillOnDevice:
    def __init__(self, case, dev, layer=0):
        ensure_built()
        self.case = case
        self.q = case.q[layer].to(dev)
        self.k_pages = case.k_pages[layer].to(dev)
        self.v_pages = case.v_pages[layer].to(dev)
        self.k_new = case.k_new[layer].to(dev)
        self.v_new = case.v_new[layer].to(dev)
        self.slots = i32(case.slot_mapping, dev)
        self.block_table = i32(case.block_table, dev)
        self.prefix = i32(case.prefix_lens, dev)
        self.cu = i32(case.cu_q_lens, dev)
        self.out = torch.full_like(self.q, float("nan"))
        self.ws = pkv.Workspace(pkv.prefill_workspace_bytes(len(case.prefix_lens), int(case.q_lens.max())), dev)
        self.max_q_len = int(case.q_lens.max())

    def run(self):
        pkv.append(self.k_new, self.v_new, self.slots, self.k_pages, self.v_pages, self.ws)
        pkv.prefill_chunk_attn(self.q, self.k_pages, self.v_pages, self.block_table, self.prefix, self.cu, self.out,
                               self.case.geom.scale, self.max_q_len, self.ws)
        torch.cuda.synchronize()
        return self.out

    def oracle_pools(self):
        c = self.case
        return oracle.append(c.k_new[0], c.v_new[0], c.slot_mapping, c.k_pages[0], c.v_pages[0])


def _check(case, dev, rows=None, what=""):
    run = PrefillOnDevice(case, dev)
    out = run.run()
    kp, vp = run.oracle_pools()
    assert np.array_equal(bits(run.k_pages), kp) and np.array_equal(bits(run.v_pages), vp)
    want = oracle.prefill(case.q[0], kp, vp, case.block_table, case.prefix_lens, case.cu_q_lens, case.geom.scale,
                          rows=rows)
    got = bf16_to_f64(out)
    got = got if rows is None else got[np.asarray(rows)]
    assert_close(got, want, what)
    assert run.ws.status() == 0
    return run


@pytest.mark.parametrize("prefix,qlen", [(0, 128), (0, 300), (5, 77), (130, 1), (16, 200), (1000, 257)])
def test_small_chunks_all_rows(cuda_device, prefix, qlen):
    case = W.prefill_case(40 + qlen, [prefix], [qlen], poison=True)
    _check(case, cuda_device, what=f"P={prefix} L={qlen}")


def test_several_requests_in_one_call(cuda_device):
    case = W.prefill_case(41, [0, 33, 500], [129, 64, 250], poison=True)
    _check(case, cuda_device, what="3 requests")


SAMPLE_STRIDE = 13  # coprime to the 128-row query tile: the samples reach every row offset


def _sample_rows(total):
    rows = list(range(0, total, SAMPLE_STRIDE)) + list(range(max(0, total - 64), total))
    return sorted(set(rows))


def split_cut_tiles(prefix_lens, q_lens, workers, item_cost=2, kv_heads=8, tile=128, item_mode_pct=75):
    """(request, query tile) pairs whose key tiles the prefill kernel's split schedule divides
    between CTAs; empty when its item schedule runs. A test-side model of the schedule's rule, used
    only to choose which rows to compare: items are ordered by request, KV head, query tile; an item
    costs item_cost units plus one per key tile; CTA c of G = min(workers, U) takes units
    [c U / G, (c + 1) U / G); the item schedule runs when the largest item has at least
    item_mode_pct % of a CTA's average key tiles."""
    items = []
    for n, (P, L) in enumerate(zip(prefix_lens, q_lens)):
        T = -(-int(L) // tile)
        for g in range(kv_heads):
            for t in range(T):
                items.append((n, t, -(-(int(P) + min(int(L), tile * (t + 1))) // tile)))
    if not items:
        return []
    tiles_all = sum(nt for _, _, nt in items)
    if 100 * max(nt for _, _, nt in items) * workers >= item_mode_pct * tiles_all:
        return []
    U = sum(item_cost + nt for _, _, nt in items)
    G = min(workers, U)
    cta_of = lambda f: ((f + 1) * G + U - 1) // U - 1
    cut, f = set(), 0
    for n, t, nt in items:
        if cta_of(f + item_cost) != cta_of(f + item_cost + nt - 1):
            cut.add((n, t))
        f += item_cost + nt
    return sorted(cut)


def _workers(dev):
    return torch.cuda.get_device_properties(dev).multi_processor_count


def _cut_rows(case, dev, max_tiles):
    """All rows of up to max_tiles query tiles (spread over the list) that the split schedule cuts."""
    cut = split_cut_tiles(case.prefix_lens, case.q_lens, _workers(dev))
    pick = cut[:: max(1, len(cut) // max_tiles)][:max_tiles] if cut else []
    rows = set()
    for n, t in pick:
        lo = int(case.cu_q_lens[n]) + 128 * t
        rows |= set(range(lo, min(lo + 128, int(case.cu_q_lens[n + 1]))))
    return rows, len(cut)


@pytest.mark.parametrize("prefix", [0, 8192, 32768])
def test_full_chunk_sampled_rows(cuda_device, prefix):
    case = W.prefill_case(42, [prefix], [W.PREFILL_CHUNK], poison=True)
    cut_rows, n_cut = _cut_rows(case, cuda_device, max_tiles=2)
    if prefix > 0:
        # long cached prefixes run the split schedule (equal shares of key tiles that cut items)
        assert n_cut > 0 and len(cut_rows) == 256
    rows = sorted(set(_sample_rows(W.PREFILL_CHUNK)) | cut_rows)
    assert {r % 128 for r in rows} == set(range(128))
    _check(case, cuda_device, rows=rows, what=f"chunk 4096 after {prefix}")


def test_split_schedule_several_requests(cuda_device):
    # three requests of 1536 rows after 3000 cached tokens: the key tiles outnumber what
    # whole query tiles can balance over the SMs, so CTAs take equal shares that cut
    # through (request, head, query tile) items, some across request boundaries, and
    # the split items are merged; sampled rows of every request (every row offset of a
    # query tile) and every row of three cut query tiles
    case = W.prefill_case(44, [3000, 3000, 3000], [1536, 1536, 1536], poison=True)
    cut_rows, n_cut = _cut_rows(case, cuda_device, max_tiles=3)
    assert n_cut > 0
    rows = sorted({r for n in range(3) for r in range(n * 1536, (n + 1) * 1536, SAMPLE_STRIDE)} |
                  {n * 1536 + r for n in range(3) for r in range(1536 - 16, 1536)} | cut_rows)
    run = _check(case, cuda_device, rows=rows, what="split schedule, 3 requests")
    # merges run in an order fixed by the item, whichever CTA completes it: same bits again
    again = PrefillOnDevice(case, cuda_device).run()
    assert torch.equal(run.out.view(torch.int16), again.view(torch.int16))


def test_chunk_longer_than_max_q_len_is_reported(cuda_device):
    # max_q_len = 100 sizes the call for one 128-row query tile; a 300-row chunk then has rows the
    # call does not compute, and the status word says so (the first tile's rows are still right)
    case = W.prefill_case(46, [50], [300], poison=True)
    run = PrefillOnDevice(case, cuda_device)
    run.max_q_len = 100
    run.ws = pkv.Workspace(pkv.prefill_workspace_bytes(1, 100), cuda_device)
    out = run.run()
    assert run.ws.status() == pkv.ERR_CODES["PKV_ERR_OUT_OF_BOUNDS"]
    kp, vp = run.oracle_pools()
    want = oracle.prefill(case.q[0], kp, vp, case.block_table, case.prefix_lens, case.cu_q_lens, case.geom.scale,
                          rows=range(128))
    assert_close(bf16_to_f64(out[:128]), want, "first query tile of an over-long chunk")


def test_causality_on_gpu(cuda_device):
    # perturbing keys/values at positions after row i's limit leaves row i bit-identical
    case = W.prefill_case(43, [40], [200], poison=False)
    base = PrefillOnDevice(case, cuda_device).run().clone()
    lim_row = 100  # rows <= 100 see keys <= 140
    kn = case.k_new.clone()
    vn = case.v_new.clone()
    kn[0, lim_row + 1:] = -kn[0, lim_row + 1:]
    vn[0, lim_row + 1:] = vn[0, lim_row + 1:] * 2
    case.k_new, case.v_new = kn, vn
    pert = PrefillOnDevice(case, cuda_device).run()
    assert torch.equal(base[: lim_row + 1].view(torch.int16), pert[: lim_row + 1].view(torch.int16))
    assert not torch.equal(base[lim_row + 1:].view(torch.int16), pert[lim_row + 1:].view(torch.int16))


def test_mixed_step_graph_with_parallel_branches_equals_eager(cuda_device):
    # the mixed step of workload 4 (a chunk after cached tokens plus concurrent decode requests),
    # captured as one CUDA graph whose chunk branch (append, prefill) and decode branch (append,
    # attention) run on different streams: replays give the same bits as sequential eager calls
    case = W.prefill_case(45, [500], [700], dec_seq_lens=[90, 1000, 17, 2500], poison=True)
    dev = cuda_device

    def state():
        c = case
        return dict(kp=c.k_pages[0].to(dev), vp=c.v_pages[0].to(dev), out=torch.zeros_like(c.q[0], device=dev),
                    dout=torch.zeros_like(c.dec_q[0], device=dev))

    q, kn, vn = case.q[0].to(dev), case.k_new[0].to(dev), case.v_new[0].to(dev)
    dq, dk, dv = case.dec_q[0].to(dev), case.dec_k_new[0].to(dev), case.dec_v_new[0].to(dev)
    slots, bt = i32(case.slot_mapping, dev), i32(case.block_table, dev)
    prefix, cu = i32(case.prefix_lens, dev), i32(case.cu_q_lens, dev)
    dslots, dbt, dlens = i32(case.dec_slot_mapping, dev), i32(case.dec_block_table, dev), i32(case.dec_seq_lens, dev)
    ensure_built()
    pws = pkv.Workspace(pkv.prefill_workspace_bytes(1, 700), dev)
    dws = pkv.Workspace(pkv.decode_workspace_bytes(4, case.dec_block_table.shape[1]), dev)
    scale = case.geom.scale

    def step(s, side=None):
        pkv.append(kn, vn, slots, s["kp"], s["vp"], pws)
        pkv.prefill_chunk_attn(q, s["kp"], s["vp"], bt, prefix, cu, s["out"], scale, 700, pws)
        ctx = torch.cuda.stream(side) if side is not None else None
        if ctx:
            side.wait_stream(torch.cuda.current_stream())
            ctx.__enter__()
        pkv.append(dk, dv, dslots, s["kp"], s["vp"], dws)
        pkv.decode_attn(dq, s["kp"], s["vp"], dbt, dlens, s["dout"], scale, dws)
        if ctx:
            ctx.__exit__(None, None, None)
            torch.cuda.current_stream().wait_stream(side)

    eager = state()
    step(eager)
    torch.cuda.synchronize()
    graphed = state()
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        step(state(), side)  # warm-up outside the graph
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        step(graphed, side)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for key in ("out", "dout", "kp", "vp"):
        assert torch.equal(eager[key].view(torch.int16), graphed[key].view(torch.int16)), key
    assert pws.status() == 0 and dws.status() == 0


def _mixed_graph(case, dev):
    """Workload 4's step as one CUDA graph with two branches: the chunk's append and prefill on
    the capturing stream, the decode requests' append and attention on a side stream (disjoint
    slots, separate workspaces). Returns the graph and the device state it writes."""
    s = dict(kp=case.k_pages[0].to(dev), vp=case.v_pages[0].to(dev),
             out=torch.full_like(case.q[0], float("nan"), device=dev),
             dout=torch.full_like(case.dec_q[0], float("nan"), device=dev))
    q, kn, vn = case.q[0].to(dev), case.k_new[0].to(dev), case.v_new[0].to(dev)
    dq, dk, dv = case.dec_q[0].to(dev), case.dec_k_new[0].to(dev), case.dec_v_new[0].to(dev)
    slots, bt = i32(case.slot_mapping, dev), i32(case.block_table, dev)
    prefix, cu = i32(case.prefix_lens, dev), i32(case.cu_q_lens, dev)
    dslots, dbt, dlens = i32(case.dec_slot_mapping, dev), i32(case.dec_block_table, dev), i32(case.dec_seq_lens, dev)
    max_q = int(case.q_lens.max())
    pws = pkv.Workspace(pkv.prefill_workspace_bytes(len(case.prefix_lens), max_q), dev)
    dws = pkv.Workspace(pkv.decode_workspace_bytes(len(case.dec_seq_lens), case.dec_block_table.shape[1]), dev)
    side = torch.cuda.Stream()
    scale = case.geom.scale

    def step():
        main = torch.cuda.current_stream()
        side.wait_stream(main)
        pkv.append(kn, vn, slots, s["kp"], s["vp"], pws)
        pkv.prefill_chunk_attn(q, s["kp"], s["vp"], bt, prefix, cu, s["out"], scale, max_q, pws)
        with torch.cuda.stream(side):
            pkv.append(dk, dv, dslots, s["kp"], s["vp"], dws)
            pkv.decode_attn(dq, s["kp"], s["vp"], dbt, dlens, s["dout"], scale, dws)
        main.wait_stream(side)

    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        step()  # once outside the graph (the appends rewrite the same rows in every run)
        cap.synchronize()
        with torch.cuda.graph(g, stream=cap):
            step()
    torch.cuda.synchronize()
    return g, s, pws, dws


@pytest.mark.parametrize("prefix", [0, 32768])
def test_mixed_step_graph_matches_oracle(cuda_device, prefix):
    # workload 4 at full size: a 4096-row chunk after `prefix` cached tokens and 15 decode
    # requests U{500..5000} in one pool, as the two-branch graph; pools bit-exact against the
    # oracle's appends, sampled chunk rows (every row offset, the split schedule's cut tiles)
    # and all 15 decode rows against the oracle
    dev = cuda_device
    ensure_built()
    case = W.prefill_case(4, [prefix], [W.PREFILL_CHUNK], dec_seq_lens=W.mixed_decode_lens(4), poison=True)
    g, s, pws, dws = _mixed_graph(case, dev)
    for _ in range(2):  # a replay rewrites the same rows: the second sees the first's pools
        g.replay()
    torch.cuda.synchronize()
    assert pws.status() == 0 and dws.status() == 0
    kp, vp = oracle.append(case.k_new[0], case.v_new[0], case.slot_mapping, case.k_pages[0], case.v_pages[0])
    kp, vp = oracle.append(case.dec_k_new[0], case.dec_v_new[0], case.dec_slot_mapping, kp, vp)
    assert np.array_equal(bits(s["kp"]), kp) and np.array_equal(bits(s["vp"]), vp)
    cut_rows, _ = _cut_rows(case, dev, max_tiles=2)
    rows = sorted(set(_sample_rows(W.PREFILL_CHUNK)) | cut_rows)
    want = oracle.prefill(case.q[0], kp, vp, case.block_table, case.prefix_lens, case.cu_q_lens, case.geom.scale,
                          rows=rows)
    assert_close(bf16_to_f64(s["out"])[np.asarray(rows)], want, f"mixed step: chunk after {prefix}")
    want_d = oracle.decode(case.dec_q[0], kp, vp, case.dec_block_table, case.dec_seq_lens, case.geom.scale)
    assert_close(bf16_to_f64(s["dout"]), want_d, f"mixed step: 15 decode requests (chunk after {prefix})")


# ---------------------------------------------------------------------------- the mixed-step kernel

def mixed_workers(case, sms, pages_per_tile=24, item_mode_pct=75, kv_heads=8, tile=128):
    """Persistent prefill workers of the mixed-step kernel's split schedule: the SMs less the ones kept
    for the decode CTAs, in proportion to the decode pages' share of the SM time (a test-side model of
    the kernel's rule, used to pick the rows the split schedule cuts)."""
    tiles = [(-(-(int(P) + min(int(L), tile * (t + 1))) // tile))
             for P, L in zip(case.prefix_lens, case.q_lens) for t in range(-(-int(L) // tile))]
    tiles_all = kv_heads * sum(tiles)
    if not tiles or 100 * max(tiles) * sms >= item_mode_pct * tiles_all:
        return sms
    dec_pages = kv_heads * sum(-(-int(n) // 16) for n in case.dec_seq_lens)
    if dec_pages == 0:
        return sms
    dec_tiles = -(-dec_pages // pages_per_tile)
    k = -(-(sms * dec_tiles) // (dec_tiles + tiles_all))
    return sms - min(max(k, 1), sms // 2)


def _mixed_kernel_run(case, dev):
    """pkv_append of the chunk and the decode tokens, then one pkv_mixed_step_attn launch."""
    ensure_built()
    kp, vp = case.k_pages[0].to(dev), case.v_pages[0].to(dev)
    S = len(case.prefix_lens)
    max_q = int(case.q_lens.max()) if S else 0
    ws = pkv.Workspace(pkv.mixed_workspace_bytes(S, max_q, len(case.dec_seq_lens), case.dec_block_table.shape[1]), dev)
    q = case.q[0].to(dev)
    out = torch.full_like(q, float("nan"))
    dq = case.dec_q[0].to(dev)
    dout = torch.full_like(dq, float("nan"))
    if S:
        pkv.append(case.k_new[0].to(dev), case.v_new[0].to(dev), i32(case.slot_mapping, dev), kp, vp, ws)
    pkv.append(case.dec_k_new[0].to(dev), case.dec_v_new[0].to(dev), i32(case.dec_slot_mapping, dev), kp, vp, ws)
    pkv.mixed_step_attn(q if S else None, kp, vp, i32(case.block_table, dev) if S else None,
                        i32(case.prefix_lens, dev) if S else None, i32(case.cu_q_lens, dev) if S else None,
                        out if S else None, max_q, dq, i32(case.dec_block_table, dev), i32(case.dec_seq_lens, dev),
                        dout, case.geom.scale, ws)
    torch.cuda.synchronize()
    assert ws.status() == 0
    want_k, want_v = oracle.append(case.k_new[0], case.v_new[0], case.slot_mapping, case.k_pages[0], case.v_pages[0])
    want_k, want_v = oracle.append(case.dec_k_new[0], case.dec_v_new[0], case.dec_slot_mapping, want_k, want_v)
    assert np.array_equal(bits(kp), want_k) and np.array_equal(bits(vp), want_v)
    return out, dout, want_k, want_v


@pytest.mark.parametrize("prefix", [0, 8192, 32768])
def test_mixed_step_kernel_matches_oracle(cuda_device, prefix):
    # workload 4 at full size through the one-launch mixed step: a 4096-row chunk after `prefix` cached
    # tokens and 15 decode requests U{500..5000}; sampled chunk rows (every row offset, every row of two
    # tiles the split schedule cuts) and all decode rows against the oracle
    case = W.prefill_case(4, [prefix], [W.PREFILL_CHUNK], dec_seq_lens=W.mixed_decode_lens(4), poison=True)
    out, dout, kp, vp = _mixed_kernel_run(case, cuda_device)
    workers = mixed_workers(case, _workers(cuda_device))
    cut = split_cut_tiles(case.prefix_lens, case.q_lens, workers)
    if prefix > 0:
        assert cut and workers < _workers(cuda_device)  # split schedule, SMs kept for the decode CTAs
    rows = set(_sample_rows(W.PREFILL_CHUNK))
    for n, t in cut[:: max(1, len(cut) // 2)][:2]:
        rows |= set(range(128 * t, min(128 * t + 128, W.PREFILL_CHUNK)))
    rows = sorted(rows)
    want = oracle.prefill(case.q[0], kp, vp, case.block_table, case.prefix_lens, case.cu_q_lens, case.geom.scale,
                          rows=rows)
    assert_close(bf16_to_f64(out)[np.asarray(rows)], want, f"mixed kernel: chunk after {prefix}")
    want_d = oracle.decode(case.dec_q[0], kp, vp, case.dec_block_table, case.dec_seq_lens, case.geom.scale)
    assert_close(bf16_to_f64(dout), want_d, f"mixed kernel: decode requests (chunk after {prefix})")


def test_mixed_step_kernel_small_all_rows(cuda_device):
    # two chunks and a ragged decode batch (empty, one-token, page-boundary and a 9-page request) in one
    # pool; every output row against the oracle
    case = W.prefill_case(47, [130, 0], [300, 77], dec_seq_lens=[0, 1, 16, 17, 129, 2000, 33], poison=True)
    out, dout, kp, vp = _mixed_kernel_run(case, cuda_device)
    want = oracle.prefill(case.q[0], kp, vp, case.block_table, case.prefix_lens, case.cu_q_lens, case.geom.scale)
    assert_close(bf16_to_f64(out), want, "mixed kernel: small chunks")
    want_d = oracle.decode(case.dec_q[0], kp, vp, case.dec_block_table, case.dec_seq_lens, case.geom.scale)
    assert_close(bf16_to_f64(dout), want_d, "mixed kernel: ragged decode batch")
    assert torch.count_nonzero(dout[0].view(torch.int16)).item() == 0  # the empty request: zeros
    # one-token request: that value row exactly
    assert torch.equal(dout[1].view(torch.int16).cpu(), torch.from_numpy(
        np.repeat(vp[case.dec_block_table[1, 0], :, 0, :].view(np.int16), 2, axis=0)))


def test_mixed_step_kernel_decode_only(cuda_device):
    # no chunk: the launch is decode attention alone
    case = W.prefill_case(48, [], [], dec_seq_lens=[300, 0, 5000, 16], poison=True)
    _, dout, kp, vp = _mixed_kernel_run(case, cuda_device)
    want_d = oracle.decode(case.dec_q[0], kp, vp, case.dec_block_table, case.dec_seq_lens, case.geom.scale)
    assert_close(bf16_to_f64(dout), want_d, "mixed kernel: decode only")


def test_many_requests_in_one_call(cuda_device):
    # 70 chunks (the length scan runs over three warps' worth of requests) of 1..300 rows after 0..2000
    # cached tokens, every row against the oracle
    rng = np.random.default_rng(70)
    prefix = rng.integers(0, 2000, size=70)
    qlens = rng.integers(1, 300, size=70)
    case = W.prefill_case(70, prefix, qlens, poison=True)
    _check(case, cuda_device, what="70 chunks")


def test_many_requests_split_schedule(cuda_device):
    # 40 chunks of 512 rows after 6000..9000 cached tokens: the split schedule, shares cutting items of many
    # requests; every 13th row and the last rows of every request
    rng = np.random.default_rng(71)
    prefix = rng.integers(6000, 9000, size=40)
    case = W.prefill_case(71, prefix, [512] * 40, poison=True)
    assert split_cut_tiles(case.prefix_lens, case.q_lens, _workers(cuda_device))
    rows = sorted({r for n in range(40) for r in range(512 * n, 512 * (n + 1), SAMPLE_STRIDE)} |
                  {512 * n + 511 for n in range(40)})
    _check(case, cuda_device, rows=rows, what="40 chunks, split schedule")


def test_mixed_step_kernel_many_requests(cuda_device):
    # 5 chunks and 64 decode requests of 1..6000 tokens (several 64-page chunks each) in one launch
    rng = np.random.default_rng(72)
    case = W.prefill_case(72, rng.integers(0, 3000, size=5), rng.integers(1, 700, size=5),
                          dec_seq_lens=rng.integers(0, 6000, size=64), poison=True)
    out, dout, kp, vp = _mixed_kernel_run(case, cuda_device)
    want = oracle.prefill(case.q[0], kp, vp, case.block_table, case.prefix_lens, case.cu_q_lens, case.geom.scale)
    assert_close(bf16_to_f64(out), want, "mixed kernel: 5 chunks")
    want_d = oracle.decode(case.dec_q[0], kp, vp, case.dec_block_table, case.dec_seq_lens, case.geom.scale)
    assert_close(bf16_to_f64(dout), want_d, "mixed kernel: 64 decode requests")
