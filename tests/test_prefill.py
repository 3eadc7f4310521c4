"""Chunked-prefill attention on the GPU (tcgen05 kernel) against the fp64 oracle.

Small cases compare every output row; full-size chunks (4096 rows after 0,
8192 or 32768 cached tokens) compare sampled rows (every 64th row, the last
64 rows, all heads), which the oracle computes one by one. Bar as elsewhere:
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


def _sample_rows(total):
    rows = list(range(0, total, 64)) + list(range(max(0, total - 64), total))
    return sorted(set(rows))


@pytest.mark.parametrize("prefix", [0, 8192, 32768])
def test_full_chunk_sampled_rows(cuda_device, prefix):
    case = W.prefill_case(42, [prefix], [W.PREFILL_CHUNK], poison=True)
    _check(case, cuda_device, rows=_sample_rows(W.PREFILL_CHUNK), what=f"chunk 4096 after {prefix}")


def test_split_schedule_several_requests(cuda_device):
    # three requests of 1536 rows after 3000 cached tokens: the key tiles outnumber what
    # whole query tiles can balance over the SMs, so CTAs take equal shares that cut
    # through (request, head, query tile) items, some across request boundaries, and
    # the split items are merged; sampled rows of every request
    case = W.prefill_case(44, [3000, 3000, 3000], [1536, 1536, 1536], poison=True)
    rows = sorted({r for n in range(3) for r in range(n * 1536, (n + 1) * 1536, 48)} |
                  {n * 1536 + r for n in range(3) for r in range(1536 - 16, 1536)})
    run = _check(case, cuda_device, rows=rows, what="split schedule, 3 requests")
    # merges run in an order fixed by the item, whichever CTA completes it: same bits again
    again = PrefillOnDevice(case, cuda_device).run()
    assert torch.equal(run.out.view(torch.int16), again.view(torch.int16))


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
