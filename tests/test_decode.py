"""Decode attention on the GPU against the fp64 oracle.

Bar: max |diff| <= 1e-2, mean |diff| <= 1e-3 and relative L2 <= 1e-2 over
every output element (tests/parity.py). Exact cases (one cached token, page
placement, empty rows) are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_gb300 as pkv
from gpu_util import DecodeOnDevice, bits, ensure_built, i32
from parity import assert_close, bf16_to_f64
from paged_kv_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _oracle_after_append(case, layer, dev_run):
    kp, vp = dev_run.pools_cpu()  # pools after the GPU append (append itself is checked bit-exact elsewhere)
    if case.k_new is not None:
        want_k, want_v = oracle.append(case.k_new[layer], case.v_new[layer], case.slot_mapping,
                                       case.k_pages[layer], case.v_pages[layer])
        assert np.array_equal(bits(kp), want_k) and np.array_equal(bits(vp), want_v)
        return want_k, want_v
    return kp, vp


def _check_case(case, dev, layers=(0,), what=""):
    for layer in layers:
        run = DecodeOnDevice(case, layer, dev)
        out = run.step()
        torch.cuda.synchronize()
        kp, vp = _oracle_after_append(case, layer, run)
        want = oracle.decode(case.q[layer], kp, vp, case.block_table, case.seq_lens, case.geom.scale)
        assert_close(bf16_to_f64(out), want, f"{what} layer {layer}")
        assert run.ws.status() == 0


def test_tiny_config(cuda_device):
    case = W.decode_case(1, W.config_seq_lens(1), pending_append=True, poison=False)
    assert case.num_pages == 17  # 16 request pages + the unused last page
    _check_case(case, cuda_device, what="tiny")


def test_qwen3_bs16_two_layers(cuda_device):
    case = W.decode_case(2, W.config_seq_lens(2), layers=2, pending_append=True, poison=True)
    _check_case(case, cuda_device, layers=(0, 1), what="bs16")


@pytest.mark.parametrize("context", [4096, 16384, 40000, 65536])
def test_long_context(cuda_device, context):
    case = W.decode_case(3, W.config_seq_lens(3, context=context), pending_append=True, poison=True)
    _check_case(case, cuda_device, what=f"context {context}")


def test_cfg_pairs(cuda_device):
    case = W.decode_case(5, W.config_seq_lens(5), pending_append=True, poison=True)
    _check_case(case, cuda_device, what="cfg")


def test_mixed_step_decode_part(cuda_device):
    case = W.decode_case(4, W.mixed_decode_lens(), pending_append=True, poison=True)
    _check_case(case, cuda_device, what="mixed decode")


@pytest.mark.parametrize("lens", [[1], [17], [15, 16, 17, 31, 32, 33], list(range(1, 65)),
                                  [40000, 16, 16, 16, 16], [3, 30000, 5, 9000]])
def test_ragged_lengths(cuda_device, lens):
    case = W.decode_case(6, lens, pending_append=True, poison=True)
    _check_case(case, cuda_device, what=f"ragged {lens[:4]}")


def test_maximum_batch(cuda_device):
    # 1024 requests (the kernel's limit): every CTA holds many whole pieces, and
    # empty rows, one-token rows and long rows mix
    lens = np.random.default_rng(17).choice([0, 1, 17, 300, 2000], size=1024)
    case = W.decode_case(17, lens, pending_append=True, poison=True)
    _check_case(case, cuda_device, what="batch 1024")


def test_graph_bucket_padding_rows_are_zero(cuda_device):
    lens = [700, 0, 33, 0, 0, 1, 2900, 0]
    case = W.decode_case(7, lens, pending_append=True, poison=True)
    run = DecodeOnDevice(case, 0, cuda_device)
    run.out.fill_(7.0)
    out = run.step()
    torch.cuda.synchronize()
    for b, n in enumerate(lens):
        if n == 0:
            assert torch.count_nonzero(out[b]).item() == 0
    kp, vp = _oracle_after_append(case, 0, run)
    want = oracle.decode(case.q[0], kp, vp, case.block_table, case.seq_lens, case.geom.scale)
    assert_close(bf16_to_f64(out), want, "padded bucket")


def test_all_rows_empty(cuda_device):
    case = W.decode_case(8, [0, 0, 0, 0], pending_append=False, poison=True)
    run = DecodeOnDevice(case, 0, cuda_device)
    run.out.fill_(1.0)
    out = run.step()
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0
    assert run.ws.status() == 0


def test_single_cached_token_is_exact(cuda_device):
    # softmax over one key is 1; 1 * v is exact in fp32 and rounds back to the same bf16
    case = W.decode_case(9, [1] * 16, pending_append=False, poison=True)
    run = DecodeOnDevice(case, 0, cuda_device)
    out = run.step().cpu()
    for b in range(16):
        page = case.block_table[b, 0]
        for h in range(16):
            assert torch.equal(out[b, h].view(torch.int16), case.v_pages[0, page, h // 2, 0].view(torch.int16))


def test_page_placement_gives_identical_bits(cuda_device):
    case = W.decode_case(10, W.config_seq_lens(2), pending_append=False, poison=True)
    out1 = DecodeOnDevice(case, 0, cuda_device).step().clone()
    rng = np.random.default_rng(1234)
    perm = rng.permutation(case.num_pages)
    kp2 = torch.empty_like(case.k_pages)
    vp2 = torch.empty_like(case.v_pages)
    kp2[:, perm] = case.k_pages
    vp2[:, perm] = case.v_pages
    case.k_pages, case.v_pages = kp2, vp2
    case.block_table = perm[case.block_table].astype(np.int32)
    out2 = DecodeOnDevice(case, 0, cuda_device).step()
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_peaked_scores(cuda_device):
    # one key per (request, KV head) made a large multiple of the query: the softmax is
    # nearly one-hot, so a wrong page, slot or head shows up as an O(1) error
    case = W.decode_case(11, [300, 1234, 2900, 45], pending_append=False, poison=True)
    rng = np.random.default_rng(5)
    for b, n in enumerate(case.seq_lens):
        for g in range(8):
            j = int(rng.integers(0, n))
            page, slot = case.block_table[b, j // 16], j % 16
            case.k_pages[0, page, g, slot] = (case.q[0, b, 2 * g].float() * 0.5).to(torch.bfloat16)
    run = DecodeOnDevice(case, 0, cuda_device)
    out = run.step()
    torch.cuda.synchronize()
    want = oracle.decode(case.q[0], case.k_pages[0], case.v_pages[0], case.block_table, case.seq_lens,
                         case.geom.scale)
    assert_close(bf16_to_f64(out), want, "peaked")


def test_cuda_graph_replay_matches_eager(cuda_device):
    case = W.decode_case(12, W.config_seq_lens(2), layers=2, pending_append=False, poison=True)
    runs = [DecodeOnDevice(case, layer, cuda_device) for layer in range(2)]
    eager = [r.step().clone() for r in runs]
    for r in runs:
        r.out.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for r in runs:  # warm-up on the capture stream
            r.step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for r in runs:
            r.step()
    for r in runs:
        r.out.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for r, e in zip(runs, eager):
        assert torch.equal(r.out.view(torch.int16), e.view(torch.int16))
        assert r.ws.status() == 0


def _split_scratch(ws, batch):
    """(counters, tagged records) views of a decode workspace. Layout: status
    header, int32 counters [batch][8] padded to 256 B, fp32 records, tagged
    records; each record area holds two 1056-byte records per CTA of the grid
    (two CTAs per SM)."""
    sms = torch.cuda.get_device_properties(ws.tensor.device).multi_processor_count
    slots = 2 * min(2 * sms, 2048)
    cnt_bytes = (batch * 8 * 4 + 255) // 256 * 256
    off = pkv.PKV_STATUS_BYTES
    counters = ws.tensor[off:off + cnt_bytes]
    tagged = ws.tensor[off + cnt_bytes + slots * 1056:off + cnt_bytes + 2 * slots * 1056]
    assert off + cnt_bytes + 2 * slots * 1056 == ws.nbytes
    return counters, tagged


@pytest.mark.parametrize("lens", [[40000], "bs16", [1, 17, 0, 33, 250, 4095, 16, 15, 3000, 2]])
def test_repeated_calls_reuse_the_workspace(cuda_device, lens):
    # the split counters return to zero and the merging CTAs clear every tagged
    # record they read, so a second call on the same workspace gives the same bits
    lens = W.config_seq_lens(2) if lens == "bs16" else lens
    case = W.decode_case(13, lens, pending_append=False, poison=True)
    run = DecodeOnDevice(case, 0, cuda_device)
    a = run.step().clone()
    torch.cuda.synchronize()
    counters, tagged = _split_scratch(run.ws, case.batch)
    assert torch.count_nonzero(counters).item() == 0 and torch.count_nonzero(tagged).item() == 0
    b = run.step().clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.count_nonzero(counters).item() == 0 and torch.count_nonzero(tagged).item() == 0
    assert run.ws.status() == 0


def test_page_id_outside_pool_is_reported_not_read(cuda_device):
    case = W.decode_case(14, [100, 200], pending_append=False, poison=True)
    case.block_table[1, 3] = case.num_pages + 1000
    run = DecodeOnDevice(case, 0, cuda_device)
    run.step()
    torch.cuda.synchronize()
    assert run.ws.status() == -7


def test_length_beyond_table_is_clamped_and_reported(cuda_device):
    case = W.decode_case(15, [100, 200], pending_append=False, poison=False)
    ensure_built()
    run = DecodeOnDevice(case, 0, cuda_device)
    run.seq_lens = i32([100, case.max_pages * 16 + 50], cuda_device)
    run.step()
    torch.cuda.synchronize()
    assert run.ws.status() == -7


def test_workspace_too_small_is_rejected(cuda_device):
    case = W.decode_case(16, [100, 200], pending_append=False)
    run = DecodeOnDevice(case, 0, cuda_device)
    run.ws = pkv.Workspace(512, cuda_device)
    with pytest.raises(pkv.PkvError) as e:
        run.step()
    assert e.value.code == -4


# ---------------------------------------------------------------------------- fused append + decode

def _fused(case, layer, dev):
    run = DecodeOnDevice(case, layer, dev)
    pkv.decode_append_attn(run.q, run.k_new, run.v_new, run.k_pages, run.v_pages, run.block_table, run.seq_lens,
                           run.out, case.geom.scale, run.ws)
    torch.cuda.synchronize()
    return run


@pytest.mark.parametrize("cfg", ["tiny", "bs16", "40k", "cfg", "ragged", "padded"])
def test_fused_append_decode_matches_oracle(cuda_device, cfg):
    lens = {"tiny": W.config_seq_lens(1), "bs16": W.config_seq_lens(2), "40k": W.config_seq_lens(3),
            "cfg": W.config_seq_lens(5), "ragged": [1, 15, 16, 17, 32, 33, 1000],
            "padded": [700, 0, 33, 0, 1, 2900]}[cfg]
    case = W.decode_case(17, lens, pending_append=True, poison=True)
    run = _fused(case, 0, cuda_device)
    # the pools equal the oracle's slot scatter: new rows written, every other slot untouched
    want_k, want_v = oracle.append(case.k_new[0], case.v_new[0], case.slot_mapping, case.k_pages[0], case.v_pages[0])
    assert np.array_equal(bits(run.k_pages), want_k) and np.array_equal(bits(run.v_pages), want_v)
    want = oracle.decode(case.q[0], want_k, want_v, case.block_table, case.seq_lens, case.geom.scale)
    assert_close(bf16_to_f64(run.out), want, f"fused {cfg}")
    for b, n in enumerate(case.seq_lens):
        if n == 0:
            assert torch.count_nonzero(run.out[b]).item() == 0
    assert run.ws.status() == 0


def test_fused_equals_separate_calls_bitwise(cuda_device):
    case = W.decode_case(18, W.config_seq_lens(2), pending_append=True, poison=True)
    sep = DecodeOnDevice(case, 0, cuda_device)
    out_sep = sep.step().clone()
    fused = _fused(case, 0, cuda_device)
    assert torch.equal(out_sep.view(torch.int16), fused.out.view(torch.int16))
    assert torch.equal(sep.k_pages.view(torch.int16), fused.k_pages.view(torch.int16))


@pytest.mark.parametrize("early,rope,cfg", [(False, False, "bs16"), (True, False, "bs16"), (True, True, "bs16"),
                                             (True, True, "40k")])
def test_fused_layer_chain_in_a_graph(cuda_device, early, rope, cfg):
    # two layers, each its own pool, replayed from a CUDA graph; with early prefetch each
    # layer's kernel may start reading its pool while the previous layer's kernel finishes (with the
    # rotary embedding, the pages before a chunk's first new row before the predecessor completes)
    lens = {"bs16": W.config_seq_lens(2), "40k": W.config_seq_lens(3)}[cfg]
    case = W.decode_case(19, lens, layers=2, pending_append=True, poison=True)
    runs = [DecodeOnDevice(case, layer, cuda_device) for layer in range(2)]
    cs = oracle.rope_cache(ROPE_THETA, case.geom.head_dim, int(max(lens)) + 1) if rope else None
    cs_dev = torch.from_numpy(cs).to(cuda_device) if rope else None

    def step():
        for r in runs:
            if rope:
                pkv.decode_append_rope_attn(r.q, r.k_new, r.v_new, r.k_pages, r.v_pages, r.block_table, r.seq_lens,
                                            cs_dev, r.out, case.geom.scale, r.ws, early_prefetch=early)
            else:
                pkv.decode_append_attn(r.q, r.k_new, r.v_new, r.k_pages, r.v_pages, r.block_table, r.seq_lens,
                                       r.out, case.geom.scale, r.ws, early_prefetch=early)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for r in runs:
        r.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    pos = np.asarray(case.seq_lens, dtype=np.int64) - 1
    for layer, r in enumerate(runs):
        k_new = oracle.rope_bf16(case.k_new[layer], pos, cs) if rope else case.k_new[layer]
        want_k, want_v = oracle.append(k_new, case.v_new[layer], case.slot_mapping, case.k_pages[layer],
                                       case.v_pages[layer])
        assert np.array_equal(bits(r.k_pages), want_k) and np.array_equal(bits(r.v_pages), want_v)
        q = oracle.rope_f64(case.q[layer], pos, cs) if rope else case.q[layer]
        want = oracle.decode(q, want_k, want_v, case.block_table, case.seq_lens, case.geom.scale)
        assert_close(bf16_to_f64(r.out), want, f"graph layer {layer} early={early} rope={rope} {cfg}")
        assert r.ws.status() == 0


def test_fused_rejects_unknown_flags(cuda_device):
    case = W.decode_case(20, [40, 50], pending_append=True)
    run = DecodeOnDevice(case, 0, cuda_device)
    from paged_kv_decode_gb300 import _lib
    import ctypes
    d = pkv.desc(case.num_pages)
    rc = _lib.load().pkv_decode_append_attn(run.q.data_ptr(), run.k_new.data_ptr(), run.v_new.data_ptr(),
                                            run.k_pages.data_ptr(), run.v_pages.data_ptr(), run.block_table.data_ptr(),
                                            run.seq_lens.data_ptr(), run.out.data_ptr(), 1.0, None, ctypes.byref(d),
                                            2, case.max_pages, run.ws.tensor.data_ptr(), run.ws.nbytes, 6)
    assert rc == -3


# ---------------------------------------------------------------------------- fused rotary embedding

ROPE_THETA = 1e6  # "Fun-ASR-Nano Native Runtime Design", section "Decoder And Prompt"


@pytest.mark.parametrize("cfg", ["tiny", "bs16", "40k", "ragged", "padded"])
def test_fused_rope_append_decode_matches_oracle(cuda_device, cfg):
    lens = {"tiny": W.config_seq_lens(1), "bs16": W.config_seq_lens(2), "40k": W.config_seq_lens(3),
            "ragged": [1, 15, 16, 17, 32, 33, 1000], "padded": [700, 0, 33, 0, 1, 2900]}[cfg]
    case = W.decode_case(19, lens, pending_append=True, poison=True)
    cs = oracle.rope_cache(ROPE_THETA, case.geom.head_dim, int(max(lens)) + 3)
    run = DecodeOnDevice(case, 0, cuda_device)
    pkv.decode_append_rope_attn(run.q, run.k_new, run.v_new, run.k_pages, run.v_pages, run.block_table,
                                run.seq_lens, torch.from_numpy(cs).to(cuda_device), run.out, case.geom.scale, run.ws)
    torch.cuda.synchronize()
    pos = np.asarray(case.seq_lens, dtype=np.int64) - 1  # -1 for empty requests: nothing appended
    k_rot = oracle.rope_bf16(case.k_new[0], pos, cs)
    want_k, want_v = oracle.append(k_rot, case.v_new[0], case.slot_mapping, case.k_pages[0], case.v_pages[0])
    # the rotated key rows land bit-exactly; every other slot is untouched
    assert np.array_equal(bits(run.k_pages), want_k) and np.array_equal(bits(run.v_pages), want_v)
    want = oracle.decode(oracle.rope_f64(case.q[0], pos, cs), want_k, want_v, case.block_table, case.seq_lens,
                         case.geom.scale)
    assert_close(bf16_to_f64(run.out), want, f"rope {cfg}")
    for b, n in enumerate(case.seq_lens):
        if n == 0:
            assert torch.count_nonzero(run.out[b]).item() == 0
    assert run.ws.status() == 0


@pytest.mark.parametrize("head_dim", [128, 64])
def test_library_rope_table_matches_the_oracle_table(cuda_device, head_dim):
    # pkv_rope_table (the device kernel, double angles rounded to float) and the oracle's C table
    # follow the same definition independently: within one float ulp, nearly all equal
    a = pkv.rope_cos_sin(ROPE_THETA, 50000, head_dim, device=cuda_device).cpu().numpy()
    b = oracle.rope_cache(ROPE_THETA, head_dim, 50000)
    assert a.shape == b.shape == (50000, head_dim)
    ulp = np.spacing(np.abs(b).astype(np.float32))
    assert (np.abs(a.astype(np.float64) - b.astype(np.float64)) <= ulp).all()
    assert (a == b).mean() > 0.999


def test_fused_rope_position_beyond_table_is_reported(cuda_device):
    case = W.decode_case(20, [300, 40], pending_append=True, poison=False)
    cs = oracle.rope_cache(ROPE_THETA, case.geom.head_dim, 100)  # 300 - 1 is past the last row
    run = DecodeOnDevice(case, 0, cuda_device)
    pkv.decode_append_rope_attn(run.q, run.k_new, run.v_new, run.k_pages, run.v_pages, run.block_table,
                                run.seq_lens, torch.from_numpy(cs).to(cuda_device), run.out, case.geom.scale, run.ws)
    torch.cuda.synchronize()
    assert run.ws.status() == -7  # PKV_ERR_OUT_OF_BOUNDS
