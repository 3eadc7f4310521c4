"""Pins for the fp64 oracle (CPU only).

Each test ties the oracle to something other than itself: torch's
scaled_dot_product_attention on a dense (unpaged) layout, closed forms,
invariants of softmax attention (identical keys, one key, zero scale, head
grouping, page placement, causality), and the definition of the slot scatter.
A plausible mistake anywhere in the oracle -- a wrong page or slot index, a
wrong KV-head map, a dropped or extra key, a missing scale, a top-left causal
mask -- fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from parity import stats, within
from paged_kv_decode_gb300 import workloads as W

G_SMALL = W.Geometry(n_q_heads=4, n_kv_heads=2, head_dim=8, page_size=4)


def _bf16(x) -> torch.Tensor:
    return torch.as_tensor(x, dtype=torch.float64).to(torch.bfloat16)


def _dense_to_paged(dense_k, dense_v, lens, page_size, rng, spare=0):
    """Scatter dense [B, T, Hkv, D] K/V into a permuted page pool, by the layout's definition."""
    B, T, Hkv, D = dense_k.shape
    need = [(-(-int(n) // page_size)) for n in lens]
    total = sum(need) + spare
    perm = rng.permutation(total)
    max_pages = max(1, max(need))
    bt = np.full((B, max_pages), total - 1 if spare else 0, dtype=np.int32)
    kp = torch.zeros((total, Hkv, page_size, D), dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    cur = 0
    for b in range(B):
        for p in range(need[b]):
            bt[b, p] = perm[cur]
            cur += 1
        for j in range(int(lens[b])):
            page, slot = bt[b, j // page_size], j % page_size
            kp[page, :, slot, :] = dense_k[b, j]
            vp[page, :, slot, :] = dense_v[b, j]
    return kp, vp, bt


def _sdpa_decode(q, dense_k, dense_v, lens, scale, group):
    """torch SDPA in fp64 on the dense layout, one query per request."""
    B, Hq, D = q.shape
    T = dense_k.shape[1]
    qd = q.to(torch.float64).reshape(B, Hq, 1, D)
    kd = dense_k.to(torch.float64).permute(0, 2, 1, 3).repeat_interleave(group, dim=1)
    vd = dense_v.to(torch.float64).permute(0, 2, 1, 3).repeat_interleave(group, dim=1)
    mask = torch.zeros((B, 1, 1, T), dtype=torch.bool)
    for b in range(B):
        mask[b, 0, 0, : int(lens[b])] = True
    out = F.scaled_dot_product_attention(qd, kd, vd, attn_mask=mask, scale=scale)
    return out.reshape(B, Hq, D).numpy()


@pytest.mark.parametrize("geom,lens", [(G_SMALL, [5, 37, 1, 16]), (W.QWEN3, [37, 200])])
def test_decode_matches_sdpa_on_dense_layout(geom, lens):
    rng = np.random.default_rng(11)
    gen = torch.Generator().manual_seed(11)
    B, T = len(lens), max(lens)
    dk = torch.randn((B, T, geom.n_kv_heads, geom.head_dim), generator=gen).to(torch.bfloat16)
    dv = torch.randn((B, T, geom.n_kv_heads, geom.head_dim), generator=gen).to(torch.bfloat16)
    q = torch.randn((B, geom.n_q_heads, geom.head_dim), generator=gen).to(torch.bfloat16)
    kp, vp, bt = _dense_to_paged(dk, dv, lens, geom.page_size, rng)
    got = oracle.decode(q, kp, vp, bt, np.array(lens, dtype=np.int32), geom.scale)
    want = _sdpa_decode(q, dk, dv, lens, geom.scale, geom.n_q_heads // geom.n_kv_heads)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_two_key_closed_form():
    # q = a * e0, k0 = e0, k1 = 0 -> s0 = scale * a, s1 = 0;
    # out = (e^{s0} v0 + v1) / (e^{s0} + 1) for every query head of the group.
    g = W.Geometry(n_q_heads=2, n_kv_heads=1, head_dim=4, page_size=2)
    a, scale = 3.0, 0.5
    q = torch.zeros((1, 2, 4))
    q[0, :, 0] = a
    kp = torch.zeros((1, 1, 2, 4))
    kp[0, 0, 0, 0] = 1.0
    vp = torch.tensor([[[[1.0, 2.0, -4.0, 0.5], [-3.0, 0.25, 8.0, 1.0]]]])
    got = oracle.decode(_bf16(q), _bf16(kp), _bf16(vp), np.array([[0]], np.int32), np.array([2], np.int32), scale)
    w0 = math.exp(scale * a) / (math.exp(scale * a) + 1.0)
    v0, v1 = vp[0, 0, 0].double().numpy(), vp[0, 0, 1].double().numpy()
    want = w0 * v0 + (1 - w0) * v1
    for h in range(2):
        np.testing.assert_allclose(got[0, h], want, rtol=0, atol=1e-15)


def test_identical_keys_give_mean_of_values():
    case = W.decode_case(3, [29, 64], geom=G_SMALL, pending_append=False, poison=True)
    kp = case.k_pages[0].clone()
    kp[:] = kp[0, 0, 0]  # every row the same key (poison rows too, they stay unread)
    out = oracle.decode(case.q[0], kp, case.v_pages[0], case.block_table, case.seq_lens, G_SMALL.scale)
    for b, n in enumerate(case.seq_lens):
        rows = []
        for j in range(int(n)):
            page, slot = case.block_table[b, j // 4], j % 4
            rows.append(case.v_pages[0, page, :, slot, :].double().numpy())
        mean = np.mean(np.stack(rows), axis=0)  # [Hkv, D]
        for h in range(G_SMALL.n_q_heads):
            np.testing.assert_allclose(out[b, h], mean[h // 2], rtol=0, atol=1e-12)


def test_zero_scale_gives_mean_of_values():
    case = W.decode_case(4, [13], geom=G_SMALL, pending_append=False)
    out = oracle.decode(case.q[0], case.k_pages[0], case.v_pages[0], case.block_table, case.seq_lens, 0.0)
    bt = case.block_table
    rows = np.stack([case.v_pages[0, bt[0, j // 4], :, j % 4].double().numpy() for j in range(13)])
    for h in range(4):
        np.testing.assert_allclose(out[0, h], rows.mean(axis=0)[h // 2], rtol=0, atol=1e-12)


def test_single_token_returns_its_value_row_exactly():
    case = W.decode_case(5, [1, 1, 17], geom=G_SMALL, pending_append=False)
    out = oracle.decode(case.q[0], case.k_pages[0], case.v_pages[0], case.block_table, case.seq_lens, G_SMALL.scale)
    for b in range(2):
        page = case.block_table[b, 0]
        for h in range(4):
            assert np.array_equal(out[b, h], case.v_pages[0, page, h // 2, 0].double().numpy())


def test_query_head_reads_kv_head_h_div_group():
    # V of KV head g is the constant g + 1, so out[h] == h // 2 + 1 exactly (h % 8 would fail).
    g = W.Geometry(n_q_heads=16, n_kv_heads=8, head_dim=8, page_size=4)
    case = W.decode_case(6, [23], geom=g, pending_append=False, poison=False)
    vp = case.v_pages[0].clone()
    for kv in range(8):
        vp[:, kv] = float(kv + 1)
    out = oracle.decode(case.q[0], case.k_pages[0], vp, case.block_table, case.seq_lens, g.scale)
    for h in range(16):
        np.testing.assert_allclose(out[0, h], h // 2 + 1, rtol=0, atol=1e-12)


def test_page_placement_does_not_change_output_bits():
    case = W.decode_case(7, [45, 3, 130], geom=G_SMALL, pending_append=False, poison=False)
    out1 = oracle.decode(case.q[0], case.k_pages[0], case.v_pages[0], case.block_table, case.seq_lens, G_SMALL.scale)
    rng = np.random.default_rng(99)
    perm = rng.permutation(case.num_pages)  # new physical id of each old page
    kp2 = torch.empty_like(case.k_pages[0])
    vp2 = torch.empty_like(case.v_pages[0])
    kp2[perm] = case.k_pages[0]
    vp2[perm] = case.v_pages[0]
    bt2 = perm[case.block_table].astype(np.int32)
    out2 = oracle.decode(case.q[0], kp2, vp2, bt2, case.seq_lens, G_SMALL.scale)
    assert np.array_equal(out1, out2)


def test_peaked_query_selects_the_addressed_position():
    # Make key j* = 40 * q (per KV head); softmax is then one-hot at j* to within e^-... and
    # out ~= v_{j*}: the position -> (page, slot) map must find j*'s row.
    g = W.Geometry(n_q_heads=2, n_kv_heads=1, head_dim=16, page_size=4)
    case = W.decode_case(8, [37], geom=g, pending_append=False, poison=False)
    jstar = 22
    kp = case.k_pages[0].clone()
    page, slot = case.block_table[0, jstar // 4], jstar % 4
    q = case.q[0].clone()
    q[0, 1] = q[0, 0]
    kp[page, 0, slot] = (q[0, 0].float() * 2.0).to(torch.bfloat16)
    out = oracle.decode(q, kp, case.v_pages[0], case.block_table, case.seq_lens, 1.0)
    want = case.v_pages[0, page, 0, slot].double().numpy()
    np.testing.assert_allclose(out[0, 0], want, rtol=0, atol=1e-6)


def test_unread_slots_may_hold_nan_and_empty_rows_give_zeros():
    case = W.decode_case(9, [0, 17, 5], geom=G_SMALL, pending_append=False, poison=True)
    out = oracle.decode(case.q[0], case.k_pages[0], case.v_pages[0], case.block_table, case.seq_lens, G_SMALL.scale)
    assert np.isfinite(out).all()
    assert np.array_equal(out[0], np.zeros_like(out[0]))


def test_out_of_range_page_is_an_error():
    case = W.decode_case(10, [9], geom=G_SMALL, pending_append=False)
    bt = case.block_table.copy()
    bt[0, 1] = case.num_pages + 5
    with pytest.raises(ValueError):
        oracle.decode(case.q[0], case.k_pages[0], case.v_pages[0], bt, case.seq_lens, 1.0)


# ---------------------------------------------------------------------------- prefill

def _sdpa_prefill(q, dense_k, dense_v, prefix, scale, group):
    """torch SDPA in fp64 with an explicit bottom-right causal mask (row i sees keys <= prefix + i)."""
    Lq, Hq, D = q.shape
    T = dense_k.shape[0]
    qd = q.to(torch.float64).permute(1, 0, 2).unsqueeze(0)
    kd = dense_k.to(torch.float64).permute(1, 0, 2).repeat_interleave(group, dim=0).unsqueeze(0)
    vd = dense_v.to(torch.float64).permute(1, 0, 2).repeat_interleave(group, dim=0).unsqueeze(0)
    i = torch.arange(Lq).unsqueeze(1)
    j = torch.arange(T).unsqueeze(0)
    mask = (j <= prefix + i).reshape(1, 1, Lq, T)
    out = F.scaled_dot_product_attention(qd, kd, vd, attn_mask=mask, scale=scale)
    return out.squeeze(0).permute(1, 0, 2).numpy()


@pytest.mark.parametrize("prefix,qlen", [(0, 21), (19, 13), (64, 1)])
def test_prefill_matches_sdpa_with_bottom_right_mask(prefix, qlen):
    g = G_SMALL
    rng = np.random.default_rng(21)
    gen = torch.Generator().manual_seed(21)
    T = prefix + qlen
    dk = torch.randn((1, T, g.n_kv_heads, g.head_dim), generator=gen).to(torch.bfloat16)
    dv = torch.randn((1, T, g.n_kv_heads, g.head_dim), generator=gen).to(torch.bfloat16)
    q = torch.randn((qlen, g.n_q_heads, g.head_dim), generator=gen).to(torch.bfloat16)
    kp, vp, bt = _dense_to_paged(dk, dv, [T], g.page_size, rng)
    got = oracle.prefill(q, kp, vp, bt, np.array([prefix], np.int32), np.array([0, qlen], np.int32), g.scale)
    want = _sdpa_prefill(q, dk[0], dv[0], prefix, g.scale, 2)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_prefill_two_requests_and_row_sampling():
    case = W.prefill_case(22, [8, 0], [7, 5], geom=G_SMALL, poison=True)
    kp, vp = oracle.append(case.k_new[0], case.v_new[0], case.slot_mapping, case.k_pages[0], case.v_pages[0])
    full = oracle.prefill(case.q[0], kp, vp, case.block_table, case.prefix_lens, case.cu_q_lens, G_SMALL.scale)
    assert np.isfinite(full).all()
    rows = [11, 0, 6, 7]
    part = oracle.prefill(case.q[0], kp, vp, case.block_table, case.prefix_lens, case.cu_q_lens, G_SMALL.scale,
                          rows=rows)
    assert np.array_equal(part, full[rows])


def test_prefill_row_equals_decode_over_its_visible_prefix():
    case = W.prefill_case(23, [11], [9], geom=G_SMALL, poison=True)
    kp, vp = oracle.append(case.k_new[0], case.v_new[0], case.slot_mapping, case.k_pages[0], case.v_pages[0])
    pre = oracle.prefill(case.q[0], kp, vp, case.block_table, case.prefix_lens, case.cu_q_lens, G_SMALL.scale)
    for i in range(9):
        dec = oracle.decode(case.q[0][i:i + 1], kp, vp, case.block_table, np.array([11 + i + 1], np.int32),
                            G_SMALL.scale)
        assert np.array_equal(dec[0], pre[i])


def test_prefill_causality():
    case = W.prefill_case(24, [6], [10], geom=G_SMALL, poison=False)
    kp, vp = oracle.append(case.k_new[0], case.v_new[0], case.slot_mapping, case.k_pages[0], case.v_pages[0])
    base = oracle.prefill(case.q[0], kp, vp, case.block_table, case.prefix_lens, case.cu_q_lens, G_SMALL.scale)
    i0 = 4  # perturb every key/value after absolute position 6 + 4
    kp2, vp2 = kp.copy(), vp.copy()
    for j in range(6 + i0 + 1, 16):
        page, slot = case.block_table[0, j // 4], j % 4
        kp2[page, :, slot, :] ^= 0x0100
        vp2[page, :, slot, :] ^= 0x0100
    pert = oracle.prefill(case.q[0], kp2, vp2, case.block_table, case.prefix_lens, case.cu_q_lens, G_SMALL.scale)
    assert np.array_equal(pert[: i0 + 1], base[: i0 + 1])
    assert not np.array_equal(pert[i0 + 1:], base[i0 + 1:])


# ---------------------------------------------------------------------------- append

def test_append_scatter_definition():
    case = W.decode_case(30, [5, 16, 33, 0], geom=G_SMALL, pending_append=True, poison=True)
    kp0 = case.k_pages[0].contiguous().view(torch.int16).numpy().view(np.uint16)
    kp, vp = oracle.append(case.k_new[0], case.v_new[0], case.slot_mapping, case.k_pages[0], case.v_pages[0])
    kn = case.k_new[0].contiguous().view(torch.int16).numpy().view(np.uint16)
    vn = case.v_new[0].contiguous().view(torch.int16).numpy().view(np.uint16)
    touched = np.zeros(kp.shape[:1] + kp.shape[2:3], dtype=bool)  # [page, slot]
    for b, n in enumerate(case.seq_lens):
        if n == 0:
            assert case.slot_mapping[b] == -1
            continue
        j = int(n) - 1  # the appended token is the last visible position
        page, slot = case.block_table[b, j // 4], j % 4
        assert np.array_equal(kp[page, :, slot], kn[b]) and np.array_equal(vp[page, :, slot], vn[b])
        touched[page, slot] = True
    mask = ~touched
    kp_m = np.transpose(kp, (0, 2, 1, 3))[mask]
    kp0_m = np.transpose(kp0, (0, 2, 1, 3))[mask]
    assert np.array_equal(kp_m, kp0_m)


def test_append_out_of_range_slot_is_an_error():
    case = W.decode_case(31, [5], geom=G_SMALL)
    sm = np.array([case.num_pages * 4 + 1], np.int32)
    with pytest.raises(ValueError):
        oracle.append(case.k_new[0], case.v_new[0], sm, case.k_pages[0], case.v_pages[0])


# ---------------------------------------------------------------------------- tolerance teeth

def test_tolerance_rejects_a_dropped_page_and_a_wrong_head_map():
    """Plant mistakes on the oracle side (CPU) and check the parity bar catches them."""
    case = W.decode_case(40, [600, 1200], pending_append=False, poison=False)
    g = W.QWEN3
    args = (case.k_pages[0], case.v_pages[0])
    want = oracle.decode(case.q[0], *args, case.block_table, case.seq_lens, g.scale)
    # (a) one page of request 1 read from the wrong physical page
    bt = case.block_table.copy()
    bt[1, 30] = bt[0, 3]
    dropped = oracle.decode(case.q[0], *args, bt, case.seq_lens, g.scale)
    # (b) query heads mapped h % 8 instead of h // 2
    # place query head h where the correct map sends it to KV head h % 8, then read it back
    slot_of = [2 * (h % 8) + h // 8 for h in range(16)]
    q2 = torch.empty_like(case.q[0])
    q2[:, slot_of] = case.q[0]
    swapped = oracle.decode(q2, *args, case.block_table, case.seq_lens, g.scale)[:, slot_of]
    # (c) a page dropped from the context entirely
    short = oracle.decode(case.q[0], *args, case.block_table, case.seq_lens - 16, g.scale)
    for bad in (dropped, swapped, short):
        assert not within(stats(bad, want))
    assert within(stats(want, want))


@pytest.mark.parametrize("base,peak", [(0.0, 8.0), (-10.0, -9.0)])
def test_huge_scores_do_not_overflow_or_underflow(base, peak):
    # Scores of order +-800: exp() of the raw scores overflows (or underflows to 0) in
    # double, so only a max-shifted softmax gives the right answer, here the value row
    # of the last position, which holds the largest score.
    g = W.Geometry(n_q_heads=2, n_kv_heads=1, head_dim=4, page_size=4)
    case = W.decode_case(12, [7], geom=g, pending_append=False, poison=False)
    q = torch.zeros((1, 2, 4))
    q[0, :, 0] = 100.0
    kp = case.k_pages[0].float().clone()
    bt = case.block_table
    for j in range(7):
        kp[bt[0, j // 4], 0, j % 4] = 0.0
        kp[bt[0, j // 4], 0, j % 4, 0] = peak if j == 6 else base
    out = oracle.decode(_bf16(q), kp.to(torch.bfloat16), case.v_pages[0], bt, case.seq_lens, 1.0)
    want = case.v_pages[0, bt[0, 1], 0, 6 % 4].double().numpy()
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out[0, 0], want, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------- rotary position embedding
# RoPE with theta 1e6 ("Fun-ASR-Nano Native Runtime Design", section "Decoder And Prompt"),
# rotate-half pairs (i, i + 64) of a 128-dim head.

THETA = 1e6


def _rope_ref_pair(x1, x2, ang):
    return x1 * math.cos(ang) - x2 * math.sin(ang), x2 * math.cos(ang) + x1 * math.sin(ang)


def test_rope_cache_row0_and_angle_addition():
    cs = oracle.rope_cache(THETA, 128, 64).astype(np.float64)
    assert np.array_equal(cs[0, :64], np.ones(64)) and np.array_equal(cs[0, 64:], np.zeros(64))
    # angles grow linearly with the position: cos((p+1)w) = cos(pw)cos(w) - sin(pw)sin(w), and the
    # same for sin, for every frequency (float rounding of the table only)
    c, s = cs[:, :64], cs[:, 64:]
    c1, s1 = c[1], s[1]
    assert np.abs(c[1:] - (c[:-1] * c1 - s[:-1] * s1)).max() < 3e-7 * 64
    assert np.abs(s[1:] - (s[:-1] * c1 + c[:-1] * s1)).max() < 3e-7 * 64
    assert np.abs(c ** 2 + s ** 2 - 1).max() < 2e-7


def test_rope_cache_frequencies_follow_theta():
    cs = oracle.rope_cache(THETA, 128, 2).astype(np.float64)
    w = np.arcsin(np.clip(cs[1, 64:], -1, 1))  # sin(w_i) at position 1; w_0 = 1 < pi/2
    assert abs(w[0] - 1.0) < 1e-7  # w_0 = theta^0
    # w_i = theta^(-2i/128): log-linear in i with slope -2 ln(theta) / 128
    slope = np.polyfit(np.arange(1, 64), np.log(w[1:]), 1)[0]
    assert abs(slope - (-2 * math.log(THETA) / 128)) < 1e-6
    assert abs(w[63] / THETA ** (-126 / 128) - 1) < 1e-5


def test_rope_unit_vectors_pin_pairing_and_direction():
    cs = oracle.rope_cache(THETA, 128, 8)
    x = np.zeros((4, 1, 128), dtype=np.float32)
    x[0, 0, 0] = 1.0   # e_0 at position 5 -> cos(5) e_0 + sin(5) e_64
    x[1, 0, 64] = 1.0  # e_64 at position 5 -> -sin(5) e_0 + cos(5) e_64
    x[2, 0, 1] = 1.0   # e_1 pairs with e_65, frequency w_1
    x[3, 0, 7] = 1.0   # position -1: unrotated
    xb = torch.from_numpy(x).to(torch.bfloat16)
    y = oracle.rope_f64(xb, [5, 5, 3, -1], cs)
    c5, s5 = float(cs[5, 0]), float(cs[5, 64])
    assert abs(c5 - math.cos(5)) < 1e-7 and abs(s5 - math.sin(5)) < 1e-7
    want = np.zeros((4, 1, 128))
    want[0, 0, 0], want[0, 0, 64] = c5, s5
    want[1, 0, 0], want[1, 0, 64] = -s5, c5
    want[2, 0, 1], want[2, 0, 65] = float(cs[3, 1]), float(cs[3, 65])
    want[3, 0, 7] = 1.0
    assert np.array_equal(y, want)
    w1 = THETA ** (-2 / 128)
    assert abs(float(cs[3, 1]) - math.cos(3 * w1)) < 1e-7 and abs(float(cs[3, 65]) - math.sin(3 * w1)) < 1e-7


def test_rope_position0_identity_and_pair_norms():
    cs = oracle.rope_cache(THETA, 128, 50000)
    g = torch.Generator().manual_seed(7)
    x = torch.randn(6, 4, 128, generator=g).to(torch.bfloat16)
    pos = [0, 1, 17, 4095, 40000, 49999]
    y = oracle.rope_f64(x, pos, cs)
    xf = x.to(torch.float64).numpy()
    assert np.array_equal(y[0], xf[0])
    n_in = xf[..., :64] ** 2 + xf[..., 64:] ** 2
    n_out = y[..., :64] ** 2 + y[..., 64:] ** 2
    assert np.abs(n_out - n_in).max() <= 1e-6 * n_in.max()
    # bf16 form: position 0 returns the input bits
    assert np.array_equal(oracle.rope_bf16(x, [0] * 6, cs), x.view(torch.int16).numpy().view(np.uint16))


def test_rope_scores_depend_on_relative_position_only():
    # <R(m) q, R(n) k> = <R(m - n) q, k>: with a table built here in double from the definition,
    # the oracle's rotation reproduces it to float-table rounding
    d = 128
    w = THETA ** (-2 * np.arange(64) / d)
    pos_max = 3000
    ang = np.arange(pos_max)[:, None] * w[None, :]
    cs = np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)
    g = torch.Generator().manual_seed(8)
    q = torch.randn(1, 1, d, generator=g).to(torch.bfloat16)
    k = torch.randn(1, 1, d, generator=g).to(torch.bfloat16)
    for m, n in [(2900, 2000), (1234, 5), (77, 77)]:
        lhs = float(np.dot(oracle.rope_f64(q, [m], cs).ravel(), oracle.rope_f64(k, [n], cs).ravel()))
        rhs = float(np.dot(oracle.rope_f64(q, [m - n], cs).ravel(), k.to(torch.float64).numpy().ravel()))
        assert abs(lhs - rhs) < 1e-4 * (1 + abs(rhs)), (m, n, lhs, rhs)


def test_rope_bf16_is_a_neighbour_of_the_exact_rotation():
    cs = oracle.rope_cache(THETA, 128, 41000)
    g = torch.Generator().manual_seed(9)
    x = (torch.randn(64, 8, 128, generator=g) * 3).to(torch.bfloat16)
    pos = np.random.default_rng(9).integers(0, 41000, 64).astype(np.int32)
    exact = oracle.rope_f64(x, pos, cs)
    got = torch.from_numpy(oracle.rope_bf16(x, pos, cs).view(np.int16)).view(torch.bfloat16).double().numpy()
    # bf16 keeps 8 significant bits: |got - exact| within one step of the bf16 grid at exact's magnitude
    step = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(exact), 1e-30))) - 7)
    assert (np.abs(got - exact) <= step * 1.0001).all()
    # and mostly the nearest value
    nearest = torch.from_numpy(exact).to(torch.bfloat16).double().numpy()
    assert (got == nearest).mean() > 0.99


def test_decode_with_float64_queries_matches_bf16_queries():
    case = W.decode_case(11, [37, 200], pending_append=False, poison=False)
    q = case.q[0]
    a = oracle.decode(q, case.k_pages[0], case.v_pages[0], case.block_table, case.seq_lens, case.geom.scale)
    b = oracle.decode(q.to(torch.float64).numpy(), case.k_pages[0], case.v_pages[0], case.block_table,
                      case.seq_lens, case.geom.scale)
    assert np.isfinite(a).all() and np.array_equal(a, b)
