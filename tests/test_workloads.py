"""The seeded generators: shapes, determinism, page placement and poison (CPU only)."""
import json
import os

import numpy as np
import torch

from paged_kv_decode_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_geometry_matches_the_pages():
    g = json.load(open(os.path.join(GOLDEN, "qwen3_decoder.json")))
    assert (W.N_Q_HEADS, W.N_KV_HEADS, W.N_LAYERS) == (g["n_q_heads"], g["n_kv_heads"], g["n_layers"])
    s = json.load(open(os.path.join(GOLDEN, "serving_shapes.json")))
    assert W.PREFILL_CHUNK == s["chunked_prefill"]["chunk_tokens"]
    assert len(W.config_seq_lens(2)) == s["benchmark_setup"]["max_running_requests"]


def test_config_lengths_in_range_and_seeded():
    a, b = W.config_seq_lens(2), W.config_seq_lens(2)
    assert np.array_equal(a, b) and a.min() >= 300 and a.max() <= 3000 and len(a) == 16
    c = W.config_seq_lens(5)
    assert len(c) == 32 and c[0::2].min() >= 1000 and c[0::2].max() <= 8000
    assert c[1::2].min() >= 8 + 16 and c[1::2].max() <= 64 + 512
    d = W.mixed_decode_lens()
    assert len(d) == 15 and d.min() >= 500 and d.max() <= 5000
    assert list(W.config_seq_lens(1)) == [37, 200]
    assert list(W.config_seq_lens(3, context=65536)) == [65536]


def test_block_table_is_a_placement_of_distinct_pages():
    rng = np.random.default_rng(0)
    lens = np.array([37, 200, 16, 0])
    bt, num_pages, poison = W.place_pages(rng, lens, 16)
    need = (lens + 15) // 16
    used = np.concatenate([bt[b, :n] for b, n in enumerate(need)])
    assert len(np.unique(used)) == len(used) == need.sum()
    assert used.max() < poison == num_pages - 1
    for b, n in enumerate(need):
        assert (bt[b, n:] == poison).all()


def test_decode_case_poison_and_determinism():
    g = W.Geometry(4, 2, 8, 4)
    c1 = W.decode_case(5, [6, 9], geom=g, pending_append=True, poison=True)
    c2 = W.decode_case(5, [6, 9], geom=g, pending_append=True, poison=True)
    assert torch.equal(c1.k_pages.view(torch.int16), c2.k_pages.view(torch.int16))
    kp = c1.k_pages[0].float()
    for b, n in enumerate(c1.seq_lens):
        for j in range(int(n) - 1):
            assert torch.isfinite(kp[c1.block_table[b, j // 4], :, j % 4]).all()
        # the pending slot and the tail are poison
        for j in range(int(n) - 1, ((int(n) + 3) // 4) * 4):
            assert torch.isnan(kp[c1.block_table[b, j // 4], :, j % 4]).all()
        page, slot = c1.block_table[b, (n - 1) // 4], (n - 1) % 4
        assert c1.slot_mapping[b] == page * 4 + slot
    assert torch.isnan(kp[c1.poison_page]).all()


