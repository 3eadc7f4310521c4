"""KV append on the GPU: bit-exact against the oracle's slot scatter."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_gb300 as pkv
from gpu_util import bits, ensure_built, i32
from paged_kv_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run_append(k_new, v_new, slots, kp, vp, dev):
    ensure_built()
    kd, vd = kp.to(dev), vp.to(dev)
    ws = pkv.Workspace(pkv.PKV_STATUS_BYTES, dev)
    pkv.append(k_new.to(dev), v_new.to(dev), i32(slots, dev), kd, vd, ws)
    torch.cuda.synchronize()
    return kd, vd, ws


@pytest.mark.parametrize("lens", [W.config_seq_lens(2), W.config_seq_lens(5), [1, 0, 17, 33]])
def test_decode_step_append_bit_exact(cuda_device, lens):
    case = W.decode_case(101, lens, pending_append=True, poison=True)
    kd, vd, ws = _run_append(case.k_new[0], case.v_new[0], case.slot_mapping, case.k_pages[0], case.v_pages[0],
                             cuda_device)
    want_k, want_v = oracle.append(case.k_new[0], case.v_new[0], case.slot_mapping, case.k_pages[0], case.v_pages[0])
    assert np.array_equal(bits(kd), want_k)  # touched slots equal, untouched (NaN canaries) unchanged
    assert np.array_equal(bits(vd), want_v)
    assert ws.status() == 0


@pytest.mark.parametrize("prefix,qlen", [(0, 4096), (8192, 4096), (5, 37)])
def test_prefill_chunk_append_bit_exact(cuda_device, prefix, qlen):
    case = W.prefill_case(102, [prefix], [qlen], poison=True)
    kd, vd, ws = _run_append(case.k_new[0], case.v_new[0], case.slot_mapping, case.k_pages[0], case.v_pages[0],
                             cuda_device)
    want_k, want_v = oracle.append(case.k_new[0], case.v_new[0], case.slot_mapping, case.k_pages[0], case.v_pages[0])
    assert np.array_equal(bits(kd), want_k) and np.array_equal(bits(vd), want_v)
    assert ws.status() == 0


def test_negative_slots_skip_and_bad_slot_reports(cuda_device):
    case = W.decode_case(103, [40, 41, 42, 43], pending_append=True, poison=True)
    slots = case.slot_mapping.copy()
    slots[1] = -1
    bad = slots.copy()
    bad[2] = case.num_pages * 16 + 3  # past the pool: skipped, reported
    kd, vd, ws = _run_append(case.k_new[0], case.v_new[0], bad, case.k_pages[0], case.v_pages[0], cuda_device)
    keep = slots.copy()
    keep[2] = -1
    want_k, want_v = oracle.append(case.k_new[0], case.v_new[0], keep, case.k_pages[0], case.v_pages[0])
    assert np.array_equal(bits(kd), want_k) and np.array_equal(bits(vd), want_v)
    assert ws.status() == -7
