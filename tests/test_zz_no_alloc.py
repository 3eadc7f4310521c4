"""pkv_decode_attn_noalloc: decode attention for callers that may not allocate
device memory (a plug-in whose host runtime owns all device memory, a serving
loop that reserves memory once and must not allocate afterwards). Its split-KV
scratch is a fixed array inside the library instead of a caller workspace.

Checked here through the C ABI: two calls in a row give the same output as
pkv_decode_attn (the entry point with a workspace). Both run the same kernel
with the same grid and merge order, so the outputs are compared bit for bit,
and the result is also checked against the fp64 oracle at the parity
tolerance. The cases: a batch whose contexts are split over many CTAs (so the
scratch partials and counters are used), one long context (the counted
merge) and a ragged batch with padding rows. This file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_gb300 as pkv
from gpu_util import DecodeOnDevice
from parity import assert_close, bf16_to_f64
from paged_kv_decode_gb300 import _lib
from paged_kv_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seq_lens", [W.config_seq_lens(2), [40000], [0, 37, 200, 0]])
def test_noalloc_matches_workspace_entry_point_on_two_calls(cuda_device, seq_lens):
    case = W.decode_case(21, seq_lens, pending_append=False, poison=True)
    run = DecodeOnDevice(case, 0, cuda_device)
    ref = run.step().clone()
    torch.cuda.synchronize()
    assert run.ws.status() == 0
    want = oracle.decode(case.q[0], case.k_pages[0], case.v_pages[0], case.block_table, case.seq_lens,
                         case.geom.scale)
    for _ in range(2):
        out = torch.full_like(run.q, float("nan"))
        pkv.decode_attn_noalloc(run.q, run.k_pages, run.v_pages, run.block_table, run.seq_lens, out,
                                case.geom.scale)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), "noalloc differs from the workspace call"
        assert_close(bf16_to_f64(out), want, "noalloc vs oracle")


def test_noalloc_rejects_batch_beyond_its_scratch(cuda_device):
    d = pkv.desc(16)
    dummy = torch.zeros(64, dtype=torch.bfloat16, device=cuda_device)
    p = dummy.data_ptr()
    rc = _lib.load().pkv_decode_attn_noalloc(p, p, p, p, p, p, 1.0, None, ctypes.byref(d), 257, 1)
    assert rc == -4
