"""Failure detection without faulting the GPU: a device-side wait that nothing
completes gives up after its bound, records PKV_ERR_DEVICE_TIMEOUT in the
status word, and the context keeps working (a decode call afterwards is
correct)."""
import ctypes

import pytest
import torch

import oracle
import paged_kv_decode_gb300 as pkv
from gpu_util import DecodeOnDevice, ensure_built
from parity import assert_close, bf16_to_f64
from paged_kv_decode_gb300 import _lib
from paged_kv_decode_gb300 import workloads as W


def test_selftest_rejects_bad_arguments_on_the_host():
    ensure_built()
    lib = _lib.load()
    assert lib.pkv_selftest_wait_timeout(None, 0, 100, None) == -1
    buf = ctypes.create_string_buffer(64)
    assert lib.pkv_selftest_wait_timeout(buf, 64, 100, None) == -4
    big = ctypes.create_string_buffer(512)
    assert lib.pkv_selftest_wait_timeout(big, 512, -1, None) == -2


@pytest.mark.gpu
def test_wait_that_never_completes_times_out_and_reports(cuda_device):
    ensure_built()
    ws = pkv.Workspace(pkv.PKV_STATUS_BYTES, cuda_device)
    assert ws.status() == 0
    st = torch.cuda.current_stream()
    rc = _lib.load().pkv_selftest_wait_timeout(ctypes.c_void_p(ws.tensor.data_ptr()), ws.nbytes, 2_000_000,
                                               ctypes.c_void_p(st.cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert ws.status() == -6  # PKV_ERR_DEVICE_TIMEOUT
    # the context is still usable: a decode call afterwards matches the oracle
    case = W.decode_case(50, [300, 77], pending_append=False, poison=True)
    run = DecodeOnDevice(case, 0, cuda_device)
    out = run.step()
    torch.cuda.synchronize()
    want = oracle.decode(case.q[0], case.k_pages[0], case.v_pages[0], case.block_table, case.seq_lens,
                         case.geom.scale)
    assert_close(bf16_to_f64(out), want, "after timeout")
    assert run.ws.status() == 0
