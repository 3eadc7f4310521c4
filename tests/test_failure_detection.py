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


class _FakeLib:
    """Stands in for libpkv on the CPU: a status word the test sets, and a record of re-inits."""

    def __init__(self, status):
        self.status = status
        self.inits = []

    def pkv_read_status(self, ws, stream):
        return self.status

    def pkv_workspace_init(self, ws, nbytes, stream):
        self.inits.append((ws.value, nbytes))
        self.status = 0
        return 0

    def pkv_status_string(self, code):
        return b"fake"


@pytest.mark.parametrize("code", [-6, -7])
def test_workspace_is_zeroed_again_after_a_device_error(monkeypatch, code):
    # the documented rule: after a call whose status word is not PKV_OK, the workspace is
    # initialised again before its next use (stale counters or tagged records would otherwise
    # be taken for the next call's own); Workspace.check does that before raising
    fake = _FakeLib(code)
    monkeypatch.setattr(_lib, "load", lambda: fake)
    monkeypatch.setattr(pkv, "_stream", lambda s: ctypes.c_void_p(0))
    ws = object.__new__(pkv.Workspace)
    ws.tensor = torch.zeros(1024, dtype=torch.uint8)
    with pytest.raises(pkv.PkvError) as e:
        ws.check("decode")
    assert e.value.code == code
    assert fake.inits == [(ws.tensor.data_ptr(), 1024)]
    ws.check("decode")  # clean now: no error, no further init
    assert len(fake.inits) == 1
