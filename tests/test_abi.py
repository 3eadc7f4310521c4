"""The C-ABI library: it builds, loads, exports every symbol include/pkv.h
declares, and rejects bad arguments on the host before touching a device.
CPU only: no call here launches or queries a GPU."""
import ctypes

import pytest

from paged_kv_decode_gb300 import _lib
from paged_kv_decode_gb300.build import build_library


@pytest.fixture(scope="module")
def lib():
    build_library()
    return _lib.load()


def test_exports_every_declared_function(lib):
    declared = _lib.header_functions()
    assert len(declared) >= 8
    assert set(declared) == set(_lib.PROTOTYPES), "binding prototypes out of sync with include/pkv.h"
    for name in declared:
        assert hasattr(lib, name), f"libpkv.so does not export {name}"


def test_status_strings(lib):
    for code in [0, -1, -2, -3, -4, -5, -6, -7, -8]:
        s = lib.pkv_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.pkv_status_string(12345).decode() == "unknown status"


def _desc(**kw):
    d = dict(num_q_heads=16, num_kv_heads=8, head_dim=128, page_size=16, num_pages=4)
    d.update(kw)
    return _lib.CacheDesc(**d)


def test_host_argument_checks(lib):
    d = _desc()
    # NULL descriptor
    assert lib.pkv_append(None, None, None, 1, None, None, None, None, None, 0) == -1
    # unsupported geometry: decode, append, the fused append + decode and prefill take page size 16,
    # head_dim 64 or 128 and 1 to 8 query heads per KV head; the RoPE call only 16/8/128/16
    for bad in (_desc(head_dim=96), _desc(num_q_heads=36, num_kv_heads=4), _desc(num_q_heads=20),
                _desc(page_size=32), _desc(num_q_heads=32, num_kv_heads=2)):
        assert lib.pkv_append(None, None, None, 1, None, None, ctypes.byref(bad), None, None, 0) == -3
        assert lib.pkv_decode_attn(None, None, None, None, None, None, 1.0, None, ctypes.byref(bad), 1, 1, None,
                                   0) == -3
        assert lib.pkv_prefill_chunk_attn(None, None, None, None, None, None, 1, 1, None, 1.0, None,
                                          ctypes.byref(bad), 1, 1, None, 0) == -3
    for other in (_desc(head_dim=64), _desc(num_q_heads=32, num_kv_heads=8), _desc(num_q_heads=8),
                  _desc(num_q_heads=40), _desc(num_q_heads=28, num_kv_heads=4), _desc(num_q_heads=24)):
        # served by the decode path with run-time head counts: past the geometry check, stopped at the NULL
        # pointers
        assert lib.pkv_decode_attn(None, None, None, None, None, None, 1.0, None, ctypes.byref(other), 1, 1, None,
                                   0) == -1
        assert lib.pkv_append(None, None, None, 1, None, None, ctypes.byref(other), None, None, 0) == -1
        assert lib.pkv_decode_append_attn(None, None, None, None, None, None, None, None, 1.0, None,
                                          ctypes.byref(other), 1, 1, None, 0, 0) == -1
        # (a table address the host never reads: past the geometry check, stopped at the NULL pointers)
        assert lib.pkv_decode_append_rope_attn(None, None, None, None, None, None, None, 256, 1, None, 1.0, None,
                                               ctypes.byref(other), 1, 1, None, 0, 0) == -1
        assert lib.pkv_prefill_chunk_attn(None, None, None, None, None, None, 1, 1, None, 1.0, None,
                                          ctypes.byref(other), 1, 1, None, 0) == -1
    # sizes
    assert lib.pkv_append(None, None, None, -1, None, None, ctypes.byref(d), None, None, 0) == -2
    assert lib.pkv_decode_attn(None, None, None, None, None, None, 1.0, None, ctypes.byref(d), -1, 1, None, 0) == -2
    assert lib.pkv_decode_attn(None, None, None, None, None, None, 1.0, None, ctypes.byref(d), 1, 0, None, 0) == -2
    zero_pages = _desc(num_pages=0)
    assert lib.pkv_append(None, None, None, 1, None, None, ctypes.byref(zero_pages), None, None, 0) == -2
    # the decode kernel counts (request, KV head, page) triples in 32 bits: batch * max_pages * max(KV heads, 8)
    # must stay below 2^31 (1024 * 65536 * 32 = 2^31 is refused for 32 KV heads, the same table for 8 is not)
    mha = _desc(num_q_heads=32, num_kv_heads=32)
    assert lib.pkv_decode_attn(None, None, None, None, None, None, 1.0, None, ctypes.byref(mha), 1024, 65536,
                               None, 0) == -2
    assert lib.pkv_decode_append_attn(None, None, None, None, None, None, None, None, 1.0, None, ctypes.byref(mha),
                                      1024, 65536, None, 0, 0) == -2
    assert lib.pkv_decode_attn(None, None, None, None, None, None, 1.0, None, ctypes.byref(d), 1024, 65536,
                               None, 0) == -1
    # nothing to do is fine, without any device
    assert lib.pkv_append(None, None, None, 0, None, None, ctypes.byref(d), None, None, 0) == 0
    # missing pointers
    assert lib.pkv_append(None, None, None, 3, None, None, ctypes.byref(d), None, None, 0) == -1
    assert lib.pkv_decode_attn(None, None, None, None, None, None, 1.0, None, ctypes.byref(d), 2, 4, None, 0) == -1
    # a workspace smaller than the status header
    ws = ctypes.create_string_buffer(64)
    assert lib.pkv_append(None, None, None, 0, None, None, ctypes.byref(d), None, ws, 64) == -4
    # more requests than one decode launch takes
    assert lib.pkv_decode_attn(None, None, None, None, None, None, 1.0, None, ctypes.byref(d), 1025, 1, None,
                               0) == -3
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(d), 1025, 1) == 0
    # workspace queries refuse bad arguments
    assert lib.pkv_decode_workspace_bytes(None, 1, 1) == 0
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(d), -1, 1) == 0
    assert lib.pkv_decode_workspace_bytes(ctypes.byref(d), 1, 0) == 0


def test_rope_table_host_argument_checks(lib):
    # pkv_rope_table checks its arguments before it looks at any device
    buf = ctypes.create_string_buffer(64)
    p = (ctypes.addressof(buf) + 15) // 16 * 16  # never written: every call below is rejected
    f = lib.pkv_rope_table
    assert f(None, 8, 128, 1e6, None) == -1
    assert f(p, 0, 128, 1e6, None) == -2
    assert f(p, 8, 127, 1e6, None) == -2
    assert f(p, 8, 2048, 1e6, None) == -2
    assert f(p, 8, 128, 0.0, None) == -2
    assert f(p, 8, 128, float("nan"), None) == -2
    assert f(p + 4, 8, 128, 1e6, None) == -8


def test_mixed_step_host_argument_checks(lib):
    # pkv_mixed_step_attn serves 16/8/128 and checks both halves' arguments before any device lookup
    f = lib.pkv_mixed_step_attn
    buf = ctypes.create_string_buffer(1024)
    p = (ctypes.addressof(buf) + 255) // 256 * 256  # aligned host address, never dereferenced
    d = _desc()

    def call(desc=d, num_seqs=1, total_q=8, max_q=8, dec_batch=2, dec_pages=4, ws=p, ws_bytes=256, q=None, dq=None,
             kp=None):
        q = p if q is None else q
        dq = p if dq is None else dq
        kp = p if kp is None else kp
        return f(q, kp, kp, p, p, p, num_seqs, total_q, q, 4, max_q, dq, p, p, dq, dec_batch, dec_pages, 1.0, None,
                 None if desc is None else ctypes.byref(desc), ws, ws_bytes)

    assert call(desc=None) == -1
    for other in (_desc(num_q_heads=32), _desc(head_dim=64)):
        assert call(desc=other) == -3
    assert call(num_seqs=-1) == -2
    assert call(dec_batch=-1) == -2
    assert call(dec_pages=0) == -2
    assert call(dec_batch=1025) == -3
    assert call(ws=None) == -1
    assert call(ws_bytes=64) == -4
    assert call(num_seqs=0, dec_batch=0) == 0  # nothing to do
    assert call(kp=0) == -1
    assert call(q=p + 2) == -8
    assert call(dq=p + 4) == -8
    assert lib.pkv_mixed_workspace_bytes(None, 1, 8, 2, 4) == 0
    assert lib.pkv_mixed_workspace_bytes(ctypes.byref(_desc(num_q_heads=32)), 1, 8, 2, 4) == 0
    assert lib.pkv_mixed_workspace_bytes(ctypes.byref(d), 1, 8, -1, 4) == 0


def test_noalloc_host_argument_checks(lib):
    # pkv_decode_attn_noalloc rejects bad arguments before it looks up its device array
    f = lib.pkv_decode_attn_noalloc
    d = _desc()
    dummy = ctypes.create_string_buffer(64)
    p = (ctypes.addressof(dummy) + 15) // 16 * 16  # 16-byte aligned host address, never dereferenced
    args = lambda batch=1, max_pages=1, desc=d, ptr=p, q=None: (q or ptr, ptr, ptr, ptr, ptr, ptr, 1.0, None,
                                                                   None if desc is None else ctypes.byref(desc),
                                                                   batch, max_pages)
    assert f(*args(desc=None)) == -1
    # only the 16/8/128/16 geometry, also where pkv_decode_attn serves others
    for other in (_desc(num_q_heads=32, num_kv_heads=8), _desc(head_dim=64), _desc(num_q_heads=8)):
        assert f(*args(desc=other)) == -3
    assert f(*args(desc=_desc(num_pages=0))) == -2
    assert f(*args(batch=-1)) == -2
    assert f(*args(max_pages=0)) == -2
    # more requests than the fixed array holds partial results for
    assert f(*args(batch=257)) == -4
    # a block table too large for the kernels' 32-bit indexing
    assert f(*args(batch=256, max_pages=1 << 20)) == -2
    # an empty batch is a no-op, without any device
    assert f(*args(batch=0)) == 0
    # missing and misaligned pointers
    assert f(*args(ptr=None)) == -1
    assert f(*args(q=p + 2)) == -8


def test_no_cpu_fallback_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.load()
