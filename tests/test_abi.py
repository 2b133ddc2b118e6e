"""The C-ABI library without a GPU: it loads, exports every symbol that
include/mkv.h declares, its structs match the binding's layout, and its
host-only entry points (config validation, layout sizes, status strings)
behave.  No call here launches a kernel."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

from oracle import mosaickv as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mkv.h")


@pytest.fixture(scope="module")
def M():
    from two_compressed_kv_gb300 import build_lib
    if not os.path.exists(build_lib.LIB):
        build_lib.build()
    from two_compressed_kv_gb300 import mkv
    return mkv


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(mkv_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(M):
    names = declared_functions()
    assert len(names) >= 11, names
    lib = ctypes.CDLL(M.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_struct_layout_matches_binding(M):
    src = r'''
#include <stdio.h>
#include <stddef.h>
#include "mkv.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu\n", sizeof(mkv_config), offsetof(mkv_config, max_pool_bytes),
         offsetof(mkv_config, device), sizeof(mkv_segment_header), sizeof(mkv_stats_t),
         offsetof(mkv_stats_t, kernel_launches));
  return 0;
}
'''
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "l.c")
        exe = os.path.join(d, "l")
        open(c, "w").write(src)
        subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe])
        got = [int(x) for x in subprocess.check_output([exe]).split()]
    want = [ctypes.sizeof(M.mkv_config), M.mkv_config.max_pool_bytes.offset,
            M.mkv_config.device.offset, ctypes.sizeof(M.mkv_segment_header),
            ctypes.sizeof(M.mkv_stats_t), M.mkv_stats_t.kernel_launches.offset]
    assert got == want


def test_segment_bytes_match_oracle_layout(M):
    for st in (0, 1, 2, 3):
        for c in range(8, 129, 8):
            for rows in (1, 2, 7, 16, 44, 64, 128, 255, 256):
                assert M.mkv_segment_bytes(st, rows, c) == O.segment_cost(st, rows, c)
    assert M.mkv_segment_bytes(4, 10, 8) == 0
    assert M.mkv_segment_bytes(0, 0, 8) == 0


def _cfg(M, **kw):
    base = dict(batch=1, n_kv_heads=8, n_q_heads=32, max_ctx=4096, segment=64, c=64, tau=0.9,
                top_k=256)
    base.update(kw)
    return M.make_config(**base)


def test_validate_config(M):
    assert M.mkv_validate_config(_cfg(M)) == M.MKV_OK
    bad = [dict(head_dim=64), dict(n_q_heads=30), dict(n_q_heads=8 * 17), dict(segment=8),
           dict(segment=72), dict(segment=272), dict(c=4), dict(c=36), dict(c=136),
           dict(tau=0.0), dict(tau=1.5), dict(tau=float("nan")), dict(top_k=0),
           dict(max_ctx=0), dict(batch=0), dict(attn_chunk=4), dict(attn_chunk=12),
           dict(flags=16), dict(device=-1), dict(attn_chunk=136)]
    for b in bad:
        assert M.mkv_validate_config(_cfg(M, **b)) == M.MKV_ERR_INVALID_ARG, b
    for good in [dict(segment=16), dict(segment=256), dict(c=8), dict(c=128), dict(tau=1.0),
                 dict(attn_chunk=8), dict(attn_chunk=128), dict(n_kv_heads=4, n_q_heads=28)]:
        assert M.mkv_validate_config(_cfg(M, **good)) == M.MKV_OK, good


def test_create_rejects_bad_config_without_gpu(M):
    h = ctypes.c_void_p()
    cfg = _cfg(M, c=36)
    assert M.lib.mkv_create(ctypes.byref(cfg), ctypes.byref(h)) == M.MKV_ERR_INVALID_ARG
    assert h.value is None
    assert M.lib.mkv_create(None, ctypes.byref(h)) == M.MKV_ERR_INVALID_ARG


def test_status_strings_and_null_safety(M):
    for s in range(7):
        assert M.mkv_status_string(s).startswith("MKV_")
    M.mkv_free(None)
    assert M.lib.mkv_decode(None, None, None, None, None) == M.MKV_ERR_INVALID_ARG
    assert M.lib.mkv_compress(None, None, None, 1, None) == M.MKV_ERR_INVALID_ARG
    assert M.lib.mkv_stats(None, None) == M.MKV_ERR_INVALID_ARG


def test_basis_static_rejects_before_any_cuda_call(M):
    """Oversized, NULL and unaligned requests fail on the host; the pointers
    below are never dereferenced."""
    p = ctypes.c_void_p(1 << 20)
    assert M.lib.mkv_basis_static(p, p, 16, 9, 64, p, p, None) == M.MKV_ERR_INVALID_ARG
    msg = M.mkv_last_error_string()
    assert "288 streams" in msg and str(M.MKV_BASIS_STATIC_MAX_BYTES) in msg
    assert M.lib.mkv_basis_static(None, p, 1, 1, 64, p, p, None) == M.MKV_ERR_INVALID_ARG
    assert M.lib.mkv_basis_static(p, p, 1, 1, 0, p, p, None) == M.MKV_ERR_INVALID_ARG
    q = ctypes.c_void_p((1 << 20) + 8)
    assert M.lib.mkv_basis_static(q, p, 1, 1, 64, p, p, None) == M.MKV_ERR_INVALID_ARG


def test_basis_static_binding_rejects_mixed_devices(M, monkeypatch):
    """The binding refuses tensors on different devices before it calls the
    library (the library works on the current device only)."""
    import torch
    calls = []
    monkeypatch.setattr(M._lib, "mkv_basis_static", lambda *a: calls.append(a) or 0,
                        raising=False)
    k = torch.empty((1, 1, 16, 128), dtype=torch.float16, device="meta")
    v = torch.empty((1, 1, 16, 128), dtype=torch.float16, device="cpu")
    R = torch.empty((2, 1, 128, 128), dtype=torch.float32, device="meta")
    lam = torch.empty((2, 1, 128), dtype=torch.float32, device="meta")
    with pytest.raises(ValueError, match="one device"):
        M.mkv_basis_static(k, v, R, lam)
    assert not calls


def test_debug_hooks_reject_bad_arguments_without_gpu(M):
    assert M.lib.mkv_debug_wait_test(None, 1_000_000, None) == M.MKV_ERR_INVALID_ARG
    fake = ctypes.c_void_p(1 << 20)     # never dereferenced: the limit is checked first
    assert M.lib.mkv_debug_wait_test(fake, 10, None) == M.MKV_ERR_INVALID_ARG
    assert M.lib.mkv_debug_wait_test(fake, 3_000_000_000, None) == M.MKV_ERR_INVALID_ARG
    assert M.lib.mkv_debug_set_check_extent(None, 0) == M.MKV_ERR_INVALID_ARG


def test_decode_layers_rejects_bad_arguments_without_gpu(M):
    """Argument checks of mkv_decode_layers run before any CUDA call."""
    ok = M.MKV_ERR_INVALID_ARG
    assert M.mkv_decode_layers_raw(None, 1, [1], [1]) == ok
    assert M.mkv_decode_layers_raw([None], 1, [1], [1]) == ok
    assert M.mkv_decode_layers_raw([1], 1, None, [1]) == ok
    assert M.mkv_decode_layers_raw([1], 1, [1], None) == ok
    assert M.mkv_decode_layers_raw([1], 0, [1], [1]) == ok
    assert M.mkv_decode_layers_raw([1] * 65, 65, [1] * 65, [1] * 65) == ok
    assert M.MKV_MAX_FUSED_LAYERS == 64

