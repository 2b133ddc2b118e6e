"""Failure detection on the GPU without any fault, trap or hang.

* A bounded device-side wait that runs out: a test hook runs the library's own
  mbarrier wait on a barrier no thread arrives on, with a 1 ms limit; the
  kernel must return, mkv_check_device must report MKV_ERR_TIMEOUT once, and
  the ctx must keep working.
* The kernels' packed-cache bounds checks: a test hook shrinks the checked
  extent below the real pool, so that ordinary in-bounds accesses count as
  violations (no access ever leaves the allocated pool); the library must
  report MKV_ERR_DEVICE_CHECK and work again once the extent is restored.
"""
import numpy as np
import pytest
import torch

from two_compressed_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def M():
    from two_compressed_kv_gb300 import mkv
    return mkv


def _ctx(M, w):
    cfg = M.make_config(w.batch, w.n_kv_heads, w.n_q_heads, w.ctx, w.segment, w.c, w.tau,
                        w.top_k)
    return M.Mkv(cfg)


def test_bounded_wait_gives_up_and_ctx_stays_usable(M):
    w = W.small_workload("wait", ctx=1000, top_k=64)
    K, V = W.draw_kv(w, device=DEV)
    q = W.draw_queries(w, K)
    with _ctx(M, w) as m:
        m.compress(K, V)
        sel0 = torch.empty(1, 2, 64, dtype=torch.int32, device=DEV)
        out0 = m.decode(q, sel=sel0).cpu()
        assert M.mkv_check_device(m.ctx) == M.MKV_OK
        M.mkv_debug_wait_test(m.ctx, 1_000_000)
        assert M.mkv_check_device(m.ctx) == M.MKV_ERR_TIMEOUT
        assert "wait" in M.mkv_last_error_string()
        # reported once, then cleared; later work is unaffected
        assert M.mkv_check_device(m.ctx) == M.MKV_OK
        sel1 = torch.empty_like(sel0)
        out1 = m.decode(q, sel=sel1).cpu()
        assert M.mkv_check_device(m.ctx) == M.MKV_OK
        assert torch.equal(out0, out1) and torch.equal(sel0, sel1)
    with pytest.raises(M.MkvError):
        with _ctx(M, w) as m2:
            M.mkv_debug_wait_test(m2.ctx, 10)      # below the 1 us minimum


def test_bounds_checks_report_device_check(M):
    w = W.small_workload("checks", ctx=2000, top_k=128, n_q_heads=8)
    K, V = W.draw_kv(w, device=DEV)
    q = W.draw_queries(w, K)
    with _ctx(M, w) as m:
        m.compress(K, V)
        out0 = m.decode(q).cpu()
        assert M.mkv_check_device(m.ctx) == M.MKV_OK
        st = m.stats()
        packed = st["payload_bytes"][0] + st["payload_bytes"][1]
        # decode: the score pass and the attention gathers read past half the pool
        M.mkv_debug_set_check_extent(m.ctx, packed // 2)
        m.decode(q)
        assert M.mkv_check_device(m.ctx) == M.MKV_ERR_DEVICE_CHECK
        assert "extent" in M.mkv_last_error_string()
        M.mkv_debug_set_check_extent(m.ctx, 0)
        out1 = m.decode(q).cpu()
        assert M.mkv_check_device(m.ctx) == M.MKV_OK
        assert torch.equal(out0, out1)
        # compression: packing writes past a 4 KiB extent
        M.mkv_debug_set_check_extent(m.ctx, 4096)
        m.compress(K, V)
        assert M.mkv_check_device(m.ctx) == M.MKV_ERR_DEVICE_CHECK
        M.mkv_debug_set_check_extent(m.ctx, 0)
        m.compress(K, V)
        out2 = m.decode(q).cpu()
        assert M.mkv_check_device(m.ctx) == M.MKV_OK
        assert torch.equal(out0, out2)
        # an extent larger than the pool changes nothing
        M.mkv_debug_set_check_extent(m.ctx, 1 << 40)
        out3 = m.decode(q).cpu()
        assert M.mkv_check_device(m.ctx) == M.MKV_OK
        assert torch.equal(out0, out3)
