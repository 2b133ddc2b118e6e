"""mkv_basis_static, the allocation-free basis call, against mkv_compress.

mkv_basis_static computes the per-stream bases and eigenvalues that
mkv_compress computes, without a ctx and with its scratch in a static device
buffer of the library.  Its results are compared with what mkv_compress stores
(read back with mkv_export), on two calls in a row with different inputs, so
that anything left in the shared buffer by the first call would show in the
second.  This file is collected last, so that it runs both after the other GPU
tests and, on its own, in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from two_compressed_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
EIG_LAM = 3e-4     # eigenvalue error, relative to the largest eigenvalue
EIG_GAP = 1e-2     # eigenvectors compared where the relative eigengap exceeds this
EIG_COS = 1e-3     # 1 - |cos| allowed for those eigenvectors


@pytest.fixture(scope="module")
def M():
    from two_compressed_kv_gb300 import mkv
    return mkv


def _compress_reference(M, w, K, V):
    """Bases and eigenvalues as mkv_compress stores them: [2][B*H][128][128], [2][B*H][128]."""
    cfg = M.make_config(w.batch, w.n_kv_heads, w.n_q_heads, K.shape[2], w.segment, w.c, w.tau,
                        w.top_k)
    R = np.zeros((2, w.batch * w.n_kv_heads, 128, 128), np.float32)
    lam = np.zeros((2, w.batch * w.n_kv_heads, 128), np.float32)
    with M.Mkv(cfg) as m:
        m.compress(K, V)
        torch.cuda.synchronize()
        for x in range(2):
            for b in range(w.batch):
                for h in range(w.n_kv_heads):
                    Rs, ls, _, _ = m.export(b, h, x)
                    R[x, b * w.n_kv_heads + h] = Rs
                    lam[x, b * w.n_kv_heads + h] = ls
    return R, lam


def _static(M, K, V):
    B, H = K.shape[0], K.shape[1]
    R = torch.full((2, B * H, 128, 128), float("nan"), dtype=torch.float32, device=DEV)
    lam = torch.full((2, B * H, 128), float("nan"), dtype=torch.float32, device=DEV)
    M.mkv_basis_static(K, V, R, lam)
    torch.cuda.synchronize()
    return R.cpu().numpy(), lam.cpu().numpy()


def _assert_close(R, lam, R_ref, lam_ref):
    assert np.isfinite(R).all() and np.isfinite(lam).all()
    for x in range(R.shape[0]):
        for s in range(R.shape[1]):
            lr = lam_ref[x, s].astype(np.float64)
            scale = max(abs(lr[0]), 1e-30)
            assert np.abs(lam[x, s] - lr).max() <= EIG_LAM * scale, (x, s)
            gap = np.full(128, np.inf)
            d = np.abs(np.diff(lr)) / scale
            gap[:-1] = np.minimum(gap[:-1], d)
            gap[1:] = np.minimum(gap[1:], d)
            cols = np.nonzero(gap > EIG_GAP)[0]
            cos = np.abs(np.einsum("rj,rj->j", R[x, s][:, cols].astype(np.float64),
                                   R_ref[x, s][:, cols].astype(np.float64)))
            assert (cos >= 1 - EIG_COS).all(), (x, s, cos.min())


def test_two_calls_in_a_row_match_compress(M):
    """Same Gram chunking as mkv_compress here (2*1*2 streams x 16 chunks fit
    the buffer): the results are checked within tolerance and are expected to
    be the same bits."""
    w1 = W.small_workload("no-alloc-a", batch=1, n_kv_heads=2, n_q_heads=4, ctx=4096, seed=21)
    w2 = W.small_workload("no-alloc-b", batch=1, n_kv_heads=2, n_q_heads=4, ctx=4096, seed=22)
    inputs = []
    for w in (w1, w2):
        K, V = W.draw_kv(w)
        inputs.append((w, K.to(DEV), V.to(DEV)))
    refs = [_compress_reference(M, w, K, V) for w, K, V in inputs]
    got = [_static(M, K, V) for _, K, V in inputs]
    for (R, lam), (R_ref, lam_ref) in zip(got, refs):
        _assert_close(R, lam, R_ref, lam_ref)
        assert np.array_equal(R, R_ref) and np.array_equal(lam, lam_ref)
    # the two inputs differ, so the second call did not reuse the first's result
    assert not np.array_equal(got[0][0], got[1][0])


def test_fewer_chunks_when_the_buffer_is_short(M):
    """2*2*8 = 32 streams x 19 chunks would need 38 MiB: the call uses 8 chunks
    per stream instead, a different summation order, so the results agree to
    fp32 rounding."""
    w = W.small_workload("no-alloc-c", batch=2, n_kv_heads=8, n_q_heads=32, ctx=8192, seed=23)
    K, V = W.draw_kv(w)
    K, V = K.to(DEV), V.to(DEV)
    R_ref, lam_ref = _compress_reference(M, w, K, V)
    for _ in range(2):
        R, lam = _static(M, K, V)
        _assert_close(R, lam, R_ref, lam_ref)


def test_calls_do_not_change_free_device_memory(M):
    w = W.small_workload("no-alloc-d", batch=1, n_kv_heads=2, n_q_heads=4, ctx=2048, seed=24)
    K, V = W.draw_kv(w)
    K, V = K.to(DEV), V.to(DEV)
    R = torch.empty((2, 2, 128, 128), dtype=torch.float32, device=DEV)
    lam = torch.empty((2, 2, 128), dtype=torch.float32, device=DEV)
    M.mkv_basis_static(K, V, R, lam)   # the first call on a device may load the buffer
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        M.mkv_basis_static(K, V, R, lam)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


def test_oversized_request_is_rejected(M):
    K = torch.zeros((16, 9, 16, 128), dtype=torch.float16, device=DEV)
    R = torch.zeros((2, 16 * 9, 128, 128), dtype=torch.float32, device=DEV)
    lam = torch.zeros((2, 16 * 9, 128), dtype=torch.float32, device=DEV)
    with pytest.raises(M.MkvError) as e:
        M.mkv_basis_static(K, K, R, lam)
    assert e.value.status == M.MKV_ERR_INVALID_ARG
    assert str(M.MKV_BASIS_STATIC_MAX_BYTES) in M.mkv_last_error_string()
    # the rejection launched nothing and left the outputs alone
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(R)) == 0
    st = M.lib.mkv_basis_static(ctypes.c_void_p(K.data_ptr() + 2), ctypes.c_void_p(K.data_ptr()),
                                1, 1, 16, ctypes.c_void_p(R.data_ptr()),
                                ctypes.c_void_p(lam.data_ptr()), None)
    assert st == M.MKV_ERR_INVALID_ARG
