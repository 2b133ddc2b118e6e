"""Parity of the CUDA library (through its C ABI) with the CPU oracle.

Every stream is checked on the small workloads; at the full workload sizes the
oracle recomputes sampled streams one by one.  See parity_util for the rules.
"""
import math

import numpy as np
import pytest
import torch

from oracle import mosaickv as O
from parity_util import (assert_budgets, check_basis, compare_compressed, compare_decode,
                         compare_oracle_packed)
from two_compressed_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def M():
    from two_compressed_kv_gb300 import mkv
    return mkv


def run_gpu(M, w, K, V, q, attn_chunk=0, max_ctx=None, flags=0):
    cfg = M.make_config(w.batch, w.n_kv_heads, w.n_q_heads, max_ctx or K.shape[2], w.segment,
                        w.c, w.tau, w.top_k, attn_chunk=attn_chunk, flags=flags)
    m = M.Mkv(cfg)
    m.compress(K.to(DEV), V.to(DEV))
    kk = min(w.top_k, K.shape[2])
    sel = torch.empty(w.batch, w.n_kv_heads, kk, dtype=torch.int32, device=DEV)
    out = m.decode(q.to(DEV), sel=sel)
    torch.cuda.synchronize()
    return m, out.cpu().numpy(), sel.cpu().numpy()


def check_streams(w, K, V, q, m, out, sel, streams, basis=True, oracle_packed=True,
                  bitmask_pv=False):
    rep = {}
    g = w.group
    T = K.shape[2]
    for b, h in streams:
        RK, lamK, hk, pk = m.export(b, h, 0)
        RV, lamV, hv, pv = m.export(b, h, 1)
        Kn = K[b, h].cpu().numpy()
        Vn = V[b, h].cpu().numpy()
        if basis:
            check_basis(Kn, RK, lamK, rep)
            check_basis(Vn, RV, lamV, rep)
        ck = compare_compressed(Kn, RK, hk, pk, w.segment, w.c, w.tau, rep, bitmask_pv)
        cv = compare_compressed(Vn, RV, hv, pv, w.segment, w.c, w.tau, rep, bitmask_pv)
        Kh = O.unpack_stream(hk, pk, T, w.segment, w.c)
        Vh = O.unpack_stream(hv, pv, T, w.segment, w.c)
        qn = q[b, h * g:(h + 1) * g].cpu().numpy()
        compare_decode(qn, RK, RV, Kh, Vh, w.top_k, sel[b, h], out[b, h * g:(h + 1) * g], rep)
        if oracle_packed:
            compare_oracle_packed(qn, ck, cv, w.top_k, sel[b, h], out[b, h * g:(h + 1) * g], Kh,
                                  rep)
    return rep


def all_streams(w):
    return [(b, h) for b in range(w.batch) for h in range(w.n_kv_heads)]


def _near_tie_budget(rep, name=None, crowded=False):
    import os
    assert_budgets(name or os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], rep,
                   crowded)


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------
def test_tiny_4k_every_stream(M):
    w = W.TINY_4K
    K, V = W.draw_kv(w)
    q = W.draw_queries(w, K)
    m, out, sel = run_gpu(M, w, K, V, q)
    rep = check_streams(w, K, V, q, m, out, sel, all_streams(w))
    _near_tie_budget(rep)
    st = m.stats()
    assert st["strategy_count"][0][0] > 0
    m.close()


def test_layer_32k_every_stream(M):
    w = W.LAYER_32K
    K, V = W.draw_kv(w, device=DEV)
    q = W.draw_queries(w, K)
    m, out, sel = run_gpu(M, w, K, V, q)
    rep = check_streams(w, K, V, q, m, out, sel, all_streams(w), basis=False)
    # bases: a few streams against fp64 (the eigen-solve is the same code for all)
    check_basis(K[0, 0].cpu().numpy(), *m.export(0, 0, 0)[:2], rep)
    check_basis(V[3, 7].cpu().numpy(), *m.export(3, 7, 1)[:2], rep)
    _near_tie_budget(rep)
    m.close()


@pytest.mark.parametrize("w,streams", [
    (W.HEADLINE_128K, [(0, 0), (7, 7)]),
    (W.MILLION_1M, [(0, 0), (0, 5)]),
    (W.MIXED_256K, [(0, 0), (3, 3)]),
], ids=["headline-128K-b8", "million-1M", "mixed-256K"])
def test_full_size_sampled_streams(M, w, streams):
    K, V = W.draw_kv(w, layer=0, device=DEV)
    q = W.draw_queries(w, K)
    m, out, sel = run_gpu(M, w, K, V, q)
    rep = check_streams(w, K, V, q, m, out, sel, streams)
    _near_tie_budget(rep)
    # properties that hold for every stream: ascending unique in-range selections
    T = K.shape[2]
    kk = min(w.top_k, T)
    assert sel.shape == (w.batch, w.n_kv_heads, kk)
    assert (np.diff(sel, axis=2) > 0).all() and sel.min() >= 0 and sel.max() < T
    assert np.isfinite(out).all()
    st = m.stats()
    if w.mixed_regimes:
        for x in range(2):
            assert min(st["strategy_count"][x]) >= 0
        assert sum(st["strategy_count"][0][i] > 0 for i in range(3)) + \
            sum(st["strategy_count"][1][i] > 0 for i in range(3)) >= 5, st
    m.close()
    del K, V
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# Edge cases: ragged tails, tiny and huge k, extreme c and S, group sizes
# ---------------------------------------------------------------------------
EDGE = {
    "ragged-T300-S64": dict(ctx=300, segment=64),
    "T-less-than-k": dict(ctx=40, top_k=64),
    "k1": dict(ctx=200, top_k=1),
    "T1": dict(ctx=1, top_k=4),
    "T17-S16": dict(ctx=17, segment=16, top_k=5),
    "c8": dict(ctx=256, c=8, tau=0.3),
    "c128": dict(ctx=256, c=128),
    "S16": dict(ctx=256, segment=16),
    "S256-ragged": dict(ctx=700, segment=256),
    "g1": dict(n_q_heads=2, ctx=300),
    "g7": dict(n_kv_heads=1, n_q_heads=7, ctx=300),
    "g16": dict(n_kv_heads=1, n_q_heads=16, ctx=130, top_k=100),
    "tau1": dict(ctx=256, tau=1.0),
    "mixed-regimes": dict(ctx=640, segment=64, c=48, tau=0.9, mixed_regimes=True),
    "b3": dict(batch=3, n_kv_heads=2, n_q_heads=4, ctx=333, segment=32, top_k=50),
}


@pytest.mark.parametrize("name", list(EDGE))
def test_edge_cases(M, name):
    w = W.small_workload(name, **EDGE[name])
    K, V = W.draw_kv(w)
    q = W.draw_queries(w, K)
    m, out, sel = run_gpu(M, w, K, V, q)
    rep = check_streams(w, K, V, q, m, out, sel, all_streams(w), basis=False)
    _near_tie_budget(rep)
    m.close()


# ---------------------------------------------------------------------------
# Bitmask-indexed per-vector segments (MKV_FLAG_BITMASK_PV)
# ---------------------------------------------------------------------------
PVB_CASES = {
    "mixed-regimes-c48": dict(ctx=900, segment=64, c=48, tau=0.9, mixed_regimes=True),
    "c40-ragged": dict(ctx=700, segment=64, c=40, tau=0.93),
    "c16-tie-to-PV": dict(ctx=400, segment=32, c=16, tau=0.6),
    "c8-PV-cheaper": dict(ctx=300, segment=32, c=8, tau=0.4),
    "g7-S16": dict(n_kv_heads=1, n_q_heads=7, ctx=333, segment=16, c=40, tau=0.93),
}


@pytest.mark.parametrize("name", list(PVB_CASES))
def test_bitmask_pv_segments(M, name):
    w = W.small_workload("pvb-" + name, **PVB_CASES[name])
    K, V = W.draw_kv(w)
    q = W.draw_queries(w, K)
    m, out, sel = run_gpu(M, w, K, V, q, flags=M.MKV_FLAG_BITMASK_PV)
    rep = check_streams(w, K, V, q, m, out, sel, all_streams(w), basis=False, bitmask_pv=True)
    _near_tie_budget(rep)
    counts = m.stats()["strategy_count"]
    if w.c > 16:
        assert counts[0][M.MKV_STRATEGY_PV] + counts[1][M.MKV_STRATEGY_PV] == 0
        assert counts[1][M.MKV_STRATEGY_PVB] > 0
    else:
        assert counts[0][M.MKV_STRATEGY_PVB] + counts[1][M.MKV_STRATEGY_PVB] == 0
    m.close()


def test_bitmask_pv_full_size_headline_stream(M):
    """The 128K batch-8 layer with bitmask PV segments (V is mostly per-vector
    there): sampled streams against the oracle, all selections valid."""
    w = W.HEADLINE_128K
    K, V = W.draw_kv(w, layer=0, device=DEV)
    q = W.draw_queries(w, K)
    m, out, sel = run_gpu(M, w, K, V, q, flags=M.MKV_FLAG_BITMASK_PV)
    st = m.stats()
    assert st["strategy_count"][1][M.MKV_STRATEGY_PVB] > 0
    rep = check_streams(w, K, V, q, m, out, sel, [(0, 0), (5, 3)], basis=False,
                        bitmask_pv=True)
    _near_tie_budget(rep)
    assert (np.diff(sel, axis=2) > 0).all() and np.isfinite(out).all()
    m.close()
    del K, V
    torch.cuda.empty_cache()


def test_zero_and_constant_streams(M):
    """All-zero K and V (no energy: every fraction is 1) and a constant query."""
    w = W.small_workload("zeros", ctx=130, segment=32, top_k=20)
    K = torch.zeros(1, 2, 130, 128, dtype=torch.float16)
    V = torch.zeros_like(K)
    V[0, 1, :, 5] = 1.0
    K[0, 1, :, 3] = 2.0
    q = torch.ones(1, 4, 128, dtype=torch.float16)
    m, out, sel = run_gpu(M, w, K, V, q)
    rep = check_streams(w, K, V, q, m, out, sel, all_streams(w), basis=False)
    _near_tie_budget(rep)
    # all scores tie: the lowest token ids are selected
    assert (sel[0, 0] == np.arange(20)).all()
    m.close()


# ---------------------------------------------------------------------------
# Top-k with more than 8192 tokens in the k-th score's level-1 bin: the
# selection then finds the threshold from its global scratch and places the
# tokens by re-reading the scores.  Cluster sizes: 8 CTAs per stream (one
# stream of 65536 tokens), 4 (two streams of 32768), 1 (80 streams).
# ---------------------------------------------------------------------------
def test_many_candidates_all_equal_scores_cluster8(M):
    """A zero query: every score is exactly 0, so all 65536 tokens tie and the
    4096 lowest token ids are the selection (ties to the lower token)."""
    w = W.small_workload("ties-65536", batch=1, n_kv_heads=1, n_q_heads=4, ctx=65536,
                         segment=128, c=40, tau=0.85, top_k=4096, seed=31)
    K, V = W.draw_kv(w)
    q = torch.zeros(1, 4, 128, dtype=torch.float16)
    m, out, sel = run_gpu(M, w, K, V, q)
    assert np.array_equal(sel[0, 0], np.arange(4096))
    rep = check_streams(w, K, V, q, m, out, sel, all_streams(w), basis=False)
    _near_tie_budget(rep)
    m.close()


def test_many_candidates_one_bin_distinct_scores_cluster4(M):
    """Keys = one fixed vector per head + 1% noise, queries = that vector
    scaled so that the GQA-summed score sits in the middle of a level-1 bin
    (fp32 key bits 31..20: sign, exponent and 3 mantissa bits): all 32768
    scores of a stream share that bin but differ, so the threshold comes from
    the two finer radix digits over > 8192 candidates."""
    w = W.small_workload("one-bin-32768", batch=1, n_kv_heads=2, n_q_heads=8, ctx=32768,
                         segment=128, c=40, tau=0.85, top_k=1000, seed=32)
    g = torch.Generator().manual_seed(32)
    base = torch.randn(2, 128, generator=g, dtype=torch.float64)
    K = (base.view(1, 2, 1, 128) + 0.01 * torch.randn(1, 2, 32768, 128, generator=g,
                                                      dtype=torch.float64)).to(torch.float16)
    _, V = W.draw_kv(w)
    q = torch.empty(1, 8, 128, dtype=torch.float64)
    for h in range(2):
        s0 = 4.0 * float(base[h] @ base[h])          # 4 query heads per KV head
        e = math.floor(math.log2(s0))
        j = math.floor((s0 / 2.0 ** e - 1.0) * 8)
        target = 2.0 ** e * (1.0 + (j + 0.5) / 8)
        q[0, 4 * h:4 * h + 4] = base[h] * (target / s0)
    q = q.to(torch.float16)
    m, out, sel = run_gpu(M, w, K, V, q)
    for h in range(2):
        RK = m.export(0, h, 0)[0].astype(np.float64)
        cs = O.compress_stream(K[0, h].numpy(), w.segment, w.c, w.tau, R=RK)
        sc = (O.rotate_queries(q[0, 4 * h:4 * h + 4].numpy(), RK) @ cs.dense_hat().T).sum(axis=0)
        bins = np.float32(sc).view(np.uint32) >> 20
        assert (bins == bins[0]).all(), "scores do not share one level-1 bin"
        assert len(np.unique(sc)) > 8192
    rep = check_streams(w, K, V, q, m, out, sel, all_streams(w), basis=False)
    # ~400 tokens per stream lie within 1e-4 of the k-th score here
    _near_tie_budget(rep, crowded=True)
    m.close()


def test_many_candidates_all_equal_scores_cluster1(M):
    """80 streams (one CTA per stream in the selection), zero query, 16384
    tokens each, k = 100: every stream selects tokens 0..99."""
    w = W.small_workload("ties-80x16384", batch=10, n_kv_heads=8, n_q_heads=8, ctx=16384,
                         segment=64, c=40, tau=0.85, top_k=100, seed=33)
    K, V = W.draw_kv(w, device=DEV)
    q = torch.zeros(10, 8, 128, dtype=torch.float16)
    m, out, sel = run_gpu(M, w, K, V, q)
    assert (sel == np.arange(100)).all()
    rep = check_streams(w, K.cpu(), V.cpu(), q, m, out, sel, [(0, 0), (9, 7)], basis=False)
    _near_tie_budget(rep)
    m.close()


def test_dense_reduction_matches_textbook_attention(M):
    """c = 128 and k = T: the library computes plain softmax(q K^T / sqrt(d)) V
    on the original fp16 K and V, up to fp16 storage rounding of the rotated
    values (independent of the oracle and of the basis)."""
    w = W.small_workload("dense", ctx=512, segment=64, c=128, top_k=512, n_kv_heads=2,
                         n_q_heads=8)
    K, V = W.draw_kv(w)
    q = W.draw_queries(w, K)
    m, out, sel = run_gpu(M, w, K, V, q)
    for h in range(2):
        Kf = K[0, h].double().numpy()
        Vf = V[0, h].double().numpy()
        qq = q[0, h * 4:(h + 1) * 4].double().numpy()
        lg = qq @ Kf.T / math.sqrt(128)
        p = np.exp(lg - lg.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        ref = p @ Vf
        assert np.abs(out[0, h * 4:(h + 1) * 4] - ref).max() <= 2e-3
    assert (sel[0] == np.arange(512)).all()
    m.close()


# ---------------------------------------------------------------------------
# Split-K invariance, determinism, error paths
# ---------------------------------------------------------------------------
def test_split_count_invariance(M):
    w = W.small_workload("split", ctx=4000, segment=64, top_k=1000, n_q_heads=8)
    K, V = W.draw_kv(w)
    q = W.draw_queries(w, K)
    outs, sels = [], []
    for ch in (8, 64, 120, 128):
        m, out, sel = run_gpu(M, w, K, V, q, attn_chunk=ch)
        outs.append(out)
        sels.append(sel)
        m.close()
    for o, s in zip(outs[1:], sels[1:]):
        assert np.array_equal(s, sels[0])
        assert np.abs(o - outs[0]).max() <= 1e-5


def test_determinism(M):
    w = W.small_workload("det", ctx=2000, segment=64, top_k=300, n_q_heads=8)
    K, V = W.draw_kv(w)
    q = W.draw_queries(w, K)
    m1, o1, s1 = run_gpu(M, w, K, V, q)
    m2, o2, s2 = run_gpu(M, w, K, V, q)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)
    for h in range(w.n_kv_heads):
        for x in range(2):
            e1, e2 = m1.export(0, h, x), m2.export(0, h, x)
            assert np.array_equal(e1[0], e2[0]) and e1[3] == e2[3]
    # repeated decode on one ctx is bit-identical too
    o3 = m1.decode(q.to(DEV)).cpu().numpy()
    assert np.array_equal(o1, o3)
    assert M.mkv_check_device(m1.ctx) == M.MKV_OK
    m1.close()
    m2.close()


def test_error_paths(M):
    w = W.small_workload("err", ctx=256, segment=64, top_k=16)
    K, V = W.draw_kv(w)
    q = W.draw_queries(w, K).to(DEV)
    cfg = M.make_config(1, 2, 4, 512, 64, 40, 0.85, 16)
    m = M.Mkv(cfg)
    out = torch.empty(1, 4, 128, dtype=torch.float32, device=DEV)
    with pytest.raises(M.MkvError) as e:
        m.decode(q, out)
    assert e.value.status == M.MKV_ERR_STATE
    Kd, Vd = K.to(DEV), V.to(DEV)
    with pytest.raises(M.MkvError) as e:       # ctx_len beyond max_ctx
        M.mkv_compress(m.ctx, Kd, Vd, 1000)
    assert e.value.status == M.MKV_ERR_INVALID_ARG
    st = M.lib.mkv_decode(m.ctx, None, out.data_ptr(), None, None)
    assert st == M.MKV_ERR_INVALID_ARG
    m.close()
    # allocation failure injected through the pool cap: the old cache survives
    w2 = W.small_workload("err2", ctx=512, segment=64, top_k=16)
    K2, V2 = W.draw_kv(w2)
    cfg = M.make_config(1, 2, 4, 512, 64, 40, 0.85, 16, max_pool_bytes=140_000)
    m = M.Mkv(cfg)
    m.compress(Kd, Vd)
    before = m.decode(q).cpu().numpy()
    with pytest.raises(M.MkvError) as e:
        m.compress(K2.to(DEV), V2.to(DEV))
    assert e.value.status == M.MKV_ERR_OOM
    after = m.decode(q).cpu().numpy()
    assert np.array_equal(before, after)
    assert m.stats()["ctx_len"] == 256
    m.close()


def test_recompress_replaces_cache(M):
    w = W.small_workload("re", ctx=300, segment=64, top_k=32)
    K, V = W.draw_kv(w)
    q = W.draw_queries(w, K)
    cfg = M.make_config(1, 2, 4, 1000, 64, 40, 0.85, 32)
    m = M.Mkv(cfg)
    w2 = W.small_workload("re2", ctx=900, segment=64, top_k=32, seed=99)
    K2, V2 = W.draw_kv(w2)
    m.compress(K2.to(DEV), V2.to(DEV))
    m.compress(K.to(DEV), V.to(DEV))
    m.T = 300
    sel = torch.empty(1, 2, 32, dtype=torch.int32, device=DEV)
    out = m.decode(q.to(DEV), sel=sel)
    torch.cuda.synchronize()
    rep = check_streams(w, K, V, q, m, out.cpu().numpy(), sel.cpu().numpy(), all_streams(w),
                        basis=False)
    _near_tie_budget(rep)
    m.close()
