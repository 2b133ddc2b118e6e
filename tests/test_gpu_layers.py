"""mkv_decode_layers: the decode steps of several layers with one launch of
each decode kernel.  The fused call must return exactly what mkv_decode
returns layer by layer (same kernels, same arithmetic order), and match the
oracle's decode on sampled streams."""
import dataclasses

import pytest
import torch

from test_gpu_parity import _near_tie_budget, check_streams
from two_compressed_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def M():
    from two_compressed_kv_gb300 import mkv
    return mkv


def _layers(M, w, n, dense_first=False, max_ctx=None):
    """n ctxs of w's shape, layer l drawn as layer l of w; with dense_first the
    first layer uses the mixed regimes (dense segments), the others do not."""
    cfg = M.make_config(w.batch, w.n_kv_heads, w.n_q_heads, max_ctx or w.ctx, w.segment, w.c,
                        w.tau, w.top_k)
    ms, data = [], []
    for l in range(n):
        wl = dataclasses.replace(w, mixed_regimes=bool(dense_first and l == 0))
        K, V = W.draw_kv(wl, layer=l)
        q = W.draw_queries(wl, K, layer=l)
        m = M.Mkv(cfg)
        m.compress(K.to(DEV), V.to(DEV))
        ms.append(m)
        data.append((wl, K, V, q.to(DEV)))
    return ms, data


def _per_layer_and_fused(M, ms, data):
    kk = ms[0].stats()["ctx_len"]
    w = data[0][0]
    kk = min(w.top_k, kk)
    ref = []
    for m, (_, _, _, q) in zip(ms, data):
        sel = torch.empty(w.batch, w.n_kv_heads, kk, dtype=torch.int32, device=DEV)
        out = m.decode(q, sel=sel)
        ref.append((out, sel))
    outs = [torch.full_like(o, float("nan")) for o, _ in ref]
    sels = [torch.full_like(s, -7) for _, s in ref]
    M.mkv_decode_layers([m.ctx for m in ms], [d[3] for d in data], outs, sels)
    torch.cuda.synchronize()
    return ref, outs, sels


def test_fused_equals_per_layer_and_oracle(M):
    w = W.small_workload("fused", batch=2, n_kv_heads=2, n_q_heads=8, ctx=700, segment=64, c=40,
                         tau=0.9, top_k=48)
    ms, data = _layers(M, w, 3, dense_first=True)
    dense = [m.stats()["strategy_count"][0][2] + m.stats()["strategy_count"][1][2] for m in ms]
    assert dense[0] > 0 and min(dense[1:]) == 0, dense     # slots of different widths
    ref, outs, sels = _per_layer_and_fused(M, ms, data)
    for (o, s), fo, fs in zip(ref, outs, sels):
        assert torch.equal(o, fo)
        assert torch.equal(s, fs)
    # the fused outputs of two layers against the oracle
    for l in (0, 2):
        wl, K, V, q = data[l]
        rep = check_streams(wl, K, V, q.cpu(), ms[l], outs[l].cpu().numpy(), sels[l].cpu().numpy(),
                            [(1, 1), (0, 0)], basis=False)
        _near_tie_budget(rep, f"fused layer {l}")
    for m in ms:
        m.close()


def test_fused_after_appends(M):
    w = W.small_workload("fused-append", batch=1, n_kv_heads=2, n_q_heads=4, ctx=300, segment=64,
                         c=40, tau=0.9, top_k=40)
    ms, data = _layers(M, w, 2, max_ctx=600)
    for l, m in enumerate(ms):
        wl = dataclasses.replace(w, ctx=150)
        K2, V2 = W.draw_kv(wl, layer=10 + l)
        m.append(K2.to(DEV), V2.to(DEV))
    assert ms[0].stats()["ctx_len"] == 450
    ref, outs, sels = _per_layer_and_fused(M, ms, data)
    for (o, s), fo, fs in zip(ref, outs, sels):
        assert torch.equal(o, fo)
        assert torch.equal(s, fs)
    for m in ms:
        m.close()


def test_fused_32k_layers(M):
    """Four layers of the 32K batch-4 shape: fused == per layer."""
    w = W.LAYER_32K
    ms, data = _layers(M, w, 4)
    ref, outs, sels = _per_layer_and_fused(M, ms, data)
    for (o, s), fo, fs in zip(ref, outs, sels):
        assert torch.equal(o, fo)
        assert torch.equal(s, fs)
    for m in ms:
        m.close()
    torch.cuda.empty_cache()


def test_fused_rejects_mismatches(M):
    w = W.small_workload("fused-bad", ctx=300, top_k=32)
    ms, data = _layers(M, w, 2)
    q = data[0][3]
    out = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    # a ctx twice
    with pytest.raises(M.MkvError) as e:
        M.mkv_decode_layers([ms[0].ctx, ms[0].ctx], [q, q], [out, out])
    assert e.value.status == M.MKV_ERR_INVALID_ARG
    # another context length
    w2 = dataclasses.replace(w, ctx=256)
    other, _ = _layers(M, w2, 1, max_ctx=300)
    with pytest.raises(M.MkvError) as e:
        M.mkv_decode_layers([ms[0].ctx, other[0].ctx], [q, q], [out, out])
    assert e.value.status == M.MKV_ERR_INVALID_ARG
    # a ctx without a cache
    cfg = M.make_config(w.batch, w.n_kv_heads, w.n_q_heads, w.ctx, w.segment, w.c, w.tau, w.top_k)
    empty = M.Mkv(cfg)
    with pytest.raises(M.MkvError) as e:
        M.mkv_decode_layers([ms[0].ctx, empty.ctx], [q, q], [out, out])
    assert e.value.status == M.MKV_ERR_STATE
    # too many layers
    assert M.mkv_decode_layers_raw([ms[0].ctx.value] * 65, 65, [q.data_ptr()] * 65,
                                   [out.data_ptr()] * 65) == M.MKV_ERR_INVALID_ARG
    # the ctxs still decode afterwards
    o2 = torch.empty_like(out)
    M.mkv_decode_layers([ms[0].ctx, ms[1].ctx], [q, data[1][3]], [out, o2])
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(o2).all()
    for m in ms + other + [empty]:
        m.close()
