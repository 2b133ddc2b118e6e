"""Decode-time appends on the GPU against the oracle.

A prefill is compressed (ragged or on a segment boundary), then tokens are
appended in uneven pieces that cross segment boundaries three times.  After
every append the decode (selected tokens, attention output) is compared with
the oracle's decode of the grown stream given the library's bases; at the end
every committed segment's bytes are compared with the oracle's compression of
the same tokens with the stream's basis.
"""
import numpy as np
import pytest
import torch

from oracle import mosaickv as O
from parity_util import NEAR_REL, OUT_TOL, assert_budgets, compare_compressed
from two_compressed_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module")
def M():
    from two_compressed_kv_gb300 import mkv
    return mkv


def _library_hat(m, b, h, x, T0, S, c, n_commit):
    """[prefill + committed tokens, 128] from the library's exported bytes."""
    R, _, hdr, pay = m.export(b, h, x)
    nseg0 = -(-T0 // S)
    buf = np.frombuffer(pay, dtype=np.uint8)
    pre = O.unpack_stream(hdr[:nseg0], pay, T0, S, c)
    parts = [pre]
    for i in range(n_commit):
        hd = hdr[nseg0 + i:nseg0 + i + 1].copy()
        off = int(hd[0]["off16"]) * 16
        hd[0]["off16"] = 0
        parts.append(O.unpack_stream(hd, buf[off:].tobytes(), S, S, c))
    return R.astype(np.float64), np.concatenate(parts, axis=0)


@pytest.mark.parametrize("T0,pieces,bitmask", [(300, [5, 59, 1, 70, 65], False),
                                               (256, [5, 59, 1, 70, 65], False),
                                               (100, [64, 200, 130, 50], False),
                                               (256, [5, 59, 1, 70, 65], True)],
                         ids=["ragged-prefill", "aligned-prefill", "pool-growth", "bitmask-pv"])
def test_appends_across_segment_boundaries(M, T0, pieces, bitmask):
    """pool-growth: 6 commits (444 appended tokens, S = 64), more than the room
    mkv_compress reserves (2), so the pool is moved to a larger allocation
    during the appends.  bitmask-pv: MKV_FLAG_BITMASK_PV, mixed regimes, so
    that commits include bitmask-indexed per-vector segments."""
    S, c, tau, k = 64, 40, 0.85, 96
    w = W.small_workload(f"append-{T0}", n_kv_heads=2, n_q_heads=8, ctx=T0 + sum(pieces),
                         segment=S, c=c, tau=tau, top_k=k, seed=41, mixed_regimes=bitmask)
    K, V = W.draw_kv(w)
    cfg = M.make_config(w.batch, w.n_kv_heads, w.n_q_heads, w.ctx, S, c, tau, k,
                        flags=M.MKV_FLAG_BITMASK_PV if bitmask else 0)
    m = M.Mkv(cfg)
    m.compress(K[:, :, :T0].contiguous().to(DEV), V[:, :, :T0].contiguous().to(DEV))
    g = w.group
    rep = {}
    grown = {}
    for h in range(2):
        for x, X in ((0, K), (1, V)):
            R = m.export(0, h, x)[0].astype(np.float64)
            base = O.compress_stream(X[0, h, :T0].numpy(), S, c, tau, R=R, bitmask_pv=bitmask)
            grown[(h, x)] = O.GrownStream(base=base)
    T = T0
    for step, n in enumerate(pieces):
        m.append(K[:, :, T:T + n].contiguous().to(DEV), V[:, :, T:T + n].contiguous().to(DEV))
        for key in grown:
            X = K if key[1] == 0 else V
            grown[key] = O.append_stream(grown[key], X[0, key[0], T:T + n].numpy(), tau,
                                         bitmask_pv=bitmask)
        T += n
        q = W.draw_queries(w, K[:, :, :T], step=step)
        kk = min(k, T)
        sel = torch.empty(1, 2, kk, dtype=torch.int32, device=DEV)
        out = m.decode(q.to(DEV), sel=sel).cpu().numpy()
        sel = sel.cpu().numpy()
        n_commit = len(grown[(0, 0)].committed)
        assert m.stats()["ctx_len"] == T and m.n_segments() == -(-T0 // S) + n_commit
        for h in range(2):
            RK, Kp = _library_hat(m, 0, h, 0, T0, S, c, n_commit)
            RV, Vp = _library_hat(m, 0, h, 1, T0, S, c, n_commit)
            gk, gv = grown[(h, 0)], grown[(h, 1)]
            tail_k = O.append_rows(gk.tail, RK) if gk.n_tail else np.zeros((0, 128))
            tail_v = O.append_rows(gv.tail, RV) if gv.n_tail else np.zeros((0, 128))
            Kh = np.concatenate([Kp, tail_k])
            Vh = np.concatenate([Vp, tail_v])
            # the packed part is the library's own bytes; it must also equal
            # the oracle's grown stream up to stored-value rounding
            assert Kh.shape[0] == T and np.allclose(Kh, O.grown_dense_hat(gk), atol=2e-2)
            qn = q[0, h * g:(h + 1) * g].numpy()
            r = O.decode_stream(qn, RK, RV, Kh, Vh, k)
            s_all = r.scores
            sk = np.sort(s_all)[::-1][kk - 1]
            # tail rows are rounded from an fp32 rotation on the GPU: one fp16
            # step per stored value bounds their score difference
            qb = np.abs(O.rotate_queries(qn, RK).sum(axis=0))
            tail_win = (np.abs(tail_k) * 2.0 ** -10) @ qb if len(tail_k) else np.zeros(0)
            diff = np.setxor1d(sel[0, h], r.sel)
            for t in diff:
                win = NEAR_REL * abs(sk)
                if t >= T - len(tail_k):
                    win += 2 * tail_win.max()
                assert abs(s_all[t] - sk) <= win, f"step {step} head {h}: token {t} differs"
            rep["sel_near"] = rep.get("sel_near", 0) + len(diff) // 2
            rep["selected"] = rep.get("selected", 0) + kk
            qt = O.rotate_queries(qn, RK)
            ref, _ = O.attend(qt, RV, Kh, Vh, sel[0, h].astype(np.int64))
            err = float(np.abs(ref - out[0, h * g:(h + 1) * g]).max())
            rep["out_err"] = max(rep.get("out_err", 0.0), err)
            assert err <= OUT_TOL, f"step {step} head {h}: output error {err}"
    # committed segments: bytes against the oracle's compression of their tokens
    n_commit = len(grown[(0, 0)].committed)
    assert n_commit == sum(pieces) // S
    nseg0 = -(-T0 // S)
    n_pvb = 0
    for h in range(2):
        for x, X in ((0, K), (1, V)):
            R, _, hdr, pay = m.export(0, h, x)
            n_pvb += int((hdr[nseg0:nseg0 + n_commit]["strategy"] == O.PVB).sum())
            buf = np.frombuffer(pay, dtype=np.uint8)
            for i in range(n_commit):
                hd = hdr[nseg0 + i:nseg0 + i + 1].copy()
                off = int(hd[0]["off16"]) * 16
                hd[0]["off16"] = 0
                t0 = T0 + i * S
                compare_compressed(X[0, h, t0:t0 + S].numpy(), R, hd, buf[off:].tobytes(), S, c,
                                   tau, rep, bitmask)
    assert_budgets(f"appends T0={T0} commits={n_commit}" + (" bitmask" if bitmask else ""), rep)
    if bitmask:
        assert n_pvb > 0, "no committed segment used the bitmask strategy"
    # a repeated decode is bit-identical
    q = W.draw_queries(w, K, step=99)
    o1 = m.decode(q.to(DEV)).cpu()
    o2 = m.decode(q.to(DEV)).cpu()
    assert torch.equal(o1, o2)
    assert M.mkv_check_device(m.ctx) == M.MKV_OK
    m.close()


def test_append_errors_and_reset(M):
    w = W.small_workload("append-err", ctx=200, segment=64, top_k=16)
    K, V = W.draw_kv(w)
    cfg = M.make_config(1, 2, 4, 210, 64, 40, 0.85, 16)
    m = M.Mkv(cfg)
    one = K[:, :, :1].contiguous().to(DEV)
    with pytest.raises(M.MkvError) as e:          # before any compression
        m.append(one, one)
    assert e.value.status == M.MKV_ERR_STATE
    m.compress(K.to(DEV), V.to(DEV))
    m.append(K[:, :, :10].contiguous().to(DEV), V[:, :, :10].contiguous().to(DEV))
    assert m.stats()["ctx_len"] == 210
    with pytest.raises(M.MkvError) as e:          # past max_ctx
        m.append(one, one)
    assert e.value.status == M.MKV_ERR_INVALID_ARG
    assert m.stats()["ctx_len"] == 210
    m.compress(K.to(DEV), V.to(DEV))              # a new prefill drops the appended tokens
    assert m.stats()["ctx_len"] == 200
    m.close()
    # no room for appends when the prefill fills max_ctx
    m = M.Mkv(M.make_config(1, 2, 4, 200, 64, 40, 0.85, 16))
    m.compress(K.to(DEV), V.to(DEV))
    with pytest.raises(M.MkvError):
        m.append(one, one)
    m.close()
