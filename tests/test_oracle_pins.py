"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test states what fixes the expected value: a hand-derived case
(tests/golden/), a closed form, an invariant, brute-force enumeration on a tiny
input, or a special case that reduces to textbook dense attention.  The last
group plants plausible mistakes in the oracle (on the CPU) and checks that the
pins catch every one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import mosaickv as O
from two_compressed_kv_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _frac(s):
    a, b = s.split("/") if "/" in s else (s, "1")
    return float(a) / float(b)


def _hand():
    with open(os.path.join(GOLDEN, "hand_case_d16.json")) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Hand-derived golden case: selection, statistics, strategy, layout, decode
# ---------------------------------------------------------------------------
def check_hand_case():
    g = _hand()
    p, e = g["params"], g["expected"]
    X = np.array(g["X"], dtype=np.float16)
    d = p["d"]
    I = np.eye(d)
    cs = O.compress_stream(X, p["S"], p["c"], p["tau"], R=I)
    assert np.array_equal(cs.P, np.array(e["P"])), "per-token channels"
    for si, s in enumerate(cs.segs):
        assert math.isclose(s.f_pv, _frac(e["f_pv"][si]), rel_tol=1e-15), f"f_pv seg {si}"
        assert math.isclose(s.f_sm, _frac(e["f_sm"][si]), rel_tol=1e-15), f"f_sm seg {si}"
        assert list(s.mask) == e["mask"][si], f"mask seg {si}"
        assert O.STRATEGY_NAMES[s.strategy] == e["strategy"][si], f"strategy seg {si}"
    hdr, payload = O.pack_stream(cs)
    got_h = [[int(h["off16"]), int(h["strategy"]), int(h["rows"])] for h in hdr]
    assert got_h == e["headers"], "headers"
    want = bytes.fromhex("".join(e["payload_hex"]).replace(" ", ""))
    assert payload == want, "payload bytes"
    khat = O.unpack_stream(hdr, payload, p["T"], p["S"], p["c"], d)
    assert np.array_equal(khat, cs.dense_hat()), "unpack(pack(x)) round trip"
    q = np.zeros((p["g"], d), dtype=np.float16)
    q[0, 0] = 1
    q[1, 1] = 1
    r = O.decode_stream(q, I, I, khat, khat, p["k"])
    assert np.array_equal(r.scores, np.array(e["scores"], dtype=float)), "scores"
    assert list(r.sel) == e["sel"], "selected tokens"
    want_out = np.array([[eval(x, {"e": math.e}) for x in row] for row in e["out"]])
    assert np.allclose(r.out, want_out, rtol=0, atol=1e-13), "attention output"


def test_hand_case_d16():
    check_hand_case()


# ---------------------------------------------------------------------------
# Basis: closed forms and invariants
# ---------------------------------------------------------------------------
def check_basis_closed_forms():
    # G = [[6, -2], [-2, 6]]: eigenpairs 8 -> (1, -1)/sqrt2, 4 -> (1, 1)/sqrt2.
    X = np.array([[1, 1], [1, 1], [2, -2]], dtype=np.float16)
    lam, R = O.basis(X)
    s = 1 / math.sqrt(2)
    assert np.allclose(lam, [8, 4], atol=1e-12)
    assert np.allclose(R, [[s, s], [-s, s]], atol=1e-12), "2x2 basis / sign rule"
    Xt = O.rotate(X, R)
    assert np.allclose(Xt, [[0, math.sqrt(2)], [0, math.sqrt(2)], [2 * math.sqrt(2), 0]],
                       atol=1e-12), "rotation x R"
    # Diagonal G = diag(1, 9, 4): basis is the permutation (e1, e2, e0).
    X = np.array([[0, -3, 0], [1, 0, 0], [0, 0, 2]], dtype=np.float16)
    lam, R = O.basis(X)
    assert np.allclose(lam, [9, 4, 1])
    assert np.array_equal(np.abs(R).round(12), np.array([[0, 0, 1], [1, 0, 0], [0, 1, 0]]))
    assert (R.max(axis=0) > 0).all()


def test_basis_closed_forms():
    check_basis_closed_forms()


def check_basis_invariants(X):
    lam, R = O.basis(X)
    X64 = X.astype(np.float64)
    G = X64.T @ X64
    d = R.shape[0]
    assert np.abs(R.T @ R - np.eye(d)).max() <= 1e-12, "orthogonality"
    assert np.linalg.norm(G @ R - R * lam) / np.linalg.norm(G) <= 1e-10, "eigen-residual"
    assert (np.diff(lam) <= 0).all(), "descending"
    C = O.rotate(X, R).T @ O.rotate(X, R)
    off = C - np.diag(np.diag(C))
    assert np.abs(off).max() <= 1e-9 * np.abs(C).max(), "rotated columns decorrelated"
    assert np.allclose(np.diag(C), lam, rtol=1e-9, atol=1e-9 * lam[0])
    for j in range(d):
        r = int(np.argmax(np.abs(R[:, j])))
        assert R[r, j] > 0, "sign rule"


def test_basis_invariants_random():
    rng = np.random.default_rng(5)
    X = (rng.standard_normal((700, 128)) * np.exp(-np.arange(128) / 30)).astype(np.float16)
    check_basis_invariants(X)


def test_basis_recovers_generator_rotation():
    """K = (Z*M) diag(sigma) Q_h: the leading right singular vectors span the
    leading rows of Q_h (textbook PCA of a rotated diagonal covariance).  The
    4-dimensional principal subspace is compared (single vectors can swap when
    two sample eigenvalues are close)."""
    w = W.small_workload("pin", ctx=65536, n_kv_heads=1, n_q_heads=1)
    K, _ = W.draw_kv(w)
    Q = W.haar_orthogonal(1, W._gen(w.seed, 0, 11, "cpu"))[0].double().numpy()
    _, R = O.basis(K[0, 0].numpy())
    P = R[:, :4].T @ Q[:4].T
    assert (P ** 2).sum() / 4 >= 0.98
    assert abs(float(R[:, 0] @ Q[0])) >= 0.99


# ---------------------------------------------------------------------------
# Selection: brute force on tiny inputs with exact ties
# ---------------------------------------------------------------------------
def _brute_topc(v, c):
    """Max-energy c-subset; among equal energies the lexicographically
    smallest index tuple (which is what 'ties to the lower channel' gives)."""
    best = None
    for sub in itertools.combinations(range(len(v)), c):
        en = sum(int(v[j]) ** 2 for j in sub)
        key = (-en, sub)
        if best is None or key < best:
            best = key
    return list(best[1])


def test_top_c_bruteforce():
    rng = np.random.default_rng(1)
    V = rng.integers(-4, 5, size=(60, 8))
    for row in V:
        assert list(O.top_c_channels(row.astype(float), 3)) == _brute_topc(row, 3)


def test_segment_mask_bruteforce():
    rng = np.random.default_rng(2)
    for _ in range(40):
        seg = rng.integers(-3, 4, size=(5, 8)).astype(float)
        P = O.top_c_channels(seg, 3)
        st = O.segment_stats(seg, P, 3)
        col = (seg ** 2).sum(axis=0)
        brute = max(itertools.combinations(range(8), 3),
                    key=lambda s: (sum(col[j] for j in s), [-j for j in s]))
        assert list(st.mask) == sorted(brute)
        if st.e_tot > 0:
            assert st.f_sm <= st.f_pv + 1e-15, "shared mask never beats per-vector"


def test_top_k_counting_definition():
    rng = np.random.default_rng(3)
    for T, k in [(50, 1), (50, 7), (50, 50), (50, 80), (9, 4)]:
        s = rng.integers(-5, 6, size=T).astype(float)
        sel = O.top_k_tokens(s, k)
        kk = min(k, T)
        want = [t for t in range(T)
                if sum(1 for u in range(T) if s[u] > s[t] or (s[u] == s[t] and u < t)) < kk]
        assert list(sel) == want
    s = rng.standard_normal(100)
    assert list(O.top_k_tokens(s, 1)) == [int(np.argmax(s))]


# ---------------------------------------------------------------------------
# Strategy costs and choice (hand table)
# ---------------------------------------------------------------------------
def check_costs_and_choice():
    # (strategy, rows, c) -> bytes, worked by hand from the layout
    table = [(O.SM, 128, 40, 48 + 10240), (O.PV, 128, 40, 10240 + 5120),
             (O.DENSE, 128, 40, 32768), (O.SM, 1, 8, 32), (O.PV, 1, 8, 32),
             (O.PV, 3, 8, 48 + 32), (O.SM, 64, 64, 64 + 8192), (O.PV, 44, 40, 3520 + 1760)]
    for st, rows, c, want in table:
        assert O.segment_cost(st, rows, c) == want
    assert O.choose_strategy(0.95, 0.97, 128, 40, 0.9) == O.SM
    assert O.choose_strategy(0.80, 0.97, 128, 40, 0.9) == O.PV
    assert O.choose_strategy(0.80, 0.85, 128, 40, 0.9) == O.DENSE
    assert O.choose_strategy(0.9, 0.9, 128, 40, 0.9) == O.SM            # inclusive
    assert O.choose_strategy(1.0, 1.0, 1, 8, 0.9) == O.SM               # SM/PV tie -> SM
    assert O.choose_strategy(1.0, 1.0, 16, 128, 0.5) == O.DENSE         # c = d: dense cheapest


def test_costs_and_choice():
    check_costs_and_choice()


# ---------------------------------------------------------------------------
# Reduction to textbook dense attention (c = d, k = T), basis invariance,
# dense round trip
# ---------------------------------------------------------------------------
def _dense_attention(q, K, V):
    q = q.astype(np.float64)
    K = K.astype(np.float64)
    V = V.astype(np.float64)
    lg = q @ K.T / math.sqrt(K.shape[1])
    lg -= lg.max(axis=1, keepdims=True)
    p = np.exp(lg)
    p /= p.sum(axis=1, keepdims=True)
    return p @ V


@pytest.mark.parametrize("T,S", [(256, 64), (200, 48)])
def test_dense_attention_reduction(T, S):
    w = W.small_workload("dense", ctx=T, n_kv_heads=1, n_q_heads=4)
    K, V = W.draw_kv(w)
    q = W.draw_queries(w, K)[0].numpy()
    K, V = K[0, 0].numpy(), V[0, 0].numpy()
    ck = O.compress_stream(K, S, 128, 0.85)
    cv = O.compress_stream(V, S, 128, 0.85)
    assert all(s.strategy == O.DENSE for s in ck.segs + cv.segs)
    r = O.decode_stream(q, ck.R, cv.R, ck.dense_hat(), cv.dense_hat(), T)
    assert np.abs(r.out - _dense_attention(q, K, V)).max() <= 2e-3
    # any orthonormal basis gives the same result up to fp16 storage rounding
    Qr = np.linalg.qr(np.random.default_rng(0).standard_normal((128, 128)))[0]
    ck2 = O.compress_stream(K, S, 128, 0.85, R=Qr)
    cv2 = O.compress_stream(V, S, 128, 0.85, R=np.eye(128))
    r2 = O.decode_stream(q, ck2.R, cv2.R, ck2.dense_hat(), cv2.dense_hat(), T)
    assert np.abs(r2.out - r.out).max() <= 2e-3


def test_dense_segment_round_trip():
    w = W.small_workload("rt", ctx=128, n_kv_heads=1, n_q_heads=1)
    K, _ = W.draw_kv(w)
    X = K[0, 0].numpy()
    cs = O.compress_stream(X, 32, 8, 1.0)       # tau = 1 with c < d: dense segments
    assert all(s.strategy == O.DENSE for s in cs.segs)
    hdr, payload = O.pack_stream(cs)
    vals = np.frombuffer(payload, dtype="<f2").reshape(128, 128)
    assert np.array_equal(vals.view(np.uint16), O.to_fp16(cs.Xt).view(np.uint16))
    xhat = O.unpack_stream(hdr, payload, 128, 32, 8) @ cs.R.T
    ulp = np.spacing(np.abs(O.to_fp16(cs.Xt)).astype(np.float16)).astype(np.float64)
    bound = (ulp / 2) @ np.abs(cs.R.T) + 1e-12
    assert (np.abs(xhat - X.astype(np.float64)) <= bound).all()


def test_retained_energy_and_ragged_tail():
    w = W.small_workload("ret", ctx=300, n_kv_heads=1, n_q_heads=1)
    K, V = W.draw_kv(w)
    for X in (K[0, 0].numpy(), V[0, 0].numpy()):
        cs = O.compress_stream(X, 64, 40, 0.85)
        assert [s.rows for s in cs.segs] == [64, 64, 64, 64, 44]
        for s in cs.segs:
            assert s.f_sm <= s.f_pv + 1e-12
            f = {O.SM: s.f_sm, O.PV: s.f_pv, O.DENSE: 1.0}[s.strategy]
            assert f >= np.float32(0.85)
        hdr, payload = O.pack_stream(cs)
        assert len(payload) == sum(O.segment_cost(s.strategy, s.rows, 40) for s in cs.segs)
        assert int(hdr[-1]["rows"]) == 44


def test_energy_identity():
    rng = np.random.default_rng(4)
    X = rng.standard_normal((50, 128)).astype(np.float16)
    cs = O.compress_stream(X, 16, 40, 0.5)
    assert np.allclose((cs.Xt ** 2).sum(1), (X.astype(np.float64) ** 2).sum(1), rtol=1e-12)
    for (a, b), s in zip(O.segment_bounds(50, 16), cs.segs):
        assert math.isclose(s.e_tot, float((X[a:b].astype(np.float64) ** 2).sum()), rel_tol=1e-12)


def check_gqa_closed_form():
    """Query head i attends with KV head i // g, pinned without restating the
    rule: when every V row of KV head h equals one vector a_h, each query
    head's output is a_(i // g) whatever its weights (they sum to one), and
    another mapping (i mod H) would return the other vector for head 1."""
    T, H, g = 64, 2, 3
    rng = np.random.default_rng(5)
    K = rng.standard_normal((1, H, T, 128)).astype(np.float16)
    a = np.stack([rng.standard_normal(128), 3.0 + rng.standard_normal(128)])
    V = np.broadcast_to(a[None, :, None, :], (1, H, T, 128)).astype(np.float16)
    q = rng.standard_normal((1, H * g, 128)).astype(np.float16)
    layer = O.compress_layer(K, np.ascontiguousarray(V), 32, 40, 0.85)
    out, _, _ = O.decode_layer(layer, q, 16)
    a16 = a.astype(np.float16).astype(np.float64)
    for i in range(H * g):
        assert np.abs(out[0, i] - a16[i // g]).max() <= 2e-2, i
    assert np.abs(out[0, 1] - a16[1 % H]).max() > 1.0


def test_gqa_mapping_closed_form():
    check_gqa_closed_form()


def test_gqa_head_mapping():
    """Query head i attends with KV head i // g (g = Hq / H)."""
    w = W.small_workload("gqa", ctx=96, n_kv_heads=2, n_q_heads=6)
    K, V = W.draw_kv(w)
    q = W.draw_queries(w, K).numpy()
    layer = O.compress_layer(K.numpy(), V.numpy(), 32, 40, 0.85)
    out, sel, scores = O.decode_layer(layer, q, 20)
    for i in range(6):
        h = i // 3
        ck, cv = layer.K[0][h], layer.V[0][h]
        r = O.decode_stream(q[0, h * 3:(h + 1) * 3], ck.R, cv.R, ck.dense_hat(), cv.dense_hat(), 20)
        assert np.array_equal(out[0, i], r.out[i - 3 * h])
    # the summed score equals the score of the summed rotated query
    ck = layer.K[0][1]
    qt = q[0, 3:6].astype(np.float64) @ ck.R
    assert np.allclose(scores[0, 1], ck.dense_hat() @ qt.sum(0), rtol=1e-12, atol=1e-9)


def check_zero_energy():
    """A stream with no energy (all zeros): every retained fraction is 1 by the
    rule for an empty segment, every per-token and shared channel choice is a
    tie resolved to the lowest channels, SM and PV cost the same here and the
    tie goes to SM; all scores are 0, so the first k tokens are selected and
    the softmax is uniform (all logits 0), giving a zero output."""
    d, T, S, c, k = 16, 10, 4, 4, 3
    X = np.zeros((T, d), dtype=np.float16)
    I = np.eye(d)
    cs = O.compress_stream(X, S, c, 0.9, R=I)
    assert np.array_equal(cs.P, np.tile(np.arange(c), (T, 1)))
    for seg in cs.segs:
        assert seg.e_tot == 0.0 and seg.f_pv == 1.0 and seg.f_sm == 1.0
        assert list(seg.mask) == list(range(c))
        assert O.segment_cost(O.SM, seg.rows, c, d) == O.segment_cost(O.PV, seg.rows, c, d)
        assert seg.strategy == O.SM
    hdr, payload = O.pack_stream(cs)
    want = b""
    for rows in (4, 4, 2):
        want += bytes(range(c)) + bytes(16 - c) + bytes(2 * c * rows)
    assert payload == want
    assert [int(h["off16"]) for h in hdr] == [0, 3, 6]
    q = np.ones((2, d), dtype=np.float16)
    khat = O.unpack_stream(hdr, payload, T, S, c, d)
    r = O.decode_stream(q, I, I, khat, khat, k)
    assert list(r.sel) == [0, 1, 2]
    assert np.all(r.scores == 0.0) and np.all(r.logits == 0.0)
    assert np.all(r.out == 0.0)


def test_zero_energy_stream_closed_form():
    check_zero_energy()


def test_kv_size_arithmetic_from_paper():
    """§1 and §2.1 of the paper: eight Llama-3.1-8B requests at 128K tokens need
    128 GB of KV cache, and 1 TB at 1M tokens (fp16, 32 layers, 8 KV heads)."""
    with open(os.path.join(GOLDEN, "kv_cache_size.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        got = W.kv_cache_bytes(case["requests"], case["tokens"], 32, 8)
        assert got == case["bytes"]


# ---------------------------------------------------------------------------
# Planted mistakes: every one must be caught by the pins above
# ---------------------------------------------------------------------------
def _mut_rotate_transposed(mp):
    mp.setattr(O, "rotate", lambda X, R: np.asarray(X, np.float64) @ np.asarray(R, np.float64).T)


def _mut_ties_high(mp):
    def f(values, c):
        v = np.atleast_2d(np.abs(np.asarray(values, dtype=np.float64)))[:, ::-1]
        order = v.shape[1] - 1 - np.argsort(-v, axis=1, kind="stable")[:, :c]
        out = np.sort(order, axis=1)
        return out[0] if np.ndim(values) == 1 else out
    mp.setattr(O, "top_c_channels", f)


def _mut_most_retained(mp):
    def f(f_sm, f_pv, rows, c, tau, d=128, bitmask_pv=False):
        return O.PV if f_pv >= tau else (O.SM if f_sm >= tau else O.DENSE)
    mp.setattr(O, "choose_strategy", f)


def _mut_topk_ties_high(mp):
    def f(s, k):
        T = s.shape[0]
        order = np.lexsort((-np.arange(T), -np.asarray(s, dtype=np.float64)))
        return np.sort(order[:min(k, T)])
    mp.setattr(O, "top_k_tokens", f)


def _mut_no_scale(mp):
    orig = O.decode_stream

    def f(q, R_K, R_V, K_hat, V_hat, k):
        return orig(np.asarray(q, np.float64) * math.sqrt(np.atleast_2d(q).shape[1]) ** 0.5,
                    R_K, R_V, K_hat, V_hat, k)
    mp.setattr(O, "decode_stream", f)


def _mut_sign_flipped(mp):
    orig = O.basis

    def f(X):
        lam, R = orig(X)
        return lam, -R
    mp.setattr(O, "basis", f)


def _mut_ascending(mp):
    orig = O.basis

    def f(X):
        lam, R = orig(X)
        return lam[::-1].copy(), R[:, ::-1].copy()
    mp.setattr(O, "basis", f)


def _mut_stats_drop_pad(mp):
    orig = O.segment_cost

    def f(strategy, rows, c, d=128):
        v = orig(strategy, rows, c, d)
        return v - (O.pad16(c) if strategy == O.SM else 0)
    mp.setattr(O, "segment_cost", f)


def _mut_empty_segment_unkept(mp):
    orig = O.segment_stats

    def f(Xt_seg, P_seg, c):
        st = orig(Xt_seg, P_seg, c)
        if st.e_tot == 0.0:
            st.f_pv = st.f_sm = 0.0
        return st
    mp.setattr(O, "segment_stats", f)


def _mut_gqa_interleaved(mp):
    """query head i attends with KV head i mod H instead of i // g"""
    def wrong(layer, q, k):
        B, Hq, d = q.shape
        kk = min(k, layer.T)
        out = np.zeros((B, Hq, d))
        sel = np.zeros((B, layer.H, kk), dtype=np.int64)
        scores = np.zeros((B, layer.H, layer.T))
        for b in range(B):
            for h in range(layer.H):
                heads = np.arange(h, Hq, layer.H)
                ck, cv = layer.K[b][h], layer.V[b][h]
                r = O.decode_stream(q[b, heads], ck.R, cv.R, ck.dense_hat(), cv.dense_hat(), k)
                out[b, heads] = r.out
                sel[b, h] = r.sel
                scores[b, h] = r.scores
        return out, sel, scores
    mp.setattr(O, "decode_layer", wrong)


MUTATIONS = [_mut_rotate_transposed, _mut_ties_high, _mut_most_retained, _mut_topk_ties_high,
             _mut_no_scale, _mut_sign_flipped, _mut_ascending, _mut_stats_drop_pad,
             _mut_empty_segment_unkept, _mut_gqa_interleaved]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=[m.__name__ for m in MUTATIONS])
def test_pins_catch_planted_mistake(mutation, monkeypatch):
    mutation(monkeypatch)
    rng = np.random.default_rng(5)
    Xr = (rng.standard_normal((300, 16)) * np.exp(-np.arange(16) / 4)).astype(np.float16)
    checks = [check_hand_case, check_basis_closed_forms, check_costs_and_choice,
              lambda: check_basis_invariants(Xr), check_zero_energy, check_gqa_closed_form]
    caught = 0
    for chk in checks:
        try:
            chk()
        except AssertionError:
            caught += 1
    assert caught >= 1, "no pin caught the planted mistake"
