"""Pins for the oracle's decode-time appends (buffer of new tokens, commit of
full segments with the stream's basis).

What fixes the expected values: textbook dense attention over the original
tokens when nothing is dropped (c = d, k = T); the prefill compression of the
concatenated tokens when the prefill ends on a segment boundary; the fp16
round-trip bound of dense rows; counting.  Planted mistakes (wrong token
order, committing with a fresh basis instead of the stream's, buffer rows not
rotated, committing one token late) must each fail a pin.
"""
import math

import numpy as np
import pytest

from oracle import mosaickv as O


def _stream(seed, T, d=16, decay=3.0):
    rng = np.random.default_rng(seed)
    Q, _ = np.linalg.qr(rng.standard_normal((d, d)))
    sig = np.exp(-np.arange(d) / decay)
    return ((rng.standard_normal((T, d)) * sig) @ Q).astype(np.float16)


def _grow(X0, Xs, S, c, tau, R=None):
    gs = O.GrownStream(base=O.compress_stream(X0, S, c, tau, R=R))
    for X in Xs:
        gs = O.append_stream(gs, X, tau)
    return gs


def test_append_rows_round_trip():
    X = _stream(1, 50)
    _, R = O.basis(X)
    rows = O.append_rows(X, R)
    back = rows @ R.T
    bound = (np.abs(R).sum(axis=1)[None, :] * np.abs(O.rotate(X, R)).max() * 2 ** -11)
    assert np.abs(back - X.astype(np.float64)).max() <= bound.max()
    assert np.array_equal(rows, O.to_fp16(O.rotate(X, R)).astype(np.float64))


def test_commit_count_and_tail_length():
    X0 = _stream(2, 40)
    gs = _grow(X0, [_stream(3, 5), _stream(4, 30), _stream(5, 1)], S=16, c=4, tau=0.9)
    assert len(gs.committed) == 2 and gs.n_tail == 36 - 32
    assert gs.T == 40 + 36
    assert O.grown_segment_starts(40, 16, 2) == [0, 16, 32, 40, 56]
    assert O.grown_dense_hat(gs).shape == (76, 16)
    # a buffer that reaches exactly S tokens is committed at once
    gs = O.append_stream(gs, _stream(10, 12), 0.9)
    assert len(gs.committed) == 3 and gs.n_tail == 0 and gs.T == 88


def test_aligned_prefill_equals_compressing_the_concatenation():
    """Prefill of 48 tokens (3 segments of 16) + 40 appended tokens in uneven
    pieces: the committed segments and the buffer must decode exactly like the
    prefill compression of all 88 tokens with the same basis (2 more full
    segments; the last 8 tokens as dense rows)."""
    X = _stream(6, 88)
    _, R = O.basis(X[:48])
    gs = _grow(X[:48], [X[48:51], X[51:70], X[70:88]], S=16, c=5, tau=0.8, R=R)
    whole = O.compress_stream(X[:80], 16, 5, 0.8, R=R)
    got = O.grown_dense_hat(gs)
    assert np.array_equal(got[:80], whole.dense_hat())
    assert np.array_equal(got[80:], O.append_rows(X[80:], R))
    for i, cs in enumerate(gs.committed):
        assert cs.segs[0].strategy == whole.segs[3 + i].strategy


def test_ragged_prefill_commits_after_its_end():
    """Prefill of 40 tokens with S = 16 ends in a ragged segment of 8; the
    first committed segment is tokens 40..55, compressed on its own."""
    X = _stream(7, 70)
    _, R = O.basis(X[:40])
    gs = _grow(X[:40], [X[40:70]], S=16, c=4, tau=0.85, R=R)
    seg = O.compress_stream(X[40:56], 16, 4, 0.85, R=R)
    assert len(gs.committed) == 1
    assert np.array_equal(O.grown_dense_hat(gs)[40:56], seg.dense_hat())
    assert np.array_equal(O.grown_dense_hat(gs)[56:], O.append_rows(X[56:], R))


def test_dense_decode_after_appends_is_textbook_attention():
    """c = d and k = T: attention over the grown stream equals softmax(q X^T /
    sqrt(d)) V over the original tokens, up to the fp16 storage of rotated
    values."""
    d, S = 16, 8
    K = _stream(8, 45, d)
    V = _stream(9, 45, d, decay=5.0)
    _, RK = O.basis(K[:20])
    _, RV = O.basis(V[:20])
    gk = _grow(K[:20], [K[20:29], K[29:45]], S, d, 0.5, R=RK)
    gv = _grow(V[:20], [V[20:29], V[29:45]], S, d, 0.5, R=RV)
    q = (K[[3, 33]].astype(np.float64) + 0.1).astype(np.float16)
    r = O.decode_stream(q, RK, RV, O.grown_dense_hat(gk), O.grown_dense_hat(gv), 45)
    lg = q.astype(np.float64) @ K.astype(np.float64).T / math.sqrt(d)
    p = np.exp(lg - lg.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    ref = p @ V.astype(np.float64)
    assert np.abs(r.out - ref).max() <= 2e-3
    assert np.array_equal(r.sel, np.arange(45))


# ---------------------------------------------------------------------------
# Planted mistakes: each must fail one of the pins above
# ---------------------------------------------------------------------------
def _planted(monkeypatch, which):
    if which == "fresh_basis":
        orig = O.compress_stream

        def commit_fresh(X, S, c, tau, R=None, **kw):
            return orig(X, S, c, tau, R=None if X.shape[0] == S else R, **kw)
        monkeypatch.setattr(O, "compress_stream", commit_fresh)
    elif which == "unrotated_tail":
        monkeypatch.setattr(O, "append_rows",
                            lambda X, R: O.to_fp16(np.asarray(X, dtype=np.float64)).astype(np.float64))
    elif which == "tail_first":
        def order(gs):
            parts = [gs.base.dense_hat()]
            if gs.n_tail:
                parts.append(O.append_rows(gs.tail, gs.base.R))
            parts += [cs.dense_hat() for cs in gs.committed]
            return np.concatenate(parts, axis=0)
        monkeypatch.setattr(O, "grown_dense_hat", order)
    elif which == "late_commit":
        orig_append = O.append_stream

        def late(gs, X_new, tau, bitmask_pv=False):
            tail = X_new if gs.tail is None else np.concatenate([gs.tail, X_new])
            committed = list(gs.committed)
            while tail.shape[0] > gs.S:
                seg, tail = tail[:gs.S], tail[gs.S:]
                committed.append(O.compress_stream(seg, gs.S, gs.base.c, tau, R=gs.base.R))
            return O.GrownStream(base=gs.base, committed=committed, tail=tail)
        monkeypatch.setattr(O, "append_stream", late)


@pytest.mark.parametrize("which", ["fresh_basis", "unrotated_tail", "tail_first", "late_commit"])
def test_planted_mistakes_are_caught(monkeypatch, which):
    _planted(monkeypatch, which)
    pins = [test_append_rows_round_trip, test_commit_count_and_tail_length,
            test_aligned_prefill_equals_compressing_the_concatenation,
            test_ragged_prefill_commits_after_its_end,
            test_dense_decode_after_appends_is_textbook_attention]
    failed = 0
    for pin in pins:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1, f"planted mistake {which} passed every pin"


def test_bitmask_commits_follow_the_prefill_rule():
    """With bitmask-indexed per-vector segments enabled, a committed segment
    is compressed by the same rule as the prefill: here (aligned prefill) the
    grown stream decodes exactly like compressing all tokens with bitmask PV
    and the same basis (fitted to the prefill only), and the committed
    segment is a PVB one (its per-token outliers keep tau per vector but not
    under one shared mask, and c = 40 > 16 makes PVB cheaper than PV)."""
    rng = np.random.default_rng(9)
    d, T, S = 128, 96, 32
    Q, _ = np.linalg.qr(rng.standard_normal((d, d)))
    Z = rng.standard_normal((T, d)) * np.where(rng.random((T, d)) < 0.05, 20.0, 1.0)
    X = (Z @ Q).astype(np.float16)
    _, R = O.basis(X[:64])
    gs = O.GrownStream(base=O.compress_stream(X[:64], S, 40, 0.8, R=R, bitmask_pv=True))
    gs = O.append_stream(gs, X[64:75], 0.8, bitmask_pv=True)
    gs = O.append_stream(gs, X[75:96], 0.8, bitmask_pv=True)
    whole = O.compress_stream(X, S, 40, 0.8, R=R, bitmask_pv=True)
    assert len(gs.committed) == 1 and gs.n_tail == 0
    assert gs.committed[0].segs[0].strategy == whole.segs[2].strategy == O.PVB
    assert np.array_equal(O.grown_dense_hat(gs), whole.dense_hat())
    # without the flag the same tokens commit as a PV segment
    plain = O.append_stream(O.GrownStream(base=O.compress_stream(X[:64], S, 40, 0.8, R=R)),
                            X[64:96], 0.8)
    assert plain.committed[0].segs[0].strategy == O.PV

