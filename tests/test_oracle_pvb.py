"""Pins for the bitmask-indexed per-vector strategy (PVB) of the oracle.

What fixes the expected values: bytes worked out by hand for a tiny case; the
cost table; the identity between PV and PVB reconstructions (same channels,
same values, only the channel encoding differs); the choice rule (PVB wins
over PV exactly when 16 < c, loses ties to PV).  Planted mistakes (bit order
within a word reversed, word order reversed, PVB preferred on a cost tie)
must each fail a pin.
"""
import numpy as np
import pytest

from oracle import mosaickv as O


def test_bitmask_bytes_by_hand():
    P = np.array([[0, 5, 31, 32, 127], [1, 2, 3, 64, 100]])
    m = O.channel_bitmask(P)
    # row 0: word0 bits 0,5,31 = 0x80000021; word1 bit 0 = 0x1; word3 bit 31 = 0x80000000
    assert m[0].tobytes() == bytes.fromhex("21000080" "01000000" "00000000" "00000080")
    # row 1: word0 bits 1,2,3 = 0xe; word2 bit 0 = 0x1; word3 bit 4 (100 - 96) = 0x10
    assert m[1].tobytes() == bytes.fromhex("0e000000" "00000000" "01000000" "10000000")
    assert list(O.bitmask_channels(m[0])) == [0, 5, 31, 32, 127]
    assert list(O.bitmask_channels(m[1])) == [1, 2, 3, 64, 100]


def test_costs_and_choice():
    assert O.segment_cost(O.PVB, 10, 40) == 10 * (80 + 16)
    assert O.segment_cost(O.PV, 10, 40) == 800 + 400
    # c = 16: PVB and PV cost the same; the tie goes to PV
    assert O.segment_cost(O.PVB, 4, 16) == O.segment_cost(O.PV, 4, 16) == 192
    assert O.choose_strategy(0.0, 0.95, 4, 16, 0.9, bitmask_pv=True) == O.PV
    assert O.choose_strategy(0.0, 0.95, 4, 40, 0.9, bitmask_pv=True) == O.PVB
    assert O.choose_strategy(0.0, 0.95, 4, 8, 0.9, bitmask_pv=True) == O.PV
    assert O.choose_strategy(0.0, 0.95, 4, 40, 0.9) == O.PV          # off unless asked
    assert O.choose_strategy(0.95, 0.96, 4, 40, 0.9, bitmask_pv=True) == O.SM
    assert O.choose_strategy(0.0, 0.5, 4, 40, 0.9, bitmask_pv=True) == O.DENSE


def _stream(seed, T=96, d=128):
    """Flat spectrum with 5% outliers x20 at random places: per-token channels
    keep ~97% of the energy, one shared mask ~86%."""
    rng = np.random.default_rng(seed)
    Q, _ = np.linalg.qr(rng.standard_normal((d, d)))
    Z = rng.standard_normal((T, d)) * np.where(rng.random((T, d)) < 0.05, 20.0, 1.0)
    return (Z @ Q).astype(np.float16)


def test_pvb_reconstructs_like_pv_and_is_smaller():
    X = _stream(3)
    a = O.compress_stream(X, 32, 40, 0.9)
    b = O.compress_stream(X, 32, 40, 0.9, R=a.R, bitmask_pv=True)
    assert any(s.strategy == O.PV for s in a.segs), "the case must have PV segments"
    for sa, sb in zip(a.segs, b.segs):
        assert sb.strategy == (O.PVB if sa.strategy == O.PV else sa.strategy)
    assert np.array_equal(a.dense_hat(), b.dense_hat())
    ha, pa = O.pack_stream(a)
    hb, pb = O.pack_stream(b)
    n_pv = sum(s.strategy == O.PV for s in a.segs)
    assert len(pa) - len(pb) == n_pv * 32 * (40 - 16)
    assert np.array_equal(O.unpack_stream(hb, pb, 96, 32, 40), b.dense_hat())


def _planted(monkeypatch, which):
    if which == "bit_order":
        orig = O.channel_bitmask

        def rev(P):
            m = orig(P)
            return np.frombuffer(np.array([int(f"{int(w):032b}"[::-1], 2) for w in
                                           m.view("<u4").reshape(-1)], dtype="<u4").tobytes(),
                                 dtype=np.uint8).reshape(m.shape)
        monkeypatch.setattr(O, "channel_bitmask", rev)
    elif which == "word_order":
        orig = O.channel_bitmask
        monkeypatch.setattr(O, "channel_bitmask",
                            lambda P: orig(P).reshape(-1, 4, 4)[:, ::-1, :].reshape(-1, 16).copy())
    elif which == "tie_to_pvb":
        orig = O.choose_strategy

        def pref(f_sm, f_pv, rows, c, tau, d=128, bitmask_pv=False):
            r = orig(f_sm, f_pv, rows, c, tau, d, bitmask_pv)
            if (bitmask_pv and r == O.PV and
                    O.segment_cost(O.PVB, rows, c, d) == O.segment_cost(O.PV, rows, c, d)):
                return O.PVB
            return r
        monkeypatch.setattr(O, "choose_strategy", pref)


@pytest.mark.parametrize("which", ["bit_order", "word_order", "tie_to_pvb"])
def test_planted_mistakes_are_caught(monkeypatch, which):
    _planted(monkeypatch, which)
    failed = 0
    for pin in (test_bitmask_bytes_by_hand, test_costs_and_choice,
                test_pvb_reconstructs_like_pv_and_is_smaller):
        try:
            pin()
        except (AssertionError, ValueError):
            failed += 1
    assert failed >= 1, f"planted mistake {which} passed every pin"
