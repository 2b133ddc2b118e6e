"""Oracle: a plain, slow, fp64 CPU restatement of MosaicKV's decode path over a
two-D compressed KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the tests, the smoke check and the benchmark's CPU
baseline leg do.  It shares no code with the CUDA library.

Source: "MosaicKV: Serving Long-Context LLM with Dynamic Two-D KV Cache
Compression" (arXiv 2607.00760).  The paper's text available here covers the
abstract and §1 Introduction; the method is described there in one paragraph
each, so every concrete rule below is the plainest reading of those paragraphs,
and each reading is marked READING.

  * §1, "Observation & Method 1: dynamic two-D compression": KV vectors are
    rotated by an SVD basis; important elements are picked per vector
    ("per-vector element selection"); the cache is cut into segments and each
    segment gets a suitable compression strategy ("dynamic compression
    strategy").
  * §1, prior-work paragraph: ThinK applies one channel mask to all key vectors
    (the segment-shared mask strategy here), Quest selects tokens per query at
    run time (the top-k token selection here).
  * §1, "Observation & Method 2: compressed KV cache management": the sparse
    KV matrix is packed into a dense format in GPU memory and attention runs on
    it without unpacking (the packed layout here).

Notation: a stream is one (batch b, KV head h, X in {K, V}); X is [T, d] with
fp16 entries (converted exactly to fp64 here); d = 128 in the library, any d
here so that tiny hand-checkable cases can be written.  S = segment size,
c = kept channels, tau = retained-energy threshold, k = token budget,
g = query heads per KV head.

Functions whose results have no independent pin are marked "parity unpinned"
in their docstring.  At present every function is pinned by a test in
tests/test_oracle_pins.py (the append functions by tests/test_oracle_append.py).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

SM, PV, DENSE, PVB = 0, 1, 2, 3
STRATEGY_NAMES = {SM: "SM", PV: "PV", DENSE: "D", PVB: "PVB"}
HEADER_DTYPE = np.dtype([("off16", "<u4"), ("strategy", "u1"), ("rsv", "u1"), ("rows", "<u2")])


def pad16(n: int) -> int:
    return (int(n) + 15) // 16 * 16


# ---------------------------------------------------------------------------
# Step 1: per-stream SVD basis  (§1 Observation & Method 1: "SVD rotation")
# ---------------------------------------------------------------------------
def basis(X: np.ndarray):
    """Right singular vectors of X, i.e. eigenvectors of G = X^T X.

    READING: no mean-centering (an SVD, not a PCA); eigenvalues in descending
    order, equal eigenvalues keep the solver's order; each column's entry of
    largest magnitude is made positive, the lowest row winning a magnitude tie.
    Returns (lam [d] descending, R [d, d], columns = basis vectors)."""
    X64 = np.asarray(X, dtype=np.float64)
    G = X64.T @ X64
    lam, E = np.linalg.eigh(G)
    order = np.argsort(-lam, kind="stable")
    lam = lam[order]
    E = E[:, order].copy()
    for j in range(E.shape[1]):
        r = int(np.argmax(np.abs(E[:, j])))        # first (lowest) row on ties
        if E[r, j] < 0:
            E[:, j] = -E[:, j]
    return lam, E


# ---------------------------------------------------------------------------
# Step 2: rotation and fp16 storage rounding
# ---------------------------------------------------------------------------
def rotate(X: np.ndarray, R: np.ndarray) -> np.ndarray:
    """x~_t = x_t R (row vectors), fp64."""
    return np.asarray(X, dtype=np.float64) @ np.asarray(R, dtype=np.float64)


def to_fp16(x: np.ndarray) -> np.ndarray:
    """Storage rounding: fp16, round-to-nearest-even (READING)."""
    return np.asarray(x, dtype=np.float64).astype(np.float16)


# ---------------------------------------------------------------------------
# Step 3: per-vector element selection and per-segment statistics
# ---------------------------------------------------------------------------
def top_c_channels(values: np.ndarray, c: int) -> np.ndarray:
    """Indices of the c entries of largest magnitude in each row of `values`
    (ties go to the lower channel), returned in ascending channel order.

    Works on a 1-D vector or row-wise on a 2-D array."""
    v = np.atleast_2d(np.abs(np.asarray(values, dtype=np.float64)))
    order = np.argsort(-v, axis=1, kind="stable")[:, :c]
    out = np.sort(order, axis=1)
    return out[0] if np.ndim(values) == 1 else out


def segment_bounds(T: int, S: int):
    """[(start, end)] of each segment; the last one holds T mod S rows when S
    does not divide T (READING)."""
    return [(a, min(T, a + S)) for a in range(0, T, S)]


@dataclass
class SegmentStats:
    rows: int
    e_tot: float
    f_pv: float
    f_sm: float
    mask: np.ndarray           # segment-shared channels (ascending), length c
    strategy: int = -1


def segment_stats(Xt_seg: np.ndarray, P_seg: np.ndarray, c: int) -> SegmentStats:
    """Retained-energy fractions of one segment.

    f_PV: energy kept when every token keeps its own top-c channels.
    f_SM: energy kept by the c channels with the largest column energy
          (ties to the lower channel), shared by every token of the segment.
    Both are 1 when the segment has no energy (READING)."""
    sq = Xt_seg * Xt_seg
    e_tot = float(sq.sum())
    kept = float(np.take_along_axis(sq, P_seg, axis=1).sum())
    col = sq.sum(axis=0)
    mask = top_c_channels(col, c)
    if e_tot > 0.0:
        f_pv = kept / e_tot
        f_sm = float(col[mask].sum()) / e_tot
    else:
        f_pv = f_sm = 1.0
    return SegmentStats(rows=Xt_seg.shape[0], e_tot=e_tot, f_pv=f_pv, f_sm=f_sm, mask=mask)


# ---------------------------------------------------------------------------
# Step 4: strategy choice and packed sizes (§1 Observation & Method 1/2)
# ---------------------------------------------------------------------------
def segment_cost(strategy: int, rows: int, c: int, d: int = 128) -> int:
    """Packed bytes of one segment (READING: the cost that "cheapest" means).

    SM : c uint8 channel indices padded to 16 B, then rows x c fp16 values.
    PV : rows x c fp16 values, then rows x c uint8 indices padded to 16 B.
    D  : rows x d fp16 values.
    PVB: rows x c fp16 values, then one 16-byte channel bitmask per row
         (READING of the pages' open "suitable strategy": the per-vector
         selection with its channels as a bitmask, cheaper than c index bytes
         when c > 16)."""
    if strategy == SM:
        return pad16(c) + 2 * c * rows
    if strategy == PV:
        return 2 * c * rows + pad16(c * rows)
    if strategy == DENSE:
        return 2 * d * rows
    if strategy == PVB:
        return 2 * c * rows + 16 * rows
    raise ValueError(strategy)


def choose_strategy(f_sm: float, f_pv: float, rows: int, c: int, tau: float, d: int = 128,
                    bitmask_pv: bool = False) -> int:
    """The cheapest strategy whose retained fraction is >= tau; dense is always
    allowed; equal costs resolve in the order SM, PV, PVB, D (READING).  PVB
    (per-vector channels as a bitmask) is a candidate only when bitmask_pv;
    it keeps exactly PV's channels, so it is eligible whenever PV is."""
    order = {SM: 0, PV: 1, PVB: 2, DENSE: 3}
    cands = []
    if f_sm >= tau:
        cands.append((segment_cost(SM, rows, c, d), order[SM], SM))
    if f_pv >= tau:
        cands.append((segment_cost(PV, rows, c, d), order[PV], PV))
        if bitmask_pv:
            cands.append((segment_cost(PVB, rows, c, d), order[PVB], PVB))
    cands.append((segment_cost(DENSE, rows, c, d), order[DENSE], DENSE))
    return min(cands)[2]


@dataclass
class CompressedStream:
    """Logical content of one compressed stream."""
    T: int
    d: int
    S: int
    c: int
    R: np.ndarray                       # [d, d] basis actually used
    lam: Optional[np.ndarray]           # eigenvalues (None when the basis was given)
    Xt: np.ndarray                      # [T, d] fp64 rotated values (unrounded)
    P: np.ndarray                       # [T, c] per-token top-c channels (ascending)
    segs: List[SegmentStats] = field(default_factory=list)

    def kept_channels(self, t: int) -> np.ndarray:
        s = self.segs[t // self.S]
        if s.strategy == SM:
            return s.mask
        if s.strategy in (PV, PVB):
            return self.P[t]
        return np.arange(self.d)

    def dense_hat(self) -> np.ndarray:
        """[T, d] fp64 of the stored fp16 values on kept channels, 0 elsewhere."""
        out = np.zeros((self.T, self.d))
        q16 = to_fp16(self.Xt).astype(np.float64)
        for si, (a, b) in enumerate(segment_bounds(self.T, self.S)):
            st = self.segs[si].strategy
            if st == DENSE:
                out[a:b] = q16[a:b]
            elif st == SM:
                m = self.segs[si].mask
                out[a:b, m] = q16[a:b][:, m]
            else:
                rows = np.arange(a, b)[:, None]
                out[rows, self.P[a:b]] = q16[rows, self.P[a:b]]
        return out


def compress_stream(X: np.ndarray, S: int, c: int, tau: float,
                    R: Optional[np.ndarray] = None, bitmask_pv: bool = False) -> CompressedStream:
    """Steps 1-4 for one stream.  `R` (an orthonormal basis) replaces step 1
    when given; the parity tests use that to check the steps that follow a
    basis produced elsewhere (a basis is only unique up to column signs and
    rotations inside degenerate eigenspaces)."""
    X = np.asarray(X)
    T, d = X.shape
    lam = None
    if R is None:
        lam, R = basis(X)
    R = np.asarray(R, dtype=np.float64)
    Xt = rotate(X, R)
    P = top_c_channels(Xt, c)
    cs = CompressedStream(T=T, d=d, S=S, c=c, R=R, lam=lam, Xt=Xt, P=P)
    tau = float(np.float32(tau))            # the threshold is an fp32 value (READING)
    for (a, b) in segment_bounds(T, S):
        st = segment_stats(Xt[a:b], P[a:b], c)
        st.strategy = choose_strategy(st.f_sm, st.f_pv, b - a, c, tau, d, bitmask_pv)
        cs.segs.append(st)
    return cs


# ---------------------------------------------------------------------------
# Packed layout (§1 Observation & Method 2: sparse KV packed dense)
# ---------------------------------------------------------------------------
def channel_bitmask(P: np.ndarray) -> np.ndarray:
    """16-byte little-endian channel bitmask of each row of channel lists P
    ([rows, c]): bit j % 32 of 32-bit word j // 32 is set for every channel j
    in the row."""
    rows = P.shape[0]
    words = np.zeros((rows, 4), dtype=np.uint64)
    for r in range(rows):
        for j in P[r]:
            words[r, int(j) // 32] |= np.uint64(1) << np.uint64(int(j) % 32)
    return words.astype("<u4").view(np.uint8).reshape(rows, 16)


def bitmask_channels(mask16: np.ndarray) -> np.ndarray:
    """Ascending channels whose bits are set in one 16-byte bitmask."""
    words = np.frombuffer(np.ascontiguousarray(mask16).tobytes(), dtype="<u4")
    return np.array([32 * w + b for w in range(4) for b in range(32)
                     if (int(words[w]) >> b) & 1], dtype=np.int64)


def pack_stream(cs: CompressedStream):
    """(headers, payload bytes) of one stream.

    Header per segment: {uint32 off16, uint8 strategy, uint8 0, uint16 rows};
    off16 = payload offset / 16 from the stream's first byte.  Values are
    fp16 (RNE) in ascending channel order; channel indices are uint8."""
    c, d = cs.c, cs.d
    q16 = to_fp16(cs.Xt)
    hdr = np.zeros(len(cs.segs), dtype=HEADER_DTYPE)
    chunks = []
    off = 0
    for si, (a, b) in enumerate(segment_bounds(cs.T, cs.S)):
        s = cs.segs[si]
        rows = b - a
        if s.strategy == SM:
            idx = np.zeros(pad16(c), dtype=np.uint8)
            idx[:c] = s.mask
            vals = q16[a:b][:, s.mask]
            blob = idx.tobytes() + vals.astype("<f2").tobytes()
        elif s.strategy == PV:
            P = cs.P[a:b]
            vals = np.take_along_axis(q16[a:b], P, axis=1)
            idx = np.zeros(pad16(c * rows), dtype=np.uint8)
            idx[:c * rows] = P.reshape(-1)
            blob = vals.astype("<f2").tobytes() + idx.tobytes()
        elif s.strategy == PVB:
            P = cs.P[a:b]
            vals = np.take_along_axis(q16[a:b], P, axis=1)
            blob = vals.astype("<f2").tobytes() + channel_bitmask(P).tobytes()
        else:
            blob = q16[a:b].astype("<f2").tobytes()
        assert len(blob) == segment_cost(s.strategy, rows, c, d)
        hdr[si] = (off // 16, s.strategy, 0, rows)
        chunks.append(blob)
        off += len(blob)
    return hdr, b"".join(chunks)


def unpack_stream(hdr: np.ndarray, payload: bytes, T: int, S: int, c: int, d: int = 128) -> np.ndarray:
    """Inverse of the layout: [T, d] fp64 with stored values on kept channels
    and zeros elsewhere.  Validates every header against the layout."""
    buf = np.frombuffer(payload, dtype=np.uint8)
    out = np.zeros((T, d))
    for si, (a, b) in enumerate(segment_bounds(T, S)):
        off = int(hdr[si]["off16"]) * 16
        st = int(hdr[si]["strategy"])
        rows = int(hdr[si]["rows"])
        if rows != b - a:
            raise ValueError(f"segment {si}: rows {rows} != {b - a}")
        size = segment_cost(st, rows, c, d)
        if off + size > len(buf):
            raise ValueError(f"segment {si} overruns the payload")
        seg = buf[off:off + size]
        if st == SM:
            idx = seg[:c].astype(np.int64)
            vals = seg[pad16(c):].view("<f2").reshape(rows, c).astype(np.float64)
            out[a:b][:, idx] = vals
        elif st == PV:
            vals = seg[:2 * c * rows].view("<f2").reshape(rows, c).astype(np.float64)
            idx = seg[2 * c * rows:2 * c * rows + c * rows].reshape(rows, c).astype(np.int64)
            r = np.arange(a, b)[:, None]
            out[r, idx] = vals
        elif st == DENSE:
            out[a:b] = seg.view("<f2").reshape(rows, d).astype(np.float64)
        elif st == PVB:
            vals = seg[:2 * c * rows].view("<f2").reshape(rows, c).astype(np.float64)
            masks = seg[2 * c * rows:].reshape(rows, 16)
            for r in range(rows):
                ch = bitmask_channels(masks[r])
                if len(ch) != c:
                    raise ValueError(f"segment {si} row {r}: bitmask holds {len(ch)} channels")
                out[a + r, ch] = vals[r]
        else:
            raise ValueError(f"segment {si}: bad strategy {st}")
    return out


# ---------------------------------------------------------------------------
# Steps 5-6: decode (query-aware token selection + attention on the packed
# cache; §1 prior-work paragraph and Observation & Method 2)
# ---------------------------------------------------------------------------
def top_k_tokens(s: np.ndarray, k: int) -> np.ndarray:
    """The min(k, T) highest scores, ties to the lower token index, returned
    in ascending token order (READING)."""
    T = s.shape[0]
    kk = min(int(k), T)
    order = np.lexsort((np.arange(T), -np.asarray(s, dtype=np.float64)))
    return np.sort(order[:kk])


@dataclass
class DecodeResult:
    scores: np.ndarray      # [T] GQA-summed scores
    sel: np.ndarray         # [kk] ascending token ids
    out: np.ndarray         # [g, d] attention output in the original basis
    logits: np.ndarray      # [g, kk]


def rotate_queries(q: np.ndarray, R_K: np.ndarray) -> np.ndarray:
    """q~_i = q_i R_K for each query head of the group (fp64)."""
    return np.atleast_2d(np.asarray(q, dtype=np.float64)) @ np.asarray(R_K, dtype=np.float64)


def attend(qt: np.ndarray, R_V: np.ndarray, K_hat: np.ndarray, V_hat: np.ndarray,
           sel: np.ndarray):
    """Softmax attention of the rotated queries over the selected tokens:
    logits q~_i . k^_t / sqrt(d), max-subtracted softmax, o~_i = sum_t p_it v^_t
    in the rotated V basis, o_i = o~_i R_V^T.  Returns (out [g, d], logits)."""
    d = qt.shape[1]
    logits = (qt @ K_hat[sel].T) / math.sqrt(d)
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    p /= p.sum(axis=1, keepdims=True)
    ot = p @ V_hat[sel]
    return ot @ np.asarray(R_V, dtype=np.float64).T, logits


def decode_stream(q: np.ndarray, R_K: np.ndarray, R_V: np.ndarray,
                  K_hat: np.ndarray, V_hat: np.ndarray, k: int) -> DecodeResult:
    """One decode step for one KV head and its g query heads.

    q~_i = q_i R_K; s_t = sum_i q~_i . k^_t (the GQA group's scores summed);
    Sel = top-k of s; then `attend` over Sel."""
    qt = rotate_queries(q, R_K)
    s = (qt @ K_hat.T).sum(axis=0)
    sel = top_k_tokens(s, k)
    out, logits = attend(qt, R_V, K_hat, V_hat, sel)
    return DecodeResult(scores=s, sel=sel, out=out, logits=logits)


# ---------------------------------------------------------------------------
# Layer-level convenience (loops over streams; query head i -> KV head i // g)
# ---------------------------------------------------------------------------
@dataclass
class CompressedLayer:
    B: int
    H: int
    T: int
    S: int
    c: int
    K: List[List[CompressedStream]]
    V: List[List[CompressedStream]]


def compress_layer(K: np.ndarray, V: np.ndarray, S: int, c: int, tau: float,
                   bases_K=None, bases_V=None) -> CompressedLayer:
    """K, V: [B, H, T, d] fp16.  bases_*: optional [B, H, d, d]."""
    B, H, T, d = K.shape
    outK, outV = [], []
    for b in range(B):
        rk, rv = [], []
        for h in range(H):
            rk.append(compress_stream(K[b, h], S, c, tau,
                                      None if bases_K is None else bases_K[b, h]))
            rv.append(compress_stream(V[b, h], S, c, tau,
                                      None if bases_V is None else bases_V[b, h]))
        outK.append(rk)
        outV.append(rv)
    return CompressedLayer(B=B, H=H, T=T, S=S, c=c, K=outK, V=outV)


def decode_layer(layer: CompressedLayer, q: np.ndarray, k: int):
    """q: [B, Hq, d] fp16.  Returns (out [B, Hq, d] fp64, sel [B, H, kk],
    scores [B, H, T])."""
    B, Hq, d = q.shape
    g = Hq // layer.H
    kk = min(k, layer.T)
    out = np.zeros((B, Hq, d))
    sel = np.zeros((B, layer.H, kk), dtype=np.int64)
    scores = np.zeros((B, layer.H, layer.T))
    for b in range(B):
        for h in range(layer.H):
            ck, cv = layer.K[b][h], layer.V[b][h]
            r = decode_stream(q[b, h * g:(h + 1) * g], ck.R, cv.R,
                              ck.dense_hat(), cv.dense_hat(), k)
            out[b, h * g:(h + 1) * g] = r.out
            sel[b, h] = r.sel
            scores[b, h] = r.scores
    return out, sel, scores


# ---------------------------------------------------------------------------
# Decode-time appends (§1 "Observation & Method 2: compressed KV cache
# management": newly generated KV stay in a GPU-side buffer, are attended in
# later decode steps, and full segments are compressed and switched in)
# ---------------------------------------------------------------------------
def append_rows(X_new: np.ndarray, R: np.ndarray) -> np.ndarray:
    """READING: a newly generated token waits in the buffer as its rotated
    vector x R (the stream's existing basis) in fp16 with every channel kept,
    i.e. a dense row.  Returns the stored values as [n, d] fp64."""
    return to_fp16(rotate(X_new, R)).astype(np.float64)


@dataclass
class GrownStream:
    """A compressed stream with decode-time appends.

    READING: the prefill part keeps its segments (the last one possibly
    ragged); appended tokens fill a buffer of up to S tokens; whenever the
    buffer holds S tokens they are compressed as one segment with the
    stream's basis, by the same steps as the prefill (compress_stream with
    R given), and committed after the prefill part and earlier commits.
    Token order: prefill tokens, committed segments, then the buffer."""
    base: CompressedStream
    committed: List[CompressedStream] = field(default_factory=list)
    tail: Optional[np.ndarray] = None        # [n, d] fp16 tokens not yet committed

    @property
    def S(self) -> int:
        return self.base.S

    @property
    def T(self) -> int:
        return self.base.T + self.S * len(self.committed) + self.n_tail

    @property
    def n_tail(self) -> int:
        return 0 if self.tail is None else self.tail.shape[0]


def append_stream(gs: GrownStream, X_new: np.ndarray, tau: float,
                  bitmask_pv: bool = False) -> GrownStream:
    """Adds tokens [n, d] (fp16) to the buffer, committing every full S.
    A commit uses the strategy set of the prefill (bitmask_pv as there)."""
    X_new = np.asarray(X_new)
    d = gs.base.d
    tail = np.zeros((0, d), dtype=X_new.dtype) if gs.tail is None else gs.tail
    tail = np.concatenate([tail, X_new], axis=0)
    committed = list(gs.committed)
    while tail.shape[0] >= gs.S:
        seg, tail = tail[:gs.S], tail[gs.S:]
        committed.append(compress_stream(seg, gs.S, gs.base.c, tau, R=gs.base.R,
                                         bitmask_pv=bitmask_pv))
    return GrownStream(base=gs.base, committed=committed, tail=tail)


def grown_dense_hat(gs: GrownStream) -> np.ndarray:
    """[T, d] fp64 of the values decode reads: the prefill part's stored
    values, the committed segments', then the buffer's dense rows."""
    parts = [gs.base.dense_hat()] + [cs.dense_hat() for cs in gs.committed]
    if gs.n_tail:
        parts.append(append_rows(gs.tail, gs.base.R))
    return np.concatenate(parts, axis=0)


def grown_segment_starts(T0: int, S: int, n_committed: int) -> List[int]:
    """First token of every segment: the prefill segments at multiples of S,
    then one committed segment per S tokens after the prefill's end."""
    return list(range(0, T0, S)) + [T0 + i * S for i in range(n_committed)]
