"""Dropout masks from a counter-based generator, and the tensor-parallel RNG
tracker.

"02 - How a whole Transformer block is split", section 5 (TP-specific RNG):
outside the tensor-parallel region the activations are replicated, so every
rank must drop the same elements; inside it (attention scores, split hidden)
each rank holds a different shard and must draw its own mask. Three generator
states are registered at once:
    data-parallel    seed                          (outside the TP region)
    model-parallel   seed + 2718 + tp_rank         (inside the TP region)
    expert-parallel  seed + 1024 + 100*ep_rank + etp_rank   (MoE experts)
and a fork() context switches to one of them and back, so dropout inside the
region uses the model-parallel state; recomputation (activation
checkpointing) must reproduce the same mask.

Readings (the pages fix no generator):
  * The generator is Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel
    random numbers: as easy as 1, 2, 3", SC 2011): a state is (seed, offset);
    the key is the seed's low and high 32-bit words; the stream is the four
    32-bit outputs of counters (q, 0, 0, 0), q = 0, 1, ..., each word split
    into four bytes, lowest byte first. Byte position `offset + e` is the
    uniform of element e of a site, so a mask is a pure function of
    (seed, offset, element index): replay is exact by construction.
  * An element is kept iff its byte < thr = floor((1 - p) * 256 + 1/2)
    (round half up, in double precision from the caller's p); kept elements
    are scaled by 256 / thr (the realized keep probability is thr / 256).
  * The tracker's draw(n) hands out the current state's (seed, offset) and
    advances the offset by n rounded up to a multiple of 16 (one counter).
  * Sites of the layer: the attention probabilities (inside the TP region;
    element ((b*nq + h)*S + i)*Sp + j, Sp = S rounded up to 16, so each row
    starts on a counter), then the hidden dropouts after the output
    projection and after fc2 (outside; element t*H + c of [T, H]), each drawn
    in that order.

Written from the definitions with plain numpy integer arithmetic. Test
infrastructure only; pinned by tests/test_oracle_dropout.py (against the
curand host generator's Philox4x32-10 stream among others).
"""
import contextlib

import numpy as np

# Philox4x32 round multipliers and Weyl key increments (Salmon et al., SC 2011)
PHILOX_M0, PHILOX_M1 = 0xD2511F53, 0xCD9E8D57
PHILOX_W0, PHILOX_W1 = 0x9E3779B9, 0xBB67AE85
MASK32 = 0xFFFFFFFF


def philox4x32(counters, key, rounds=10):
    """counters [N, 4] uint32, key (k0, k1) -> [N, 4] uint32 outputs."""
    c = np.asarray(counters, dtype=np.uint64) & MASK32
    c0, c1, c2, c3 = (c[:, i].copy() for i in range(4))
    k0, k1 = np.uint64(key[0] & MASK32), np.uint64(key[1] & MASK32)
    m0, m1 = np.uint64(PHILOX_M0), np.uint64(PHILOX_M1)
    s32, m32 = np.uint64(32), np.uint64(MASK32)
    for r in range(rounds):
        p0 = m0 * c0            # < 2^64: both factors < 2^32
        p1 = m1 * c2
        hi0, lo0 = p0 >> s32, p0 & m32
        hi1, lo1 = p1 >> s32, p1 & m32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        if r + 1 < rounds:
            k0 = (k0 + np.uint64(PHILOX_W0)) & m32
            k1 = (k1 + np.uint64(PHILOX_W1)) & m32
    return np.stack([c0, c1, c2, c3], axis=1).astype(np.uint32)


def uniform_bytes(seed, offset, n):
    """Bytes at stream positions offset .. offset + n - 1 of state (seed, offset=0)."""
    if n == 0:
        return np.zeros(0, dtype=np.uint8)
    q0, q1 = offset // 16, (offset + n - 1) // 16
    q = np.arange(q0, q1 + 1, dtype=np.uint64)
    ctr = np.zeros((q.size, 4), dtype=np.uint64)
    ctr[:, 0] = q & np.uint64(MASK32)
    ctr[:, 1] = q >> np.uint64(32)
    words = philox4x32(ctr, (seed & MASK32, (seed >> 32) & MASK32))
    stream = words.reshape(-1).view(np.uint8)  # little-endian: lowest byte first
    if stream.dtype.byteorder == ">":
        raise RuntimeError("big-endian host")
    start = offset - q0 * 16
    return stream[start:start + n].copy()


def keep_threshold(p):
    """Bytes below this value are kept."""
    if not 0.0 <= p < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    return int(np.floor((1.0 - float(p)) * 256.0 + 0.5))


def keep_scale(p):
    return 256.0 / keep_threshold(p)


def dropout_keep(seed, offset, shape, p, row_pad=None):
    """Boolean keep mask of `shape` for a site at stream position `offset`.
    row_pad: the element index uses rows of this length (>= the last dim)."""
    shape = tuple(shape)
    last = shape[-1]
    rows = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
    ld = row_pad if row_pad is not None else last
    u = uniform_bytes(seed, offset, rows * ld).reshape(rows, ld)[:, :last]
    return (u.astype(np.int64) < keep_threshold(p)).reshape(shape)


def pad16(n):
    return (n + 15) // 16 * 16


class RNGTracker:
    """Named generator states (seed, offset) with a current one; fork()
    switches to a named state and back (the TP RNG tracker)."""

    DATA, MODEL, EXPERT = "data-parallel", "model-parallel", "expert-parallel"

    def __init__(self):
        self.states = {}
        self.current = None

    def add(self, name, seed):
        if name in self.states:
            raise ValueError(f"state {name} exists")
        self.states[name] = [int(seed), 0]
        if self.current is None:
            self.current = name

    @contextlib.contextmanager
    def fork(self, name=MODEL):
        prev = self.current
        self.current = name
        try:
            yield
        finally:
            self.current = prev

    def draw(self, n):
        """(seed, offset) for n uniforms from the current state; advances it."""
        st = self.states[self.current]
        out = (st[0], st[1])
        st[1] += pad16(n)
        return out


def model_parallel_seed(seed, tp_rank=0, ep_rank=0, etp_rank=0):
    """The three states of section 5; the data-parallel one is current."""
    t = RNGTracker()
    t.add(RNGTracker.DATA, seed)
    t.add(RNGTracker.MODEL, seed + 2718 + tp_rank)
    t.add(RNGTracker.EXPERT, seed + 1024 + 100 * ep_rank + etp_rank)
    return t


def layer_dropout(cfg, tracker, p_attn, p_hidden):
    """Draws the layer's three sites from the tracker (attention inside the TP
    region, the two hidden dropouts outside) and returns the keep masks:
    {"attn": (keep [B, nq, S, S], scale) or None, "proj": (keep [T, H], scale)
    or None, "fc2": ...} plus the drawn states under "states"."""
    B, S, H = cfg.batch, cfg.seq, cfg.hidden
    T, nq = B * S, cfg.n_q_heads
    out, states = {}, {}
    n_attn = B * nq * S * pad16(S)
    with tracker.fork(RNGTracker.MODEL):
        states["attn"] = tracker.draw(n_attn)
    states["proj"] = tracker.draw(T * H)
    states["fc2"] = tracker.draw(T * H)
    if p_attn > 0:
        s, o = states["attn"]
        out["attn"] = (dropout_keep(s, o, (B, nq, S, S), p_attn, row_pad=pad16(S)), keep_scale(p_attn))
    else:
        out["attn"] = None
    for site in ("proj", "fc2"):
        if p_hidden > 0:
            s, o = states[site]
            out[site] = (dropout_keep(s, o, (T, H), p_hidden), keep_scale(p_hidden))
        else:
            out[site] = None
    out["states"] = states
    return out
