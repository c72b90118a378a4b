"""Philox4x64-10 counter-based generator and the verify step's uniforms / Gumbel noise.

Written from the published definition (Salmon, Moraes, Dror, Shaw, "Parallel
random numbers: as easy as 1, 2, 3", SC'11): a 4x64-bit counter and a 2x64-bit
key; each of the 10 rounds multiplies counter words 0 and 2 by two fixed odd
constants, keeps the 128-bit products' high and low halves, XORs the high
halves with the other two counter words and the key, and permutes; the key is
bumped by two Weyl constants between rounds.

The pages say only that sampling verification draws random numbers; the
generator and the counter layout are this project's reading (stated in the
design notes).  Use for the round:

    key     = (seed, 0)
    acceptance test i at node (b, node), stream 0:
        counter = (round_id, b * 2**32 + node, i, 0)
        U  = (w0 >> 40) * 2**-24                   (w0: the first output word)
    Gumbel noise of token x at node (b, node), stream 1 (stream 2 for the
    children of a sampled draft, node = the expanded node's slot): one block
    serves four tokens,
        counter = (round_id, b * 2**32 + node, x // 4, stream)
        U' = ((w >> 40) + 0.5) * 2**-24            (w: output word x % 4)
        gumbel = -log(-log U')

The four output words of a Philox block are independent uniform 64-bit
words (the generator's design), so every token still gets its own
independent Gumbel variable.

ORACLE / TEST INFRASTRUCTURE ONLY.
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
PHILOX_M0 = 0xD2E7470EE14C6C93
PHILOX_M1 = 0xCA5A826395121157
PHILOX_W0 = 0x9E3779B97F4A7C15  # golden ratio
PHILOX_W1 = 0xBB67AE8584CAA73B  # sqrt(3) - 1
ROUNDS = 10


def philox4x64_scalar(ctr, key, rounds: int = ROUNDS):
    """One Philox4x64 block with Python integers (the definition, word by word)."""
    c0, c1, c2, c3 = (int(x) & MASK64 for x in ctr)
    k0, k1 = (int(x) & MASK64 for x in key)
    for r in range(rounds):
        if r:
            k0 = (k0 + PHILOX_W0) & MASK64
            k1 = (k1 + PHILOX_W1) & MASK64
        p0 = PHILOX_M0 * c0
        p1 = PHILOX_M1 * c2
        hi0, lo0 = p0 >> 64, p0 & MASK64
        hi1, lo1 = p1 >> 64, p1 & MASK64
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


_U32 = np.uint64(0xFFFFFFFF)
_S32 = np.uint64(32)


def _mulhilo(a: np.ndarray, b: int):
    """128-bit product of uint64 arrays by a constant, split into (hi, lo)."""
    bl, bh = np.uint64(b & 0xFFFFFFFF), np.uint64(b >> 32)
    al, ah = a & _U32, a >> _S32
    ll = al * bl
    lh = al * bh
    hl = ah * bl
    hh = ah * bh
    cross = (ll >> _S32) + (hl & _U32) + (lh & _U32)
    hi = hh + (hl >> _S32) + (lh >> _S32) + (cross >> _S32)
    lo = a * np.uint64(b)
    return hi, lo


def philox4x64(c0, c1, c2, c3, k0: int, k1: int = 0, rounds: int = ROUNDS):
    """Vectorised Philox4x64 over broadcastable uint64 counter arrays."""
    with np.errstate(over="ignore"):
        c0, c1, c2, c3 = np.broadcast_arrays(*(np.asarray(x, dtype=np.uint64) for x in (c0, c1, c2, c3)))
        c0, c1, c2, c3 = c0.copy(), c1.copy(), c2.copy(), c3.copy()
        k0, k1 = k0 & MASK64, k1 & MASK64
        for r in range(rounds):
            if r:
                k0 = (k0 + PHILOX_W0) & MASK64
                k1 = (k1 + PHILOX_W1) & MASK64
            hi0, lo0 = _mulhilo(c0, PHILOX_M0)
            hi1, lo1 = _mulhilo(c2, PHILOX_M1)
            c0, c1, c2, c3 = hi1 ^ c1 ^ np.uint64(k0), lo1, hi0 ^ c3 ^ np.uint64(k1), lo0
    return c0, c1, c2, c3


def _words(seed, round_id, b, node, idx, stream):
    c1 = (np.asarray(b, dtype=np.uint64) << _S32) + np.asarray(node, dtype=np.uint64)
    return philox4x64(round_id, c1, idx, stream, int(seed))


def _word0(seed, round_id, b, node, idx, stream):
    return _words(seed, round_id, b, node, idx, stream)[0]


def uniform(seed, round_id, b, node, idx):
    """Acceptance uniform in [0, 1): 24 top bits of word 0, stream 0."""
    w = _word0(seed, round_id, b, node, idx, 0)
    return (w >> np.uint64(40)).astype(np.float64) * 2.0 ** -24


def gumbel(seed, round_id, b, node, idx, stream=1):
    """Gumbel(0, 1) noise of token idx: word idx % 4 of block idx // 4 of the
    stream (1: the verify step's residual draw; 2: the sampled draft's children,
    node = the expanded node's slot), through the open-interval uniform U'."""
    idx = np.asarray(idx, dtype=np.uint64)
    ws = _words(seed, round_id, b, node, idx >> np.uint64(2), stream)
    w = np.choose((idx & np.uint64(3)).astype(np.int64), ws)
    u = ((w >> np.uint64(40)).astype(np.float64) + 0.5) * 2.0 ** -24
    return -np.log(-np.log(u))
