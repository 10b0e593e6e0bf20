"""Philox4x32-10 counter-based generator, CPU (NumPy) version.

Test infrastructure: only the tests, the smoke check and the benchmark's CPU-baseline
leg use this module. It shares no code with the CUDA library, which carries its own
implementation of the same published definition.

Definition followed: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
1, 2, 3" (SC'11), section 4 (Philox): a 4x32-bit counter and a 2x32-bit key; each round
multiplies counter words 0 and 2 by the constants M0, M1 into 64-bit hi/lo halves and
permutes them with the other two words and the key; the key is bumped by the Weyl
constants W0, W1 between rounds; 10 rounds. Pinned by the published known-answer
vectors (tests/golden/philox4x32_10_kat.txt).

The step-verification draws (the draw layout is this library's own choice; the pages
give only the distributions):
  key      = (seed & 0xffffffff, seed >> 32)
  accept   counter = (request, offset_lo, offset_hi, j)          words 0..3 -> steps 4j..4j+3
  resample counter = (request, offset_lo, offset_hi, 0x80000000 | (v >> 2))  word v & 3 -> token v
  noise    counter = (request, position, offset_lo, 0x40000000 | (v >> 2))  word v & 3 -> the
           shared Gumbel noise of token v at absolute output position `position`
  uniform  u = (2 * (w >> 9) + 1) * 2**-24, an odd multiple of 2**-24 in (0, 1); exactly
           representable in fp32 and fp64, so both sides see the same value.
"""
from __future__ import annotations

import numpy as np

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
MASK32 = 0xFFFFFFFF
RESAMPLE_TAG = 0x80000000
NOISE_TAG = 0x40000000


def philox4x32_10(counter, key):
    """counter: uint32 array [..., 4]; key: uint32 array [..., 2] (broadcast against
    the counter's leading dimensions). Returns the uint32 array [..., 4] of outputs."""
    c = np.asarray(counter, dtype=np.uint32)
    key = np.asarray(key, dtype=np.uint32)
    lead = np.broadcast_shapes(c.shape[:-1], key.shape[:-1])
    c = np.broadcast_to(c, lead + (4,)).astype(np.uint64)
    k0 = np.broadcast_to(key[..., 0], lead).astype(np.uint64)
    k1 = np.broadcast_to(key[..., 1], lead).astype(np.uint64)
    m32 = np.uint64(MASK32)
    s32 = np.uint64(32)
    c0, c1, c2, c3 = c[..., 0], c[..., 1], c[..., 2], c[..., 3]
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + np.uint64(W0)) & m32
            k1 = (k1 + np.uint64(W1)) & m32
        p0 = c0 * np.uint64(M0)          # < 2**64: no wrap-around
        p1 = c2 * np.uint64(M1)
        c0, c1, c2, c3 = ((p1 >> s32) ^ c1 ^ k0), (p1 & m32), ((p0 >> s32) ^ c3 ^ k1), (p0 & m32)
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def philox_scalar(counter, key):
    """Pure-Python integer version of the same function (for small cross-checks)."""
    c = [int(x) & MASK32 for x in counter]
    k0, k1 = int(key[0]) & MASK32, int(key[1]) & MASK32
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + W0) & MASK32
            k1 = (k1 + W1) & MASK32
        p0 = M0 * c[0]
        p1 = M1 * c[2]
        c = [((p1 >> 32) ^ c[1] ^ k0) & MASK32, p1 & MASK32,
             ((p0 >> 32) ^ c[3] ^ k1) & MASK32, p0 & MASK32]
    return c


def word_to_uniform(w):
    """uint32 -> odd multiple of 2**-24 in (0, 1), returned as float64."""
    w = np.asarray(w, dtype=np.uint64)
    return ((w >> np.uint64(9)) * np.uint64(2) + np.uint64(1)).astype(np.float64) * 2.0 ** -24


def _key(seed):
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return np.array([seed & MASK32, seed >> 32], dtype=np.uint32)


def accept_uniforms(seed, offset, request, n):
    """Uniforms u_1..u_n of one request's acceptance tests (step order)."""
    offset = int(offset) & 0xFFFFFFFFFFFFFFFF
    calls = (n + 3) // 4
    ctr = np.zeros((calls, 4), dtype=np.uint32)
    ctr[:, 0] = request
    ctr[:, 1] = offset & MASK32
    ctr[:, 2] = offset >> 32
    ctr[:, 3] = np.arange(calls, dtype=np.uint32)
    words = philox4x32_10(ctr, _key(seed)).reshape(-1)[:n]
    return word_to_uniform(words)


def resample_uniforms(seed, offset, request, V):
    """Uniforms u_v, v = 0..V-1, of one request's residual resampling race."""
    offset = int(offset) & 0xFFFFFFFFFFFFFFFF
    calls = (V + 3) // 4
    ctr = np.zeros((calls, 4), dtype=np.uint32)
    ctr[:, 0] = request
    ctr[:, 1] = offset & MASK32
    ctr[:, 2] = offset >> 32
    ctr[:, 3] = RESAMPLE_TAG | np.arange(calls, dtype=np.uint32)
    words = philox4x32_10(ctr, _key(seed)).reshape(-1)[:V]
    return word_to_uniform(words)


def noise_uniforms(seed, offset, request, position, V):
    """Uniforms u_{a,v}, v = 0..V-1, behind the shared Gumbel noise of one request at
    absolute output position a (only the low 32 bits of the offset enter)."""
    offset = int(offset) & 0xFFFFFFFFFFFFFFFF
    calls = (V + 3) // 4
    ctr = np.zeros((calls, 4), dtype=np.uint32)
    ctr[:, 0] = request
    ctr[:, 1] = int(position) & MASK32
    ctr[:, 2] = offset & MASK32
    ctr[:, 3] = NOISE_TAG | np.arange(calls, dtype=np.uint32)
    words = philox4x32_10(ctr, _key(seed)).reshape(-1)[:V]
    return word_to_uniform(words)
