"""Philox4x32-10 counter-based generator and the verifier's uniform streams.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Philox4x32-10 follows its published definition [Philox] (Salmon et al.,
SC'11, section 3.2): a 128-bit counter (four 32-bit words) and a 64-bit key
(two words) go through ten rounds.  One round multiplies counter words 0 and 2
by the constants M0 = 0xD2511F53 and M1 = 0xCD9E8D57 into 64-bit products and
mixes the high halves with the other two words and the key; the key is bumped
by the Weyl constants W0 = 0x9E3779B9, W1 = 0xBB67AE85 between rounds.

Uniform streams used by tree verification (the pages fix no generator, so the
reading is: counter-based, so any request/row can be drawn independently):
  * accept test of tree row ``i`` of request ``b``:
      counter = (i, b, 2*offset_hi + 0, offset_lo), key = (seed_lo, seed_hi),
      output word 0;
  * exponential-race uniform of vocabulary id ``y`` for request ``b``:
      counter = (y >> 2, b, 2*offset_hi + 1, offset_lo), output word (y & 3).
A 32-bit output ``x`` becomes ``u = (2*(x >> 9) + 1) * 2**-24`` which lies in
(0, 1) and is exactly representable in both fp32 and fp64, so the CPU and the
GPU see bit-identical uniforms.
"""

import numpy as np

M0 = np.uint64(0xD2511F53)
M1 = np.uint64(0xCD9E8D57)
W0 = np.uint64(0x9E3779B9)
W1 = np.uint64(0xBB67AE85)
MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32-10.  Inputs are uint32-valued arrays or scalars.

    Returns a tuple of four uint64 arrays holding the 32-bit output words.
    """
    c = [np.asarray(v, dtype=np.uint64) & MASK32 for v in (c0, c1, c2, c3)]
    c = list(np.broadcast_arrays(*c))
    c = [v.copy() for v in c]
    k0 = np.uint64(int(k0) & 0xFFFFFFFF)
    k1 = np.uint64(int(k1) & 0xFFFFFFFF)
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + W0) & MASK32
            k1 = (k1 + W1) & MASK32
        p0 = c[0] * M0  # < 2**64, exact in uint64
        p1 = c[2] * M1
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK32
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK32
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return tuple(c)


def bits_to_uniform(x):
    """Map 32-bit words to u = (2*(x>>9)+1) * 2^-24 in (0,1), exact in fp32."""
    x = np.asarray(x, dtype=np.uint64)
    return ((x >> np.uint64(9)).astype(np.float64) * 2.0 + 1.0) * 2.0 ** -24


def _key(seed):
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return seed & 0xFFFFFFFF, seed >> 32


def _c2c3(offset, stream):
    offset = int(offset) & 0xFFFFFFFFFFFFFFFF
    hi, lo = offset >> 32, offset & 0xFFFFFFFF
    if hi >= 2 ** 31:
        raise ValueError("offset must be below 2**63")
    return 2 * hi + stream, lo


def accept_uniforms(seed, offset, B, R):
    """Accept-test uniforms, array [B, R] (fp64 holding fp32-exact values)."""
    k0, k1 = _key(seed)
    c2, c3 = _c2c3(offset, 0)
    i = np.arange(R, dtype=np.uint64)[None, :]
    b = np.arange(B, dtype=np.uint64)[:, None]
    w = philox4x32_10(i, b, c2, c3, k0, k1)
    return bits_to_uniform(w[0])


def race_uniforms(seed, offset, b, V):
    """Exponential-race uniforms of request ``b`` for ids 0..V-1, array [V]."""
    k0, k1 = _key(seed)
    c2, c3 = _c2c3(offset, 1)
    y = np.arange(V, dtype=np.uint64)
    w = philox4x32_10(y >> np.uint64(2), np.uint64(b), c2, c3, k0, k1)
    words = np.stack(w, axis=0)  # [4, V]
    x = words[(y & np.uint64(3)).astype(np.int64), np.arange(V)]
    return bits_to_uniform(x)


def race_uniforms_batch(seed, offset, B, V):
    """Exponential-race uniforms for requests 0..B-1, array [B, V]."""
    k0, k1 = _key(seed)
    c2, c3 = _c2c3(offset, 1)
    y = np.arange(V, dtype=np.uint64)[None, :]
    b = np.arange(B, dtype=np.uint64)[:, None]
    w = philox4x32_10(y >> np.uint64(2), b, c2, c3, k0, k1)
    words = np.stack(w, axis=0)  # [4, B, V]
    sel = np.broadcast_to((y & np.uint64(3)).astype(np.int64), (B, V))
    x = np.take_along_axis(words, sel[None], axis=0)[0]
    return bits_to_uniform(x)
