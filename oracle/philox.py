"""Philox4x32-10 counter-based generator and the sampler's uniforms.

Test infrastructure only (see the package docstring).

The S³R pages use exact speculative sampling ([wispaper] "S3R drafts sparsely
and verifies densely"; [ritwork] "Как разреженный черновик ...") but say
nothing about random numbers.  Both the oracle and the CUDA library draw them
from Philox4x32 with 10 rounds, each side written independently from the
published definition: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3", SC'11, section 3.2 (Philox).

Definition used here (SC'11 section 3.2):
  * state: four 32-bit words (c0, c1, c2, c3); key: two 32-bit words (k0, k1)
  * one round with multipliers M0 = 0xD2511F53, M1 = 0xCD9E8D57:
        (hi0, lo0) = M0 * c0 as a 64-bit product
        (hi1, lo1) = M1 * c2
        (c0, c1, c2, c3) <- (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0)
  * the key is bumped between rounds by the Weyl constants
        k0 += 0x9E3779B9 (golden ratio), k1 += 0xBB67AE85 (sqrt(3) - 1)
  * Philox4x32-10 applies 10 rounds (9 key bumps).

How the sampler uses it (a reading: the pages give no RNG):
  counter = (n, position, stream, offset), key = (seed low 32, seed high 32),
  uniform u = (first output word >> 8) * 2^-24, a value in [0, 1) that is exact
  in float32 and float64, so both sides compare the same u.

Parity status: pinned by tests/test_oracle_philox.py against the published
known-answer vectors (tests/golden/philox4x32_10_kat.txt) and, on the GPU, by
tests/test_gpu_philox.py against CUDA's curand Philox4x32-10 device routine.
"""

import numpy as np

M0 = 0xD2511F53
M1 = 0xCD9E8D57
W0 = 0x9E3779B9
W1 = 0xBB67AE85
MASK32 = 0xFFFFFFFF

STREAM_ACCEPT = 0
STREAM_RESAMPLE = 1
STREAM_DRAFT = 2


def _mulhilo(m, x):
    prod = np.uint64(m) * x.astype(np.uint64)
    return (prod >> np.uint64(32)).astype(np.uint64), (prod & np.uint64(MASK32)).astype(np.uint64)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32-10: arrays (broadcastable) of 32-bit words in,
    the four output words (uint32 arrays) out."""
    c = [np.asarray(w, dtype=np.uint64) & np.uint64(MASK32) for w in (c0, c1, c2, c3)]
    c = list(np.broadcast_arrays(*c))
    k0 = np.asarray(k0, dtype=np.uint64) & np.uint64(MASK32)
    k1 = np.asarray(k1, dtype=np.uint64) & np.uint64(MASK32)
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + np.uint64(W0)) & np.uint64(MASK32)
            k1 = (k1 + np.uint64(W1)) & np.uint64(MASK32)
        hi0, lo0 = _mulhilo(M0, c[0])
        hi1, lo1 = _mulhilo(M1, c[2])
        c = [hi1 ^ c[1] ^ k0, lo1, hi0 ^ c[3] ^ k1, lo0]
    return tuple(w.astype(np.uint32) for w in c)


def philox_uniform(seed, offset, n, position, stream):
    """u in [0, 1) for counter (n, position, stream, offset) and key = seed."""
    seed = int(seed)
    offset = int(offset)
    if not 0 <= offset <= MASK32:
        raise ValueError("offset must fit in 32 bits")
    w0, _, _, _ = philox4x32_10(n, position, stream, offset, seed & MASK32, (seed >> 32) & MASK32)
    return (w0 >> np.uint32(8)).astype(np.float64) * (2.0 ** -24)
