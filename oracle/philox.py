"""Philox-4x32-10 counter-based generator (oracle copy; test infrastructure).

The pages give no random-number scheme; [SpS] "实验结果" only remarks that SpS
and ordinary sampling differ in their pseudo-random seed handling. The build
therefore fixes one: Philox-4x32 with 10 rounds, as published by Salmon,
Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11).
This file is written from that definition; the CUDA library carries its own,
independent copy, and the two are cross-checked on the GPU.

Counter and key layout used everywhere in this project:

    key     = (seed & 0xffffffff, seed >> 32)
    counter = (row & 0xffffffff, row >> 32, position, purpose)

``row`` is ``offset + b`` (the sequence's global row id), ``position`` the
draft position k, ``purpose`` one of the PURPOSE_* constants below. Output
word 0 is turned into a uniform u = ((w0 >> 9) + 0.5) * 2**-23, which lies in
(0, 1), takes 2**23 equally likely values and, having 24 significant bits, is
exact in fp32 as well as fp64 (the 24-bit variant (w0 >> 8) + 0.5 would need 25
bits and round in fp32).
"""

import numpy as np

PURPOSE_ACCEPT = 0    # the acceptance uniform u_k
PURPOSE_RESAMPLE = 1  # the resample / bonus uniform u'
PURPOSE_DRAFT = 2     # draft-token sampling (spec_sample)
PURPOSE_NOISE = 3     # reserved for input generation

_MASK = np.uint64(0xFFFFFFFF)
_M0 = np.uint64(0xD2511F53)  # round multiplier applied to counter word 0
_M1 = np.uint64(0xCD9E8D57)  # round multiplier applied to counter word 2
_W0 = np.uint64(0x9E3779B9)  # key schedule (Weyl) increment, key word 0
_W1 = np.uint64(0xBB67AE85)  # key schedule (Weyl) increment, key word 1


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Philox-4x32-10 block function, vectorised over broadcastable inputs.

    One round maps (c0, c1, c2, c3) with key (k0, k1) to
    (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0));
    the key is bumped by the Weyl constants between rounds (Salmon et al.,
    SC'11, section on the Philox family). Returns four uint32 arrays.
    """
    c0, c1, c2, c3, k0, k1 = (np.asarray(v, dtype=np.uint64) & _MASK for v in (c0, c1, c2, c3, k0, k1))
    c0, c1, c2, c3, k0, k1 = np.broadcast_arrays(c0, c1, c2, c3, k0, k1)
    c0, c1, c2, c3, k0, k1 = (v.copy() for v in (c0, c1, c2, c3, k0, k1))
    for r in range(10):
        if r > 0:
            k0 = (k0 + _W0) & _MASK
            k1 = (k1 + _W1) & _MASK
        p0 = _M0 * c0  # < 2**64: no wrap-around in uint64
        p1 = _M1 * c2
        hi0, lo0 = p0 >> np.uint64(32), p0 & _MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & _MASK
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return tuple(v.astype(np.uint32) for v in (c0, c1, c2, c3))


def uniform(seed, row, position, purpose):
    """u in (0,1) for (seed, row, position, purpose); arrays broadcast.

    u = ((w0 >> 9) + 0.5) * 2**-23 with w0 the first Philox output word.
    """
    seed = np.uint64(seed)
    row = np.asarray(row, dtype=np.uint64)
    w0, _, _, _ = philox4x32_10(row & _MASK, row >> np.uint64(32), position, purpose,
                                seed & _MASK, seed >> np.uint64(32))
    return ((w0 >> np.uint32(9)).astype(np.float64) + 0.5) * 2.0 ** -23
