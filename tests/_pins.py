"""Independent formulations used to pin the oracle (test-side only).

Nothing here is shared with the CUDA path, and nothing reuses the oracle's
code: the total order is rebuilt from Python floats (bf16 widened by a bit
shift, not by the oracle's exponent/fraction decoding), and the selection is
checked by enumerating subsets rather than sorting.
"""
from __future__ import annotations

import itertools
import math
import struct


def order_key(bits: int, is_bf16: bool):
    """A Python sort key realising IEEE 754 totalOrder on a bit pattern."""
    if is_bf16:
        bits &= 0xFFFF
        f = struct.unpack("<f", struct.pack("<I", bits << 16))[0]
        neg = bits >> 15
        payload = bits & 0x7F
    else:
        bits &= 0xFFFFFFFF
        f = struct.unpack("<f", struct.pack("<I", bits))[0]
        neg = bits >> 31
        payload = bits & 0x7FFFFF
    if math.isnan(f):
        return (-2, -payload, 0) if neg else (2, payload, 0)
    if f == 0.0:
        return (0, 0.0, -1 if neg else 1)
    return (0, f, 0)


def brute_force_select(row_bits, v: int, K: int, num_init: int, num_local: int,
                       is_bf16: bool):
    """All size-n subsets of [0, v) that contain every forced id and in which
    every selected non-forced id beats every excluded id (higher order key,
    or equal key and lower id).  Returns the list of such subsets (sorted)."""
    n = min(K, v)
    forced = {b for b in range(v) if b < num_init or b >= v - num_local}
    keys = [order_key(int(row_bits[b]), is_bf16) for b in range(v)]
    found = []
    for subset in itertools.combinations(range(v), n):
        s = set(subset)
        if not forced.issubset(s) and len(forced) <= n:
            continue
        ok = True
        for a in s - forced:
            for x in set(range(v)) - s:
                if not (keys[a] > keys[x] or (keys[a] == keys[x] and a < x)):
                    ok = False
                    break
            if not ok:
                break
        if ok:
            found.append(sorted(s))
    return found
