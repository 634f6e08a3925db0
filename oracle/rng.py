"""The oracle's own counter-based generator for the method's random draws.

The method draws a random rotation, random signs and a Gaussian QJL matrix
([Reconstruction] §5 Step 2, §6 "The 1-Bit QJL Transform", §9 table;
[Design study] §Dense and structured transform comparison: "deterministic
seeded Rademacher pattern").  The pages name no generator; the one used is
SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014; the widely published 64-bit reference form by
Vigna), stepped one output at a time, with

* uniform in [0, 1):        (x >> 11) * 2^-53
* standard normal pairs:    Box-Muller, r = sqrt(-2 ln(1 - u1)),
                            z0 = r cos(2 pi u2), z1 = r sin(2 pi u2)
* Rademacher sign:          bit 0 of the output (1 -> -1, 0 -> +1)

Stream selection (reading; the pages give none): the initial state for
(seed, layer, head, role) is seed XOR splitmix64_mix(key) with
key = (layer << 24) | (head << 8) | role, layer < 2^20, head < 2^16, role < 2^8.
"""

from __future__ import annotations

import numpy as np

_M64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15


def splitmix64_mix(z: int) -> int:
    """The SplitMix64 output function applied to (z + golden gamma)."""
    z = (z + GOLDEN) & _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def stream_state(seed: int, layer: int, head: int, role: int) -> int:
    if not (0 <= layer < (1 << 20) and 0 <= head < (1 << 16) and 0 <= role < (1 << 8)):
        raise ValueError("layer/head/role out of range")
    key = (layer << 24) | (head << 8) | role
    return (seed & _M64) ^ splitmix64_mix(key)


class SplitMix64:
    """Plain SplitMix64, one output per call."""

    def __init__(self, state: int):
        self.state = state & _M64

    def next_u64(self) -> int:
        self.state = (self.state + GOLDEN) & _M64
        z = self.state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
        return z ^ (z >> 31)

    def outputs(self, n: int) -> np.ndarray:
        """The next n outputs as uint64 (vectorised, same sequence as next_u64)."""
        k = np.arange(1, n + 1, dtype=np.uint64)
        with np.errstate(over="ignore"):
            z = np.uint64(self.state) + k * np.uint64(GOLDEN)
            z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
            z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
            z = z ^ (z >> np.uint64(31))
        self.state = (self.state + n * GOLDEN) & _M64
        return z

    def uniforms(self, n: int) -> np.ndarray:
        return (self.outputs(n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)

    def normals(self, n: int) -> np.ndarray:
        """n standard normals; each Box-Muller pair consumes two outputs."""
        m = (n + 1) // 2
        u = self.uniforms(2 * m)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log(1.0 - u1))
        z = np.empty(2 * m, dtype=np.float64)
        z[0::2] = r * np.cos(2.0 * np.pi * u2)
        z[1::2] = r * np.sin(2.0 * np.pi * u2)
        return z[:n]

    def rademacher(self, n: int) -> np.ndarray:
        bit = self.outputs(n) & np.uint64(1)
        return np.where(bit == 1, -1.0, 1.0)
