"""java.util.Random, restated from its published specification.

The pages seed several worked examples with ``new Random(seed)`` and print the
results; reproducing the generator lets those printed numbers pin the oracle.
Specification (Java SE API documentation of java.util.Random):
  * state: 48 bits, initialised to (seed XOR 0x5DEECE66D) mod 2^48;
  * next(bits): state = (state * 0x5DEECE66D + 0xB) mod 2^48, return the top
    ``bits`` bits as a signed 32-bit int;
  * nextDouble(): ((next(26) << 27) + next(27)) * 2^-53;
  * nextGaussian(): the polar method of Box, Muller and Marsaglia, caching the
    second value: v1, v2 = 2*nextDouble()-1 until 0 < s = v1^2+v2^2 < 1, then
    m = sqrt(-2 ln(s) / s), return v1*m and keep v2*m for the next call.
"""
import math

_MULT = 0x5DEECE66D
_MASK = (1 << 48) - 1


class JavaRandom:
    def __init__(self, seed: int):
        self.state = (seed ^ _MULT) & _MASK
        self._next_gaussian = None

    def next(self, bits: int) -> int:
        self.state = (self.state * _MULT + 0xB) & _MASK
        r = self.state >> (48 - bits)
        if r >= 1 << 31:
            r -= 1 << 32
        return r

    def next_double(self) -> float:
        return ((self.next(26) << 27) + self.next(27)) * 2.0 ** -53

    def next_gaussian(self) -> float:
        if self._next_gaussian is not None:
            g, self._next_gaussian = self._next_gaussian, None
            return g
        while True:
            v1 = 2 * self.next_double() - 1
            v2 = 2 * self.next_double() - 1
            s = v1 * v1 + v2 * v2
            if 0 < s < 1:
                break
        m = math.sqrt(-2 * math.log(s) / s)
        self._next_gaussian = v2 * m
        return v1 * m


def java_round(x: float) -> int:
    """Math.round(double): the closest long, ties towards positive infinity."""
    return math.floor(x + 0.5)
