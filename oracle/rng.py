"""Counter-based random streams for the method's own random matrices (Pi, S).

The pages only say that Pi is a random orthogonal matrix ([P4] §4.1) and that
QJL uses a random projection ([P4] §4.3); they fix no generator.  Both sides of
this project draw them from the published SplitMix64 generator (Steele, Lea &
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014; the
64-bit finalizer constants of Vigna's reference splitmix64.c), used in counter
form, and turn pairs of uniforms into normals with the Box-Muller transform.

Definition (restated here, implemented independently in the CUDA library):
  state(stream, i) = seed + stream * 2**40 + (i + 1) * 0x9E3779B97F4A7C15  (mod 2**64)
  out(stream, i)   = mix64(state)
  uniform(i)       = ((out >> 11) + 0.5) * 2**-53            in (0, 1)
  normal(2j)       = sqrt(-2 ln uniform(2j)) * cos(2 pi uniform(2j+1))
  normal(2j+1)     = sqrt(-2 ln uniform(2j)) * sin(2 pi uniform(2j+1))
Stream 1 fills the d x d Gaussian matrix G that becomes Pi, stream 2 fills S.
"""

import math

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MASK64 = (1 << 64) - 1


def _mix64(z):
    """SplitMix64 output finalizer on a uint64 numpy array (wrapping arithmetic)."""
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= np.uint64(0xBF58476D1CE4E5B9)
    z ^= z >> np.uint64(27)
    z *= np.uint64(0x94D049BB133111EB)
    z ^= z >> np.uint64(31)
    return z


def splitmix64_stream(seed, stream, n, start=0):
    """Raw 64-bit outputs out(stream, start .. start+n-1) as uint64."""
    base = (int(seed) + int(stream) * (1 << 40)) & MASK64
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = np.uint64(base) + idx * np.uint64(GAMMA)
        return _mix64(state)


def uniform_stream(seed, stream, n, start=0):
    """Uniforms in (0, 1): ((out >> 11) + 0.5) * 2**-53, exact in fp64."""
    raw = splitmix64_stream(seed, stream, n, start)
    return ((raw >> np.uint64(11)).astype(np.float64) + 0.5) * 2.0 ** -53


def gaussian_stream(seed, stream, n):
    """n standard normals by Box-Muller from consecutive uniform pairs."""
    npairs = (n + 1) // 2
    u = uniform_stream(seed, stream, 2 * npairs)
    u1, u2 = u[0::2], u[1::2]
    # math.log/cos/sin (the C library's) element by element, so both sides of
    # the project call the same libm routines.
    out = np.empty(2 * npairs)
    for j in range(npairs):
        r = math.sqrt(-2.0 * math.log(u1[j]))
        t = 2.0 * math.pi * u2[j]
        out[2 * j] = r * math.cos(t)
        out[2 * j + 1] = r * math.sin(t)
    return out[:n]
