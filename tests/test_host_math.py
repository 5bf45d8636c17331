"""Host-side integer math used by the kernels' index decomposition.

The tile kernels divide 31-bit task indices by per-call constants with one
64-bit multiply and a shift (m = ceil(2^(32+s)/d), s = ceil(log2 d)).  This
checks the formula, as the library computes it, against exact division."""
import numpy as np


def make_fastdiv(d):
    s = 0
    while (1 << s) < d:
        s += 1
    shift = 32 + s
    return ((1 << shift) + d - 1) // d, shift


def test_fastdiv_exact_below_2_pow_31():
    rng = np.random.default_rng(1)
    divisors = list(range(1, 600)) + [2**k + o for k in range(10, 31) for o in (-1, 0, 1)] + [2**31 - 1]
    divisors += rng.integers(1, 2**31 - 1, 300).tolist()
    edge = [0, 1, 2**31 - 1, 2**31 - 2, 2**30, 2**30 - 1]
    for d in divisors:
        m, shift = make_fastdiv(d)
        assert m < 2**33
        ns = np.concatenate([rng.integers(0, 2**31, 2000), np.array(edge), np.array([d - 1, d, d + 1, 2 * d - 1, 2 * d]) % 2**31])
        for n in ns.tolist():
            assert (n * m) >> shift == n // d, (n, d)
            assert n * m < 2**64
