"""The kernel decodes work-unit indices with division by invariant integers
(Granlund and Montgomery, 1994, unsigned case): q = (mulhi(mul, n) + n) >> l with
l = ceil(log2 d) and mul = floor(2^32 (2^l - d) / d) + 1. This restates that
method and checks it exactly against integer division over the range the kernel
uses (0 <= n < 2^31, 1 <= d < 2^31), at boundaries and on random values."""
import random


def make(d):
    l = 0
    while (1 << l) < d:
        l += 1
    return ((1 << 32) * ((1 << l) - d)) // d + 1, l


def fdiv(n, mul, l):
    return (((n * mul) >> 32) + n) >> l


def test_division_by_invariant_integers():
    rng = random.Random(7)
    ds = list(range(1, 400)) + [2 ** k + o for k in range(1, 31) for o in (-1, 0, 1)]
    ds += [rng.randrange(1, 2 ** 31) for _ in range(3000)]
    for d in ds:
        if not 1 <= d < 2 ** 31:
            continue
        mul, l = make(d)
        assert 0 < mul < 2 ** 32
        ns = [0, 1, d - 1, d, d + 1, 2 * d - 1, 2 * d, 2 ** 31 - 1, 2 ** 31 - d]
        ns += [rng.randrange(0, 2 ** 31) for _ in range(100)]
        for n in ns:
            if 0 <= n < 2 ** 31:
                assert fdiv(n, mul, l) == n // d, (n, d)
                assert ((n * mul) >> 32) + n < 2 ** 32
