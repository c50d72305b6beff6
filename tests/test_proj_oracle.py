"""CPU pins of the projection oracle (oracle/proj.py) against values fixed by arithmetic:
exact products of small integers, one-hot weights, identities, and a brute-force search
for the nearest bfloat16."""
import numpy as np
import pytest

from oracle.proj import bf16_round, skinny_proj


def nearest_bf16_brute(a):
    """The 8-significant-bit value nearest to a, ties to the even significand, by search."""
    if a == 0:
        return 0.0
    e = int(np.floor(np.log2(abs(a))))
    best = None
    for ee in (e - 1, e, e + 1):
        ulp = 2.0 ** (ee - 7)
        for mq in range(128, 256):
            c = np.copysign(mq * ulp, a)
            d = abs(c - a)
            if best is None or d < best[0] or (d == best[0] and mq % 2 == 0):
                best = (d, c)
    return best[1]


def test_bf16_round_is_the_nearest_bf16():
    rng = np.random.default_rng(5)
    v = rng.standard_normal(300) * np.exp(rng.uniform(-20, 20, 300))
    got = bf16_round(v)
    for a, g in zip(v, got):
        assert g == nearest_bf16_brute(a), (a, g)


def test_bf16_round_ties_and_exact_values():
    # exactly representable values stay; halfway cases go to the even significand
    assert np.array_equal(bf16_round(np.array([1.0, -3.0, 2.0 ** -20, 255.0 * 2 ** 10])),
                          np.array([1.0, -3.0, 2.0 ** -20, 255.0 * 2 ** 10]))
    assert bf16_round(np.array([1.0 + 2.0 ** -8]))[0] == 1.0                    # 128.5 -> 128
    assert bf16_round(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6      # 129.5 -> 130
    assert bf16_round(np.array([-(1.0 + 2.0 ** -8 + 2.0 ** -30)]))[0] == -(1.0 + 2.0 ** -7)


@pytest.mark.parametrize("m", [1, 5])
def test_skinny_proj_closed_forms(m):
    k, n_ab, r, n_b = 64, 32, 16, 24
    x = np.ones((m, k))
    w_ab = np.ones((n_ab, k))
    y, z = skinny_proj(x, w_ab, np.ones((n_b, r)), r)
    assert np.all(y == k)                      # every entry sums k ones
    assert np.all(z == r * k)                  # k is a bf16 value: r terms of k
    # one-hot second weights select columns of bf16(y): z[:, j] = bf16(y)[:, j mod r]
    rng = np.random.default_rng(6)
    xv = rng.integers(-3, 4, (m, k)).astype(np.float64)
    wv = rng.integers(-3, 4, (n_ab, k)).astype(np.float64)
    wb = np.zeros((n_b, r))
    wb[np.arange(n_b), np.arange(n_b) % r] = 1.0
    y, z = skinny_proj(xv, wv, wb, r)
    brute = np.array([[sum(xv[i, t] * wv[j, t] for t in range(k)) for j in range(n_ab)]
                      for i in range(m)])
    assert np.array_equal(y, brute)            # integers: exact
    assert np.array_equal(z, bf16_round(brute)[:, np.arange(n_b) % r])


def test_skinny_proj_identity_and_scaling():
    rng = np.random.default_rng(7)
    k = 32
    x = bf16_round(rng.standard_normal((3, k)))
    y, z = skinny_proj(x, np.eye(k), np.eye(16), 16)
    assert np.array_equal(y, x) and np.array_equal(z, x[:, :16])
    w = bf16_round(rng.standard_normal((16, k)))
    y1, _ = skinny_proj(x, w, np.eye(16), 16)
    y2, _ = skinny_proj(2.0 * x, w, np.eye(16), 16)
    assert np.array_equal(y2, 2.0 * y1)        # scaling by a power of two is exact
