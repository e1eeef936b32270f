"""Why three 9-bit digits and six digit products are enough: a numpy model of
the tcgen05 engine's arithmetic, checked against float64 on the CPU.

The scheme (restated from its definition, not from the CUDA code): every
operand row is cut into 128-wide blocks along K, each with a power-of-two scale
sigma, the smallest at or above the block's largest magnitude, and each element
is held as x = sigma / 256 (P1 + P2 + P3) with P1 = d1, P2 = d2 2^-9,
P3 = d3 2^-18 and integer digits |d| <= 256 (exact in bf16).  A product sums,
per 128-wide chunk, the exact integer level S0 = sum P1 Q1 and the level
S1 = sum of the five pairs (P1, Q2), (P2, Q1), (P1, Q3), (P2, Q2), (P3, Q1)
(fp32 accumulation, one K16 step at a time), and adds
sigma_A sigma_B 2^-16 (S0 + S1) to fp32 sums with one fused multiply-add per
chunk.

Pinned below:
* the digits hold any fp32 value to 2^-27 of its block scale, and exactly when
  it is within a factor 8 of the scale;
* S0 of a 128-wide chunk stays at or below 2^23, so its fp32 accumulation is
  exact in any order;
* the modelled product meets the bound the GPU self-test holds the kernel to
  (2^-20 sum |a||b| + 2^-23 |a.b|) on operands whose rows and blocks span many
  orders of magnitude;
* dropping the second-level pairs (or any one of them), or the third digit,
  breaks that bound by a factor of 5 or more, while the full scheme stays
  within a quarter of it: each part of the scheme is needed.
"""
import numpy as np
import pytest

CHUNK = 128
SIX_PAIRS = [(0, 0), (0, 1), (1, 0), (0, 2), (1, 1), (2, 0)]     # digit indices, 0-based


def pow2_ceil(m):
    """Smallest power of two at or above m (1 where m is 0)."""
    m = np.asarray(m, dtype=np.float64)
    f, e = np.frexp(np.where(m > 0, m, 1.0))
    return np.ldexp(1.0, e - (f == 0.5))


def block_scales(X):
    """sigma per (row, 128-column block)."""
    M, K = X.shape
    nb = (K + CHUNK - 1) // CHUNK
    out = np.empty((M, nb))
    for c in range(nb):
        out[:, c] = pow2_ceil(np.max(np.abs(X[:, c * CHUNK:(c + 1) * CHUNK]), axis=1))
    return out


def digits(X, sigma, ndig=3, bits=9):
    """Integer digits of X / sigma: d1 from 2^(bits-1) X / sigma, then each
    remainder times 2^bits, rounded to nearest (ties to even)."""
    y = np.asarray(X, dtype=np.float64) / sigma * 2.0 ** (bits - 1)
    out = []
    for _ in range(ndig):
        d = np.rint(y)
        out.append(d)
        y = (y - d) * 2.0 ** bits
    return out


def planes(X, sigma, ndig=3, bits=9):
    return [d * 2.0 ** (-bits * s) for s, d in enumerate(digits(X, sigma, ndig, bits))]


def digit_gemm(A, B, pairs=SIX_PAIRS, ndig=3):
    """The modelled C = A B^T."""
    A = np.asarray(A, dtype=np.float32)
    B = np.asarray(B, dtype=np.float32)
    M, K = A.shape
    N = B.shape[0]
    sa_all, sb_all = block_scales(A), block_scales(B)
    acc = np.zeros((M, N), dtype=np.float32)
    for c in range(sa_all.shape[1]):
        ks = slice(c * CHUNK, min((c + 1) * CHUNK, K))
        sa, sb = sa_all[:, c], sb_all[:, c]
        P = planes(A[:, ks], sa[:, None], ndig)
        Q = planes(B[:, ks], sb[:, None], ndig)
        s0 = np.zeros((M, N), dtype=np.float32)
        s1 = np.zeros((M, N), dtype=np.float32)
        for k0 in range(0, ks.stop - ks.start, 16):
            kk = slice(k0, k0 + 16)
            lead = sum(P[i][:, kk] @ Q[j][:, kk].T for i, j in pairs if i + j == 0)
            rest = sum((P[i][:, kk] @ Q[j][:, kk].T for i, j in pairs if i + j > 0), np.zeros((M, N)))
            s0 = (s0 + np.asarray(lead, dtype=np.float32)).astype(np.float32)
            s1 = (s1 + rest.astype(np.float32)).astype(np.float32)
        v = (s0 + s1).astype(np.float32)
        t = (v * sb[None, :].astype(np.float32)).astype(np.float32)
        acc = (t.astype(np.float64) * sa[:, None] + acc.astype(np.float64)).astype(np.float32)
    return acc.astype(np.float64) * 2.0 ** -16


def operands(M, N, K, seed):
    """Rows over 12 (A) and 6 (B) orders of magnitude, and blocks of K scaled
    apart, so that the per-(row, block) scales matter."""
    rng = np.random.default_rng(seed)
    A = rng.standard_normal((M, K))
    B = rng.standard_normal((N, K))
    A *= 10.0 ** rng.uniform(-6, 6, size=(M, 1))
    B *= 10.0 ** rng.uniform(-3, 3, size=(N, 1))
    A *= np.repeat(10.0 ** rng.uniform(-4, 4, size=(1, (K + CHUNK - 1) // CHUNK)), CHUNK, axis=1)[:, :K]
    return A.astype(np.float32), B.astype(np.float32)


def worst_over_bound(C, A, B):
    A64, B64 = A.astype(np.float64), B.astype(np.float64)
    ref = A64 @ B64.T
    bound = 2.0 ** -20 * (np.abs(A64) @ np.abs(B64).T) + 2.0 ** -23 * np.abs(ref)
    return float(np.max(np.abs(C - ref) / np.maximum(bound, 1e-300)))


def test_scales_are_the_smallest_power_of_two_at_or_above():
    m = np.array([0.0, 1.0, 0.75, 0.5, 3.0, 2.0 ** -30 * 1.5, 1e30])
    s = pow2_ceil(m)
    assert np.all(s >= m) and np.all((s / 2 < m) | (m == 0))
    assert list(s[:5]) == [1.0, 1.0, 1.0, 0.5, 4.0]


def test_digits_hold_fp32_values():
    rng = np.random.default_rng(0)
    X = (rng.standard_normal((64, 512)) * 10.0 ** rng.uniform(-8, 8, size=(64, 1))).astype(np.float32)
    X[:, 200:260] *= np.float32(1e-5)                       # small entries beside large ones in a block
    X[3, :] = 0.0
    sig = np.repeat(block_scales(X), CHUNK, axis=1)[:, :X.shape[1]]
    d = digits(X, sig)
    assert all(np.all(np.abs(x) <= 256) for x in d)         # 9 bits: exact in bf16
    rec = sig / 256.0 * (d[0] + d[1] * 2.0 ** -9 + d[2] * 2.0 ** -18)
    err = np.abs(rec - X.astype(np.float64))
    assert np.all(err <= 2.0 ** -27 * sig)
    near = np.abs(X) >= sig / 8                              # 27 digit bits cover fp32's 24 there
    assert np.all(err[near] == 0.0)
    assert np.count_nonzero(err) > 0                         # the small entries do round


def test_leading_chunk_sums_are_exact_in_fp32():
    # the extreme case: every digit 256, one 128-wide chunk
    d = np.full(CHUNK, 256.0)
    assert float(d @ d) == 2.0 ** 23
    rng = np.random.default_rng(1)
    for _ in range(20):
        a = rng.integers(-256, 257, size=CHUNK).astype(np.float64)
        b = rng.integers(-256, 257, size=CHUNK).astype(np.float64)
        s = np.float32(0.0)
        for k in rng.permutation(CHUNK):                    # any order
            s = np.float32(s + np.float32(a[k] * b[k]))
            assert abs(float(s)) <= 2.0 ** 23
        assert float(s) == float(a @ b)


@pytest.mark.parametrize("shape", [(48, 40, 300), (33, 17, 129), (16, 64, 1024)])
def test_six_digit_products_meet_the_kernel_bound(shape):
    A, B = operands(*shape, seed=sum(shape))
    assert worst_over_bound(digit_gemm(A, B), A, B) <= 0.25


@pytest.mark.parametrize("variant", ["three pairs", "two digits", "without (0, 2)", "without (1, 1)",
                                     "without (2, 0)"])
def test_fewer_terms_break_the_bound(variant):
    A, B = operands(48, 40, 300, seed=7)
    if variant == "three pairs":
        C = digit_gemm(A, B, pairs=SIX_PAIRS[:3])
    elif variant == "two digits":
        C = digit_gemm(A, B, pairs=[p for p in SIX_PAIRS if max(p) < 2], ndig=2)
    else:
        dropped = tuple(int(x) for x in variant[9:-1].split(", "))
        C = digit_gemm(A, B, pairs=[p for p in SIX_PAIRS if p != dropped])
    assert worst_over_bound(C, A, B) > 5.0
