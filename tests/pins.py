"""Checks that pin the CPU oracle to facts other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with what the Fathom page and the mathematics fix:
library routines (numpy float16 rounding), exact rational arithmetic, closed
properties (the t-plane prefix is the t-bit quantiser), brute force on tiny
inputs, hand-derived fixtures in ``tests/golden`` and textbook softmax
attention.  ``tests/test_oracle_pins.py`` runs them on the oracle as built;
``tests/test_oracle_mutants.py`` runs them on builds with planted mistakes and
expects each mistake to trip at least one of them.
"""
from __future__ import annotations

import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------ helpers

def bf16_bits_of(x) -> np.ndarray:
    """Round float values to bf16 (torch's round-to-nearest-even) -> uint16 patterns."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_value(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def unpack_codes(planes: np.ndarray, n: int, t: int = 4) -> np.ndarray:
    """t-bit prefix codes [n][D] read from planes [D][4][nb] with numpy's
    little-endian bit unpacking (word bit i = token i of the block)."""
    D, _, nb = planes.shape
    by = np.ascontiguousarray(planes).view(np.uint8).reshape(D, 4, nb * 8)
    bits = np.unpackbits(by, axis=-1, bitorder="little")[:, :, :n].astype(np.int64)
    c = np.zeros((D, n), dtype=np.int64)
    for p in range(t):
        c = (c << 1) | bits[:, p, :]
    return c.T


def block_scale(a: float) -> float:
    """fp16 scale of a block with max |k| = a, by numpy's float16 rounding,
    saturating at 65504."""
    x = a / 8.0
    if x >= 65504.0:
        return 65504.0
    return float(np.float16(x))


def exact_codes(k_bits: np.ndarray, t: int = 4) -> np.ndarray:
    """Direct t-bit quantiser clip(floor(k / (s 2^(4-t))), -2^(t-1), 2^(t-1)-1) + 2^(t-1)
    with exact rational arithmetic; s from numpy's float16 rounding of blockmax/8."""
    n, D = k_bits.shape
    kv = bf16_value(k_bits)
    out = np.zeros((n, D), dtype=np.int64)
    if t == 0:
        return out
    half = 1 << (t - 1)
    for b0 in range(0, n, 64):
        blk = kv[b0:b0 + 64]
        for j in range(D):
            a = float(np.max(np.abs(blk[:, j])))
            s = block_scale(a)
            for r in range(blk.shape[0]):
                if s == 0.0:
                    out[b0 + r, j] = half
                    continue
                f = math.floor(Fraction(blk[r, j]) / (Fraction(s) * (2 ** (4 - t))))
                out[b0 + r, j] = min(max(f, -half), half - 1) + half
    return out


def dequant_direct(k_bits: np.ndarray, depth: np.ndarray) -> np.ndarray:
    """Keys read at depth t_j, built straight from k (numpy float64):
    s ((c_t + 1/2) 2^(4-t) - 8), zero at t = 0."""
    n, D = k_bits.shape
    kv = bf16_value(k_bits)
    out = np.zeros((n, D), dtype=np.float64)
    for b0 in range(0, n, 64):
        blk = kv[b0:b0 + 64]
        for j in range(D):
            t = int(depth[j])
            if t == 0:
                continue
            s = block_scale(float(np.max(np.abs(blk[:, j]))))
            if s == 0.0:
                continue
            cell = s * 2.0 ** (4 - t)
            half = 1 << (t - 1)
            ct = np.clip(np.floor(blk[:, j] / cell), -half, half - 1) + half
            out[b0:b0 + blk.shape[0], j] = s * ((ct + 0.5) * 2.0 ** (4 - t) - 8.0)
    return out


def _keys(rng, n, D, spread=True):
    sig = np.exp(0.75 * rng.standard_normal(D)) if spread else np.ones(D)
    return bf16_bits_of(rng.standard_normal((n, D)) * sig)


# ------------------------------------------------------------------ scalars

def pin_fp16(o):
    rng = np.random.default_rng(11)
    xs = list(np.exp(rng.uniform(np.log(2.0 ** -30), np.log(70000.0), 4000)))
    # exact halfway points between neighbouring halves (ties to even)
    for base in [1.0, 1.5, 0.75, 1024.0, 2.0 ** -15, 2.0 ** -20, 60000.0]:
        h = np.float16(base)
        nxt = np.nextafter(h, np.float16(np.inf))
        xs.append((float(h) + float(nxt)) / 2)
    for x in xs:
        got = o.fp16_bits(float(x))
        if x >= 65504.0:
            assert got == 0x7BFF, (x, got)
        else:
            want = int(np.array([x], dtype=np.float64).astype(np.float16).view(np.uint16)[0])
            assert got == want, (x, hex(got), hex(want))
    pats = np.arange(0, 0x7C00, dtype=np.uint16)
    vals = pats.view(np.float16).astype(np.float64)
    for p in range(0, 0x7C00, 7):
        assert o.fp16_value(int(p)) == vals[p]


# ------------------------------------------------------------------ encode

def _bf16_below(x: float) -> int:
    """Bit pattern of the largest bf16 value below x."""
    b = int(bf16_bits_of([x])[0])
    if x > 0:
        return b - 1
    if x < 0:
        return b + 1
    return 0x8001


def _adversarial_block(D):
    """One 64-token block per channel with keys on and just below every cell
    boundary: blockmax 8 (s = 1) on even channels, 3 (s = 0.375) on odd ones."""
    out = np.zeros((64, D), dtype=np.uint16)
    for j in range(D):
        sc = 1.0 if j % 2 == 0 else 0.375
        pats = []
        for m in range(-8, 9):
            pats.append(int(bf16_bits_of([m * sc])[0]))
            pats.append(_bf16_below(m * sc))
        pats = (pats * 2)[:64]
        pats[0], pats[1] = int(bf16_bits_of([8 * sc])[0]), int(bf16_bits_of([-8 * sc])[0])
        out[:, j] = pats
    return out


def pin_codes_exact(o):
    rng = np.random.default_rng(12)
    n, D = 3 * 64 + 17, 16
    k = _keys(rng, n, D)
    k[:, 3] = 0  # an all-zero channel
    k[:64] = _adversarial_block(D)
    nb = (n + 63) // 64
    scales, planes = o.encode(k, nb + 2)
    got = unpack_codes(planes, n)
    want = exact_codes(k)
    assert np.array_equal(got, want), np.argwhere(got != want)[:5]
    kv = bf16_value(k)
    for b in range(nb):
        for j in range(D):
            a = float(np.max(np.abs(kv[64 * b:64 * b + 64, j])))
            w = np.array([block_scale(a)], dtype=np.float16).view(np.uint16)[0]
            assert scales[j, b] == w, (b, j, hex(scales[j, b]), hex(w))
    # blocks past the data are untouched, and absent tokens of the tail block are 0 bits
    assert not planes[:, :, nb:].any() and not scales[:, nb:].any()
    tail = planes[:, :, nb - 1]
    assert not (tail >> np.uint64(n - 64 * (nb - 1))).any()


def pin_prefix_quantiser(o):
    rng = np.random.default_rng(13)
    n, D = 2 * 64 + 5, 12
    k = _keys(rng, n, D)
    k[64:128] = _adversarial_block(D)
    _, planes = o.encode(k, 3)
    for t in range(5):
        assert np.array_equal(unpack_codes(planes, n, t), exact_codes(k, t)), t


def pin_special_values(o):
    D = 4
    k = np.zeros((64, D), dtype=np.float32)
    k[:, 0] = np.linspace(-1.0, 1.0, 64)
    k[5, 0], k[6, 0], k[7, 0] = 1.25, -1.25, 0.0   # +a, -a, 0 with a = 1.25
    k[:, 1] = 0.0                                   # all-zero channel
    k[:, 2] = 2.0 ** -30                            # blockmax/8 underflows fp16
    k[:, 3] = 1e30                                  # blockmax/8 above fp16 range
    kb = bf16_bits_of(k)
    scales, planes = o.encode(kb, 1)
    c = unpack_codes(planes, 64)
    assert c[5, 0] == 15 and c[6, 0] == 0 and c[7, 0] == 8
    assert scales[1, 0] == 0 and np.all(c[:, 1] == 8)
    assert scales[2, 0] == 0 and np.all(c[:, 2] == 8)
    assert scales[3, 0] == 0x7BFF and np.all(c[:, 3] == 15)


def pin_bit_order_golden(o):
    g = json.load(open(os.path.join(GOLDEN, "bitplane_order.json")))
    k = np.array([(i % 16) - 8 for i in range(64)], dtype=np.float32)[:, None]
    scales, planes = o.encode(bf16_bits_of(k), 1)
    assert int(scales[0, 0]) == int(g["scale_fp16"], 16)
    for p in range(4):
        assert int(planes[0, p, 0]) == int(g["planes"][p], 16), (p, hex(int(planes[0, p, 0])))


# ------------------------------------------------------------------ scores

def pin_scores(o):
    rng = np.random.default_rng(14)
    n, D, G = 150, 128, 4
    k = _keys(rng, n, D)
    q = rng.standard_normal((G, D)).astype(np.float32)
    scales, planes = o.encode(k, 3)
    for depth in [np.full(D, 4, np.uint8), rng.integers(0, 5, D).astype(np.uint8),
                  np.array([1, 2] * 64, np.uint8)]:
        got = o.scores(n, scales, planes, depth, q)
        want = q.astype(np.float64) @ dequant_direct(k, depth).T
        scale = np.abs(q).astype(np.float64) @ np.abs(dequant_direct(k, depth)).T
        assert np.all(np.abs(got - want) <= 1e-12 * (scale + 1e-300)), np.max(np.abs(got - want))
    # full depth = dot product with s (c - 7.5), c the exact 4-bit codes
    c = exact_codes(k[:64])
    kv = bf16_value(k[:64])
    s = np.array([block_scale(float(np.max(np.abs(kv[:, j])))) for j in range(D)])
    khat = s[None, :] * (c - 7.5)
    got = o.scores(64, scales, planes, np.full(D, 4, np.uint8), q)
    assert np.allclose(got, q.astype(np.float64) @ khat.T, rtol=1e-12, atol=1e-12)
    # a channel read at depth 0 contributes exactly nothing
    depth = rng.integers(1, 5, D).astype(np.uint8)
    depth[7] = 0
    k2 = k.copy()
    k2[:, 7] = bf16_bits_of(rng.standard_normal(n) * 50)
    s2, p2 = o.encode(k2, 3)
    assert np.array_equal(o.scores(n, scales, planes, depth, q), o.scores(n, s2, p2, depth, q))
    # a code has four planes: depth values above 4 read the whole code (the
    # full-depth closed form above), never the next channel's planes
    for big in (5, 17, 255):
        depth = rng.integers(0, 5, D).astype(np.uint8)
        depth[rng.choice(D, 20, replace=False)] = big
        got = o.scores(n, scales, planes, depth, q)
        want = q.astype(np.float64) @ dequant_direct(k, np.minimum(depth, 4)).T
        scale = np.abs(q).astype(np.float64) @ np.abs(dequant_direct(k, np.minimum(depth, 4))).T
        assert np.all(np.abs(got - want) <= 1e-12 * (scale + 1e-300)), (big, np.max(np.abs(got - want)))


# ------------------------------------------------------------------ depths

def _importance32(q, sigma2):
    acc = np.zeros(q.shape[1], np.float32)
    for h in range(q.shape[0]):
        acc = (acc + (q[h] * q[h]) * sigma2).astype(np.float32)
    return acc


def _cost_q(t):
    t = np.asarray(t)
    return 4 * t.sum(axis=-1) + (t > 0).sum(axis=-1)


_ALL8 = None


def _all_depth_vectors():
    global _ALL8
    if _ALL8 is None:
        _ALL8 = np.array(list(itertools.product(range(5), repeat=8)), dtype=np.int64)
    return _ALL8


def pin_alloc_bruteforce(o):
    T = _all_depth_vectors()
    planes_used = T.sum(axis=1)
    pw = 4.0 ** (-T.astype(np.float64))
    rng = np.random.default_rng(15)
    for trial in range(6):
        q = rng.standard_normal((4, 8)).astype(np.float32)
        sigma2 = np.exp(rng.standard_normal(8)).astype(np.float32)
        if trial == 5:
            q[:, 2] = 0.0  # a channel of no importance is never read
        g = _importance32(q, sigma2).astype(np.float64)
        obj_all = pw @ g
        for B in range(0, 137, 3):
            t = o.alloc_depths(q, sigma2, B).astype(np.int64)
            assert _cost_q(t) <= B
            m = planes_used <= t.sum()
            best = obj_all[m].min()
            mine = float(pw[np.ravel_multi_index(t, (5,) * 8)] @ g)
            assert mine <= best * (1 + 1e-12) + 1e-300, (trial, B, t, mine, best)
            # stop rule: the next item in value order is absent, worthless or does not fit
            cand = [(g[j] * 4.0 ** -t[j], -j) for j in range(8) if t[j] < 4]
            if cand:
                v, mj = max(cand)
                j = -mj
                step = 5 if t[j] == 0 else 4
                assert v <= 0 or _cost_q(t) + step > B, (trial, B, t)
            if trial == 5:
                assert t[2] == 0


def pin_alloc_golden(o):
    g = json.load(open(os.path.join(GOLDEN, "alloc_cases.json")))
    for case in g["cases"]:
        D = len(case["q_head0"])
        q = np.zeros((4, D), np.float32)
        q[0] = case["q_head0"]
        sigma2 = np.array(case["sigma2"], np.float32)
        for B, want in zip(case["budgets_q"], case["depths"]):
            got = o.alloc_depths(q, sigma2, B)
            assert list(got) == want, (case["why"][:40], B, list(got), want)
    u = g["uniform"]
    q = np.ones((4, u["D"]), np.float32)
    for bits, n_ch in u["cases"]:
        got = o.alloc_depths(q, np.ones(u["D"], np.float32), 4 * bits)
        assert list(got) == [1] * n_ch + [0] * (u["D"] - n_ch), bits


def pin_fixed_depths(o):
    from workload.bytes_model import depth_bits
    rng = np.random.default_rng(16)
    q = rng.standard_normal((4, 128)).astype(np.float32)
    q[:, 40] = q[:, 41]  # an exact tie: the lower index ranks first
    a = np.zeros(128, np.float32)
    for h in range(4):
        a = (a + np.abs(q[h])).astype(np.float32)
    order = sorted(range(128), key=lambda j: (-float(a[j]), j))
    for r, t, bits in [(32, 4, 136), (16, 4, 68), (128, 2, 288), (200, 1, 160)]:
        d = o.fixed_depths(q, r, t)
        want = np.zeros(128, np.uint8)
        want[order[:r]] = t
        assert np.array_equal(d, want), (r, t)
        assert depth_bits(d) == bits


def _dyadic_calibration(rng, m_q, G, m_k, D):
    """Calibration data whose sums, means and products are exact in double:
    |q| multiples of 1/4 in [0, 8], |k| multiples of 1/8 in [0, 4] (exact in
    bf16), random signs, m_q G and m_k powers of two."""
    q = rng.integers(0, 33, (m_q, G, D)) / 4.0 * rng.choice([-1.0, 1.0], (m_q, G, D))
    k = rng.integers(0, 33, (m_k, D)) / 8.0 * rng.choice([-1.0, 1.0], (m_k, D))
    return q.astype(np.float32), k


def _calibration_order(q, k):
    """Channels by (mean|q| mean|k| desc, index asc), in exact rational arithmetic."""
    from fractions import Fraction
    m_q, G, D = q.shape
    st = []
    for j in range(D):
        a = sum(Fraction(float(abs(x))) for x in q[:, :, j].ravel()) / (m_q * G)
        b = sum(Fraction(float(abs(x))) for x in k[:, j]) / k.shape[0]
        st.append(a * b)
    return sorted(range(D), key=lambda j: (-st[j], j)), st


def pin_calibrated_channels(o):
    from workload.bytes_model import depth_bits
    rng = np.random.default_rng(20)
    D, G, m_q, m_k = 32, 4, 8, 16
    q, k = _dyadic_calibration(rng, m_q, G, m_k, D)
    # an exact tie of equal columns, and one of equal products from different
    # factors (twice the queries, half the keys): both go to the lower index
    q[:, :, 9], k[:, 9] = q[:, :, 4], k[:, 4]
    q[:, :, 12], k[:, 12] = 2 * q[:, :, 6], k[:, 6] / 2
    # a channel with the largest queries and near-zero keys, one with the
    # largest keys and small queries: neither statistic alone decides
    q[:, :, 0], k[:, 0] = 8.0, 0.125
    q[:, :, 1], k[:, 1] = 0.25, 4.0
    # heads differ: the mean runs over every head of the group
    q[:, 1:, 2] = 0.0
    q[:, 0, 2] = 8.0
    k[:, 2] = 2.0
    order, st = _calibration_order(q, k)
    assert st[9] == st[4] and st[12] == st[6]
    kb = bf16_bits_of(k)
    for c, t in [(8, 4), (16, 2), (32, 1), (0, 4), (40, 3)]:
        d = o.calibrate_channels(q, kb, c, t)
        want = np.zeros(D, np.uint8)
        want[order[:c]] = t
        assert np.array_equal(d, want), (c, t, list(d), list(want))
    # storage order of the calibration tokens does not matter (exact sums)
    pq, pk = rng.permutation(m_q), rng.permutation(m_k)
    assert np.array_equal(o.calibrate_channels(q[pq], kb[pk], 8, 4), o.calibrate_channels(q, kb, 8, 4))
    # one calibration query and keys of equal magnitude: the SparQ set of that query
    q1 = rng.standard_normal((1, 4, 128)).astype(np.float32)
    k1 = bf16_bits_of(np.where(rng.random((8, 128)) < 0.5, -1.5, 1.5))
    a = np.zeros(128, np.float64)
    for h in range(4):
        a = a + np.abs(q1[0, h]).astype(np.float64)
    sparq = sorted(range(128), key=lambda j: (-a[j], j))
    d = o.calibrate_channels(q1, k1, 32, 4)
    want = np.zeros(128, np.uint8)
    want[sparq[:32]] = 4
    assert np.array_equal(d, want)
    assert depth_bits(d) == 136  # 32 channels x 4 bits + their scales
    # a channel permutation permutes the set (tie-free random data)
    qr = rng.standard_normal((16, 4, 128)).astype(np.float32)
    kr = bf16_bits_of(rng.standard_normal((64, 128)) * np.exp(0.75 * rng.standard_normal(128)))
    perm = rng.permutation(128)
    d0 = o.calibrate_channels(qr, kr, 32, 4)
    assert np.array_equal(o.calibrate_channels(qr[:, :, perm], kr[:, perm], 32, 4), d0[perm])
    # and matches means formed by numpy's own reductions
    stat = np.abs(qr.astype(np.float64)).mean(axis=(0, 1)) * np.abs(bf16_value(kr)).mean(axis=0)
    want = np.zeros(128, np.uint8)
    want[np.argsort(-stat, kind="stable")[:32]] = 4
    assert np.array_equal(d0, want)


def _round_fp32(v):
    """Nearest float32 to the rational v (ties to even), as a Fraction."""
    from fractions import Fraction
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)                      # subnormals share the lowest exponent
    ulp = Fraction(2) ** (e - 23)
    q, r = divmod(a / ulp, 1)
    q = int(q)
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and q % 2 == 1):
        q += 1
    return sign * q * ulp


def _bf16_of_fraction(v) -> int:
    """bf16 pattern of a float32 value given as a Fraction (round to nearest even)."""
    f = np.float32(float(v))              # exact: v is a float32 value
    u = int(np.array([f], np.float32).view(np.uint32)[0])
    u += 0x7FFF + ((u >> 16) & 1)
    return (u >> 16) & 0xFFFF


def pin_basis(o):
    from fractions import Fraction
    rng = np.random.default_rng(21)
    D = 128
    # exact: each output is a chain of float32 fused multiply-adds in channel order
    x = (rng.standard_normal((2, D)) * np.exp(rng.standard_normal((2, D)))).astype(np.float32)
    R = rng.standard_normal((D, D)).astype(np.float32)
    y = o.rotate(x, R)
    for r in range(2):
        for l in range(0, D, 9):
            acc = Fraction(0)
            for j in range(D):
                acc = _round_fp32(Fraction(float(x[r, j])) * Fraction(float(R[j, l])) + acc)
            assert y[r, l] == np.float32(float(acc)), (r, l)
    kb = bf16_bits_of(rng.standard_normal((3, D)) * 3)
    yk = o.rotate_keys(kb, R)
    xk = bf16_value(kb).astype(np.float32)
    for r in range(3):
        for l in range(0, D, 13):
            acc = Fraction(0)
            for j in range(D):
                acc = _round_fp32(Fraction(float(xk[r, j])) * Fraction(float(R[j, l])) + acc)
            assert int(yk[r, l]) == _bf16_of_fraction(acc), (r, l)
    # identity and permutation bases move bits, nothing else
    k = bf16_bits_of(rng.standard_normal((50, D)) * 2)
    assert np.array_equal(o.rotate_keys(k, np.eye(D, dtype=np.float32)), k)
    perm = rng.permutation(D)
    P = np.zeros((D, D), np.float32)
    P[perm, np.arange(D)] = 1.0
    assert np.array_equal(o.rotate_keys(k, P), k[:, perm])
    # an orthogonal basis (signed, normalised Hadamard) keeps inner products
    H = np.array([[1.0]])
    while H.shape[0] < D:
        H = np.block([[H, H], [H, -H]])
    Hs = (H * rng.choice([-1.0, 1.0], D)[:, None] / np.sqrt(D)).astype(np.float32)
    q = rng.standard_normal((4, D)).astype(np.float32)
    kk = rng.standard_normal((6, D)).astype(np.float32)
    ref = q.astype(np.float64) @ kk.astype(np.float64).T
    got = o.rotate(q, Hs).astype(np.float64) @ o.rotate(kk, Hs).astype(np.float64).T
    assert np.allclose(got, ref, rtol=0, atol=1e-4 * np.abs(ref).max())
    # the identity basis is a no-op for a whole decode of one unit
    n = 300
    kb2, vb2 = bf16_bits_of(rng.standard_normal((n, D)) * 2), bf16_bits_of(rng.standard_normal((n, D)))
    q2 = rng.standard_normal((4, D)).astype(np.float32)
    s2 = np.exp(rng.standard_normal(D)).astype(np.float32)
    a = o.decode_unit(kb2, vb2, q2, s2, 92, 64)
    b = o.decode_unit(kb2, vb2, q2, s2, 92, 64, basis=np.eye(D, dtype=np.float32))
    for key in ("planes", "scales", "depth", "idx", "out"):
        assert np.array_equal(a[key], b[key]), key


# ------------------------------------------------------------------ selection

def _topk_brute(score, k, n_sink=4, n_recent=32):
    n = len(score)
    lo = min(n_sink, n)
    hi = max(n - n_recent, lo)
    sel = set(range(lo)) | set(range(hi, n))
    cands = sorted(range(lo, hi), key=lambda i: (-score[i], i))
    sel |= set(cands[:max(k - n_sink - n_recent, 0)])
    out = sorted(sel)
    return out + [-1] * (k - len(out))


def pin_topk(o):
    rng = np.random.default_rng(17)
    for n in [0, 1, 3, 4, 20, 36, 37, 40, 64, 100, 256]:
        for k in [36, 40, 64]:
            s = np.round(rng.standard_normal(n) * 3) / 3  # many exact ties
            assert list(o.topk(s, k)) == _topk_brute(list(s), k), (n, k)
    s = rng.standard_normal(200)
    assert list(o.topk(s, 48, 0, 0)) == _topk_brute(list(s), 48, 0, 0)


def pin_union(o):
    rng = np.random.default_rng(18)
    for k in [1, 8, 40]:
        idx = np.stack([np.sort(rng.choice(60, size=k, replace=False)) for _ in range(4)]).astype(np.int32)
        idx[2, k // 2:] = -1
        uidx, umask = o.union(idx)
        want = sorted({int(i) for i in idx.ravel() if i >= 0})
        assert list(uidx) == want
        for i, m in zip(uidx, umask):
            assert m == sum(1 << h for h in range(4) if i in set(idx[h].tolist())), (i, m)


# ------------------------------------------------------------------ attention

def _softmax_attend(q, kv, vv):
    lg = (q.astype(np.float64) @ kv.T) / math.sqrt(q.shape[1])
    lg -= lg.max(axis=1, keepdims=True)
    w = np.exp(lg)
    w /= w.sum(axis=1, keepdims=True)
    return w @ vv


def pin_attention(o):
    rng = np.random.default_rng(19)
    n, D, G = 70, 128, 4
    k = bf16_bits_of(rng.standard_normal((n, D)) * 2)
    v = bf16_bits_of(rng.standard_normal((n, D)))
    q = rng.standard_normal((G, D)).astype(np.float32)
    all_idx = np.tile(np.arange(n, dtype=np.int32), (G, 1))
    ref = _softmax_attend(q, bf16_value(k), bf16_value(v))
    assert np.allclose(o.attend(q, k, v, all_idx), ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(o.dense_attend(q, k, v, n), ref, rtol=1e-12, atol=1e-12)
    # each head over its own subset, padding ignored
    idx = np.full((G, 20), -1, np.int32)
    for h in range(G):
        sub = np.sort(rng.choice(n, size=10 + h, replace=False))
        idx[h, :len(sub)] = sub
        want = _softmax_attend(q[h:h + 1], bf16_value(k[sub]), bf16_value(v[sub]))
        got = o.attend(q, k, v, idx)[h]
        assert np.allclose(got, want[0], rtol=1e-12, atol=1e-12)
    # one row: the output is that row's value; two equal keys: the mean of their values
    one = np.full((G, 2), -1, np.int32)
    one[:, 0] = 9
    assert np.array_equal(o.attend(q, k, v, one), np.tile(bf16_value(v[9]), (G, 1)))
    k2 = k.copy()
    k2[11] = k2[10]
    two = np.tile(np.array([10, 11], np.int32), (G, 1))
    assert np.allclose(o.attend(q, k2, v, two), np.tile((bf16_value(v[10]) + bf16_value(v[11])) / 2, (G, 1)),
                       rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ value-side depth (ReadKV, stage 2)

def exact_row_codes(v_bits: np.ndarray, t: int = 4) -> np.ndarray:
    """Direct t-bit codes of value rows [n][D] with the row's scale
    s = fp16(rowmax / 8) (numpy float16 rounding), exact rational floor."""
    n, D = v_bits.shape
    vv = bf16_value(v_bits)
    out = np.zeros((n, D), dtype=np.int64)
    if t == 0:
        return out
    half = 1 << (t - 1)
    for i in range(n):
        s = block_scale(float(np.max(np.abs(vv[i]))))
        for j in range(D):
            if s == 0.0:
                out[i, j] = half
                continue
            f = math.floor(Fraction(vv[i, j]) / (Fraction(s) * (2 ** (4 - t))))
            out[i, j] = min(max(f, -half), half - 1) + half
    return out


def unpack_row_codes(vplanes: np.ndarray, t: int = 4) -> np.ndarray:
    """t-bit prefix codes [n][D] from token-major planes [n][4][D/64] (numpy
    little-endian bit unpacking: bit b of word w = channel 64 w + b)."""
    n, _, W = vplanes.shape
    by = np.ascontiguousarray(vplanes).view(np.uint8).reshape(n, 4, W * 8)
    bits = np.unpackbits(by, axis=-1, bitorder="little").astype(np.int64)  # [n][4][D]
    c = np.zeros((n, W * 64), dtype=np.int64)
    for p in range(t):
        c = (c << 1) | bits[:, p, :]
    return c


def pin_value_codes(o):
    rng = np.random.default_rng(21)
    n, D = 9, 128
    v = bf16_bits_of(rng.standard_normal((n, D)) * np.exp(rng.standard_normal((n, 1))))
    v[2] = 0                                              # an all-zero row: scale 0, codes 8
    adv = _adversarial_block(2)[:, 0]                     # values on and below every cell edge, s = 1
    v[4, :64], v[4, 64:] = adv, adv
    vscales, vplanes = o.v_encode(v)
    for t in range(5):
        got, want = unpack_row_codes(vplanes, t), exact_row_codes(v, t)
        assert np.array_equal(got, want), (t, np.argwhere(got != want)[:5])
    vv = bf16_value(v)
    for i in range(n):
        w = np.array([block_scale(float(np.max(np.abs(vv[i]))))], dtype=np.float16).view(np.uint16)[0]
        assert vscales[i] == w, (i, hex(vscales[i]), hex(w))
    # reconstruction: the mid-rise cell midpoint of the t-bit code, zero at t = 0
    for i in (0, 4):
        s = block_scale(float(np.max(np.abs(vv[i]))))
        for t in range(5):
            ct = exact_row_codes(v[i:i + 1], t)[0]
            want = np.zeros(D) if t == 0 else s * ((ct + 0.5) * 2.0 ** (4 - t) - 8.0)
            assert np.array_equal(o.v_row(vscales, vplanes, i, t), want), (i, t)
    assert not o.v_row(vscales, vplanes, 2, 4).any()


def pin_value_bit_order_golden(o):
    g = json.load(open(os.path.join(GOLDEN, "value_plane_order.json")))
    v = bf16_bits_of(np.array([[(j % 16) - 8 for j in range(128)]], dtype=np.float32))
    vscales, vplanes = o.v_encode(v)
    assert int(vscales[0]) == int(g["scale_fp16"], 16)
    for p in range(4):
        for w in range(2):
            assert int(vplanes[0, p, w]) == int(g["planes"][p][w], 16), (p, w, hex(int(vplanes[0, p, w])))
    depth, used = o.v_alloc(np.ones(3), 1)
    assert list(depth) == [1, 0, 0] and used == 1


def pin_value_alloc_bruteforce(o):
    """The greedy depths minimise sum_r a_r 4^-t_r over every depth vector with
    as many planes (a concave separable objective: greedy is optimal), use
    min(budget, 4 n) planes when every weight is positive, and never read a
    row of zero weight."""
    n = 6
    T = np.array(list(itertools.product(range(5), repeat=n)), dtype=np.int64)
    used_all = T.sum(axis=1)
    pw = 4.0 ** (-T.astype(np.float64))
    rng = np.random.default_rng(22)
    for trial in range(5):
        a = rng.random(n) ** 3
        if trial == 4:
            a[1] = 0.0
        obj = pw @ a
        for B in range(0, 4 * n + 3):
            t, used = o.v_alloc(a, B)
            t = t.astype(np.int64)
            assert used == int(t.sum()) <= B
            if trial < 4:
                assert used == min(B, 4 * n), (trial, B, used)
            m = used_all <= used
            mine = float(pw[np.ravel_multi_index(t, (5,) * n)] @ a)
            assert mine <= obj[m].min() * (1 + 1e-12) + 1e-300, (trial, B, t)
            if trial == 4:
                assert t[1] == 0


def pin_value_attention(o):
    rng = np.random.default_rng(23)
    n, D, G = 40, 128, 4
    k = bf16_bits_of(rng.standard_normal((n, D)) * 1.5)
    v = bf16_bits_of(rng.standard_normal((n, D)))
    q = rng.standard_normal((G, D)).astype(np.float32)
    vscales, vplanes = o.v_encode(v)
    # a union of 25 rows; head h selects a subset, every row at least one head
    uidx = np.sort(rng.choice(n, size=25, replace=False)).astype(np.int32)
    umask = rng.integers(1, 16, size=25).astype(np.uint8)
    kv = bf16_value(k)
    p = np.zeros((G, 25))
    for h in range(G):
        sel = np.nonzero((umask >> h) & 1)[0]
        lg = (q[h].astype(np.float64) @ kv[uidx[sel]].T) / math.sqrt(D)
        w = np.exp(lg - lg.max())
        p[h, sel] = w / w.sum()
    weight = (p * p).sum(axis=0)
    # full depth: textbook attention over each head's rows with the 4-bit values
    full = o.attend_vdepth(q, k, vscales, vplanes, uidx, umask, 4 * 25)
    assert np.all(full["depth"] == 4)
    assert np.allclose(full["weight"], weight, rtol=1e-12, atol=1e-15)
    c4 = exact_row_codes(v[uidx], 4)
    s = np.array([block_scale(float(np.max(np.abs(bf16_value(v[i]))))) for i in uidx])
    vhat4 = s[:, None] * (c4 - 7.5)
    assert np.allclose(full["out"], p @ vhat4, rtol=1e-12, atol=1e-12)
    # a partial budget: the depths are the greedy allocation of the weights,
    # each row read through its own prefix
    part = o.attend_vdepth(q, k, vscales, vplanes, uidx, umask, 37)
    t = part["depth"].astype(np.int64)
    assert int(t.sum()) == 37
    assert np.array_equal(part["depth"], o.v_alloc(weight, 37)[0])
    vhat = np.zeros((25, D))
    for r in range(25):
        if t[r]:
            ct = exact_row_codes(v[uidx[r]:uidx[r] + 1], int(t[r]))[0]
            vhat[r] = s[r] * ((ct + 0.5) * 2.0 ** (4 - t[r]) - 8.0)
    assert np.allclose(part["out"], p @ vhat, rtol=1e-12, atol=1e-12)
    # the heaviest row is read deepest
    assert t[int(np.argmax(weight))] == t.max()
    # given depths: the same output as the allocation that produced them, and
    # any other depth vector is read through each row's own prefix too
    again = o.attend_vdepth(q, k, vscales, vplanes, uidx, umask, 0, depth_in=part["depth"])
    assert np.array_equal(again["out"], part["out"]) and np.array_equal(again["depth"], part["depth"])
    other = rng.integers(0, 5, size=25).astype(np.uint8)
    got = o.attend_vdepth(q, k, vscales, vplanes, uidx, umask, 0, depth_in=other)
    vo = np.zeros((25, D))
    for r in range(25):
        if other[r]:
            ct = exact_row_codes(v[uidx[r]:uidx[r] + 1], int(other[r]))[0]
            vo[r] = s[r] * ((ct + 0.5) * 2.0 ** (4 - int(other[r])) - 8.0)
    assert np.allclose(got["out"], p @ vo, rtol=1e-12, atol=1e-12)


ALL_PINS = [pin_fp16, pin_codes_exact, pin_prefix_quantiser, pin_special_values, pin_bit_order_golden,
            pin_scores, pin_alloc_bruteforce, pin_alloc_golden, pin_fixed_depths, pin_calibrated_channels,
            pin_basis, pin_topk, pin_union, pin_attention, pin_value_codes, pin_value_bit_order_golden,
            pin_value_alloc_bruteforce, pin_value_attention]
