"""Pins for the oracle's quantizer, record layout, pack/unpack and encode."""
import os

import numpy as np
import pytest

import oracle


def _cases(golden_dir):
    out = []
    for line in open(os.path.join(golden_dir, "pack_cases.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        parts = dict(p.strip().split("=", 1) for p in line.split("|"))
        out.append(([int(x) for x in parts["bits"].split(",")],
                    [int(x, 0) for x in parts["codes"].split(",")],
                    [int(x, 16) for x in parts["words"].split(",")]))
    return out


def test_pack_hand_built_records(golden_dir):
    cases = _cases(golden_dir)
    assert len(cases) >= 6
    for bits, codes, words in cases:
        rec = oracle.pack(codes, bits)
        assert [int(w) for w in rec] == words, (bits, [hex(int(w)) for w in rec])
        assert list(oracle.unpack(rec, bits)) == codes


def test_layout_fields_aligned_and_disjoint():
    rng = np.random.default_rng(3)
    for _ in range(50):
        bits = np.sort(rng.integers(0, 9, size=128))[::-1]
        off = oracle.layout(bits)
        used = np.zeros(int(bits.sum()), dtype=int)
        for j in range(128):
            for s in range(4):
                if bits[j] >> s & 1:
                    o, w = off[j, s], 1 << s
                    assert o % w == 0                       # aligned to its width
                    assert o // 32 == (o + w - 1) // 32     # never crosses a word
                    used[o:o + w] += 1
                else:
                    assert off[j, s] == -1
        assert np.all(used == 1)                            # every bit used exactly once


def test_pack_unpack_roundtrip_random():
    rng = np.random.default_rng(4)
    for trial in range(200):
        d = int(rng.integers(1, 130))
        bits = rng.integers(0, 9, size=d)
        extra = (-bits.sum()) % 32                          # pad the budget to whole words
        bits = np.concatenate([bits, np.full(extra // 8, 8), [extra % 8] if extra % 8 else []]).astype(int)
        u = np.array([rng.integers(0, 1 << b) if b else 0 for b in bits])
        rec = oracle.pack(u, bits)
        assert len(rec) * 32 == bits.sum()
        assert np.array_equal(oracle.unpack(rec, bits), u)


def test_quantizer_levels_and_error_bound():
    step = np.array([0.5, 0.25, 2.0, 1.0], dtype=np.float32)
    bits = np.array([1, 3, 8, 0])
    # b=1: levels +-step/2; b=3: 8 levels centered on zero
    assert list(oracle.quantize([-0.1, 0.0, 0.0, 5.0], step, bits)[:2]) == [0, 4]
    assert list(oracle.dequantize([0, 1, 0, 0], step, bits)) == [-0.25, -0.625, -255.0, 0.0]
    rng = np.random.default_rng(5)
    for b in range(1, 9):
        N = 2 ** b
        s = np.float32(0.37)
        c = rng.uniform(-N * s / 2, N * s / 2, size=2000) * 0.999
        u = np.array([oracle.quantize([x], [s], [b])[0] for x in c[:200]])
        assert u.min() >= 0 and u.max() <= N - 1
        ch = np.array([oracle.dequantize([k], [s], [b])[0] for k in u])
        assert np.all(np.abs(ch - c[:200]) <= s / 2 * (1 + 1e-6))
    # clamping outside the range
    assert oracle.quantize([1e9], [1.0], [4])[0] == 15 and oracle.quantize([-1e9], [1.0], [4])[0] == 0
    # round half to even on an exact fp32 tie: v = 0/1 + 0.5 -> 0 ; v = 1.5 -> 2
    assert oracle.quantize([0.0], [1.0], [1])[0] == 0
    assert oracle.quantize([1.0], [1.0], [2])[0] == 2


def test_encode_reconstruct_error_matches_quantizer_mse():
    """Gaussian coefficients through the KLT: measured MSE per channel matches
    lam_j * MSE_b(s_b), the model the step sizes were chosen under."""
    rng = np.random.default_rng(6)
    d, n = 64, 100000
    lam = 0.9 ** np.arange(d)
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    X = (rng.standard_normal((n, d)) * np.sqrt(lam)) @ Qm.T
    T = Qm.T                                  # exact KLT of the source
    bits, _ = oracle.allocate_bits(lam, 160)
    step = oracle.steps(lam, bits)
    rec, codes, _ = oracle.encode(X, T, np.zeros(d), step, bits, want_codes=True)
    Xh = oracle.reconstruct(rec, Qm, np.zeros(d), step, bits)
    c, ch = X @ T.T, (Xh @ Qm)
    for j in range(d):
        pred = lam[j] * (oracle.gauss_uniform_mse(bits[j], oracle.gauss_uniform_step(bits[j]))
                         if bits[j] else 1.0)
        e2 = (c[:, j] - ch[:, j]) ** 2
        meas, se = e2.mean(), e2.std() / np.sqrt(n)      # tails make the overload part noisy
        assert abs(meas - pred) < 4 * se + 0.01 * pred, (j, bits[j], meas, pred, se)
    assert np.array_equal(oracle.unpack(rec[17], bits), codes[17])


def test_compression_ratio_arithmetic():
    """16-bit cache over the average bits per element: about 5.8x at 2.75 bits."""
    for rbar, ratio, nbytes in ((2.75, 5.818, 44), (2.0, 8.0, 32), (4.0, 4.0, 64)):
        bits, _ = oracle.allocate_bits(0.95 ** np.arange(128), int(rbar * 128))
        rec = oracle.pack(np.zeros(128, dtype=int), bits)
        assert rec.nbytes == nbytes
        assert abs(16 * 128 / (rec.nbytes * 8) - ratio) < 1e-3
    assert round(16 / 2.75, 1) == 5.8
