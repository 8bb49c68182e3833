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


def test_layout_codes_contiguous_and_disjoint():
    """Every record bit belongs to exactly one code; pruned channels take none."""
    rng = np.random.default_rng(3)
    for _ in range(50):
        bits = np.sort(rng.integers(0, 9, size=128))[::-1]
        off = oracle.layout(bits)
        order = oracle.record_order(bits)
        assert sorted(order.tolist()) == [j for j in range(128) if bits[j] > 0]
        used = np.zeros(int(bits.sum()), dtype=int)
        pos = 0
        for j in order:                                     # codes follow the order, back to back
            assert off[j] == pos
            used[pos:pos + bits[j]] += 1
            pos += bits[j]
        assert np.all(off[bits == 0] == -1)
        assert np.all(used == 1)


def test_order_keeps_three_consecutive_codes_at_seven_bits():
    """On the workloads' spectra the order rule leaves no byte of a record
    holding parts of more than four codes."""
    for lam_decay, B in ((0.95, 352), (0.93, 352), (0.9, 352), (0.95, 256), (0.95, 512)):
        bits, _ = oracle.allocate_bits(lam_decay ** np.arange(128), B)
        off = oracle.layout(bits)
        per_byte = np.zeros(B // 8, dtype=int)
        for j in range(128):
            if bits[j]:
                per_byte[off[j] // 8:(off[j] + bits[j] - 1) // 8 + 1] += 1
        assert per_byte.max() <= 4, (lam_decay, B, per_byte.max())


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


def test_cache_tiling_hand_positions():
    """Positions worked out by hand from the tiling rule (W = 11 words): keys of
    token 19 word 9 -> tile word 176 + 128 + 6 + 2 + 1 = 313; token 45 word 2
    -> 352 + 6*8 + 4 + 1 = 405.  Values: half-word e of token 19 -> word
    16 e + 9 (high half); of token 45 -> 352 + 16 e + 6 (high half)."""
    W, L = 11, 64
    rec = np.array([[(t << 8) | w for w in range(W)] for t in range(L)], dtype=np.uint32)
    kc = oracle.cache_put(rec, oracle.KEYS)
    assert kc.size == L * W
    assert kc[313] == rec[19, 9] and kc[405] == rec[45, 2]
    assert kc[0] == rec[0, 0] and kc[1] == rec[1, 0] and kc[2] == rec[0, 1]
    vc = oracle.cache_put(rec, oracle.VALUES)
    for e in range(2 * W):
        hw = lambda t: (int(rec[t, e // 2]) >> (16 * (e % 2))) & 0xFFFF  # noqa: E731
        assert int(vc[16 * e + 9]) >> 16 == hw(19)
        assert int(vc[352 + 16 * e + 6]) >> 16 == hw(45)
        assert int(vc[16 * e]) & 0xFFFF == hw(0) and int(vc[16 * e]) >> 16 == hw(1)


def test_cache_tiling_is_a_permutation_and_round_trips():
    rng = np.random.default_rng(7)
    for W in (8, 11, 16, 5, 1):
        L = 96
        rec = rng.integers(0, 2 ** 32, size=(L, W), dtype=np.uint64).astype(np.uint32)
        for kind in (oracle.KEYS, oracle.VALUES):
            c = oracle.cache_put(rec, kind)
            assert np.array_equal(oracle.cache_get(c, W, kind, L), rec)
            # each cache bit comes from exactly one record bit: place one-hot records
            seen = np.zeros(L * W * 32, dtype=int)
            for t in (0, 1, 15, 16, 31, 32, 63, 95):
                for w in range(W):
                    for k in (0, 13, 16, 31):
                        one = np.zeros((L, W), dtype=np.uint32)
                        one[t, w] = np.uint32(1 << k)
                        cc = oracle.cache_put(one, kind)
                        nz = np.flatnonzero(cc)
                        assert nz.size == 1
                        bit = nz[0] * 32 + int(np.log2(int(cc[nz[0]])))
                        seen[bit] += 1
            assert seen.max() == 1
        # partial writes leave other tokens alone
        c = oracle.cache_put(rec, oracle.VALUES)
        new = rng.integers(0, 2 ** 32, size=(3, W), dtype=np.uint64).astype(np.uint32)
        oracle.cache_put(new, oracle.VALUES, cache=c, start=33)
        back = oracle.cache_get(c, W, oracle.VALUES, L)
        assert np.array_equal(back[33:36], new)
        assert np.array_equal(back[:33], rec[:33]) and np.array_equal(back[36:], rec[36:])


def test_prequant_hand_values():
    """The pre-rounding value v = c/Delta + (2^b - 1)/2, rounded once to fp32,
    worked out by hand ("End-to-End Implementation": rotate, then quantize per
    channel; mid-rise levels), and the code each one gives."""
    cases = [
        # c,          step,  b, v (exact),                 code
        (0.0,         1.596, 1, 0.5,                       0),    # exact fp32 tie -> even (0)
        (0.8,         1.6,   1, 1.0,                       1),    # 0.8/1.6 in fp64 -> 1.0 after fp32 rounding
        (0.25,        0.5,   3, 4.0,                       4),
        (-1.0,        0.5,   3, 1.5,                       2),    # tie -> even (2)
        (1.0,         0.25,  8, 131.5,                     132),  # tie -> even (132)
        (-40.0,       0.25,  8, -32.5,                     0),    # below the range: clamped
        (40.0,        0.25,  8, 287.5,                     255),  # above the range: clamped
        (1.0 / 3.0,   1.0,   2, np.float32(11.0 / 6.0),    2),    # 11/6 rounded to the nearest fp32
        (1.0 + 1e-9,  1.0,   2, 2.5,                       2),    # 2.500000001 rounds to fp32 2.5: tie -> 2
        (5.0,         1.0,   0, 0.0,                       0),    # pruned channel
    ]
    for c, s, b, v, u in cases:
        got = oracle.prequant([c], [s], [b])[0]
        assert got.dtype == np.float32
        assert got == np.float32(v), (c, s, b, got, v)
        assert oracle.quantize([c], [s], [b])[0] == u, (c, s, b)
    # the fp32 rounding is the one the decision uses: just above a half-integer
    # in fp64 but equal to it in fp32 rounds to even, just above it in fp32 rounds up
    up = float(np.nextafter(np.float32(2.5), np.float32(3.0)))
    assert oracle.prequant([up - 1.5], [1.0], [2])[0] == np.float32(up)
    assert oracle.quantize([up - 1.5], [1.0], [2])[0] == 3


def test_quantize_is_clamped_rint_of_prequant():
    """quantize(c) == clamp(rint(prequant(c)), 0, 2^b - 1) (half to even) for
    every width, negative coefficients and values far outside the range."""
    rng = np.random.default_rng(8)
    d = 4000
    bits = rng.integers(0, 9, size=d)
    step = (0.05 + rng.random(d)).astype(np.float32)
    top = (1 << bits) - 1
    c = rng.standard_normal(d) * step * np.maximum(top, 1) * 0.8    # mostly inside the range
    c[::7] *= 5.0                                                     # some far outside, both signs
    c[::11] = (rng.integers(-3, 300, size=c[::11].size) + 0.5 - top[::11] / 2.0) * step[::11]  # exact ties
    pre = oracle.prequant(c, step, bits)
    u = oracle.quantize(c, step, bits)
    expect = np.clip(np.rint(pre.astype(np.float64)), 0, top).astype(np.int64)
    expect[bits == 0] = 0
    assert np.array_equal(u, expect)
    assert np.all(pre[bits == 0] == 0)
    assert np.sum((bits > 0) & (pre - np.floor(pre) == 0.5)) > 100     # ties were exercised
    # encode reports the same pre-rounding values for the coefficients T (x - mu)
    dd = 16
    T = rng.standard_normal((dd, dd))
    X = rng.standard_normal((50, dd))
    mu = rng.standard_normal(dd)
    b16 = np.array([8, 6, 5, 4, 3, 3, 2, 1, 0, 0, 0, 0, 0, 0, 0, 0])   # 32 bits: one record word
    st16 = (0.1 + rng.random(dd)).astype(np.float32)
    _, codes, pre_e = oracle.encode(X, T, mu, st16, b16, want_codes=True, want_pre=True)
    for i in range(50):
        cc = T @ (X[i] - mu)
        assert np.array_equal(pre_e[i], oracle.prequant(cc, st16, b16))
        assert np.array_equal(codes[i], oracle.quantize(cc, st16, b16))
