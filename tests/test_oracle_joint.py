"""Pins of the oracle's attention-aware token weights and joint K/V allocation.

"Attention-Aware Transform Coding Guide: KV Compression", section "Theorem:
Additive Error Decomposition": the value error is weighted by sum_i A_i^2,
and the key error by (1/d) sum_i A_i^2 |v_i - o|^2.  Section "Optimal Bit
Allocation via Reverse Water-Filling": one water level over the weighted
channel variances.  The weights are checked against closed forms (uniform
attention, an exact two-key tie) and invariances of the softmax.  The joint
allocation is checked against brute force over every bit vector on tiny
cases, and against the global top-B rule over the union of K and V gains.
"""
import itertools

import numpy as np
import pytest

import oracle


def _cost(lam, bits, alpha):
    return alpha * float(np.sum(np.asarray(lam) * 4.0 ** (-np.asarray(bits, dtype=np.float64))))


# ----------------------------------------------------------------- token weights
def test_uniform_attention_closed_form():
    """q = 0: every key gets A_i = 1/n, so alpha_V = 1/n and
    alpha_K = (1/d) (1/n^2) sum_i |v_i - mean(v)|^2."""
    rng = np.random.default_rng(1)
    n, d = 37, 16
    K, V = rng.standard_normal((n, d)), rng.standard_normal((n, d)) * 3 + 1
    ak, av = oracle.attention_weights(np.zeros((5, d)), K, V)
    vbar = V.mean(axis=0)
    assert av == pytest.approx(1.0 / n, rel=1e-13)
    assert ak == pytest.approx(np.sum((V - vbar) ** 2) / (d * n * n), rel=1e-12)


def test_two_key_tie_closed_form():
    """Two keys share the top score and the rest are far below: A = (1/2, 1/2, 0...),
    o = (v0 + v1) / 2, alpha_V = 1/2, alpha_K = |v0 - v1|^2 / (8 d)."""
    d, n = 8, 6
    K = np.zeros((n, d))
    K[0, 0] = K[1, 0] = 1.0
    K[2:, 0] = -1.0
    q = np.zeros((1, d))
    q[0, 0] = 2000.0                      # score gap 2000 * 2 / sqrt(8): exp(-1414) = 0
    rng = np.random.default_rng(2)
    V = rng.standard_normal((n, d))
    ak, av = oracle.attention_weights(q, K, V)
    assert av == pytest.approx(0.5, rel=1e-14)
    assert ak == pytest.approx(np.sum((V[0] - V[1]) ** 2) / (8 * d), rel=1e-12)


def test_token_weight_invariances():
    rng = np.random.default_rng(3)
    m, n, d = 6, 50, 12
    Q, K, V = rng.standard_normal((m, d)), rng.standard_normal((n, d)), rng.standard_normal((n, d))
    ak, av = oracle.attention_weights(Q, K, V)
    assert 1.0 / n <= av <= 1.0 and ak > 0
    # the same vector added to every key shifts each query's scores by a constant
    ak2, av2 = oracle.attention_weights(Q, K + rng.standard_normal(d), V)
    assert ak2 == pytest.approx(ak, rel=1e-9) and av2 == pytest.approx(av, rel=1e-9)
    # token order does not matter
    p = rng.permutation(n)
    ak3, av3 = oracle.attention_weights(Q, K[p], V[p])
    assert ak3 == pytest.approx(ak, rel=1e-12) and av3 == pytest.approx(av, rel=1e-12)
    # a shift of every value leaves v_i - o alone; a scale s multiplies alpha_K by s^2
    ak4, av4 = oracle.attention_weights(Q, K, V + 5.0)
    assert ak4 == pytest.approx(ak, rel=1e-9) and av4 == pytest.approx(av, rel=1e-12)
    ak5, av5 = oracle.attention_weights(Q, K, 3.0 * V)
    assert ak5 == pytest.approx(9.0 * ak, rel=1e-12) and av5 == pytest.approx(av, rel=1e-12)


# ----------------------------------------------------------------- joint allocation
@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("granule", [1, 2, 3])
def test_joint_allocation_is_the_brute_force_optimum(seed, granule):
    """d = 2 channels per tensor: every (bK, bV) in [0, 8]^4 with the right total
    and a granule-aligned K budget; the oracle's cost is the least one."""
    rng = np.random.default_rng(seed)
    lk, lv = rng.uniform(0.1, 10.0, 2), rng.uniform(0.1, 10.0, 2)
    ak, av = rng.uniform(0.2, 3.0), rng.uniform(0.2, 3.0)
    for B in range(0, 33, granule):
        best = np.inf
        for bk in itertools.product(range(9), repeat=2):
            if sum(bk) % granule:
                continue
            for bv in itertools.product(range(9), repeat=2):
                if sum(bk) + sum(bv) != B:
                    continue
                best = min(best, _cost(lk, bk, ak) + _cost(lv, bv, av))
        gk, gv, Bk, cost = oracle.joint_allocation(lk, lv, ak, av, B, granule)
        assert gk.sum() == Bk and gk.sum() + gv.sum() == B and Bk % granule == 0
        assert cost == pytest.approx(best, rel=1e-12), (B, granule)
        assert cost == pytest.approx(_cost(lk, gk, ak) + _cost(lv, gv, av), rel=1e-12)


def test_unit_granule_matches_the_union_top_b():
    """Granule 1: the joint optimum is the top-B rule over the union of the
    gains alpha_K lam_K 4^-t and alpha_V lam_V 4^-t."""
    rng = np.random.default_rng(7)
    d = 128
    lk, lv = np.sort(rng.gamma(0.7, 2.0, d))[::-1], np.sort(rng.gamma(0.7, 1.0, d))[::-1]
    ak, av = 0.8, 1.7
    for B in (0, 100, 511, 704, 1500, 2048):
        union, _ = oracle.allocate_bits(np.concatenate([ak * lk, av * lv]), B)
        ucost = _cost(ak * lk, union[:d], 1.0) + _cost(av * lv, union[d:], 1.0)
        _, _, _, cost = oracle.joint_allocation(lk, lv, ak, av, B, 1)
        assert cost == pytest.approx(ucost, rel=1e-12), B


def test_joint_allocation_symmetry_monotonicity_and_gain():
    d = 128
    lam = 0.95 ** np.arange(d)
    bk, bv, Bk, cost = oracle.joint_allocation(lam, lam, 1.0, 1.0, 704)
    assert Bk == 352 and np.array_equal(bk, bv)           # identical tensors split evenly
    lv = 0.93 ** np.arange(d)
    last = -1
    for ak in (0.01, 0.1, 0.3, 1.0, 3.0, 10.0, 100.0):
        bk, bv, Bk, cost = oracle.joint_allocation(lam, lv, ak, 1.0, 704)
        assert Bk >= last and Bk % 32 == 0                 # heavier keys never get fewer bits
        last = Bk
        ek, _ = oracle.allocate_bits(lam, 352)
        ev, _ = oracle.allocate_bits(lv, 352)
        assert cost <= _cost(lam, ek, ak) + _cost(lv, ev, 1.0) * (1 + 1e-15)   # never worse than 352 + 352
    with pytest.raises(ValueError):
        oracle.joint_allocation(lam, lv, 1.0, 1.0, 704 + 16)        # not a multiple of the granule


def test_joint_split_on_the_tiny_workload():
    """The calibration path end to end: token weights from the calibration
    queries, then the word-aligned split of the 2 x 352-bit pair budget.  The
    even split is one of the candidates, so the joint cost is never above it,
    and each side's bits are that side's exact top-B allocation."""
    from quantized_attention_kv_b300 import synth
    wl = synth.WORKLOADS["tiny"]
    k, v, q = synth.calib_inputs(wl, n_calib=256)
    cal = oracle.calibrate(k.double().numpy(), v.double().numpy(), q.double().numpy(), wl.bits)
    res = oracle.joint_split(k.numpy(), v.numpy(), q.numpy(), cal)
    assert len(res) == wl.n_kv_heads
    for h, r in enumerate(res):
        assert r["B_k"] + r["B_v"] == 2 * 32 * cal["W"] and r["B_k"] % 32 == 0
        assert r["alpha_k"] > 0 and 0 < r["alpha_v"] <= 1
        assert r["cost"] <= r["cost_even"] * (1 + 1e-12)
        bk, _ = oracle.allocate_bits(cal["lam_k"][h], r["B_k"])
        assert np.array_equal(bk, r["bits_k"])


@pytest.mark.parametrize("granule", [1, 2])
def test_layer_split_is_the_brute_force_optimum(granule):
    """Two heads share one split (one record width per tensor for the layer):
    brute force over the common B_K and every per-head bit vector."""
    rng = np.random.default_rng(11 + granule)
    lk, lv = rng.uniform(0.1, 10.0, (2, 2)), rng.uniform(0.1, 10.0, (2, 2))
    ak, av = rng.uniform(0.2, 3.0, 2), rng.uniform(0.2, 3.0, 2)
    vecs = list(itertools.product(range(9), repeat=2))
    for B in range(0, 33, granule):
        best = np.inf
        for Bk in range(0, B + 1, granule):
            tot = 0.0
            for h in range(2):
                ck = min((_cost(lk[h], b, ak[h]) for b in vecs if sum(b) == Bk), default=np.inf)
                cv = min((_cost(lv[h], b, av[h]) for b in vecs if sum(b) == B - Bk), default=np.inf)
                tot += ck + cv
            best = min(best, tot)
        bk, bv, Bk, cost = oracle.joint_allocation_layer(lk, lv, ak, av, B, granule)
        assert np.all(bk.sum(axis=1) == Bk) and np.all(bk.sum(axis=1) + bv.sum(axis=1) == B)
        assert cost == pytest.approx(best, rel=1e-12), B


def _tiny_cals():
    from quantized_attention_kv_b300 import synth
    wl = synth.WORKLOADS["tiny"]
    k, v, q = synth.calib_inputs(wl)
    args = (k.double().numpy(), v.double().numpy(), q.double().numpy(), wl.bits)
    return wl, oracle.calibrate(*args), oracle.calibrate(*args, joint=True)


def test_joint_calibration_fields():
    wl, ce, cj = _tiny_cals()
    W = ce["W"]
    assert cj["W_k"] + cj["W_v"] == 2 * W and cj["W_k"] != cj["W_v"] and cj["W"] is None
    for h in range(wl.n_kv_heads):
        assert cj["bits_k"][h].sum() == 32 * cj["W_k"] and cj["bits_v"][h].sum() == 32 * cj["W_v"]
        assert np.array_equal(cj["bits_k"][h], oracle.allocate_bits(cj["lam_k"][h], 32 * cj["W_k"])[0])
        assert np.array_equal(cj["step_v"][h], oracle.steps(cj["lam_v"][h], cj["bits_v"][h]))
    for key in ("T_k", "T_v", "lam_k", "lam_v", "mu_k", "mu_v"):      # the transforms do not change
        assert np.array_equal(cj[key], ce[key])


def test_decode_with_unequal_record_widths():
    """Records of W_K and W_V words: attention over the packed caches equals
    attention over the keys and values reconstructed from the same records."""
    from quantized_attention_kv_b300 import synth
    wl, _, cj = _tiny_cals()
    kc, vc = synth.cache_inputs(wl, seq_len=200, batch=1)
    q = synth.query_inputs(wl, batch=1, step=5)
    K, V, Q = kc.double().numpy(), vc.double().numpy(), q.double().numpy()
    kr, _, _ = oracle.encode_cache(K, cj, "k")
    vr, _, _ = oracle.encode_cache(V, cj, "v")
    assert kr.shape[-1] == cj["W_k"] and vr.shape[-1] == cj["W_v"]
    got = oracle.decode_attention(Q, kr, vr, cj)
    Kh = oracle.reconstruct(kr[0, 0], cj["T_k_inv"][0], cj["mu_k"][0], cj["step_k"][0], cj["bits_k"][0])
    Vh = oracle.reconstruct(vr[0, 0], cj["U_v"][0], cj["mu_v"][0], cj["step_v"][0], cj["bits_v"][0])
    for g in range(Q.shape[1]):
        np.testing.assert_allclose(got[0, g], oracle.attention(Q[0, g], Kh, Vh), rtol=1e-12, atol=1e-12)


def test_joint_allocation_lowers_the_attention_error():
    """The theorem's weighting in use: on the tiny workload, the attention error
    of the joint split (relative to the output's variation around the value
    mean) is below that of the even split."""
    from quantized_attention_kv_b300 import synth
    wl, ce, cj = _tiny_cals()
    kc, vc = synth.cache_inputs(wl, seq_len=512, batch=2)
    q = synth.query_inputs(wl, batch=2, step=3)
    K, V, Q = kc.double().numpy(), vc.double().numpy(), q.double().numpy()
    errs = []
    for cal in (ce, cj):
        kr, _, _ = oracle.encode_cache(K, cal, "k")
        vr, _, _ = oracle.encode_cache(V, cal, "v")
        o_hat = oracle.decode_attention(Q, kr, vr, cal)
        num = den = 0.0
        for b in range(2):
            for g in range(Q.shape[1]):
                o = oracle.attention(Q[b, g], K[b, 0], V[b, 0])
                num += np.sum((o - o_hat[b, g]) ** 2)
                den += np.sum((o - V[b, 0].mean(axis=0)) ** 2)
        errs.append(num / den)
    assert errs[1] < 0.8 * errs[0], errs
