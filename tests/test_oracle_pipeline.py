"""Pins for the oracle's per-head calibration on the smallest workload."""
import numpy as np

import oracle
from quantized_attention_kv_b300 import synth


def test_calibration_on_tiny_workload():
    wl = synth.WORKLOADS["tiny"]
    k, v, q = (t.double().numpy() for t in synth.calib_inputs(wl))
    cal = oracle.calibrate(k, v, q, wl.bits)
    assert cal["ok"] and cal["W"] == 11 and cal["G"] == 16
    d = wl.head_dim
    # query metric pooled over the 16 query heads of the group (plain numpy)
    Q = q.reshape(-1, d)
    Sq = Q.T @ Q / Q.shape[0]
    Ti = cal["T_k_inv"][0]
    assert np.abs(Ti.T @ Sq @ Ti - np.eye(d)).max() < 1e-8
    Sk = np.cov(k[0].T, bias=True)
    C = cal["T_k"][0] @ Sk @ cal["T_k"][0].T
    assert np.abs(C - np.diag(np.diag(C))).max() < 1e-6 * np.trace(C)
    Sv = np.cov(v[0].T, bias=True)
    Cv = cal["T_v"][0] @ Sv @ cal["T_v"][0].T
    assert np.abs(Cv - np.diag(np.diag(Cv))).max() < 1e-6 * np.trace(Cv)
    for t in ("k", "v"):
        b = cal["bits_" + t][0]
        assert b.sum() == 352 and np.all(np.diff(b) <= 0)
        s = cal["step_" + t][0]
        assert np.all((s > 0) == (b > 0))
    # the encode -> decode round trip on the tiny cache is close to exact attention
    kc, vc = (t.double().numpy() for t in synth.cache_inputs(wl))
    qq = synth.query_inputs(wl).double().numpy()
    kp, _, _ = oracle.encode_cache(kc, cal, "k")
    vp, _, _ = oracle.encode_cache(vc, cal, "v")
    out = oracle.decode_attention(qq, kp, vp, cal)
    for g in range(wl.n_q_heads):
        ex = oracle.attention(qq[0, g], kc[0, 0], vc[0, 0])
        rel = np.abs(out[0, g] - ex).max() / np.abs(ex).max()
        assert rel < 0.35, (g, rel)
