"""fp64 CPU oracle for Attention-Aware Transform Coding (AATC) of KV caches.

TEST INFRASTRUCTURE ONLY.  This package is the reference the CUDA path is
checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it;
the product package never does, and the two share no code.

The arithmetic lives in ``aatc_oracle.c`` (plain C, fp64, compiled with gcc
on first use or by ``build()``); this module only marshals numpy arrays.
Each wrapper names the page section it follows, as the C file does.

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
library routines, brute force or published values -- none is "parity
unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "aatc_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

MAXB = 8


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (IEEE fp64, no fast-math) into liboracle.so."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11",
                               "-D_DEFAULT_SOURCE", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        Lg = ctypes.c_long
        D = ctypes.c_double
        sig = {
            "orc_abi_version": (I, []),
            "orc_mean": (None, [P, Lg, I, P]),
            "orc_moment": (None, [P, Lg, I, P, P]),
            "orc_jacobi_eig": (I, [P, I, I, D, P, P]),
            "orc_key_transform": (I, [P, P, I, I, D, P, P, P, P, P]),
            "orc_waterfill_theta": (D, [P, I, D, P, P]),
            "orc_allocate_bits": (I, [P, I, I, P, P]),
            "orc_attention_weights": (None, [P, P, P, Lg, Lg, I, P, P]),
            "orc_joint_allocation": (I, [P, P, I, I, P, P, I, I, P, P, P, P]),
            "orc_gauss_uniform_mse": (D, [I, D]),
            "orc_gauss_uniform_step": (D, [I]),
            "orc_steps": (None, [P, P, I, P]),
            "orc_quantize": (None, [P, P, P, I, P]),
            "orc_prequant": (None, [P, P, P, I, P]),
            "orc_dequantize": (None, [P, P, P, I, P]),
            "orc_record_order": (I, [P, I, P]),
            "orc_layout": (None, [P, I, P]),
            "orc_cache_put": (None, [P, Lg, I, I, Lg, P]),
            "orc_cache_get": (None, [P, Lg, I, I, Lg, P]),
            "orc_pack": (None, [P, P, I, I, P]),
            "orc_unpack": (None, [P, P, I, P]),
            "orc_unpack_rows": (None, [P, Lg, I, P, I, P]),
            "orc_encode": (None, [P, Lg, I, P, P, P, P, I, P, P, P]),
            "orc_attention": (None, [P, P, P, Lg, I, P]),
            "orc_reconstruct": (None, [P, Lg, I, I, P, P, P, P, P]),
            "orc_decode_head": (None, [P, I, P, P, Lg, I, I, I, P, P, P, P, P, P, P, P, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


# ---------------------------------------------------------------- statistics
def mean(X) -> np.ndarray:
    """Channel mean of X [n][d] (KLT section: calibration statistics)."""
    X = _f64(X)
    n, d = X.shape
    mu = np.empty(d)
    lib().orc_mean(_p(X), n, d, _p(mu))
    return mu


def moment(X, center=None) -> np.ndarray:
    """(1/n) sum (x-c)(x-c)^T; center=None gives the uncentered second moment."""
    X = _f64(X)
    n, d = X.shape
    S = np.empty((d, d))
    c = None if center is None else _f64(center)
    lib().orc_moment(_p(X), n, d, None if c is None else _p(c), _p(S))
    return S


# ---------------------------------------------------------------- eigen
def jacobi_eig(A, max_sweeps: int = 50, tol: float = 1e-15):
    """Cyclic Jacobi; returns (evals desc, evecs [d][d] columns, sweeps or -1)."""
    A = _f64(A)
    d = A.shape[0]
    w = np.empty(d)
    V = np.empty((d, d))
    sw = lib().orc_jacobi_eig(_p(A), d, max_sweeps, tol, _p(w), _p(V))
    return w, V, sw


def key_transform(Sk, Sq, max_sweeps: int = 50, tol: float = 1e-15):
    """Whitened key KLT: returns dict(T, T_inv, A, lam, lam_q, ok)."""
    Sk, Sq = _f64(Sk), _f64(Sq)
    d = Sk.shape[0]
    T, Ti, A = np.empty((d, d)), np.empty((d, d)), np.empty((d, d))
    lam, lamq = np.empty(d), np.empty(d)
    rc = lib().orc_key_transform(_p(Sk), _p(Sq), d, max_sweeps, tol, _p(T), _p(Ti), _p(A),
                                 _p(lam), _p(lamq))
    return dict(T=T, T_inv=Ti, A=A, lam=lam, lam_q=lamq, ok=(rc == 0))


# ---------------------------------------------------------------- water-filling
def waterfill_theta(lam, total_bits: float):
    """Continuous reverse water-filling: (theta, R, D)."""
    lam = _f64(lam)
    d = lam.shape[0]
    R, D = np.empty(d), np.empty(d)
    th = lib().orc_waterfill_theta(_p(lam), d, float(total_bits), _p(R), _p(D))
    return th, R, D


def allocate_bits(lam, B_bits: int):
    """Exact integer allocation (top-B gains); returns (bits int32[d], cut margin)."""
    lam = _f64(lam)
    d = lam.shape[0]
    b = np.empty(d, dtype=np.int32)
    m = ctypes.c_double(0.0)
    rc = lib().orc_allocate_bits(_p(lam), d, int(B_bits), _p(b), ctypes.byref(m))
    if rc != 0:
        raise ValueError("unsupported budget")
    return b, m.value


def attention_weights(Q, K, V):
    """Token weights of the distortion theorem for one KV head: (alpha_K, alpha_V)
    averaged over the calibration queries Q [m][d] attending keys K [n][d] and
    values V [n][d]: alpha_V = sum_i A_i^2, alpha_K = (1/d) sum_i A_i^2 |v_i - o|^2."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    m, d = Q.shape
    n = K.shape[0]
    ak, av = ctypes.c_double(0.0), ctypes.c_double(0.0)
    lib().orc_attention_weights(_p(Q), _p(K), _p(V), m, n, d, ctypes.byref(ak), ctypes.byref(av))
    return ak.value, av.value


def joint_allocation_layer(lam_k, lam_v, alpha_k, alpha_v, B_total: int, granule: int = 32):
    """One water level over K and V for the H heads of a layer (lam_k, lam_v
    [H][d], alpha_k, alpha_v [H]) with one split B_k + B_v = B_total common to
    the heads (multiples of `granule`).  Returns (bits_k, bits_v [H][d], B_k, cost)."""
    lam_k, lam_v = np.atleast_2d(_f64(lam_k)), np.atleast_2d(_f64(lam_v))
    H, d = lam_k.shape
    ak, av = _f64(np.atleast_1d(alpha_k)), _f64(np.atleast_1d(alpha_v))
    bk, bv = np.empty((H, d), dtype=np.int32), np.empty((H, d), dtype=np.int32)
    Bk, cost = ctypes.c_int(0), ctypes.c_double(0.0)
    rc = lib().orc_joint_allocation(_p(lam_k), _p(lam_v), H, d, _p(ak), _p(av), int(B_total), int(granule),
                                    _p(bk), _p(bv), ctypes.byref(Bk), ctypes.byref(cost))
    if rc != 0:
        raise ValueError("unsupported budget")
    return bk, bv, Bk.value, cost.value


def joint_allocation(lam_k, lam_v, alpha_k: float, alpha_v: float, B_total: int, granule: int = 32):
    """joint_allocation_layer for one head: returns (bits_k, bits_v [d], B_k, cost)."""
    bk, bv, Bk, cost = joint_allocation_layer(lam_k, lam_v, [alpha_k], [alpha_v], B_total, granule)
    return bk[0], bv[0], Bk, cost


def joint_split(k_cal, v_cal, q_cal, cal, granule: int = 32):
    """Joint K/V allocation per KV head from a calibration `cal` (its lam_k of the
    whitened key covariance and lam_v): the token weights of the G query heads'
    calibration queries attending the head's calibration keys and values, then
    one water level over K and V with the pair budget 2 * 32 * W.  Returns a
    list of dicts (alpha_k, alpha_v, B_k, B_v, bits_k, bits_v, cost, cost_even)."""
    k_cal, v_cal, q_cal = _f64(k_cal), _f64(v_cal), _f64(q_cal)
    Hkv, Hq = k_cal.shape[0], q_cal.shape[0]
    G = Hq // Hkv
    B = 32 * int(cal["W"])
    out = []
    for h in range(Hkv):
        Qh = q_cal[h * G:(h + 1) * G].reshape(-1, q_cal.shape[-1])
        ak, av = attention_weights(Qh, k_cal[h], v_cal[h])
        lk, lv = cal["lam_k"][h], cal["lam_v"][h]
        bk, bv, Bk, cost = joint_allocation(lk, lv, ak, av, 2 * B, granule)
        even = ak * float(np.sum(lk * 4.0 ** -cal["bits_k"][h].astype(np.float64))) + \
            av * float(np.sum(lv * 4.0 ** -cal["bits_v"][h].astype(np.float64)))
        out.append(dict(alpha_k=ak, alpha_v=av, B_k=Bk, B_v=2 * B - Bk, bits_k=bk, bits_v=bv, cost=cost,
                        cost_even=even))
    return out


def gauss_uniform_mse(b: int, step: float) -> float:
    return lib().orc_gauss_uniform_mse(int(b), float(step))


def gauss_uniform_step(b: int) -> float:
    return lib().orc_gauss_uniform_step(int(b))


def steps(lam, bits) -> np.ndarray:
    lam, bits = _f64(lam), _i32(bits)
    out = np.empty(lam.shape[0], dtype=np.float32)
    lib().orc_steps(_p(lam), _p(bits), lam.shape[0], _p(out))
    return out


# ---------------------------------------------------------------- codec
def quantize(c, step, bits) -> np.ndarray:
    c, step, bits = _f64(c), _f32(step), _i32(bits)
    u = np.empty(c.shape[0], dtype=np.int32)
    lib().orc_quantize(_p(c), _p(step), _p(bits), c.shape[0], _p(u))
    return u


def prequant(c, step, bits) -> np.ndarray:
    """fp32 pre-rounding values v_j = c_j/Delta_j + (2^b_j - 1)/2 of quantize
    (0 for pruned channels): where the rounding decision is taken."""
    c, step, bits = _f64(c), _f32(step), _i32(bits)
    v = np.empty(c.shape[0], dtype=np.float32)
    lib().orc_prequant(_p(c), _p(step), _p(bits), c.shape[0], _p(v))
    return v


def dequantize(u, step, bits) -> np.ndarray:
    u, step, bits = _i32(u), _f32(step), _i32(bits)
    c = np.empty(u.shape[0])
    lib().orc_dequantize(_p(u), _p(step), _p(bits), u.shape[0], _p(c))
    return c


def record_order(bits) -> np.ndarray:
    """Order in which the codes of the non-pruned channels follow one another
    in a record (see orc_record_order)."""
    bits = _i32(bits)
    order = np.empty(max(1, bits.shape[0]), dtype=np.int32)
    n = lib().orc_record_order(_p(bits), bits.shape[0], _p(order))
    return order[:n].copy()


def layout(bits) -> np.ndarray:
    """Record bit offset of each channel's code: int32 [d], -1 = pruned."""
    bits = _i32(bits)
    off = np.empty(bits.shape[0], dtype=np.int32)
    lib().orc_layout(_p(bits), bits.shape[0], _p(off))
    return off


KEYS, VALUES = 0, 1
TILE = 32


def cache_put(rec, kind: int, cache=None, start: int = 0, L_cap=None) -> np.ndarray:
    """Place records rec [n][W] of tokens start.. into a tiled cache slab
    (uint32 [L_cap * W]); a new zeroed slab is made if cache is None."""
    rec = np.ascontiguousarray(np.asarray(rec, dtype=np.uint32))
    n, W = rec.shape
    if cache is None:
        L_cap = L_cap if L_cap is not None else -(-(start + n) // TILE) * TILE
        cache = np.zeros(L_cap * W, dtype=np.uint32)
    assert cache.dtype == np.uint32 and cache.flags["C_CONTIGUOUS"]
    assert cache.size % (TILE * W) == 0 and start + n <= cache.size // W
    lib().orc_cache_put(_p(rec), n, W, int(kind), int(start), _p(cache))
    return cache


def cache_get(cache, W: int, kind: int, n: int, start: int = 0) -> np.ndarray:
    """Records [n][W] of tokens start..start+n-1 from a tiled cache slab."""
    cache = np.ascontiguousarray(np.asarray(cache, dtype=np.uint32)).reshape(-1)
    assert start + n <= cache.size // W
    rec = np.empty((n, W), dtype=np.uint32)
    lib().orc_cache_get(_p(cache), int(n), int(W), int(kind), int(start), _p(rec))
    return rec


def to_cache(rec, kind: int, L_cap: int) -> np.ndarray:
    """Records [B][H][L][W] -> tiled caches uint32 [B][H][L_cap*W]."""
    rec = np.asarray(rec, dtype=np.uint32)
    Bsz, H, L, W = rec.shape
    out = np.zeros((Bsz, H, L_cap * W), dtype=np.uint32)
    for b in range(Bsz):
        for h in range(H):
            cache_put(rec[b, h], kind, out[b, h])
    return out


def from_cache(cache, W: int, kind: int, L: int) -> np.ndarray:
    """Tiled caches [B][H][L_cap*W] -> records [B][H][L][W]."""
    cache = np.asarray(cache).view(np.uint32) if np.asarray(cache).dtype != np.uint32 else np.asarray(cache)
    Bsz, H = cache.shape[:2]
    cache = cache.reshape(Bsz, H, -1)
    out = np.empty((Bsz, H, L, W), dtype=np.uint32)
    for b in range(Bsz):
        for h in range(H):
            out[b, h] = cache_get(np.ascontiguousarray(cache[b, h]), W, kind, L)
    return out


def pack(u, bits) -> np.ndarray:
    u, bits = _i32(u), _i32(bits)
    B = int(bits.sum())
    assert B % 32 == 0
    rec = np.empty(B // 32, dtype=np.uint32)
    lib().orc_pack(_p(u), _p(bits), bits.shape[0], B // 32, _p(rec))
    return rec


def unpack(rec, bits) -> np.ndarray:
    rec = np.ascontiguousarray(np.asarray(rec, dtype=np.uint32))
    bits = _i32(bits)
    u = np.empty(bits.shape[0], dtype=np.int32)
    lib().orc_unpack(_p(rec), _p(bits), bits.shape[0], _p(u))
    return u


def unpack_rows(rec, bits) -> np.ndarray:
    """unpack for records rec [..][W] -> codes int32 [..][d]."""
    rec = np.ascontiguousarray(np.asarray(rec, dtype=np.uint32))
    bits = _i32(bits)
    W = rec.shape[-1]
    n = rec.size // W
    u = np.empty(rec.shape[:-1] + (bits.shape[0],), dtype=np.int32)
    lib().orc_unpack_rows(_p(rec), n, W, _p(bits), bits.shape[0], _p(u))
    return u


def encode(X, T, mu, step, bits, want_codes=False, want_pre=False):
    """Encode rows X [n][d] -> records uint32 [n][W] (+ codes, pre-rounding values)."""
    X, T, mu, step, bits = _f64(X), _f64(T), _f64(mu), _f32(step), _i32(bits)
    n, d = X.shape
    W = int(bits.sum()) // 32
    rec = np.empty((n, W), dtype=np.uint32)
    codes = np.empty((n, d), dtype=np.int32) if want_codes else None
    pre = np.empty((n, d), dtype=np.float32) if want_pre else None
    lib().orc_encode(_p(X), n, d, _p(T), _p(mu), _p(step), _p(bits), W, _p(rec),
                     None if codes is None else _p(codes), None if pre is None else _p(pre))
    return rec, codes, pre


def reconstruct(rec, T_inv, mu, step, bits) -> np.ndarray:
    rec = np.ascontiguousarray(np.asarray(rec, dtype=np.uint32))
    T_inv, mu, step, bits = _f64(T_inv), _f64(mu), _f32(step), _i32(bits)
    n, W = rec.shape
    d = mu.shape[0]
    X = np.empty((n, d))
    lib().orc_reconstruct(_p(rec), n, d, W, _p(T_inv), _p(mu), _p(step), _p(bits), _p(X))
    return X


def attention(q, K, V) -> np.ndarray:
    """Exact softmax(q K^T / sqrt(d)) V for one query q [d]."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    L, d = K.shape
    o = np.empty(d)
    lib().orc_attention(_p(q), _p(K), _p(V), L, d, _p(o))
    return o


# ---------------------------------------------------------------- pipeline
def calibrate(k_cal, v_cal, q_cal, bits_per_element: float, max_sweeps: int = 50, joint: bool = False):
    """Per-KV-head calibration.

    k_cal, v_cal: [H_kv][N][d]; q_cal: [H_q][N][d] (query head h uses KV head
    h // G).  Returns a dict of per-head arrays (leading axis H_kv):
    mu_k, mu_v, T_k, T_k_inv, A_k, lam_k, T_v (= U_v^T), U_v, lam_v, lam_q,
    bits_k, bits_v, step_k, step_v, margin_k, margin_v, W_k, W_v, W, ok.
    Each tensor gets B = bits_per_element * d bits per token (W = B / 32 words)
    unless `joint`: then the pair budget 2B is split between K and V by the
    attention-aware token weights (joint_allocation_layer, one split for the
    layer), W_k + W_v = 2W, and W is None when the widths differ.
    """
    k_cal, v_cal, q_cal = (np.asarray(a) for a in (k_cal, v_cal, q_cal))
    Hkv, N, d = k_cal.shape
    Hq = q_cal.shape[0]
    if Hq % Hkv:
        raise ValueError("n_q_heads must be a multiple of n_kv_heads")
    G = Hq // Hkv
    B_bits = int(round(bits_per_element * d))
    if abs(B_bits - bits_per_element * d) > 1e-9 or B_bits % 32 or B_bits > MAXB * d or B_bits <= 0:
        raise ValueError("unsupported budget")
    out = {k: [] for k in ("mu_k", "mu_v", "T_k", "T_k_inv", "A_k", "lam_k", "T_v", "U_v",
                           "lam_v", "lam_q", "bits_k", "bits_v", "step_k", "step_v",
                           "margin_k", "margin_v")}
    ok = True
    for h in range(Hkv):
        K = _f64(k_cal[h])
        V = _f64(v_cal[h])
        Q = _f64(q_cal[h * G:(h + 1) * G].reshape(G * N, d))
        mu_k, mu_v = mean(K), mean(V)
        Sk, Sv = moment(K, mu_k), moment(V, mu_v)
        Sq = moment(Q)
        kt = key_transform(Sk, Sq, max_sweeps)
        lam_v, U_v, sw = jacobi_eig(Sv, max_sweeps)
        ok = ok and kt["ok"] and sw >= 0
        bk, mk = allocate_bits(kt["lam"], B_bits)
        bv, mv = allocate_bits(lam_v, B_bits)
        for key, val in (("mu_k", mu_k), ("mu_v", mu_v), ("T_k", kt["T"]), ("T_k_inv", kt["T_inv"]),
                         ("A_k", kt["A"]), ("lam_k", kt["lam"]), ("T_v", U_v.T.copy()), ("U_v", U_v),
                         ("lam_v", lam_v), ("lam_q", kt["lam_q"]), ("bits_k", bk), ("bits_v", bv),
                         ("step_k", steps(kt["lam"], bk)), ("step_v", steps(lam_v, bv)),
                         ("margin_k", mk), ("margin_v", mv)):
            out[key].append(val)
    res = {k: np.stack([np.asarray(x) for x in v]) for k, v in out.items()}
    res["W_k"] = res["W_v"] = res["W"] = B_bits // 32
    if joint:
        ak, av = [], []
        for h in range(Hkv):
            Q = _f64(q_cal[h * G:(h + 1) * G].reshape(G * N, d))
            a = attention_weights(Q, _f64(k_cal[h]), _f64(v_cal[h]))
            ak.append(a[0])
            av.append(a[1])
        bk, bv, Bk, _ = joint_allocation_layer(res["lam_k"], res["lam_v"], ak, av, 2 * B_bits)
        res["bits_k"], res["bits_v"] = bk, bv
        res["step_k"] = np.stack([steps(res["lam_k"][h], bk[h]) for h in range(Hkv)])
        res["step_v"] = np.stack([steps(res["lam_v"][h], bv[h]) for h in range(Hkv)])
        res["margin_k"] = np.array([allocate_bits(res["lam_k"][h], Bk)[1] for h in range(Hkv)])
        res["margin_v"] = np.array([allocate_bits(res["lam_v"][h], 2 * B_bits - Bk)[1] for h in range(Hkv)])
        res["alpha_k"], res["alpha_v"] = np.array(ak), np.array(av)
        res["W_k"], res["W_v"] = Bk // 32, (2 * B_bits - Bk) // 32
        res["W"] = res["W_k"] if res["W_k"] == res["W_v"] else None
    res["G"] = G
    res["ok"] = ok
    return res


def encode_cache(X, cal, tensor: str, want_codes=False, want_pre=False):
    """Encode a cache X [B][H_kv][L][d] with calibration `cal` ('k' or 'v')."""
    X = np.asarray(X)
    Bsz, Hkv, L, d = X.shape
    W = cal.get("W_" + tensor, cal["W"])
    T = cal["T_k"] if tensor == "k" else cal["T_v"]
    rec = np.empty((Bsz, Hkv, L, W), dtype=np.uint32)
    codes = np.empty((Bsz, Hkv, L, d), dtype=np.int32) if want_codes else None
    pre = np.empty((Bsz, Hkv, L, d), dtype=np.float32) if want_pre else None
    for b in range(Bsz):
        for h in range(Hkv):
            r, c, p = encode(X[b, h], T[h], cal["mu_" + tensor][h], cal["step_" + tensor][h],
                             cal["bits_" + tensor][h], want_codes, want_pre)
            rec[b, h] = r
            if want_codes:
                codes[b, h] = c
            if want_pre:
                pre[b, h] = p
    return rec, codes, pre


def decode_attention(q, kp, vp, cal, seq_lens=None):
    """Exact attention of q [B][H_q][d] over packed caches kp, vp [B][H_kv][L_cap][W].

    Tokens 0..seq_lens[b]-1 of batch row b are attended (all L_cap if None).
    Returns fp64 [B][H_q][d].
    """
    q = _f64(q)
    Bsz, Hq, d = q.shape
    Hkv = kp.shape[1]
    G = Hq // Hkv
    Wk, Wv = cal.get("W_k", cal["W"]), cal.get("W_v", cal["W"])
    out = np.zeros((Bsz, Hq, d))
    for b in range(Bsz):
        L = kp.shape[2] if seq_lens is None else int(seq_lens[b])
        for h in range(Hkv):
            kr = np.ascontiguousarray(kp[b, h, :L], dtype=np.uint32)
            vr = np.ascontiguousarray(vp[b, h, :L], dtype=np.uint32)
            o = np.empty((G, d))
            qq = _f64(q[b, h * G:(h + 1) * G])
            args = [_f64(cal["T_k_inv"][h]), _f64(cal["mu_k"][h]), _f32(cal["step_k"][h]),
                    _i32(cal["bits_k"][h]), _f64(cal["U_v"][h]), _f64(cal["mu_v"][h]),
                    _f32(cal["step_v"][h]), _i32(cal["bits_v"][h])]
            lib().orc_decode_head(_p(qq), G, _p(kr), _p(vr), L, d, Wk, Wv, *[_p(a) for a in args], _p(o))
            out[b, h * G:(h + 1) * G] = o
    return out
