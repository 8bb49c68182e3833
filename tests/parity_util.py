"""Helpers shared by the GPU parity tests: comparisons and tolerances.

Tolerances (all written here, used by every GPU test):
  * bit allocations, record layout, pack/unpack: bit-exact;
  * quantization codes: at most 1e-4 of the entries may differ, each by +-1,
    and only where the oracle's fp32 pre-rounding value lies within 1e-3 of a
    half-integer (a rounding tie);
  * attention outputs: max over (batch row, query head) of
    |o_gpu - o_ref|_inf / |o_ref|_inf <= 1e-3 (norm-wise relative error).
"""
import numpy as np
import torch

import oracle

CODE_MISMATCH_FRAC = 1e-4
TIE_WINDOW = 1e-3
ATTN_RTOL = 1e-3


def as_u32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().view(np.uint32)


def compare_codes(gpu_rec: np.ndarray, ref_codes: np.ndarray, ref_pre: np.ndarray, bits: np.ndarray):
    """Check GPU records against oracle codes (same bits).  Returns the mismatch fraction."""
    got = oracle.unpack_rows(gpu_rec, bits)
    diff = got.astype(np.int64) - ref_codes
    bad = diff != 0
    nbad = int(bad.sum())
    active = np.broadcast_to(bits > 0, ref_codes.shape)
    frac = nbad / max(1, int(active.sum()))
    assert frac <= CODE_MISMATCH_FRAC, "code mismatch fraction %.3g" % frac
    if nbad:
        assert np.abs(diff[bad]).max() == 1, "a code differs by more than one level"
        pre = ref_pre[bad].astype(np.float64)
        dist = np.abs(pre - np.floor(pre) - 0.5)
        assert dist.max() < TIE_WINDOW, "mismatch away from a rounding tie (%.3g)" % dist.max()
    return frac


def attn_rel_err(out_gpu: np.ndarray, out_ref: np.ndarray) -> float:
    """max over leading indices of |a - b|_inf / |b|_inf."""
    a = out_gpu.reshape(-1, out_gpu.shape[-1]).astype(np.float64)
    b = out_ref.reshape(-1, out_ref.shape[-1]).astype(np.float64)
    num = np.abs(a - b).max(axis=1)
    den = np.abs(b).max(axis=1)
    rel = np.where(den > 0, num / np.where(den > 0, den, 1), num)
    return float(rel.max())


def to_np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def records(cache_t, W, kind, L, start=0):
    """Records [B][H][L][W] of tokens start.. read from a GPU cache through the oracle's tiling."""
    c = as_u32(cache_t)
    Bsz, H = c.shape[:2]
    c = c.reshape(Bsz, H, -1)
    out = np.empty((Bsz, H, L, W), dtype=np.uint32)
    for b in range(Bsz):
        for h in range(H):
            out[b, h] = oracle.cache_get(np.ascontiguousarray(c[b, h]), W, kind, L, start)
    return out


def upload(rec, kind, L_cap):
    """Oracle records [B][H][L][W] placed in a tiled GPU cache of L_cap tokens."""
    Bsz, H, _, W = rec.shape
    c = oracle.to_cache(rec, kind, L_cap).view(np.int32).reshape(Bsz, H, L_cap, W)
    return torch.from_numpy(c).cuda()


def synthetic_calibration(G, bits_k, bits_v, seed=0, H=1):
    """A calibration with chosen bit allocations (orthogonal transforms from
    QR, steps from the oracle), to reach every decode path; H KV heads that
    share it."""
    rng = np.random.default_rng(seed)
    d = 128
    cal = {}
    Qk, _ = np.linalg.qr(rng.standard_normal((d, d)))
    Qv, _ = np.linalg.qr(rng.standard_normal((d, d)))
    lam_k = 0.95 ** np.arange(d)
    lam_v = 0.93 ** np.arange(d)
    rep = lambda a: np.repeat(np.asarray(a)[None], H, axis=0)  # noqa: E731
    cal["mu_k"] = rep(rng.standard_normal(d))
    cal["mu_v"] = rep(rng.standard_normal(d))
    cal["T_k"] = rep(Qk.T)
    cal["T_k_inv"] = rep(Qk)
    cal["A_k"] = rep(Qk.T)
    cal["T_v"] = rep(Qv.T)
    cal["U_v"] = rep(Qv)
    cal["lam_k"], cal["lam_v"], cal["lam_q"] = rep(lam_k), rep(lam_v), rep(np.ones(d))
    cal["bits_k"] = rep(np.asarray(bits_k, dtype=np.int32))
    cal["bits_v"] = rep(np.asarray(bits_v, dtype=np.int32))
    cal["step_k"] = rep(oracle.steps(lam_k, bits_k))
    cal["step_v"] = rep(oracle.steps(lam_v, bits_v))
    cal["W"] = int(np.sum(bits_k)) // 32
    cal["W_k"], cal["W_v"] = cal["W"], int(np.sum(bits_v)) // 32
    cal["G"] = G
    return cal
