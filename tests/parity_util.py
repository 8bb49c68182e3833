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
