"""aatc_decode_attention_static: decode attention for callers that cannot
allocate device memory (an engine plugin whose memory planner owns all device
memory, or a latency-critical path where cudaMalloc is not allowed).  It must
give the same output as aatc_decode_attention with a caller workspace, call
after call, even though every call reuses the same built-in scratch array.

Kept in a file of its own, collected last, so a stop-at-first-failure run has
run everything else before it."""
import ctypes

import numpy as np
import pytest
import torch

from parity_util import ATTN_RTOL, attn_rel_err
from quantized_attention_kv_b300 import aatc, synth

pytestmark = pytest.mark.gpu


def _static_fn():
    from quantized_attention_kv_b300 import build
    build.build()
    f = aatc.lib().aatc_decode_attention_static
    P, I = ctypes.c_void_p, ctypes.c_int
    f.restype = I
    f.argtypes = [P, P, P, P, I, P, I, I, P, P]
    return f


def _call_static(f, cal, q, kp, vp, L, seq_lens, out):
    return f(cal.handle, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kp.data_ptr()),
             ctypes.c_void_p(vp.data_ptr()), kp.shape[2],
             None if seq_lens is None else ctypes.c_void_p(seq_lens.data_ptr()), L, q.shape[0],
             ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_static_scratch_decode_matches_workspace_decode_twice():
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    f = _static_fn()
    wl = synth.WORKLOADS["tiny"]
    k, v, q = synth.calib_inputs(wl, device="cuda")
    cal = aatc.calibrate(k, v, q, wl.bits)
    B, L = 3, 1024
    kc, vc = synth.cache_inputs(wl, device="cuda", seq_len=L, batch=B)
    kp = aatc.alloc_cache(cal, B, L)
    vp = aatc.alloc_cache(cal, B, L)
    aatc.encode(cal, kc, vc, kp, vp)
    # two calls in a row with different queries, lengths and split plans:
    # the second must not see anything the first left in the shared scratch
    cases = [(synth.query_inputs(wl, device="cuda", batch=B, step=0), L,
              torch.tensor([1024, 517, 3], dtype=torch.int32, device="cuda")),
             (synth.query_inputs(wl, device="cuda", batch=B, step=1), 300, None)]
    for qd, Lc, sl in cases:
        ref = aatc.decode_attention(cal, qd, kp, vp, Lc, seq_lens=sl)
        got = torch.full_like(ref, float("nan"))
        st = _call_static(f, cal, qd, kp, vp, Lc, sl, got)
        assert st == aatc.OK, aatc.last_error()
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
        assert attn_rel_err(got.cpu().numpy(), ref.cpu().numpy()) <= ATTN_RTOL


def test_static_scratch_general_path_matches_workspace_decode_twice():
    """Records of 20 words take the general decode path (query prep, split and
    combine kernels, with q' and the partials laid out differently in the
    scratch): two calls in a row of different lengths still match the
    workspace decode."""
    f = _static_fn()
    wl = synth.WORKLOADS["tiny"]
    k, v, q = synth.calib_inputs(wl, device="cuda")
    cal = aatc.calibrate(k, v, q, 5.0)
    assert cal.W == 20
    B, L = 3, 1024
    assert 0 < aatc.workspace_size(cal, B, L) <= (4 << 20)
    kc, vc = synth.cache_inputs(wl, device="cuda", seq_len=L, batch=B)
    kp = aatc.alloc_cache(cal, B, L)
    vp = aatc.alloc_cache(cal, B, L)
    aatc.encode(cal, kc, vc, kp, vp)
    for step, Lc in ((0, 1024), (1, 300)):
        qd = synth.query_inputs(wl, device="cuda", batch=B, step=step)
        ref = aatc.decode_attention(cal, qd, kp, vp, Lc)
        got = torch.full_like(ref, float("nan"))
        st = _call_static(f, cal, qd, kp, vp, Lc, None, got)
        assert st == aatc.OK, aatc.last_error()
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
        assert attn_rel_err(got.cpu().numpy(), ref.cpu().numpy()) <= ATTN_RTOL, Lc


def test_static_scratch_checks_arguments_before_its_size():
    """Bad arguments get the same status as aatc_decode_attention gives them,
    not a scratch-size error worked out from them."""
    f = _static_fn()
    wl = synth.WORKLOADS["tiny"]
    k, v, q = synth.calib_inputs(wl, device="cuda")
    cal = aatc.calibrate(k, v, q, wl.bits)
    qd = synth.query_inputs(wl, device="cuda")
    kp = aatc.alloc_cache(cal, 1, 64)
    out = torch.zeros(1, wl.n_q_heads, 128, device="cuda")
    st = _call_static(f, cal, qd, kp, kp, 65, None, out)        # L above L_cap
    assert st == aatc.ERR_CAPACITY and "L_cap" in aatc.last_error()
    P = ctypes.c_void_p
    st = f(cal.handle, P(qd.data_ptr()), P(kp.data_ptr()), P(kp.data_ptr()), 64, None, 64, 70000,
           P(out.data_ptr()), P(torch.cuda.current_stream().cuda_stream))
    assert st == aatc.ERR_INVALID_ARG and "too large" in aatc.last_error()
    st = f(cal.handle, P(qd.data_ptr()), None, None, 64, None, 64, 1, P(out.data_ptr()), None)
    assert st == aatc.ERR_INVALID_ARG and "packed caches" in aatc.last_error()
    assert torch.all(out == 0)                # nothing was launched


def test_static_scratch_rejects_shapes_beyond_its_size():
    f = _static_fn()
    wl = synth.WORKLOADS["tiny"]
    k, v, q = synth.calib_inputs(wl, device="cuda")
    cal = aatc.calibrate(k, v, q, 5.0)        # 20-word records: the general decode path
    B = 600                                   # needs more than the 4 MiB of built-in scratch
    assert aatc.workspace_size(cal, B, 128) > (4 << 20)
    qd = torch.zeros(B, wl.n_q_heads, 128, dtype=wl.dtype, device="cuda")
    kp = aatc.alloc_cache(cal, B, 128)
    out = torch.zeros(B, wl.n_q_heads, 128, device="cuda")
    st = _call_static(f, cal, qd, kp, kp, 128, None, out)
    assert st == aatc.ERR_CAPACITY
    assert "scratch" in aatc.last_error()
    assert torch.all(out == 0)                # nothing was launched
