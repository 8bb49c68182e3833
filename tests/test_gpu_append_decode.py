"""aatc_append_decode_attention: a serving engine's decode step in one launch
("Attention-Aware Transform Coding Guide: KV Compression", "Deployment Guide:
Integrating AATC with vLLM": calibrate offline, then every decode step appends
the new tokens to the compressed cache and attends over it).

The fused call must write the same records as aatc_encode at positions
L_old.. and give the attention aatc_decode_attention gives over all
L_old + n_new tokens; both are checked, and the output is compared with the
oracle's attention over the records the call wrote."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import ATTN_RTOL, attn_rel_err, records, to_np64
from quantized_attention_kv_b300 import aatc, synth

pytestmark = pytest.mark.gpu

# GPU vs GPU from identical records: only the summation order differs (the new
# tokens' scores are fp32 dot products in the fused call, mma.sync sums in the
# split kernel, and the merge has one more partial)
SAME_CODES_RTOL = 2e-4

# (workload, batch rows, cached tokens, new tokens per row).  The fused
# kernel fits shapes whose plain decode has several splits per (row, KV head
# group) or no cached tokens; the others run append then decode.  Each case
# runs with the kernel used whenever it fits and with the default rule (used
# where it pays).
CASES = [
    ("tiny", 1, 0, 1),          # an empty cache: the new token alone (appenders only, two head groups)
    ("tiny", 1, 5, 1),          # one split per unit: the two calls
    ("tiny", 2, 31, 1),         # the new token ends a tile (the two calls)
    ("tiny", 2, 64, 4),         # new tokens open a tile
    ("tiny", 2, 95, 2),         # new tokens across a tile boundary
    ("tiny", 3, 1000, 4),       # the most new tokens the fused kernel takes
    ("tiny", 2, 300, 5),        # beyond it: the two separate calls
    ("tiny", 1, 40, 17),        # beyond the append encoder too: the prefill encoder
    ("llama_32k", 1, 4095, 1),
    ("llama_32k", 4, 1000, 2),  # appenders with two pairs each
    ("llama_32k", 20, 256, 1),  # more units than SMs: the two calls
    ("qwen_128k", 2, 2047, 3),  # GQA group 7: a head group with one dead head
]

_cals = {}


def _cal(name):
    if name not in _cals:
        wl = synth.WORKLOADS[name]
        k, v, q = synth.calib_inputs(wl, device="cuda")
        _cals[name] = (wl, aatc.calibrate(k, v, q, wl.bits))
    return _cals[name]


def _caches(cal, B, L_cap, kc, vc, L_old):
    kp, vp = aatc.alloc_cache(cal, B, L_cap, tensor="k"), aatc.alloc_cache(cal, B, L_cap, tensor="v")
    if L_old:
        aatc.encode(cal, kc[:, :, :L_old].contiguous(), vc[:, :, :L_old].contiguous(), kp, vp)
    return kp, vp


@pytest.fixture(params=[2, 1], ids=["fused_whenever_it_fits", "fused_when_it_pays"])
def fuse_mode(request):
    aatc.set_fused_step(request.param)
    yield request.param
    aatc.set_fused_step(1)


@pytest.mark.parametrize("name,B,L_old,n_new", CASES)
def test_fused_step_matches_append_then_decode_and_oracle(name, B, L_old, n_new, fuse_mode):
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    wl, cal = _cal(name)
    L = L_old + n_new
    L_cap = 32 * (L // 32 + 2)
    kc, vc = synth.cache_inputs(wl, layer=6, device="cuda", seq_len=L, batch=B)
    kn, vn = kc[:, :, L_old:].contiguous(), vc[:, :, L_old:].contiguous()
    qd = synth.query_inputs(wl, device="cuda", batch=B, step=L)
    kpa, vpa = _caches(cal, B, L_cap, kc, vc, L_old)
    kpb, vpb = _caches(cal, B, L_cap, kc, vc, L_old)
    ws = aatc.new_append_workspace(cal, B, L_old, n_new)
    out_f = aatc.append_decode_attention(cal, kn, vn, qd, kpa, vpa, L_old, workspace=ws)
    aatc.encode(cal, kn, vn, kpb, vpb, start_pos=L_old)
    out_s = aatc.decode_attention(cal, qd, kpb, vpb, L)
    torch.cuda.synchronize()
    cal.check()
    assert torch.equal(kpa, kpb) and torch.equal(vpa, vpb), "records differ from aatc_encode's"
    assert torch.isfinite(out_f).all()
    assert attn_rel_err(out_f.cpu().numpy(), out_s.cpu().numpy()) <= SAME_CODES_RTOL
    assert int(ws[:1024].count_nonzero()) == 0, "split counters not left at zero"
    gcal = cal.export()
    rk = records(kpa, gcal["W_k"], oracle.KEYS, L)
    rv = records(vpa, gcal["W_v"], oracle.VALUES, L)
    ref = oracle.decode_attention(to_np64(qd), rk, rv, gcal)
    assert attn_rel_err(out_f.cpu().numpy(), ref) <= ATTN_RTOL


def test_fused_step_mode_argument():
    with pytest.raises(aatc.AatcError) as e:
        aatc.set_fused_step(3)
    assert e.value.status == aatc.ERR_INVALID_ARG


def test_fused_steps_in_a_row_share_one_workspace():
    """Three decode steps, one token each, with one workspace (and a plain
    decode in between on the same workspace): each step matches the oracle."""
    wl, cal = _cal("llama_32k")
    B, L0 = 2, 2000
    L_cap = 2048
    kc, vc = synth.cache_inputs(wl, layer=7, device="cuda", seq_len=L0 + 3, batch=B)
    kp, vp = _caches(cal, B, L_cap, kc, vc, L0)
    ws = aatc.new_append_workspace(cal, B, L0 + 3, 1)
    gcal = cal.export()
    for step in range(3):
        Lo = L0 + step
        qd = synth.query_inputs(wl, device="cuda", batch=B, step=step)
        out = aatc.append_decode_attention(cal, kc[:, :, Lo:Lo + 1].contiguous(), vc[:, :, Lo:Lo + 1].contiguous(),
                                           qd, kp, vp, Lo, workspace=ws)
        plain = aatc.decode_attention(cal, qd, kp, vp, Lo + 1, workspace=ws)
        torch.cuda.synchronize()
        cal.check()
        rk = records(kp, gcal["W_k"], oracle.KEYS, Lo + 1)
        rv = records(vp, gcal["W_v"], oracle.VALUES, Lo + 1)
        ref = oracle.decode_attention(to_np64(qd), rk, rv, gcal)
        assert attn_rel_err(out.cpu().numpy(), ref) <= ATTN_RTOL, step
        assert attn_rel_err(out.cpu().numpy(), plain.cpu().numpy()) <= SAME_CODES_RTOL, step
        assert int(ws[:1024].count_nonzero()) == 0


def test_fused_step_arguments():
    wl, cal = _cal("tiny")
    B = 1
    kp, vp = aatc.alloc_cache(cal, B, 64), aatc.alloc_cache(cal, B, 64)
    kn = torch.zeros(B, wl.n_kv_heads, 1, 128, dtype=wl.dtype, device="cuda")
    qd = synth.query_inputs(wl, device="cuda", batch=B)
    with pytest.raises(aatc.AatcError) as e:   # L_old + n_new > L_cap
        aatc.append_decode_attention(cal, kn, kn, qd, kp, vp, 64)
    assert e.value.status == aatc.ERR_CAPACITY
    out = aatc.append_decode_attention(cal, kn[:, :, :0], kn[:, :, :0], qd, kp, vp, 10)   # n_new = 0: a plain decode
    ref = aatc.decode_attention(cal, qd, kp, vp, 10)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
