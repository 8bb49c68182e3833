"""The bounded waits of the decode kernels report TIMEOUT instead of hanging.

Every wait of a decode kernel on its own bulk copies gives up after a fixed
number of tries and sets the handle's TIMEOUT status.  A testing hook of the
library (aatc_test_wait_fault) leaves one tile copy unissued, with a short
limit on the wait for it, so the wait runs out without any fault: the call
returns, aatc_check reports TIMEOUT, and the next normal call is correct."""
import time

import pytest
import torch

import oracle
from parity_util import ATTN_RTOL, attn_rel_err, to_np64
from quantized_attention_kv_b300 import aatc, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantized_attention_kv_b300 import build
    build.build()
    aatc.lib()
    yield
    aatc.test_wait_fault(False)
    torch.cuda.synchronize()


@pytest.mark.parametrize("B,L", [(1, 5000), (160, 700)])   # several splits + combine; one split per unit
def test_wait_that_runs_out_reports_timeout_and_the_context_stays_usable(B, L):
    wl = synth.WORKLOADS["tiny"]
    k, v, q = synth.calib_inputs(wl, device="cuda")
    ocal = oracle.calibrate(to_np64(k), to_np64(v), to_np64(q), wl.bits)
    g = aatc.import_calib(ocal, wl.n_q_heads, wl.dtype)
    kc, vc = synth.cache_inputs(wl, device="cuda", seq_len=L, batch=B)
    kp = aatc.alloc_cache(g, B, L)
    vp = aatc.alloc_cache(g, B, L)
    aatc.encode(g, kc, vc, kp, vp)
    qd = synth.query_inputs(wl, device="cuda", batch=B)
    torch.cuda.synchronize()
    g.check()
    try:
        aatc.test_wait_fault(True, 500)            # about 10 ms at most for the one wait
        t0 = time.perf_counter()
        aatc.decode_attention(g, qd, kp, vp, L)
        torch.cuda.synchronize()
        took = time.perf_counter() - t0
    finally:
        aatc.test_wait_fault(False)
    assert took < 1.0, took                        # gave up within the short limit, no hang
    with pytest.raises(aatc.AatcError) as e:
        g.check()
    assert e.value.status == aatc.ERR_TIMEOUT
    g.check()                                      # the status was cleared
    # the next call, with the hook off, is correct
    out = aatc.decode_attention(g, qd, kp, vp, L).cpu().numpy()
    g.check()
    rows = [0] if B == 1 else [0, B - 1]
    okp, _, _ = oracle.encode_cache(to_np64(kc[rows]), ocal, "k")
    ovp, _, _ = oracle.encode_cache(to_np64(vc[rows]), ocal, "v")
    ref = oracle.decode_attention(to_np64(qd[rows]), okp, ovp, ocal)
    assert attn_rel_err(out[rows], ref) <= ATTN_RTOL
