"""GPU parity of the joint K/V budget split (attention-aware token weights).

"Theorem: Additive Error Decomposition" weights value noise by A_i^2 and key
noise by A_i^2 |v_i - o|^2 (and the query metric); "Optimal Bit Allocation via
Reverse Water-Filling" then puts one water level over the channels of both
tensors.  With one record width per tensor for a layer, the pair budget 2B is
split word-aligned between keys and values (W_K + W_V = 2W).

* An oracle joint calibration (W_K != W_V) imported into the library: codes of
  every encoder (fp32, append, tensor-core prefill) follow the tie rule, the
  caches are laid out with each tensor's own width, and decode (fast path,
  contiguous and paged) matches the oracle from identical codes.
* GPU calibration with joint_kv against the oracle's joint calibration: the
  same split and bit allocations (unless the oracle's best split is a cost tie
  within 1e-9 of another), then encode and decode parity end to end.
Tolerances are those of tests/parity_util.py.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import ATTN_RTOL, as_u32, attn_rel_err, compare_codes, records, to_np64, upload
from quantized_attention_kv_b300 import aatc, synth

pytestmark = pytest.mark.gpu
WL = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantized_attention_kv_b300 import build
    build.build()
    aatc.lib()
    yield
    torch.cuda.synchronize()


# (workload, KV heads kept, calibration tokens): fewer heads and tokens than the
# full workloads keep the fp64 oracle's calibration attention to seconds
CASES = {
    "tiny": ("tiny", 1, 512),
    "llama": ("llama_32k", 2, 1024),
    "qwen": ("qwen_128k", 2, 1024),
}
_cache = {}


def _case(name):
    if name not in _cache:
        wname, H, N = CASES[name]
        wl = synth.dataclasses.replace(WL[wname], n_kv_heads=H, n_q_heads=H * WL[wname].group)
        k, v, q = synth.calib_inputs(wl, device="cuda", n_calib=N)
        ocal = oracle.calibrate(to_np64(k), to_np64(v), to_np64(q), wl.bits, joint=True)
        _cache[name] = (wl, k, v, q, ocal)
    return _cache[name]


def _split_cost(ocal, Bk):
    """The oracle's layer cost of a given split (its token weights and eigenvalues)."""
    H = ocal["lam_k"].shape[0]
    Bpair = 32 * (ocal["W_k"] + ocal["W_v"])
    tot = 0.0
    for h in range(H):
        bk, _ = oracle.allocate_bits(ocal["lam_k"][h], Bk)
        bv, _ = oracle.allocate_bits(ocal["lam_v"][h], Bpair - Bk)
        tot += ocal["alpha_k"][h] * np.sum(ocal["lam_k"][h] * 4.0 ** -bk) + \
            ocal["alpha_v"][h] * np.sum(ocal["lam_v"][h] * 4.0 ** -bv)
    return tot


@pytest.mark.parametrize("name", ["tiny", "llama", "qwen"])
def test_imported_joint_calibration_encode_and_decode(name):
    wl, k, v, q, ocal = _case(name)
    Wk, Wv = ocal["W_k"], ocal["W_v"]
    assert Wk != Wv and Wk + Wv == 2 * int(wl.bits * 4)
    H = wl.n_kv_heads
    g = aatc.import_calib(ocal, wl.n_q_heads, wl.dtype)
    assert (g.W_k, g.W_v) == (Wk, Wv)
    with pytest.raises(ValueError):
        g.W                                          # no common width
    B, L = 2, 700
    kc, vc = synth.cache_inputs(wl, device="cuda", seq_len=L, batch=B)
    kn, vn = synth.cache_inputs(wl, layer=1, device="cuda", seq_len=3, batch=B)
    kp = aatc.alloc_cache(g, B, L + 3, tensor="k")
    vp = aatc.alloc_cache(g, B, L + 3, tensor="v")
    assert kp.shape[-1] == Wk and vp.shape[-1] == Wv
    aatc.encode(g, kc, vc, kp, vp)                   # prefill (tensor-core path for bf16)
    aatc.encode(g, kn, vn, kp, vp, start_pos=L)      # append path
    torch.cuda.synchronize()
    g.check()
    kall, vall = torch.cat([kc, kn], dim=2), torch.cat([vc, vn], dim=2)
    for t, kind, x, p in (("k", oracle.KEYS, kall, kp), ("v", oracle.VALUES, vall, vp)):
        _, codes, pre = oracle.encode_cache(to_np64(x), ocal, t, want_codes=True, want_pre=True)
        got = records(p, ocal["W_" + t], kind, L + 3)
        for h in range(H):
            compare_codes(got[:, h], codes[:, h], pre[:, h], ocal["bits_" + t][h])
    # decode from identical codes: the GPU's records, the oracle's calibration
    qd = synth.query_inputs(wl, device="cuda", batch=B, step=2)
    lens = torch.tensor([L + 3, 401], dtype=torch.int32, device="cuda")
    out = aatc.decode_attention(g, qd, kp, vp, L + 3, seq_lens=lens).cpu().numpy()
    g.check()
    rk, rv = records(kp, Wk, oracle.KEYS, L + 3), records(vp, Wv, oracle.VALUES, L + 3)
    ref = oracle.decode_attention(to_np64(qd), rk, rv, ocal, seq_lens=[L + 3, 401])
    assert attn_rel_err(out, ref) <= ATTN_RTOL, attn_rel_err(out, ref)
    # the same caches on shuffled 32-token blocks of paged pools: exactly the same output
    L_cap = kp.shape[2]
    bpr = L_cap // 32
    perm = torch.randperm(B * bpr + 3, generator=torch.Generator().manual_seed(7))
    table = perm[:B * bpr].reshape(B, bpr).to(torch.int32).cuda()
    pools = []
    for c, t in ((kp, "k"), (vp, "v")):
        W = c.shape[-1]
        pool = aatc.alloc_pool(g, B * bpr + 3, 32, tensor=t)
        pool[table.long()] = c.reshape(B, H, bpr, 32, W).permute(0, 2, 1, 3, 4)
        pools.append(pool)
    out_p = aatc.decode_attention_paged(g, qd, pools[0], pools[1], table, L + 3, seq_lens=lens)
    assert torch.equal(out_p, torch.from_numpy(out).cuda())


@pytest.mark.parametrize("name", ["tiny", "llama", "qwen"])
def test_gpu_joint_calibration_matches_oracle(name):
    wl, k, v, q, ocal = _case(name)
    g = aatc.calibrate(k, v, q, wl.bits, joint=True)
    gcal = g.export()
    Bk_o, Bk_g = 32 * ocal["W_k"], gcal["B_k"]
    assert gcal["B_k"] + gcal["B_v"] == 32 * (ocal["W_k"] + ocal["W_v"])
    assert 32 <= Bk_o <= 32 * (ocal["W_k"] + ocal["W_v"]) - 32   # inside the library's candidates
    if Bk_g != Bk_o:
        # only a cost tie may pick another split
        co, cg = _split_cost(ocal, Bk_o), _split_cost(ocal, Bk_g)
        assert abs(cg - co) <= 1e-9 * co, (Bk_g, Bk_o, cg, co)
        g.free()
        return
    H = wl.n_kv_heads
    for t in ("k", "v"):
        for h in range(H):
            gb, ob = gcal["bits_" + t][h], ocal["bits_" + t][h]
            if not np.array_equal(gb, ob):
                assert ocal["margin_" + t][h] < 1e-9, (t, h)
    # end to end on a cache: codes by the tie rule, decode from identical codes
    B, L = 1, 640
    kc, vc = synth.cache_inputs(wl, device="cuda", seq_len=L, batch=B)
    kp = aatc.alloc_cache(g, B, L, tensor="k")
    vp = aatc.alloc_cache(g, B, L, tensor="v")
    aatc.encode(g, kc, vc, kp, vp)
    qd = synth.query_inputs(wl, device="cuda", batch=B, step=4)
    out = aatc.decode_attention(g, qd, kp, vp, L).cpu().numpy()
    g.check()
    for t, kind, x, p in (("k", oracle.KEYS, kc, kp), ("v", oracle.VALUES, vc, vp)):
        _, codes, pre = oracle.encode_cache(to_np64(x), ocal, t, want_codes=True, want_pre=True)
        got = records(p, ocal["W_" + t], kind, L)
        for h in range(H):
            if np.array_equal(gcal["bits_" + t][h], ocal["bits_" + t][h]):
                compare_codes(got[:, h], codes[:, h], pre[:, h], ocal["bits_" + t][h])
    rk, rv = records(kp, gcal["W_k"], oracle.KEYS, L), records(vp, gcal["W_v"], oracle.VALUES, L)
    ref = oracle.decode_attention(to_np64(qd), rk, rv, gcal)
    assert attn_rel_err(out, ref) <= ATTN_RTOL
    g.free()
