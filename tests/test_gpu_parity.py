"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle.

Per-kernel checks import the oracle's calibration into a GPU handle and feed
identical inputs (and, for decode, identical oracle-packed records), so each
kernel is isolated.  End-to-end checks run GPU calibration + encode + decode
on the full workload sizes and compare with the oracle's own pipeline on
sampled heads.  Tolerances are those of tests/parity_util.py.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import (ATTN_RTOL, as_u32, attn_rel_err, compare_codes, records, synthetic_calibration,
                         to_np64, upload)
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


def _oracle_cal(k, v, q, bits):
    return oracle.calibrate(to_np64(k), to_np64(v), to_np64(q), bits)


# ----------------------------------------------------------------- calibration
_tiny_cache = {}


def _tiny():
    if not _tiny_cache:
        wl = WL["tiny"]
        k, v, q = synth.calib_inputs(wl, device="cuda")
        _tiny_cache.update(wl=wl, k=k, v=v, q=q, ocal=_oracle_cal(k, v, q, wl.bits))
    return _tiny_cache


def _check_calibration(gcal: dict, ocal: dict, H: int):
    ties = 0
    for t in ("k", "v"):
        for h in range(H):
            gb, ob = gcal["bits_" + t][h], ocal["bits_" + t][h]
            if not np.array_equal(gb, ob):
                assert ocal["margin_" + t][h] < 1e-9, ("allocation differs away from a tie", t, h)
                ties += 1
                continue
            assert gb.sum() == ocal["W"] * 32
            gs, os_ = gcal["step_" + t][h], ocal["step_" + t][h]
            ulp = np.spacing(np.abs(os_).astype(np.float32))
            assert np.all(np.abs(gs.astype(np.float64) - os_) <= 1.0 * ulp), (t, h)
        lam_g, lam_o = gcal["lam_" + t], ocal["lam_" + t]
        assert np.abs(lam_g - lam_o).max() <= 1e-10 * np.abs(lam_o).max()
    np.testing.assert_allclose(gcal["mu_k"], ocal["mu_k"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(gcal["mu_v"], ocal["mu_v"], rtol=0, atol=1e-12)
    for key in ("T_k", "A_k", "T_k_inv", "T_v", "U_v"):
        g, o = gcal[key], ocal[key]
        assert np.abs(g - o).max() <= 1e-7 * np.abs(o).max(), key
    return ties


def test_calibration_matches_oracle_tiny():
    c = _tiny()
    g = aatc.calibrate(c["k"], c["v"], c["q"], c["wl"].bits)
    gcal = g.export()
    assert gcal["W"] == 11
    _check_calibration(gcal, c["ocal"], 1)
    # generalized Parseval with the GPU transform and the data's query moment
    Q = to_np64(c["q"]).reshape(-1, 128)
    Sq = Q.T @ Q / Q.shape[0]
    Ti = gcal["T_k_inv"][0]
    assert np.abs(Ti.T @ Sq @ Ti - np.eye(128)).max() < 1e-8


def test_calibration_errors_reported():
    c = _tiny()
    with pytest.raises(aatc.AatcError) as e:
        aatc.calibrate(c["k"], c["v"], c["q"], c["wl"].bits, jacobi_max_sweeps=1)
    assert e.value.status == aatc.ERR_NO_CONVERGENCE
    kb = c["k"].clone()
    kb[0, 17, 5] = float("nan")
    with pytest.raises(aatc.AatcError) as e:
        aatc.calibrate(kb, c["v"], c["q"], c["wl"].bits)
    assert e.value.status == aatc.ERR_NONFINITE
    # the context stays usable afterwards
    aatc.calibrate(c["k"], c["v"], c["q"], c["wl"].bits).free()


# ----------------------------------------------------------------- encode
_records = records


@pytest.mark.parametrize("L_new,start,L_cap", [(1024, 0, 1024), (1000, 24, 1056), (1, 7, 32), (129, 0, 160),
                                               (45, 31, 96)])
def test_encode_matches_oracle_with_imported_calibration(L_new, start, L_cap):
    c = _tiny()
    wl, ocal = c["wl"], c["ocal"]
    W = ocal["W"]
    g = aatc.import_calib(ocal, wl.n_q_heads, wl.dtype)
    kc, vc = synth.cache_inputs(wl, device="cuda", seq_len=L_new, batch=2)
    kp = torch.full((2, 1, L_cap, W), -1, dtype=torch.int32, device="cuda")
    vp = kp.clone()
    aatc.encode(g, kc, vc, kp, vp, start_pos=start)
    torch.cuda.synchronize()
    for t, kind, x, p in (("k", oracle.KEYS, kc, kp), ("v", oracle.VALUES, vc, vp)):
        _, codes, pre = oracle.encode_cache(to_np64(x), ocal, t, want_codes=True, want_pre=True)
        compare_codes(_records(p, W, kind, L_new, start), codes, pre, ocal["bits_" + t][0])
        # every bit of every other token is untouched: overwrite the written
        # tokens with ones through the oracle's tiling and expect all ones
        cc = as_u32(p).reshape(2, -1).copy()
        ones = np.full((L_new, W), 0xFFFFFFFF, dtype=np.uint32)
        for b in range(2):
            oracle.cache_put(ones, kind, cache=cc[b], start=start)
        assert np.all(cc == 0xFFFFFFFF), t
    g.check()


_bf16_cache = {}


def _bf16_two_heads():
    """Llama-shaped bf16 calibration of two KV heads (oracle), for the tensor-core encoder."""
    if not _bf16_cache:
        wl = synth.dataclasses.replace(WL["llama_32k"], n_kv_heads=2, n_q_heads=8)
        k, v, q = synth.calib_inputs(wl, device="cuda")
        _bf16_cache.update(wl=wl, ocal=_oracle_cal(k, v, q, wl.bits))
    return _bf16_cache


@pytest.mark.parametrize("L_new,start,L_cap,B", [(1024, 0, 1024, 2), (1000, 24, 1056, 2), (17, 7, 32, 1),
                                                 (300, 64, 384, 3), (257, 0, 288, 1)])
def test_encode_bf16_tensor_core_path(L_new, start, L_cap, B):
    """bf16 inputs go through the tensor-core encoder: full aligned 128-token
    blocks leave by bulk store, ragged or unaligned ones by per-token stores."""
    c = _bf16_two_heads()
    wl, ocal = c["wl"], c["ocal"]
    W = ocal["W"]
    g = aatc.import_calib(ocal, wl.n_q_heads, wl.dtype)
    kc, vc = synth.cache_inputs(wl, device="cuda", seq_len=L_new, batch=B)
    kp = torch.full((B, 2, L_cap, W), -1, dtype=torch.int32, device="cuda")
    vp = kp.clone()
    aatc.encode(g, kc, vc, kp, vp, start_pos=start)
    torch.cuda.synchronize()
    for t, kind, x, p in (("k", oracle.KEYS, kc, kp), ("v", oracle.VALUES, vc, vp)):
        _, codes, pre = oracle.encode_cache(to_np64(x), ocal, t, want_codes=True, want_pre=True)
        got = _records(p, W, kind, L_new, start)
        for h in range(2):
            compare_codes(got[:, h], codes[:, h], pre[:, h], ocal["bits_" + t][h])
        cc = as_u32(p).reshape(B * 2, -1).copy()
        ones = np.full((L_new, W), 0xFFFFFFFF, dtype=np.uint32)
        for r in range(B * 2):
            oracle.cache_put(ones, kind, cache=cc[r], start=start)
        assert np.all(cc == 0xFFFFFFFF), t
    g.check()


_bf16_wide = {}


@pytest.mark.parametrize("bits", [5.0, 8.0])
@pytest.mark.parametrize("L_new,start,L_cap,B", [(1024, 0, 1024, 2), (1000, 24, 1056, 1)])
def test_encode_bf16_tensor_core_wide_records(bits, L_new, start, L_cap, B):
    """The tensor-core encoder with records of 20 and 32 words: key words past
    the 16th in the tiled layout, and the two-stage instance (records above 12
    words)."""
    if bits not in _bf16_wide:
        wl = synth.dataclasses.replace(WL["llama_32k"], n_kv_heads=2, n_q_heads=8)
        k, v, q = synth.calib_inputs(wl, device="cuda")
        _bf16_wide[bits] = (wl, _oracle_cal(k, v, q, bits))
    wl, ocal = _bf16_wide[bits]
    W = ocal["W"]
    assert W == int(bits * 4)
    g = aatc.import_calib(ocal, wl.n_q_heads, wl.dtype)
    kc, vc = synth.cache_inputs(wl, device="cuda", seq_len=L_new, batch=B)
    kp = torch.full((B, 2, L_cap, W), -1, dtype=torch.int32, device="cuda")
    vp = kp.clone()
    aatc.encode(g, kc, vc, kp, vp, start_pos=start)
    torch.cuda.synchronize()
    _check_written(kp, kc, ocal, "k", oracle.KEYS, start, 2)
    _check_written(vp, vc, ocal, "v", oracle.VALUES, start, 2)
    g.check()


def _check_written(p, x, ocal, t, kind, start, heads):
    """Codes of the written tokens vs the oracle (rounding-tie rule), and every
    bit of every other token untouched (the cache started as all ones)."""
    W = ocal["W"]
    Bsz, L_new = x.shape[0], x.shape[2]
    _, codes, pre = oracle.encode_cache(to_np64(x), ocal, t, want_codes=True, want_pre=True)
    got = _records(p, W, kind, L_new, start)
    for h in range(heads):
        compare_codes(got[:, h], codes[:, h], pre[:, h], ocal["bits_" + t][h])
    cc = as_u32(p).reshape(Bsz * heads, -1).copy()
    ones = np.full((L_new, W), 0xFFFFFFFF, dtype=np.uint32)
    for r in range(Bsz * heads):
        oracle.cache_put(ones, kind, cache=cc[r], start=start)
    assert np.all(cc == 0xFFFFFFFF), t


@pytest.mark.parametrize("case,L_new,start,L_cap,B", [("tiny", 1, 0, 32, 2), ("tiny", 16, 24, 64, 2),
                                                      ("tiny", 3, 31, 64, 1), ("bf16", 1, 1023, 1024, 1),
                                                      ("bf16", 5, 62, 96, 3), ("bf16", 16, 0, 32, 1),
                                                      ("bf16", 2, 33, 64, 2)])
def test_encode_append_path(case, L_new, start, L_cap, B):
    """Up to 16 new tokens per row (a decode step) take the append kernel:
    one CTA per (KV head, tensor, row), fp32 transform, records placed token
    by token (tile boundaries and odd value half-word slots included)."""
    c = _tiny() if case == "tiny" else _bf16_two_heads()
    wl, ocal = c["wl"], c["ocal"]
    H = wl.n_kv_heads
    g = aatc.import_calib(ocal, wl.n_q_heads, wl.dtype)
    kc, vc = synth.cache_inputs(wl, layer=2, device="cuda", seq_len=L_new, batch=B)
    kp = torch.full((B, H, L_cap, ocal["W"]), -1, dtype=torch.int32, device="cuda")
    vp = kp.clone()
    aatc.encode(g, kc, vc, kp, vp, start_pos=start)
    torch.cuda.synchronize()
    _check_written(kp, kc, ocal, "k", oracle.KEYS, start, H)
    _check_written(vp, vc, ocal, "v", oracle.VALUES, start, H)
    g.check()


def test_encode_token_by_token_matches_one_shot_oracle():
    """A decode loop: 40 appends of one token each (every value word is
    shared by two tokens written by different launches) give the oracle's
    codes for all 40 tokens."""
    c = _bf16_two_heads()
    wl, ocal = c["wl"], c["ocal"]
    W = ocal["W"]
    g = aatc.import_calib(ocal, wl.n_q_heads, wl.dtype)
    L = 40
    kc, vc = synth.cache_inputs(wl, layer=3, device="cuda", seq_len=L, batch=2)
    kp = aatc.alloc_cache(g, 2, L)
    vp = aatc.alloc_cache(g, 2, L)
    for i in range(L):
        aatc.encode(g, kc[:, :, i:i + 1].contiguous(), vc[:, :, i:i + 1].contiguous(), kp, vp, start_pos=i)
    torch.cuda.synchronize()
    for t, kind, x, p in (("k", oracle.KEYS, kc, kp), ("v", oracle.VALUES, vc, vp)):
        _, codes, pre = oracle.encode_cache(to_np64(x), ocal, t, want_codes=True, want_pre=True)
        got = _records(p, W, kind, L)
        for h in range(2):
            compare_codes(got[:, h], codes[:, h], pre[:, h], ocal["bits_" + t][h])
    g.check()


def test_encode_writes_the_oracle_cache_bit_for_bit():
    """Away from rounding ties the whole tiled cache equals the oracle's."""
    c = _tiny()
    wl, ocal = c["wl"], c["ocal"]
    W = ocal["W"]
    g = aatc.import_calib(ocal, wl.n_q_heads, wl.dtype)
    kc, vc = synth.cache_inputs(wl, device="cuda", seq_len=200, batch=1)
    kp = aatc.alloc_cache(g, 1, 200)
    vp = aatc.alloc_cache(g, 1, 200)
    aatc.encode(g, kc, vc, kp, vp)
    for t, kind, x, p in (("k", oracle.KEYS, kc, kp), ("v", oracle.VALUES, vc, vp)):
        rec, codes, pre = oracle.encode_cache(to_np64(x), ocal, t, want_codes=True, want_pre=True)
        ref = oracle.to_cache(rec, kind, p.shape[2])
        got = as_u32(p).reshape(ref.shape)
        near_tie = np.abs(pre - np.floor(pre) - 0.5) < 1e-3
        clean = ~near_tie.any(axis=-1)[0, 0]          # tokens with no near-tie code
        gr = oracle.from_cache(got, W, kind, 200)[0, 0]
        assert np.array_equal(gr[clean], rec[0, 0][clean])
        if clean.all():
            assert np.array_equal(got, ref)


def test_encode_rejects_capacity_and_flags_nonfinite():
    c = _tiny()
    g = aatc.import_calib(c["ocal"], 16, torch.float32)
    kc, vc = synth.cache_inputs(c["wl"], device="cuda", seq_len=16)
    kp = torch.zeros(1, 1, 32, 11, dtype=torch.int32, device="cuda")
    vp = kp.clone()
    with pytest.raises(aatc.AatcError) as e:
        aatc.encode(g, kc, vc, kp, vp, start_pos=20)
    assert e.value.status == aatc.ERR_CAPACITY
    bad = torch.zeros(1, 1, 20, 11, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):                 # the binding checks the cache shape
        aatc.encode(g, kc, vc, bad, bad, start_pos=0)
    import ctypes
    st = aatc.lib().aatc_encode(g.handle, ctypes.c_void_p(kc.data_ptr()), ctypes.c_void_p(vc.data_ptr()), 1, 16, 0,
                                20, ctypes.c_void_p(bad.data_ptr()), ctypes.c_void_p(bad.data_ptr()), None)
    assert st == aatc.ERR_INVALID_ARG and "multiple of 32" in aatc.last_error()
    kc[0, 0, 3, 3] = float("inf")
    aatc.encode(g, kc, vc, kp, vp, start_pos=0)
    with pytest.raises(aatc.AatcError) as e:
        g.check()
    assert e.value.status == aatc.ERR_NONFINITE
    g.check()      # the status was cleared


# ----------------------------------------------------------------- decode
def _oracle_records(wl, ocal, B, L, layer=0):
    kc, vc = synth.cache_inputs(wl, layer=layer, device="cpu", seq_len=L, batch=B)
    kp, _, _ = oracle.encode_cache(to_np64(kc), ocal, "k")
    vp, _, _ = oracle.encode_cache(to_np64(vc), ocal, "v")
    return kp, vp


_upload = upload


@pytest.mark.parametrize("lens", [[1024], [1, 1024, 0], [127, 129, 1000], [31, 32, 33, 64, 2]])
def test_decode_matches_oracle_from_identical_codes(lens):
    c = _tiny()
    wl, ocal = c["wl"], c["ocal"]
    B, L = len(lens), max(lens)
    kp, vp = _oracle_records(wl, ocal, B, 1024)
    q = synth.query_inputs(wl, device="cuda", batch=B)
    ref = oracle.decode_attention(to_np64(q), kp, vp, ocal, seq_lens=lens)
    g = aatc.import_calib(ocal, wl.n_q_heads, wl.dtype)
    kpt, vpt = _upload(kp, oracle.KEYS, 1024), _upload(vp, oracle.VALUES, 1024)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = aatc.decode_attention(g, q, kpt, vpt, L, seq_lens=sl).cpu().numpy()
    for b in range(B):
        if lens[b] == 0:
            assert np.all(out[b] == 0)
        else:
            assert attn_rel_err(out[b], ref[b]) <= ATTN_RTOL, (b, attn_rel_err(out[b], ref[b]))
    # without seq_lens every row attends L tokens
    out2 = aatc.decode_attention(g, q, kpt, vpt, L).cpu().numpy()
    ref2 = oracle.decode_attention(to_np64(q), kp, vp, ocal, seq_lens=[L] * B)
    assert attn_rel_err(out2, ref2) <= ATTN_RTOL
    g.check()


_synthetic_calibration = synthetic_calibration


@pytest.mark.parametrize("case", ["G1", "G7", "G8", "wide_W20", "many_pieces", "key_pieces8", "key_pieces8_G8",
                                  "bits2", "bits4", "bits8"])
def test_decode_paths_match_oracle(case):
    """Fast path (GQA groups of 1..8, 2.0..4.0 bits, key bytes of up to eight
    code pieces) and the general path (records above 16 words up to the
    32-word maximum, value bytes holding more than four code pieces, key bytes
    of more than four pieces with GQA groups above 4); each also through a
    paged pool on shuffled 32-token blocks, which must give the contiguous
    output exactly."""
    lam = 0.95 ** np.arange(128)
    G, B_bits = 4, 352
    if case == "G1":
        G = 1
    elif case in ("G7", "G8", "key_pieces8_G8"):
        G = int(case[-1:])
    elif case == "wide_W20":
        B_bits = 640
    elif case == "bits2":
        B_bits = 256
    elif case == "bits4":
        B_bits = 512
    elif case == "bits8":
        B_bits = 1024
    bk, _ = oracle.allocate_bits(lam, B_bits)
    bv, _ = oracle.allocate_bits(0.93 ** np.arange(128), B_bits)
    if case == "many_pieces":
        # 96 two-bit and 32 one-bit codes: the order rule puts the last 1-bit
        # codes eight to a byte, beyond what the fast decoder reads
        bk = np.array([2] * 96 + [1] * 32, dtype=np.int32)
        bv = bk.copy()
    if case.startswith("key_pieces8"):
        # the same key record (eight 1-bit codes to a byte at its end), values of 11 words
        bk = np.array([2] * 96 + [1] * 32, dtype=np.int32)
    cal = _synthetic_calibration(G, bk, bv)
    L, Bsz = 333, 2
    rng = np.random.default_rng(1)
    kp = np.stack([[oracle.pack(rng.integers(0, 2 ** np.maximum(bk, 1)) * (bk > 0), bk) for _ in range(L)]
                   for _ in range(Bsz)])[:, None]
    vp = np.stack([[oracle.pack(rng.integers(0, 2 ** np.maximum(bv, 1)) * (bv > 0), bv) for _ in range(L)]
                   for _ in range(Bsz)])[:, None]
    q = torch.from_numpy(rng.standard_normal((Bsz, G, 128)).astype(np.float32) * 3).cuda()
    g = aatc.import_calib(cal, G, torch.float32)
    L_cap = aatc.cache_capacity(L)
    kc, vc = _upload(kp, oracle.KEYS, L_cap), _upload(vp, oracle.VALUES, L_cap)
    out = aatc.decode_attention(g, q, kc, vc, L)
    ref = oracle.decode_attention(to_np64(q), kp, vp, cal)
    err = attn_rel_err(out.cpu().numpy(), ref)
    assert err <= ATTN_RTOL, (case, err)
    # the same caches on shuffled 32-token blocks of a pool
    bpr = L_cap // 32
    perm = torch.randperm(Bsz * bpr + 5, generator=torch.Generator().manual_seed(3))
    table = perm[:Bsz * bpr].reshape(Bsz, bpr).to(torch.int32).cuda()
    pools = []
    for c, t in ((kc, "k"), (vc, "v")):
        pool = aatc.alloc_pool(g, Bsz * bpr + 5, 32, tensor=t)
        pool[table.long()] = c.reshape(Bsz, 1, bpr, 32, c.shape[-1]).permute(0, 2, 1, 3, 4)
        pools.append(pool)
    out_p = aatc.decode_attention_paged(g, q, pools[0], pools[1], table, L)
    assert torch.equal(out_p, out), case
    g.check()


def test_decode_workspace_reuse_across_shapes():
    """One workspace, zeroed once, for calls of different shapes in a row:
    each call leaves its split counters at zero and nothing else it left
    leaks into the next call.  A workspace that was not zeroed is reported."""
    c = _tiny()
    wl, ocal = c["wl"], c["ocal"]
    g = aatc.import_calib(ocal, wl.n_q_heads, wl.dtype)
    kp, vp = _oracle_records(wl, ocal, 3, 700)
    kpt, vpt = _upload(kp, oracle.KEYS, 704), _upload(vp, oracle.VALUES, 704)
    ws = aatc.new_workspace(g, 3, 700)
    ws[1024:] = 0x7F                              # only the counters must start at zero
    for Bsz, L in ((3, 700), (1, 40), (2, 513), (3, 700)):
        q = synth.query_inputs(wl, device="cuda", batch=Bsz, step=L)
        out = aatc.decode_attention(g, q, kpt[:Bsz], vpt[:Bsz], L, workspace=ws).cpu().numpy()
        ref = oracle.decode_attention(to_np64(q), kp[:Bsz], vp[:Bsz], ocal, seq_lens=[L] * Bsz)
        assert attn_rel_err(out, ref) <= ATTN_RTOL, (Bsz, L)
        assert torch.all(ws[:1024] == 0)          # the counters are back at zero
    g.check()
    bad = torch.full_like(ws, 0x7F)               # never zeroed
    aatc.decode_attention(g, q, kpt[:3], vpt[:3], 700, workspace=bad)
    with pytest.raises(aatc.AatcError) as e:
        g.check()
    assert e.value.status == aatc.ERR_INVALID_ARG and "zeroed" in str(e.value)


def test_decode_workspace_and_capacity_errors():
    c = _tiny()
    g = aatc.import_calib(c["ocal"], 16, torch.float32)
    q = synth.query_inputs(c["wl"], device="cuda")
    kp = torch.zeros(1, 1, 64, 11, dtype=torch.int32, device="cuda")
    with pytest.raises(aatc.AatcError) as e:
        aatc.decode_attention(g, q, kp, kp, 65)
    assert e.value.status == aatc.ERR_CAPACITY
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(aatc.AatcError) as e:
        aatc.decode_attention(g, q, kp, kp, 64, workspace=ws)
    assert e.value.status == aatc.ERR_INVALID_ARG
    out = aatc.decode_attention(g, q, kp, kp, 0)
    assert torch.all(out == 0)


# ----------------------------------------------------------------- end to end
PIPELINE_RTOL = 1e-2


def _end_to_end(wl, sample, layer=0, seq_len=None, bits=None, decode_step=False):
    """GPU pipeline on the full workload vs the oracle pipeline on sampled (b, h)."""
    bits = bits or wl.bits
    L = seq_len or wl.seq_len
    k, v, q = synth.calib_inputs(wl, layer=layer, device="cuda")
    g = aatc.calibrate(k, v, q, bits)
    ocal = _oracle_cal(k, v, q, bits)
    gcal = g.export()
    ties = _check_calibration(gcal, ocal, wl.n_kv_heads)
    kc, vc = synth.cache_inputs(wl, layer=layer, device="cuda", seq_len=L)
    kp = aatc.alloc_cache(g, wl.batch, L + 1)
    vp = aatc.alloc_cache(g, wl.batch, L + 1)
    aatc.encode(g, kc, vc, kp, vp)
    Ltot = L
    if decode_step:
        # one decode step: encode the new token at position L, attend over L + 1
        kn, vn = synth.cache_inputs(wl, layer=layer + 1, device="cuda", seq_len=1, batch=wl.batch)
        aatc.encode(g, kn, vn, kp, vp, start_pos=L)
        kc = torch.cat([kc, kn], dim=2)
        vc = torch.cat([vc, vn], dim=2)
        Ltot = L + 1
    qd = synth.query_inputs(wl, layer=layer, device="cuda")
    out = aatc.decode_attention(g, qd, kp, vp, Ltot).cpu().numpy()
    g.check()
    G = wl.group
    worst = 0.0
    for (b, h) in sample:
        if not np.array_equal(gcal["bits_k"][h], ocal["bits_k"][h]) or \
                not np.array_equal(gcal["bits_v"][h], ocal["bits_v"][h]):
            continue        # a reported allocation tie: codes are not comparable
        sub = {key: (val[h:h + 1] if isinstance(val, np.ndarray) and val.ndim >= 1 and val.shape[0] == wl.n_kv_heads
                     else val) for key, val in ocal.items()}
        xk = to_np64(kc[b:b + 1, h:h + 1, :Ltot])
        xv = to_np64(vc[b:b + 1, h:h + 1, :Ltot])
        rk, ck, pk = oracle.encode_cache(xk, sub, "k", want_codes=True, want_pre=True)
        rv, cv, pv = oracle.encode_cache(xv, sub, "v", want_codes=True, want_pre=True)
        compare_codes(_records(kp[b:b + 1, h:h + 1], ocal["W"], oracle.KEYS, Ltot), ck, pk, sub["bits_k"][0])
        compare_codes(_records(vp[b:b + 1, h:h + 1], ocal["W"], oracle.VALUES, Ltot), cv, pv, sub["bits_v"][0])
        qq = to_np64(qd[b:b + 1, h * G:(h + 1) * G])
        # decode parity from identical codes: the oracle decodes the GPU's own
        # records with the GPU's calibration tables
        gsub = {key: (val[h:h + 1] if isinstance(val, np.ndarray) and val.ndim >= 1 and
                      val.shape[0] == wl.n_kv_heads else val) for key, val in gcal.items()}
        gk = _records(kp[b:b + 1, h:h + 1], gcal["W"], oracle.KEYS, Ltot)
        gv = _records(vp[b:b + 1, h:h + 1], gcal["W"], oracle.VALUES, Ltot)
        ref = oracle.decode_attention(qq, gk, gv, gsub)
        err = attn_rel_err(out[b, h * G:(h + 1) * G], ref[0])
        worst = max(worst, err)
        assert err <= ATTN_RTOL, (b, h, err)
        # the oracle's own pipeline (its calibration, its codes): codes may differ
        # by one level at rounding ties, which moves the output by more than the
        # identical-code tolerance; this only guards against gross errors
        pipe = attn_rel_err(out[b, h * G:(h + 1) * G], oracle.decode_attention(qq, rk, rv, sub)[0])
        assert pipe <= PIPELINE_RTOL, (b, h, pipe)
    g.free()
    return worst, ties


# every KV head of at least one row is compared in each workload
def test_end_to_end_llama_32k_with_decode_step():
    _end_to_end(WL["llama_32k"], sample=[(0, h) for h in range(8)], decode_step=True)


def test_end_to_end_llama_b16_8k():
    _end_to_end(WL["llama_b16_8k"], sample=[(0, h) for h in range(8)] + [(15, 7)])


def test_end_to_end_qwen_128k():
    _end_to_end(WL["qwen_128k"], sample=[(3, h) for h in range(4)])


@pytest.mark.parametrize("bits", [2.0, 2.75, 4.0])
def test_end_to_end_stack_layer_budgets(bits):
    _end_to_end(WL["llama_stack"], sample=[(0, h) for h in range(8)], layer=31, seq_len=4096, bits=bits)


def test_kernel_variant_reused_with_more_shared_memory():
    """Two record widths served by one decode kernel variant, the narrower
    (less shared memory) planned after the wider had launched: the wider must
    still launch (sizing a new shape must not lower the variant's
    shared-memory limit below what an earlier launch set)."""
    rng = np.random.default_rng(5)
    lam = 0.95 ** np.arange(128)
    bv, _ = oracle.allocate_bits(0.93 ** np.arange(128), 352)
    outs = []
    for bk_bits in (352, 224, 352):     # 11/11 words, then 7/11, then 11/11 again
        bk, _ = oracle.allocate_bits(lam, bk_bits)
        cal = _synthetic_calibration(4, bk, bv)
        L, Bsz = 2000, 1
        kp = np.stack([[oracle.pack(rng.integers(0, 2 ** np.maximum(bk, 1)) * (bk > 0), bk) for _ in range(L)]])[:, None]
        vp = np.stack([[oracle.pack(rng.integers(0, 2 ** np.maximum(bv, 1)) * (bv > 0), bv) for _ in range(L)]])[:, None]
        q = torch.from_numpy(rng.standard_normal((Bsz, 4, 128)).astype(np.float32)).cuda()
        g = aatc.import_calib(cal, 4, torch.float32)
        L_cap = aatc.cache_capacity(L)
        out = aatc.decode_attention(g, q, _upload(kp, oracle.KEYS, L_cap), _upload(vp, oracle.VALUES, L_cap), L)
        ref = oracle.decode_attention(to_np64(q), kp, vp, cal)
        assert attn_rel_err(out.cpu().numpy(), ref) <= ATTN_RTOL, bk_bits
        g.check()
        outs.append(out)
