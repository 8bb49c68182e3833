"""GPU decode parity where the fast decoder's schedule is most stressed.

* Refill path: every warp of the split kernel streams more 32-token tiles than
  it has pipeline stages, so stages are reused and mbarrier phases flip, for
  the 2.0-bit (8-word) and 4.0-bit (16-word) records, with several splits per
  (row, KV head) and with one.
* Peaked softmax: the decoder raises its running maximum lazily (only when a
  score exceeds it by 8 in log2 units) and rescales its sums then.  Keys are
  built so that one code decides every score: a dominant token at chosen
  positions (the last token of a row and of tiles and warps' ranges), scores
  rising monotonically along the row, all keys equal, and queries scaled by 50.

Decode is compared from identical codes: the oracle decodes the same records
with the same calibration ("Attention-Aware Transform Coding Guide: KV
Compression", section "Formal Attention Distortion Model": exact softmax
attention over the reconstructed keys and values).  Tolerances are those of
tests/parity_util.py.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import ATTN_RTOL, attn_rel_err, records, synthetic_calibration, to_np64, upload
from quantized_attention_kv_b300 import aatc, synth

pytestmark = pytest.mark.gpu
WL = synth.WORKLOADS
LOG2E = 1.4426950408889634


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantized_attention_kv_b300 import build
    build.build()
    aatc.lib()
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("bits", [2.0, 4.0])
@pytest.mark.parametrize("layout", ["splits", "single"])
def test_decode_refill_path_matches_oracle(bits, layout):
    """Llama-shaped stack layer (8 KV heads, GQA group 4) calibrated and encoded
    on the GPU; decode of the GPU's records against the oracle's decode of the
    same records.  "splits": one row of 40,000 tokens, 8 (row, KV head) units
    of 18 splits of 70 tiles (4-5 tiles per warp).  "single": 19 rows of 2,100
    tokens, 152 units that each fill one CTA (66 tiles, 4-5 per warp) and
    finish without a combine."""
    wl = WL["llama_stack"]
    B, L = (1, 40000) if layout == "splits" else (19, 2100)
    k, v, q = synth.calib_inputs(wl, layer=31, device="cuda")
    g = aatc.calibrate(k, v, q, bits)
    gcal = g.export()
    W = gcal["W"]
    assert W == {2.0: 8, 4.0: 16}[bits]
    # the two layouts take the two ends of the call: partial slots + combine, or none
    assert (aatc.workspace_size(g, B, L) > 0) == (layout == "splits")
    kc, vc = synth.cache_inputs(wl, layer=31, device="cuda", seq_len=L, batch=B)
    kp = aatc.alloc_cache(g, B, L)
    vp = aatc.alloc_cache(g, B, L)
    aatc.encode(g, kc, vc, kp, vp)
    qd = synth.query_inputs(wl, layer=31, device="cuda", batch=B)
    out = aatc.decode_attention(g, qd, kp, vp, L).cpu().numpy()
    g.check()
    rows = [0] if B == 1 else [0, 7, 18]
    rk = records(kp[rows], W, oracle.KEYS, L)
    rv = records(vp[rows], W, oracle.VALUES, L)
    ref = oracle.decode_attention(to_np64(qd[rows]), rk, rv, gcal)
    err = attn_rel_err(out[rows], ref)
    assert err <= ATTN_RTOL, (bits, layout, err)


def _allocs(B_bits):
    bk, _ = oracle.allocate_bits(0.95 ** np.arange(128), B_bits)
    bv, _ = oracle.allocate_bits(0.93 ** np.arange(128), B_bits)
    return bk, bv


def _key_records(bk, n, u0, base=None):
    """n key records whose channel-0 code is u0[i] and whose other codes are
    those of `base` (all zero if None); built from one packed record per
    distinct u0 value."""
    base = np.zeros(128, dtype=np.int64) if base is None else np.asarray(base, dtype=np.int64)
    levels = np.unique(u0)
    table = {}
    for lv in levels:
        u = base.copy()
        u[0] = lv
        table[int(lv)] = oracle.pack(u, bk)
    W = int(bk.sum()) // 32
    out = np.empty((n, W), dtype=np.uint32)
    for lv, rec in table.items():
        out[u0 == lv] = rec
    return out


def _queries(cal, B, G, gap_log2, rng):
    """Queries whose scores depend on the channel-0 key code alone (q' along
    channel 0, since A_k = Qk^T here): a code step from 0 to the top level adds
    gap_log2 * (1 + g/4) to the log2 score of query head g."""
    Qk = cal["T_k_inv"][0]
    top = (1 << int(cal["bits_k"][0][0])) - 1
    unit = LOG2E * float(cal["step_k"][0][0]) / np.sqrt(128.0) * top   # log2 score gap per unit of q along Qk[:,0]
    q = np.empty((B, G, 128))
    for g in range(G):
        s = gap_log2 * (1 + g / 4) / unit
        q[:, g] = s * Qk[:, 0] + 1e-3 * rng.standard_normal((B, 128))
    return q


GEOMS = {
    # one row, one KV head: 148 splits of 64 tiles each (4 per warp), ragged end
    "splits": (1, 148 * 64 * 32 + 17),
    # 150 rows that each fill one CTA: 66 tiles each (4-5 per warp)
    "single": (150, 2093),
}


@pytest.mark.parametrize("G", [4, 8])
@pytest.mark.parametrize("geom", ["splits", "single"])
@pytest.mark.parametrize("case", ["dominant", "rising", "equal_keys", "q_x50"])
def test_decode_peaked_softmax_from_identical_codes(case, geom, G):
    rng = np.random.default_rng({"dominant": 1, "rising": 2, "equal_keys": 3, "q_x50": 4}[case])
    B, L = GEOMS[geom]
    bk, bv = _allocs(352)
    cal = synthetic_calibration(G, bk, bv, seed=5)
    W = cal["W"]
    top = (1 << int(bk[0])) - 1
    # values: random words are random codes (every record bit belongs to one code)
    vp = rng.integers(0, 2 ** 32, size=(B, 1, L, W), dtype=np.uint64).astype(np.uint32)
    base = rng.integers(0, 2 ** np.maximum(bk, 1)) * (bk > 0)
    if case == "dominant":
        # one token per row with the top channel-0 code, the rest at code 0: the
        # row's last token, the last token of a tile, the last token of a warp's
        # first tile, the first token, and random positions
        u0 = np.zeros((B, L), dtype=np.int64)
        picks = [L - 1, 32 * 40 - 1, 32 * 16 - 1, 0, 31, L // 2]
        for b in range(B):
            u0[b, picks[b] if b < len(picks) else int(rng.integers(0, L))] = top
        kp = np.stack([_key_records(bk, L, u0[b], base) for b in range(B)])[:, None]
        q = _queries(cal, B, G, 24.0, rng)          # 24..(24 * 2.75) log2 units above the rest
    elif case == "rising":
        # the channel-0 code rises with the position: scores rise monotonically
        # along the row, by 40..110 log2 units in all, so every warp keeps
        # raising its maximum
        u0 = np.minimum(np.arange(L) * (top + 1) // L, top)
        kp = np.broadcast_to(_key_records(bk, L, u0, base), (B, 1, L, W)).copy()
        q = _queries(cal, B, G, 40.0, rng)
    elif case == "equal_keys":
        # every key the same: uniform weights, the output is the mean value
        kp = np.broadcast_to(oracle.pack(base, bk), (B, 1, L, W)).copy()
        q = rng.standard_normal((B, G, 128)) * 3
    else:
        kp = rng.integers(0, 2 ** 32, size=(B, 1, L, W), dtype=np.uint64).astype(np.uint32)
        q = rng.standard_normal((B, G, 128)) * 50
    g = aatc.import_calib(cal, G, torch.float32)
    L_cap = aatc.cache_capacity(L)
    kc, vc = upload(kp, oracle.KEYS, L_cap), upload(vp, oracle.VALUES, L_cap)
    qt = torch.from_numpy(q.astype(np.float32)).cuda()
    out = aatc.decode_attention(g, qt, kc, vc, L).cpu().numpy()
    g.check()
    rows = list(range(B)) if B <= 8 else [0, 1, 2, 3, 4, 5, 77, B - 1]
    ref = oracle.decode_attention(q[rows].astype(np.float32).astype(np.float64), kp[rows], vp[rows], cal)
    err = attn_rel_err(out[rows], ref)
    assert err <= ATTN_RTOL, (case, geom, G, err)
    if case == "dominant":
        # the reference itself is peaked: most weight on the dominant token
        Vh = oracle.reconstruct(vp[0, 0], cal["U_v"][0], cal["mu_v"][0], cal["step_v"][0], bv)
        j = int(np.flatnonzero(u0[0] == top)[0])
        assert np.abs(ref[0, G - 1] - Vh[j]).max() < 0.05 * np.abs(Vh[j]).max()
