"""GPU tests of the paged cache (block tables).

A paged pool holds the same 32-token tiles as a contiguous cache, placed
block by block through a block table, and every kernel does the same
arithmetic on them.  So (1) encoding into a pool and gathering its blocks
back in logical order gives exactly the contiguous cache that aatc_encode
writes from the same inputs, and paged decode gives exactly the contiguous
decode's output; (2) paged decode over oracle-packed records scattered into
a pool matches the oracle's attention; (3) bad block tables and positions are
reported, and writes outside a row's blocks are skipped.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import ATTN_RTOL, attn_rel_err, to_np64
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


_cals = {}


def _case(name):
    """Oracle calibration of the tiny fp32 workload, or of two Llama-shaped bf16 KV heads."""
    if name not in _cals:
        if name == "tiny":
            wl = WL["tiny"]
        else:
            wl = synth.dataclasses.replace(WL["llama_32k"], n_kv_heads=2, n_q_heads=8)
        k, v, q = synth.calib_inputs(wl, device="cuda")
        _cals[name] = (wl, oracle.calibrate(to_np64(k), to_np64(v), to_np64(q), wl.bits))
    return _cals[name]


def _table(B, bpr, n_blocks, seed):
    """Block table: the rows' logical blocks on distinct, shuffled physical blocks."""
    g = torch.Generator().manual_seed(seed)
    return torch.randperm(n_blocks, generator=g)[:B * bpr].reshape(B, bpr).to(torch.int32).cuda()


def _gather(pool, table):
    """Pool [n_blocks][H][bt][W] -> contiguous cache [B][H][bpr*bt][W] in logical order."""
    B, bpr = table.shape
    _, H, bt, W = pool.shape
    return pool[table.long()].permute(0, 2, 1, 3, 4).reshape(B, H, bpr * bt, W)


def _scatter(cont, table, pool):
    B, H, Lc, W = cont.shape
    bt = pool.shape[2]
    pool[table.long()] = cont.reshape(B, H, Lc // bt, bt, W).permute(0, 2, 1, 3, 4)


@pytest.mark.parametrize("name,bt,B,L", [("tiny", 32, 3, 300), ("tiny", 128, 2, 1000), ("bf16", 64, 3, 300),
                                         ("bf16", 32, 3, 300), ("bf16", 128, 16, 8192), ("bf16", 256, 2, 5000),
                                         ("bf16", 64, 40, 2000), ("bf16", 32, 16, 8192)])
def test_paged_matches_contiguous_bit_for_bit(name, bt, B, L):
    """Prefill (tensor-core or fp32 encoder) and one appended token per row at
    per-row positions, into a shuffled pool and into a contiguous cache: the
    gathered pool equals the cache word for word, and paged decode equals
    contiguous decode exactly.  The shapes cover split and single-split decode
    units, warps that refill their stages (and read block entries ahead of
    them), ragged tails and blocks of 1 to 8 tiles."""
    wl, ocal = _case(name)
    H = wl.n_kv_heads
    g = aatc.import_calib(ocal, wl.n_q_heads, wl.dtype)
    bpr = -(-(L + 1) // bt)
    n_blocks = B * bpr + 7
    table = _table(B, bpr, n_blocks, seed=bt + B)
    kpool, vpool = aatc.alloc_pool(g, n_blocks, bt), aatc.alloc_pool(g, n_blocks, bt)
    kp, vp = aatc.alloc_cache(g, B, bpr * bt), aatc.alloc_cache(g, B, bpr * bt)
    kc, vc = synth.cache_inputs(wl, device="cuda", seq_len=L, batch=B)
    aatc.encode_paged(g, kc, vc, kpool, vpool, table, start_pos=0)
    aatc.encode(g, kc, vc, kp, vp, start_pos=0)
    pos = [L - (7 * b) % 50 for b in range(B)]
    kn, vn = synth.cache_inputs(wl, layer=1, device="cuda", seq_len=1, batch=B)
    aatc.encode_paged(g, kn, vn, kpool, vpool, table, row_start=torch.tensor(pos, dtype=torch.int32, device="cuda"))
    for b in range(B):
        aatc.encode(g, kn[b:b + 1].contiguous(), vn[b:b + 1].contiguous(), kp[b:b + 1], vp[b:b + 1],
                    start_pos=pos[b])
    torch.cuda.synchronize()
    assert torch.equal(_gather(kpool, table), kp)
    assert torch.equal(_gather(vpool, table), vp)

    lens = torch.tensor([p + 1 for p in pos], dtype=torch.int32, device="cuda")
    q = synth.query_inputs(wl, device="cuda", batch=B, step=L)
    o_paged = aatc.decode_attention_paged(g, q, kpool, vpool, table, L + 1, seq_lens=lens)
    o_cont = aatc.decode_attention(g, q, kp, vp, L + 1, seq_lens=lens)
    torch.cuda.synchronize()
    assert torch.equal(o_paged, o_cont)
    g.check()


@pytest.mark.parametrize("bt,lens", [(64, [1024, 1, 517]), (32, [33, 0, 700])])
def test_paged_decode_matches_oracle(bt, lens):
    """Oracle-packed records scattered into a pool: paged decode vs the oracle's attention."""
    wl, ocal = _case("tiny")
    g = aatc.import_calib(ocal, wl.n_q_heads, wl.dtype)
    B, L = len(lens), max(lens)
    kc, vc = synth.cache_inputs(wl, layer=4, device="cpu", seq_len=L, batch=B)
    kr, _, _ = oracle.encode_cache(to_np64(kc), ocal, "k")
    vr, _, _ = oracle.encode_cache(to_np64(vc), ocal, "v")
    bpr = -(-L // bt)
    table = _table(B, bpr, B * bpr + 3, seed=11)
    pools = []
    for rec, kind in ((kr, oracle.KEYS), (vr, oracle.VALUES)):
        c = oracle.to_cache(rec, kind, bpr * bt).view(np.int32).reshape(B, wl.n_kv_heads, bpr * bt, ocal["W"])
        pool = aatc.alloc_pool(g, B * bpr + 3, bt)
        _scatter(torch.from_numpy(c).cuda(), table, pool)
        pools.append(pool)
    q = synth.query_inputs(wl, device="cuda", batch=B, step=L)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = aatc.decode_attention_paged(g, q, pools[0], pools[1], table, L, seq_lens=sl).cpu().numpy()
    ref = oracle.decode_attention(to_np64(q), kr, vr, ocal, seq_lens=lens)
    assert attn_rel_err(out, ref) <= ATTN_RTOL
    g.check()


def test_paged_errors():
    wl, ocal = _case("tiny")
    g = aatc.import_calib(ocal, wl.n_q_heads, wl.dtype)
    W, H = ocal["W"], wl.n_kv_heads
    kc, vc = synth.cache_inputs(wl, device="cuda", seq_len=40)
    q = synth.query_inputs(wl, device="cuda")
    table = torch.tensor([[2, 0]], dtype=torch.int32, device="cuda")
    # block_tokens not 32 times a power of two (the binding passes the shape through)
    for bt in (48, 96):
        odd = torch.zeros(3, H, bt, W, dtype=torch.int32, device="cuda")
        with pytest.raises(aatc.AatcError) as e:
            aatc.encode_paged(g, kc, vc, odd, odd, table)
        assert e.value.status == aatc.ERR_INVALID_ARG
    kpool, vpool = aatc.alloc_pool(g, 3, 32), aatc.alloc_pool(g, 3, 32)
    # more tokens than the row's blocks hold
    big_k, big_v = synth.cache_inputs(wl, device="cuda", seq_len=65)
    with pytest.raises(aatc.AatcError) as e:
        aatc.encode_paged(g, big_k, big_v, kpool, vpool, table)
    assert e.value.status == aatc.ERR_CAPACITY
    with pytest.raises(aatc.AatcError) as e:
        aatc.decode_attention_paged(g, q, kpool, vpool, table, 65)
    assert e.value.status == aatc.ERR_CAPACITY
    # a device-side position past the row's blocks: the write is skipped and reported
    aatc.encode_paged(g, kc[:, :, :1].contiguous(), vc[:, :, :1].contiguous(), kpool, vpool, table,
                      row_start=torch.tensor([64], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert int(kpool.count_nonzero()) == 0 and int(vpool.count_nonzero()) == 0
    with pytest.raises(aatc.AatcError) as e:
        g.check()
    assert e.value.status == aatc.ERR_CAPACITY
    g.check()   # cleared
    # a block table entry outside the pool, inside the row's length: reported
    aatc.encode_paged(g, kc, vc, kpool, vpool, table)
    bad = torch.tensor([[2, 3]], dtype=torch.int32, device="cuda")
    aatc.decode_attention_paged(g, q, kpool, vpool, bad, 40)
    torch.cuda.synchronize()
    with pytest.raises(aatc.AatcError) as e:
        g.check()
    assert e.value.status == aatc.ERR_CAPACITY
    # the same entry past the row's length is never read
    aatc.decode_attention_paged(g, q, kpool, vpool, bad, 32)
    torch.cuda.synchronize()
    g.check()
