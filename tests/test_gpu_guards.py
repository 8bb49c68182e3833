"""Guard words after every caller-owned output buffer (compute-sanitizer is not
available, so out-of-bounds writes are looked for directly).

Each output -- packed caches, paged pools, the decode output and workspaces
of exactly the size the library asks for -- is the front of a larger buffer
whose tail holds a sentinel.  After every encode and decode call, on odd sizes
(1, 15, 33 and 32769 tokens, ragged rows), the tails must be intact.
"""
import math

import pytest
import torch

import oracle
from parity_util import to_np64
from quantized_attention_kv_b300 import aatc, synth

pytestmark = pytest.mark.gpu
SENTINEL = 0x5A5A5A5A
GUARD = 256   # 32-bit words after each buffer


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantized_attention_kv_b300 import build
    build.build()
    aatc.lib()
    yield
    torch.cuda.synchronize()


class Guarded:
    """A tensor of `shape` at the front of an int32 buffer with GUARD sentinel words after it."""

    def __init__(self, shape, dtype):
        nbytes = math.prod(shape) * torch.empty(0, dtype=dtype).element_size()
        assert nbytes % 4 == 0
        self.n = nbytes // 4
        self.full = torch.full((self.n + GUARD,), SENTINEL, dtype=torch.int32, device="cuda")
        self.full[:self.n].zero_()
        self.t = self.full[:self.n].view(dtype).view(shape)

    def intact(self):
        return bool(torch.all(self.full[self.n:] == SENTINEL))


_cals = {}


def _case(name):
    if name not in _cals:
        wl = WL_TINY if name == "tiny" else synth.dataclasses.replace(synth.WORKLOADS["llama_32k"],
                                                                         n_kv_heads=2, n_q_heads=8)
        k, v, q = synth.calib_inputs(wl, device="cuda")
        _cals[name] = (wl, oracle.calibrate(to_np64(k), to_np64(v), to_np64(q), wl.bits))
    return _cals[name]


WL_TINY = synth.WORKLOADS["tiny"]


@pytest.mark.parametrize("name,L", [("bf16", 1), ("bf16", 15), ("bf16", 33), ("bf16", 32769), ("tiny", 33),
                                    ("tiny", 1)])
def test_no_write_past_any_output(name, L):
    wl, ocal = _case(name)
    g = aatc.import_calib(ocal, wl.n_q_heads, wl.dtype)
    B, H, W = 3, wl.n_kv_heads, ocal["W"]
    L_cap = aatc.cache_capacity(L)
    kc, vc = synth.cache_inputs(wl, device="cuda", seq_len=L, batch=B)
    kp, vp = Guarded((B, H, L_cap, W), torch.int32), Guarded((B, H, L_cap, W), torch.int32)
    aatc.encode(g, kc, vc, kp.t, vp.t, start_pos=0)
    torch.cuda.synchronize()
    assert kp.intact() and vp.intact()

    lens = torch.tensor([L, max(L - 7, 0), (L + 1) // 2], dtype=torch.int32, device="cuda")
    q = synth.query_inputs(wl, device="cuda", batch=B, step=L)
    out = Guarded((B, wl.n_q_heads, 128), torch.float32)
    need = aatc.workspace_size(g, B, L)          # a multiple of 256 bytes (or 0)
    ws = Guarded((need // 4,), torch.int32) if need else None
    aatc.decode_attention(g, q, kp.t, vp.t, L, seq_lens=lens, out=out.t,
                          workspace=ws.t.view(torch.uint8) if ws else None)
    torch.cuda.synchronize()
    assert out.intact() and (ws is None or ws.intact()) and kp.intact() and vp.intact()

    # paged: 32-token blocks, shuffled; a one-token append per row at its own position
    bpr = L_cap // 32 + 1
    nb = B * bpr + 2
    table = torch.randperm(nb, generator=torch.Generator().manual_seed(L))[:B * bpr].reshape(B, bpr)
    table = table.to(torch.int32).cuda()
    kq, vq = Guarded((nb, H, 32, W), torch.int32), Guarded((nb, H, 32, W), torch.int32)
    aatc.encode_paged(g, kc, vc, kq.t, vq.t, table, start_pos=0)
    kn, vn = synth.cache_inputs(wl, layer=1, device="cuda", seq_len=1, batch=B)
    aatc.encode_paged(g, kn, vn, kq.t, vq.t, table, row_start=lens)
    out2 = Guarded((B, wl.n_q_heads, 128), torch.float32)
    need2 = aatc.workspace_size(g, B, L + 1)
    ws2 = Guarded((need2 // 4,), torch.int32) if need2 else None
    aatc.decode_attention_paged(g, q, kq.t, vq.t, table, L + 1, seq_lens=lens + 1, out=out2.t,
                                workspace=ws2.t.view(torch.uint8) if ws2 else None)
    torch.cuda.synchronize()
    assert kq.intact() and vq.intact() and out2.intact() and (ws2 is None or ws2.intact())
    g.check()
