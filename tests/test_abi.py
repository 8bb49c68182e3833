"""Host-side checks of the C ABI: the library loads, exports every entry point
declared in include/aatc.h, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from quantized_attention_kv_b300 import aatc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", f)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(aatc_\w+)\s*\(", txt))
    return names


@pytest.fixture(scope="module")
def L():
    from quantized_attention_kv_b300 import build
    build.build()
    return aatc.lib()


def test_library_exports_every_declared_symbol(L):
    names = _declared()
    assert {"aatc_calibrate", "aatc_encode", "aatc_decode_attention", "aatc_free"} <= names
    for n in names:
        assert hasattr(L, n), n
    assert set(aatc.EXPORTED) <= names


def test_null_and_bad_arguments_rejected_on_host(L):
    P = ctypes.c_void_p
    h = P()
    assert L.aatc_calibrate(None, None, None, None, ctypes.byref(h), None) == aatc.ERR_INVALID_ARG
    d = aatc.CalibDesc(64, 1, 1, 100, 2.75, 0, 0)
    assert L.aatc_calibrate(ctypes.byref(d), P(16), P(16), P(16), ctypes.byref(h), None) == aatc.ERR_UNSUPPORTED
    d = aatc.CalibDesc(128, 2, 3, 100, 2.75, 0, 0)
    assert L.aatc_calibrate(ctypes.byref(d), P(16), P(16), P(16), ctypes.byref(h), None) == aatc.ERR_INVALID_ARG
    for bits in (2.7, 0.0, 9.0, 2.6, 8.25):
        d = aatc.CalibDesc(128, 1, 4, 100, bits, 0, 0)
        assert L.aatc_calibrate(ctypes.byref(d), P(16), P(16), P(16), ctypes.byref(h), None) == aatc.ERR_UNSUPPORTED
    d = aatc.CalibDesc(128, 1, 4, 100, 2.75, 0, 0)
    assert L.aatc_calibrate(ctypes.byref(d), P(17), P(16), P(16), ctypes.byref(h), None) == aatc.ERR_INVALID_ARG
    assert "aligned" in aatc.last_error()
    assert L.aatc_encode(None, None, None, 1, 1, 0, 1, None, None, None) == aatc.ERR_INVALID_ARG
    assert L.aatc_decode_attention(None, None, None, None, 1, None, 1, 1, None, None, 0, None) == aatc.ERR_INVALID_ARG
    assert L.aatc_decode_workspace_size(None, 1, 1) == 0
    pg = aatc.Pages(None, 1, 32, 1)
    assert L.aatc_encode_paged(None, None, None, 1, 1, 0, None, None, None, ctypes.byref(pg), None) == \
        aatc.ERR_INVALID_ARG
    assert L.aatc_decode_attention_paged(None, None, None, None, ctypes.byref(pg), None, 1, 1, None, None, 0,
                                         None) == aatc.ERR_INVALID_ARG
    assert L.aatc_record_words(None) == -1
    L.aatc_free(None)
    assert L.aatc_check(None) == aatc.ERR_INVALID_ARG


def _blob_arrays(H=2, bits_sum=352):
    d = 128
    bits = np.zeros((H, d), dtype=np.int32)
    bits[:, : bits_sum // 4] = 4
    rng = np.random.default_rng(0)
    return dict(mu_k=np.zeros((H, d)), mu_v=np.zeros((H, d)),
                T_k=np.tile(np.eye(d), (H, 1, 1)), T_k_inv=np.tile(np.eye(d), (H, 1, 1)),
                A_k=np.tile(np.eye(d), (H, 1, 1)), T_v=np.tile(np.eye(d), (H, 1, 1)),
                U_v=np.tile(np.eye(d), (H, 1, 1)), lam_k=rng.random((H, d)), lam_v=rng.random((H, d)),
                lam_q=np.ones((H, d)), bits_k=bits, bits_v=bits.copy(),
                step_k=np.ones((H, d), np.float32), step_v=np.ones((H, d), np.float32))


def test_blob_roundtrip_and_import_validation(L):
    cal = _blob_arrays()
    blob = aatc.make_blob(cal, 8, torch.bfloat16)
    back = aatc.parse_blob(blob)
    for k, v in cal.items():
        assert np.array_equal(back[k], v), k
    assert back["W"] == 11 and back["G"] == 4
    h = ctypes.c_void_p()
    bad = bytearray(blob)
    bad[0] ^= 1
    assert L.aatc_import_calib(bytes(bad), len(bad), ctypes.byref(h)) == aatc.ERR_INVALID_ARG
    assert L.aatc_import_calib(blob, len(blob) - 4, ctypes.byref(h)) == aatc.ERR_INVALID_ARG
    cal2 = dict(cal)
    cal2["bits_v"] = cal["bits_v"].copy()
    cal2["bits_v"][1, 0] += 1            # no longer sums to the budget
    b2 = aatc.make_blob(cal2, 8, torch.bfloat16)
    assert L.aatc_import_calib(b2, len(b2), ctypes.byref(h)) == aatc.ERR_INVALID_ARG
    cal3 = dict(cal)
    cal3["bits_k"] = cal["bits_k"].copy()
    cal3["bits_k"][0, :3] = [9, 0, 3]    # width above 8, same total
    b3 = aatc.make_blob(cal3, 8, torch.bfloat16)
    assert L.aatc_import_calib(b3, len(b3), ctypes.byref(h)) == aatc.ERR_INVALID_ARG
    assert not h.value


def test_binding_refuses_cpu_tensors(L):
    with pytest.raises(ValueError):
        aatc._ptr(torch.zeros(4))
