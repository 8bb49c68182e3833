"""Thin ctypes binding of libaatc.so (C ABI in include/aatc.h).

Argument marshalling only: every computation runs in the CUDA library.  The
functions take torch CUDA tensors (for device memory and the current stream)
and pass raw pointers and sizes across the ABI.  If the library is missing
``lib()`` raises; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import struct
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libaatc.so")

(OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_NO_CONVERGENCE, ERR_NONFINITE, ERR_CAPACITY,
 ERR_TIMEOUT) = range(8)
STATUS_NAMES = ["OK", "INVALID_ARG", "UNSUPPORTED", "CUDA", "NO_CONVERGENCE", "NONFINITE", "CAPACITY", "TIMEOUT"]
TILE = 32      # cache tiles hold 32 tokens; L_cap is a multiple of this
F32, BF16 = 0, 1
D = 128
BLOB_MAGIC, BLOB_VERSION = 0x43544141, 2

EXPORTED = ["aatc_calibrate", "aatc_encode", "aatc_decode_attention", "aatc_decode_workspace_size",
            "aatc_encode_paged", "aatc_decode_attention_paged",
            "aatc_record_words", "aatc_record_words_kv", "aatc_export_calib", "aatc_import_calib", "aatc_check",
            "aatc_free", "aatc_last_error", "aatc_test_wait_fault", "aatc_append_decode_attention",
            "aatc_append_decode_workspace_size", "aatc_decode_launches", "aatc_set_fused_step"]


class AatcError(RuntimeError):
    def __init__(self, status: int, msg: str):
        self.status = status
        super().__init__("%s: %s" % (STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else status, msg))


class CalibDesc(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int), ("n_kv_heads", ctypes.c_int), ("n_q_heads", ctypes.c_int),
                ("n_calib_tokens", ctypes.c_int), ("bits_per_element", ctypes.c_double),
                ("dtype", ctypes.c_int), ("jacobi_max_sweeps", ctypes.c_int), ("joint_kv", ctypes.c_int)]


class Pages(ctypes.Structure):
    """aatc_pages: block table (device int32 [B][blocks_per_row]) of a paged pool."""
    _fields_ = [("block_table", ctypes.c_void_p), ("blocks_per_row", ctypes.c_int), ("block_tokens", ctypes.c_int),
                ("n_blocks", ctypes.c_int)]


_lib = None


def lib():
    """Load libaatc.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libaatc.so is not built; run `python -m quantized_attention_kv_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        sig = {
            "aatc_calibrate": (I, [ctypes.POINTER(CalibDesc), P, P, P, ctypes.POINTER(P), P]),
            "aatc_encode": (I, [P, P, P, I, I, I, I, P, P, P]),
            "aatc_decode_attention": (I, [P, P, P, P, I, P, I, I, P, P, S, P]),
            "aatc_decode_workspace_size": (S, [P, I, I]),
            "aatc_encode_paged": (I, [P, P, P, I, I, I, P, P, P, ctypes.POINTER(Pages), P]),
            "aatc_decode_attention_paged": (I, [P, P, P, P, ctypes.POINTER(Pages), P, I, I, P, P, S, P]),
            "aatc_record_words": (I, [P]),
            "aatc_record_words_kv": (I, [P, I]),
            "aatc_export_calib": (I, [P, P, ctypes.POINTER(S)]),
            "aatc_import_calib": (I, [P, S, ctypes.POINTER(P)]),
            "aatc_check": (I, [P]),
            "aatc_free": (None, [P]),
            "aatc_last_error": (ctypes.c_char_p, []),
            "aatc_test_wait_fault": (I, [I, I]),
            "aatc_append_decode_attention": (I, [P, P, P, I, P, P, P, I, I, I, P, P, S, P]),
            "aatc_append_decode_workspace_size": (S, [P, I, I, I]),
            "aatc_decode_launches": (I, [P]),
            "aatc_set_fused_step": (I, [I]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def last_error() -> str:
    return lib().aatc_last_error().decode()


def _check(st: int):
    if st != OK:
        raise AatcError(st, last_error())


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device: Optional[torch.device] = None):
    """The cudaStream_t of `stream`, or of the current stream of `device`."""
    if stream is None:
        if _raw_stream is not None and device is not None and device.index is not None:
            return _raw_stream(device.index)      # the current stream without building a Stream object
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to the library must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t.data_ptr()


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return F32
    if dt == torch.bfloat16:
        return BF16
    raise ValueError("inputs must be float32 or bfloat16")


class Calib:
    """Owning wrapper of an aatc_calib handle."""

    def __init__(self, handle: ctypes.c_void_p, dtype: torch.dtype, n_kv_heads: int, n_q_heads: int):
        self.handle = handle
        self.dtype = dtype
        self.n_kv_heads = n_kv_heads
        self.n_q_heads = n_q_heads
        # record widths never change for a handle
        self._wk = lib().aatc_record_words_kv(handle, 0)
        self._wv = lib().aatc_record_words_kv(handle, 1)

    @property
    def W(self) -> int:
        """Record words of keys and values when they are the same (else an error)."""
        if self._wk != self._wv:
            raise ValueError("keys and values have different record widths: use W_k / W_v")
        return self._wk

    @property
    def W_k(self) -> int:
        return self._wk

    @property
    def W_v(self) -> int:
        return self._wv

    def words(self, tensor: str) -> int:
        """Record words of 'k' or 'v'."""
        return self.W_k if tensor == "k" else self.W_v

    def free(self):
        if self.handle:
            lib().aatc_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass

    def check(self):
        _check(lib().aatc_check(self.handle))

    def decode_launches(self) -> int:
        """Kernels one decode_attention call launches (1: fast path, 3: general path)."""
        return int(lib().aatc_decode_launches(self.handle))

    def export(self) -> dict:
        """The calibration as numpy arrays (via aatc_export_calib)."""
        n = ctypes.c_size_t(0)
        _check(lib().aatc_export_calib(self.handle, None, ctypes.byref(n)))
        buf = ctypes.create_string_buffer(n.value)
        _check(lib().aatc_export_calib(self.handle, buf, ctypes.byref(n)))
        return parse_blob(buf.raw[:n.value])


def calibrate(k_cal: torch.Tensor, v_cal: torch.Tensor, q_cal: torch.Tensor, bits_per_element: float,
              jacobi_max_sweeps: int = 0, joint: bool = False, stream=None) -> Calib:
    """aatc_calibrate: k_cal, v_cal [H_kv][N][128], q_cal [H_q][N][128] on the GPU.
    joint: split the pair budget between keys and values by the attention-aware
    token weights (then W_k and W_v may differ)."""
    Hkv, N, d = k_cal.shape
    desc = CalibDesc(d, Hkv, q_cal.shape[0], N, float(bits_per_element), _dtype_code(k_cal.dtype),
                     int(jacobi_max_sweeps), 1 if joint else 0)
    h = ctypes.c_void_p()
    _check(lib().aatc_calibrate(ctypes.byref(desc), _ptr(k_cal), _ptr(v_cal), _ptr(q_cal),
                                ctypes.byref(h), _stream(stream, k_cal.device)))
    return Calib(h, k_cal.dtype, Hkv, q_cal.shape[0])


def make_blob(cal: dict, n_q_heads: int, dtype: torch.dtype) -> bytes:
    """Serialize calibration arrays into the aatc_import_calib blob format."""
    H = np.asarray(cal["mu_k"]).shape[0]
    Bk = int(np.asarray(cal["bits_k"])[0].sum())
    Bv = int(np.asarray(cal["bits_v"])[0].sum())
    hdr = struct.pack("<8i", BLOB_MAGIC, BLOB_VERSION, D, H, n_q_heads, Bk, _dtype_code(dtype), Bv)
    parts = [hdr]
    for key in ("mu_k", "mu_v", "T_k", "T_k_inv", "A_k", "T_v", "U_v", "lam_k", "lam_v", "lam_q"):
        parts.append(np.ascontiguousarray(cal[key], dtype="<f8").tobytes())
    for key in ("bits_k", "bits_v"):
        parts.append(np.ascontiguousarray(cal[key], dtype="<i4").tobytes())
    for key in ("step_k", "step_v"):
        parts.append(np.ascontiguousarray(cal[key], dtype="<f4").tobytes())
    return b"".join(parts)


def parse_blob(blob: bytes) -> dict:
    hdr = struct.unpack_from("<8i", blob, 0)
    if hdr[0] != BLOB_MAGIC or hdr[1] not in (1, BLOB_VERSION):
        raise ValueError("not a calibration blob")
    H = hdr[3]
    Bk, Bv = hdr[5], (hdr[5] if hdr[1] == 1 else hdr[7])
    off = 32
    out = {"n_q_heads": hdr[4], "B_bits": Bk, "B_k": Bk, "B_v": Bv, "dtype": hdr[6],
           "W_k": Bk // 32, "W_v": Bv // 32, "W": Bk // 32 if Bk == Bv else None, "G": hdr[4] // H}

    def take(key, dt, shape):
        nonlocal off
        n = int(np.prod(shape))
        out[key] = np.frombuffer(blob, dtype=dt, count=n, offset=off).reshape(shape).copy()
        off += n * np.dtype(dt).itemsize

    for key in ("mu_k", "mu_v"):
        take(key, "<f8", (H, D))
    for key in ("T_k", "T_k_inv", "A_k", "T_v", "U_v"):
        take(key, "<f8", (H, D, D))
    for key in ("lam_k", "lam_v", "lam_q"):
        take(key, "<f8", (H, D))
    for key in ("bits_k", "bits_v"):
        take(key, "<i4", (H, D))
    for key in ("step_k", "step_v"):
        take(key, "<f4", (H, D))
    return out


def import_calib(cal: dict, n_q_heads: int, dtype: torch.dtype) -> Calib:
    """aatc_import_calib from a dict of arrays (e.g. another calibration's export)."""
    blob = make_blob(cal, n_q_heads, dtype)
    h = ctypes.c_void_p()
    _check(lib().aatc_import_calib(blob, len(blob), ctypes.byref(h)))
    return Calib(h, dtype, np.asarray(cal["mu_k"]).shape[0], n_q_heads)


def cache_capacity(L: int) -> int:
    """Smallest valid L_cap (a multiple of 32) holding L tokens."""
    return max(TILE, -(-int(L) // TILE) * TILE)


def alloc_cache(calib: Calib, B: int, L: int, device="cuda", tensor: Optional[str] = None) -> torch.Tensor:
    """A zeroed packed cache for B rows of up to L tokens: int32 [B][H_kv][L_cap][W]
    words with L_cap = cache_capacity(L), in the tiled layout of aatc_encode
    (the [L_cap][W] axes are the slab's size, not one record per row).
    tensor: 'k' or 'v' for that tensor's record width; None when both are the same."""
    W = calib.W if tensor is None else calib.words(tensor)
    return torch.zeros(B, calib.n_kv_heads, cache_capacity(L), W, dtype=torch.int32, device=device)


def _check_cache(calib: Calib, B: int, kc: torch.Tensor, vc: torch.Tensor) -> int:
    """Caches must be [B][H_kv][L_cap][W_k] and [B][H_kv][L_cap][W_v] (the tiled
    slabs of aatc_encode); returns L_cap."""
    for c, W in ((kc, calib._wk), (vc, calib._wv)):
        if c.dim() != 4 or tuple(c.shape[:2]) != (B, calib.n_kv_heads) or c.shape[3] != W or \
                c.shape[2] % TILE or c.element_size() != 4:
            raise ValueError("packed caches must be 4-byte [B=%d][H_kv=%d][L_cap (multiple of %d)][W=%d], got %s"
                             % (B, calib.n_kv_heads, TILE, W, tuple(c.shape)))
    if kc.shape[2] != vc.shape[2]:
        raise ValueError("key and value caches must have the same L_cap")
    return kc.shape[2]


def encode(calib: Calib, k: torch.Tensor, v: torch.Tensor, k_packed: torch.Tensor, v_packed: torch.Tensor,
           start_pos: int = 0, stream=None):
    """aatc_encode: k, v [B][H_kv][L_new][128] into tokens start_pos.. of the packed caches."""
    B, H, L_new, _ = k.shape
    _check_cache(calib, B, k_packed, v_packed)
    _check(lib().aatc_encode(calib.handle, _ptr(k), _ptr(v), B, L_new, int(start_pos), k_packed.shape[2],
                             _ptr(k_packed), _ptr(v_packed), _stream(stream, k.device)))


def workspace_size(calib: Calib, B: int, L: int) -> int:
    return int(lib().aatc_decode_workspace_size(calib.handle, B, L))


def new_workspace(calib: Calib, B: int, L: int, device="cuda") -> torch.Tensor:
    """A decode workspace for B rows of up to L tokens, zeroed as the library
    requires before its first use (later calls leave it ready)."""
    return torch.zeros(max(workspace_size(calib, B, L), 16), dtype=torch.uint8, device=device)


def decode_attention(calib: Calib, q: torch.Tensor, k_packed: torch.Tensor, v_packed: torch.Tensor, L: int,
                     seq_lens: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """aatc_decode_attention: q [B][H_q][128] -> fp32 [B][H_q][128]."""
    B = q.shape[0]
    _check_cache(calib, B, k_packed, v_packed)
    if out is None:
        out = torch.empty(B, calib.n_q_heads, D, dtype=torch.float32, device=q.device)
    if workspace is None:   # (a given workspace is checked against the need by the library)
        workspace = new_workspace(calib, B, L, q.device)
    _check(lib().aatc_decode_attention(calib.handle, _ptr(q), _ptr(k_packed), _ptr(v_packed), k_packed.shape[2],
                                       _ptr(seq_lens), int(L), B, _ptr(out), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream, q.device)))
    return out


def set_fused_step(mode: int):
    """aatc_set_fused_step: 0 never fuse the serving step, 1 when it pays (default), 2 whenever it fits."""
    _check(lib().aatc_set_fused_step(int(mode)))


def append_workspace_size(calib: Calib, B: int, L_old: int, n_new: int) -> int:
    return int(lib().aatc_append_decode_workspace_size(calib.handle, B, L_old, n_new))


def new_append_workspace(calib: Calib, B: int, L_old: int, n_new: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace for append_decode_attention (it may also serve decode_attention)."""
    n = max(append_workspace_size(calib, B, L_old, n_new), workspace_size(calib, B, L_old + n_new), 16)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def append_decode_attention(calib: Calib, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor,
                            k_packed: torch.Tensor, v_packed: torch.Tensor, L_old: int,
                            out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    """aatc_append_decode_attention: one decode step in one launch -- the
    n_new tokens k_new, v_new [B][H_kv][n_new][128] are encoded into positions
    L_old.. of the caches and q [B][H_q][128] attends all L_old + n_new tokens."""
    B, H, n_new, _ = k_new.shape
    _check_cache(calib, B, k_packed, v_packed)
    if out is None:
        out = torch.empty(B, calib.n_q_heads, D, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = new_append_workspace(calib, B, L_old, n_new, q.device)
    _check(lib().aatc_append_decode_attention(calib.handle, _ptr(k_new), _ptr(v_new), n_new, _ptr(q),
                                              _ptr(k_packed), _ptr(v_packed), k_packed.shape[2], int(L_old), B,
                                              _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                              _stream(stream, q.device)))
    return out


# ----------------------------------------------------------------- paged cache
def alloc_pool(calib: Calib, n_blocks: int, block_tokens: int, device="cuda",
               tensor: Optional[str] = None) -> torch.Tensor:
    """A zeroed pool of n_blocks blocks of block_tokens tokens (32 times a power of two):
    int32 [n_blocks][H_kv][block_tokens][W]; head h of block p is tiled like a
    contiguous cache with L_cap = block_tokens.  tensor: 'k' or 'v' for that
    tensor's record width; None when both are the same."""
    tpb = block_tokens // TILE
    if block_tokens <= 0 or block_tokens % TILE or tpb & (tpb - 1):
        raise ValueError("block_tokens must be %d times a power of two" % TILE)
    W = calib.W if tensor is None else calib.words(tensor)
    return torch.zeros(n_blocks, calib.n_kv_heads, block_tokens, W, dtype=torch.int32, device=device)


def _pages(calib: Calib, block_table: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor) -> Pages:
    if block_table.dim() != 2 or block_table.dtype != torch.int32:
        raise ValueError("block_table must be int32 [B][blocks_per_row]")
    for p, W in ((k_pool, calib.W_k), (v_pool, calib.W_v)):
        if p.dim() != 4 or p.shape[1] != calib.n_kv_heads or p.shape[3] != W or p.element_size() != 4:
            raise ValueError("pools must be 4-byte [n_blocks][H_kv=%d][block_tokens][W=%d], got %s"
                             % (calib.n_kv_heads, W, tuple(p.shape)))
    if k_pool.shape[:3] != v_pool.shape[:3]:
        raise ValueError("key and value pools must have the same blocks")
    bt = _ptr(block_table)
    return Pages(bt, block_table.shape[1], k_pool.shape[2], k_pool.shape[0])


def encode_paged(calib: Calib, k: torch.Tensor, v: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                 block_table: torch.Tensor, start_pos: int = 0, row_start: Optional[torch.Tensor] = None,
                 stream=None):
    """aatc_encode_paged: token n of row b to logical position row_start[b] + n
    (or start_pos + n) of row b's blocks."""
    B, H, L_new, _ = k.shape
    if block_table.shape[0] != B:
        raise ValueError("block_table must have one row per batch row")
    if row_start is not None and (row_start.dtype != torch.int32 or row_start.numel() < B):
        raise ValueError("row_start must be int32 with one entry per batch row")
    pg = _pages(calib, block_table, k_pool, v_pool)
    _check(lib().aatc_encode_paged(calib.handle, _ptr(k), _ptr(v), B, L_new, int(start_pos), _ptr(row_start),
                                   _ptr(k_pool), _ptr(v_pool), ctypes.byref(pg), _stream(stream, k.device)))


def decode_attention_paged(calib: Calib, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                           block_table: torch.Tensor, L: int, seq_lens: Optional[torch.Tensor] = None,
                           out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                           stream=None) -> torch.Tensor:
    """aatc_decode_attention_paged: q [B][H_q][128] -> fp32 [B][H_q][128]."""
    B = q.shape[0]
    if block_table.shape[0] != B:
        raise ValueError("block_table must have one row per batch row")
    pg = _pages(calib, block_table, k_pool, v_pool)
    if out is None:
        out = torch.empty(B, calib.n_q_heads, D, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = new_workspace(calib, B, L, q.device)
    _check(lib().aatc_decode_attention_paged(calib.handle, _ptr(q), _ptr(k_pool), _ptr(v_pool), ctypes.byref(pg),
                                             _ptr(seq_lens), int(L), B, _ptr(out), _ptr(workspace),
                                             workspace.numel() * workspace.element_size(), _stream(stream, q.device)))
    return out


def test_wait_fault(skip_tile_copy: bool, wait_tries: int = 0):
    """aatc_test_wait_fault (testing hook): while set, fast-path decode calls
    leave one tile copy unissued so that a bounded wait gives up and the
    handle reports TIMEOUT; (False, 0) restores normal operation."""
    _check(lib().aatc_test_wait_fault(1 if skip_tile_copy else 0, int(wait_tries)))
