"""Compressed sparse attention (c4a / c128a) for GB300: Python binding of libcsa.

A thin ctypes layer over the C ABI declared in include/csa.h.  It only
marshals arguments: torch tensors become device pointers, the current torch
stream becomes the launch stream.  Every step of the path runs in the CUDA
kernels of libcsa.so; there is no Python or CPU fallback, and every call
raises if the compiled library is missing.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa.so")

F32, BF16, E4M3, E2M1, E4M3R = 0, 1, 2, 3, 4
DTYPES = {"f32": F32, "bf16": BF16, "e4m3": E4M3, "e2m1": E2M1, "e4m3r": E4M3R}

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE_BOUNDS, ERR_WORKSPACE, ERR_TIMEOUT = 0, -1, -2, -3, -4, -5, -6


class CsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class Paged(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("rows_per_block", ctypes.c_int32), ("dim", ctypes.c_int32),
                ("tail_bf16", ctypes.c_int32)]


class BlockTableC(ctypes.Structure):
    _fields_ = [("table", ctypes.c_void_p), ("num_seqs", ctypes.c_int32), ("stride", ctypes.c_int32)]


class QueryNormC(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("q_dtype", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("gamma", ctypes.c_void_p), ("q_out", ctypes.c_void_p), ("out_dtype", ctypes.c_int32)]


class Layer(ctypes.Structure):
    _fields_ = [("ratio", ctypes.c_int32), ("window", ctypes.c_int32), ("dim", ctypes.c_int32),
                ("rope_dim", ctypes.c_int32), ("heads", ctypes.c_int32), ("swa", ctypes.c_int32),
                ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float), ("scale", ctypes.c_float)]


_lib = None

_VP, _I32, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
_PP, _PB, _PL = ctypes.POINTER(Paged), ctypes.POINTER(BlockTableC), ctypes.POINTER(Layer)
_PQ = ctypes.POINTER(QueryNormC)

_SIGS = {
    "csa_compress_insert": (_I32, [_PL, _VP, _VP, _I32, _I32, _VP, _VP, _VP, _VP, _VP, _PP, _PB, _PP, _PB, _PP,
                                   _PB, _VP, _VP]),
    "csa_compress_insert_qnorm": (_I32, [_PL, _VP, _VP, _I32, _I32, _VP, _VP, _VP, _VP, _VP, _PP, _PB, _PP, _PB,
                                         _PP, _PB, _PQ, _VP, _VP]),
    "csa_cache_store": (_I32, [_VP, _I32, _VP, _VP, _PP, _PB, _VP, _VP]),
    "csa_indexer_topk": (_I32, [_VP, _I32, _VP, _I32, _I32, _I32, _VP, _VP, _I32, _I32, _PP, _PB, _I32, _I32, _VP,
                                _VP, _SZ, _VP, _VP]),
    "csa_indexer_topk_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "csa_sparse_attn_decode": (_I32, [_PL, _VP, _I32, _I32, _VP, _VP, _PP, _PB, _VP, _I32, _I32, _PP, _PB, _VP, _I32,
                                      _VP, _VP, _SZ, _VP, _VP]),
    "csa_sparse_attn_prefill": (_I32, [_PL, _VP, _I32, _I32, _VP, _VP, _PP, _PB, _VP, _I32, _I32, _PP, _PB, _VP,
                                       _I32, _VP, _VP, _SZ, _VP, _VP]),
    "csa_sparse_attn_workspace_size": (_SZ, [_PL, _I32, _I32]),
    "csa_indexer_topk_noalloc": (_I32, [_VP, _I32, _VP, _I32, _I32, _I32, _VP, _VP, _I32, _I32, _PP, _PB, _I32,
                                        _I32, _VP, _VP, _VP]),
    "csa_read_status": (_I32, [_VP, _I32, _VP]),
    "csa_status_string": (ctypes.c_char_p, [_I32]),
    "csa_version": (_I32, []),
    "csa_launch_count": (ctypes.c_uint64, []),
}

EXPORTED = tuple(_SIGS)


def lib():
    """The loaded libcsa.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libcsa.so is not built ({LIB_PATH}); run "
                               "`python -m compressed_sparse_long_c128a_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().csa_status_string(int(status)).decode()


def version() -> int:
    return int(lib().csa_version())


def launch_count() -> int:
    """Kernel launches the library has enqueued in this process (host-side count)."""
    return int(lib().csa_launch_count())


def _check(status: int, what: str):
    if status != OK:
        raise CsaError(status, what)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on the CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _tdtype(t) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise ValueError(f"unsupported input dtype {t.dtype}")


@dataclass
class PagedCache:
    """A paged cache in device memory: `data` [num_blocks, rows_per_block, row] and,
    for quantised dtypes, `scales` (E4M3, E4M3R: float [num_blocks, rows_per_block];
    E2M1: uint8 [num_blocks, rows_per_block, dim/16]).  An E4M3R row is
    dim - tail_bf16 code bytes followed by tail_bf16 bf16 values."""

    data: torch.Tensor
    scales: torch.Tensor | None
    dtype: int
    rows_per_block: int
    dim: int
    tail_bf16: int = 0

    @staticmethod
    def empty(num_blocks: int, rows_per_block: int, dim: int, dtype: int, device="cuda",
              tail_bf16: int = 0) -> "PagedCache":
        shape = (num_blocks, rows_per_block)
        scales = None
        if dtype == F32:
            data = torch.zeros(*shape, dim, dtype=torch.float32, device=device)
        elif dtype == BF16:
            data = torch.zeros(*shape, dim, dtype=torch.bfloat16, device=device)
        elif dtype == E4M3:
            data = torch.zeros(*shape, dim, dtype=torch.uint8, device=device)
            scales = torch.zeros(*shape, dtype=torch.float32, device=device)
        elif dtype == E2M1:
            data = torch.zeros(*shape, dim // 2, dtype=torch.uint8, device=device)
            scales = torch.zeros(*shape, dim // 16, dtype=torch.uint8, device=device)
        elif dtype == E4M3R:
            data = torch.zeros(*shape, dim + tail_bf16, dtype=torch.uint8, device=device)
            scales = torch.zeros(*shape, dtype=torch.float32, device=device)
        else:
            raise ValueError(dtype)
        return PagedCache(data, scales, dtype, rows_per_block, dim, tail_bf16 if dtype == E4M3R else 0)

    @property
    def num_blocks(self) -> int:
        return self.data.shape[0]

    def c(self) -> Paged:
        return Paged(_ptr(self.data), _ptr(self.scales), self.dtype, self.num_blocks, self.rows_per_block, self.dim,
                     self.tail_bf16)


def block_table(t: torch.Tensor) -> BlockTableC:
    """C view of an int32 [num_seqs, stride] device block table."""
    if t.dtype != torch.int32 or t.dim() != 2:
        raise ValueError("block table must be int32 [num_seqs, stride]")
    return BlockTableC(_ptr(t), t.shape[0], t.shape[1])


def make_layer(ratio, window, dim, rope_dim, heads, swa=128, rope_theta=10000.0, rms_eps=1e-6, scale=None) -> Layer:
    return Layer(ratio, window, dim, rope_dim, heads, swa, rope_theta, rms_eps,
                 dim ** -0.5 if scale is None else scale)


# ------------------------------------------------------------------ entry points


def compress_insert(layer: Layer, kv, gate, seq_id, pos, bias, gamma_c, gamma_swa, state: PagedCache, state_bt,
                    swa: PagedCache | None, swa_bt, comp: PagedCache, comp_bt, err, stream=None):
    """swa=None (swa_bt and gamma_swa then ignored) writes no sliding-window rows:
    the indexer-key compressor, whose keys go to an indexer cache (comp may be E2M1)."""
    no_swa = swa is None
    st = lib().csa_compress_insert(ctypes.byref(layer), _ptr(kv), _ptr(gate), _tdtype(kv), kv.shape[0],
                                   _ptr(seq_id), _ptr(pos), _ptr(bias), _ptr(gamma_c),
                                   None if no_swa else _ptr(gamma_swa),
                                   ctypes.byref(state.c()), ctypes.byref(block_table(state_bt)),
                                   None if no_swa else ctypes.byref(swa.c()),
                                   None if no_swa else ctypes.byref(block_table(swa_bt)),
                                   ctypes.byref(comp.c()), ctypes.byref(block_table(comp_bt)), _ptr(err),
                                   _stream(stream))
    _check(st, "csa_compress_insert")


def compress_insert_qnorm(layer: Layer, kv, gate, seq_id, pos, bias, gamma_c, gamma_swa, state: PagedCache,
                          state_bt, swa: PagedCache | None, swa_bt, comp: PagedCache, comp_bt, q, gamma_q, q_out,
                          err, stream=None):
    """compress_insert plus q_out[j, h] := RMSNorm(q[j, h]; gamma_q) in the same launch.
    q, q_out: [n_tok, heads, D] (f32 or bf16; q_out may be q itself)."""
    if q.dim() != 3 or q_out.shape != q.shape or q.shape[0] != kv.shape[0]:
        raise ValueError("q and q_out must be [n_tok, heads, D] with n_tok rows of kv")
    qn = QueryNormC(_ptr(q), _tdtype(q), q.shape[1], _ptr(gamma_q), _ptr(q_out), _tdtype(q_out))
    no_swa = swa is None
    st = lib().csa_compress_insert_qnorm(ctypes.byref(layer), _ptr(kv), _ptr(gate), _tdtype(kv), kv.shape[0],
                                         _ptr(seq_id), _ptr(pos), _ptr(bias), _ptr(gamma_c),
                                         None if no_swa else _ptr(gamma_swa),
                                         ctypes.byref(state.c()), ctypes.byref(block_table(state_bt)),
                                         None if no_swa else ctypes.byref(swa.c()),
                                         None if no_swa else ctypes.byref(block_table(swa_bt)),
                                         ctypes.byref(comp.c()), ctypes.byref(block_table(comp_bt)),
                                         ctypes.byref(qn), _ptr(err), _stream(stream))
    _check(st, "csa_compress_insert_qnorm")


def cache_store(rows, seq_id, row_idx, cache: PagedCache, bt, err, stream=None):
    if rows.dtype != torch.float32:
        raise ValueError("rows must be float32")
    st = lib().csa_cache_store(_ptr(rows), rows.shape[0], _ptr(seq_id), _ptr(row_idx), ctypes.byref(cache.c()),
                               ctypes.byref(block_table(bt)), _ptr(err), _stream(stream))
    _check(st, "csa_cache_store")


def indexer_topk_workspace_size(n_rows: int, max_n: int, k: int) -> int:
    return int(lib().csa_indexer_topk_workspace_size(n_rows, max_n, k))


def indexer_topk(q_idx, w, seq_id, pos, ratio: int, window: int, idx_cache: PagedCache, bt, k: int, max_n: int,
                 out_idx, ws, err, stream=None):
    n_rows, heads, dim = q_idx.shape
    st = lib().csa_indexer_topk(_ptr(q_idx), _tdtype(q_idx), _ptr(w), n_rows, heads, dim, _ptr(seq_id), _ptr(pos),
                                ratio, window, ctypes.byref(idx_cache.c()), ctypes.byref(block_table(bt)), k, max_n,
                                _ptr(out_idx), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                _ptr(err), _stream(stream))
    _check(st, "csa_indexer_topk")


def indexer_topk_noalloc(q_idx, w, seq_id, pos, ratio: int, window: int, idx_cache: PagedCache, bt, k: int,
                         max_n: int, out_idx, err, stream=None):
    """indexer_topk without a workspace, for callers that cannot allocate device
    memory: its scratch is a fixed 16 MiB array inside the library, shared by
    every call (calls that may overlap on the GPU race; the first call on a
    device should come before any stream capture)."""
    n_rows, heads, dim = q_idx.shape
    st = lib().csa_indexer_topk_noalloc(_ptr(q_idx), _tdtype(q_idx), _ptr(w), n_rows, heads, dim, _ptr(seq_id),
                                        _ptr(pos), ratio, window, ctypes.byref(idx_cache.c()),
                                        ctypes.byref(block_table(bt)), k, max_n, _ptr(out_idx), _ptr(err),
                                        _stream(stream))
    _check(st, "csa_indexer_topk_noalloc")


def sparse_attn_workspace_size(layer: Layer, n_rows: int, k_or_max_n: int) -> int:
    return int(lib().csa_sparse_attn_workspace_size(ctypes.byref(layer), n_rows, k_or_max_n))


def _attn(name, layer, q, seq_id, pos, comp, comp_bt, topk, k, max_n, swa, swa_bt, out, out_dtype, out_scales, ws,
          err, stream):
    fn = getattr(lib(), name)
    st = fn(ctypes.byref(layer), _ptr(q), _tdtype(q), q.shape[0], _ptr(seq_id), _ptr(pos), ctypes.byref(comp.c()),
            ctypes.byref(block_table(comp_bt)), _ptr(topk), k, max_n, ctypes.byref(swa.c()),
            ctypes.byref(block_table(swa_bt)), _ptr(out), out_dtype, _ptr(out_scales), _ptr(ws),
            0 if ws is None else ws.numel() * ws.element_size(), _ptr(err), _stream(stream))
    _check(st, name)


def sparse_attn_decode(layer: Layer, q, seq_id, pos, comp: PagedCache, comp_bt, topk, k: int, max_n: int,
                       swa: PagedCache, swa_bt, out, out_dtype: int, out_scales, ws, err, stream=None):
    _attn("csa_sparse_attn_decode", layer, q, seq_id, pos, comp, comp_bt, topk, k, max_n, swa, swa_bt, out,
          out_dtype, out_scales, ws, err, stream)


def sparse_attn_prefill(layer: Layer, q, seq_id, pos, comp: PagedCache, comp_bt, topk, k: int, max_n: int,
                        swa: PagedCache, swa_bt, out, out_dtype: int, out_scales, ws, err, stream=None):
    _attn("csa_sparse_attn_prefill", layer, q, seq_id, pos, comp, comp_bt, topk, k, max_n, swa, swa_bt, out,
          out_dtype, out_scales, ws, err, stream)


def read_status(err, reset: bool = True, stream=None) -> int:
    return int(lib().csa_read_status(_ptr(err), 1 if reset else 0, _stream(stream)))
