"""Block-sparse FP8 attention prefill over a paged KV cache on GB300 (sm_103a).

A thin ctypes binding over the C ABI in include/bsa_fp8.h: it marshals PyTorch CUDA tensors
(device pointers) and the current stream into ``bsa_fp8_prefill`` / ``bsa_fp8_compact_tiles``
and the quantise step ``bsa_fp8_quantize_rows`` / ``bsa_fp8_append_kv``; ``prefill_host``
marshals CPU tensors into ``bsa_fp8_prefill_host``, which copies them in and the results out.
Every step of the computation runs in the library's CUDA kernels; there is no CPU path.
The library must have been built (``block_sparse_fp8_gb300._build.build()``); importing the
binding on a machine without it raises immediately.
"""
from __future__ import annotations

import ctypes
import math
import os

from . import _build

__all__ = ["Dims", "AppendDims", "Tensors", "TENSOR_NAMES", "Q_TND", "Q_NTD", "KV_HND",
           "KV_NHD", "prefill", "prefill_host", "compact_tiles", "quantize_rows", "append_kv",
           "workspace_size", "status_string", "set_wait_limit_ns", "lib",
           "SCALE_PER_TENSOR", "SCALE_PER_TOKEN_HEAD", "SCALE_PER_HEAD", "BsaError",
           "DESCALE_AMAX", "DESCALE_UE8M0",
           "DEV_BAD_INDEX", "DEV_BAD_PAGE", "DEV_BAD_SEQLEN", "DEV_TIMEOUT"]

SCALE_PER_TENSOR = 0
SCALE_PER_TOKEN_HEAD = 1
SCALE_PER_HEAD = 2

DEV_BAD_INDEX = 1
DEV_BAD_PAGE = 2
DEV_BAD_SEQLEN = 4
DEV_TIMEOUT = 8

EXPORTED = ("bsa_fp8_prefill", "bsa_fp8_prefill_workspace_size", "bsa_fp8_compact_tiles",
            "bsa_fp8_prefill_noalloc", "bsa_fp8_prefill_host", "bsa_fp8_quantize_rows",
            "bsa_fp8_quantize_rows_ue8m0", "bsa_fp8_append_kv", "bsa_fp8_set_wait_limit_ns",
            "bsa_status_string")

# descale rules of the quantise step
DESCALE_AMAX = 0    # amax / 448
DESCALE_UE8M0 = 1   # amax / 448 rounded up to a power of two


class BsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "B", "N1", "N2", "D", "page_size", "max_q_len", "max_kv_len", "num_pages",
        "max_pages_per_seq", "total_q", "k_scale_kind", "v_scale_kind", "causal", "q_layout",
        "kv_layout", "tiles_per_step")]


# the tensors of one call, in bsa_fp8_tensors_t's order (prefill's argument names; out, lse)
TENSOR_NAMES = ("q", "k_pages", "v_pages", "q_descale", "k_descale", "v_descale",
                "cu_seqlens_q", "seqused_kv", "block_table", "block_mask", "sparse_indices",
                "sparse_seq_len", "out", "lse")


class Tensors(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in TENSOR_NAMES]


Q_TND, Q_NTD = 0, 1
KV_HND, KV_NHD = 0, 1


class AppendDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "B", "N2", "D", "page_size", "num_pages", "max_pages_per_seq", "total_new",
        "k_scale_kind", "v_scale_kind", "kv_layout", "k_descale_rule")]


_lib = None


def lib():
    """The loaded libbsa_fp8.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise ImportError(
                f"{_build.LIB} is missing: build it with block_sparse_fp8_gb300._build.build()")
        L = ctypes.CDLL(_build.LIB)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.bsa_fp8_prefill.restype = i32
        L.bsa_fp8_prefill.argtypes = [ctypes.POINTER(Dims)] + [vp] * 12 + [f32, f32, vp, vp, vp,
                                                                           sz, vp, vp]
        L.bsa_fp8_prefill_workspace_size.restype = sz
        L.bsa_fp8_prefill_workspace_size.argtypes = [ctypes.POINTER(Dims)]
        L.bsa_fp8_prefill_noalloc.restype = i32
        L.bsa_fp8_prefill_noalloc.argtypes = [ctypes.POINTER(Dims)] + [vp] * 12 + [f32, f32, vp,
                                                                                  vp, vp, vp]
        L.bsa_fp8_prefill_host.restype = i32
        L.bsa_fp8_prefill_host.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(Tensors),
                                           ctypes.POINTER(Tensors), f32, f32, vp, sz, vp, vp]
        L.bsa_fp8_compact_tiles.restype = i32
        L.bsa_fp8_compact_tiles.argtypes = [ctypes.POINTER(Dims)] + [vp] * 9
        L.bsa_fp8_quantize_rows.restype = i32
        L.bsa_fp8_quantize_rows.argtypes = [vp, ctypes.c_longlong, vp, vp, vp]
        L.bsa_fp8_quantize_rows_ue8m0.restype = i32
        L.bsa_fp8_quantize_rows_ue8m0.argtypes = [vp, ctypes.c_longlong, vp, vp, vp]
        L.bsa_fp8_append_kv.restype = i32
        L.bsa_fp8_append_kv.argtypes = [ctypes.POINTER(AppendDims)] + [vp] * 12
        L.bsa_fp8_set_wait_limit_ns.restype = i32
        L.bsa_fp8_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
        L.bsa_status_string.restype = ctypes.c_char_p
        L.bsa_status_string.argtypes = [i32]
        _lib = L
    return _lib


def set_wait_limit_ns(ns: int) -> None:
    """Limit of every bounded wait inside the prefill kernel for later launches (0: the
    default, 2 s).  A wait that runs out sets DEV_TIMEOUT in the device status word."""
    lib().bsa_fp8_set_wait_limit_ns(int(ns))


def status_string(status: int) -> str:
    return lib().bsa_status_string(status).decode()


def _p(t):
    return None if t is None else t.data_ptr()


def _stream_handle(stream):
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def make_dims(q, k_pages, block_table, cu_seqlens_q, max_q_len, max_kv_len, k_scale_kind,
              v_scale_kind, causal=True, q_layout=Q_TND, kv_layout=KV_HND,
              tiles_per_step=1) -> Dims:
    if q_layout == Q_NTD:
        N1, T, D = q.shape
    else:
        T, N1, D = q.shape
    if kv_layout == KV_NHD:
        P, ps, N2, D2 = k_pages.shape
    else:
        P, N2, ps, D2 = k_pages.shape
    return Dims(B=cu_seqlens_q.shape[0] - 1, N1=N1, N2=N2, D=D, page_size=ps,
                max_q_len=int(max_q_len), max_kv_len=int(max_kv_len), num_pages=P,
                max_pages_per_seq=block_table.shape[1], total_q=T,
                k_scale_kind=int(k_scale_kind), v_scale_kind=int(v_scale_kind),
                causal=int(bool(causal)), q_layout=int(q_layout), kv_layout=int(kv_layout),
                tiles_per_step=int(tiles_per_step))


def workspace_size(dims: Dims) -> int:
    return int(lib().bsa_fp8_prefill_workspace_size(ctypes.byref(dims)))


def prefill(q, k_pages, v_pages, q_descale, k_descale, v_descale, cu_seqlens_q, seqused_kv,
            block_table, max_q_len: int, max_kv_len: int, block_mask=None, sparse_indices=None,
            sparse_seq_len=None, softmax_scale: float | None = None, p_scale: float = 256.0,
            causal: bool = True, out=None, lse=None, return_lse: bool = True, dev_status=None,
            workspace=None, stream=None, k_scale_kind: int | None = None,
            v_scale_kind: int | None = None, q_layout: int = Q_TND, kv_layout: int = KV_HND,
            tiles_per_step: int = 1):
    """Block-sparse FP8 prefill.  Tensors are CUDA tensors in the C ABI's layouts:
    q uint8/float8_e4m3fn [T, N1, 128] (q_layout Q_TND) or [N1, T, 128] (Q_NTD, with q_descale
    [N1, T]); k_pages, v_pages [P, N2, page, 128] (KV_HND) or [P, page, N2, 128] (KV_NHD);
    q_descale f32 [T, N1]; k_descale f32 [1] or [P, N2, page]; v_descale f32 [1] or [N2];
    cu_seqlens_q i32
    [B+1]; seqused_kv i32 [B] or None; block_table i32 [B, L]; block_mask u8 [B, N1, Qb, Kb]
    or sparse_indices i32 [B, N1, Qb, Kb] + sparse_seq_len i32 [B, N1, Qb].
    max_q_len / max_kv_len are host integers (upper bounds of the per-sequence lengths).
    The scale kinds default to what the descale shapes imply (K [P, N2, page] = per token and
    head; V [N2] = per head, which for N2 = 1 is the same as per tensor).
    tiles_per_step = 2 runs the online softmax over 256-wide macro blocks (two list tiles
    per step).  Returns (out bf16 [T, N1, 128], lse f32 [N1, T] or None)."""
    import torch

    n2 = k_pages.shape[2] if kv_layout == KV_NHD else k_pages.shape[1]
    k_kind = k_scale_kind if k_scale_kind is not None else (
        SCALE_PER_TOKEN_HEAD if k_descale.dim() == 3 else SCALE_PER_TENSOR)
    v_kind = v_scale_kind if v_scale_kind is not None else (
        SCALE_PER_HEAD if v_descale.numel() == n2 else SCALE_PER_TENSOR)
    dims = make_dims(q, k_pages, block_table, cu_seqlens_q, max_q_len, max_kv_len, k_kind,
                     v_kind, causal, q_layout, kv_layout, tiles_per_step)
    T, N1, D = dims.total_q, dims.N1, dims.D
    if out is None:
        out = torch.empty((T, N1, D), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((N1, T), dtype=torch.float32, device=q.device)
    ws_bytes = workspace_size(dims)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    st = lib().bsa_fp8_prefill(
        ctypes.byref(dims), _p(q), _p(k_pages), _p(v_pages), _p(q_descale), _p(k_descale),
        _p(v_descale), _p(cu_seqlens_q), _p(seqused_kv), _p(block_table), _p(block_mask),
        _p(sparse_indices), _p(sparse_seq_len), float(softmax_scale), float(p_scale), _p(out),
        _p(lse), _p(workspace), ws_bytes, _p(dev_status), _stream_handle(stream))
    if st != 0:
        raise BsaError(st, "bsa_fp8_prefill")
    return out, lse


def prefill_host(host: dict, dev: dict, max_q_len: int, max_kv_len: int,
                 softmax_scale: float | None = None, p_scale: float = 256.0, causal: bool = True,
                 workspace=None, dev_status=None, stream=None, k_scale_kind: int | None = None,
                 v_scale_kind: int | None = None, q_layout: int = Q_TND,
                 kv_layout: int = KV_HND, tiles_per_step: int = 1) -> None:
    """The prefill on host tensors (bsa_fp8_prefill_host).  `host` maps the names in
    TENSOR_NAMES to CPU tensors (page-locked ones make the copies asynchronous; absent or None
    = not given); "out" and "lse" receive the results once `stream` has been synchronised.
    `dev` maps the same names to CUDA tensors of the same shapes, which the call fills and
    computes on.  Scale kinds default as in prefill()."""
    import torch

    k_descale, v_descale = host["k_descale"], host["v_descale"]
    k_pages = host["k_pages"]
    n2 = k_pages.shape[2] if kv_layout == KV_NHD else k_pages.shape[1]
    k_kind = k_scale_kind if k_scale_kind is not None else (
        SCALE_PER_TOKEN_HEAD if k_descale.dim() == 3 else SCALE_PER_TENSOR)
    v_kind = v_scale_kind if v_scale_kind is not None else (
        SCALE_PER_HEAD if v_descale.numel() == n2 else SCALE_PER_TENSOR)
    dims = make_dims(host["q"], k_pages, host["block_table"], host["cu_seqlens_q"], max_q_len,
                     max_kv_len, k_kind, v_kind, causal, q_layout, kv_layout, tiles_per_step)
    ws_bytes = workspace_size(dims)
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev["q"].device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(dims.D)
    th = Tensors(*(_p(host.get(n)) for n in TENSOR_NAMES))
    td = Tensors(*(_p(dev.get(n)) for n in TENSOR_NAMES))
    st = lib().bsa_fp8_prefill_host(ctypes.byref(dims), ctypes.byref(th), ctypes.byref(td),
                                    float(softmax_scale), float(p_scale), _p(workspace),
                                    ws_bytes, _p(dev_status), _stream_handle(stream))
    if st != 0:
        raise BsaError(st, "bsa_fp8_prefill_host")


def compact_tiles(cu_seqlens_q, seqused_kv, dims: Dims, block_mask=None, sparse_indices=None,
                  sparse_seq_len=None, dev_status=None, stream=None):
    """Active-tile lists [B, N1, Qb, Kb] (-1 past the count) and counts [B, N1, Qb]."""
    import torch

    Qb = -(-dims.max_q_len // 128)
    Kb = -(-dims.max_kv_len // 128)
    dev = cu_seqlens_q.device
    lists = torch.empty((dims.B, dims.N1, Qb, Kb), dtype=torch.int32, device=dev)
    counts = torch.empty((dims.B, dims.N1, Qb), dtype=torch.int32, device=dev)
    st = lib().bsa_fp8_compact_tiles(ctypes.byref(dims), _p(cu_seqlens_q), _p(seqused_kv),
                                     _p(block_mask), _p(sparse_indices), _p(sparse_seq_len),
                                     _p(lists), _p(counts), _p(dev_status),
                                     _stream_handle(stream))
    if st != 0:
        raise BsaError(st, "bsa_fp8_compact_tiles")
    return lists, counts


def quantize_rows(x, codes=None, descale=None, stream=None, rule: int = DESCALE_AMAX):
    """bf16 tensor [..., 128] -> (e4m3 codes uint8 [..., 128], fp32 descale [...]): per row
    descale = amax / 448 (1 for a zero row), rounded up to a power of two under
    DESCALE_UE8M0; code = e4m3(x / descale)."""
    import torch

    if x.dtype != torch.bfloat16 or x.shape[-1] != 128 or not x.is_contiguous():
        raise ValueError("x must be a contiguous bf16 tensor [..., 128]")
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if descale is None:
        descale = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    fn = lib().bsa_fp8_quantize_rows_ue8m0 if rule == DESCALE_UE8M0 else lib().bsa_fp8_quantize_rows
    st = fn(_p(x), x.numel() // 128, _p(codes), _p(descale), _stream_handle(stream))
    if st != 0:
        raise BsaError(st, "bsa_fp8_quantize_rows")
    return codes, descale


def append_kv(k_new, v_new, cu_seqlens_new, cache_seqlens, block_table, k_pages, v_pages,
              k_descale=None, k_scale=None, v_scale=None, k_scale_kind=SCALE_PER_TOKEN_HEAD,
              v_scale_kind=SCALE_PER_HEAD, dev_status=None, stream=None, kv_layout=KV_HND,
              k_descale_rule: int = DESCALE_AMAX):
    """Writes bf16 K/V tokens [T_new, N2, 128] into the paged cache (k_pages / v_pages
    [P, N2, page_size, 128] (KV_HND) or [P, page_size, N2, 128] (KV_NHD) uint8 e4m3,
    k_descale [P, N2, page_size] for per-token K, computed under k_descale_rule) at positions
    cache_seqlens[b] + i through block_table [B, L]; in place."""
    if kv_layout == KV_NHD:
        P, ps, N2, D = k_pages.shape
    else:
        P, N2, ps, D = k_pages.shape
    dims = AppendDims(B=cu_seqlens_new.numel() - 1, N2=N2, D=D, page_size=ps, num_pages=P,
                      max_pages_per_seq=block_table.shape[1], total_new=k_new.shape[0],
                      k_scale_kind=k_scale_kind, v_scale_kind=v_scale_kind,
                      kv_layout=int(kv_layout), k_descale_rule=int(k_descale_rule))
    st = lib().bsa_fp8_append_kv(ctypes.byref(dims), _p(k_new), _p(v_new), _p(cu_seqlens_new),
                                 _p(cache_seqlens), _p(block_table), _p(k_scale), _p(v_scale),
                                 _p(k_pages), _p(v_pages), _p(k_descale), _p(dev_status),
                                 _stream_handle(stream))
    if st != 0:
        raise BsaError(st, "bsa_fp8_append_kv")
    return k_pages, v_pages, k_descale
