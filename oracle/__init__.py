"""CPU oracle for block-sparse FP8 attention prefill (fp64, plain C, ctypes wrapper).

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg import this package.  The product library (``block_sparse_fp8_gb300``) never
does.  The C source, ``bsa_oracle.c``, restates the formula of "Quant Block Sparse Attention"
(CANNBotDSL, section 算子介绍) and the fixed P-scale online softmax of "hpc-ops Block-Sparse
FP8 Attention" (section 固定 P-scale 量化技巧); its header lists the readings it takes.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py`` (brute-force
dense attention, closed forms, invariants, the exhaustive e4m3 table; the quantise and
KV-append step against numpy fp32 arithmetic with PyTorch's e4m3 cast and hand-derived
codes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sysconfig

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "bsa_oracle.c")
LIB = os.path.join(HERE, "_build", "libbsa_oracle.so")

EXACT = 0
PEMU = 1

ERR_BAD_INDEX = 1
ERR_BAD_PAGE = 2
ERR_BAD_ARG = 4


class OracleDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "B", "N1", "N2", "D", "page_size", "max_q_len", "max_kv_len", "num_pages",
        "max_pages_per_seq", "total_q", "k_scale_kind", "v_scale_kind", "causal")]


class OracleInputs(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k_pages", ctypes.c_void_p), ("v_pages", ctypes.c_void_p),
        ("q_descale", ctypes.c_void_p), ("k_descale", ctypes.c_void_p),
        ("v_descale", ctypes.c_void_p), ("cu_seqlens_q", ctypes.c_void_p),
        ("seqused_kv", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
        ("block_mask", ctypes.c_void_p), ("sparse_indices", ctypes.c_void_p),
        ("sparse_seq_len", ctypes.c_void_p), ("softmax_scale", ctypes.c_double),
        ("p_scale", ctypes.c_double)]


def build(src: str = SRC, out: str = LIB, openmp: bool = True) -> str:
    """Compiles the oracle with gcc (fp64, no fast-math).  Returns the library path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
            "-ffp-contract=off", src, "-o", out, "-lm"]
    if openmp:
        r = subprocess.run(base[:-3] + ["-fopenmp"] + base[-3:], capture_output=True, text=True)
        if r.returncode == 0:
            return out
    subprocess.run(base, check=True)
    return out


_lib = None


def load(path: str | None = None):
    global _lib
    if path is not None:
        lib = ctypes.CDLL(path)
    else:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
            build()
        lib = ctypes.CDLL(LIB)
    lib.oracle_e4m3_decode.restype = ctypes.c_double
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
    lib.oracle_active_tiles.restype = ctypes.c_int
    lib.oracle_active_tiles.argtypes = [ctypes.POINTER(OracleDims), ctypes.POINTER(OracleInputs),
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
    lib.oracle_all_lists.restype = ctypes.c_int
    lib.oracle_all_lists.argtypes = [ctypes.POINTER(OracleDims), ctypes.POINTER(OracleInputs),
                                     ctypes.c_void_p, ctypes.c_void_p]
    lib.oracle_attention_rows.restype = ctypes.c_int
    lib.oracle_attention_rows.argtypes = [ctypes.POINTER(OracleDims),
                                          ctypes.POINTER(OracleInputs), ctypes.c_int,
                                          ctypes.c_void_p, ctypes.c_long, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_int]
    lib.oracle_attention_rows_split.restype = ctypes.c_int
    lib.oracle_attention_rows_split.argtypes = [ctypes.POINTER(OracleDims),
                                                ctypes.POINTER(OracleInputs), ctypes.c_int,
                                                ctypes.c_int, ctypes.c_void_p, ctypes.c_long,
                                                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.oracle_attention_rows_grouped.restype = ctypes.c_int
    lib.oracle_attention_rows_grouped.argtypes = [ctypes.POINTER(OracleDims),
                                                  ctypes.POINTER(OracleInputs), ctypes.c_int,
                                                  ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                                  ctypes.c_long, ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_int]
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_quantize_rows.restype = None
    lib.oracle_quantize_rows.argtypes = [ctypes.c_void_p, ctypes.c_long, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_void_p]
    lib.oracle_append_kv.restype = ctypes.c_int
    lib.oracle_append_kv.argtypes = [ctypes.c_int] * 8 + [ctypes.c_void_p] * 10
    if path is None:
        _lib = lib
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p).value


class Oracle:
    """Binds one workloads.Case (host arrays) to the C oracle."""

    def __init__(self, case, lib=None):
        self.case = case
        self.lib = lib if lib is not None else load()
        c = case
        self._keep = [np.ascontiguousarray(a) if a is not None else None for a in (
            c.q, c.k_pages, c.v_pages, c.q_descale, c.k_descale, c.v_descale, c.cu_seqlens_q,
            c.seqused_kv, c.block_table, c.block_mask, c.sparse_indices, c.sparse_seq_len)]
        self.dims = OracleDims(**c.dims())
        k = self._keep
        self.inputs = OracleInputs(
            _ptr(k[0]), _ptr(k[1]), _ptr(k[2]), _ptr(k[3]), _ptr(k[4]), _ptr(k[5]),
            _ptr(k[6]), _ptr(k[7]), _ptr(k[8]), _ptr(k[9]), _ptr(k[10]), _ptr(k[11]),
            float(c.softmax_scale), float(c.p_scale))

    def lists(self):
        """(lists [B,N1,Qb,Kb] int32 with -1 past the count, counts [B,N1,Qb] int32, err)."""
        c = self.case
        lists = np.full((c.B, c.N1, c.Qb, c.Kb), -1, dtype=np.int32)
        counts = np.zeros((c.B, c.N1, c.Qb), dtype=np.int32)
        err = self.lib.oracle_all_lists(ctypes.byref(self.dims), ctypes.byref(self.inputs),
                                        _ptr(lists), _ptr(counts))
        return lists, counts, err

    def rows(self, rows, mode=EXACT, nthreads=0, splits=1, group=1):
        """rows: int array [n, 2] of (token, head).  Returns (o [n,128] f64, lse [n] f64, err).
        splits > 1 (P-emulating mode): the active list cut into that many consecutive slices,
        each with its own online softmax, merged by log-sum-exp weights.  group (P-emulating
        mode): list tiles per online-softmax step, 1 (128-token tiles) or 2 (256-wide macro
        blocks of two tiles, an odd last tile alone)."""
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 2))
        n = rows.shape[0]
        o = np.zeros((n, 128), dtype=np.float64)
        lse = np.zeros(n, dtype=np.float64)
        err = self.lib.oracle_attention_rows_grouped(ctypes.byref(self.dims),
                                                     ctypes.byref(self.inputs), mode,
                                                     int(splits), int(group), _ptr(rows), n,
                                                     _ptr(o), _ptr(lse), nthreads)
        return o, lse, err

    def all_rows(self, mode=EXACT, nthreads=0, splits=1, group=1):
        """Full O [T, N1, 128] and LSE [N1, T]."""
        c = self.case
        tok, h = np.meshgrid(np.arange(c.T), np.arange(c.N1), indexing="ij")
        rows = np.stack([tok.ravel(), h.ravel()], axis=1)
        o, lse, err = self.rows(rows, mode, nthreads, splits, group)
        return o.reshape(c.T, c.N1, 128), lse.reshape(c.T, c.N1).T.copy(), err


DESCALE_AMAX, DESCALE_UE8M0 = 0, 1


def quantize_rows(x_bf16: np.ndarray, lib=None, rule: int = DESCALE_AMAX):
    """x_bf16: uint16 bf16 bit patterns [..., 128].  Returns (codes uint8 [..., 128], descale
    float32 [...]): per row descale = amax/448 (1 for a zero row), with DESCALE_UE8M0 rounded
    up to a power of two (FlashMLA page, 量化 / 解量化的源码实现), code = e4m3(x / descale)."""
    lib = lib if lib is not None else load()
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    assert x.shape[-1] == 128
    rows = x.size // 128
    codes = np.zeros(x.shape, dtype=np.uint8)
    desc = np.zeros(x.shape[:-1], dtype=np.float32)
    lib.oracle_quantize_rows(_ptr(x), rows, int(rule), _ptr(codes), _ptr(desc))
    return codes, desc


def append_kv(k_new, v_new, cu_new, cache_len, block_table, k_pages, v_pages, k_descale,
              k_scale_kind, v_scale_kind, k_scale=None, v_scale=None, lib=None,
              k_descale_rule: int = DESCALE_AMAX):
    """Writes bf16 K/V tokens [T_new, N2, 128] (uint16 bit patterns) into copies of the paged
    cache arrays; per-token K descales follow k_descale_rule.  Returns (k_pages, v_pages,
    k_descale, err)."""
    lib = lib if lib is not None else load()
    k_new = np.ascontiguousarray(k_new, dtype=np.uint16)
    v_new = np.ascontiguousarray(v_new, dtype=np.uint16)
    cu_new = np.ascontiguousarray(cu_new, dtype=np.int32)
    cache_len = np.ascontiguousarray(cache_len, dtype=np.int32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    kp = np.array(k_pages, dtype=np.uint8, copy=True)
    vp = np.array(v_pages, dtype=np.uint8, copy=True)
    kd = np.array(k_descale, dtype=np.float32, copy=True)
    ks = np.ascontiguousarray(np.atleast_1d(k_scale if k_scale is not None else 1.0), dtype=np.float32)
    vs = np.ascontiguousarray(np.atleast_1d(v_scale if v_scale is not None else 1.0), dtype=np.float32)
    P, N2, ps, D = kp.shape
    B = cu_new.size - 1
    err = lib.oracle_append_kv(B, N2, ps, P, bt.shape[1], int(k_scale_kind), int(v_scale_kind),
                               int(k_descale_rule),
                               _ptr(k_new), _ptr(v_new), _ptr(cu_new), _ptr(cache_len), _ptr(bt),
                               _ptr(ks), _ptr(vs), _ptr(kp), _ptr(vp), _ptr(kd))
    return kp, vp, kd, err


def e4m3_decode(code: int) -> float:
    return load().oracle_e4m3_decode(code)


def e4m3_encode(x: float) -> int:
    return load().oracle_e4m3_encode(x)


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return sysconfig.get_platform()
