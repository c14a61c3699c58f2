"""The C-ABI library loads, exports every symbol include/bsa_fp8.h declares, and validates its
arguments on the host (no GPU needed: every call here returns before touching CUDA)."""
from __future__ import annotations

import ctypes
import os
import re
import shutil

import numpy as np

import pytest

import block_sparse_fp8_gb300 as bsa
from block_sparse_fp8_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "bsa_fp8.h")
INVALID, UNSUPPORTED = 1, 2


@pytest.fixture(scope="module")
def L():
    if _build.needs_build():
        if shutil.which(_build.nvcc()) is None and not os.path.exists(_build.nvcc()):
            pytest.skip("nvcc not available")
        _build.build()
    return bsa.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bsa_\w+)\s*\(", src)))


def test_header_declares_the_binding_set():
    assert declared_functions() == sorted(bsa.EXPORTED)


def test_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings(L):
    for code in range(5):
        assert bsa.status_string(code)
    assert "unknown" in bsa.status_string(99)


def _dims(**kw):
    base = dict(B=1, N1=8, N2=1, D=128, page_size=64, max_q_len=1024, max_kv_len=1024,
                num_pages=16, max_pages_per_seq=16, total_q=1024, k_scale_kind=0,
                v_scale_kind=0, causal=1)
    base.update(kw)
    return bsa.Dims(**base)


def _prefill(L, dims, **ptrs):
    fake = 0x10000  # never dereferenced: every case below fails validation first
    args = dict(q=fake, k=fake, v=fake, qd=fake, kd=fake, vd=fake, cu=fake, su=fake, bt=fake,
                mask=None, idx=None, sl=None, scale=0.088, pscale=256.0, out=fake, lse=fake)
    args.update(ptrs)
    return L.bsa_fp8_prefill(ctypes.byref(dims), args["q"], args["k"], args["v"], args["qd"],
                             args["kd"], args["vd"], args["cu"], args["su"], args["bt"],
                             args["mask"], args["idx"], args["sl"], args["scale"],
                             args["pscale"], args["out"], args["lse"], None, 0, None, None)


@pytest.mark.parametrize("bad", [
    dict(D=64), dict(page_size=48), dict(page_size=128), dict(N1=6, N2=4), dict(N1=34, N2=2),
    dict(N1=0), dict(N2=0), dict(max_q_len=-1), dict(max_kv_len=-5), dict(total_q=-1),
    dict(max_pages_per_seq=15), dict(k_scale_kind=2), dict(v_scale_kind=1),
    dict(causal=2), dict(B=-1), dict(q_layout=2), dict(kv_layout=-1), dict(tiles_per_step=3),
    dict(tiles_per_step=-1)])
def test_invalid_dims(L, bad):
    assert _prefill(L, _dims(**bad)) == INVALID


def test_too_many_kv_tiles_unsupported(L):
    d = _dims(max_kv_len=4097 * 128, max_pages_per_seq=4097 * 2, num_pages=8194 * 1)
    assert _prefill(L, d) == UNSUPPORTED


def test_too_many_tasks_unsupported(L):
    # B * N1 * Qb above 2^30: the int work-item counter must not wrap
    d = _dims(B=1 << 12, N1=16, N2=1, max_q_len=(1 << 14) * 128 + 1)
    assert _prefill(L, d) == UNSUPPORTED


def test_invalid_scalars_and_pointers(L):
    d = _dims()
    assert _prefill(L, d, scale=float("inf")) == INVALID
    assert _prefill(L, d, scale=float("nan")) == INVALID
    assert _prefill(L, d, pscale=float("nan")) == INVALID
    assert _prefill(L, d, pscale=float("inf")) == INVALID
    assert _prefill(L, d, mask=0x20000, idx=0x30000, sl=0x40000) == INVALID   # both forms
    assert _prefill(L, d, idx=0x30000) == INVALID                              # no seq_len
    for k in ("q", "k", "v", "qd", "kd", "vd", "cu", "bt", "out"):
        assert _prefill(L, d, **{k: None}) == INVALID, k
    assert _prefill(L, d, q=0x10001) == INVALID     # TMA needs 16-byte aligned bases
    assert _prefill(L, d, k=0x10008) == INVALID
    assert _prefill(L, d, lse=0x10002) == INVALID   # fp32 LSE needs 4-byte alignment
    assert _prefill(L, _dims(num_pages=0)) == INVALID


def test_empty_problem_is_a_no_op(L):
    assert _prefill(L, _dims(B=0, total_q=0)) == 0
    assert _prefill(L, _dims(total_q=0)) == 0
    assert _prefill(L, _dims(max_q_len=0, total_q=0)) == 0


def test_compact_validation(L):
    d = _dims(page_size=16)
    assert L.bsa_fp8_compact_tiles(ctypes.byref(d), 1, None, None, None, None, 1, 1, None,
                                   None) == INVALID
    d = _dims()
    assert L.bsa_fp8_compact_tiles(ctypes.byref(d), 0x100, None, 0x200, 0x300, 0x400, 0x500,
                                   0x600, None, None) == INVALID


def test_workspace_query(L):
    assert bsa.workspace_size(_dims()) == 256
    assert bsa.workspace_size(_dims(D=64)) == 0


def test_workspace_required(L):
    d = _dims()
    fake = 0x10000
    args = [fake] * 9 + [None, None, None]
    call = lambda ws, nbytes: L.bsa_fp8_prefill(ctypes.byref(d), *args, 0.088, 256.0, fake,
                                                fake, ws, nbytes, None, None)
    assert call(None, 0) == 4                 # BSA_ERR_WORKSPACE
    assert call(0x20000, 255) == 4            # too small
    assert call(0x20002, 256) == 4            # misaligned


def _noalloc(L, dims, **ptrs):
    fake = 0x10000  # never dereferenced: every case below fails validation first
    args = dict(q=fake, k=fake, v=fake, qd=fake, kd=fake, vd=fake, cu=fake, su=fake, bt=fake,
                mask=None, idx=None, sl=None, scale=0.088, pscale=256.0, out=fake, lse=fake)
    args.update(ptrs)
    return L.bsa_fp8_prefill_noalloc(ctypes.byref(dims), args["q"], args["k"], args["v"],
                                     args["qd"], args["kd"], args["vd"], args["cu"], args["su"],
                                     args["bt"], args["mask"], args["idx"], args["sl"],
                                     args["scale"], args["pscale"], args["out"], args["lse"],
                                     None, None)


@pytest.mark.parametrize("bad", [dict(D=64), dict(page_size=48), dict(N1=6, N2=4),
                                 dict(max_pages_per_seq=15), dict(causal=2)])
def test_noalloc_validates_like_prefill(L, bad):
    """The array-backed entry point checks its arguments before it touches the device, so its
    error codes are those of bsa_fp8_prefill (no GPU is needed to reach them)."""
    d = _dims(**bad)
    assert _noalloc(L, d) == _prefill(L, d) == INVALID


def test_noalloc_scalar_pointer_and_size_checks(L):
    d = _dims()
    assert _noalloc(L, d, scale=float("nan")) == INVALID
    assert _noalloc(L, d, mask=0x20000, idx=0x30000, sl=0x40000) == INVALID
    for k in ("q", "k", "v", "qd", "kd", "vd", "cu", "bt", "out"):
        assert _noalloc(L, d, **{k: None}) == INVALID, k
    assert _noalloc(L, d, q=0x10001) == INVALID
    assert _noalloc(L, _dims(max_kv_len=4097 * 128, max_pages_per_seq=4097 * 2,
                             num_pages=8194)) == UNSUPPORTED
    assert _noalloc(L, _dims(B=0, total_q=0)) == 0


def _host(L, dims, host=None, dev=None, **over):
    """bsa_fp8_prefill_host with fake addresses (never dereferenced: every case below fails
    validation before a copy is queued).  `over` sets "host.<name>" / "dev.<name>"."""
    fake = 0x10000
    sets = {}
    for side in ("host", "dev"):
        t = dict.fromkeys(bsa.TENSOR_NAMES, fake)
        t.update(block_mask=None, sparse_indices=None, sparse_seq_len=None)
        for key, val in over.items():
            s, name = key.split(".")
            if s == side:
                t[name] = val
        sets[side] = bsa.Tensors(*(t[n] for n in bsa.TENSOR_NAMES))
    h = None if host == "null" else ctypes.byref(sets["host"])
    d = None if dev == "null" else ctypes.byref(sets["dev"])
    return L.bsa_fp8_prefill_host(ctypes.byref(dims), h, d, 0.088, 256.0, fake, 256, None, None)


@pytest.mark.parametrize("bad", [dict(D=64), dict(page_size=48), dict(N1=6, N2=4),
                                 dict(max_pages_per_seq=15), dict(tiles_per_step=3)])
def test_host_call_validates_dims_like_prefill(L, bad):
    d = _dims(**bad)
    assert _host(L, d) == _prefill(L, d) == INVALID


def test_host_call_tensor_checks(L):
    d = _dims()
    assert _host(L, d, host="null") == INVALID
    assert _host(L, d, dev="null") == INVALID
    for name in ("q", "k_pages", "v_pages", "q_descale", "k_descale", "v_descale",
                 "cu_seqlens_q", "block_table", "out"):
        assert _host(L, d, **{f"host.{name}": None}) == INVALID, name   # host side missing
        assert _host(L, d, **{f"dev.{name}": None}) == INVALID, name    # device side missing
    for name in ("seqused_kv", "lse"):   # optional tensors: given on both sides or neither
        assert _host(L, d, **{f"host.{name}": None}) == INVALID, name
        assert _host(L, d, **{f"dev.{name}": None}) == INVALID, name
    assert _host(L, d, **{"host.block_mask": 0x20000}) == INVALID
    assert _host(L, d, **{"dev.sparse_indices": 0x20000, "dev.sparse_seq_len": 0x30000}) == INVALID
    assert _host(L, d, **{"dev.q": 0x10001}) == INVALID                 # the device set's alignment
    assert _host(L, d, **{"host.block_mask": 0x20000, "dev.block_mask": 0x30000,
                          "host.sparse_indices": 0x20000, "dev.sparse_indices": 0x30000,
                          "host.sparse_seq_len": 0x20000,
                          "dev.sparse_seq_len": 0x30000}) == INVALID    # both sparse forms


def test_host_call_empty_problem_is_a_no_op(L):
    nothing = {f"{s}.{n}": None for s in ("host", "dev") for n in bsa.TENSOR_NAMES}
    assert _host(L, _dims(B=0, total_q=0), **nothing) == 0
    assert _host(L, _dims(total_q=0), **nothing) == 0


def test_append_descale_rule_checked(L):
    fake = 0x10000
    for rule, want in ((2, INVALID), (-1, INVALID)):
        d = bsa.AppendDims(B=1, N2=2, D=128, page_size=64, num_pages=4, max_pages_per_seq=4,
                           total_new=8, k_scale_kind=1, v_scale_kind=2, kv_layout=0,
                           k_descale_rule=rule)
        assert L.bsa_fp8_append_kv(ctypes.byref(d), *([fake] * 12)) == want


def test_quantize_ue8m0_validation(L):
    assert L.bsa_fp8_quantize_rows_ue8m0(None, 0, None, None, None) == 0
    assert L.bsa_fp8_quantize_rows_ue8m0(None, -1, None, None, None) == INVALID
    assert L.bsa_fp8_quantize_rows_ue8m0(0x10008, 4, 0x20000, 0x30000, None) == INVALID


def test_generator_token_group_power_of_two_k_scales():
    """The seeded generator's K scales per token group: one value per group of consecutive
    tokens of a sequence and KV head, a power of two not below the group's amax / 448."""
    import workloads as W

    case = W.make_case("kg", 5, [300, 77], [300, 90], 4, 2, 32, W.SCALE_PER_TOKEN_HEAD,
                       W.SCALE_PER_HEAD, "none", k_token_group=16, k_pow2=True,
                       keep_logical=True)
    kd = case.meta["k_descale_tok"]                           # [tokens, N2], token order
    s0 = 0
    for kv in (300, 90):
        for g0 in range(0, kv, 16):
            grp = kd[s0 + g0: s0 + min(kv, g0 + 16)]
            assert np.all(grp == grp[0])
        s0 += kv
    lg = np.log2(kd.astype(np.float64))
    assert np.all(lg == np.round(lg))
