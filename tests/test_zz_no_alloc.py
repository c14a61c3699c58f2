"""bsa_fp8_prefill_noalloc: the prefill for callers that cannot allocate device memory.

Such a caller -- a plugin handed only its input and output buffers, code running from a
fixed device-memory budget, or a path that must not pay cudaMalloc's implicit
synchronisation -- gets the same result through this entry point, which uses the library's
own 256-byte device array where bsa_fp8_prefill uses the caller's workspace.  These tests
call it through the C ABI:

  * where bsa_fp8_prefill does not split the KV lists either, both entry points run the same
    plan, so two calls in a row must reproduce bsa_fp8_prefill's output bit for bit;
  * where bsa_fp8_prefill would split (few tasks over a long KV), this entry point runs the
    lists unsplit, so it is checked against the oracle instead: the exact fp64 band and the
    tight band around the P-emulating mode over the whole list (one slice).

The file is named to be collected last, so that a run stopping at the first failure has run
every other test before this one; it also passes on its own in a fresh process.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_helpers import (EXACT_ATOL, EXACT_RTOL, PEMU_ATOL, PEMU_RTOL, SPLIT_CASES, check_lse,
                         check_o, ensure_built, sample_rows, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_built()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _call(lib, name, case, d, out, lse, status, extra):
    import block_sparse_fp8_gb300 as bsa

    dims = bsa.Dims(**case.dims())
    fn = getattr(lib, name)
    args = [ctypes.byref(dims), _ptr(d["q"]), _ptr(d["k_pages"]), _ptr(d["v_pages"]),
            _ptr(d["q_descale"]), _ptr(d["k_descale"]), _ptr(d["v_descale"]),
            _ptr(d["cu_seqlens_q"]), _ptr(d["seqused_kv"]), _ptr(d["block_table"]),
            _ptr(d["block_mask"]), _ptr(d["sparse_indices"]), _ptr(d["sparse_seq_len"]),
            case.softmax_scale, case.p_scale, _ptr(out), _ptr(lse)]
    args += extra + [_ptr(status), torch.cuda.current_stream().cuda_stream]
    return fn(*args)


def _noalloc(lib, case, d):
    """One bsa_fp8_prefill_noalloc call into NaN-filled outputs; returns (out, lse)."""
    out = torch.full((case.T, case.N1, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((case.N1, case.T), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _call(lib, "bsa_fp8_prefill_noalloc", case, d, out, lse, st, []) == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    return out, lse


def _splits_of_prefill(case):
    """Slices bsa_fp8_prefill cuts each task into: more than one when its workspace query asks
    for more than the 256-byte counter."""
    import block_sparse_fp8_gb300 as bsa

    return bsa.workspace_size(bsa.Dims(**case.dims())) > 256


def test_noalloc_matches_prefill_twice(lib):
    import block_sparse_fp8_gb300 as bsa

    # per-token K descales and more tasks than resident CTAs: every part of the kernel runs,
    # and the shared task counter is reused by consecutive calls
    case = W.make_case("noalloc", 77, [2000, 1300, 129], [2000, 1500, 129], 16, 4, 64,
                       W.SCALE_PER_TOKEN_HEAD, W.SCALE_PER_HEAD, "bernoulli", keep=0.5)
    assert not _splits_of_prefill(case)
    d = to_device(case)
    ref_out = torch.full((case.T, case.N1, 128), float("nan"), dtype=torch.bfloat16,
                         device="cuda")
    ref_lse = torch.full((case.N1, case.T), float("nan"), dtype=torch.float32, device="cuda")
    ref_st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws_bytes = bsa.workspace_size(bsa.Dims(**case.dims()))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    assert _call(lib, "bsa_fp8_prefill", case, d, ref_out, ref_lse, ref_st,
                 [_ptr(ws), ws_bytes]) == 0
    torch.cuda.synchronize()
    assert int(ref_st.item()) == 0
    for call in range(2):
        out, lse = _noalloc(lib, case, d)
        # the same unsplit plan as bsa_fp8_prefill: the same bits
        assert torch.equal(out, ref_out), f"call {call}: O differs from bsa_fp8_prefill"
        assert torch.equal(lse, ref_lse), f"call {call}: LSE differs from bsa_fp8_prefill"


@pytest.mark.parametrize("name", sorted(SPLIT_CASES))
def test_noalloc_unsplit_where_prefill_splits(lib, name):
    case = W.make_case(name, **SPLIT_CASES[name])
    assert _splits_of_prefill(case), "the case is meant to be one bsa_fp8_prefill splits"
    d = to_device(case)
    orc = O.Oracle(case)
    o_ex, l_ex, err = orc.all_rows(O.EXACT)
    o_pe, _, _ = orc.all_rows(O.PEMU, splits=1)
    assert err == 0
    first = None
    for call in range(2):
        out, lse = _noalloc(lib, case, d)
        got = out.float().cpu().numpy()
        check_o(got, o_ex, EXACT_ATOL, EXACT_RTOL, f"{name} call {call} vs exact")
        check_o(got, o_pe, PEMU_ATOL, PEMU_RTOL, f"{name} call {call} vs P-emulating")
        check_lse(lse.cpu().numpy(), l_ex, f"{name} call {call} LSE")
        if first is None:
            first = (out, lse)
        else:
            assert torch.equal(out, first[0]) and torch.equal(lse, first[1])


def test_noalloc_longest_supported_kv(lib):
    """Kb = 4096 KV tiles over four tasks: bsa_fp8_prefill splits this; the array-backed entry
    point runs each 4096-tile list in one pipeline.  Sampled rows against the oracle."""
    case = W.make_case("max_kb", 301, [256], [4096 * 128], 2, 1, 64, W.SCALE_PER_TOKEN_HEAD,
                       W.SCALE_PER_HEAD, "local_sink", n_local=2, p_far=0.01)
    assert case.Kb == 4096 and _splits_of_prefill(case)
    d = to_device(case)
    rows = sample_rows(case, 96, seed=3)
    orc = O.Oracle(case)
    o_ex, l_ex, err = orc.rows(rows, O.EXACT)
    o_pe, _, _ = orc.rows(rows, O.PEMU, splits=1)
    assert err == 0
    for call in range(2):
        out, lse = _noalloc(lib, case, d)
        got = out.float()[rows[:, 0], rows[:, 1]].cpu().numpy()
        check_o(got, o_ex, EXACT_ATOL, EXACT_RTOL, f"call {call} vs exact")
        check_o(got, o_pe, PEMU_ATOL, PEMU_RTOL, f"call {call} vs P-emulating")
        check_lse(lse[rows[:, 1], rows[:, 0]].cpu().numpy(), l_ex, f"call {call} LSE")
