"""bsa_fp8_prefill_noalloc: the prefill for callers that cannot allocate device memory.

Such a caller -- a plugin handed only its input and output buffers, code running from a
fixed device-memory budget, or a path that must not pay cudaMalloc's implicit
synchronisation -- gets the same result through this entry point, which uses the library's
own 256-byte device array where bsa_fp8_prefill uses the caller's workspace.  This test calls
it through the C ABI twice in a row and checks both results against bsa_fp8_prefill's.

The file is named to be collected last, so that a run stopping at the first failure has run
every other test before this one; it also passes on its own in a fresh process.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import (LSE_ATOL, LSE_RTOL, MAX_OUTSIDE, PEMU_ATOL, PEMU_RTOL, band_fraction,
                         ensure_built, to_device)

pytestmark = pytest.mark.gpu


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


def test_noalloc_matches_prefill_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = ensure_built()
    import block_sparse_fp8_gb300 as bsa

    # per-token K descales and more tasks than resident CTAs: every part of the kernel runs,
    # and the shared task counter is reused by consecutive calls
    case = W.make_case("noalloc", 77, [2000, 1300, 129], [2000, 1500, 129], 16, 4, 64,
                       W.SCALE_PER_TOKEN_HEAD, W.SCALE_PER_HEAD, "bernoulli", keep=0.5)
    d = to_device(case)
    new = lambda *shape, dt: torch.full(shape, float("nan"), dtype=dt, device="cuda")

    ref_out = new(case.T, case.N1, 128, dt=torch.bfloat16)
    ref_lse = new(case.N1, case.T, dt=torch.float32)
    ref_st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws_bytes = bsa.workspace_size(bsa.Dims(**case.dims()))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    assert _call(lib, "bsa_fp8_prefill", case, d, ref_out, ref_lse, ref_st,
                 [_ptr(ws), ws_bytes]) == 0
    torch.cuda.synchronize()
    assert int(ref_st.item()) == 0

    for call in range(2):
        out = new(case.T, case.N1, 128, dt=torch.bfloat16)
        lse = new(case.N1, case.T, dt=torch.float32)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _call(lib, "bsa_fp8_prefill_noalloc", case, d, out, lse, st, []) == 0
        torch.cuda.synchronize()
        assert int(st.item()) == 0, f"call {call}: device status {int(st.item())}"
        got = out.float().cpu().numpy()
        ref = ref_out.float().cpu().numpy()
        assert np.all(np.isfinite(got)), f"call {call}: unwritten or non-finite output"
        frac, _ = band_fraction(got, ref, PEMU_ATOL, PEMU_RTOL)
        assert frac <= MAX_OUTSIDE, f"call {call}: {frac:.4%} of O outside the band"
        frac, _ = band_fraction(lse.cpu().numpy(), ref_lse.cpu().numpy(), LSE_ATOL, LSE_RTOL)
        assert frac <= MAX_OUTSIDE, f"call {call}: {frac:.4%} of LSE outside the band"
