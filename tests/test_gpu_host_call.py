"""bsa_fp8_prefill_host: host tensors in, host results out, through one C-ABI call.

The call copies every input to the caller's device buffers, runs the prefill on them and
copies O and the LSE back, all on one stream.  Its results must be bit for bit those of
bsa_fp8_prefill on the same inputs already on the device (same kernel, same plan), and
within the exact band of the oracle's formula.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_helpers import (EXACT_ATOL, EXACT_RTOL, SPLIT_CASES, check_o, ensure_built, run,
                         sample_rows, to_device)
from test_gpu_parity import SMALL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _host_call(case, pinned=True, with_lse=True, stream=None, dev=None, **kw):
    import block_sparse_fp8_gb300 as bsa

    host = {n: torch.from_numpy(np.ascontiguousarray(getattr(case, n)))
            for n in bsa.TENSOR_NAMES[:-2] if getattr(case, n) is not None}
    host["out"] = torch.full((case.T, case.N1, 128), float("nan"), dtype=torch.bfloat16)
    if with_lse:
        host["lse"] = torch.full((case.N1, case.T), float("nan"))
    if pinned:
        host = {k: v.pin_memory() for k, v in host.items()}
    if dev is None:
        dev = {k: (None if v is None else torch.empty(v.shape, dtype=v.dtype, device="cuda"))
               for k, v in host.items()}
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsa.prefill_host(host, dev, case.max_q_len, case.max_kv_len,
                     softmax_scale=case.softmax_scale, p_scale=case.p_scale,
                     causal=bool(case.causal), dev_status=st, stream=stream,
                     k_scale_kind=case.k_scale_kind, v_scale_kind=case.v_scale_kind, **kw)
    torch.cuda.synchronize()
    return host["out"], host.get("lse"), int(st.item())


CASES = {**{n: SMALL[n] for n in ("bern_ragged", "bern_pt_p32", "indices_empty", "chunked_off")},
         "split_long_kv": SPLIT_CASES["split_long_kv"]}


@pytest.mark.parametrize("name", sorted(CASES))
def test_host_call_matches_device_call_bitwise(name):
    case = W.make_case(name, **CASES[name])
    ref_out, ref_lse, st = run(case)
    assert st == 0
    out, lse, st = _host_call(case)
    assert st == 0
    assert torch.equal(out, ref_out.cpu()) and torch.equal(lse, ref_lse.cpu())


def test_host_call_against_the_oracle_pageable_no_lse():
    """Pageable host memory, no LSE, a side stream: the same output, within the exact band."""
    case = W.make_case("bern_pt_p32", **SMALL["bern_pt_p32"])
    side = torch.cuda.Stream()
    out, lse, st = _host_call(case, pinned=False, with_lse=False, stream=side)
    assert st == 0 and lse is None
    rows = sample_rows(case, 1024, seed=5)
    o_ex, l_ex, err = O.Oracle(case).rows(rows, O.EXACT)
    assert err == 0
    check_o(out.float()[rows[:, 0], rows[:, 1]].numpy(), o_ex, EXACT_ATOL, EXACT_RTOL,
            "host call vs exact")
    ref_out, _, _ = run(case)
    assert torch.equal(out, ref_out.cpu())


def test_host_call_macro_blocks_and_reused_buffers():
    """Two calls on the same device buffers (the second overwrites every input), one of them
    with 256-wide macro blocks: each gives its own kernel's result."""
    case = W.make_case("indices_empty", **SMALL["indices_empty"])
    d = to_device(case)
    out1, lse1, _ = run(case, d)
    out2, lse2, _ = run(case, d, tiles_per_step=2)
    dev = {k: (None if v is None else torch.empty_like(v)) for k, v in d.items()}
    dev["out"] = torch.empty_like(out1)
    dev["lse"] = torch.empty_like(lse1)
    h1, l1, st = _host_call(case, dev=dev)
    assert st == 0
    h2, l2, st = _host_call(case, dev=dev, tiles_per_step=2)
    assert st == 0
    assert torch.equal(h1, out1.cpu()) and torch.equal(l1, lse1.cpu())
    assert torch.equal(h2, out2.cpu()) and torch.equal(l2, lse2.cpu())


def test_host_call_other_layouts():
    """Q [N1, T, 128] with q_descale [N1, T] and NHD pages [P, page, N2, 128] from host
    memory: the same copies (layout-independent sizes) and the TND / HND result bit for bit."""
    import block_sparse_fp8_gb300 as bsa

    case = W.make_case("bern_ragged", **SMALL["bern_ragged"])
    ref_out, ref_lse, _ = run(case)
    host = {n: torch.from_numpy(np.ascontiguousarray(getattr(case, n)))
            for n in bsa.TENSOR_NAMES[:-2] if getattr(case, n) is not None}
    host["q"] = host["q"].permute(1, 0, 2).contiguous()
    host["q_descale"] = host["q_descale"].t().contiguous()
    host["k_pages"] = host["k_pages"].permute(0, 2, 1, 3).contiguous()
    host["v_pages"] = host["v_pages"].permute(0, 2, 1, 3).contiguous()
    host["out"] = torch.zeros((case.T, case.N1, 128), dtype=torch.bfloat16)
    host["lse"] = torch.zeros((case.N1, case.T))
    host = {k: v.pin_memory() for k, v in host.items()}
    dev = {k: torch.empty(v.shape, dtype=v.dtype, device="cuda") for k, v in host.items()}
    bsa.prefill_host(host, dev, case.max_q_len, case.max_kv_len,
                     softmax_scale=case.softmax_scale, p_scale=case.p_scale,
                     causal=bool(case.causal), k_scale_kind=case.k_scale_kind,
                     v_scale_kind=case.v_scale_kind, q_layout=bsa.Q_NTD, kv_layout=bsa.KV_NHD)
    torch.cuda.synchronize()
    assert torch.equal(host["out"], ref_out.cpu()) and torch.equal(host["lse"], ref_lse.cpu())
