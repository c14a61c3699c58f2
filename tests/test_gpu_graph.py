"""The prefill inside CUDA graphs.

Every entry point queues its work on the caller's stream and never synchronises, so a call
can be captured once and replayed: a replay must give exactly the eager call's result, and
a replay after the inputs were overwritten in place must give the eager result on the new
inputs.  Covered: the device call (unsplit and split-KV, whose counters are cleared by a
captured memset) and the host-buffer call (its copies are captured with it).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import SPLIT_CASES, ensure_built, run, to_device
from test_gpu_parity import SMALL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _call(case, d, out, lse, ws, status):
    import block_sparse_fp8_gb300 as bsa

    bsa.prefill(d["q"], d["k_pages"], d["v_pages"], d["q_descale"], d["k_descale"],
                d["v_descale"], d["cu_seqlens_q"], d["seqused_kv"], d["block_table"],
                case.max_q_len, case.max_kv_len, block_mask=d["block_mask"],
                sparse_indices=d["sparse_indices"], sparse_seq_len=d["sparse_seq_len"],
                softmax_scale=case.softmax_scale, p_scale=case.p_scale,
                causal=bool(case.causal), out=out, lse=lse, workspace=ws, dev_status=status,
                k_scale_kind=case.k_scale_kind, v_scale_kind=case.v_scale_kind)


@pytest.mark.parametrize("name", ["indices_empty", "split_long_kv"])
def test_device_call_replays(name):
    import block_sparse_fp8_gb300 as bsa

    params = SMALL.get(name) or SPLIT_CASES[name]
    case = W.make_case(name, **params)
    d = to_device(case)
    ref_out, ref_lse, st = run(case, d)          # eager; also sets the kernel attributes
    assert st == 0
    out, lse = torch.empty_like(ref_out), torch.empty_like(ref_lse)
    ws = torch.empty(max(bsa.workspace_size(bsa.Dims(**case.dims())), 256), dtype=torch.uint8,
                     device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _call(case, d, out, lse, ws, status)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    # new Q values in the captured buffer: the replay follows them
    case2 = W.make_case(name, **{**params, "seed": params["seed"] + 1000})
    d["q"].copy_(torch.from_numpy(case2.q).cuda())
    d["q_descale"].copy_(torch.from_numpy(case2.q_descale).cuda())
    g.replay()
    torch.cuda.synchronize()
    eager_out, eager_lse, st = run(case, d)
    assert st == 0 and int(status.item()) == 0
    assert torch.equal(out, eager_out) and torch.equal(lse, eager_lse)
    assert not torch.equal(out, ref_out)


def test_host_call_replays():
    """The whole end-to-end step -- copies in from pinned host memory, the prefill, copies
    out -- captured from one bsa_fp8_prefill_host call."""
    import block_sparse_fp8_gb300 as bsa

    case = W.make_case("bern_ragged", **SMALL["bern_ragged"])
    ref_out, ref_lse, _ = run(case)
    host = {n: torch.from_numpy(np.ascontiguousarray(getattr(case, n))).pin_memory()
            for n in bsa.TENSOR_NAMES[:-2] if getattr(case, n) is not None}
    host["out"] = torch.zeros((case.T, case.N1, 128), dtype=torch.bfloat16).pin_memory()
    host["lse"] = torch.zeros((case.N1, case.T)).pin_memory()
    dev = {k: torch.empty(v.shape, dtype=v.dtype, device="cuda") for k, v in host.items()}
    ws = torch.empty(max(bsa.workspace_size(bsa.Dims(**case.dims())), 256), dtype=torch.uint8,
                     device="cuda")
    kw = dict(softmax_scale=case.softmax_scale, p_scale=case.p_scale, causal=bool(case.causal),
              workspace=ws, k_scale_kind=case.k_scale_kind, v_scale_kind=case.v_scale_kind)
    bsa.prefill_host(host, dev, case.max_q_len, case.max_kv_len, **kw)   # eager first
    torch.cuda.synchronize()
    assert torch.equal(host["out"], ref_out.cpu()) and torch.equal(host["lse"], ref_lse.cpu())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bsa.prefill_host(host, dev, case.max_q_len, case.max_kv_len, **kw)
    host["out"].zero_()
    host["lse"].zero_()
    dev["out"].zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(host["out"], ref_out.cpu()) and torch.equal(host["lse"], ref_lse.cpu())
    # new host Q: the replay copies it in and the result follows
    case2 = W.make_case("bern_ragged", **{**SMALL["bern_ragged"], "seed": 2101})
    host["q"].copy_(torch.from_numpy(case2.q))
    host["q_descale"].copy_(torch.from_numpy(case2.q_descale))
    g.replay()
    torch.cuda.synchronize()
    case.q, case.q_descale = case2.q, case2.q_descale
    new_out, new_lse, _ = run(case)
    assert torch.equal(host["out"], new_out.cpu()) and torch.equal(host["lse"], new_lse.cpu())
