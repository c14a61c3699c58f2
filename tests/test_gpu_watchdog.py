"""The bounded waits inside the prefill kernel, made to run out on a healthy workload.

bsa_fp8_set_wait_limit_ns lowers the limit of every wait for later launches.  At one
microsecond, waits that are legitimate but longer (a producer waiting for a task slot, the
MMA thread waiting for P) run out: the launch must set BSA_DEV_TIMEOUT, let every copy and
tensor-core operation it issued finish, free its tensor memory and return.  Nothing is
withheld or broken on purpose; the inputs are a normal problem.  Afterwards, with the default
limit, the same problem must give exactly the result it gave before the aborted launches --
the context survived and nothing of the aborted launches leaked into later ones.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_helpers import (EXACT_ATOL, EXACT_RTOL, check_lse, check_o, ensure_built, run,
                         sample_rows, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


CASES = {
    # about seven tasks per pipeline of ~16 tiles: producers wait for task slots
    "per_token_k": dict(seed=140, q_lens=[8192], kv_lens=[8192], N1=32, N2=8, page_size=64,
                        k_scale_kind=W.SCALE_PER_TOKEN_HEAD, v_scale_kind=W.SCALE_PER_HEAD,
                        mask="bernoulli", keep=0.5),
    # index lists, page 32, ragged sequences
    "indices_p32": dict(seed=141, q_lens=[3000, 1500, 700], kv_lens=[3000, 1600, 700], N1=16,
                        N2=4, page_size=32, k_scale_kind=W.SCALE_PER_TOKEN_HEAD,
                        v_scale_kind=W.SCALE_PER_HEAD, mask="indices", sparse_frac=0.4,
                        n_empty=5),
}


@pytest.mark.parametrize("tiles_per_step", [1, 2])
@pytest.mark.parametrize("name", sorted(CASES))
def test_short_wait_limit_aborts_and_the_context_survives(name, tiles_per_step):
    """Both kernels: one 128-token tile per online-softmax step, and 256-wide macro blocks."""
    import block_sparse_fp8_gb300 as bsa

    case = W.make_case(name, **CASES[name])
    d = to_device(case)
    ref_out, ref_lse, st = run(case, d, tiles_per_step=tiles_per_step)
    assert st == 0
    rows = sample_rows(case, 2048, seed=9)
    o_ex, l_ex, err = O.Oracle(case).rows(rows, O.EXACT)
    assert err == 0
    check_o(ref_out.float()[rows[:, 0], rows[:, 1]].cpu().numpy(), o_ex, EXACT_ATOL, EXACT_RTOL,
            f"{name} before")
    bsa.set_wait_limit_ns(1000)
    try:
        for i in range(3):
            _, _, st = run(case, d, tiles_per_step=tiles_per_step)
            assert st & bsa.DEV_TIMEOUT, f"launch {i}: no wait ran out (status {st})"
            assert st & ~bsa.DEV_TIMEOUT == 0, f"launch {i}: status {st}"
    finally:
        bsa.set_wait_limit_ns(0)
    out, lse, st = run(case, d, tiles_per_step=tiles_per_step)
    assert st == 0
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    check_lse(lse[rows[:, 1], rows[:, 0]].cpu().numpy(), l_ex, f"{name} after")
