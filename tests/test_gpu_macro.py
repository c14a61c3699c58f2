"""256-wide macro blocks (dims.tiles_per_step = 2) against the oracle.

The Quant Block Sparse Attention kernel description pairs two sparse 128-token KV blocks into
one 256-wide macro block per online-softmax step, with odd counts, KV tail blocks and empty
tasks handled at the edges.  The oracle's P-emulating mode with group=2 takes the same steps
(consecutive list tiles in pairs, an odd last tile alone); the kernel must sit in the tight
band around it and in the exact band around the formula.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_helpers import (EXACT_ATOL, EXACT_RTOL, NEG_FLT_MAX, PEMU_ATOL, PEMU_RTOL, check_lse,
                         check_o, ensure_built, run, run_lists, to_device)
from test_gpu_parity import SMALL, task_rows, task_sample

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


@pytest.mark.parametrize("name", sorted(SMALL))
def test_macro_block_all_rows(name):
    case = W.make_case(name, **SMALL[name])
    out, lse, st = run(case, tiles_per_step=2)
    assert st == 0
    orc = O.Oracle(case)
    o_pe, _, _ = orc.all_rows(O.PEMU, group=2)
    o_ex, l_ex, _ = orc.all_rows(O.EXACT)
    got = out.float().cpu().numpy().astype(np.float64)
    gl = lse.cpu().numpy().astype(np.float64)
    check_o(got, o_pe, PEMU_ATOL, PEMU_RTOL, f"{name} vs P-emulating, two tiles per step")
    check_lse(gl, l_ex, f"{name} lse")
    emu_out = np.mean(np.abs(o_pe - o_ex) > EXACT_ATOL + EXACT_RTOL * np.abs(o_ex))
    gpu_out = np.mean(np.abs(got - o_ex) > EXACT_ATOL + EXACT_RTOL * np.abs(o_ex))
    print(f"{name}: outside the exact band: kernel {gpu_out:.4%}, P-emulating oracle "
          f"{emu_out:.4%}")
    assert gpu_out <= max(0.005, emu_out + 0.002), (name, gpu_out, emu_out)
    empty = l_ex == NEG_FLT_MAX
    assert np.all(gl[empty] == np.float32(NEG_FLT_MAX))
    assert not got.transpose(1, 0, 2)[empty].any()


def test_macro_block_odd_and_even_counts():
    """Every task length from 1 to 8 tiles (dense causal: Q tile qt has qt + 1 tiles), so odd
    last steps, pairs, and a one-tile task all occur; per-token K, page 32, ragged tail."""
    case = W.make_case("counts", 150, [1000], [1000], 4, 1, 32, W.SCALE_PER_TOKEN_HEAD,
                       W.SCALE_PER_HEAD, "none")
    out, lse, st = run(case, tiles_per_step=2)
    assert st == 0
    orc = O.Oracle(case)
    o_pe, _, _ = orc.all_rows(O.PEMU, group=2)
    o_ex, l_ex, _ = orc.all_rows(O.EXACT)
    got = out.float().cpu().numpy()
    check_o(got, o_pe, PEMU_ATOL, PEMU_RTOL, "counts vs P-emulating, two tiles per step")
    check_o(got, o_ex, EXACT_ATOL, EXACT_RTOL, "counts vs exact")
    check_lse(lse.cpu().numpy(), l_ex, "counts lse")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["prefill_2x8k_h32kv8_bsm50_outliers",
                                  "varlen_4x16k_h64kv8_idx25"])
def test_macro_block_workload(name):
    """Full-size workloads: a seeded 1/32 of whole tasks (every Q tile of every sequence, the
    empty tasks), exact and pair-P-emulating bands; repeated runs agree bit for bit."""
    case = W.make_workload(name)
    d = to_device(case)
    ref_l, ref_c, _ = O.Oracle(case).lists()
    lists, counts, st = run_lists(case, d)
    assert st == 0 and np.array_equal(counts, ref_c) and np.array_equal(lists, ref_l)
    out, lse, st = run(case, d, tiles_per_step=2)
    assert st == 0
    tasks = task_sample(case, seed=11, frac=1 / 32)
    rows = task_rows(case, tasks)
    orc = O.Oracle(case)
    o_ex, l_ex, err = orc.rows(rows, O.EXACT)
    assert err == 0
    got = out.float()[rows[:, 0], rows[:, 1]].cpu().numpy()
    check_o(got, o_ex, EXACT_ATOL, EXACT_RTOL, f"{name} vs exact")
    check_lse(lse[rows[:, 1], rows[:, 0]].cpu().numpy(), l_ex, f"{name} lse")
    prow = task_rows(case, tasks[::4])
    o_pe, _, _ = orc.rows(prow, O.PEMU, group=2)
    check_o(out.float()[prow[:, 0], prow[:, 1]].cpu().numpy(), o_pe, PEMU_ATOL, PEMU_RTOL,
            f"{name} vs P-emulating, two tiles per step")
    o2, l2, st = run(case, d, tiles_per_step=2)
    assert st == 0 and torch.equal(out, o2) and torch.equal(lse, l2)


@pytest.mark.parametrize("tiles_per_step", [1, 2])
def test_grouping_is_the_one_asked_for(tiles_per_step):
    """Two tiles whose maxima rise from the first to the second (s = -0.1, then 0): in one
    step per tile the first tile's P is 256 exactly and O at the last row is the exact
    (2 + e) / (1 + e) = 1.525; in one step per pair the first tile's P rounds from 231.64 to
    224 and O = 736 / (256 (1 + e)) = 1.509 (e = e^-0.1).  The 1% gap is wider than bf16's
    rounding, so the output tells which grouping the kernel ran."""
    from oracle_pins import _rising_tiles_case

    case = _rising_tiles_case(2)
    out, lse, st = run(case, tiles_per_step=tiles_per_step)
    assert st == 0
    orc = O.Oracle(case)
    mine, _, _ = orc.all_rows(O.PEMU, group=tiles_per_step)
    other, _, _ = orc.all_rows(O.PEMU, group=3 - tiles_per_step)
    got = out.float().cpu().numpy()[255, 0]
    assert np.all(np.abs(got - mine[255, 0]) <= 0.004 * np.abs(mine[255, 0]))
    assert np.all(np.abs(got - other[255, 0]) > 0.006 * np.abs(other[255, 0]))


def test_macro_block_longest_supported_kv():
    """Kb = 4096 KV tiles with two list tiles per step: the longest list the one-pipeline kernel
    holds in shared memory (it never splits), sampled rows against the exact formula and the
    pair-P-emulating mode."""
    from gpu_helpers import sample_rows

    case = W.make_case("max_kb", 301, [256], [4096 * 128], 2, 1, 64, W.SCALE_PER_TOKEN_HEAD,
                       W.SCALE_PER_HEAD, "local_sink", n_local=2, p_far=0.01)
    assert case.Kb == 4096
    d = to_device(case)
    out, lse, st = run(case, d, tiles_per_step=2)
    assert st == 0
    rows = sample_rows(case, 96, seed=3)
    orc = O.Oracle(case)
    o_ex, l_ex, err = orc.rows(rows, O.EXACT)
    o_pe, _, _ = orc.rows(rows, O.PEMU, group=2)
    assert err == 0
    got = out.float()[rows[:, 0], rows[:, 1]].cpu().numpy()
    check_o(got, o_ex, EXACT_ATOL, EXACT_RTOL, "max Kb, two tiles per step, vs exact")
    check_o(got, o_pe, PEMU_ATOL, PEMU_RTOL, "max Kb vs P-emulating, two tiles per step")
    check_lse(lse[rows[:, 1], rows[:, 0]].cpu().numpy(), l_ex, "max Kb lse, two tiles per step")
