"""Helpers for the GPU parity tests: upload a workloads.Case, run the library, compare.

Tolerances (from the acceptance rules of the Quant Block Sparse Attention page, section
精度测试, and the exact-result band used for the fp64 formula):
  * O vs the exact fp64 oracle:          |err| <= 0.02 + 0.02 |ref|
  * O vs the e4m3-P emulating oracle:    |err| <= 1e-4 + 0.0078125 |ref|
  * LSE vs either oracle:                |err| <= 2.5e-5 + 0.005 |ref|
with at most 0.5% of the compared elements outside; active-tile lists are bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import block_sparse_fp8_gb300 as bsa

NEG_FLT_MAX = -3.4028234663852886e38

EXACT_ATOL, EXACT_RTOL = 0.02, 0.02
PEMU_ATOL, PEMU_RTOL = 1e-4, 0.0078125
LSE_ATOL, LSE_RTOL = 2.5e-5, 0.005
MAX_OUTSIDE = 0.005

# few (b, h, q-tile) tasks over a long KV: bsa_fp8_prefill cuts each task's active list into
# slices (split-KV) for these
SPLIT_CASES = {
    "split_long_kv": dict(seed=201, q_lens=[256], kv_lens=[8229], N1=2, N2=1, page_size=64,
                          k_scale_kind=1, v_scale_kind=2, mask="bernoulli", keep=0.5),
    "split_chunked": dict(seed=202, q_lens=[384], kv_lens=[16384], N1=4, N2=2, page_size=32,
                          k_scale_kind=1, v_scale_kind=2, mask="local_sink", n_local=2,
                          p_far=0.3),
    "split_dense_noncausal": dict(seed=203, q_lens=[130, 70], kv_lens=[9000, 8300], N1=2,
                                  N2=2, page_size=64, mask="none", causal=0),
}


def ensure_built():
    from block_sparse_fp8_gb300 import _build

    if _build.needs_build():
        _build.build()
    return bsa.lib()


def to_device(case, dev="cuda"):
    t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return dict(q=t(case.q), k_pages=t(case.k_pages), v_pages=t(case.v_pages),
                q_descale=t(case.q_descale), k_descale=t(case.k_descale),
                v_descale=t(case.v_descale), cu_seqlens_q=t(case.cu_seqlens_q),
                seqused_kv=t(case.seqused_kv), block_table=t(case.block_table),
                block_mask=t(case.block_mask), sparse_indices=t(case.sparse_indices),
                sparse_seq_len=t(case.sparse_seq_len))


def run(case, dev_tensors=None, status=True, **kw):
    d = dev_tensors if dev_tensors is not None else to_device(case)
    st = torch.zeros(1, dtype=torch.int32, device="cuda") if status else None
    out, lse = bsa.prefill(
        d["q"], d["k_pages"], d["v_pages"], d["q_descale"], d["k_descale"], d["v_descale"],
        d["cu_seqlens_q"], d["seqused_kv"], d["block_table"], case.max_q_len, case.max_kv_len,
        block_mask=d["block_mask"], sparse_indices=d["sparse_indices"],
        sparse_seq_len=d["sparse_seq_len"], softmax_scale=case.softmax_scale,
        p_scale=case.p_scale, causal=bool(case.causal), dev_status=st,
        k_scale_kind=case.k_scale_kind, v_scale_kind=case.v_scale_kind, **kw)
    torch.cuda.synchronize()
    return out, lse, (int(st.item()) if status else 0)


def dims_of(case):
    return bsa.Dims(**case.dims())


def run_lists(case, dev_tensors=None):
    d = dev_tensors if dev_tensors is not None else to_device(case)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lists, counts = bsa.compact_tiles(d["cu_seqlens_q"], d["seqused_kv"], dims_of(case),
                                      block_mask=d["block_mask"],
                                      sparse_indices=d["sparse_indices"],
                                      sparse_seq_len=d["sparse_seq_len"], dev_status=st)
    torch.cuda.synchronize()
    return lists.cpu().numpy(), counts.cpu().numpy(), int(st.item())


def band_fraction(got, ref, atol, rtol):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bad = ~(np.abs(got - ref) <= atol + rtol * np.abs(ref))
    return float(bad.mean()) if bad.size else 0.0, bad


def check_o(got, ref, atol, rtol, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    frac, bad = band_fraction(got, ref, atol, rtol)
    if frac > MAX_OUTSIDE:
        err = np.abs(np.asarray(got, np.float64) - ref)
        i = np.unravel_index(np.argmax(err - rtol * np.abs(ref)), err.shape)
        raise AssertionError(f"{what}: {frac:.4%} outside atol={atol} rtol={rtol}; worst at {i}:"
                             f" got {got[i]} ref {ref[i]}")
    return frac


def check_lse(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    empty = ref == NEG_FLT_MAX
    assert np.all(got[empty] == np.float32(NEG_FLT_MAX)), f"{what}: empty rows must be -FLT_MAX"
    frac, _ = band_fraction(got[~empty], ref[~empty], LSE_ATOL, LSE_RTOL)
    assert frac <= MAX_OUTSIDE, f"{what}: LSE {frac:.4%} outside"
    return frac


def sample_rows(case, n, seed):
    """(token, head) rows: sequence starts/ends, tile edges, plus a seeded random sample."""
    rng = np.random.default_rng(seed)
    rows = set()
    for b in range(case.B):
        q0, ql = int(case.cu_seqlens_q[b]), case.q_lens[b]
        if ql == 0:
            continue
        for i in {0, 1, 127, 128, ql // 2, ql - 129, ql - 128, ql - 2, ql - 1}:
            if 0 <= i < ql:
                for h in (0, case.N1 - 1, int(rng.integers(case.N1))):
                    rows.add((q0 + i, h))
    while len(rows) < n:
        rows.add((int(rng.integers(case.T)), int(rng.integers(case.N1))))
    return np.array(sorted(rows), dtype=np.int32)
