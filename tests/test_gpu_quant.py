"""The quantise step on the GPU against the oracle: bit-exact codes and descales.

bsa_fp8_quantize_rows (Q [T, N1, 128] bf16 -> e4m3 + q_descale) and bsa_fp8_append_kv (new
K/V tokens into the paged cache) follow the FlashMLA page's quantisation rule (scale =
amax / 448, stored value e4m3(x / scale)), and under the UE8M0 rule the same page's cast of
the scale up to a power of two; codes are integers, so the bar is equality.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_helpers import ensure_built
from oracle_pins import _quant_rows_fixture, bf16_bits_to_f32, f32_to_bf16_bits

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _rows(seed, n, scale=1.0):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((n, 128)) * scale).astype(np.float32)
    if n > 4:
        x[n // 2] = 0.0
        x[1] *= 1e-6
    return f32_to_bf16_bits(x)


RULES = [O.DESCALE_AMAX, O.DESCALE_UE8M0]


def _gpu_quantize(xb, rule=O.DESCALE_AMAX):
    import block_sparse_fp8_gb300 as bsa

    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    codes, desc = bsa.quantize_rows(x, rule=rule)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), desc.cpu().numpy()


def _check_rows(xb, rule):
    codes, desc = _gpu_quantize(xb, rule)
    o_codes, o_desc = O.quantize_rows(xb, rule=rule)
    assert np.array_equal(desc.view(np.uint32), o_desc.view(np.uint32)), \
        f"{int((desc.view(np.uint32) != o_desc.view(np.uint32)).sum())} descales differ"
    assert np.array_equal(codes, o_codes), f"{int((codes != o_codes).sum())} codes differ"


@pytest.mark.parametrize("rule", RULES)
@pytest.mark.parametrize("n", [1, 15, 16, 17, 37, 1003])
def test_quantize_rows_bit_exact(n, rule):
    _need_gpu()
    _check_rows(_rows(100 + n, n, scale=3.0), rule)


@pytest.mark.parametrize("rule", RULES)
def test_quantize_rows_edge_values(rule):
    _need_gpu()
    _check_rows(_quant_rows_fixture(), rule)


def test_quantize_rows_ue8m0_subnormal_descales():
    """Rows whose amax / 448 is an fp32 subnormal (amax down to the smallest bf16, 2^-133),
    powers of two among them, and rows just above and at powers of two times 448."""
    _need_gpu()
    rows = []
    for bits in (0x0001, 0x0002, 0x0003, 0x0005, 0x0010, 0x0011, 0x007F, 0x0080, 0x0081, 0x00FF,
                 0x0100, 0x0123, 0x03FF, 0x0400, 0x0401):
        r = np.zeros(128, dtype=np.uint16)
        r[bits % 128] = bits
        r[(bits + 5) % 128] = bits // 2 | 0x8000        # a smaller negative value
        rows.append(r)
    for e in (-20, -1, 0, 1, 7, 40):
        for m in (448.0, 450.0, 446.0):
            rows.append(f32_to_bf16_bits(np.full(128, m * 2.0 ** e, dtype=np.float32) *
                                         np.linspace(-1, 1, 128, dtype=np.float32)))
    _check_rows(np.stack(rows), O.DESCALE_UE8M0)


@pytest.mark.parametrize("rule", RULES)
def test_quantize_rows_extreme_scales(rule):
    """Rows whose descale lies outside and at the edges of the range where the kernel uses the
    corrected-reciprocal quotient (2^-90 .. 2^90) and so divides directly."""
    _need_gpu()
    rng = np.random.default_rng(31)
    base = rng.standard_normal((8, 128)).astype(np.float32)
    base[:, 0] = 448.0                                     # amax 448 * 2^k -> descale 2^k
    exps = [-110, -91, -90, -89, 89, 90, 91, 110]
    x = np.stack([base[i] * np.float32(2.0 ** e) for i, e in enumerate(exps)])
    _check_rows(f32_to_bf16_bits(x), rule)
    # non-power-of-two descales near both edges
    x2 = np.stack([base[i] * np.float32(1.37 * 2.0 ** e) for i, e in enumerate(exps)])
    _check_rows(f32_to_bf16_bits(x2), rule)


def test_quantize_rows_full_q_of_the_bench_workload():
    """Q of the 2 x 8192-token, 32-head workload: 524,288 rows, every code compared."""
    _need_gpu()
    T, N1 = 16384, 32
    rng = np.random.default_rng(7)
    x = rng.standard_normal((T, N1, 128)).astype(np.float32)
    ch = rng.choice(N1 * 128, size=41, replace=False)             # 1% outlier channels x8
    x.reshape(T, -1)[:, ch] *= 8.0
    xb = f32_to_bf16_bits(x)
    codes, desc = _gpu_quantize(xb)
    o_codes, o_desc = O.quantize_rows(xb)
    assert desc.shape == (T, N1)
    assert np.array_equal(desc.view(np.uint32), o_desc.view(np.uint32))
    assert np.array_equal(codes, o_codes), f"{int((codes != o_codes).sum())} codes differ"


def test_quantize_rows_zero_rows_is_noop():
    _need_gpu()
    import block_sparse_fp8_gb300 as bsa

    st = bsa.lib().bsa_fp8_quantize_rows(None, 0, None, None, None)
    assert st == 0
    assert bsa.lib().bsa_fp8_quantize_rows(None, -1, None, None, None) == 1


def _append_case(ps, k_kind, v_kind, seed=5):
    rng = np.random.default_rng(seed)
    B, N2 = 3, 4
    cache_len = np.array([0, 37, 100], dtype=np.int32)
    n_new = np.array([50, 1, 129], dtype=np.int32)
    cu_new = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    L = int(max(-(-(cache_len + n_new) // ps)))
    P = B * L + 3
    perm = rng.permutation(P).astype(np.int32)
    bt = perm[: B * L].reshape(B, L).copy()
    T = int(cu_new[-1])
    kb = f32_to_bf16_bits(rng.standard_normal((T, N2, 128)).astype(np.float32) * 2.0)
    vb = f32_to_bf16_bits(rng.standard_normal((T, N2, 128)).astype(np.float32))
    kp = np.full((P, N2, ps, 128), 0x55, dtype=np.uint8)
    vp = np.full((P, N2, ps, 128), 0x55, dtype=np.uint8)
    kd = np.full((P, N2, ps), -7.0, dtype=np.float32)
    k_scale = np.array([0.0123], dtype=np.float32)
    v_scale = (np.array([0.01, 0.02, 0.005, 0.04], dtype=np.float32)
               if v_kind == W.SCALE_PER_HEAD else np.array([0.01], dtype=np.float32))
    return dict(kb=kb, vb=vb, cu_new=cu_new, cache_len=cache_len, bt=bt, kp=kp, vp=vp, kd=kd,
                k_scale=k_scale, v_scale=v_scale, k_kind=k_kind, v_kind=v_kind)


def _run_append(c, nhd=False, rule=O.DESCALE_AMAX):
    """Runs the append; with nhd the cache is held as NHD pages and returned as HND."""
    import block_sparse_fp8_gb300 as bsa

    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    perm = (0, 2, 1, 3)
    kp = t(c["kp"].transpose(perm) if nhd else c["kp"])
    vp = t(c["vp"].transpose(perm) if nhd else c["vp"])
    kd = t(c["kd"])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsa.append_kv(bf(c["kb"]), bf(c["vb"]), t(c["cu_new"]), t(c["cache_len"]), t(c["bt"]), kp, vp,
                  k_descale=kd, k_scale=t(c["k_scale"]), v_scale=t(c["v_scale"]),
                  k_scale_kind=c["k_kind"], v_scale_kind=c["v_kind"], dev_status=st,
                  kv_layout=bsa.KV_NHD if nhd else bsa.KV_HND, k_descale_rule=rule)
    torch.cuda.synchronize()
    kp, vp = kp.cpu().numpy(), vp.cpu().numpy()
    if nhd:
        kp, vp = kp.transpose(perm), vp.transpose(perm)
    return kp, vp, kd.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("nhd", [False, True])
@pytest.mark.parametrize("ps", [32, 64])
@pytest.mark.parametrize("kinds", [(W.SCALE_PER_TOKEN_HEAD, W.SCALE_PER_HEAD, O.DESCALE_AMAX),
                                   (W.SCALE_PER_TOKEN_HEAD, W.SCALE_PER_HEAD, O.DESCALE_UE8M0),
                                   (W.SCALE_PER_TENSOR, W.SCALE_PER_TENSOR, O.DESCALE_AMAX)])
def test_append_kv_bit_exact(ps, kinds, nhd):
    _need_gpu()
    c = _append_case(ps, *kinds[:2])
    kp, vp, kd, st = _run_append(c, nhd, rule=kinds[2])
    okp, ovp, okd, err = O.append_kv(c["kb"], c["vb"], c["cu_new"], c["cache_len"], c["bt"],
                                     c["kp"], c["vp"], c["kd"], c["k_kind"], c["v_kind"],
                                     c["k_scale"], c["v_scale"], k_descale_rule=kinds[2])
    assert st == 0 and err == 0
    assert np.array_equal(kp, okp), f"{int((kp != okp).sum())} K bytes differ"
    assert np.array_equal(vp, ovp), f"{int((vp != ovp).sum())} V bytes differ"
    assert np.array_equal(kd.view(np.uint32), okd.view(np.uint32))


def test_append_kv_missing_page_reported_and_skipped():
    _need_gpu()
    c = _append_case(32, W.SCALE_PER_TOKEN_HEAD, W.SCALE_PER_HEAD)
    c["bt"] = c["bt"].copy()
    c["bt"][2, 4] = -1                                   # positions 128..159 of sequence 2
    kp, vp, kd, st = _run_append(c)
    okp, ovp, okd, err = O.append_kv(c["kb"], c["vb"], c["cu_new"], c["cache_len"], c["bt"],
                                     c["kp"], c["vp"], c["kd"], c["k_kind"], c["v_kind"],
                                     c["k_scale"], c["v_scale"])
    assert st == 2 and err == O.ERR_BAD_PAGE                # BSA_DEV_BAD_PAGE
    assert np.array_equal(kp, okp) and np.array_equal(vp, ovp)
    assert np.array_equal(kd.view(np.uint32), okd.view(np.uint32))


@pytest.mark.parametrize("rule", RULES)
def test_quantised_inputs_feed_the_prefill(rule):
    """bf16 Q/K/V -> quantise step on the GPU -> prefill; the result matches the oracle run on
    the same quantised inputs (the formats of the two steps agree end to end), with the
    descales of Q and K plain or rounded up to powers of two."""
    _need_gpu()
    import block_sparse_fp8_gb300 as bsa
    from gpu_helpers import EXACT_ATOL, EXACT_RTOL, MAX_OUTSIDE, band_fraction, to_device

    ps, N1, N2 = 64, 8, 2
    q_len = kv_len = 300
    base = W.make_case("quant_e2e", 41, [q_len], [kv_len], N1, N2, ps, W.SCALE_PER_TOKEN_HEAD,
                       W.SCALE_PER_HEAD, "bernoulli", keep=0.6)
    rng = np.random.default_rng(8)
    qb = f32_to_bf16_bits(rng.standard_normal((q_len, N1, 128)).astype(np.float32))
    kb = f32_to_bf16_bits(rng.standard_normal((kv_len, N2, 128)).astype(np.float32))
    vb = f32_to_bf16_bits(rng.standard_normal((kv_len, N2, 128)).astype(np.float32))
    vx = bf16_bits_to_f32(vb)
    v_scale = (np.abs(vx).max(axis=(0, 2)) / np.float32(448)).astype(np.float32)
    P = base.k_pages.shape[0]
    c = dict(kb=kb, vb=vb, cu_new=np.array([0, kv_len], np.int32),
             cache_len=np.array([0], np.int32), bt=base.block_table,
             kp=np.zeros((P, N2, ps, 128), np.uint8), vp=np.zeros((P, N2, ps, 128), np.uint8),
             kd=np.zeros((P, N2, ps), np.float32), k_scale=np.array([1.0], np.float32),
             v_scale=v_scale, k_kind=W.SCALE_PER_TOKEN_HEAD, v_kind=W.SCALE_PER_HEAD)
    kp, vp, kd, st = _run_append(c, rule=rule)
    q8, qd = _gpu_quantize(qb.reshape(-1, 128), rule)
    assert st == 0
    if rule == O.DESCALE_UE8M0:
        lg = np.log2(np.concatenate([qd.ravel(), kd[kd > 0]]).astype(np.float64))
        assert np.all(lg == np.round(lg))
    base.q, base.q_descale = q8.reshape(q_len, N1, 128), qd.reshape(q_len, N1)
    base.k_pages, base.v_pages, base.k_descale, base.v_descale = kp, vp, kd, v_scale
    d = to_device(base)
    out, lse = bsa.prefill(d["q"], d["k_pages"], d["v_pages"], d["q_descale"], d["k_descale"],
                           d["v_descale"], d["cu_seqlens_q"], d["seqused_kv"], d["block_table"],
                           base.max_q_len, base.max_kv_len, block_mask=d["block_mask"],
                           softmax_scale=base.softmax_scale, p_scale=base.p_scale, causal=True)
    torch.cuda.synchronize()
    ref, ref_lse, err = O.Oracle(base).all_rows(O.EXACT)
    assert err == 0
    frac, _ = band_fraction(out.float().cpu().numpy(), ref, EXACT_ATOL, EXACT_RTOL)
    assert frac <= MAX_OUTSIDE
