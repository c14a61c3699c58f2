"""Pins for the CPU oracle: checks against things other than the oracle itself.

Every pin takes a loaded oracle library (``oracle.load(path)``) so that the same pins can be
run against deliberately broken builds of the oracle (tests/test_oracle_mutants.py).

What the pins compare against:
  * the OCP E4M3 table (tests/golden/e4m3_points.json) and PyTorch's float8_e4m3fn cast;
  * brute-force dense softmax attention written as matrix algebra (numpy + scipy logsumexp)
    over page-free, token-ordered copies of K and V, with the tile mask expanded to a dense
    [q, kv] boolean matrix -- none of the oracle's page, list or kend logic;
  * closed forms (K = 0 gives uniform weights; constant V; the first causal row);
  * invariances the method must have (masked tiles never read, page permutation, index list
    vs block mask, GQA replication, p_scale independence of the exact result, zero-filled
    tails, empty tasks);
  * a hand-derived fixed-P-scale example for the e4m3-emulating mode.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
from scipy.special import logsumexp

import oracle as O
import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
NEG_FLT_MAX = -3.4028234663852886e38


def _oracle(case, lib):
    return O.Oracle(case, lib=lib)


def torch_decode(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn)
    return t.to(torch.float32).numpy().astype(np.float64)


# ----------------------------------------------------------------------------------------
# brute-force reference (independent of the oracle's page / list code)
# ----------------------------------------------------------------------------------------

def tile_sets(case):
    """Python sets of enabled KV tiles per (b, h, qt) straight from the mask inputs."""
    B, N1, Qb, Kb = case.B, case.N1, case.Qb, case.Kb
    sets = {}
    for b in range(B):
        for h in range(N1):
            for qt in range(Qb):
                if case.block_mask is not None:
                    sets[b, h, qt] = {t for t in range(Kb) if case.block_mask[b, h, qt, t]}
                elif case.sparse_indices is not None:
                    n = int(case.sparse_seq_len[b, h, qt])
                    sets[b, h, qt] = {int(t) for t in case.sparse_indices[b, h, qt, :n]}
                else:
                    sets[b, h, qt] = set(range(Kb))
    return sets


def brute_force(case):
    """Dense softmax attention with an explicit [q, kv] allowed-matrix; O [T,N1,D], LSE [N1,T]."""
    k_codes = case.meta["k_codes"]
    v_codes = case.meta["v_codes"]
    Q = torch_decode(case.q) * case.q_descale[..., None].astype(np.float64)
    K = torch_decode(k_codes)
    if case.k_scale_kind == W.SCALE_PER_TOKEN_HEAD:
        K = K * case.meta["k_descale_tok"][..., None].astype(np.float64)
    else:
        K = K * float(case.k_descale[0])
    V = torch_decode(v_codes)
    if case.v_scale_kind == W.SCALE_PER_HEAD:
        V = V * case.v_descale[None, :, None].astype(np.float64)
    else:
        V = V * float(case.v_descale[0])
    G = case.N1 // case.N2
    sets = tile_sets(case)
    out = np.zeros((case.T, case.N1, W.HEAD_DIM))
    lse = np.full((case.N1, case.T), NEG_FLT_MAX)
    kv0 = 0
    for b in range(case.B):
        ql, kl = case.q_lens[b], case.kv_lens[b]
        q0 = int(case.cu_seqlens_q[b])
        i = np.arange(ql)[:, None]
        j = np.arange(kl)[None, :]
        for h in range(case.N1):
            g = h // G
            S = case.softmax_scale * (Q[q0:q0 + ql, h] @ K[kv0:kv0 + kl, g].T)
            allowed = np.ones((ql, kl), dtype=bool)
            if case.causal:
                allowed &= j <= i + (kl - ql)
            tm = np.zeros((max(case.Qb, 1), max(case.Kb, 1)), dtype=bool)
            for qt in range(case.Qb):
                for t in sets[b, h, qt]:
                    if 0 <= t < case.Kb:
                        tm[qt, t] = True
            allowed &= tm[i // W.TILE, j // W.TILE]
            S = np.where(allowed, S, -np.inf)
            has = allowed.any(axis=1)
            if has.any():
                ls = logsumexp(S[has], axis=1)
                P = np.exp(S[has] - ls[:, None])
                out[q0 + np.nonzero(has)[0], h] = P @ V[kv0:kv0 + kl, g]
                lse[h, q0 + np.nonzero(has)[0]] = ls
        kv0 += kl
    return out, lse


def _close(a, b, tol=1e-9):
    a = np.asarray(a)
    b = np.asarray(b)
    assert a.shape == b.shape, (a.shape, b.shape)
    err = np.abs(a - b)
    lim = tol * (1.0 + np.abs(b))
    assert np.all(err <= lim), f"max err {err.max()} at {np.unravel_index(err.argmax(), err.shape)}"


# ----------------------------------------------------------------------------------------
# e4m3 codec
# ----------------------------------------------------------------------------------------

def pin_e4m3_spec_points(lib):
    with open(os.path.join(GOLDEN, "e4m3_points.json")) as f:
        pts = json.load(f)["points"]
    for p in pts:
        c = int(p["code"], 16)
        v = lib.oracle_e4m3_decode(c)
        if p["value"] == "nan":
            assert math.isnan(v), p
        else:
            assert v == p["value"] and math.copysign(1, v) == math.copysign(1, p["value"]), (p, v)


def pin_e4m3_decode_all_codes(lib):
    ref = torch_decode(np.arange(256, dtype=np.uint8))
    for c in range(256):
        v = lib.oracle_e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c] and math.copysign(1, v) == math.copysign(1, ref[c]), (c, v, ref[c])


def pin_e4m3_encode(lib):
    # every finite code round-trips
    for c in range(256):
        v = lib.oracle_e4m3_decode(c)
        if not math.isnan(v):
            assert lib.oracle_e4m3_encode(v) == c, (hex(c), v)
    # midpoints between neighbouring codes (ties) and random values agree with torch's RNE
    fin = sorted({torch_decode(np.array([c], np.uint8))[0] for c in range(256)} - {float("nan")})
    fin = [x for x in fin if not math.isnan(x)]
    mids = [(a + b) / 2 for a, b in zip(fin[:-1], fin[1:])]
    rng = np.random.default_rng(7)
    rnd = list(rng.standard_normal(3000) * 40) + list(rng.standard_normal(1000) * 0.01)
    xs = np.array(mids + rnd + [447.9, 440.0, 1e-30, -1e-30], dtype=np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for x, r in zip(xs, ref):
        assert lib.oracle_e4m3_encode(float(x)) == r, (float(x), hex(r))
    # saturation (the cast used for P is satfinite)
    assert lib.oracle_e4m3_encode(1e6) == 0x7E
    assert lib.oracle_e4m3_encode(-1e6) == 0xFE
    assert lib.oracle_e4m3_encode(float("inf")) == 0x7E
    assert lib.oracle_e4m3_encode(470.0) == 0x7E
    assert lib.oracle_e4m3_encode(float("nan")) & 0x7F == 0x7F


# ----------------------------------------------------------------------------------------
# lists
# ----------------------------------------------------------------------------------------

def _small_cases():
    return [
        W.make_case("bern", 11, [300, 129, 1], [300, 129, 1], 4, 2, 64,
                    W.SCALE_PER_TOKEN_HEAD, W.SCALE_PER_HEAD, "bernoulli", keep=0.5,
                    keep_logical=True),
        W.make_case("chunk", 12, [200], [700], 2, 1, 32, mask="local_sink", n_local=1,
                    p_far=0.3, keep_logical=True),
        W.make_case("idx", 13, [520, 260], [520, 260], 4, 1, 32, W.SCALE_PER_TOKEN_HEAD,
                    W.SCALE_PER_HEAD, "indices", sparse_frac=0.5, n_empty=1, keep_logical=True),
        W.make_case("dense", 14, [257], [257], 2, 2, 64, mask="none", keep_logical=True),
        W.make_case("qlong", 15, [300], [170], 2, 1, 64, mask="ones", keep_logical=True),
        W.make_case("noncausal", 16, [200, 140], [330, 140], 4, 2, 32, W.SCALE_PER_TOKEN_HEAD,
                    W.SCALE_PER_HEAD, "ones", causal=0, keep_logical=True),
        # a sequence with no KV tokens at all: every row of it sees no key
        W.make_case("kv0", 17, [200, 130], [0, 300], 4, 2, 64, W.SCALE_PER_TOKEN_HEAD,
                    W.SCALE_PER_HEAD, "bernoulli", keep=0.6, keep_logical=True),
    ]


_CASES = None


def small_cases():
    global _CASES
    if _CASES is None:
        _CASES = _small_cases()
    return _CASES


def pin_lists_vs_sets(lib):
    """A tile is listed iff it is enabled and holds a key some row of the task can see."""
    for case in small_cases():
        lists, counts, err = _oracle(case, lib).lists()
        assert err == 0
        sets = tile_sets(case)
        for b in range(case.B):
            ql, kl = case.q_lens[b], case.kv_lens[b]
            for h in range(case.N1):
                for qt in range(case.Qb):
                    rows = range(qt * W.TILE, min(ql, qt * W.TILE + W.TILE))
                    want = []
                    for t in sorted(sets[b, h, qt]):
                        if not 0 <= t < case.Kb:
                            continue
                        keys = range(t * W.TILE, min(kl, t * W.TILE + W.TILE))
                        if any((not case.causal) or k <= r + (kl - ql) for r in rows for k in keys):
                            want.append(t)
                    got = lists[b, h, qt, :counts[b, h, qt]].tolist()
                    assert got == want, (case.name, b, h, qt, got, want)
                    assert np.all(lists[b, h, qt, counts[b, h, qt]:] == -1)


# ----------------------------------------------------------------------------------------
# attention results
# ----------------------------------------------------------------------------------------

def pin_brute_force(lib):
    for case in small_cases():
        o, lse, err = _oracle(case, lib).all_rows(O.EXACT)
        assert err == 0
        bo, blse = brute_force(case)
        _close(o, bo)
        _close(lse, blse)


def pin_ones_equals_dense(lib):
    a = W.make_case("a", 21, [300, 90], [300, 400], 4, 2, 64, W.SCALE_PER_TOKEN_HEAD,
                    W.SCALE_PER_HEAD, "ones")
    b = W.make_case("b", 21, [300, 90], [300, 400], 4, 2, 64, W.SCALE_PER_TOKEN_HEAD,
                    W.SCALE_PER_HEAD, "none")
    oa, la, _ = _oracle(a, lib).all_rows()
    ob, lb, _ = _oracle(b, lib).all_rows()
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def _uniform_k_case(seed, pemu_exact=True):
    c = W.make_case("k0", seed, [260, 70], [260, 330], 4, 2, 32, mask="bernoulli", keep=0.6,
                    keep_logical=True)
    c.k_pages[:] = 0
    return c


def pin_closed_form_zero_k(lib):
    """K = 0: every visible key has weight 1/|A_i|, LSE = ln |A_i| (both modes)."""
    case = _uniform_k_case(31)
    sets = tile_sets(case)
    V = torch_decode(case.meta["v_codes"]) * float(case.v_descale[0])
    G = case.N1 // case.N2
    for mode in (O.EXACT, O.PEMU):
        o, lse, _ = _oracle(case, lib).all_rows(mode)
        kv0 = 0
        for b in range(case.B):
            ql, kl = case.q_lens[b], case.kv_lens[b]
            q0 = int(case.cu_seqlens_q[b])
            for h in range(case.N1):
                for i in range(ql):
                    vis = [j for j in range(kl) if j <= i + kl - ql and (j // 128) in sets[b, h, i // 128]]
                    if not vis:
                        assert lse[h, q0 + i] == NEG_FLT_MAX and not o[q0 + i, h].any()
                        continue
                    want = V[[kv0 + j for j in vis], h // G].mean(axis=0)
                    _close(o[q0 + i, h], want, 1e-12)
                    assert abs(lse[h, q0 + i] - math.log(len(vis))) < 1e-12
            kv0 += kl


def pin_closed_form_const_v(lib):
    """Every V row equal to c gives O_i = c * v_descale for every row with a visible key."""
    case = W.make_case("cv", 32, [200], [200], 2, 1, 64, W.SCALE_PER_TOKEN_HEAD,
                       W.SCALE_PER_HEAD, "bernoulli", keep=0.7)
    row = np.arange(128, dtype=np.uint8) % 0x70          # a fixed pattern of finite codes
    case.v_pages[:] = row
    want = torch_decode(row) * float(case.v_descale[0])
    o, lse, _ = _oracle(case, lib).all_rows(O.EXACT)
    for tok in range(case.T):
        for h in range(case.N1):
            _close(o[tok, h], want, 1e-12)


def pin_first_row(lib):
    """Row 0 of a sequence with kv_len = q_len sees only key 0: O_0 = V^_0, LSE_0 = s_00."""
    case = W.make_case("r0", 33, [150, 40], [150, 40], 4, 2, 64, W.SCALE_PER_TOKEN_HEAD,
                       W.SCALE_PER_HEAD, "bernoulli", keep_logical=True)
    o, lse, _ = _oracle(case, lib).all_rows()
    Q = torch_decode(case.q) * case.q_descale[..., None]
    K = torch_decode(case.meta["k_codes"]) * case.meta["k_descale_tok"][..., None]
    V = torch_decode(case.meta["v_codes"]) * case.v_descale[None, :, None]
    kv0 = 0
    for b in range(case.B):
        q0 = int(case.cu_seqlens_q[b])
        for h in range(case.N1):
            g = h // 2
            _close(o[q0, h], V[kv0, g], 1e-12)
            s00 = case.softmax_scale * float(Q[q0, h] @ K[kv0, g])
            assert abs(lse[h, q0] - s00) < 1e-12 * (1 + abs(s00))
        kv0 += case.kv_lens[b]


def pin_masked_tiles_never_read(lib):
    """Pages of tiles that no task of a KV group enables are filled with e4m3 NaN: O unchanged."""
    case = W.make_case("poison", 34, [256], [1024], 4, 2, 64, mask="local_sink", n_local=0,
                       p_far=0.0)
    o_ref, l_ref, _ = _oracle(case, lib).all_rows()
    used = set()
    G = case.N1 // case.N2
    for (b, h, qt), s in tile_sets(case).items():
        used |= {(h // G, t) for t in s}
    ps = case.page_size
    n_poison = 0
    for g in range(case.N2):
        for t in range(case.Kb):
            if (g, t) in used:
                continue
            for lp in range(t * 128 // ps, (t + 1) * 128 // ps):
                pg = case.block_table[0, lp]
                case.k_pages[pg, g] = 0x7F
                case.v_pages[pg, g] = 0x7F
                n_poison += 1
    assert n_poison > 0
    o, l, _ = _oracle(case, lib).all_rows()
    assert np.array_equal(o, o_ref) and np.array_equal(l, l_ref)


def pin_page_permutation(lib):
    kw = dict(q_lens=[300, 77], kv_lens=[300, 500], N1=4, N2=2, page_size=32,
              k_scale_kind=W.SCALE_PER_TOKEN_HEAD, v_scale_kind=W.SCALE_PER_HEAD)
    a = W.make_case("perm", 35, identity_pages=True, **kw)
    b = W.make_case("perm", 35, identity_pages=False, **kw)
    assert not np.array_equal(a.block_table, b.block_table)
    oa, la, _ = _oracle(a, lib).all_rows()
    ob, lb, _ = _oracle(b, lib).all_rows()
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def pin_indices_equal_mask(lib):
    m = W.make_case("m", 36, [400, 130], [400, 130], 4, 2, 64, mask="bernoulli", keep=0.4)
    rng = np.random.default_rng(36)
    idx = np.full(m.block_mask.shape, -1, dtype=np.int32)
    n = np.zeros(m.block_mask.shape[:3], dtype=np.int32)
    for key in np.ndindex(*m.block_mask.shape[:3]):
        on = np.nonzero(m.block_mask[key])[0]
        rng.shuffle(on)
        idx[key][:len(on)] = on
        n[key] = len(on)
    s = W.make_case("m", 36, [400, 130], [400, 130], 4, 2, 64, mask="none")
    s.sparse_indices, s.sparse_seq_len = idx, n
    om, lm = _oracle(m, lib), _oracle(s, lib)
    la, ca, _ = om.lists()
    lb, cb, _ = lm.lists()
    assert np.array_equal(la, lb) and np.array_equal(ca, cb)
    oa, xa, _ = om.all_rows()
    ob, xb, _ = lm.all_rows()
    assert np.array_equal(oa, ob) and np.array_equal(xa, xb)


def pin_gqa_replicated(lib):
    """N1 = 4, N2 = 2 equals N1 = 4, N2 = 4 with KV heads (0, 0, 1, 1)."""
    g2 = W.make_case("g", 37, [260], [260], 4, 2, 64, W.SCALE_PER_TOKEN_HEAD, W.SCALE_PER_HEAD,
                     "bernoulli")
    g1 = W.make_case("g", 37, [260], [260], 4, 2, 64, W.SCALE_PER_TOKEN_HEAD, W.SCALE_PER_HEAD,
                     "bernoulli")
    rep = [0, 0, 1, 1]
    g1.N2 = 4
    g1.k_pages = np.ascontiguousarray(g2.k_pages[:, rep])
    g1.v_pages = np.ascontiguousarray(g2.v_pages[:, rep])
    g1.k_descale = np.ascontiguousarray(g2.k_descale[:, rep])
    g1.v_descale = np.ascontiguousarray(g2.v_descale[rep])
    oa, la, _ = _oracle(g2, lib).all_rows()
    ob, lb, _ = _oracle(g1, lib).all_rows()
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def pin_exact_independent_of_pscale(lib):
    a = W.make_case("p", 38, [200], [200], 2, 1, 64, mask="bernoulli")
    b = W.make_case("p", 38, [200], [200], 2, 1, 64, mask="bernoulli", p_scale=100.5)
    oa, la, _ = _oracle(a, lib).all_rows()
    ob, lb, _ = _oracle(b, lib).all_rows()
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def pin_empty_tasks(lib):
    case = W.make_case("e", 39, [300, 200], [300, 200], 4, 1, 32, mask="indices",
                       sparse_frac=0.5, n_empty=3)
    _, counts, _ = _oracle(case, lib).lists()
    o, lse, _ = _oracle(case, lib).all_rows(O.EXACT)
    o2, lse2, _ = _oracle(case, lib).all_rows(O.PEMU)
    empties = 0
    for b in range(case.B):
        q0 = int(case.cu_seqlens_q[b])
        for h in range(case.N1):
            for qt in range(-(-case.q_lens[b] // 128)):
                if case.sparse_seq_len[b, h, qt] == 0:
                    empties += 1
                    assert counts[b, h, qt] == 0
                    r = slice(q0 + qt * 128, q0 + min(case.q_lens[b], qt * 128 + 128))
                    for oo, ll in ((o, lse), (o2, lse2)):
                        assert not oo[r, h].any()
                        assert np.all(ll[h, r] == NEG_FLT_MAX)
    assert empties == 3


def pin_tail_slots_unused(lib):
    kw = dict(q_lens=[300, 100], kv_lens=[300, 100], N1=2, N2=1, page_size=64,
              k_scale_kind=W.SCALE_PER_TOKEN_HEAD, v_scale_kind=W.SCALE_PER_HEAD, mask="ones")
    a = W.make_case("t", 40, **kw)
    b = W.make_case("t", 40, tail_fill=1.0, **kw)
    assert not np.array_equal(a.k_pages, b.k_pages)
    for mode in (O.EXACT, O.PEMU):
        oa, la, _ = _oracle(a, lib).all_rows(mode)
        ob, lb, _ = _oracle(b, lib).all_rows(mode)
        assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def _two_key_case():
    """T = 2, one head; q = e0, k_0 = 0, k_1 = -e0, v_0 = 1, v_1 = 2, softmax_scale = 0.1."""
    q = np.zeros((2, 1, 128), np.uint8)
    q[:, 0, 0] = 0x38                                     # 1.0
    kp = np.zeros((1, 1, 32, 128), np.uint8)
    kp[0, 0, 1, 0] = 0xB8                                 # -1.0
    vp = np.zeros((1, 1, 32, 128), np.uint8)
    vp[0, 0, 0, :] = 0x38                                 # 1.0
    vp[0, 0, 1, :] = 0x40                                 # 2.0
    return W.Case(name="two", B=1, N1=1, N2=1, page_size=32, q_lens=[2], kv_lens=[2],
                  k_scale_kind=0, v_scale_kind=0, causal=1, softmax_scale=0.1, p_scale=256.0,
                  q=q, k_pages=kp, v_pages=vp, q_descale=np.ones((2, 1), np.float32),
                  k_descale=np.ones(1, np.float32), v_descale=np.ones(1, np.float32),
                  cu_seqlens_q=np.array([0, 2], np.int32), seqused_kv=np.array([2], np.int32),
                  block_table=np.array([[0]], np.int32),
                  block_mask=np.ones((1, 1, 1, 1), np.uint8))


def pin_fixed_pscale_worked_example(lib):
    """Row 1 sees s = (0, -0.1).  Exact: O = (1 + 2e^-0.1)/(1 + e^-0.1).  With P-scale 256:
    p = (1, e^-0.1 = 0.904837...), 256p = (256, 231.638...); 231.638 lies below the midpoint 232
    of the e4m3 neighbours 224 and 240, so it becomes 224, and
    O = (256*1 + 224*2) / (256 * (1 + e^-0.1)) = 704 / (256 * 1.904837...).
    Row 0 sees only key 0: O = 1, LSE = 0."""
    case = _two_key_case()
    e = math.exp(-0.1)
    o, lse, _ = _oracle(case, lib).all_rows(O.EXACT)
    assert abs(o[1, 0, 0] - (1 + 2 * e) / (1 + e)) < 1e-12
    assert abs(lse[0, 1] - math.log(1 + math.exp(-0.1))) < 1e-9
    assert o[0, 0, 5] == 1.0 and lse[0, 0] == 0.0
    o2, lse2, _ = _oracle(case, lib).all_rows(O.PEMU)
    assert abs(o2[1, 0, 7] - 704.0 / (256.0 * (1 + e))) < 1e-6
    assert abs(lse2[0, 1] - math.log(1 + e)) < 1e-6
    assert o2[0, 0, 0] == 1.0 and lse2[0, 0] == 0.0


def _two_tile_case():
    """256 keys, one head, q = e0, softmax_scale 0.1.  Keys 0..127 (tile 0): k = 0, v = 1.
    Keys 128..255 (tile 1): k = -e0, v = 2.  So s = 0 on tile 0 and -0.1 on tile 1."""
    q = np.zeros((256, 1, 128), np.uint8)
    q[:, 0, 0] = 0x38
    kp = np.zeros((4, 1, 64, 128), np.uint8)
    vp = np.zeros((4, 1, 64, 128), np.uint8)
    kp[2:, 0, :, 0] = 0xB8                                # -1.0 on pages of tile 1
    vp[:2] = 0x38                                         # 1.0
    vp[2:] = 0x40                                         # 2.0
    return W.Case(name="two_tiles", B=1, N1=1, N2=1, page_size=64, q_lens=[256],
                  kv_lens=[256], k_scale_kind=0, v_scale_kind=0, causal=1, softmax_scale=0.1,
                  p_scale=256.0, q=q, k_pages=kp, v_pages=vp,
                  q_descale=np.ones((256, 1), np.float32), k_descale=np.ones(1, np.float32),
                  v_descale=np.ones(1, np.float32), cu_seqlens_q=np.array([0, 256], np.int32),
                  seqused_kv=np.array([256], np.int32),
                  block_table=np.array([[0, 1, 2, 3]], np.int32),
                  block_mask=np.ones((1, 1, 2, 2), np.uint8))


def pin_fixed_pscale_running_max(lib):
    """Row 255 sees all 256 keys, tile 0 first.  The running max after tile 0 is 0 and stays 0
    (tile 1's scores are -0.1), so tile 1's p = e^-0.1 is scaled to 231.638... and rounds to
    224: O = (128*256*1 + 128*224*2) / (256 * (128 + 128 e^-0.1)) = 704 / (256 (1 + e^-0.1)),
    LSE = ln(128 (1 + e^-0.1)).  The sum l is over the unrounded p.  Row 127 sees tile 0
    only: O = 1, LSE = ln 128."""
    case = _two_tile_case()
    e = math.exp(float(np.float32(-0.1)))
    o, lse, _ = _oracle(case, lib).all_rows(O.PEMU)
    assert abs(o[255, 0, 3] - 704.0 / (256.0 * (1 + e))) < 1e-6
    assert abs(lse[0, 255] - math.log(128 * (1 + e))) < 1e-6
    assert abs(o[127, 0, 9] - 1.0) < 1e-12 and abs(lse[0, 127] - math.log(128)) < 1e-12
    o, lse, _ = _oracle(case, lib).all_rows(O.EXACT)
    ee = math.exp(-0.1)
    assert abs(o[255, 0, 3] - (1 + 2 * ee) / (1 + ee)) < 1e-12


def _rising_tiles_case(ntiles):
    """128·ntiles keys, one head, q = e0, softmax_scale 0.1, identity pages of 64.  Tile 0:
    k = -e0 (s = -0.1), v = 1; tile 1: k = 0 (s = 0), v = 2; tile 2: k = -2e0 (s = -0.2),
    v = 3; tile 3: k = e0 (s = 0.1), v = 4.  The row max rises at tile 1, so a step holding
    tiles 0 and 1 quantises tile 0's P against tile 1's maximum."""
    n = 128 * ntiles
    q = np.zeros((n, 1, 128), np.uint8)
    q[:, 0, 0] = 0x38                                     # 1.0
    npages = 2 * ntiles
    kp = np.zeros((npages, 1, 64, 128), np.uint8)
    vp = np.zeros((npages, 1, 64, 128), np.uint8)
    kcode = {0: 0xB8, 1: 0x00, 2: 0xC0, 3: 0x38}          # -1.0, 0, -2.0, 1.0
    vcode = {0: 0x38, 1: 0x40, 2: 0x44, 3: 0x48}          # 1.0, 2.0, 3.0, 4.0
    for t in range(ntiles):
        kp[2 * t:2 * t + 2, 0, :, 0] = kcode[t]
        vp[2 * t:2 * t + 2] = vcode[t]
    return W.Case(name="rising", B=1, N1=1, N2=1, page_size=64, q_lens=[n], kv_lens=[n],
                  k_scale_kind=0, v_scale_kind=0, causal=1, softmax_scale=0.1, p_scale=256.0,
                  q=q, k_pages=kp, v_pages=vp, q_descale=np.ones((n, 1), np.float32),
                  k_descale=np.ones(1, np.float32), v_descale=np.ones(1, np.float32),
                  cu_seqlens_q=np.array([0, n], np.int32), seqused_kv=np.array([n], np.int32),
                  block_table=np.arange(npages, dtype=np.int32)[None, :],
                  block_mask=np.ones((1, 1, ntiles, ntiles), np.uint8))


def pin_macro_block_pairs(lib):
    """Two tiles, the last row sees both (s = -0.1 on tile 0, 0 on tile 1).  One tile per
    step: tile 0 is quantised against its own maximum (p = 1 -> 256 exactly), then rescaled
    by e^-0.1 when tile 1 raises the maximum, which gives the exact answer (2 + e)/(1 + e),
    e = e^-0.1.  Both tiles in one step (the 256-wide macro block): tile 0's p = e^-0.1 is
    scaled to 231.64 and rounds to 224, so O = (128*224*1 + 128*256*2) / (256*128 (1 + e)) =
    736 / (256 (1 + e)).  LSE = ln(128 (1 + e)) either way; row 127 sees tile 0 only: O = 1."""
    case = _rising_tiles_case(2)
    e = math.exp(float(np.float32(-0.1)))
    a = _oracle(case, lib)
    o2, l2, _ = a.all_rows(O.PEMU, group=2)
    assert abs(o2[255, 0, 5] - 736.0 / (256.0 * (1 + e))) < 1e-6
    assert abs(l2[0, 255] - math.log(128 * (1 + e))) < 1e-6
    assert abs(o2[127, 0, 5] - 1.0) < 1e-12
    o1, _, _ = a.all_rows(O.PEMU, group=1)
    assert abs(o1[255, 0, 5] - (2 + e) / (1 + e)) < 1e-6


def pin_macro_block_odd_tail(lib):
    """Three tiles (s = -0.1, 0, -0.2; v = 1, 2, 3), the last row sees all of them.  Two per
    step: tiles 0 and 1 share the maximum 0 (224 and 256, as above); tile 2 is a step of its
    own, below the maximum, p = e^-0.2 scaled to 209.59, which rounds to 208.  O = 128 (224*1 +
    256*2 + 208*3) / (256*128 (e1 + 1 + e2)) = 1360 / (256 (e1 + 1 + e2)), e1 = e^-0.1,
    e2 = e^-0.2."""
    case = _rising_tiles_case(3)
    e1 = math.exp(float(np.float32(-0.1)))
    e2 = math.exp(float(np.float32(-0.2)))
    o, lse, _ = _oracle(case, lib).all_rows(O.PEMU, group=2)
    assert abs(o[383, 0, 7] - 1360.0 / (256.0 * (e1 + 1 + e2))) < 1e-6
    assert abs(lse[0, 383] - math.log(128 * (e1 + 1 + e2))) < 1e-6


def pin_macro_block_second_pair(lib):
    """Four tiles (s = -0.1, 0, -0.2, 0.1; v = 1, 2, 3, 4), the last row sees all of them, in
    steps (0, 1), (2, 3).  Step 1: maximum 0, P = 224 and 256 as above, l1 = 128 (e1 + 1).
    Step 2: the maximum rises to 0.1, a = e^-0.1; tile 2's p = e^-0.3 scaled to 189.65 rounds
    to 192, tile 3's p = 1 gives 256.  O = (a*128*736 + 128 (192*3 + 256*4)) /
    (256 (a*l1 + 128 (e3 + 1))), e3 = e^-0.3; LSE = 0.1 + ln(a*l1 + 128 (e3 + 1))."""
    case = _rising_tiles_case(4)
    f = lambda x: float(np.float32(x))
    e1 = math.exp(f(-0.1))
    a = math.exp(-f(0.1))
    e3 = float(np.float32(math.exp(f(-0.2) - f(0.1))))
    l1 = 128 * (float(np.float32(e1)) + 1)
    lt = a * l1 + 128 * (e3 + 1)
    o, lse, _ = _oracle(case, lib).all_rows(O.PEMU, group=2)
    assert abs(o[511, 0, 11] - (a * 128 * 736 + 128 * (192 * 3 + 256 * 4)) / (256 * lt)) < 1e-6
    assert abs(lse[0, 511] - (f(0.1) + math.log(lt))) < 1e-6


def pin_macro_block_closed_form_zero_k(lib):
    """K = 0: every visible key has p = 1 whatever the grouping, so two tiles per step gives
    the plain mean of the visible V and LSE = ln |A_i|, as the exact formula does."""
    case = _uniform_k_case(31)
    a = _oracle(case, lib)
    o2, l2, _ = a.all_rows(O.PEMU, group=2)
    oe, le, _ = a.all_rows(O.EXACT)
    _close(o2, oe, 1e-9)
    _close(l2, le, 1e-9)


def pin_macro_block_near_exact(lib):
    """Two tiles per step stays within the exact band on a random block-sparse case."""
    case = W.make_case("macro", 32, [700, 300], [700, 300], 4, 2, 64, 1, 2, "bernoulli",
                       keep=0.6)
    a = _oracle(case, lib)
    o2, l2, _ = a.all_rows(O.PEMU, group=2)
    oe, le, _ = a.all_rows(O.EXACT)
    bad = np.abs(o2 - oe) > 0.02 + 0.02 * np.abs(oe)
    assert bad.mean() < 0.005
    seen = le > -1e30
    assert np.all(np.abs(l2[seen] - le[seen]) <= 2.5e-5 + 0.005 * np.abs(le[seen]))


def pin_pemu_near_exact(lib):
    """The e4m3-rounded P stays within the exact band on all but a sliver of elements."""
    case = W.make_case("pe", 41, [512], [512], 4, 1, 64, W.SCALE_PER_TOKEN_HEAD,
                       W.SCALE_PER_HEAD, "bernoulli")
    a = _oracle(case, lib)
    o, l, _ = a.all_rows(O.EXACT)
    o2, l2, _ = a.all_rows(O.PEMU)
    bad = np.abs(o2 - o) > 0.02 + 0.02 * np.abs(o)
    assert bad.mean() < 0.005
    assert np.abs(o2 - o).max() > 1e-4          # the rounding is really applied
    assert np.all(np.abs(l2 - l) <= 2.5e-5 + 0.005 * np.abs(l))


def pin_split_two_tiles(lib):
    """The P-emulating mode with the list cut into 2 slices (one tile each, each slice its own
    online softmax, merged by log-sum-exp weights).  Row 255: slice 0 has m = 0 and p = 1;
    slice 1 has its own max m = -0.1, so its p = 1 too and 256p = 256 is exact; the merge
    weighs slice 1 by e^-0.1.  O = (128*256*1 + e*128*256*2) / (256 * 128 (1 + e)) =
    (1 + 2e) / (1 + e) -- the exact answer, unlike the unsplit mode (704 / (256 (1 + e))),
    and LSE = ln(128 (1 + e))."""
    case = _two_tile_case()
    e = math.exp(float(np.float32(-0.1)))
    o, lse, _ = _oracle(case, lib).all_rows(O.PEMU, splits=2)
    assert abs(o[255, 0, 3] - (1 + 2 * e) / (1 + e)) < 1e-9
    assert abs(lse[0, 255] - math.log(128 * (1 + e))) < 1e-9
    assert abs(o[127, 0, 9] - 1.0) < 1e-12 and abs(lse[0, 127] - math.log(128)) < 1e-12
    o1, _, _ = _oracle(case, lib).all_rows(O.PEMU, splits=1)
    assert abs(o1[255, 0, 3] - 704.0 / (256.0 * (1 + e))) < 1e-6


def pin_split_closed_form_zero_k(lib):
    """K = 0 with the list in 3 and 5 slices: still every visible key at weight 1/|A_i|."""
    case = _uniform_k_case(35)
    sets = tile_sets(case)
    V = torch_decode(case.meta["v_codes"]) * float(case.v_descale[0])
    G = case.N1 // case.N2
    for splits in (3, 5):
        o, lse, _ = _oracle(case, lib).all_rows(O.PEMU, splits=splits)
        kv0 = 0
        for b in range(case.B):
            ql, kl = case.q_lens[b], case.kv_lens[b]
            q0 = int(case.cu_seqlens_q[b])
            for h in range(case.N1):
                for i in range(ql):
                    vis = [j for j in range(kl) if j <= i + kl - ql and (j // 128) in sets[b, h, i // 128]]
                    if not vis:
                        assert lse[h, q0 + i] == NEG_FLT_MAX and not o[q0 + i, h].any()
                        continue
                    _close(o[q0 + i, h], V[[kv0 + j for j in vis], h // G].mean(axis=0), 1e-12)
                    assert abs(lse[h, q0 + i] - math.log(len(vis))) < 1e-12
            kv0 += kl


def pin_split_near_exact(lib):
    """Split P-emulation stays within the exact band like the unsplit mode."""
    case = W.make_case("pes", 42, [384], [1600], 4, 2, 64, W.SCALE_PER_TOKEN_HEAD,
                       W.SCALE_PER_HEAD, "bernoulli", keep=0.6)
    a = _oracle(case, lib)
    o, l, _ = a.all_rows(O.EXACT)
    for splits in (2, 4):
        o2, l2, _ = a.all_rows(O.PEMU, splits=splits)
        bad = np.abs(o2 - o) > 0.02 + 0.02 * np.abs(o)
        assert bad.mean() < 0.005
        assert np.all(np.abs(l2 - l) <= 2.5e-5 + 0.005 * np.abs(l))


# ----------------------------------------------------------------------------------------
# quantisation into the attention inputs (FlashMLA page, 量化 / 解量化的源码实现: scale =
# amax / 448, stored value e4m3(x / scale); readings in oracle/bsa_oracle.c)
# ----------------------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bit patterns (PyTorch's cast)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def torch_quantize_rows(xb: np.ndarray):
    """Independent restatement with numpy fp32 arithmetic and PyTorch's e4m3 cast."""
    x = bf16_bits_to_f32(xb)
    amax = np.abs(x).max(axis=-1)
    d = np.where(amax > 0, (amax / np.float32(448.0)).astype(np.float32), np.float32(1.0))
    q = np.clip((x / d[..., None]).astype(np.float32), -448.0, 448.0).astype(np.float32)
    codes = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes, d.astype(np.float32)


def _quant_rows_fixture():
    rng = np.random.default_rng(1234)
    x = rng.standard_normal((37, 128)).astype(np.float32)
    x[3] = 0.0                                       # zero row -> descale 1, zero codes
    x[5] *= 1e-4                                     # small values: subnormal e4m3 codes
    x[6, 17] = 3.0e4                                 # one large outlier
    x[7] = np.linspace(-1000.0, 1000.0, 128)         # codes spanning the whole range
    x[8] *= 2.0 ** -20
    return f32_to_bf16_bits(x)


def pin_quantize_vs_torch_cast(lib):
    xb = _quant_rows_fixture()
    codes, desc = O.quantize_rows(xb, lib=lib)
    t_codes, t_desc = torch_quantize_rows(xb)
    assert np.array_equal(desc.view(np.uint32), t_desc.view(np.uint32)), "descales differ"
    assert np.array_equal(codes, t_codes), f"{int((codes != t_codes).sum())} codes differ"


def pin_quantize_closed_forms(lib):
    vals = np.zeros((4, 128), dtype=np.float32)
    vals[0, :5] = [448.0, -448.0, 0.5, -2.0 ** -6, 2.0 ** -9]   # amax 448 -> descale 1
    vals[2, :3] = [896.0, 448.0, -1.0]                           # amax 896 -> descale 2
    vals[3] = vals[0] * 2.0 ** 40                                # scaled copy of row 0
    codes, desc = O.quantize_rows(f32_to_bf16_bits(vals), lib=lib)
    assert desc[0] == 1.0 and desc[1] == 1.0 and desc[2] == 2.0 and desc[3] == 2.0 ** 40
    assert list(codes[0, :5]) == [0x7E, 0xFE, 0x30, 0x88, 0x01]
    assert not codes[0, 5:].any() and not codes[1].any()
    assert list(codes[2, :3]) == [0x7E, 0x76, 0xB0]              # 448, 224, -0.5
    assert np.array_equal(codes[3], codes[0])
    # dequantisation error: half an e4m3 step (2^-4 relative) for normals, 2^-10 * descale
    # (half the subnormal quantum) below
    xb = _quant_rows_fixture()
    codes, desc = O.quantize_rows(xb, lib=lib)
    x = bf16_bits_to_f32(xb).astype(np.float64)
    deq = torch_decode(codes) * desc[:, None].astype(np.float64)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, desc[:, None] * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(deq - x) <= bound)


def pin_quantize_ue8m0_closed_forms(lib):
    """FlashMLA's cast of the scale to UE8M0 (FlashMLA page, 量化 / 解量化的源码实现): the
    descale is the smallest power of two not below amax / 448, worked by hand per row."""
    vals = np.zeros((6, 128), dtype=np.float32)
    vals[0, :3] = [448.0, -224.0, 1.0]   # amax / 448 = 1 is a power of two: descale 1
    vals[1, :2] = [450.0, -1.0]          # 450 / 448 just above 1 (449 is no bf16): descale
    #                                      2; 225 -> 224
    vals[2, 0] = 1.0                     # 1 / 448 in (2^-9, 2^-8): descale 2^-8, 1 -> 256
    vals[3, :2] = [300.0, 100.0]         # 300 / 448 in (1/2, 1): descale 1; 300 -> 288, 100 -> 96
    # row 4 stays zero: descale 1, zero codes, as under the plain rule
    xb = f32_to_bf16_bits(vals)
    xb[5, 0] = 0x0001                    # 2^-133, the smallest bf16: amax / 448 is an fp32
    #                                      subnormal (146 * 2^-149), descale 2^-141, code of 256
    codes, desc = O.quantize_rows(xb, lib=lib, rule=O.DESCALE_UE8M0)
    assert list(desc) == [1.0, 2.0, 2.0 ** -8, 1.0, 1.0, 2.0 ** -141], list(desc)
    assert list(codes[0, :3]) == [0x7E, 0xF6, 0x38]
    assert list(codes[1, :2]) == [0x76, 0xB0]
    assert codes[2, 0] == 0x78 and codes[5, 0] == 0x78
    assert list(codes[3, :2]) == [0x79, 0x6C]
    assert not codes[4].any()
    for r in range(6):
        assert not codes[r, 3:].any()


def pin_quantize_ue8m0_invariants(lib):
    """On rows spanning 2^-120 .. 2^120: every UE8M0 descale is a power of two in
    [amax/448, 2 amax/448) (amax/448 as an fp32 quotient), the codes are torch's e4m3 cast of
    x / descale, and each row's largest code decodes to [224, 448] (amax / descale lies in
    (224, 448] and rounds to no less than 224)."""
    rng = np.random.default_rng(7)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    x *= (2.0 ** rng.integers(-120, 120, size=(64, 1))).astype(np.float32)
    xb = f32_to_bf16_bits(x)
    codes, desc = O.quantize_rows(xb, lib=lib, rule=O.DESCALE_UE8M0)
    xf = bf16_bits_to_f32(xb)
    base = (np.abs(xf).max(axis=1) / np.float32(448.0)).astype(np.float32)
    lg = np.log2(desc.astype(np.float64))
    assert np.all(lg == np.round(lg)), "not a power of two"
    assert np.all(desc >= base) and np.all(desc / 2 < base)
    for r in range(64):
        assert np.array_equal(codes[r], _torch_codes(xf[r], desc[r])), r
    big = np.abs(torch_decode(codes)).max(axis=1)
    assert np.all(big >= 224.0) and np.all(big <= 448.0)


def _append_fixture(k_kind, v_kind):
    rng = np.random.default_rng(99)
    P, N2, ps = 9, 2, 4
    L = 4
    bt = np.full((2, L), -1, dtype=np.int32)
    perm = rng.permutation(P)
    bt[0, :3] = perm[:3]
    bt[1, :4] = perm[3:7]
    cache_len = np.array([5, 0], dtype=np.int32)
    cu_new = np.array([0, 6, 13], dtype=np.int32)      # 6 new tokens for b=0, 7 for b=1
    kx = rng.standard_normal((13, N2, 128)).astype(np.float32) * 3
    vx = rng.standard_normal((13, N2, 128)).astype(np.float32)
    kb, vb = f32_to_bf16_bits(kx), f32_to_bf16_bits(vx)
    kp = np.full((P, N2, ps, 128), 0x55, dtype=np.uint8)
    vp = np.full((P, N2, ps, 128), 0x55, dtype=np.uint8)
    kd = np.full((P, N2, ps), -7.0, dtype=np.float32)
    k_scale = np.array([0.02], dtype=np.float32)
    v_scale = np.array([0.01, 0.005], dtype=np.float32) if v_kind == W.SCALE_PER_HEAD else \
        np.array([0.01], dtype=np.float32)
    return dict(kb=kb, vb=vb, cu_new=cu_new, cache_len=cache_len, bt=bt, kp=kp, vp=vp, kd=kd,
                k_scale=k_scale, v_scale=v_scale, ps=ps)


def _torch_codes(x, scale):
    q = np.clip((x / scale).astype(np.float32), -448.0, 448.0).astype(np.float32)
    return torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def pin_append_kv_placement(lib):
    for k_kind, v_kind, rule in ((W.SCALE_PER_TOKEN_HEAD, W.SCALE_PER_HEAD, O.DESCALE_AMAX),
                                 (W.SCALE_PER_TOKEN_HEAD, W.SCALE_PER_HEAD, O.DESCALE_UE8M0),
                                 (W.SCALE_PER_TENSOR, W.SCALE_PER_TENSOR, O.DESCALE_AMAX)):
        f = _append_fixture(k_kind, v_kind)
        kp, vp, kd, err = O.append_kv(f["kb"], f["vb"], f["cu_new"], f["cache_len"], f["bt"],
                                      f["kp"], f["vp"], f["kd"], k_kind, v_kind,
                                      f["k_scale"], f["v_scale"], lib=lib, k_descale_rule=rule)
        assert err == 0
        ps = f["ps"]
        written = np.zeros(kp.shape[:3], dtype=bool)
        kx, vx = bf16_bits_to_f32(f["kb"]), bf16_bits_to_f32(f["vb"])
        for b in range(2):
            for i in range(f["cu_new"][b + 1] - f["cu_new"][b]):
                tok = f["cu_new"][b] + i
                pos = f["cache_len"][b] + i
                pg = f["bt"][b, pos // ps]
                slot = pos % ps
                for g in range(2):
                    written[pg, g, slot] = True
                    if k_kind == W.SCALE_PER_TOKEN_HEAD and rule == O.DESCALE_AMAX:
                        c, d = torch_quantize_rows(f["kb"][tok, g][None])
                        assert np.array_equal(kp[pg, g, slot], c[0]) and kd[pg, g, slot] == d[0]
                    elif k_kind == W.SCALE_PER_TOKEN_HEAD:
                        # the row's own quantisation under the same rule, checked above
                        c, d = O.quantize_rows(f["kb"][tok, g][None], lib=lib, rule=rule)
                        assert np.array_equal(kp[pg, g, slot], c[0]) and kd[pg, g, slot] == d[0]
                    else:
                        assert np.array_equal(kp[pg, g, slot], _torch_codes(kx[tok, g], f["k_scale"][0]))
                    vs = f["v_scale"][g] if v_kind == W.SCALE_PER_HEAD else f["v_scale"][0]
                    assert np.array_equal(vp[pg, g, slot], _torch_codes(vx[tok, g], vs))
        # every other slot is untouched
        assert np.all(kp[~written] == 0x55) and np.all(vp[~written] == 0x55)
        if k_kind == W.SCALE_PER_TOKEN_HEAD:
            assert np.all(kd[~written] == -7.0)
        else:
            assert np.all(kd == -7.0)
    # a missing page is reported and its tokens skipped
    f = _append_fixture(W.SCALE_PER_TOKEN_HEAD, W.SCALE_PER_HEAD)
    bt = f["bt"].copy()
    bt[1, 1] = -1
    kp, vp, kd, err = O.append_kv(f["kb"], f["vb"], f["cu_new"], f["cache_len"], bt, f["kp"],
                                  f["vp"], f["kd"], W.SCALE_PER_TOKEN_HEAD, W.SCALE_PER_HEAD,
                                  f["k_scale"], f["v_scale"], lib=lib)
    assert err == O.ERR_BAD_PAGE
    assert np.all(kp[f["bt"][1, 1]] == 0x55)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
