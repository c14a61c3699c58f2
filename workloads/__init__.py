"""Seeded synthetic inputs for block-sparse FP8 attention prefill over a paged KV cache.

This module is shared by the CPU oracle (``oracle/``), the tests and ``bench.py``.  It holds
none of the attention arithmetic: it draws random numbers, quantises them to e4m3 with
PyTorch's built-in ``float8_e4m3fn`` cast (a library routine), lays the keys and values out
in pages, and builds the block masks / sparse index lists.

Random numbers come from one counter-based generator, SplitMix64 (Steele, Lea & Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014): the i-th draw of stream s
under seed S is ``mix64(S * 2^32 + s, i)``.  Normals use the Box-Muller transform.

Workload shapes follow the two pages this library implements:
  * hpc-ops Block-Sparse FP8 Attention, "块稀疏调度" (block_mask [B, N1, Qb, Kb], 128-token
    Q/KV tiles) and "快速上手" (paged KV, 32/64-token pages, unused slots zero);
  * Quant Block Sparse Attention (CANNBotDSL), parameter table (TND query, page layout
    [P, N2, page, 128], q/k/v descale shapes, sparse_indices [B, N1, max_Qb, Kb] and
    sparse_seq_len [B, N1, max_Qb]).
"""
from __future__ import annotations

import math
import os
from dataclasses import dataclass, field

import numpy as np

TILE = 128          # Q tile and KV tile size (both pages fix it at 128 tokens)
HEAD_DIM = 128      # D; both pages support only 128
E4M3_MAX = 448.0

SCALE_PER_TENSOR = 0
SCALE_PER_TOKEN_HEAD = 1   # K only
SCALE_PER_HEAD = 2         # V only

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)

# stream ids (sub-streams of one seed)
S_Q, S_K, S_V, S_MASK, S_PERM, S_OUTLIER, S_SHUFFLE, S_EMPTY, S_MISC = range(9)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _C1
    z = (z ^ (z >> np.uint64(27))) * _C2
    return z ^ (z >> np.uint64(31))


def rand_u64(seed: int, stream: int, start: int, n: int) -> np.ndarray:
    """Draws start..start+n-1 of SplitMix64 stream `stream` under `seed`."""
    key = np.uint64((seed * (1 << 32) + stream * 0x632BE59BD9B4E019) & 0xFFFFFFFFFFFFFFFF)
    ctr = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + ctr * _GOLDEN)


def rand_uniform(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """Uniform doubles in the open interval (0, 1)."""
    u = rand_u64(seed, stream, start, n) >> np.uint64(11)
    return (u.astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def rand_normal(seed: int, stream: int, n: int, chunk: int = 1 << 20) -> np.ndarray:
    """N(0, 1) as float32 (Box-Muller cosine branch over draw pairs), generated in chunks.
    The generator is counter-based, so chunks are independent: they run on a thread pool
    (numpy releases the GIL in these array operations) and the result does not depend on
    the number of threads."""
    from concurrent.futures import ThreadPoolExecutor

    out = np.empty(n, dtype=np.float32)

    def fill(s):
        m = min(chunk, n - s)
        u = rand_uniform(seed, stream, 2 * m, start=2 * s)
        u1, u2 = u[0::2], u[1::2]
        out[s:s + m] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)

    starts = list(range(0, n, chunk))
    if len(starts) <= 1:
        for s in starts:
            fill(s)
    else:
        with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1, len(starts))) as ex:
            list(ex.map(fill, starts))
    return out


def quantize_e4m3(x: np.ndarray, descale: np.ndarray) -> np.ndarray:
    """uint8 e4m3fn codes of x / descale (descale broadcast against x), via torch's cast."""
    import torch

    y = np.clip(x / descale, -E4M3_MAX, E4M3_MAX).astype(np.float32)
    return torch.from_numpy(np.ascontiguousarray(y)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _amax_descale(amax: np.ndarray) -> np.ndarray:
    d = (amax / E4M3_MAX).astype(np.float32)
    return np.where(amax > 0, d, np.float32(1.0)).astype(np.float32)


@dataclass
class Case:
    """One synthetic problem in the library's device layout (all host numpy arrays)."""

    name: str
    B: int
    N1: int
    N2: int
    page_size: int
    q_lens: list
    kv_lens: list
    k_scale_kind: int
    v_scale_kind: int
    causal: int
    softmax_scale: float
    p_scale: float
    q: np.ndarray              # uint8 [T, N1, 128]
    k_pages: np.ndarray        # uint8 [P, N2, ps, 128]
    v_pages: np.ndarray        # uint8 [P, N2, ps, 128]
    q_descale: np.ndarray      # f32 [T, N1]
    k_descale: np.ndarray      # f32 [1] or [P, N2, ps]
    v_descale: np.ndarray      # f32 [1] or [N2]
    cu_seqlens_q: np.ndarray   # i32 [B+1]
    seqused_kv: np.ndarray     # i32 [B]
    block_table: np.ndarray    # i32 [B, L]
    block_mask: np.ndarray | None = None       # u8 [B, N1, Qb, Kb]
    sparse_indices: np.ndarray | None = None   # i32 [B, N1, Qb, Kb]
    sparse_seq_len: np.ndarray | None = None   # i32 [B, N1, Qb]
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def max_q_len(self) -> int:
        return max(self.q_lens) if self.q_lens else 0

    @property
    def max_kv_len(self) -> int:
        return max(self.kv_lens) if self.kv_lens else 0

    @property
    def Qb(self) -> int:
        return -(-self.max_q_len // TILE)

    @property
    def Kb(self) -> int:
        return -(-self.max_kv_len // TILE)

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    def dims(self) -> dict:
        return dict(B=self.B, N1=self.N1, N2=self.N2, D=HEAD_DIM, page_size=self.page_size,
                    max_q_len=self.max_q_len, max_kv_len=self.max_kv_len,
                    num_pages=self.num_pages, max_pages_per_seq=self.max_pages_per_seq,
                    total_q=self.T, k_scale_kind=self.k_scale_kind,
                    v_scale_kind=self.v_scale_kind, causal=self.causal)


# ----------------------------------------------------------------------------------------
# masks and sparse index lists
# ----------------------------------------------------------------------------------------

def diag_tile(q_len: int, kv_len: int, qt: int) -> int:
    """KV tile holding the causal diagonal of the first row of Q tile qt (right-aligned)."""
    return (qt * TILE + (kv_len - q_len)) // TILE


def mask_bernoulli(seed, B, N1, q_lens, kv_lens, keep: float) -> np.ndarray:
    """Diagonal tile kept; each earlier causal tile kept with probability `keep`."""
    Qb = -(-max(q_lens) // TILE)
    Kb = -(-max(kv_lens) // TILE)
    u = rand_uniform(seed, S_MASK, B * N1 * Qb * Kb).reshape(B, N1, Qb, Kb)
    m = np.zeros((B, N1, Qb, Kb), dtype=np.uint8)
    t = np.arange(Kb)
    for b in range(B):
        for qt in range(-(-q_lens[b] // TILE)):
            d = diag_tile(q_lens[b], kv_lens[b], qt)
            row = (t < d) & (u[b, :, qt, :] < keep)
            if 0 <= d < Kb:
                row[:, d] = True
            m[b, :, qt, :] = row
    return m


def mask_local_sink(seed, B, N1, q_lens, kv_lens, n_local: int, p_far: float) -> np.ndarray:
    """Diagonal, `n_local` tiles before it, tile 0 (sink) and far tiles with prob. p_far."""
    Qb = -(-max(q_lens) // TILE)
    Kb = -(-max(kv_lens) // TILE)
    u = rand_uniform(seed, S_MASK, B * N1 * Qb * Kb).reshape(B, N1, Qb, Kb)
    m = np.zeros((B, N1, Qb, Kb), dtype=np.uint8)
    t = np.arange(Kb)
    for b in range(B):
        for qt in range(-(-q_lens[b] // TILE)):
            d = diag_tile(q_lens[b], kv_lens[b], qt)
            row = (t >= 1) & (t <= d - n_local - 1) & (u[b, :, qt, :] < p_far)
            if d >= 0:
                row[:, max(0, d - n_local):min(d + 1, Kb)] = True
                row[:, 0] = True
            m[b, :, qt, :] = row
    return m


def sparse_from_fraction(seed, B, N1, q_lens, kv_lens, frac: float, n_empty: int):
    """For each task: n = max(min(2, c), ceil(frac*c)) distinct causal tiles, always tile 0
    and the diagonal, stored in shuffled order; entries past n are -1.  `n_empty` seeded
    tasks get sparse_seq_len = 0."""
    Qb = -(-max(q_lens) // TILE)
    Kb = -(-max(kv_lens) // TILE)
    idx = np.full((B, N1, Qb, Kb), -1, dtype=np.int32)
    nlen = np.zeros((B, N1, Qb), dtype=np.int32)
    keys = rand_uniform(seed, S_MASK, B * N1 * Qb * Kb).reshape(B, N1, Qb, Kb)
    shuf = rand_uniform(seed, S_SHUFFLE, B * N1 * Qb * Kb).reshape(B, N1, Qb, Kb)
    for b in range(B):
        for qt in range(-(-q_lens[b] // TILE)):
            d = min(diag_tile(q_lens[b], kv_lens[b], qt), Kb - 1)
            if d < 0:
                continue
            c = d + 1
            n = max(min(2, c), math.ceil(frac * c))
            base = sorted({0, d})
            extra = n - len(base)
            k = keys[b, :, qt, :c].copy()
            k[:, base] = np.inf
            order = np.argsort(k, axis=1, kind="stable")[:, :max(extra, 0)]
            for h in range(N1):
                chosen = np.array(base + sorted(order[h].tolist()), dtype=np.int32)
                perm = np.argsort(shuf[b, h, qt, :len(chosen)], kind="stable")
                idx[b, h, qt, :len(chosen)] = chosen[perm]
                nlen[b, h, qt] = len(chosen)
    if n_empty:
        valid = [(b, h, qt) for b in range(B) for h in range(N1)
                 for qt in range(-(-q_lens[b] // TILE))]
        pick = np.argsort(rand_uniform(seed, S_EMPTY, len(valid)), kind="stable")[:n_empty]
        for p in pick:
            b, h, qt = valid[int(p)]
            nlen[b, h, qt] = 0
    return idx, nlen


# ----------------------------------------------------------------------------------------
# generic case builder
# ----------------------------------------------------------------------------------------

def make_case(name: str, seed: int, q_lens, kv_lens, N1: int, N2: int, page_size: int,
              k_scale_kind: int = SCALE_PER_TENSOR, v_scale_kind: int = SCALE_PER_TENSOR,
              mask: str = "bernoulli", keep: float = 0.5, causal: int = 1,
              outlier_frac: float = 0.0, outlier_mult: float = 8.0,
              sparse_frac: float = 0.25, n_empty: int = 0, n_local: int = 4,
              p_far: float = 0.05, softmax_scale: float | None = None,
              p_scale: float = 256.0, identity_pages: bool = False,
              tail_fill: float | None = None, keep_logical: bool = False,
              k_token_group: int = 1, k_pow2: bool = False) -> Case:
    """Builds a seeded case.  mask in {"bernoulli", "local_sink", "indices", "none", "ones"}.
    With a per-token K scale, k_token_group > 1 gives every group of that many consecutive
    tokens of a sequence (per KV head) one scale, repeated over its tokens, and k_pow2 rounds
    the scales up to powers of two."""
    B = len(q_lens)
    assert len(kv_lens) == B
    D = HEAD_DIM
    ps = page_size
    T = int(sum(q_lens))
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)

    # --- Q: per-token per-head quantisation
    xq = rand_normal(seed, S_Q, T * N1 * D).reshape(T, N1, D)
    if outlier_frac > 0:
        nq = round(outlier_frac * N1 * D)
        ch = np.argsort(rand_uniform(seed, S_OUTLIER, N1 * D), kind="stable")[:nq]
        xq.reshape(T, N1 * D)[:, ch] *= outlier_mult
    q_desc = _amax_descale(np.abs(xq).max(axis=2))
    q = quantize_e4m3(xq, q_desc[:, :, None])

    # --- pages: logical KV tokens of every sequence, seeded page permutation
    pages_per = [-(-kv // ps) for kv in kv_lens]
    P = int(sum(pages_per))
    L = max(1, max(pages_per) if pages_per else 1)
    if identity_pages:
        perm = np.arange(P)
    else:
        perm = np.argsort(rand_uniform(seed, S_PERM, P), kind="stable")
    block_table = np.full((B, L), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        block_table[b, :pages_per[b]] = perm[off:off + pages_per[b]]
        off += pages_per[b]

    def logical(stream):
        tot = int(sum(kv_lens))
        x = rand_normal(seed, stream, tot * N2 * D).reshape(tot, N2, D)
        if outlier_frac > 0:
            nk = round(outlier_frac * N2 * D)
            ch = np.argsort(rand_uniform(seed, S_OUTLIER + 16 * stream, N2 * D),
                            kind="stable")[:nk]
            x.reshape(tot, N2 * D)[:, ch] *= outlier_mult
        return x

    def to_pages(codes_tok, fill=0):
        # codes_tok [tot, N2, ...] -> [P, N2, ps, ...]
        shape = (P, N2, ps) + codes_tok.shape[2:]
        out = np.full(shape, fill, dtype=codes_tok.dtype)
        s = 0
        for b in range(B):
            kv = kv_lens[b]
            for lp in range(pages_per[b]):
                pg = block_table[b, lp]
                n = min(ps, kv - lp * ps)
                out[pg, :, :n] = np.swapaxes(codes_tok[s + lp * ps: s + lp * ps + n], 0, 1)
            s += kv
        return out

    xk = logical(S_K)
    if k_scale_kind == SCALE_PER_TENSOR:
        kd_tok = None
        k_desc = _amax_descale(np.array([np.abs(xk).max() if xk.size else 0.0]))
        k_codes = quantize_e4m3(xk, k_desc[0])
    elif k_scale_kind == SCALE_PER_TOKEN_HEAD:
        amax = np.abs(xk).max(axis=2)                            # [tot, N2]
        if k_token_group > 1:
            s0 = 0
            for kv in kv_lens:
                for g0 in range(0, kv, k_token_group):
                    grp = slice(s0 + g0, s0 + min(kv, g0 + k_token_group))
                    amax[grp] = amax[grp].max(axis=0)
                s0 += kv
        kd_tok = _amax_descale(amax)
        if k_pow2:
            want = kd_tok.astype(np.float64)
            p2 = np.exp2(np.ceil(np.log2(want)))
            kd_tok = np.where(p2 < want, 2 * p2, p2).astype(np.float32)
        k_codes = quantize_e4m3(xk, kd_tok[:, :, None])
        k_desc = to_pages(kd_tok, fill=0)                        # [P, N2, ps]
    else:
        raise ValueError("K scale kind")
    k_pages = to_pages(k_codes)

    xv = logical(S_V)
    if v_scale_kind == SCALE_PER_TENSOR:
        v_desc = _amax_descale(np.array([np.abs(xv).max() if xv.size else 0.0]))
        v_codes = quantize_e4m3(xv, v_desc[0])
    elif v_scale_kind == SCALE_PER_HEAD:
        v_desc = _amax_descale(np.abs(xv).max(axis=(0, 2)) if xv.size else np.zeros(N2))
        v_codes = quantize_e4m3(xv, v_desc[None, :, None])
    else:
        raise ValueError("V scale kind")
    v_pages = to_pages(v_codes)

    if tail_fill is not None:
        # finite non-zero values in the unused slots of each sequence's last page
        for b in range(B):
            kv = kv_lens[b]
            if kv % ps:
                pg = block_table[b, pages_per[b] - 1]
                k_pages[pg, :, kv % ps:] = np.uint8(0x38)   # 1.0
                v_pages[pg, :, kv % ps:] = np.uint8(0x40)   # 2.0

    kvl = np.asarray(kv_lens, dtype=np.int32)
    case = Case(name=name, B=B, N1=N1, N2=N2, page_size=ps, q_lens=list(q_lens),
                kv_lens=list(kv_lens), k_scale_kind=k_scale_kind, v_scale_kind=v_scale_kind,
                causal=causal, softmax_scale=float(softmax_scale), p_scale=float(p_scale),
                q=q, k_pages=k_pages, v_pages=v_pages, q_descale=q_desc,
                k_descale=np.ascontiguousarray(k_desc, dtype=np.float32),
                v_descale=np.ascontiguousarray(v_desc, dtype=np.float32),
                cu_seqlens_q=cu, seqused_kv=kvl, block_table=block_table,
                meta=dict(seed=seed, mask=mask))
    if keep_logical:
        # token-ordered copies (concatenated over sequences) for page-free reference code
        case.meta.update(k_codes=k_codes, v_codes=v_codes,
                         k_descale_tok=kd_tok if kd_tok is not None else None)
    if mask == "bernoulli":
        case.block_mask = mask_bernoulli(seed, B, N1, q_lens, kv_lens, keep)
    elif mask == "local_sink":
        case.block_mask = mask_local_sink(seed, B, N1, q_lens, kv_lens, n_local, p_far)
    elif mask == "ones":
        case.block_mask = np.ones((B, N1, case.Qb, case.Kb), dtype=np.uint8)
    elif mask == "indices":
        case.sparse_indices, case.sparse_seq_len = sparse_from_fraction(
            seed, B, N1, q_lens, kv_lens, sparse_frac, n_empty)
    elif mask == "none":
        pass
    else:
        raise ValueError(mask)
    return case


# ----------------------------------------------------------------------------------------
# the five named workloads
# ----------------------------------------------------------------------------------------

WORKLOADS = {
    "prefill_1k_h8kv1_bsm50": dict(
        seed=1001, q_lens=[1024], kv_lens=[1024], N1=8, N2=1, page_size=64,
        k_scale_kind=SCALE_PER_TENSOR, v_scale_kind=SCALE_PER_TENSOR, mask="bernoulli", keep=0.5),
    "prefill_2x8k_h32kv8_bsm50_outliers": dict(
        seed=1002, q_lens=[8192, 8192], kv_lens=[8192, 8192], N1=32, N2=8, page_size=64,
        k_scale_kind=SCALE_PER_TOKEN_HEAD, v_scale_kind=SCALE_PER_HEAD, mask="bernoulli",
        keep=0.5, outlier_frac=0.01),
    "varlen_4x16k_h64kv8_idx25": dict(
        seed=1003, q_lens=[16384, 12000, 9000, 4097], kv_lens=[16384, 12000, 9000, 4097],
        N1=64, N2=8, page_size=32, k_scale_kind=SCALE_PER_TOKEN_HEAD,
        v_scale_kind=SCALE_PER_HEAD, mask="indices", sparse_frac=0.25, n_empty=2),
    "chunked_4k_over_64k_h32kv4_local_sink": dict(
        seed=1004, q_lens=[4096], kv_lens=[65536], N1=32, N2=4, page_size=64,
        k_scale_kind=SCALE_PER_TENSOR, v_scale_kind=SCALE_PER_TENSOR, mask="local_sink",
        n_local=4, p_far=0.05),
    "dense_32k_h32kv8": dict(
        seed=1005, q_lens=[32768], kv_lens=[32768], N1=32, N2=8, page_size=64,
        k_scale_kind=SCALE_PER_TOKEN_HEAD, v_scale_kind=SCALE_PER_HEAD, mask="none"),
    # few tasks over a long KV (32 tasks for 304 pipelines): the split-KV regime
    "short_q_512_over_64k_h8kv1_dense": dict(
        seed=1006, q_lens=[512], kv_lens=[65536], N1=8, N2=1, page_size=64,
        k_scale_kind=SCALE_PER_TOKEN_HEAD, v_scale_kind=SCALE_PER_HEAD, mask="none"),
}

WORKLOAD_ORDER = list(WORKLOADS)


def make_workload(name: str, **overrides) -> Case:
    kw = dict(WORKLOADS[name])
    kw.update(overrides)
    return make_case(name, **kw)


# ----------------------------------------------------------------------------------------
# algorithmic work counts (used for the effective-TFLOPS metric)
# ----------------------------------------------------------------------------------------

def active_work(case: Case, lists_counts=None):
    """(active tile pairs, effective FLOPs) over the canonical active lists.

    FLOPs per (task, tile) = 4 * 128 * rows_valid * cols_valid, where rows_valid counts the
    task's Q rows < q_len and cols_valid counts the tile's KV tokens < kv_len (no discount for
    the causal triangle inside the diagonal tile).  `lists_counts` = (lists, counts) arrays
    shaped [B, N1, Qb, Kb] and [B, N1, Qb]."""
    lists, counts = lists_counts
    tiles = 0
    flops = 0
    for b in range(case.B):
        ql, kl = case.q_lens[b], case.kv_lens[b]
        for qt in range(-(-ql // TILE)):
            rows = min(TILE, ql - qt * TILE)
            c = counts[b, :, qt]
            tiles += int(c.sum())
            for h in range(case.N1):
                ts = lists[b, h, qt, :c[h]].astype(np.int64)
                cols = np.minimum(TILE, kl - ts * TILE)
                flops += 4 * HEAD_DIM * rows * int(cols.sum())
    return tiles, flops
