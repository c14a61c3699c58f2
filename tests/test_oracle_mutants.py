"""The pins catch plausible mistakes in the oracle.

Each mutant is a copy of oracle/bsa_oracle.c with one planted mistake (a dropped term, a wrong
sign or index, a transposed operand), compiled on the CPU into a temporary directory.  The
full pin suite must fail on every mutant.  The real oracle source is never modified.
"""
import os

import pytest

import oracle as O
from oracle_pins import ALL_PINS

MUTANTS = {
    "gqa_head_map": ("int g = h / G;", "int g = h % d->N2;"),
    "causal_off_by_one": ("if (d->causal && j > i + off) continue;",
                          "if (d->causal && j >= i + off) continue;"),
    "drop_v_descale": ("o[k] += w * oracle_e4m3_decode(vr[k]) * vd;",
                       "o[k] += w * oracle_e4m3_decode(vr[k]);"),
    "ignore_block_table": (
        "int pg = in->block_table[(size_t)b * d->max_pages_per_seq + j / d->page_size];",
        "int pg = j / d->page_size + in->block_table[(size_t)b * d->max_pages_per_seq] * 0;"),
    "softmax_sign": ("double w = exp(s[a] - M);", "double w = exp(M - s[a]);"),
    "lse_drop_max": ("*lse = M + log(l);", "*lse = log(l);"),
    "subnormal_exponent": ("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);"),
    "pemu_drop_alpha_l": ("l = alpha * l + psum;", "l = l + psum;"),
    "pemu_drop_pscale": ("oracle_e4m3_encode((double)(float)(p * in->p_scale))",
                         "oracle_e4m3_encode((double)(float)(p))"),
    "kend_off_by_one": ("long c = (long)last_row + (kl - ql) + 1;",
                        "long c = (long)last_row + (kl - ql);"),
    "k_reads_v_pages": ("const uint8_t *kr = kv_row(d, in->k_pages,",
                        "const uint8_t *kr = kv_row(d, in->v_pages,"),
    "k_descale_layout": ("return in->k_descale[((size_t)pg * d->N2 + g) * d->page_size + slot];",
                         "return in->k_descale[((size_t)g * d->num_pages + pg) * d->page_size + slot];"),
    "q_descale_layout": ("double s = in->q_descale[(size_t)tok * d->N1 + h];",
                         "double s = in->q_descale[(size_t)h * d->total_q + tok];"),
    "encode_round_half_away": ("double r = nearbyint(ldexp(a, 3 - ue));",
                               "double r = round(ldexp(a, 3 - ue));"),
    "no_dedup_indices": ("sel[t] = 1;", "sel[t] = 1; list[n++] = t;"),
    "pemu_tile_max_not_running": ("double mn = m > mt ? m : mt;", "double mn = mt;"),
    "pemu_l_from_rounded_p": ("psum += p;",
                              "psum += oracle_e4m3_decode(oracle_e4m3_encode("
                              "(double)(float)(p * in->p_scale))) / in->p_scale;"),
    "pemu_exact_p_in_pv": ("tile_acc[k] += pq * oracle_e4m3_decode(vr[k]);",
                           "tile_acc[k] += p * in->p_scale * oracle_e4m3_decode(vr[k]);"),
    "macro_group_steps_by_one": ("for (int ti = t_lo; ti < t_hi; ti += group) {",
                                 "for (int ti = t_lo; ti < t_hi; ti += 1) {"),
    "macro_group_first_tile_only": (
        "int tl = tiles[(ti + group < t_hi ? ti + group : t_hi) - 1] * TILE;",
        "int tl = t0;"),
    "split_merge_weight_sign": ("double wo = (m == -INFINITY) ? 0.0 : exp(m - mn), wc = exp(mc - mn);",
                                "double wo = (m == -INFINITY) ? 0.0 : exp(m - mn), wc = exp(mn - mc);"),
    "split_slice_keeps_earlier_keys": (
        "    while (a < na && keys[a] < t0) ++a;              /* skip keys of earlier slices */",
        ""),
    "ue8m0_round_down": ("return m == 0.5f ? x : ldexpf(1.0f, e);",
                         "return m == 0.5f ? x : ldexpf(1.0f, e - 1);"),
    "ue8m0_rule_ignored": (
        "if (rule == ORACLE_DESCALE_UE8M0 && amax > 0.0f) descale = pow2_ceil(descale);", ""),
    "ue8m0_always_next_power": ("return m == 0.5f ? x : ldexpf(1.0f, e);",
                                "return ldexpf(1.0f, e);"),
    "quant_wrong_max": ("float descale = amax > 0.0f ? amax / 448.0f : 1.0f;",
                        "float descale = amax > 0.0f ? amax / 240.0f : 1.0f;"),
    "quant_zero_row_descale": ("float descale = amax > 0.0f ? amax / 448.0f : 1.0f;",
                               "float descale = amax > 0.0f ? amax / 448.0f : 0.0f;"),
    "quant_multiply_by_descale": ("float v = bf16_value(x[i]) / descale;",
                                  "float v = bf16_value(x[i]) * descale;"),
    "append_ignores_cache_len": ("long pos = (long)cache_len[b] + i;", "long pos = i;"),
    "append_slot_transposed": ("size_t row = ((size_t)pg * N2 + g) * page_size + slot;",
                               "size_t row = ((size_t)g * num_pages + pg) * page_size + slot;"),
    "append_v_scale_head0": ("float vs = v_scale_kind == SCALE_PER_HEAD ? v_scale[g] : v_scale[0];",
                             "float vs = v_scale[0];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(O.SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    lib = O.load(O.build(str(mpath), str(tmp_path / "libmutant.so")))
    failures = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except Exception as e:  # noqa: BLE001 - any failure (assert, crash in numpy) counts
            failures.append((pin.__name__, type(e).__name__))
    assert failures, f"no pin catches mutant {name}"
