"""Planted mistakes in the oracle must each trip at least one pin (CPU only).

Each mutant is a copy of ``oracle/pa_oracle.c`` with one plausible mistake
(a dropped term, a wrong index or sign, a transposed layout), compiled into a
temporary directory.  The test passes only if some pin in ``oracle_pins``
fails on that copy, which shows the pins are strong enough to catch that
class of mistake in the real oracle.
"""
import os

import pytest

import oracle
import oracle_pins

# (name, text in pa_oracle.c, replacement)
MUTANTS = [
    ("no_max_subtraction", "const double w = exp(l[t] - M);", "const double w = exp(l[t]);"),
    ("head_map_modulo", "const int kvh = h / G; /* [GQA] */",
     "const int kvh = h % s->num_kv_heads;"),
    ("no_normalisation", "for (int d = 0; d < D; ++d) out[d] /= den;", ""),
    ("slot_off_by_one",
     "l[t] = orc_logit(s, q, k_cache, b, h, kvh, blk, (int)(t % s->block_size));",
     "l[t] = orc_logit(s, q, k_cache, b, h, kvh, blk, (int)((t + 1) % s->block_size));"),
    ("layout_head_slot_swapped",
     "return (((int64_t)blk * s->num_kv_heads + kvh) * s->block_size + off) * (int64_t)s->head_dim;",
     "return (((int64_t)blk * s->block_size + off) * s->num_kv_heads + kvh) * (int64_t)s->head_dim;"),
    ("scale_dropped", "return s->scale * dot;", "return dot;"),
    ("bf16_shift", "uint32_t w = (uint32_t)bits << 16;", "uint32_t w = (uint32_t)bits << 15;"),
    ("f16_bias", "v = ldexp(1.0 + (double)fr / 1024.0, ex - 15);",
     "v = ldexp(1.0 + (double)fr / 1024.0, ex - 14);"),
    ("phase2_drops_exp_sum", "total += exp(m[p] - gmax) * sp[p];", "total += exp(m[p] - gmax);"),
    ("phase2_weight_drops_exp_sum", "const double wgt = exp(m[p] - gmax) * sp[p] / total;",
     "const double wgt = exp(m[p] - gmax) / total;"),
    ("partition_not_normalised", "for (int d = 0; d < D; ++d) opp[d] /= sum;", ""),
    ("partition_end_off_by_one", "const int64_t t1 = (t0 + P < L) ? t0 + P : L;",
     "const int64_t t1 = (t0 + P - 1 < L) ? t0 + P - 1 : L;"),
    ("phase2_first_max_only", "if (m[p] > gmax) gmax = m[p];", "gmax = m[0];"),
    ("rescale_sign", "const double wgt = exp(m[p] - gmax) * sp[p] / total;",
     "const double wgt = exp(gmax - m[p]) * sp[p] / total;"),
    # subset mode: the requested rows are ignored, or placed in reverse order
    ("rows_ignored", "const int64_t row = rows ? rows[r] : r;\n    const int b = (int)(row",
     "const int64_t row = r;\n    const int b = (int)(row"),
    ("prefill_rows_reversed",
     "const int64_t row = rows ? rows[r] : r;\n    const int64_t t = row",
     "const int64_t row = rows ? rows[n - 1 - r] : r;\n    const int64_t t = row"),
    # paged prefix prefill
    ("prefill_causal_exclusive", "const int64_t nvis = (int64_t)C + (t - qs) + 1;",
     "const int64_t nvis = (int64_t)C + (t - qs);"),
    ("prefill_context_dropped", "const int64_t nvis = (int64_t)C + (t - qs) + 1;",
     "const int64_t nvis = (t - qs) + 1;"),
    ("prefill_new_row_ignores_sequence_start",
     "*base = (((int64_t)qs + (j - C)) * s->num_kv_heads + kvh) * (int64_t)s->head_dim;",
     "*base = ((j - C) * s->num_kv_heads + kvh) * (int64_t)s->head_dim;"),
    ("prefill_context_slot_off_by_one",
     "*base = orc_row(s, blk, kvh, (int)(j % s->block_size));",
     "*base = orc_row(s, blk, kvh, (int)((j + 1) % s->block_size));"),
    ("prefill_tiled_corr_sign", "const double corr = m == -INFINITY ? 0.0 : exp(m - m_new);",
     "const double corr = m == -INFINITY ? 0.0 : exp(m_new - m);"),
    ("prefill_tiled_sum_not_corrected", "    lsum *= corr;\n", ""),
    ("prefill_tiled_skips_context", "const int64_t end = phase == 0 ? C : i + 1;",
     "const int64_t end = phase == 0 ? 0 : i + 1;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(oracle.source()).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    bad_src = os.path.join(tmp_path, "pa_oracle.c")
    with open(bad_src, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.build(force=True, src=bad_src, out=os.path.join(tmp_path, "libmutant.so"))
    mutant = oracle.Oracle(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError) as e:
            caught.append(f"{pin.__name__}: {str(e)[:80]}")
    assert caught, f"no pin catches the planted mistake {name}"
