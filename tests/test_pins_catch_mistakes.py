"""The oracle's pins must catch plausible mistakes in the oracle itself. Each case plants one
mistake in a copy of smx_oracle.c (a wrong table entry, a dropped or shifted term, a wrong sign,
index or rounding direction, a transposed operand), builds it, and runs the oracle's pin tests
against it: at least one pin must fail. Mistakes that give the same results by construction
are not planted (a different maximum in the softmax's first pass; clamping q at 464 instead of
448, since 464 is the e4m3 midpoint that rounds to 448 anyway)."""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PIN_FILES = ["tests/test_oracle_formats.py", "tests/test_oracle_index.py", "tests/test_oracle_attention.py",
             "tests/test_oracle_nvfp4.py"]

# (name, text in smx_oracle.c, replacement, occurrences replaced)
MISTAKES = [
    # element formats
    ("e2m1_table_entry", "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 5.0}", 1),
    ("e8m0_bias", "ldexp(1.0, byte - 127)", "ldexp(1.0, byte - 128)", 1),
    ("e4m3_subnormal_step", "v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);", 1),
    ("e4m3_value_bias", "ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)", 1),
    ("bf16_shift", "(uint32_t)bits << 16", "(uint32_t)bits << 15", 1),
    ("e2m1_tie_away_from_zero", "if (a <= 0.25) code = 0;", "if (a < 0.25) code = 0;", 1),
    ("e2m1_tie_1p25_up", "else if (a <= 1.25) code = 2;", "else if (a < 1.25) code = 2;", 1),
    ("e2m1_positive_zero", "uint8_t sign = signbit(v) ? 0x8 : 0x0;",
     "uint8_t sign = (signbit(v) && fabs(v) > 0.25) ? 0x8 : 0x0;", 1),
    ("e4m3_ties_away", "n = nearbyint(ldexp(a, -qexp));", "n = floor(ldexp(a, -qexp) + 0.5);", 1),
    ("e4m3_encode_bias", "return (uint8_t)(sign | ((E + 7) << 3) | m);", "return (uint8_t)(sign | ((E + 6) << 3) | m);", 1),
    # quantisers and the page layout
    ("mxfp4_scale_rule", "se = (ex - 1) - 2;", "se = (ex - 1) - 1;", 1),
    ("mxfp4_scale_clamp", "if (se < -127) se = -127;", "if (se < -126) se = -126;", 1),
    ("mxfp4_zero_group_scale", "        int se = 0;\n        if (amax > 0.0) {", "        int se = -127;\n        if (amax > 0.0) {", 1),
    ("mxfp4_nonfinite_kept", "if (!isfinite(xg[i])) nonfinite = 1;", "if (isnan(xg[i])) nonfinite = 1;", 1),
    ("nibble_order", "nib64[i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));",
     "nib64[i] = (uint8_t)(codes[2 * i + 1] | (codes[2 * i] << 4));", 2),
    ("scale_byte_slot", "memcpy(page + 8192 + (size_t)slot * 4, scale4, 4);",
     "memcpy(page + 8192 + (size_t)(slot ^ 1) * 4, scale4, 4);", 1),
    ("load_group_index", "orc_e8m0_value(sc[d / ORC_GROUP])", "orc_e8m0_value(sc[d % 4])", 1),
    ("rowscale_divisor", "amax / 448.0f", "amax / 240.0f", 1),
    ("rowscale_multiply_by_reciprocal", "float y = x[i] / s;", "float y = x[i] * (1.0f / s);", 1),
    ("rowscale_load_divides", "* (double)s;", "/ (double)s;", 1),
    ("pack_q_nan_byte", "if (isnan(v)) return 0x7F;", "if (isnan(v)) return 0xFF;", 1),
    ("pack_q_saturation", "if (v > 448.0) v = 448.0;", "if (v > 480.0) v = 480.0;", 1),
    # insert
    ("insert_position", "insert_token(sh, b, (int64_t)ctx_len[b] - sh->Q + t,",
     "insert_token(sh, b, (int64_t)ctx_len[b] - sh->Q + t - 1,", 1),
    ("insert_v_from_k", "store_kv_row(sh, kv_page(sh, v_pool, phys, h), slot, v_row + (size_t)h * ORC_D, sh->nv_scale_v);",
     "store_kv_row(sh, kv_page(sh, v_pool, phys, h), slot, k_row + (size_t)h * ORC_D, sh->nv_scale_v);", 1),
    # index score and top-k
    ("score_causal_off_by_one", "if (j > pos_t) continue;", "if (j >= pos_t) continue;", 1),
    ("score_no_causal_mask", "if (j > pos_t) continue;", "(void)pos_t;", 1),
    ("score_query_row", "const uint16_t* qt = qidx_bf16 + ((size_t)b * sh->Q + t) * ORC_D;",
     "const uint16_t* qt = qidx_bf16 + ((size_t)b * sh->Q) * ORC_D;", 1),
    ("score_min_not_max", "if (s > best) best = s;", "if (s < best || best == -INFINITY) best = s;", 1),
    ("topk_tie_to_higher_id", "    if (sa < sb) return 0;\n    return a < b;", "    if (sa < sb) return 0;\n    return a > b;", 1),
    ("topk_nan_ranks_first", "return nb;      /* a number beats NaN */", "return na;", 1),
    ("topk_one_too_many", "if (rank < k_eff) out[c++] = (int32_t)p;", "if (rank <= k_eff) out[c++] = (int32_t)p;", 1),
    ("block_min_not_max", "(isnan(m) || s[p] > m)) m = s[p];", "(isnan(m) || s[p] < m)) m = s[p];", 1),
    # split and merge
    ("attn_scale_1_over_d", "const double inv_sqrt_d = 1.0 / sqrt((double)ORC_D);",
     "const double inv_sqrt_d = 1.0 / (double)ORC_D;", 1),
    ("attn_kv_head_map", "int kvh = h / G;", "int kvh = h % sh->Hkv;", 1),
    ("attn_q_transposed", "size_t qbase = (((size_t)b * sh->Q + t) * sh->Hq + h) * ORC_D;",
     "size_t qbase = (((size_t)b * sh->Hq + h) * sh->Q + t) * ORC_D;", 1),
    ("attn_causal_mask", "if (j >= ctx || j > pos_t) continue;", "if (j >= ctx) continue;", 2),
    ("attn_v_is_k", "load_kv_row(sh, vp, slot, sh->nv_scale_v, vrow);", "load_kv_row(sh, kp, slot, sh->nv_scale_v, vrow);", 1),
    ("attn_natural_exp", "double w = exp2(dot * inv_sqrt_d * M_LOG2E - m);", "double w = exp(dot * inv_sqrt_d - m);", 1),
    ("split_partitions_overlap", "hi = (int)(((int64_t)(s + 1) * k_eff) / S);",
     "hi = (int)(((int64_t)(s + 1) * k_eff + S - 1) / S);", 1),
    ("block_first_page_only", "* ppb + e % ppb;", "* ppb;", 2),
    ("merge_natural_exp", "double w = exp2(part_m[pi] - M);", "double w = exp(part_m[pi] - M);", 1),
    ("merge_unnormalised", "for (int d = 0; d < ORC_D; ++d) o[d] /= L;", "(void)L;", 1),
    # NVFP4 pages
    ("nvfp4_scale_divisor", "volatile float six_g = 6.0f * g;", "volatile float six_g = 4.0f * g;", 1),
    ("nvfp4_scale_without_g", "volatile float s = amax / six_g;", "volatile float s = amax / 6.0f;", 1),
    ("nvfp4_no_saturation", "if (sc > 448.0) sc = 448.0;", "(void)0;", 1),
    ("nvfp4_element_scale_without_g", "volatile float S = (float)orc_e4m3_value(byte) * g;",
     "volatile float S = (float)orc_e4m3_value(byte);", 1),
    ("nvfp4_nonfinite_byte", "scale8[blk] = 0x7F;", "scale8[blk] = 0xFF;", 1),
    ("nvfp4_zero_scale_divides", "            if (S == 0.0f) {", "            if (0) {", 1),
    ("nvfp4_load_block_size", "orc_e4m3_value(sc[d / ORC_NV_BLOCK])", "orc_e4m3_value(sc[d / ORC_GROUP])", 1),
    ("nvfp4_load_without_g", "orc_e4m3_value(sc[d / ORC_NV_BLOCK]) * (double)g;", "orc_e4m3_value(sc[d / ORC_NV_BLOCK]);", 1),
    ("nvfp4_scale_slot", "memcpy(page + 8192 + (size_t)slot * 8, scale8, 8);",
     "memcpy(page + 8192 + (size_t)slot * 4, scale8, 8);", 1),
    ("nvfp4_index_takes_k_scale", "orc_nvfp4_quant_row(x, sh->nv_scale_idx, nib, sc);",
     "orc_nvfp4_quant_row(x, sh->nv_scale_k, nib, sc);", 1),
    ("nvfp4_score_takes_k_scale", "orc_nvfp4_load_row(page, slot, sh->nv_scale_idx, krow);",
     "orc_nvfp4_load_row(page, slot, sh->nv_scale_k, krow);", 1),
    ("nvfp4_v_takes_k_scale", "load_kv_row(sh, vp, slot, sh->nv_scale_v, vrow);", "load_kv_row(sh, vp, slot, sh->nv_scale_k, vrow);", 1),
    # the reusing layer's step
    ("reuse_skips_insert", "    orc_kv_insert(sh, k_new, v_new, NULL, page_table, ctx_len, k_pool, v_pool, NULL);\n",
     "", 1),
]


def _build_copy(name, src):
    d = os.path.join(ROOT, "oracle", "_build", "mistakes", name)
    os.makedirs(d, exist_ok=True)
    with open(os.path.join(d, "smx_oracle.c"), "w") as f:
        f.write(src)
    shutil.copy(os.path.join(ROOT, "oracle", "smx_oracle.h"), d)
    lib = os.path.join(d, "liboracle.so")
    oracle.compile_library(os.path.join(d, "smx_oracle.c"), lib, quiet=True)
    return lib


def _source():
    return open(os.path.join(ROOT, "oracle", "smx_oracle.c")).read()


def _build_mistake(name, old, new, count):
    src = _source()
    assert src.count(old) == count, f"{name}: the planted text occurs {src.count(old)} times"
    return _build_copy(name, src.replace(old, new))


def _run_pins(lib):
    env = dict(os.environ, SMX_ORACLE_LIB=lib, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "not gpu", *PIN_FILES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


def _one(case):
    lib = _build_mistake(*case)
    return _run_pins(lib)


def test_every_planted_mistake_fails_a_pin():
    names = [m[0] for m in MISTAKES]
    assert len(set(names)) == len(names)
    with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        results = list(ex.map(_one, MISTAKES))
    survivors = [(m[0], out) for m, (rc, out) in zip(MISTAKES, results) if rc != 1]
    assert not survivors, "mistakes no pin catches (or that broke the run):\n" + "\n".join(
        f"--- {n}\n{o}" for n, o in survivors)


def test_unchanged_copy_passes_the_pins():
    """The harness itself: the unchanged source built the same way passes every pin."""
    lib = _build_copy("unchanged", _source())
    rc, out = _run_pins(lib)
    assert rc == 0, out
