"""Planted mistakes in the oracle must fail its pins.

Each case copies the oracle's C source, plants one plausible mistake (a
dropped term, a wrong sign, a wrong index, a misplaced eps, a wrong rounding,
a reversed slot order ...), compiles the copy on the CPU, and runs every pin
of tests/test_oracle.py, tests/test_oracle_nvfp4.py and
tests/test_oracle_expert_norm.py against it.  At least one pin must fail.  The real
oracle is never modified.
"""
import importlib.util
import inspect
import os

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))

MUTATIONS = {
    "residual_dropped": [
        ("x[i * H + h] = residual_in[t * H + h] + acc;", "x[i * H + h] = acc;")],
    "weight_sign": [
        ("acc = fmaf(w[t * k + j], e, acc);", "acc = fmaf(-w[t * k + j], e, acc);")],
    "index_map_ignored": [
        ("float e = bf16_to_f32(expert_out[(int64_t)r * H + h]);",
         "float e = bf16_to_f32(expert_out[((t * k + j) % R) * H + h]);")],
    "row_col_transposed": [
        ("float e = bf16_to_f32(expert_out[(int64_t)r * H + h]);",
         "float e = bf16_to_f32(expert_out[h * R + (int64_t)r]);")],
    "eps_outside_root": [
        ("double inv = 1.0 / sqrt(ss / (double)H + (double)eps);",
         "double inv = 1.0 / (sqrt(ss / (double)H) + (double)eps);")],
    "sum_not_mean": [
        ("double inv = 1.0 / sqrt(ss / (double)H + (double)eps);",
         "double inv = 1.0 / sqrt(ss + (double)eps);")],
    "one_plus_gamma": [
        ("y[i * H + h] = (double)xr[h] * inv * mfr_oracle_bf16_to_f64(gamma[h]);",
         "y[i * H + h] = (double)xr[h] * inv * (1.0 + mfr_oracle_bf16_to_f64(gamma[h]));")],
    "gamma_dropped": [
        ("y[i * H + h] = (double)xr[h] * inv * mfr_oracle_bf16_to_f64(gamma[h]);",
         "y[i * H + h] = (double)xr[h] * inv;")],
    "bf16_truncates": [("double q = nearbyint(a / spacing);", "double q = floor(a / spacing);")],
    "bf16_ties_away": [("double q = nearbyint(a / spacing);", "double q = round(a / spacing);")],
    "bf16_wrong_width": [("double spacing = ldexp(1.0, lead - 7);",
                          "double spacing = ldexp(1.0, lead - 8);")],
    "unfused_multiply_add": [
        ("acc = fmaf(w[t * k + j], e, acc);", "acc = w[t * k + j] * e + acc;")],
    "slots_reversed": [
        ("for (int64_t j = 0; j < k; ++j) {\n                int32_t r = idx[t * k + j];\n"
         "                if (!slot_valid(r, R))\n                    continue;\n"
         "                float e",
         "for (int64_t j = k - 1; j >= 0; --j) {\n                int32_t r = idx[t * k + j];\n"
         "                if (!slot_valid(r, R))\n                    continue;\n"
         "                float e")],
    "residual_first": [
        ("            float acc = 0.0f;\n            for (int64_t j = 0; j < k; ++j) {\n"
         "                int32_t r = idx[t * k + j];\n                if (!slot_valid(r, R))\n"
         "                    continue;\n                float e",
         "            float acc = residual_in[t * H + h];\n            for (int64_t j = 0; j < k; ++j) {\n"
         "                int32_t r = idx[t * k + j];\n                if (!slot_valid(r, R))\n"
         "                    continue;\n                float e"),
        ("x[i * H + h] = residual_in[t * H + h] + acc;", "x[i * H + h] = acc;")],
    "bad_slots_not_counted": [("            ++bad;\n", "")],
    "e4m3_truncates": [("    double r = nearbyint(a / spacing) * spacing;\n    if (r > 448.0)",
                        "    double r = floor(a / spacing) * spacing;\n    if (r > 448.0)")],
    "e4m3_no_saturation": [("    if (r > 448.0)\n        r = 448.0;", "")],
    "e2m1_ties_up": [("(d == db && (i & 1) == 0 && (best & 1) == 1)", "(d == db)")],
    "nibbles_swapped": [("(uint8_t)(c0 | (c1 << 4))", "(uint8_t)(c1 | (c0 << 4))")],
    "scale_not_rounded": [("            float sv = (float)mfr_oracle_e4m3_to_f64(s8);",
                           "            float sv = v;")],
    "encode_ignores_the_given_scale": [
        ("nvfp4_encode_block(y + i * H + b * 16, (float)mfr_oracle_e4m3_to_f64(sf[i * (H / 16) + b]),",
         "nvfp4_encode_block(y + i * H + b * 16, 1.0f,")],
    "scale_tiles_without_the_row_group": [
        ("int64_t within = (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4);",
         "int64_t within = (r % 32) * 16 + (c % 4);")],
    "scale_tiles_column_major": [
        ("int64_t tile = (r / 128) * col_tiles + c / 4;",
         "int64_t tile = (c / 4) * ((n + 127) / 128) + r / 128;")],
    "amax_over_8": [("            for (int j = 0; j < 16; ++j)\n                if (fabsf(yb[j]) > amax)",
                     "            for (int j = 0; j < 8; ++j)\n                if (fabsf(yb[j]) > amax)")],
    "expert_norm_gamma_dropped": [
        ("yr[h] += wj * (mfr_oracle_bf16_to_f64(row[h]) * inv * mfr_oracle_bf16_to_f64(gamma[h]));",
         "yr[h] += wj * (mfr_oracle_bf16_to_f64(row[h]) * inv);")],
    "expert_norm_weights_ignored": [("double wj = (double)w[t * k + j];", "double wj = 1.0;")],
    "expert_norm_mean_over_k": [("ss / (double)H + (double)eps);\n            double wj",
                                 "ss / (double)k + (double)eps);\n            double wj")],
    "expert_norm_squares_carried_across_slots": [
        ("            const uint16_t* row = expert_out + (int64_t)r * H;\n            double ss = 0.0;\n",
         "            const uint16_t* row = expert_out + (int64_t)r * H;\n"),
        ("        for (int64_t j = 0; j < k; ++j) {\n            int32_t r = idx[t * k + j];\n            if (!slot_valid(r, R))\n                continue;\n            const uint16_t* row",
         "        double ss = 0.0;\n        for (int64_t j = 0; j < k; ++j) {\n            int32_t r = idx[t * k + j];\n            if (!slot_valid(r, R))\n                continue;\n            const uint16_t* row")],
    "expert_norm_bad_slot_reads_row_0": [
        ("            if (!slot_valid(r, R))\n                continue;\n            const uint16_t* row",
         "            if (!slot_valid(r, R))\n                r = 0;\n            const uint16_t* row")],
    "finalize_only_double_rounding": [
        ("out[i * H + h] = mfr_oracle_bf16_from_f64((double)acc);",
         "out[i * H + h] = mfr_oracle_bf16_from_f64((double)(acc * 1.0009765625f));")],
}


def _load_pins():
    runs = []
    for fname in ("test_oracle.py", "test_oracle_nvfp4.py", "test_oracle_expert_norm.py"):
        runs += _pins_of(fname)
    return runs


def _pins_of(fname):
    spec = importlib.util.spec_from_file_location(fname[:-3], os.path.join(HERE, fname))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    runs = []
    for name, fn in inspect.getmembers(mod, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if params:
            argnames = [a.strip() for a in params[0].args[0].split(",")]
            for values in params[0].args[1]:
                runs.append((f"{name}{values}", fn, dict(zip(argnames, values))))
        else:
            runs.append((name, fn, {}))
    return runs


PINS = _load_pins()


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistake_is_caught(mutation, tmp_path):
    src = open(oracle.SOURCE).read()
    for old, new in MUTATIONS[mutation]:
        assert old in src, f"mutation anchor not found: {old!r}"
        src = src.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(src)
    lib = oracle.compile_oracle(str(path), str(tmp_path / f"lib_{mutation}.so"))
    mutant = oracle.Oracle(lib)
    failed = []
    for name, fn, kw in PINS:
        try:
            fn(oracle_lib=mutant, **kw)
        except AssertionError:
            failed.append(name)
    assert failed, f"no pin caught the planted mistake {mutation!r}"


def test_unmutated_copy_passes_every_pin(tmp_path):
    path = tmp_path / "copy.c"
    path.write_text(open(oracle.SOURCE).read())
    same = oracle.Oracle(oracle.compile_oracle(str(path), str(tmp_path / "lib_copy.so")))
    for name, fn, kw in PINS:
        fn(oracle_lib=same, **kw)
