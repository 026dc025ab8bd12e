"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of ``oracle/oracle.c`` (a dropped
term, a wrong sign, index or operand), builds it with gcc on the CPU, and runs
every pin in ``test_oracle_pins.py``, ``test_oracle_nvfp4_pins.py`` and
``test_oracle_mxfp4_pins.py`` against it: at least one pin must fail.
The oracle itself is never modified.
"""
import inspect
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle
from tests import test_oracle_mxfp4_pins as mxfp4_pins
from tests import test_oracle_nvfp4_pins as nvfp4_pins
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    # the tolerance scale |s_p| * sum_h |w| |x_h| that every fp8 parity check uses
    "mag_rectified_dot": ("bound += fabs((double)w[h]) * fabs(x[h]);",
                          "bound += fabs((double)w[h]) * r;"),
    "mag_weight_sign_kept": ("bound += fabs((double)w[h]) * fabs(x[h]);",
                             "bound += (double)w[h] * fabs(x[h]);"),
    "mag_scale_dropped": ("J->mag[row * J->out_stride + p] = fabs(s) * bound;",
                          "J->mag[row * J->out_stride + p] = bound;"),
    "mag_extra_factor": ("J->mag[row * J->out_stride + p] = fabs(s) * bound;",
                         "J->mag[row * J->out_stride + p] = fabs(s) * bound * H;"),
    "relu_dropped": ("double r = x[h] > 0.0 ? x[h] : 0.0;", "double r = x[h];"),
    "relu_after_sum": ("J->out[row * J->out_stride + p] = s * acc;",
                       "J->out[row * J->out_stride + p] = s * (acc > 0.0 ? acc : 0.0);"),
    "scale_dropped": ("J->out[row * J->out_stride + p] = s * acc;",
                      "J->out[row * J->out_stride + p] = acc;"),
    "scale_wrong_index": ("ORC_BLOCK_KEY_BYTES + 4 * (p % ORC_BLOCK_KEYS)",
                          "ORC_BLOCK_KEY_BYTES + 4 * (p / ORC_BLOCK_KEYS)"),
    "weight_sign_lost": ("acc += (double)w[h] * r;", "acc += fabs((double)w[h]) * r;"),
    "key_transposed": ("J->e4m3[qrow[h * ORC_HEAD_DIM + d]] * J->e4m3[k[d]]",
                       "J->e4m3[qrow[h * ORC_HEAD_DIM + d]] * J->e4m3[blk[d * ORC_BLOCK_KEYS + p % ORC_BLOCK_KEYS]]"),
    "q_transposed": ("qrow[h * ORC_HEAD_DIM + d]", "qrow[d * H / 2 + h]"),
    "slot_ignored": ("const int64_t row = (int64_t)b * n + t;\n        const uint8_t* qrow = J->q + row * H * ORC_HEAD_DIM;",
                     "const int64_t row = (int64_t)b * n + t;\n        const uint8_t* qrow = J->q + (int64_t)b * n * H * ORC_HEAD_DIM;"),
    "block_table_row_ignored": ("J->block_table[(int64_t)b * J->bt_stride + p / ORC_BLOCK_KEYS]",
                                "J->block_table[p / ORC_BLOCK_KEYS]"),
    "e4m3_subnormal_scale": ("ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    "e4m3_bias": ("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    "bf16_page_stride_fixed": ("page * J->page_stride_bytes +\n                                (int64_t)(k % ORC_BLOCK_KEYS)",
                               "page * 16384 +\n                                (int64_t)(k % ORC_BLOCK_KEYS)"),
    "bf16_group_rows": ("for (int r = g * G; r < (g + 1) * G; ++r) {\n        const uint16_t* qr",
                        "for (int r = g; r < g + G; ++r) {\n        const uint16_t* qr"),
    "nvfp4_group_rows": ("for (int r = g * G; r < (g + 1) * G; ++r) {\n        const uint8_t* qp",
                         "for (int r = g; r < g + G; ++r) {\n        const uint8_t* qp"),
    "bf16_key_stride": ("(int64_t)(k % ORC_BLOCK_KEYS) * ORC_HEAD_DIM * 2", "(int64_t)(k % ORC_BLOCK_KEYS) * ORC_HEAD_DIM"),
    "schedule_ceil_split": ("int64_t base = total / num_ctas, extra = total % num_ctas;",
                            "int64_t base = (total + num_ctas - 1) / num_ctas, extra = 0;"),
    "schedule_skips_empty_wrong": ("if (start < prefix + nb) break;", "if (start <= prefix + nb) break;"),
    "nvfp4_scale_per_8": ("J->e4m3[scales[d / 16]]", "J->e4m3[scales[(d / 8) % 8]]"),
    "nvfp4_key_scale_row": ("(int64_t)key * (ORC_HEAD_DIM / 16)", "(int64_t)key * (ORC_HEAD_DIM / 32)"),
    "nvfp4_scale_stride_fixed": ("page * J->scale_page_stride_bytes", "page * 512"),
    "nvfp4_query_scale_by_group": ("J->query_scales + (int64_t)r * (ORC_HEAD_DIM / 16)",
                                   "J->query_scales + (int64_t)g * (ORC_HEAD_DIM / 16)"),
    "e2m1_bias": ("ldexp(1.0 + m / 2.0, e - 1)", "ldexp(1.0 + m / 2.0, e)"),
    "e2m1_subnormal": ("e == 0 ? 0.5 * m :", "e == 0 ? 1.0 * m :"),
    "e8m0_bias": ("ldexp(1.0, (int)code - 127)", "ldexp(1.0, (int)code - 128)"),
    "mxfp4_scale_per_16": ("orc_e8m0_decode(scales[d / 32])", "orc_e8m0_decode(scales[(d / 16) % 4])"),
    "mxfp4_key_scale_row": ("ORC_FP4_BLOCK_CODE_BYTES + (p % ORC_BLOCK_KEYS) * ORC_FP4_ROW_SCALES",
                            "ORC_FP4_BLOCK_CODE_BYTES + (p / ORC_BLOCK_KEYS) * ORC_FP4_ROW_SCALES"),
    "mxfp4_q_scale_head_ignored": ("J->q_sf + (row * H + h) * ORC_FP4_ROW_SCALES",
                                   "J->q_sf + (row * H) * ORC_FP4_ROW_SCALES"),
    "mxfp4_relu_dropped": ("const double rl = x[h] > 0.0 ? x[h] : 0.0;", "const double rl = x[h];"),
    "mxfp4_block_bytes": ("J->kv + phys * ORC_FP4_BLOCK_BYTES", "J->kv + phys * ORC_FP4_BLOCK_CODE_BYTES"),
    "mxfp4_block_table_row_ignored": ("J->block_table[J->bt_stride * (int64_t)b + p / ORC_BLOCK_KEYS]",
                                      "J->block_table[p / ORC_BLOCK_KEYS]"),
    "mxfp4_slot_ignored": ("J->q + (row * H + h) * ORC_FP4_ROW_BYTES",
                           "J->q + ((int64_t)b * n * H + h) * ORC_FP4_ROW_BYTES"),
}


def _pin_functions():
    out = []
    members = (inspect.getmembers(pins, inspect.isfunction) +
               inspect.getmembers(nvfp4_pins, inspect.isfunction) +
               inspect.getmembers(mxfp4_pins, inspect.isfunction))
    for name, fn in members:
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if params:
            argnames = [a.strip() for a in params[0].args[0].split(",")]
            for vals in params[0].args[1]:
                vals = vals if isinstance(vals, tuple) else (vals,)
                out.append((name, fn, dict(zip(argnames, vals))))
        else:
            out.append((name, fn, {}))
    return out


def _build_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique in oracle.c"
    path_c = os.path.join(tmp_path, f"{name}.c")
    path_so = os.path.join(tmp_path, f"lib{name}.so")
    with open(path_c, "w") as f:
        f.write(src.replace(old, new))
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", path_c, "-o",
                    path_so, "-lm"], check=True)
    return path_so


def test_every_mutant_fails_a_pin(tmp_path):
    names = sorted(MUTANTS)
    with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        libs = dict(zip(names, ex.map(lambda n: _build_mutant(n, str(tmp_path)), names)))
    golden = os.path.join(os.path.dirname(pins.__file__), "golden")
    survivors = []
    for name in names:
        caught = []
        with oracle.using_library(libs[name]):
            for tname, fn, kwargs in _pin_functions():
                args = dict(kwargs)
                if "tmp_path" in inspect.signature(fn).parameters:
                    args["tmp_path"] = tmp_path
                if "golden_dir" in inspect.signature(fn).parameters:
                    args["golden_dir"] = golden
                try:
                    fn(**args)
                except (AssertionError, ValueError, IndexError):
                    caught.append(tname)
                    break
        if not caught:
            survivors.append(name)
    assert not survivors, f"no pin caught: {survivors}"


def test_unmutated_copy_passes_all_pins(tmp_path):
    """Control: the same harness with the real source must pass every pin."""
    path_so = os.path.join(str(tmp_path), "libcontrol.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", SRC, "-o",
                    path_so, "-lm"], check=True)
    with oracle.using_library(path_so):
        for tname, fn, kwargs in _pin_functions():
            fn(**kwargs)
