"""Planted mistakes in the oracle: its pins must catch each one.

Each mutant is a copy of the oracle package (``oracle.c`` and
``oracle/__init__.py``) with one plausible error written into it - a dropped
term, a wrong sign, constant, index or comparison, a transposed operand.  The
copy is built in a temporary directory and ``tests/test_oracle_pins.py`` runs
against it in a subprocess; the run must fail.  A control copy without a
change must pass, which shows that the subprocess really loads the copy.

Everything here runs on the CPU; nothing touches the CUDA library."""
import os
import re
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

C, PY = "oracle.c", "__init__.py"
# (name, file, text in the oracle, the same text with the planted mistake)
MUTANTS = [
    ("control", C, "", ""),
    # number formats
    ("decode_exponent_off_by_one", C,
     "(int)e - f->bias - f->mbits);", "(int)e - f->bias - f->mbits + 1);"),
    ("encode_ties_away_from_zero", C,
     "if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) == 1.0))", "if (frac >= 0.5)"),
    ("encode_no_subnormal_quantum", C,
     "    if (E < emin)\n        E = emin;", ""),
    ("e4m3fn_max_as_ieee", C,
     "return ldexp(2.0 - 2.0 * ldexp(1.0, -f->mbits), top - f->bias);",
     "return ldexp(2.0 - ldexp(1.0, -f->mbits), top - f->bias);"),
    ("bf16_nan_not_canonical", C,
     "static const orc_fmt FMT_BF16 = {8, 7, 127, 1, 0x7FC0u};",
     "static const orc_fmt FMT_BF16 = {8, 7, 127, 1, 0x7FFFu};"),
    # unscale / check
    ("unscale_multiplies_by_S", C,
     "    float inv_s = 1.0f / scale;\n    int found = 0;", "    float inv_s = scale;\n    int found = 0;"),
    ("check_misses_nan", C,
     "            if (!isfinite(g))\n                found = 1;",
     "            if (isinf(g))\n                found = 1;"),
    # scale state machine
    ("growth_strictly_greater", C, "if (*tracker >= interval) {", "if (*tracker > interval) {"),
    ("tracker_kept_on_overflow", C,
     "        *scale = *scale * backoff;\n        *tracker = 0;", "        *scale = *scale * backoff;"),
    ("found_inf_not_cleared", C, "    *found_inf = 0;\n    for (int i = 0; i < n_amax; ++i)",
     "    for (int i = 0; i < n_amax; ++i)"),
    # AdamW
    ("skip_advances_step", C,
     "        return; /* skipped step: no state, output or counter changes */",
     "    {\n        *step = *step + 1;\n        return;\n    }"),
    ("decay_dropped", C, "            p = p * decay;\n", "\n"),
    ("first_moment_uses_beta2", C, "m = b1 * m + omb1 * g;", "m = b2 * m + omb2 * g;"),
    ("second_moment_abs_not_square", C, "v = b2 * v + omb2 * (g * g);",
     "v = b2 * v + omb2 * fabsf(g);"),
    ("eps_inside_sqrt", C, "float denom = sqrtf(v) / bc2_sqrt + epsf;",
     "float denom = sqrtf(v + epsf) / bc2_sqrt;"),
    ("bias_correction2_not_rooted", C, "float bc2_sqrt = (float)sqrt(bc2);",
     "float bc2_sqrt = (float)bc2;"),
    ("no_bias_correction1", C, "float step_size = (float)(lr / bc1);",
     "float step_size = (float)lr;"),
    ("update_sign_flipped", C, "p = p - step_size * (m / denom);", "p = p + step_size * (m / denom);"),
    ("amax_of_master_not_bf16", C,
     "float a = fabsf((float)fmt_decode(&FMT_BF16, b));", "float a = fabsf(p);"),
    # clipping
    ("sumsq_of_abs", C, "            acc += g * g;", "            acc += fabs(g);"),
    ("clip_factor_not_capped", C, "return (float)(c < 1.0 ? c : 1.0);", "return (float)c;"),
    # tensorwise FP8
    ("fp8_scale_inverted", C, "    double scale_d = fmax / clamped;", "    double scale_d = clamped / fmax;"),
    ("fp8_eps_ignored", C,
     "double clamped = isnan(ad) ? ad : (ad < eps ? eps : ad);", "double clamped = ad;"),
    ("fp8_transpose_index", C, "                out_t[j * rows + i] = q;", "                out_t[i * cols + j] = q;"),
    ("fp8_inv_scale_not_reciprocal", C, "    *inv_scale = (float)(1.0 / scale_d);",
     "    *inv_scale = (float)scale_d;"),
    ("fp8_amax_drops_nan", C,
     "            if (isnan(v) || isnan(a))\n                a = NAN;\n            else if (v > a)",
     "            if (v > a)"),
    # rowwise FP8
    ("rowwise_copy_uses_row_scale", C,
     "out_t[j * rows + i] = cast_scaled(f, load_as_f32(xdtype, x, i * cols + j), scale_col[j]);",
     "out_t[j * rows + i] = cast_scaled(f, load_as_f32(xdtype, x, i * cols + j), scale_row[i < cols ? i : 0]);"),
    # group-wise FP8
    ("groupwise_group_one_short", C,
     "int64_t j0 = g * group, j1 = j0 + group < cols ? j0 + group : cols;",
     "int64_t j0 = g * group, j1 = j0 + group - 1 < cols ? j0 + group - 1 : cols;"),
    ("groupwise_copy_groups_by_row_scale", C,
     "out_t[j * rows + i] = cast_scaled(f, load_as_f32(xdtype, x, i * cols + j), scale_cg[k]);",
     "out_t[j * rows + i] = cast_scaled(f, load_as_f32(xdtype, x, i * cols + j), scale_rg[i * ((cols + group - 1) / group) + j / group]);"),
    # Philox / stochastic rounding
    ("philox_nine_rounds", C, "for (int r = 0; r < 10; ++r) {", "for (int r = 0; r < 9; ++r) {"),
    ("philox_key_weyl_swapped", C, "        k1 += 0xBB67AE85u;", "        k1 += 0x9E3779B9u;"),
    ("sr_rounds_up_on_grid", C, "uint32_t r = lo + ((u & 0xFFFFu) < frac ? 1u : 0u);",
     "uint32_t r = lo + ((u & 0xFFFFu) <= frac ? 1u : 0u);"),
    # stochastic rounding of the FP8 copies
    ("fp8_sr_rounds_up_at_the_threshold", C, "        if ((double)(u & 0xFFFFu) < num)",
     "        if ((double)(u & 0xFFFFu) <= num)"),
    ("fp8_sr_ratio_of_hi_not_gap", C,
     "double ratio = (a - grid[i]) / (grid[i + 1] - grid[i]);",
     "double ratio = (a - grid[i]) / grid[i + 1];"),
    ("fp8_sr_sign_dropped", C, "    return (uint8_t)fmt_encode(f, signbit(y) ? -r : r);",
     "    return (uint8_t)fmt_encode(f, r);"),
    ("fp8_sr_stream_not_marked", C,
     "    return sr_bits(seed, step, (int32_t)((uint32_t)tensor | 0x80000000u), k);",
     "    return sr_bits(seed, step, tensor, k);"),
    ("fp8_sr_threshold_of_32_bits", C, "        double num = floor(ratio * 65536.0);",
     "        double num = floor(ratio * 4294967296.0) / 65536.0;"),
    # delayed scaling (the composed step, in Python)
    ("delayed_uses_current_amax", PY,
     '                if self.fp8_scaling == "delayed":\n                    h = self.hist[s]',
     '                if False:\n                    h = self.hist[s]'),
    ("delayed_history_not_shifted", PY,
     "            self.hist[:, 1:] = self.hist[:, :-1].copy()\n", ""),
]


def _run(mutant, tmp_root):
    name, fname, old, new = mutant
    pkg = os.path.join(tmp_root, name, "oracle")
    os.makedirs(pkg)
    for f in (C, PY):
        with open(os.path.join(ROOT, "oracle", f)) as fh:
            src = fh.read()
        if f == fname and old:
            assert old in src, f"{name}: the text to mutate is no longer in oracle/{f}"
            src = src.replace(old, new, 1)
        with open(os.path.join(pkg, f), "w") as fh:
            fh.write(src)
    # the copy comes first on sys.path (cwd of `python -m`); the repository
    # after it, for the input generators and the test helpers
    env = dict(os.environ, PYTHONPATH=ROOT)
    probe = subprocess.run([sys.executable, "-c", "import oracle; print(oracle.__file__)"],
                           cwd=os.path.dirname(pkg), env=env, capture_output=True, text=True)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu", PINS], cwd=os.path.dirname(pkg), env=env,
                       capture_output=True, text=True, timeout=900)
    return probe.stdout.strip(), r


@pytest.fixture(scope="module")
def runs(tmp_path_factory):
    tmp = str(tmp_path_factory.mktemp("oracle_mutants"))
    with ThreadPoolExecutor(max_workers=max(2, min(8, os.cpu_count() or 2))) as ex:
        futs = {m[0]: ex.submit(_run, m, tmp) for m in MUTANTS}
        return {k: f.result() for k, f in futs.items()}


def _caught_by(out: str) -> str:
    m = re.search(r"FAILED \S+::(\S+)", out)
    return m.group(1) if m else "?"


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_catch_the_planted_mistake(runs, name):
    loaded, r = runs[name]
    assert loaded.startswith(os.path.dirname(os.path.dirname(loaded))) and \
        os.sep + name + os.sep in loaded, f"{name}: the copy was not the oracle imported ({loaded})"
    if name == "control":
        assert r.returncode == 0, r.stdout[-3000:]
    else:
        assert r.returncode == 1, f"{name}: no pin failed\n{r.stdout[-3000:]}{r.stderr[-2000:]}"
        print(f"{name}: caught by {_caught_by(r.stdout)}")
