"""The oracle's pins catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle.c: a dropped factor or term,
a wrong sign, a swapped hyper-parameter, another rounding, a reading of the
page other than the one taken. It builds the copy as a separate library and
runs the pin tests covering the changed function against it (the oracle
package loads the library that ORACLE_LIB names). Every mutant must make a
pin fail. The control builds the unmodified source the same way and must pass
the same pins, so that a failure comes from the planted mistake and not from
the harness. The committed oracle.c is never modified.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

ENC = ["tests/test_oracle_encodings.py", "tests/test_oracle_codec.py"]
SPLIT = ["tests/test_oracle_split.py"]
OPTIM = ["tests/test_oracle_optim.py"]
FP32G = ["tests/test_oracle_fp32_grad.py"]

# (name, text in oracle.c, replacement, pin files expected to catch it)
MUTANTS = [
    # encodings
    ("bf16_ties_away", "return (toward_zero & 1u) ? away : toward_zero;", "return away;", ENC),
    ("fp16_truncates", "double r = rint(a / spacing) * spacing;", "double r = floor(a / spacing) * spacing;", ENC),
    ("fp16_no_overflow_to_inf", "if (a >= 65520.0)", "if (a >= 1e300)", ENC),
    # companding
    ("phi_m_drops_factor_2", "return (x + x) / (1.0f + fabsf(x));", "return x / (1.0f + fabsf(x));", ENC),
    ("phi_m_inv_wrong_sign", "return z / (2.0f - fabsf(z));", "return z / (2.0f + fabsf(z));", ENC),
    ("phi_v_identity", "float oracle_phi_v(float x) { return sqrtf(x); }",
     "float oracle_phi_v(float x) { return x; }", ENC),
    ("phi_v_inv_identity", "float oracle_phi_v_inv(float z) { return z * z; }",
     "float oracle_phi_v_inv(float z) { return z; }", ENC),
    # weight splitting
    ("split_symmetric_ulp", "float h = oracle_half_ulp(b, d < 0.0f ? -1 : +1);",
     "float h = oracle_half_ulp(b, +1);", SPLIT),
    ("half_ulp_is_full_ulp", "return (float)(fabs(b - a) * 0.5);", "return (float)(fabs(b - a));", SPLIT),
    ("rho_truncated", "float r = rintf(e * Q);", "float r = truncf(e * Q);", SPLIT),
    ("merge_ignores_rho_side", "float h = oracle_half_ulp(theta_p, rho < 0 ? -1 : +1);",
     "float h = oracle_half_ulp(theta_p, +1);", SPLIT),
    ("rho_levels_2_pow_b", "return rho_bits == 16 ? 32767 : 127;", "return rho_bits == 16 ? 32768 : 128;", SPLIT),
    # group quantization
    ("codes_truncated", "code = rintf(c[i] * inv);", "code = truncf(c[i] * inv);", ENC),
    ("no_fp16_scale_cap", "uint16_t s = oracle_fp16_rne(fminf(a, 65504.0f));",
     "uint16_t s = oracle_fp16_rne(a);", ENC),
    ("dequant_step_over_128", "float step = sf / (kind_signed(kind) ? 127.0f : 255.0f);",
     "float step = sf / (kind_signed(kind) ? 128.0f : 255.0f);", ENC),
    ("no_v_floor", "if (kind == ORACLE_VARIANCE_NONZERO && code < 1.0f)", "if (0)", ENC),
    ("groups_of_16", "for (int64_t g0 = 0; g0 < n; g0 += ORACLE_GROUP) {\n        int len = (int)(n - g0 < ORACLE_GROUP ? n - g0 : ORACLE_GROUP);\n        quant_group(",
     "for (int64_t g0 = 0; g0 < n; g0 += 16) {\n        int len = (int)(n - g0 < 16 ? n - g0 : 16);\n        quant_group(", ENC),
    # AdamW
    ("adamw_no_bc1", "k.step_size = (float)(hp->lr / bc1);", "k.step_size = (float)hp->lr;", OPTIM),
    ("adamw_no_bc2", "k.inv_sqrt_bc2 = (float)(1.0 / sqrt(bc2));", "k.inv_sqrt_bc2 = 1.0f;", OPTIM),
    ("adamw_bc1_off_by_one", "double bc1 = 1.0 - pow_int(hp->beta1, step);",
     "double bc1 = 1.0 - pow_int(hp->beta1, step + 1);", OPTIM),
    ("adamw_v_not_squared", "float vv = fmaf(k->beta2, *v, (k->c2 * g) * g);",
     "float vv = fmaf(k->beta2, *v, k->c2 * g);", OPTIM),
    ("adamw_eps_inside_sqrt", "float den = fmaf(sqrtf(vv), k->inv_sqrt_bc2, k->eps);",
     "float den = sqrtf(fmaf(vv, k->inv_sqrt_bc2 * k->inv_sqrt_bc2, k->eps));", OPTIM),
    ("adamw_no_weight_decay", "float th = *theta * decay;\n    float mm", "float th = *theta;\n    float mm", OPTIM),
    ("adamw_m_with_beta2", "float mm = fmaf(k->beta1, *m, k->c1 * g);", "float mm = fmaf(k->beta2, *m, k->c1 * g);",
     OPTIM),
    # SGD
    ("sgd_weight_decay_sign", "float gp = fmaf(weight_decay, *theta, g);", "float gp = fmaf(-weight_decay, *theta, g);",
     OPTIM),
    ("sgd_dampened", "float mm = fmaf(mu, *m, gp);", "float mm = fmaf(mu, *m, (1.0f - mu) * gp);", OPTIM),
    # Lion
    ("lion_sign_from_beta2", "float c = fmaf(k->beta1, *m, k->c1 * g);", "float c = fmaf(k->beta2, *m, k->c2 * g);",
     OPTIM),
    ("lion_m_with_beta1", "*m = fmaf(k->beta2, *m, k->c2 * g);", "*m = fmaf(k->beta1, *m, k->c1 * g);", OPTIM),
    # the fused step's gradient path
    ("fp32_grad_rounded_to_bf16", "float g = t->grad_is_f32 ? ((const float *)t->grad)[g0 + i]",
     "float g = t->grad_is_f32 ? oracle_bf16_to_f32(oracle_bf16_rne(((const float *)t->grad)[g0 + i]))", FP32G),
]


def _build(tmp_path, text, name):
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", *oracle.CFLAGS, "-I", os.path.dirname(oracle._SRC), "-o", str(so), str(src), "-lm"],
                   check=True, capture_output=True)
    return so


def _run_pins(so, files, extra=()):
    env = dict(os.environ, ORACLE_LIB=str(so))
    return subprocess.run([sys.executable, "-m", "pytest", *files, "-q", "-p", "no:cacheprovider",
                           "-m", "not gpu", *extra], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)


def _parallel():
    """pytest-xdist's workers for the control's full pin run, where installed."""
    try:
        import xdist  # noqa: F401
    except ImportError:
        return ()
    return ("-n", str(min(8, os.cpu_count() or 1)))


@pytest.fixture(scope="module")
def source():
    with open(oracle._SRC) as f:
        return f.read()


@pytest.fixture(scope="module")
def mutant_runs(tmp_path_factory, source):
    """Every mutant built and its pins run, several at a time (each run is a
    separate process on its own library)."""
    tmp = tmp_path_factory.mktemp("mutants")
    jobs = {}
    for name, old, new, files in MUTANTS:
        if source.count(old) == 1:
            jobs[name] = (_build(tmp, source.replace(old, new), name), files)
    with cf.ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        futures = {name: ex.submit(_run_pins, so, files, ("-x",)) for name, (so, files) in jobs.items()}
        return {name: f.result() for name, f in futures.items()}


def test_control_passes_the_pins(tmp_path, source):
    so = _build(tmp_path, source, "control")
    files = sorted({f for m in MUTANTS for f in m[3]})
    r = _run_pins(so, files, _parallel())
    assert r.returncode == 0, r.stdout[-3000:]


@pytest.mark.parametrize("name,old,new,files", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_the_mutant(source, mutant_runs, name, old, new, files):
    assert source.count(old) == 1, f"{name}: the planted text must occur once in oracle.c"
    r = mutant_runs[name]
    # exit status 1: tests ran and at least one failed (2-4 would be a usage,
    # collection or internal error of the harness, not a caught mutant)
    assert r.returncode == 1, f"{name} survived the pins:\n{r.stdout[-3000:]}"
