"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that
the pins in ``test_oracle_pins.py`` catch every one of them.

Every planted mistake keeps all memory accesses inside their buffers, so a
mutant can only compute wrong values, never corrupt the test process."""
import os

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "rope_oracle.c")

# (name, text in rope_oracle.c, replacement)
MUTANTS = [
    ("interleave sign of the rotated odd member",
     "out[2 * p] = -v[2 * p + 1];", "out[2 * p] = v[2 * p + 1];"),
    ("half mode: rotated halves swapped",
     "out[i] = -v[L / 2 + i];\n      out[L / 2 + i] = v[i];", "out[i] = v[L / 2 + i];\n      out[L / 2 + i] = -v[i];"),
    ("backward: sin applied after the rotation",
     "for (int64_t j = 0; j < L; ++j) tmp[j] = xs[j] * load_elem(sin, cs_dt, crow + j);",
     "for (int64_t j = 0; j < L; ++j) tmp[j] = xs[j] * load_elem(sin, cs_dt, crow + (j ^ 1));"),
    ("backward: forward sign of the rotated term",
     "double dx = xs[j] * load_elem(cos, cs_dt, crow + j) - xrot[j];",
     "double dx = xs[j] * load_elem(cos, cs_dt, crow + j) + xrot[j];"),
    ("interleave sin element index",
     "double sn = load_elem(sin, cs_dt, crow + j);", "double sn = load_elem(sin, cs_dt, crow + (j ^ 1));"),
    ("interleave dropped sin term",
     "double y = xs[j] * c + xrot[j] * sn;", "double y = xs[j] * c;"),
    ("interleave cos taken from the pair's even slot",
     "double c = load_elem(cos, cs_dt, crow + j);", "double c = load_elem(cos, cs_dt, crow + (j & ~(int64_t)1));"),
    ("broadcast over N always",
     "const int64_t cn = cs_shape[2] == 1 ? 0 : n;", "const int64_t cn = 0;"),
    ("NeoX halves swapped",
     "x1 = xr[i];\n      x2 = xr[half + i];", "x1 = xr[half + i];\n      x2 = xr[i];"),
    ("o2 sign",
     "double o2 = x2 * cosv[i] + x1 * sinv[i];", "double o2 = x2 * cosv[i] - x1 * sinv[i];"),
    ("o1 transposed operands",
     "double o1 = x1 * cosv[i] - x2 * sinv[i];", "double o1 = x1 * sinv[i] - x2 * cosv[i];"),
    ("GPT-J output concatenated instead of interleaved",
     "out[2 * i] = o1;\n      out[2 * i + 1] = o2;", "out[i] = o1;\n      out[half + i] = o2;"),
    ("cos and sin halves swapped",
     "if (!mrope) {\n      for (int64_t i = 0; i < half; ++i) {\n        cosv[i] = cos_sin[i];\n        sinv[i] = cos_sin[half + i];",
     "if (!mrope) {\n      for (int64_t i = 0; i < half; ++i) {\n        cosv[i] = cos_sin[half + i];\n        sinv[i] = cos_sin[i];"),
    ("mrope ignores the section row for cos",
     "cosv[i] = cos_sin[k * R + i];", "cosv[i] = cos_sin[i];"),
    ("mrope sin read from the cos half",
     "sinv[i] = cos_sin[k * R + half + i];", "sinv[i] = cos_sin[k * R + i];"),
    ("interleaved splice: row 2 bound from the wrong section",
     "for (int64_t i = 2; i < 3 * mrope_section[1] && i < half; i += 3) {",
     "for (int64_t i = 2; i < 3 * mrope_section[0] && i < half; i += 3) {"),
    ("interleaved splice: row 1 stride start off by one",
     "for (int64_t i = 1; i < 3 * mrope_section[1] && i < half; i += 3) {",
     "for (int64_t i = 0; i < 3 * mrope_section[1] && i < half; i += 3) {"),
    ("fused: mean over D - 1",
     "const double rms = sqrt(ss / (double)D + eps);",
     "const double rms = sqrt(ss / (double)(D - 1) + eps);"),
    ("fused: gamma index shifted",
     "for (int64_t j = 0; j < D; ++j) y[j] = x[j] / rms * load_elem(gamma, dt, j);",
     "for (int64_t j = 0; j < D; ++j) y[j] = x[j] / rms * load_elem(gamma, dt, (j + 1) % D);"),
    ("fused: q gamma for k",
     "const void* gamma = h < nq ? q_gamma : k_gamma;", "const void* gamma = q_gamma;"),
    ("fused: rope sign",
     "o[j] = y[j] * c - y[half + j] * s;", "o[j] = y[j] * c + y[half + j] * s;"),
    ("fused: cache offset off by one (stays inside the block)",
     "const int64_t blk = cache_it ? slot / block_size : 0, off = cache_it ? slot % block_size : 0;",
     "const int64_t blk = cache_it ? slot / block_size : 0, off = cache_it ? (slot + 1) % block_size : 0;"),
    ("fused: position off by one",
     "const int64_t position = seq_lens[b] - (qsl[b + 1] - qsl[b]) + i;",
     "const int64_t position = seq_lens[b] - (qsl[b + 1] - qsl[b]) + i + 1;"),
    ("rounding ties away from zero",
     "double m = nearbyint(ldexp(a, (f.p - 1) - E));", "double m = round(ldexp(a, (f.p - 1) - E));"),
    ("rounding by truncation",
     "double m = nearbyint(ldexp(a, (f.p - 1) - E));", "double m = trunc(ldexp(a, (f.p - 1) - E));"),
    ("subnormal scale off by one",
     "v = ldexp((double)frac, emin - (f.p - 1));", "v = ldexp((double)frac, emin - f.p);"),
    ("exponent bias off by one",
     "(int)efield - f.emax - (f.p - 1));", "(int)efield - f.emax - f.p);"),
]

PIN_TESTS = [name for name in dir(pins) if name.startswith("test_")]


def _run_pins():
    failures = []
    for name in PIN_TESTS:
        fn = getattr(pins, name)
        params = getattr(fn, "pytestmark", [])
        arg_sets = [{}]
        for mark in params:
            if mark.name != "parametrize":
                continue
            argnames = [a.strip() for a in mark.args[0].split(",")]
            new = []
            for base in arg_sets:
                for v in mark.args[1]:
                    vals = v if len(argnames) > 1 else (v,)
                    new.append({**base, **dict(zip(argnames, vals))})
            arg_sets = new
        for kw in arg_sets:
            try:
                fn(**kw)
            except Exception:  # noqa: BLE001 - any failure counts as caught
                failures.append(name)
                break
        if failures:
            return failures
    return failures


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, "mutation site not found: " + name
    lib = oracle.build_copy(text.replace(old, new), str(tmp_path / "mutant.so"))
    try:
        oracle.use_library(lib)
        caught = _run_pins()
    finally:
        oracle.use_library(None)
    assert caught, "no pin caught: " + name
