"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that the
pins catch every one. This is what shows the pins constrain the oracle rather
than merely agreeing with it."""
import os
import subprocess

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "causal bound off by one": ("const long n = P + i + 1;", "const long n = P + i + (i > 0);"),
    "causal bound ignores prefix": ("const long n = P + i + 1;", "const long n = i + 1;"),
    "head map h % HKV": ("h / group, scale, s);", "h % HKV, scale, s);"),
    "scale dropped": ("s[j] = dot * scale;", "s[j] = dot;"),
    "scale squared": ("s[j] = dot * scale;", "s[j] = dot * scale * scale;"),
    "values read from K": ("acc += s[j] * (double)v[", "acc += s[j] * (double)k["),
    "exponent sign flipped": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "no final division": ("out_row[d] = acc / Z;", "out_row[d] = acc;"),
    "key d index reversed": ("(double)kj[d];", "(double)kj[D - 1 - d];"),
    "value d index fixed": ("* D + d];", "* D + 0];"),
    "last key dropped from sum": ("Z += s[j];", "Z += (j + 1 < n) ? s[j] : 0.0;"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name!r} not unique"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", "-o", str(lib),
                    str(path), "-lm"], check=True)
    return oracle.load_variant(str(lib))


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    attention = _build_mutant(tmp_path, name, old, new)
    caught = []
    for pin in ALL_PINS:
        try:
            with __import__("warnings").catch_warnings():
                __import__("warnings").simplefilter("ignore")
                pin(attention)
        except (AssertionError, RuntimeError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the mutant {name!r}"
