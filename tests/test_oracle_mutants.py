"""Plant plausible mistakes in a copy of the oracle and check the pins catch each.

Each mutant is a textual edit of oracle/ink_oracle.c compiled into a temporary
library; the pin suite (tests/test_oracle_pins.py, a subset) then runs in a
child process against it.  The unmodified source must pass, every mutant
must fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ink_oracle.c")

MUTANTS = {
    "no bottom-right offset": ("const int64_t q_abs = i + Lk - Lq;", "const int64_t q_abs = i;"),
    "bias sign": ("sj += (double)a->rel[", "sj -= (double)a->rel["),
    "bias by kv head": ("((int64_t)t * a->H + h) * a->E + rd]", "((int64_t)t * a->H + g) * a->E + rd]"),
    "extent off by one": ("if (rd >= 0 && rd < a->E)", "if (rd >= 0 && rd + 1 < a->E)"),
    "gqa head map": ("const int32_t g = h / G;", "const int32_t g = h % a->Hkv;"),
    "window edge": ("if (a->wl >= 0 && j < q_abs - a->wl) return 0;", "if (a->wl >= 0 && j <= q_abs - a->wl) return 0;"),
    "right window edge": ("if (a->wr >= 0 && j > q_abs + a->wr) return 0;", "if (a->wr >= 0 && j >= q_abs + a->wr) return 0;"),
    "causal excludes diagonal": ("if (a->causal && j > q_abs) return 0;", "if (a->causal && j >= q_abs) return 0;"),
    "lse without log": ("lse[r] = m + log(l);", "lse[r] = m + l;"),
    "values from key cache": ("cache_elem(a, 1, vrow + d)", "cache_elem(a, 0, vrow + d)"),
    "e4m3 exponent bias": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e4m3 subnormal scale": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "e4m3 sign dropped": ("return sign ? -v : v;", "return v;"),
    "fp8 scales swapped": ("(value ? a->v_scale : a->k_scale)", "(value ? a->k_scale : a->v_scale)"),
    "fp8 value scale ignored": ("(value ? a->v_scale : a->k_scale)", "(value ? 1.0 : a->k_scale)"),
    "bias scaled": ("sj += (double)a->rel[", "sj += a->scale * (double)a->rel["),
    "row within page reversed": ("(((int64_t)page * a->BS + j % a->BS) * a->Hkv + g) * a->D;\n            double dot",
                                 "(((int64_t)page * a->BS + (a->BS - 1 - j % a->BS)) * a->Hkv + g) * a->D;\n            double dot"),
    "merge weight without l": ("const double w = exp(m - gmax) * l;", "const double w = exp(m - gmax);"),
    "unnormalised partials": ("tot[d] += w * (acc[d] / l);", "tot[d] += w * acc[d];"),
    "query of group leader": ("const uint16_t *qrow = a->q + ((int64_t)t * a->H + h) * a->D;",
                              "const uint16_t *qrow = a->q + ((int64_t)t * a->H + (h / G) * G) * a->D;"),
    "head dim half read": ("            for (int32_t d = 0; d < a->D; ++d)\n", "            for (int32_t d = 0; d < a->D / 2; ++d)\n"),
    "page index by row": ("a->bt[(int64_t)b * a->MAXBLK + j / a->BS];\n            if (page < 0",
                          "a->bt[(int64_t)b * a->MAXBLK + j % a->BS];\n            if (page < 0"),
}

PIN_SUBSET = ("dense or closed or split or zero_query or single_key or constant or diagonal or unread or sdpa "
              "or fp8")


def _build(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    lib = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c99", "-fopenmp", "-fPIC", "-shared", str(src), "-o", str(lib), "-lm"],
                   check=True)
    return str(lib)


def _pins_pass(lib) -> bool:
    env = dict(os.environ, INK_ORACLE_LIB=lib, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-x", "-q",
           "-k", PIN_SUBSET, "-p", "no:cacheprovider"]
    r = subprocess.run(cmd, env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    return r.returncode == 0


def test_unmodified_oracle_passes(tmp_path):
    assert _pins_pass(_build(tmp_path, "control", open(SRC).read()))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation site for {name!r} not found"
    lib = _build(tmp_path, "mutant", text.replace(old, new))
    assert not _pins_pass(lib), f"pins did not catch mutant {name!r}"
