"""Plant plausible mistakes in copies of the oracle's C source; the pins must catch each one.

The mutants are built on the CPU in a temporary directory; nothing here runs on a GPU.
"""

import json
import os
import subprocess
import sys

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sgemm_oracle.c")

# (name, text to replace, replacement): each occurs once in the FP64 routine.
MUTANTS = [
    ("dropped_first_term", "for (int k = 0; k < K; ++k) {\n                        const double a",
     "for (int k = 1; k < K; ++k) {\n                        const double a"),
    ("wrong_sign", "s[j] += a * b;", "s[j] -= a * b;"),
    ("transposed_A", "const double a = (double)A[(long long)i * lda + k];", "const double a = (double)A[(long long)k * lda + i];"),
    ("ld_ignored_for_B", "B + (long long)k * ldb", "B + (long long)k * N"),
    ("reads_C_when_beta_zero", "if (beta != 0.0f) {\n                        const double c",
     "if (1) {\n                        const double c"),
    ("alpha_for_beta", "v += db * c;", "v += da * c;"),
    ("beta_missing_in_magnitude", "w += fabs(db) * fabs(c);", "w += 0.0;"),
    ("column_shift", "const double b = (double)brow[j];", "const double b = (double)brow[j + (j + 1 < N)];"),
    ("alpha_zero_reads_AB", "if (alpha != 0.0f) {\n                    for", "if (1) {\n                    for"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mut = tmp_path / "mut.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11", str(mut),
                    "-o", str(so), "-lm"], check=True, capture_output=True)
    # Run the pins in a child process: a mutant that indexes out of bounds may crash it,
    # which also counts as caught.
    here = os.path.dirname(os.path.abspath(__file__))
    script = (
        "import json, sys\n"
        f"sys.path[:0] = [{here!r}, {os.path.dirname(here)!r}]\n"
        "import oracle, oracle_pins\n"
        f"orc = oracle.Oracle({str(so)!r})\n"
        "caught = []\n"
        "for pin in oracle_pins.ALL_PINS:\n"
        "    try:\n"
        "        pin(orc)\n"
        "    except (AssertionError, ValueError):\n"
        "        caught.append(pin.__name__)\n"
        "print(json.dumps(caught))\n"
    )
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, timeout=300)
    if r.returncode != 0:
        return  # crashed: caught
    caught = json.loads(r.stdout.strip().splitlines()[-1])
    assert caught, f"no pin caught mutant {name}"
