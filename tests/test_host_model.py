"""Runs the host unit test of the product's exact-math header
(tests/host_model/model_test.cpp) and the four planted mistakes of
Research-1433 ("Tests": always round a tie up, drop the binade check, drop the
upper bound check, ignore the parity when composing), each of which must fail."""
import os
import subprocess

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "tests", "host_model", "model_test.cpp")
OUT = os.path.join(ROOT, "tests", "_build")
FLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math"]


def _build(mutate=None):
    os.makedirs(OUT, exist_ok=True)
    exe = os.path.join(OUT, f"model_m{mutate}" if mutate else "model")
    cmd = ["g++", *FLAGS, "-o", exe, SRC, "-lm"]
    if mutate:
        cmd.insert(1, f"-DSEQSUM_MUTATE={mutate}")
    subprocess.check_call(cmd)
    return exe


def test_exact_math_header_on_host():
    exe = _build()
    r = subprocess.run([exe, "4000000"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "failures=0" in r.stdout


@pytest.mark.parametrize("mutate", [1, 2, 3, 4])
def test_planted_mistake_fails(mutate):
    exe = _build(mutate)
    r = subprocess.run([exe, "400000"], capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutation {mutate} was not caught:\n{r.stdout}"
