"""The pins catch plausible mistakes.  The oracle is rebuilt with each
mistake planted in it (-DORACLE_MUTANT=n, the points are marked in
oracle/mxsa_oracle.c) and the pin files must fail against every one.  A
mistake no pin notices would mean a pin is missing."""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = ["tests/test_oracle_pins.py", "tests/test_store_pins.py", "tests/test_dedup_pins.py",
        "tests/test_select_pins.py", "tests/test_nvfp4_pins.py"]
MUTANTS = {
    1: "bf16 decoding with misplaced bits",
    2: "e4m3 decoding with the wrong exponent bias",
    3: "GQA map h % Hkv instead of h / G",
    4: "softmax scale dropped",
    5: "causal position off by one",
    6: "each block's last key dropped",
    7: "page walk by block instead of by page",
    8: "cache read as [page][pos][head]",
    9: "lse in base 2",
    10: "combine averages its parts unweighted",
    11: "index drops causal blocks one position early",
    12: "index entries in descending slot order",
    13: "dedup shares partial blocks",
    14: "dedup merges nothing",
    15: "decode runs split into one item too many",
    16: "e4m3 encoding rounds ties away from zero",
    17: "selection ties go to the larger block",
    18: "selection hides the row's own causal position",
    19: "selection scores drop the last index dimension",
    20: "selection scores a block by its minimum",
    21: "schedule treats a shared key of several entries as a decode key",
    22: "NVFP4 nibbles read in the swapped order",
    23: "E2M1 decoding with exponent bias 2",
    24: "E2M1 encoding rounds ties to the odd code",
    25: "NVFP4 group scale amax / 4 instead of amax / 6",
}


@pytest.mark.parametrize("n", sorted(MUTANTS))
def test_pins_catch_the_planted_mistake(n, tmp_path):
    lib = oracle.build_mutant(n, str(tmp_path))
    env = dict(os.environ, MXSA_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", *PINS], cwd=ROOT,
                       env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 1, f"mutant {n} ({MUTANTS[n]}) passed every pin:\n{r.stdout[-2000:]}"
