"""Mutation test of the oracle's pins (CPU).

The pins in test_oracle_pins.py tie the oracle to what the pages and the
mathematics fix.  They are only worth something if a plausible mistake in the
oracle breaks one of them.  The oracle source carries a set of such mistakes
behind ORC_MUTANT (a dropped factor, a wrong constant, sign, index or operand,
a misplaced mask, the wrong logarithm, ...); each is built on its own and the
pins are run against it, and every one must fail.  Nothing here touches the GPU
or the CUDA library.
"""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))

# mutant -> what it gets wrong (the sites are marked ORC_MUT(n) in oracle/kvc_oracle.c)
MUTANTS = {
    1: "Eq. 21.2 without the factor 2 (keys only)",
    2: "Eq. 21.3 counts two positions",
    3: "bf16 bits placed one bit low in the binary32",
    4: "e4m3 subnormal step 2^-10",
    5: "e4m3 exponent bias 8",
    6: "e4m3 overflow to NaN instead of saturating",
    7: "e4m3 rounding toward zero",
    8: "int4 clamp to [-8, 7]",
    9: "int4 nibble bias 7",
    10: "int4 scale absmax / 8",
    11: "e4m3 scale absmax / 240",
    12: "block of position t taken as (t + 1) / bs",
    13: "slots reversed within a block",
    14: "pool layout with K|V outside the head index",
    15: "int4 nibbles swapped within a byte",
    16: "softmax scale dropped",
    17: "the newest position masked out",
    18: "values scaled by the key scales",
    19: "lse in log base 2",
    20: "query heads mapped to KV heads modulo H_KV",
    21: "prefill query hides its own key",
    22: "weights exponentiated twice",
    23: "uniform mean instead of softmax weights",
}


def test_every_mutant_is_named_in_the_source():
    src = open(os.path.join(os.path.dirname(oracle.__file__), "kvc_oracle.c")).read()
    for m in MUTANTS:
        assert f"ORC_MUT({m})" in src


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistake(mutant, tmp_path):
    so = str(tmp_path / f"libkvc_oracle_m{mutant}.so")
    subprocess.check_call(oracle.build_command(so, mutant))
    env = dict(os.environ, KVC_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(HERE, "test_oracle_pins.py"), "-x", "-q",
                        "-p", "no:cacheprovider"], env=env, cwd=os.path.dirname(HERE),
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, (f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin:\n"
                               + r.stdout[-2000:] + r.stderr[-2000:])
