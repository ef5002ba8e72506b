"""Each planted mistake in the oracle must be caught by at least one pin.

The mistakes are compiled into separate copies of the oracle
(-DORACLE_MUTANT=n, CPU only); the oracle proper is built with n = 0.
"""
import os
import subprocess

import pytest

import oracle
import oracle_checks as oc

MUTANTS = {
    1: "RMS norm divides by H-1",
    2: "top-k ties go to the higher expert id",
    3: "per_expert_scale gathered by slot, not by expert id",
    4: "dispatch is not stable (reverse slot order)",
    5: "nibbles read high-first",
    6: "gate and up halves swapped",
    7: "combine sums unrounded products",
    8: "RMS norm with a weight drops the weight",
    9: "MoE branch routes on the normalised expert input",
    10: "4-bit router drops the biases",
    11: "dense MLP swaps the gate and up linears",
    12: "self-conditioning adds the embeddings after the post norm",
    13: "dense branch's post norm takes the pre norm's weight",
    14: "head softcap is tanh(x) * cap",
    15: "head softcap reads the unrounded logit",
    16: "router hidden**-0.5 scalar kept in fp32, not rounded to bf16",
    17: "router norm output not rounded to bf16 before the scale multiply",
    18: "RMSNorm with a weight rounds x*r to bf16 before the weight",
}


@pytest.mark.parametrize("n", sorted(MUTANTS), ids=lambda n: f"mutant{n}")
def test_mutant_is_caught(tmp_path, n):
    """Fails if the pins cannot tell this planted mistake from the oracle."""
    so = str(tmp_path / f"liboracle_m{n}.so")
    subprocess.run(oracle.compile_cmd(so, mutant=n), check=True)
    lib = oracle.load(so)
    caught = []
    for check in oc.ALL_CHECKS:
        try:
            check(lib)
        except AssertionError:
            caught.append(check.__name__)
    assert caught, f"no pin caught mutant {n}: {MUTANTS[n]}"
