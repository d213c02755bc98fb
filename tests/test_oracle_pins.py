"""The CPU oracle against its pins (values printed by the pages, brute force, closed
forms, invariants).  See pins.py for what each pin fixes."""
import math

import pytest

import pins
import workloads


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(oracle, pin):
    pin(oracle)


def test_kv_size_formula_matches_page_claim():
    """ia-vox-magazine: Llama-3-70B, 20 requests x 8000 tokens, bf16 -> more than 40 GB."""
    for claim in pins.kv_size_claims()["claims"]:
        got = workloads.kv_cache_bytes(claim["layers"], claim["kv_heads"], claim["head_dim"],
                                       claim["tokens"], claim["batch"], claim["bytes_per_value"])
        assert got > claim["lower_bound_bytes"]
        assert math.isclose(got, 52_428_800_000, rel_tol=1e-12)


def test_oracle_threads_reported(oracle):
    assert oracle.num_threads >= 1
