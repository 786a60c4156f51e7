"""Each planted mistake in the oracle (compiled in with ORACLE_MUTATION=n) fails at
least one pin, so the pins would catch that kind of error in the real oracle."""
import pytest

import oracle
from oracle_pins import PINS

MUTATIONS = {
    1: "causal mask flipped toward the future",
    2: "query head h reads kv head h % nkv (interleaved groups)",
    3: "scale missing from dK",
    4: "D_i computed without the O factor",
    5: "dK/dV receive only one head of the group",
    6: "LSE with a base-2 log",
    7: "dQ gathers the key at the query's row",
    9: "scale applied twice to the scores",
    10: "decode leaves out the newest cached key",
}


@pytest.mark.parametrize("mutation", sorted(MUTATIONS), ids=lambda m: f"m{m}")
def test_mutation_is_caught(mutation):
    orc = oracle.OracleLib(mutation)
    failed = []
    for pin in PINS:
        try:
            pin(orc)
        except (AssertionError, FloatingPointError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutation {mutation} ({MUTATIONS[mutation]}) passed every pin"
