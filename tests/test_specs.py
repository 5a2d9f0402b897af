"""The workload shapes follow the figures the pages print (tests/golden/k3_layer_specs.json)."""
import json
import os

from latent_compressed_expert_gb300 import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "k3_layer_specs.json")))


def test_full_shapes_match_printed_specs():
    for sh in (synth.PREFILL, synth.DECODE, synth.SKEW):
        assert sh.d == GOLD["hidden_width"]["value"]
        assert sh.L == GOLD["latent_width"]["value"]
        assert sh.L * 2 == sh.d  # "exactly half"
        assert sh.E == GOLD["routed_experts"]["value"]
        assert sh.K == GOLD["active_per_token"]["value"]
        assert sh.S == GOLD["shared_experts"]["value"]
        assert sh.c == GOLD["situ_cap_magnitude"]["value"]
        assert round(100.0 * sh.K / sh.E, 1) == GOLD["activation_ratio_percent"]["value"]
    # the alternative pool has the same activation ratio
    alt = GOLD["alternative_pool"]
    assert alt["active"] / alt["experts"] == synth.PREFILL.K / synth.PREFILL.E


def test_reduced_shapes_keep_the_latent_ratio():
    for sh in (synth.TINY, synth.E64):
        assert sh.L * 2 == sh.d
        assert sh.S == GOLD["shared_experts"]["value"]
