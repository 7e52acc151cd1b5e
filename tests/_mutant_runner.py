"""Runs the oracle pins against another build of the oracle; prints CAUGHT if any pin fails."""
import sys

import oracle
from tests import test_oracle as pins

PIN_CALLS = [
    ("layout golden", pins.test_append_layout_golden),
    ("tiny vs torch", pins.test_tiny_config_vs_torch),
    ("random 3 vs torch", lambda: pins.test_random_tiny_vs_torch(3)),
    ("random 17 vs torch", lambda: pins.test_random_tiny_vs_torch(17)),
    ("one token", pins.test_one_token_context_returns_v_exactly),
    ("mean of V", pins.test_identical_keys_and_zero_query_give_mean_of_v),
    ("ratio closed form", pins.test_weights_sum_to_one_and_ratio_closed_form),
    ("large spike row", lambda: pins.test_score_row_shapes([0.5] * 5 + [2048.0] + [0.5] * 2)),
    ("dominant score", pins.test_dominant_score_selects_its_row_and_token_order),
    ("gqa mapping", pins.test_gqa_head_mapping),
]

if __name__ == "__main__":
    oracle.use_library(sys.argv[1])
    caught = []
    for name, call in PIN_CALLS:
        try:
            call()
        except AssertionError:
            caught.append(name)
    print(("CAUGHT by " + ", ".join(caught)) if caught else "MISSED")
