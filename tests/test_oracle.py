"""The fp64 oracle against its pins (CPU only)."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("name", [
    "check_fp16_golden", "check_fp16_all_patterns", "check_bf16_decode", "check_q8_golden",
    "check_tree_masks_golden", "check_row_map_mixed", "check_split_golden",
    "check_split_rule_properties", "check_gather_golden", "check_paged_equals_contiguous",
    "check_golden_attention", "check_brute_force", "check_weights_sum_to_one",
    "check_closed_forms", "check_split_invariance", "check_chain_is_tree_with_chain_parents",
    "check_direct_rows_independent_of_launch", "check_tree_commit_golden",
    "check_commit_then_chain", "check_device_split_golden", "check_device_split_properties",
])
def test_pin(name):
    getattr(P, name)()


@pytest.mark.parametrize("S", [1, 2, 8])
def test_golden_attention_split_route(S):
    P.check_golden_attention(num_splits=S)


def test_parallel_oracle_equals_the_oracle():
    """The row-parallel driver of the full-size tests only distributes rows:
    its result is the oracle's, bit for bit."""
    import numpy as np

    import oracle
    import synthetic as sy
    from oracle_parallel import oracle_full
    recipe = ("mixed_tree_direct", {"ctx": [40, 300, 17, 130, 64, 5, 90, 200]})
    case = sy.mixed_tree_direct(ctx=recipe[1]["ctx"])
    O, L = oracle_full(recipe, case)
    O2, L2 = oracle.verify_case(case)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)
