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
    "check_commit_then_chain",
])
def test_pin(name):
    getattr(P, name)()


@pytest.mark.parametrize("S", [1, 2, 8])
def test_golden_attention_split_route(S):
    P.check_golden_attention(num_splits=S)
