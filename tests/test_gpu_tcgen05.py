"""The bf16 attention paths on the tcgen05 kernel (pkv_set_attention_kernel(PKV_KERNEL_TCGEN05)).

The same parity and invariance checks as for the default kernel, rerun with the calls routed
to the 5th-generation tensor-core kernel (128-key tiles, accumulators in tensor memory):
within tolerance of the float64 oracle on every workload shape (decode, sinks, verify
windows, draft trees, prefill chunks, the index-list gather, ragged lengths at both head
sizes and block sizes, contexts beyond 64 splits), and bit for bit on the GPU for batch
versus solo, verify row versus decode, prefill row versus decode, permuted and shared
blocks, NaN in unused slots and a full in-order key list versus paged attention
(TensorSharp "高级功能", section "原生分页注意力"; TensorFold article, section
"先记住一条铁律").  The timeout path of its bounded waits is driven too.
"""
import pytest

import test_gpu_attention as A
import test_gpu_gather as Gt
import test_gpu_timeout as To
import test_gpu_tree as Tr

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_attention_forward_gb300 import pkv as m
    m.lib(build_if_missing=True)
    return m


@pytest.fixture(autouse=True)
def tcgen05_kernel(pkv):
    pkv.set_attention_kernel(pkv.PKV_KERNEL_TCGEN05)
    try:
        yield
    finally:
        pkv.set_attention_kernel(pkv.PKV_KERNEL_MMA_SYNC)


test_attention_matches_oracle = A.test_attention_matches_oracle
test_ministral_layers_match_oracle = A.test_ministral_layers_match_oracle
test_float32_output = A.test_float32_output
test_batch_vs_solo_bit_identical = A.test_batch_vs_solo_bit_identical
test_window_rows_equal_single_row_decodes = A.test_window_rows_equal_single_row_decodes
test_block_permutation_bit_identical = A.test_block_permutation_bit_identical
test_shared_prefix_vs_duplicated_blocks_bit_identical = A.test_shared_prefix_vs_duplicated_blocks_bit_identical
test_nan_in_unused_slots_changes_nothing = A.test_nan_in_unused_slots_changes_nothing
test_ragged_lengths_all_variants = A.test_ragged_lengths_all_variants
test_contexts_beyond_sixty_four_splits = A.test_contexts_beyond_sixty_four_splits
test_group_of_eight_with_sixteen_row_windows = A.test_group_of_eight_with_sixteen_row_windows
test_chunked_prefill_windows = A.test_chunked_prefill_windows
test_empty_context_and_sequences_without_rows = A.test_empty_context_and_sequences_without_rows
test_explicit_head_map_and_scale = A.test_explicit_head_map_and_scale
test_workspace_is_reusable_across_calls = A.test_workspace_is_reusable_across_calls
test_device_side_checks_report_and_do_not_fault = A.test_device_side_checks_report_and_do_not_fault
test_tree_attention_matches_oracle = Tr.test_tree_attention_matches_oracle
test_chain_masks_bit_identical_to_causal_window = Tr.test_chain_masks_bit_identical_to_causal_window
test_tree_batch_vs_solo_bit_identical = Tr.test_tree_batch_vs_solo_bit_identical
test_sparse_gather_matches_oracle = Gt.test_sparse_gather_matches_oracle
test_ragged_lists_and_shapes = Gt.test_ragged_lists_and_shapes
test_full_in_order_list_equals_paged_attention = Gt.test_full_in_order_list_equals_paged_attention
test_gather_batch_vs_solo_bit_identical = Gt.test_batch_vs_solo_bit_identical
test_bf16_waits_that_give_up_report_timeout = To.test_bf16_waits_that_give_up_report_timeout
test_index_list_gather_waits_that_give_up_report_timeout = To.test_index_list_gather_waits_that_give_up_report_timeout


def test_kernel_choice_is_checked(pkv):
    with pytest.raises(pkv.PkvError):
        pkv.set_attention_kernel(7)
