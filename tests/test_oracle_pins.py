"""The CPU oracle against facts outside itself (CPU only)."""
import pytest

import oracle_pins as P


def test_m1_pairs(oracle_lib):
    P.pin_m1_pairs(oracle_lib)


def test_m2_first_element_full_size(oracle_lib):
    P.pin_m2_first_element(oracle_lib)


def test_sentinel_start_rank(oracle_lib):
    P.pin_sentinel_start_rank(oracle_lib)


def test_bruteforce_order(oracle_lib):
    P.pin_bruteforce_order(oracle_lib)


def test_fp_error_bound(oracle_lib):
    P.pin_fp_error_bound(oracle_lib)


def test_rounding_16bit(oracle_lib):
    P.pin_rounding_16bit(oracle_lib)


def test_chunk_map(oracle_lib):
    P.pin_chunk_map(oracle_lib)


def test_fold_equals_simulation(oracle_lib):
    P.pin_fold_equals_simulation(oracle_lib)


def test_order_free_invariants(oracle_lib):
    P.pin_order_free_invariants(oracle_lib)


def test_sampled_equals_full(oracle_lib):
    P.pin_sampled_equals_full(oracle_lib)


def test_reduce_scatter_closed_form(oracle_lib):
    P.pin_reduce_scatter_closed_form(oracle_lib)


def test_reduce_scatter_order(oracle_lib):
    P.pin_reduce_scatter_order(oracle_lib)


def test_reduce_scatter_is_allreduce_blocks(oracle_lib):
    P.pin_reduce_scatter_is_allreduce_blocks(oracle_lib)


def test_rs_ag_equal_simulation(oracle_lib):
    P.pin_rs_ag_equal_simulation(oracle_lib)


def test_thread_count_does_not_change_result(oracle_lib):
    import numpy as np
    import oracle
    rng = np.random.default_rng(9)
    xs = [rng.standard_normal(10007).astype(np.float32) for _ in range(7)]
    one = oracle.allreduce(xs, "float32", "sum", 3, 256, nthreads=1, lib=oracle_lib)
    for t in (2, 5, 16):
        assert np.array_equal(one, oracle.allreduce(xs, "float32", "sum", 3, 256,
                                                    nthreads=t, lib=oracle_lib))


def test_rejects_bad_arguments(oracle_lib):
    import numpy as np
    import oracle
    xs = [np.zeros(4, np.float32)] * 2
    for chunk in (0, 8, 24):
        with pytest.raises(ValueError):
            oracle.allreduce(xs, "float32", "sum", 1, chunk, lib=oracle_lib)
    with pytest.raises(ValueError):
        oracle.allreduce(xs, "float32", "sum", 0, 16, lib=oracle_lib)


def test_tree_pages_examples(oracle_lib):
    P.pin_tree_pages_examples(oracle_lib)


def test_tree_structure(oracle_lib):
    P.pin_tree_structure(oracle_lib)


def test_tree_fold_by_hand(oracle_lib):
    P.pin_tree_fold_by_hand(oracle_lib)


def test_tree_sentinel(oracle_lib):
    P.pin_tree_sentinel(oracle_lib)


def test_tree_order_free(oracle_lib):
    P.pin_tree_order_free(oracle_lib)


def test_tree_split(oracle_lib):
    P.pin_tree_split(oracle_lib)


def test_scaled_ops(oracle_lib):
    P.pin_scaled_ops(oracle_lib)


def test_rounding_fp8(oracle_lib):
    P.pin_rounding_fp8(oracle_lib)


def test_tree_scaled_ops(oracle_lib):
    P.pin_tree_scaled_ops(oracle_lib)


def test_fp8_pairs_exhaustive(oracle_lib):
    P.pin_fp8_pairs_exhaustive(oracle_lib)
