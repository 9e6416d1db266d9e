"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import math

import numpy as np
import pytest

import oracle
import workloads as wl
from tests import oracle_checks as C

pytestmark = pytest.mark.cpu


def test_mapper_partition_and_closed_form():
    C.check_mapper(oracle)


def test_tiny_workload_request0_has_empty_shard():
    C.check_tiny_empty_shard(oracle)


def test_block_alignment():
    C.check_block_alignment(oracle)


def test_walker_roundtrip():
    C.check_walker(oracle)


def test_row_lengths_and_padding():
    C.check_row_lengths(oracle)


def test_attention_closed_forms():
    C.check_attention_closed_forms(oracle)


def test_attention_vs_torch_softmax():
    C.check_attention_vs_torch(oracle)


def test_combine_special_cases():
    C.check_combine_special_cases(oracle)


def test_combine_shard_order_invariance():
    C.check_combine_permutation(oracle)


def test_scale_from_query_row_width():
    facts = C.page_facts()
    qk_dims = int(facts["fp8_query_row_bytes"])  # one byte per fp8 element
    assert wl.TINY.scale == pytest.approx(1 / math.sqrt(qk_dims), rel=1e-15)
    assert wl.LONG_120K.scale == wl.TINY.scale


SMALL = [
    wl.TINY,
    wl.DecodeSpec("small_d8_i1_q1", seed=21, B=3, seq_lens=(1, 70, 130), H=4,
                  block_size=16, D=8, interleave=1),
    wl.DecodeSpec("small_d4_i16_bs64", seed=22, B=2, seq_lens=(200, 5), H=3,
                  block_size=64, D=4, interleave=16),
    wl.DecodeSpec("small_d2_i64_bs32", seed=23, B=2, seq_lens=(300, 64), H=2,
                  block_size=32, D=2, interleave=64),
    wl.DecodeSpec("small_q4_padding", seed=24, B=4, seq_lens=(50, 0, 3, 41), q_len=4,
                  H=2, block_size=16, D=4, interleave=1, extra_rows=3),
    wl.DecodeSpec("small_d1", seed=25, B=2, seq_lens=(9, 33), H=2, block_size=16,
                  D=1, interleave=1),
]


@pytest.mark.parametrize("spec", SMALL, ids=lambda s: s.name)
def test_decode_partials_and_identity(spec):
    """Sharded partials + combine = unsharded attention (torch float64)."""
    inp = wl.make_decode_inputs(spec)
    C.check_decode_rows_vs_torch(oracle, inp)


def test_tiny_partials_mask_empty_shard_with_nan():
    inp = wl.make_decode_inputs(wl.TINY)
    O, lse, rows = oracle.decode_partial(inp)
    assert (lse[3, 0] == -np.inf).all() and np.isnan(O[3, 0]).all()
    assert np.isfinite(lse[:3, 0]).all() and np.isfinite(lse[:, 1]).all()


def test_generator_is_deterministic_and_poisoned():
    a = wl.make_decode_inputs(SMALL[1])
    b = wl.make_decode_inputs(SMALL[1])
    for k in ("q", "kv_cache", "block_table", "seq_lens", "query_start_loc"):
        assert np.array_equal(a[k], b[k]), k
    # unused table columns hold -1; cache slots past a request's length hold NaN
    t = a["block_table"]
    assert (t[0, 1:] == -1).all()
    assert a["kv_cache"].reshape(-1, 576)[t[0, 0] * 16 + 1, 0] == wl.BF16_NAN


def test_concat_cache_is_cat_and_scatter():
    C.check_concat_cache(oracle)


def test_concat_cache_feeds_the_walker():
    C.check_concat_cache_feeds_the_walker(oracle)


def test_local_layout_matches_global():
    C.check_local_layout_matches_global(oracle)


def test_shared_prefix_blocks_and_values():
    C.check_shared_prefix(oracle)


def test_fp8_e4m3_widening():
    C.check_fp8_widening(oracle)


def test_fp8_decode_matches_its_bf16_twin():
    C.check_fp8_decode_matches_bf16_twin(oracle)
