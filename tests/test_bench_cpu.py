"""bench.py's algorithmic work counts and its choice of roofline (CPU only)."""
import numpy as np
import pytest

import bench
import workloads as wl

pytestmark = pytest.mark.cpu


def _host_dict(spec):
    seq = spec.resolved_seq_lens().astype(np.int32)
    ql = np.asarray(spec.q_lens(), dtype=np.int64)
    qsl = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    return dict(seq_lens=seq, query_start_loc=qsl, B=spec.B, T=int(qsl[-1]), H=spec.H, D=spec.D)


def test_decode_flops_counts_causal_rows_and_skips_padding():
    # request 0: q_len 2 over 5 tokens -> rows see 4 and 5 tokens; request 1
    # has no context (padding)
    inp = dict(seq_lens=np.array([5, 0], np.int32), query_start_loc=np.array([0, 2, 3], np.int32),
               B=2, T=3, H=16, D=4)
    assert bench.decode_flops(inp) == 2 * 16 * (576 + 512) * (4 + 5)
    assert bench.kv_tokens(inp) == 5


def test_roofline_is_tensor_only_where_flops_per_byte_pass_the_ridge():
    tpeak, _ = bench.tensor_peak()
    hpeak, _ = bench.peaks()
    ridge = tpeak * 1e12 / (hpeak * 1e9)
    got = {}
    for spec in (wl.LONG_120K, wl.BATCHED_B64, wl.SPEC_VERIFY_B32):
        inp = _host_dict(spec)
        got[spec.name] = bench.decode_flops(inp) / bench.decode_bytes(inp)
    # q_len 1: 2 x 128 x 1088 flop per 1152-byte KV row, less the partials'
    # share of the bytes; q_len 4 shares each row among four query rows
    assert got["long_ctx_120k_b1_d8_i1"] < ridge
    assert got["batched_b64_d8_i64"] < ridge
    assert got["spec_verify_b32_q4_d8_i1"] > ridge
    assert 200 < got["long_ctx_120k_b1_d8_i1"] < 2 * 128 * 1088 / 1152
