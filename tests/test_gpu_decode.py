"""GPU decode (+ combine) parity with the float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import mla_decode_context_gb300 as dcp
from tests import gpu_util as G

pytestmark = pytest.mark.gpu

# Sizes the oracle finishes in seconds that still span several tiles, ragged
# tails, empty shards, padding requests and rows past the last request.
SMALL = [
    wl.TINY,
    wl.DecodeSpec("h128_d8_i1_ragged", seed=31, B=3, seq_lens=(1, 700, 2049), H=128, block_size=64,
                  D=8, interleave=1),
    wl.DecodeSpec("h128_d8_i64_blocks", seed=32, B=3, seq_lens=(1500, 333, 64), H=128, block_size=64,
                  D=8, interleave=64),
    wl.DecodeSpec("h128_q4_causal_padding", seed=33, B=4, seq_lens=(0, 2, 903, 4), q_len=4, H=128,
                  block_size=64, D=8, interleave=1, extra_rows=2),
    wl.DecodeSpec("h128_d1", seed=34, B=2, seq_lens=(300, 17), H=128, block_size=16, D=1, interleave=1),
    wl.DecodeSpec("h128_d2_i16_bs32", seed=35, B=2, seq_lens=(777, 65), H=128, block_size=32, D=2,
                  interleave=16),
    wl.DecodeSpec("h64_d4_i3_unaligned", seed=36, B=2, seq_lens=(250, 40), H=64, block_size=16, D=4,
                  interleave=3),
    wl.DecodeSpec("h16_q2_bs16", seed=37, B=3, seq_lens=(5, 1, 60), q_len=2, H=16, block_size=16, D=4,
                  interleave=1),
    wl.DecodeSpec("h128_long_split", seed=38, B=1, seq_lens=(9000,), H=128, block_size=64, D=8,
                  interleave=1),
    # the largest shard count (32); 64-token blocks hold two tokens per shard
    wl.DecodeSpec("h128_d32_i1_max_shards", seed=40, B=2, seq_lens=(5000, 700), H=128, block_size=64,
                  D=32, interleave=1),
    # more heads than the tensor-core kernel takes: the CUDA-core kernel runs
    # under both parametrisations
    wl.DecodeSpec("h256_d4_i2_wide_heads", seed=41, B=2, seq_lens=(300, 1000), H=256, block_size=16, D=4,
                  interleave=2),
    # one shard, long: 32 splits of 9 tiles, more than the split merge
    # loads at once (its batched path)
    wl.DecodeSpec("h128_d1_32_splits", seed=42, B=1, seq_lens=(9000,), H=128, block_size=64, D=1,
                  interleave=1),
    # head counts that leave TMEM lane quarters partly or wholly empty
    wl.DecodeSpec("h1_d2_i1_single_head", seed=44, B=2, seq_lens=(700, 65), H=1, block_size=16, D=2,
                  interleave=1),
    wl.DecodeSpec("h33_d4_i2_odd_heads", seed=45, B=2, seq_lens=(1200, 3), q_len=2, H=33, block_size=32, D=4,
                  interleave=2),
    wl.DecodeSpec("h100_d8_i1_partial_quarter", seed=46, B=2, seq_lens=(2500, 90), H=100, block_size=64, D=8,
                  interleave=1),
    # verification widths: 8 rows a request (the widest run side by side in
    # the unit order), mixed widths that still group by 4 across requests,
    # and 9 rows (no grouping), with a block size and an interleave that are
    # not powers of two
    wl.DecodeSpec("h128_q8_rows_innermost", seed=47, B=3, seq_lens=(9, 1500, 3000), q_len=8, H=128, block_size=64,
                  D=8, interleave=1),
    wl.DecodeSpec("h128_mixed_q_group4", seed=48, B=4, seq_lens=(700, 5, 2000, 64), q_len=(4, 2, 2, 4), H=128,
                  block_size=64, D=4, interleave=2),
    wl.DecodeSpec("h64_q9_bs48_i5", seed=49, B=3, seq_lens=(400, 20, 1000), q_len=(9, 1, 5), H=64, block_size=48,
                  D=4, interleave=5),
    # shard lengths on tile and split edges (32, 256, 257 tokens a shard)
    wl.DecodeSpec("h128_tile_edges_bs80", seed=50, B=4, seq_lens=(128, 1024, 1028, 1027), H=128, block_size=80,
                  D=4, interleave=1, extra_rows=1),
    # more units than clusters, so one split per shard: 20-25 tiles per unit
    # (every stage, S buffer and P slot reused several times)
    wl.DecodeSpec("h128_b12_unsplit", seed=39, B=12,
                  seq_lens=(5000, 6100, 5300, 6400, 5700, 5100, 6000, 5500, 6300, 5200, 5900, 6200),
                  H=128, block_size=64, D=8, interleave=1),
]


def _full_check(inp, rows=None):
    t = G.to_device(inp)
    O, lse, err = G.run_decode(inp, t)
    assert err == 0
    out, out_lse = G.run_combine(O, lse, t)
    O_ref, lse_ref, rows = oracle.decode_partial(inp, rows)
    O_g = O.cpu().numpy()[:, rows]
    lse_g = lse.cpu().numpy()[:, rows]
    G.check_partials(O_g, lse_g, O_ref, lse_ref, inp["name"])
    _, _, pad = oracle.row_lengths(inp["seq_lens"], inp["query_start_loc"], inp["T"])
    out_ref, out_lse_ref = oracle.lse_combine(O_ref, lse_ref, pad[rows])
    G.check_combined(out.float().cpu().numpy()[rows], out_lse.cpu().numpy()[rows], out_ref, out_lse_ref,
                     pad[rows], inp["name"])
    return O, lse, out, out_lse


@pytest.fixture(params=["tc", "simt"])
def kernel(request, monkeypatch):
    """Default path (tensor cores where the layout allows) and the forced
    CUDA-core reference kernel."""
    if request.param == "simt":
        monkeypatch.setenv("DCP_FORCE_SIMT", "1")
    else:
        monkeypatch.delenv("DCP_FORCE_SIMT", raising=False)
    return request.param


@pytest.mark.parametrize("spec", SMALL, ids=lambda s: s.name)
def test_decode_matches_oracle(spec, kernel):
    _full_check(wl.make_decode_inputs(spec))


SPLIT_COUNTS = {1500: 6, 2300: 9, 2900: 12, 3900: 16}


@pytest.mark.parametrize("n", sorted(SPLIT_COUNTS), ids=lambda n: "%d_splits" % SPLIT_COUNTS[n])
def test_split_merge_source_counts(n, kernel):
    """One shard of n tokens splits into 6, 9, 12 or 16 chunks of 256: each
    count takes another shape of the split merge (two warps per pair up to 8
    and up to 12 sources, four warps up to 16).  The second request is short,
    so most of its splits are empty and merge as zero-weight sources."""
    spec = wl.DecodeSpec("h128_d1_%d" % n, seed=43, B=2, seq_lens=(n, 100), H=128, block_size=64, D=1,
                         interleave=1)
    inp = wl.make_decode_inputs(spec)
    # the decode and the split merge (plus the unit-order kernel when units
    # outnumber the clusters of one wave)
    assert dcp.dcp_decode_kernel_launches(inp["B"], inp["T"], 128, 1, 1, inp["max_seq_len"], 1, 1 << 30) >= 2
    _full_check(inp)


def test_decode_is_deterministic(kernel):
    inp = wl.make_decode_inputs(SMALL[1])
    t = G.to_device(inp)
    a = G.run_decode(inp, t)
    b = G.run_decode(inp, t)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_strided_rows_match_dense():
    inp = wl.make_decode_inputs(SMALL[3])
    t = G.to_device(inp)
    O, lse, _ = G.run_decode(inp, t)
    T, H = t["q"].shape[:2]
    qw = torch.zeros((T, H + 3, 576), dtype=torch.bfloat16, device="cuda")
    qw[:, :H] = t["q"]
    tw = torch.full((t["block_table"].shape[0], t["block_table"].shape[1] + 5), -7, dtype=torch.int32,
                    device="cuda")
    tw[:, :t["block_table"].shape[1]] = t["block_table"]
    O2, lse2, _ = G.run_decode(inp, t, q=qw[:, :H], block_table=tw[:, :t["block_table"].shape[1]])
    assert torch.equal(O, O2) and torch.equal(lse, lse2)


def test_unit_order_does_not_change_results():
    """More units than clusters (12 rows x 8 shards, unsplit): with the full
    workspace the long units start first; with no workspace they start in
    index order.  Every unit's arithmetic is its own, so the partials are
    bit-identical either way."""
    inp = wl.make_decode_inputs(SMALL[-1])
    t = G.to_device(inp)
    T, H = t["q"].shape[:2]
    B, D, msl = inp["B"], inp["D"], max(1, inp["max_seq_len"])
    ws_bytes = dcp.dcp_decode_workspace_size(B, T, H, D, msl, 1)
    ordered = dcp.dcp_decode_kernel_launches(B, T, H, D, inp["interleave"], msl, 1, ws_bytes)
    plain = dcp.dcp_decode_kernel_launches(B, T, H, D, inp["interleave"], msl, 1, 0)
    assert ordered == plain + 1  # the ordering kernel runs only with room for the order
    outs = []
    for ws in (torch.empty(ws_bytes, dtype=torch.uint8, device="cuda"), None):
        O = torch.empty((D, T, H, 512), dtype=torch.float32, device="cuda")
        lse = torch.empty((D, T, H), dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        dcp.dcp_mla_decode_partial(t["q"], t["kv_cache"], t["block_table"], t["seq_lens"], t["query_start_loc"],
                                   O, lse, D=D, interleave=inp["interleave"], scale=inp["scale"], max_seq_len=msl,
                                   max_q_len=1, workspace=ws, dev_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append((O, lse))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_empty_batch_is_a_noop():
    inp = wl.make_decode_inputs(wl.TINY)
    t = G.to_device(inp)
    O = torch.full((4, 0, 16, 512), 7.0, device="cuda")
    lse = torch.full((4, 0, 16), 7.0, device="cuda")
    dcp.dcp_mla_decode_partial(t["q"][:0], t["kv_cache"], t["block_table"], t["seq_lens"],
                               t["query_start_loc"], O, lse, D=4, interleave=1, scale=0.1, max_seq_len=37,
                               max_q_len=1)
    torch.cuda.synchronize()


def test_bad_block_id_is_flagged_not_trapped(kernel):
    spec = wl.DecodeSpec("bad_block", seed=39, B=2, seq_lens=(200, 90), H=128, block_size=16, D=4,
                         interleave=1)
    inp = wl.make_decode_inputs(spec)
    inp["block_table"] = inp["block_table"].copy()
    inp["block_table"][0, 3] = inp["num_blocks"] + 1000  # referenced column, outside the cache
    t = G.to_device(inp)
    O, lse, err = G.run_decode(inp, t)
    assert err & dcp.DEVERR_BAD_BLOCK
    assert not torch.isnan(O).any() and not torch.isnan(lse).any()
    # request 1 is untouched by the bad id
    O_ref, lse_ref, rows = oracle.decode_partial(inp, [1])
    G.check_partials(O.cpu().numpy()[:, rows], lse.cpu().numpy()[:, rows], O_ref, lse_ref, "req1")


def test_wait_that_runs_out_is_reported_and_the_context_survives(monkeypatch):
    """Failure detection without a fault: a test hook makes one wait of the
    tensor-core decode run out (a barrier nothing completes).  Every wait is
    bounded, so the launch ends on its own, with DCP_DEVERR_TIMEOUT in
    dev_error, and the next decode on the same context is correct."""
    monkeypatch.delenv("DCP_FORCE_SIMT", raising=False)
    spec = wl.DecodeSpec("stall_h128_d1", seed=43, B=1, seq_lens=(200,), H=128, block_size=64, D=1,
                         interleave=1)
    inp = wl.make_decode_inputs(spec)
    t = G.to_device(inp)
    monkeypatch.setenv("DCP_TEST_STALL_WAIT", "1")
    _, _, err = G.run_decode(inp, t)
    assert err & dcp.DEVERR_TIMEOUT
    monkeypatch.delenv("DCP_TEST_STALL_WAIT")
    O, lse, err = G.run_decode(inp, t)
    assert err == 0
    O_ref, lse_ref, rows = oracle.decode_partial(inp)
    G.check_partials(O.cpu().numpy()[:, rows], lse.cpu().numpy()[:, rows], O_ref, lse_ref, spec.name)


def test_seq_len_above_declared_max_is_flagged():
    inp = wl.make_decode_inputs(SMALL[7])
    t = G.to_device(inp)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dcp.decode_partial(t["q"], t["kv_cache"], t["block_table"], t["seq_lens"], t["query_start_loc"], D=4,
                       interleave=1, scale=0.1, max_seq_len=50, max_q_len=2, dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & dcp.DEVERR_SEQ_TOO_LONG


# --- the four decode workloads at full size, sampled rows ------------------
@pytest.fixture(scope="module")
def long_inputs():
    return wl.make_decode_inputs(wl.LONG_120K)


def test_long_context_120k(long_inputs):
    _full_check(long_inputs, rows=[0])


def test_long_context_repeats_are_bit_identical(long_inputs):
    """Thirty back-to-back decodes of the 120k workload (72 clusters, 53
    tiles each, every barrier ring reused many times) give bit-identical
    partials: the result does not depend on how the warps' timing falls."""
    t = G.to_device(long_inputs)
    O0, lse0, err = G.run_decode(long_inputs, t)
    assert err == 0
    for _ in range(29):
        O, lse, err = G.run_decode(long_inputs, t)
        assert err == 0
        assert torch.equal(O, O0) and torch.equal(lse, lse0)


def test_batched_b64(tmp_path):
    inp = wl.make_decode_inputs(wl.BATCHED_B64)
    seq = inp["seq_lens"]
    rows = [int(np.argmin(seq)), int(np.argmax(seq)), 5, 40]
    _full_check(inp, rows=rows)


def test_spec_verify_b32():
    inp = wl.make_decode_inputs(wl.SPEC_VERIFY_B32)
    seq = inp["seq_lens"]
    b = int(np.argmax(seq))
    rows = list(range(4 * b, 4 * b + 4)) + [4 * 7 + 1]
    O0, lse0, _, _ = _full_check(inp, rows=rows)
    # more units than clusters (launch order by length, rows of a request
    # side by side): repeats are bit-identical
    t = G.to_device(inp)
    for _ in range(4):
        O, lse, err = G.run_decode(inp, t)
        assert err == 0
        assert torch.equal(O, O0) and torch.equal(lse, lse0)
