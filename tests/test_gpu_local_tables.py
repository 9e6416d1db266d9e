"""GPU parity of the decode over per-shard (DCP rank-local) block tables:
against the oracle on both kernels (including shared prefixes and
verification rows), bit-exact token selection through position-coded rows,
and the 120,000-token workload as two requests sharing a 114,000-token
prefix in both layouts."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests import gpu_util as G
from tests import position_code as PC

pytestmark = pytest.mark.gpu

LOCAL = [
    wl.DecodeSpec("local_h128_d8_i1", seed=101, B=3, seq_lens=(1, 700, 2049), H=128, block_size=64, D=8,
                  interleave=1, layout="local"),
    wl.DecodeSpec("local_h128_d8_i64", seed=102, B=3, seq_lens=(1500, 333, 64), H=128, block_size=64, D=8,
                  interleave=64, layout="local"),
    wl.DecodeSpec("local_h64_d4_i3", seed=103, B=2, seq_lens=(250, 40), H=64, block_size=16, D=4, interleave=3,
                  layout="local"),
    wl.DecodeSpec("local_q4_causal_padding", seed=104, B=4, seq_lens=(0, 2, 903, 4), q_len=4, H=128, block_size=64,
                  D=8, interleave=1, extra_rows=2, layout="local"),
    wl.DecodeSpec("local_shared_prefix_split", seed=105, B=2, seq_lens=(9000, 8000), H=128, block_size=64, D=8,
                  interleave=1, prefix_len=6000, shared_prefix=True, layout="local"),
    wl.DecodeSpec("global_shared_prefix_split", seed=105, B=2, seq_lens=(9000, 8000), H=128, block_size=64, D=8,
                  interleave=1, prefix_len=6000, shared_prefix=True),
    wl.DecodeSpec("local_d32_i1", seed=106, B=2, seq_lens=(5000, 700), H=128, block_size=64, D=32, interleave=1,
                  layout="local"),
]


@pytest.fixture(params=["tc", "simt"])
def kernel(request, monkeypatch):
    if request.param == "simt":
        monkeypatch.setenv("DCP_FORCE_SIMT", "1")
    else:
        monkeypatch.delenv("DCP_FORCE_SIMT", raising=False)
    return request.param


def _check(inp, rows=None):
    t = G.to_device(inp)
    O, lse, err = G.run_decode(inp, t)
    assert err == 0
    O_ref, lse_ref, rows = oracle.decode_partial(inp, rows)
    G.check_partials(O.cpu().numpy()[:, rows], lse.cpu().numpy()[:, rows], O_ref, lse_ref, inp["name"])
    out, out_lse = G.run_combine(O, lse, t)
    _, _, pad = oracle.row_lengths(inp["seq_lens"], inp["query_start_loc"], inp["T"])
    out_ref, out_lse_ref = oracle.lse_combine(O_ref, lse_ref, pad[rows])
    G.check_combined(out.float().cpu().numpy()[rows], out_lse.cpu().numpy()[rows], out_ref, out_lse_ref,
                     pad[rows], inp["name"])


@pytest.mark.parametrize("spec", LOCAL, ids=lambda s: s.name)
def test_local_tables_match_oracle(spec, kernel):
    _check(wl.make_decode_inputs(spec))


@pytest.mark.parametrize("spec", [LOCAL[0], LOCAL[2], LOCAL[3], LOCAL[6]], ids=lambda s: s.name)
def test_local_walker_bit_exact(spec, kernel):
    inp = wl.make_decode_inputs(spec, kv_rows=PC.kv_rows)
    inp["scale"] = 0.0
    t = G.to_device(inp)
    O, lse, err = G.run_decode(inp, t)
    assert err == 0
    n, E, _ = PC.expected(inp)
    PC.check(O.cpu().numpy(), lse.cpu().numpy(), n, E, "%s/%s" % (spec.name, kernel))


def test_local_table_must_cover_the_largest_shard():
    """A per-shard table one column short of the largest local shard is
    refused before launch (the pages' table-width contract)."""
    import mla_decode_context_gb300 as dcp
    inp = wl.make_decode_inputs(LOCAL[0])
    t = G.to_device(inp)
    need = -(-oracle.local_len(int(inp["max_seq_len"]), 0, 8, 1) // 64)
    short = t["block_table"][:, :, :need - 1].contiguous()
    with pytest.raises(dcp.DCPError) as e:
        dcp.decode_partial(t["q"], t["kv_cache"], short, t["seq_lens"], t["query_start_loc"], D=8, interleave=1,
                           scale=inp["scale"], max_seq_len=int(inp["max_seq_len"]), max_q_len=1)
    assert e.value.status == 4  # DCP_ERR_TABLE_TOO_NARROW


@pytest.mark.parametrize("spec", [wl.LONG_120K_B2_PREFIX, wl.LONG_120K_B2_PREFIX_LOCAL], ids=lambda s: s.name)
def test_long_context_shared_prefix_b2(spec):
    _check(wl.make_decode_inputs(spec))


@pytest.mark.parametrize("spec", [LOCAL[0], LOCAL[3]], ids=lambda s: s.name)
def test_one_shard_per_call_as_a_rank_would(spec, kernel):
    """Each DCP rank computes only its own shard: calls over shard d alone
    (its table, shard_begin = d, shard_count = 1) reproduce the oracle's
    shard-d partials."""
    import mla_decode_context_gb300 as dcp
    inp = wl.make_decode_inputs(spec)
    t = G.to_device(inp)
    O_ref, lse_ref, rows = oracle.decode_partial(inp)
    D, T, H = inp["D"], inp["T"], inp["H"]
    msl, mql = max(1, inp["max_seq_len"]), max(1, inp["max_q_len"])
    for d in range(D):
        O = torch.empty((1, T, H, 512), device="cuda")
        lse = torch.empty((1, T, H), device="cuda")
        ws = dcp.decode_workspace(inp["B"], T, H, 1, msl, mql)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        dcp.dcp_mla_decode_partial_local(t["q"], t["kv_cache"], t["block_table"][d:d + 1], t["seq_lens"],
                                         t["query_start_loc"], O, lse, D=D, interleave=inp["interleave"],
                                         scale=inp["scale"], max_seq_len=msl, max_q_len=mql, shard_begin=d,
                                         shard_count=1, workspace=ws, dev_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        G.check_partials(O.cpu().numpy(), lse.cpu().numpy(), O_ref[d:d + 1], lse_ref[d:d + 1],
                         "%s shard %d" % (spec.name, d))
