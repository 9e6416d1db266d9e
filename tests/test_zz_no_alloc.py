"""The allocation-free decode entry point, for callers that cannot allocate
device memory (their device memory is owned and fully reserved by a host
framework, or they are plugins handed only their inputs and outputs): the
split-KV scratch lives in a fixed array inside the library instead of a
caller workspace.

It runs the same kernels on the same split plan as the regular entry point,
so its results must be bit-identical to it; checked on two calls in a row
(the shared array keeps the previous call's contents) for a long
single-request decode that needs split-KV scratch, and for a batch with
verification rows.  Collected last on purpose (its file name sorts last)."""
import pytest
import torch

import workloads as wl
import mla_decode_context_gb300 as dcp

pytestmark = pytest.mark.gpu

NOALLOC_SCRATCH_BYTES = 24 << 20
SPECS = [
    wl.DecodeSpec("noalloc_long_b1", seed=41, B=1, seq_lens=(20000,), H=128, block_size=64, D=8, interleave=1),
    wl.DecodeSpec("noalloc_q4_b3", seed=44, B=3, seq_lens=(7000, 0, 12000), q_len=4, H=128, block_size=64,
                  D=8, interleave=1),
]


def _workspace_decode(inp, t):
    T, H, D = inp["T"], inp["H"], inp["D"]
    msl, mql = inp["max_seq_len"], inp["max_q_len"]
    O = torch.full((D, T, H, 512), float("nan"), device="cuda")
    lse = torch.full((D, T, H), float("nan"), device="cuda")
    ws = dcp.decode_workspace(inp["B"], T, H, D, msl, mql)
    dcp.dcp_mla_decode_partial(t["q"], t["kv_cache"], t["block_table"], t["seq_lens"], t["query_start_loc"], O,
                               lse, D=D, interleave=inp["interleave"], scale=inp["scale"], max_seq_len=msl,
                               max_q_len=mql, workspace=ws)
    torch.cuda.synchronize()
    return O, lse


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.name)
def test_noalloc_matches_workspace_entry_point_twice(spec):
    inp = wl.make_decode_inputs(spec)
    t = wl.to_torch(inp)
    T, H, D = inp["T"], inp["H"], inp["D"]
    msl, mql = inp["max_seq_len"], inp["max_q_len"]
    if spec.B == 1:
        assert dcp.dcp_decode_workspace_size(inp["B"], T, H, D, msl, mql) > 0  # the split path is exercised
    O_ref, lse_ref = _workspace_decode(inp, t)
    for _ in range(2):
        O = torch.full_like(O_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        dcp.dcp_mla_decode_partial_noalloc(t["q"], t["kv_cache"], t["block_table"], t["seq_lens"],
                                           t["query_start_loc"], O, lse, D=D, interleave=inp["interleave"],
                                           scale=inp["scale"], max_seq_len=msl, max_q_len=mql, dev_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert torch.equal(O, O_ref) and torch.equal(lse, lse_ref)


def test_noalloc_limit_on_this_device():
    """Every plan with H <= 128 fits the fixed array on this GPU (the split
    plan depends on its SM count); a 1024-head long-context plan does not and
    is refused before any launch."""
    for D in (1, 2, 3, 4, 8, 16, 32):
        for T in (1, 2, 3, 4, 8, 16, 64, 128, 1024, 4096):
            for msl in (1, 300, 4096, 120000, 1 << 20):
                assert dcp.dcp_decode_workspace_size(T, T, 128, D, msl, 4) <= NOALLOC_SCRATCH_BYTES, (D, T, msl)
    D, H = 8, 1024
    assert dcp.dcp_decode_workspace_size(1, 1, H, D, 120000, 1) > NOALLOC_SCRATCH_BYTES
    q = torch.zeros((1, H, 576), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((1875, 64, 576), dtype=torch.bfloat16, device="cuda")
    tab = torch.arange(1875, dtype=torch.int32, device="cuda").reshape(1, -1)
    seq = torch.tensor([120000], dtype=torch.int32, device="cuda")
    qsl = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    O = torch.empty((D, 1, H, 512), device="cuda")
    lse = torch.empty((D, 1, H), device="cuda")
    with pytest.raises(dcp.DCPError) as e:
        dcp.dcp_mla_decode_partial_noalloc(q, kv, tab, seq, qsl, O, lse, D=D, interleave=1, scale=0.07,
                                           max_seq_len=120000, max_q_len=1)
    assert e.value.status == 5  # DCP_ERR_WORKSPACE_TOO_SMALL
