"""The allocation-free decode entry point (for callers that cannot allocate
device memory: the split-KV scratch lives in a fixed array inside the
library).  Checked against the regular entry point, which takes a caller
workspace, on a long single-request decode that needs split-KV scratch, two
calls in a row.  Collected last on purpose (its file name sorts last)."""
import numpy as np
import pytest
import torch

import workloads as wl
import mla_decode_context_gb300 as dcp
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice():
    spec = wl.DecodeSpec("noalloc_long_b1", seed=41, B=1, seq_lens=(20000,), H=128, block_size=64, D=8,
                         interleave=1)
    inp = wl.make_decode_inputs(spec)
    t = wl.to_torch(inp)
    T, H, D = inp["T"], inp["H"], inp["D"]
    msl, mql = inp["max_seq_len"], inp["max_q_len"]
    assert dcp.dcp_decode_workspace_size(inp["B"], T, H, D, msl, mql) > 0  # the split path is exercised
    O_ref, lse_ref = dcp.decode_partial(t["q"], t["kv_cache"], t["block_table"], t["seq_lens"],
                                        t["query_start_loc"], D=D, interleave=1, scale=inp["scale"],
                                        max_seq_len=msl, max_q_len=mql)
    torch.cuda.synchronize()
    for _ in range(2):
        O = torch.full_like(O_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        dcp.dcp_mla_decode_partial_noalloc(t["q"], t["kv_cache"], t["block_table"], t["seq_lens"],
                                           t["query_start_loc"], O, lse, D=D, interleave=1, scale=inp["scale"],
                                           max_seq_len=msl, max_q_len=mql, dev_error=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        G.check_partials(O.cpu().numpy(), lse.cpu().numpy(), O_ref.cpu().double().numpy(),
                         lse_ref.cpu().double().numpy(), "noalloc")
