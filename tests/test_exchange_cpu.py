"""The multi-GPU exchange around the per-shard decode, run as two gloo ranks
on the CPU (one process per GPU in deployment): the query gather along heads
is bit-exact, the all-to-all delivers every shard's slice of this rank's
heads bit-exactly, the local combine of those slices equals the single-
process combine of all shards, and a peer that never joins makes the
exchange fail with DCP_ERR_TIMEOUT instead of hanging."""
import datetime
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

pytestmark = pytest.mark.cpu


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    import workloads as wl
    spec = wl.DecodeSpec("x2", seed=121, B=3, seq_lens=(40, 1, 0), H=6, block_size=8, D=2, interleave=2,
                         layout="local", extra_rows=1)
    return wl.make_decode_inputs(spec)


def _oracle_combine(O_parts, lse_parts, seq_lens, qsl):
    import oracle
    T = O_parts.shape[1]
    _, _, pad = oracle.row_lengths(seq_lens.numpy(), qsl.numpy(), T)
    out, out_lse = oracle.lse_combine(O_parts.double().numpy(), lse_parts.double().numpy(), pad)
    return torch.from_numpy(out), torch.from_numpy(out_lse)


def _rank(rank, port, mode, q_out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    import oracle
    from mla_decode_context_gb300 import exchange as X, DCPError
    dist.init_process_group("gloo", rank=rank, world_size=2, timeout=datetime.timedelta(seconds=3))
    try:
        inp = _case()
        if mode == "timeout":
            if rank == 1:
                q_out.put((rank, "left"))  # this rank leaves before the exchange
                return
            O = torch.zeros((inp["T"], inp["H"], 512))
            lse = torch.zeros((inp["T"], inp["H"]))
            try:
                X.a2a_lse_reduce(O, lse, torch.from_numpy(inp["seq_lens"]),
                                 torch.from_numpy(inp["query_start_loc"]), combine=_oracle_combine)
                q_out.put((rank, "no error"))
            except DCPError as e:
                q_out.put((rank, "status %d" % e.status))
            return
        H = inp["H"]
        a, b = X.head_slices(H, 2)[rank]
        # the bf16 query bits, widened to int32 (gloo carries no 16-bit integers)
        q_bits = torch.from_numpy(inp["q"].astype(np.int32))
        q_full = X.query_gather(q_bits[:, a:b])
        assert torch.equal(q_full, q_bits)
        # this rank's shard partial over all heads (computed here by the
        # oracle; on a GPU by the decode over the rank's own cache)
        O_all, lse_all, _ = oracle.decode_partial(inp)
        O_r = torch.from_numpy(np.nan_to_num(O_all[rank], nan=0.0)).float()
        l_r = torch.from_numpy(lse_all[rank]).float()
        got, got_lse = X.a2a_lse_reduce(O_r, l_r, torch.from_numpy(inp["seq_lens"]),
                                        torch.from_numpy(inp["query_start_loc"]), combine=_oracle_combine)
        O32 = torch.from_numpy(np.nan_to_num(O_all, nan=0.0)).float()[:, :, a:b]
        l32 = torch.from_numpy(lse_all).float()[:, :, a:b]
        want, want_lse = _oracle_combine(O32, l32, torch.from_numpy(inp["seq_lens"]),
                                         torch.from_numpy(inp["query_start_loc"]))
        assert torch.equal(got, want) and torch.equal(got_lse, want_lse)
        q_out.put((rank, "ok"))
    finally:
        dist.destroy_process_group()


def _spawn(mode):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, mode, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    res = {}
    while not q.empty():
        r, v = q.get()
        res[r] = v
    for p in procs:
        if p.is_alive():
            p.kill()
    return res, [p.exitcode for p in procs]


def test_head_slices_partition_the_heads():
    from mla_decode_context_gb300.exchange import head_slices
    for H in (1, 6, 7, 128):
        for D in (1, 2, 3, 8):
            if D > H:
                continue
            s = head_slices(H, D)
            assert s[0][0] == 0 and s[-1][1] == H
            assert all(s[i][1] == s[i + 1][0] for i in range(D - 1))
            assert max(b - a for a, b in s) - min(b - a for a, b in s) <= 1


def test_gather_exchange_and_combine_on_two_ranks():
    res, codes = _spawn("ok")
    assert res == {0: "ok", 1: "ok"} and codes == [0, 0], (res, codes)


def test_peer_that_never_joins_ends_in_a_timeout_status():
    res, codes = _spawn("timeout")
    assert res.get(0) == "status 7", res
