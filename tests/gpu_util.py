"""Helpers shared by the GPU parity tests: move generator outputs to the
device, run the path through the C ABI, compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import mla_decode_context_gb300 as dcp
import workloads as wl

# Tolerances (GPU vs float64 oracle): attention outputs max abs 1e-2 and LSE
# abs 1e-3 (bf16 inputs, fp32 accumulation); the standalone combine on fp32
# partials 1e-5 relative to the (row, head) vector's largest magnitude, plus,
# for bf16 output, one bf16 ulp of the element (the output rounding).
ATT_OUT_ABS = 1e-2
ATT_LSE_ABS = 1e-3
COMB_REL = 1e-5


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_device(inp: dict, device="cuda") -> dict:
    return wl.to_torch(inp, device)


def run_decode(inp: dict, t: dict, q=None, block_table=None):
    """Decode through the C ABI; returns (O_part, lse_part, dev_error)."""
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    O, lse = dcp.decode_partial(
        t["q"] if q is None else q, t["kv_cache"], t["block_table"] if block_table is None else block_table,
        t["seq_lens"], t["query_start_loc"], D=inp["D"], interleave=inp["interleave"], scale=inp["scale"],
        max_seq_len=max(1, inp["max_seq_len"]), max_q_len=max(1, inp["max_q_len"]), dev_error=err)
    torch.cuda.synchronize()
    return O, lse, int(err.item())


def run_combine(O, lse, t: dict, out_dtype=torch.bfloat16):
    out, out_lse = dcp.lse_combine(O, lse, t["seq_lens"], t["query_start_loc"], out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out, out_lse


def check_partials(O_gpu: np.ndarray, lse_gpu: np.ndarray, O_ref: np.ndarray, lse_ref: np.ndarray, what=""):
    """Empty pairs bit-exact (-inf and zeros); live pairs within tolerance."""
    assert not np.isnan(O_gpu).any() and not np.isnan(lse_gpu).any(), what
    empty = lse_ref == -np.inf
    assert np.array_equal(lse_gpu == -np.inf, empty), what + ": empty-shard mask differs"
    assert (O_gpu[empty] == 0).all(), what
    live = ~empty
    if live.any():
        dl = np.abs(lse_gpu[live] - lse_ref[live]).max()
        do = np.abs(O_gpu[live] - O_ref[live]).max()
        assert dl <= ATT_LSE_ABS, "%s: lse err %g" % (what, dl)
        assert do <= ATT_OUT_ABS, "%s: out err %g" % (what, do)


def check_combined(out_gpu: np.ndarray, lse_gpu: np.ndarray, out_ref: np.ndarray, lse_ref: np.ndarray,
                   padding_rows: np.ndarray, what="", bf16_out=True):
    """Attention-level check of the combined result (decode + combine): the
    1e-2 attention tolerance on the computed values, plus half a bf16 ulp of
    the value when the output is stored as bf16 (the format's own rounding)."""
    assert not np.isnan(out_gpu).any(), what
    assert (out_gpu[padding_rows] == 0).all() and (lse_gpu[padding_rows] == -np.inf).all(), what
    dead = lse_ref == -np.inf
    assert np.array_equal(lse_gpu == -np.inf, dead), what
    live = ~dead
    if live.any():
        assert np.abs(lse_gpu[live] - lse_ref[live]).max() <= ATT_LSE_ABS, what
        tol = ATT_OUT_ABS + (0.5 * bf16_ulp(out_ref[live]) if bf16_out else 0.0)
        err = np.abs(out_gpu[live] - out_ref[live])
        assert (err <= tol).all(), "%s: out err %g" % (what, (err - tol).max() + ATT_OUT_ABS)
    assert (out_gpu[dead] == 0).all(), what


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)
