"""GPU LSE combine parity with the float64 oracle over the combine sweep."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import mla_decode_context_gb300 as dcp
from tests import gpu_util as G
from tests.oracle_checks import page_facts

pytestmark = pytest.mark.gpu


def _inputs(D, T, H=wl.COMBINE_H, seed=None):
    O, lse, seq, qsl, empty, pad = wl.make_combine_inputs(D, T, H, seed=seed, device="cuda")
    return O, lse, torch.from_numpy(seq).cuda(), torch.from_numpy(qsl).cuda(), pad


def _sample_rows(T):
    if T <= 64:
        return np.arange(T)
    rng = np.random.default_rng(T)
    return np.unique(np.concatenate([[0, T - 1], rng.choice(T, 62, replace=False)]))


@pytest.mark.parametrize("D,T", wl.COMBINE_SWEEP + [(32, 64)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_combine_sweep(D, T, out_dtype):
    # (32, 64): the largest shard count the ABI accepts (one lane per shard)
    O, lse, seq, qsl, pad = _inputs(D, T, seed=97 if (D, T) not in wl.COMBINE_SWEEP else None)
    out, out_lse = dcp.lse_combine(O, lse, seq, qsl, out_dtype=out_dtype)
    torch.cuda.synchronize()
    rows = _sample_rows(T)
    rt = torch.from_numpy(rows).cuda()
    O_h = O[:, rt].double().cpu().numpy()
    l_h = lse[:, rt].double().cpu().numpy()
    ref, ref_lse = oracle.lse_combine(O_h, l_h, pad[rows])
    got = out[rt].float().cpu().numpy().astype(np.float64)
    got_lse = out_lse[rt].cpu().numpy().astype(np.float64)
    assert not np.isnan(got).any()
    p = pad[rows]
    assert (got[p] == 0).all() and (got_lse[p] == -np.inf).all()
    assert np.array_equal(got_lse == -np.inf, ref_lse == -np.inf)
    live = ref_lse != -np.inf
    assert np.all(np.abs(got_lse[live] - ref_lse[live]) <= G.COMB_REL * np.maximum(1.0, np.abs(ref_lse[live])))
    # fp32 accumulation error scales with the vector, not with an element
    # that happens to cancel to ~0: allow COMB_REL of the (row, head) vector's
    # largest magnitude, plus one bf16 ulp of the element in bf16 mode
    scale = np.maximum(np.abs(ref).max(axis=-1, keepdims=True), 1e-30)
    if out_dtype == torch.float32:
        assert np.all(np.abs(got - ref) <= G.COMB_REL * scale)
    else:
        assert np.all(np.abs(got - ref) <= G.bf16_ulp(ref) + G.COMB_REL * scale)


@pytest.mark.parametrize("D", [2, 8, 12, 16, 32])
def test_combine_few_and_many_pairs_agree_bitwise(D):
    """Few (row, head) pairs load every source before the weights, many load
    the live ones in batches after them: the same live sources in the same
    order with the same weights, so the rows they share are bit-identical
    (empty shards' NaN payloads and padding rows included)."""
    T, n = 64, 8  # 8192 pairs, and 1024 in the first 8 rows
    O, lse, seq, qsl, pad = _inputs(D, T, seed=101)
    full, full_lse = dcp.lse_combine(O, lse, seq, qsl, out_dtype=torch.float32)
    few, few_lse = dcp.lse_combine(O[:, :n].contiguous(), lse[:, :n].contiguous(), seq[:n].contiguous(),
                                   qsl[:n + 1].contiguous(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert not torch.isnan(full).any()
    assert torch.equal(full[:n], few) and torch.equal(full_lse[:n], few_lse)


def test_combine_shard_order_invariance():
    O, lse, seq, qsl, pad = _inputs(8, 1024)
    a, al = dcp.lse_combine(O, lse, seq, qsl, out_dtype=torch.float32)
    perm = torch.randperm(8, generator=torch.Generator().manual_seed(0)).cuda()
    b, bl = dcp.lse_combine(O[perm].contiguous(), lse[perm].contiguous(), seq, qsl, out_dtype=torch.float32)
    torch.cuda.synchronize()
    live = torch.isfinite(al)
    assert torch.equal(torch.isfinite(bl), live)
    scale = a.abs().amax(dim=-1, keepdim=True).clamp_min(1e-30)
    assert ((a - b).abs() <= 1e-6 * scale).all()
    assert ((al[live] - bl[live]).abs() <= 1e-6 * al[live].abs().clamp_min(1)).all()


@pytest.mark.parametrize("T", [int(x) for x in page_facts()["merge_geometry_tokens"].split(",")])
def test_inplace_lse_matches_disjoint(T):
    """out_lse may alias lse_part's shard-0 slice (a two-way merge that reuses
    the running LSE tensor, in the pages' six-head geometry)."""
    H = int(page_facts()["merge_geometry_heads"])
    O, lse, seq, qsl, pad = _inputs(2, T, H=H, seed=99)
    ref, ref_lse = dcp.lse_combine(O, lse, seq, qsl, out_dtype=torch.float32)
    lse2 = lse.clone()
    out = torch.empty_like(ref)
    dcp.dcp_lse_combine(O, lse2, seq, qsl, out, lse2[0])
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert torch.equal(lse2[0], ref_lse)


def test_combine_reads_no_masked_payload():
    """Empty shards and padding rows hold NaN payloads; none may leak."""
    O, lse, seq, qsl, pad = _inputs(4, 64)
    assert torch.isnan(O).any()
    out, out_lse = dcp.lse_combine(O, lse, seq, qsl)
    torch.cuda.synchronize()
    assert not torch.isnan(out).any() and not torch.isnan(out_lse).any()
