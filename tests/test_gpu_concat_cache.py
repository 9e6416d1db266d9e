"""GPU parity of the decode step before attention (query concat + paged-cache
write, one launch) with the oracle: bit-exact, including strided inputs,
negative slots and a slot past the cache; then a step-by-step decode loop
(write the step's token, decode over the grown context, combine) against
the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import mla_decode_context_gb300 as dcp
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _bits(rng, *shape):
    # finite bf16 patterns of both signs
    b = rng.integers(0, 0x7F00, size=shape, dtype=np.uint16)
    return b | (rng.integers(0, 2, size=shape, dtype=np.uint16) << 15)


def _t(bits):
    return G.bf16_tensor(bits)


def _host(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("T,H", [(1, 1), (7, 16), (64, 128)])
def test_concat_cache_bit_exact(T, H):
    rng = np.random.default_rng(T * 1000 + H)
    nb, bs = 9, 16
    ql, qp = _bits(rng, T, H, 512), _bits(rng, T, H, 64)
    kc, kp = _bits(rng, T, 512), _bits(rng, T, 64)
    cache = _bits(rng, nb, bs, 576)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[::3] = -1  # padding / not owned here
    q_ref, cache_ref = oracle.concat_cache(ql, qp, kc, kp, slots, cache)
    # ql_nope laid out as the transposed per-head matmul output: [H, T, 512] viewed as [T, H, 512]
    ql_dev = _t(np.ascontiguousarray(ql.transpose(1, 0, 2))).transpose(0, 1)
    assert ql_dev.stride(1) == T * 512
    # kv_c and k_pe as column slices of one wider per-token row
    wide = _t(np.concatenate([kc, kp, np.zeros((T, 64), np.uint16)], axis=1))
    kc_dev, kp_dev = wide[:, :512], wide[:, 512:576]
    cache_dev = _t(cache)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q = dcp.decode_concat_cache(ql_dev, _t(qp), kc_dev, kp_dev, torch.from_numpy(slots).cuda(), cache_dev,
                                dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(_host(q), q_ref)
    assert np.array_equal(_host(cache_dev), cache_ref)


def test_slot_past_the_cache_is_flagged_not_written():
    rng = np.random.default_rng(3)
    T, H, nb, bs = 3, 2, 2, 8
    ql, qp, kc, kp = _bits(rng, T, H, 512), _bits(rng, T, H, 64), _bits(rng, T, 512), _bits(rng, T, 64)
    cache = _bits(rng, nb, bs, 576)
    slots = np.array([5, nb * bs + 4, 0], dtype=np.int64)
    cache_dev = _t(cache)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dcp.decode_concat_cache(_t(ql), _t(qp), _t(kc), _t(kp), torch.from_numpy(slots).cuda(), cache_dev,
                            dev_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) & dcp.DEVERR_BAD_BLOCK
    ok = slots.copy()
    ok[1] = -1  # the bad slot is skipped
    _, cache_ref = oracle.concat_cache(ql, qp, kc, kp, ok, cache)
    assert np.array_equal(_host(cache_dev), cache_ref)


def test_step_by_step_decode_loop():
    """Three decode steps: each writes the step's token of every live request
    at its next position (slot from the block table), then decodes over the
    grown context and combines; q and the cache match the oracle bit for bit,
    the attention output within the attention tolerances."""
    spec = wl.DecodeSpec("loop_h128_d8", seed=71, B=3, seq_lens=(100, 700, 0), H=128, block_size=64, D=8,
                         interleave=1)
    inp = wl.make_decode_inputs(spec)
    rng = np.random.default_rng(72)
    t = G.to_device(inp)
    cache_host = inp["kv_cache"].copy()
    seq = inp["seq_lens"].copy()
    B, H, bs = inp["B"], inp["H"], inp["block_size"]
    for step in range(3):
        normal = lambda *shape: wl.f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
        ql, qp, kc, kp = normal(B, H, 512), normal(B, H, 64), normal(B, 512), normal(B, 64)
        slots = np.full(B, -1, dtype=np.int64)
        for b in range(B):
            if seq[b] > 0:
                p = int(seq[b])  # the new token's position
                slots[b] = int(inp["block_table"][b, p // bs]) * bs + p % bs
        q_ref, cache_host = oracle.concat_cache(ql, qp, kc, kp, slots, cache_host)
        q = dcp.decode_concat_cache(_t(ql), _t(qp), _t(kc), _t(kp), torch.from_numpy(slots).cuda(), t["kv_cache"])
        seq = np.where(seq > 0, seq + 1, 0).astype(np.int32)
        t["seq_lens"] = torch.from_numpy(seq).cuda()
        torch.cuda.synchronize()
        assert np.array_equal(_host(q), q_ref)
        step_inp = dict(inp, q=q_ref, kv_cache=cache_host, seq_lens=seq, max_seq_len=int(seq.max()))
        t["q"] = q
        O, lse, err = G.run_decode(step_inp, t)
        assert err == 0
        out, out_lse = G.run_combine(O, lse, t)
        O_ref, lse_ref, rows = oracle.decode_partial(step_inp)
        G.check_partials(O.cpu().numpy(), lse.cpu().numpy(), O_ref, lse_ref, "step %d" % step)
        _, _, pad = oracle.row_lengths(seq, inp["query_start_loc"], inp["T"])
        out_ref, out_lse_ref = oracle.lse_combine(O_ref, lse_ref, pad)
        G.check_combined(out.float().cpu().numpy(), out_lse.cpu().numpy(), out_ref, out_lse_ref, pad,
                         "step %d" % step)
    assert np.array_equal(_host(t["kv_cache"]), cache_host)
