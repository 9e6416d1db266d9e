"""GPU parity of the fp8 latent cache (FP8 E4M3 codes, one fp32 scale per
slot) and of bf16 partial outputs, against the oracle: the fp8 decode on both
kernels in both table layouts (the 120,000-token split path included),
bit-exact token selection through position-coded fp8 rows, bf16 partials
from both kernels, and the combine over bf16 partials."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
import mla_decode_context_gb300 as dcp
from tests import gpu_util as G
from tests import position_code as PC

pytestmark = pytest.mark.gpu

FP8 = [
    wl.DecodeSpec("fp8_h128_d8_i1", seed=141, B=3, seq_lens=(1, 700, 2049), H=128, block_size=64, D=8, interleave=1,
                  kv_dtype="fp8_e4m3"),
    wl.DecodeSpec("fp8_q4_causal_padding", seed=142, B=4, seq_lens=(0, 2, 903, 4), q_len=4, H=128, block_size=64,
                  D=8, interleave=1, extra_rows=2, kv_dtype="fp8_e4m3"),
    wl.DecodeSpec("fp8_h64_d4_i3_local", seed=143, B=2, seq_lens=(250, 40), H=64, block_size=16, D=4, interleave=3,
                  layout="local", kv_dtype="fp8_e4m3"),
    wl.DecodeSpec("fp8_long_split", seed=144, B=1, seq_lens=(9000,), H=128, block_size=64, D=8, interleave=1,
                  kv_dtype="fp8_e4m3"),
]


@pytest.fixture(params=["tc", "simt"])
def kernel(request, monkeypatch):
    if request.param == "simt":
        monkeypatch.setenv("DCP_FORCE_SIMT", "1")
    else:
        monkeypatch.delenv("DCP_FORCE_SIMT", raising=False)
    return request.param


def _decode(inp, t, out_dtype=torch.float32):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    O, lse = dcp.decode_partial(t["q"], t["kv_cache"], t["block_table"], t["seq_lens"], t["query_start_loc"],
                                D=inp["D"], interleave=inp["interleave"], scale=inp["scale"],
                                max_seq_len=max(1, inp["max_seq_len"]), max_q_len=max(1, inp["max_q_len"]),
                                dev_error=err, kv_scale=t.get("kv_scale"), out_dtype=out_dtype)
    torch.cuda.synchronize()
    return O, lse, int(err.item())


def _check_partials_bf16(O, lse, O_ref, lse_ref, what):
    """bf16 partials: the attention tolerance plus half a bf16 ulp of the
    value (the storage rounding); LSEs stay fp32."""
    O = O.float().cpu().numpy()
    lse = lse.cpu().numpy()
    assert not np.isnan(O).any() and not np.isnan(lse).any(), what
    empty = lse_ref == -np.inf
    assert np.array_equal(lse == -np.inf, empty), what
    assert (O[empty] == 0).all(), what
    live = ~empty
    assert np.abs(lse[live] - lse_ref[live]).max() <= G.ATT_LSE_ABS, what
    tol = G.ATT_OUT_ABS + 0.5 * G.bf16_ulp(O_ref[live])
    assert (np.abs(O[live] - O_ref[live]) <= tol).all(), what


@pytest.mark.parametrize("spec", FP8, ids=lambda s: s.name)
def test_fp8_decode_matches_oracle(spec, kernel):
    inp = wl.make_decode_inputs(spec)
    t = G.to_device(inp)
    O, lse, err = _decode(inp, t)
    assert err == 0
    O_ref, lse_ref, rows = oracle.decode_partial(inp)
    G.check_partials(O.cpu().numpy(), lse.cpu().numpy(), O_ref, lse_ref, "%s/%s" % (spec.name, kernel))
    out, out_lse = G.run_combine(O, lse, t)
    _, _, pad = oracle.row_lengths(inp["seq_lens"], inp["query_start_loc"], inp["T"])
    out_ref, out_lse_ref = oracle.lse_combine(O_ref, lse_ref, pad)
    G.check_combined(out.float().cpu().numpy(), out_lse.cpu().numpy(), out_ref, out_lse_ref, pad, spec.name)


@pytest.mark.parametrize("spec", [FP8[0], FP8[2]], ids=lambda s: s.name)
def test_fp8_walker_bit_exact(spec, kernel):
    # position digits are exact in E4M3 with a power-of-two scale
    inp = wl.make_decode_inputs(spec, kv_rows=PC.kv_rows)
    inp["scale"] = 0.0
    t = G.to_device(inp)
    O, lse, err = _decode(inp, t)
    assert err == 0
    n, E, _ = PC.expected(inp)
    PC.check(O.cpu().numpy(), lse.cpu().numpy(), n, E, "%s/%s" % (spec.name, kernel))


@pytest.mark.parametrize("spec", [FP8[0], FP8[1], FP8[3]], ids=lambda s: s.name)
def test_fp8_scales_that_are_not_powers_of_two(spec, kernel):
    """Any fp32 scale: the CUDA-core kernel applies it in fp32 and matches the
    oracle on the codes and scales; the tensor-core kernel widens each
    code x scale to bf16 (the fp32 product, rounded to nearest even), so it
    matches the oracle run on the bf16 cache that holds exactly those
    values."""
    inp = wl.make_decode_inputs(spec)
    rng = np.random.default_rng(spec.seed + 1000)
    factor = rng.uniform(0.55, 0.95, size=inp["kv_scale"].shape)
    inp["kv_scale"] = (inp["kv_scale"].astype(np.float64) * factor).astype(np.float32)
    t = G.to_device(inp)
    O, lse, err = _decode(inp, t)
    assert err == 0
    ref = inp
    if kernel == "tc":
        widened = oracle.fp8_e4m3_to_f64(inp["kv_cache"]).astype(np.float32) * inp["kv_scale"][..., None]
        ref = dict(inp, kv_dtype="bf16", kv_cache=wl.f32_to_bf16_bits(widened))
        del ref["kv_scale"]
    O_ref, lse_ref, _ = oracle.decode_partial(ref)
    G.check_partials(O.cpu().numpy(), lse.cpu().numpy(), O_ref, lse_ref, "%s/%s" % (spec.name, kernel))


BF16_OUT = [
    wl.DecodeSpec("bf16out_h128_d8", seed=151, B=3, seq_lens=(1, 700, 2049), H=128, block_size=64, D=8, interleave=1),
    wl.DecodeSpec("bf16out_long_split", seed=152, B=1, seq_lens=(9000,), H=128, block_size=64, D=8, interleave=1),
    wl.DecodeSpec("bf16out_q4_causal_padding_local", seed=153, B=4, seq_lens=(0, 2, 903, 4), q_len=4, H=128,
                  block_size=64, D=8, interleave=1, extra_rows=2, layout="local"),
]


@pytest.mark.parametrize("spec", BF16_OUT, ids=lambda s: s.name)
def test_bf16_partials_match_oracle(spec, kernel):
    inp = wl.make_decode_inputs(spec)
    t = G.to_device(inp)
    O, lse, err = _decode(inp, t, out_dtype=torch.bfloat16)
    assert err == 0 and O.dtype == torch.bfloat16
    O_ref, lse_ref, rows = oracle.decode_partial(inp)
    _check_partials_bf16(O, lse, O_ref, lse_ref, "%s/%s" % (spec.name, kernel))
    out, out_lse = G.run_combine(O, lse, t)  # the combine reads the bf16 partials
    _, _, pad = oracle.row_lengths(inp["seq_lens"], inp["query_start_loc"], inp["T"])
    out_ref, out_lse_ref = oracle.lse_combine(O_ref, lse_ref, pad)
    G.check_combined(out.float().cpu().numpy(), out_lse.cpu().numpy(), out_ref, out_lse_ref, pad, spec.name)


@pytest.mark.parametrize("spec", [FP8[1], FP8[2]], ids=lambda s: s.name)
def test_fp8_cache_with_bf16_partials(spec, kernel):
    """Both options at once: the fp8 cache widened on the way in, bf16
    partials on the way out (causal verification rows with padding, and the
    per-shard layout with an unaligned interleave)."""
    inp = wl.make_decode_inputs(spec)
    t = G.to_device(inp)
    O, lse, err = _decode(inp, t, out_dtype=torch.bfloat16)
    assert err == 0 and O.dtype == torch.bfloat16
    O_ref, lse_ref, rows = oracle.decode_partial(inp)
    _check_partials_bf16(O, lse, O_ref, lse_ref, "%s/%s" % (spec.name, kernel))


def test_fp8_long_context_120k():
    """The 120,000-token context in the fp8 cache, on the tensor cores (nine
    splits per shard), against the oracle."""
    inp = wl.make_decode_inputs(wl.LONG_120K_FP8)
    t = G.to_device(inp)
    O, lse, err = _decode(inp, t)
    assert err == 0
    O_ref, lse_ref, rows = oracle.decode_partial(inp)
    G.check_partials(O.cpu().numpy(), lse.cpu().numpy(), O_ref, lse_ref, "120k fp8")


def test_bf16_partials_long_context_120k():
    inp = wl.make_decode_inputs(wl.LONG_120K)
    t = G.to_device(inp)
    O, lse, err = _decode(inp, t, out_dtype=torch.bfloat16)
    assert err == 0
    O_ref, lse_ref, rows = oracle.decode_partial(inp)
    _check_partials_bf16(O, lse, O_ref, lse_ref, "120k bf16 partials")


@pytest.mark.parametrize("D,T", [(2, 1024), (8, 64), (4, 1)])
def test_combine_over_bf16_partials(D, T):
    """The combine's arithmetic over bf16 partials: against the oracle's
    combine of the same bf16 values, at the combine tolerance."""
    O, lse, seq, qsl, empty, pad = wl.make_combine_inputs(D, T, device="cuda")
    Ob = torch.nan_to_num(O, nan=0.0).to(torch.bfloat16)
    seq_t, qsl_t = torch.from_numpy(seq).cuda(), torch.from_numpy(qsl).cuda()
    out, out_lse = dcp.lse_combine(Ob, lse, seq_t, qsl_t, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.lse_combine(Ob.double().cpu().numpy(), lse.double().cpu().numpy(), pad)
    got, got_lse = out.double().cpu().numpy(), out_lse.double().cpu().numpy()
    assert np.array_equal(got_lse == -np.inf, ref_lse == -np.inf)
    live = ref_lse != -np.inf
    assert np.all(np.abs(got_lse[live] - ref_lse[live]) <= G.COMB_REL * np.maximum(1.0, np.abs(ref_lse[live])))
    scale = np.maximum(np.abs(ref).max(axis=-1, keepdims=True), 1e-30)
    assert np.all(np.abs(got - ref) <= G.COMB_REL * scale)
