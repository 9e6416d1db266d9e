"""Bit-exact GPU check of the device's token -> shard mapper and paged
block-table walker (both decode kernels), through the C ABI.

At scale 0 every live token weighs exactly 1, and the planted cache rows
carry base-4 digits of their own logical position (tests/position_code.py),
so the integer digit sums and token counts recovered from each (row, shard)
partial must equal the oracle's, exactly.  Geometries: the 120,000-token
long-context workload at full size (D=8, interleave 1, nine splits per
shard), the batched workload's geometry at full size (64 requests,
interleave 64 = block size, permuted table), the largest shard count (32),
an interleave that does not divide the block size (3), block sizes and an
interleave that are not powers of two, and verification rows with causal
offsets and padding requests."""
import numpy as np
import pytest
import torch

import workloads as wl
from tests import gpu_util as G
from tests import position_code as PC

pytestmark = pytest.mark.gpu

GEOMETRIES = [
    wl.LONG_120K,
    wl.BATCHED_B64,
    wl.DecodeSpec("exact_d32_i1", seed=61, B=2, seq_lens=(5000, 700), H=128, block_size=64, D=32, interleave=1),
    wl.DecodeSpec("exact_d4_i3_bs16", seed=62, B=3, seq_lens=(250, 40, 3001), H=64, block_size=16, D=4,
                  interleave=3),
    wl.DecodeSpec("exact_q4_causal_padding", seed=63, B=4, seq_lens=(0, 2, 903, 4100), q_len=4, H=128,
                  block_size=64, D=8, interleave=1, extra_rows=2),
    wl.DecodeSpec("exact_d2_i16_bs32_long", seed=64, B=1, seq_lens=(40000,), H=128, block_size=32, D=2,
                  interleave=16),
    # divisors that are not powers of two (the walker divides by the
    # interleave and the block size with precomputed multipliers)
    wl.DecodeSpec("exact_d4_i5_bs48", seed=65, B=3, seq_lens=(7001, 20, 1000), q_len=(3, 1, 2), H=64, block_size=48,
                  D=4, interleave=5),
    wl.DecodeSpec("exact_d8_i1_bs80", seed=66, B=2, seq_lens=(20000, 1027), H=128, block_size=80, D=8,
                  interleave=1),
]


@pytest.fixture(params=["tc", "simt"])
def kernel(request, monkeypatch):
    if request.param == "simt":
        monkeypatch.setenv("DCP_FORCE_SIMT", "1")
    else:
        monkeypatch.delenv("DCP_FORCE_SIMT", raising=False)
    return request.param


@pytest.mark.parametrize("spec", GEOMETRIES, ids=lambda s: s.name)
def test_mapper_and_walker_bit_exact(spec, kernel):
    inp = wl.make_decode_inputs(spec, kv_rows=PC.kv_rows)
    inp["scale"] = 0.0
    t = G.to_device(inp)
    O, lse, err = G.run_decode(inp, t)
    assert err == 0
    n, E, rows = PC.expected(inp)
    PC.check(O.cpu().numpy(), lse.cpu().numpy(), n, E, "%s/%s" % (spec.name, kernel))
