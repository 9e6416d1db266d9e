"""C-ABI library: builds, loads, exports what include/dcp.h declares, and its
host-side logic (mapper copy, validation that returns before any launch).
No GPU needed: nothing here enqueues a kernel."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import mla_decode_context_gb300 as dcp
from mla_decode_context_gb300 import build_lib

pytestmark = pytest.mark.cpu
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "dcp.h")


@pytest.fixture(scope="module")
def L():
    build_lib.build()
    return dcp.lib()


def declared_symbols():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dcp_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_symbols()
    assert {n for n, _, _ in dcp.EXPORTS} == set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code, name in dcp.STATUS.items():
        assert dcp.dcp_status_str(code) == name
    assert dcp.dcp_version() >= 1


def test_shard_mapper_bit_exact_with_oracle(L):
    for D in (1, 2, 3, 4, 8, 32):
        for I in (1, 2, 5, 64, 128):
            for pos in list(range(0, 300)) + [10**6 + 7, 2**31 + 3]:
                assert dcp.dcp_shard_of(pos, D, I) == int(oracle.shard_of(pos, D, I))
            for Lq in list(range(0, 200)) + [120000, 65536, 2**31 - 1]:
                for d in range(D):
                    if Lq < 5000:
                        assert dcp.dcp_local_len(Lq, d, D, I) == oracle.local_len(Lq, d, D, I)
                    else:  # large L: closed form in exact integers
                        want = (Lq // (I * D)) * I + min(max(Lq % (I * D) - d * I, 0), I)
                        assert dcp.dcp_local_len(Lq, d, D, I) == want


def test_mapper_rejects_bad_args(L):
    assert dcp.dcp_shard_of(-1, 4, 1) == -1
    assert dcp.dcp_shard_of(3, 0, 1) == -1
    assert dcp.dcp_local_len(5, 4, 4, 1) == -1
    assert dcp.dcp_local_len(-1, 0, 4, 1) == -1


def test_workspace_size(L):
    assert dcp.dcp_decode_workspace_size(0, 0, 128, 8, 1000, 1) == 0
    # long-context single request: split-KV needs a workspace
    assert dcp.dcp_decode_workspace_size(1, 1, 128, 8, 120000, 1) > 0
    # many rows fill the GPU without splitting: only the units' launch order
    # (one int32 per unit, rounded to 256 bytes)
    assert dcp.dcp_decode_workspace_size(64, 64, 128, 8, 32768, 1) == 64 * 8 * 4
    with pytest.raises(dcp.DCPError):
        dcp.dcp_decode_workspace_size(1, 1, 128, 33, 100, 1)


def test_kernel_launch_count(L):
    assert dcp.dcp_decode_kernel_launches(0, 0, 128, 8, 1, 1000, 1, 0) == 0
    # long-context single request: decode + split merge
    ws = dcp.dcp_decode_workspace_size(1, 1, 128, 8, 120000, 1)
    assert dcp.dcp_decode_kernel_launches(1, 1, 128, 8, 1, 120000, 1, ws) == 2
    with pytest.raises(dcp.DCPError):
        dcp.dcp_decode_kernel_launches(1, 1, 128, 33, 1, 100, 1, 0)


def _decode(L, **kw):
    a = dict(q=0x1000, q_stride_tok=128 * 576, kv=0x2000, num_blocks=4, block_size=16, table=0x3000,
             bt_width=4, bt_stride=4, seq_lens=0x4000, qsl=0x5000, B=2, T=2, H=128, max_seq_len=37,
             max_q_len=1, D=4, I=1, scale=0.07, O=0x6000, lse=0x7000, ws=None, ws_bytes=0, err=None)
    a.update(kw)
    f = L.dcp_mla_decode_partial
    return f(a["q"], a["q_stride_tok"], a["kv"], a["num_blocks"], a["block_size"], a["table"], a["bt_width"],
             a["bt_stride"], a["seq_lens"], a["qsl"], a["B"], a["T"], a["H"], a["max_seq_len"], a["max_q_len"],
             a["D"], a["I"], a["scale"], a["O"], a["lse"], a["ws"], a["ws_bytes"], a["err"], None)


def test_decode_validation_returns_before_launch(L):
    assert _decode(L, B=0) == 0 and _decode(L, T=0) == 0  # nothing to do: OK, no launch
    assert _decode(L, q=None) == 1
    assert _decode(L, D=0) == 1 and _decode(L, D=33) == 1 and _decode(L, I=0) == 1
    assert _decode(L, H=0) == 1 and _decode(L, B=-1) == 1
    assert _decode(L, scale=float("nan")) == 1
    assert _decode(L, bt_stride=3) == 1
    assert _decode(L, q_stride_tok=100) == 1
    assert _decode(L, q=0x1008) == 3                       # 16-byte rule
    assert _decode(L, q_stride_tok=128 * 576 + 4) == 3
    assert _decode(L, O=0x6004) == 3
    assert _decode(L, max_seq_len=65) == 4                 # needs 5 columns of 16 > 4
    # a long single request needs split workspace (checked before any launch)
    assert _decode(L, B=1, T=1, max_seq_len=120000, block_size=64, bt_width=1875, bt_stride=1875,
                   D=8) == 5


def _combine(L, **kw):
    a = dict(O=0x1000, lse=0x2000, seq=0x3000, qsl=0x4000, B=2, T=2, H=128, D=4, out=0x100000, dt=0,
             out_lse=0x9000)
    a.update(kw)
    return L.dcp_lse_combine(a["O"], a["lse"], a["seq"], a["qsl"], a["B"], a["T"], a["H"], a["D"], a["out"],
                             a["dt"], a["out_lse"], None)


def test_combine_validation_returns_before_launch(L):
    assert _combine(L, T=0) == 0
    assert _combine(L, dt=7) == 2
    assert _combine(L, D=0) == 1 and _combine(L, D=33) == 1
    assert _combine(L, out=None) == 1
    assert _combine(L, O=0x1004) == 3
    assert _combine(L, out=0x1000 + 64) == 1  # overlaps O_part


def test_nvtx_range_never_raises():
    # the binding names its library calls on profiler timelines; without a
    # GPU or NVTX the range must be a no-op, never an error
    with dcp._Range("dcp_test_range"):
        pass


NOALLOC_SCRATCH_BYTES = 24 << 20


def test_noalloc_scratch_covers_every_128_head_plan(L):
    """The allocation-free decode's fixed scratch (24 MiB) covers every split
    plan with H = 128 heads at the sizes the library is used at (sized here
    for a 152-SM GB300, the count used when no device is visible)."""
    for D in range(1, 33):
        for T in list(range(1, 65)) + [128, 256, 1024, 2048, 4096]:
            for msl in (1, 255, 256, 4096, 32768, 120000, 1 << 20):
                n = dcp.dcp_decode_workspace_size(T, T, 128, D, msl, 4)
                assert n <= NOALLOC_SCRATCH_BYTES, (D, T, msl, n)


def test_noalloc_refuses_a_plan_beyond_its_scratch(L):
    """1024 heads over a 120,000-token context need ~150 MB of split partials:
    refused with DCP_ERR_WORKSPACE_TOO_SMALL before anything is launched
    (the pointers here are never dereferenced)."""
    f = L.dcp_mla_decode_partial_noalloc
    st = f(0x1000, 1024 * 576, 0x2000, 1875, 64, 0x3000, 1875, 1875, 0x4000, 0x5000, 1, 1, 1024, 120000, 1,
           8, 1, 0.07, 0x6000, 0x7000, None, None)
    assert st == 5


def _cpu_decode_args(**kw):
    import torch
    a = dict(q=torch.zeros((2, 16, 576), dtype=torch.bfloat16), kv=torch.zeros((4, 16, 576), dtype=torch.bfloat16),
             tab=torch.zeros((2, 4), dtype=torch.int32), seq=torch.zeros(2, dtype=torch.int32),
             qsl=torch.zeros(3, dtype=torch.int32), O=torch.zeros((4, 2, 16, 512)), lse=torch.zeros((4, 2, 16)))
    a.update(kw)
    return a


@pytest.mark.parametrize("entry", ["dcp_mla_decode_partial", "dcp_mla_decode_partial_noalloc"])
def test_decode_wrappers_check_shapes_before_the_device(entry):
    """Both decode wrappers reject, with ValueError and before touching a
    device, the shapes the C ABI cannot see: a block table with fewer than B
    rows, a flattened cache, a query_start_loc without B + 1 entries."""
    import torch
    f = getattr(dcp, entry)

    def call(a):
        f(a["q"], a["kv"], a["tab"], a["seq"], a["qsl"], a["O"], a["lse"], D=4, interleave=1, scale=0.1,
          max_seq_len=37, max_q_len=1)
    for bad, msg in ((dict(tab=torch.zeros((1, 4), dtype=torch.int32)), "disagree on B"),
                     (dict(kv=torch.zeros((64, 576), dtype=torch.bfloat16)), "kv_cache"),
                     (dict(qsl=torch.zeros(2, dtype=torch.int32)), "disagree on B"),
                     (dict(O=torch.zeros((4, 2, 16, 256))), "O_part")):
        with pytest.raises(ValueError, match=msg):
            call(_cpu_decode_args(**bad))
    with pytest.raises(ValueError, match="CUDA tensor"):  # right shapes, host memory
        call(_cpu_decode_args())


def test_combine_wrapper_checks_shapes_before_the_device():
    import torch
    O, lse = torch.zeros((4, 2, 16, 512)), torch.zeros((4, 2, 16))
    seq, qsl = torch.zeros(2, dtype=torch.int32), torch.zeros(3, dtype=torch.int32)
    out, out_lse = torch.zeros((2, 16, 512), dtype=torch.bfloat16), torch.zeros((2, 16))
    with pytest.raises(ValueError, match="O_part"):
        dcp.dcp_lse_combine(torch.zeros((4, 2, 16, 500)), lse, seq, qsl, out, out_lse)
    with pytest.raises(ValueError, match="O_part"):
        dcp.dcp_lse_combine(torch.zeros((3, 2, 16, 512)), lse, seq, qsl, out, out_lse)
    with pytest.raises(ValueError, match="B \\+ 1"):
        dcp.dcp_lse_combine(O, lse, seq, torch.zeros(2, dtype=torch.int32), out, out_lse)
    with pytest.raises(ValueError, match="CUDA tensor"):
        dcp.dcp_lse_combine(O, lse, seq, qsl, out, out_lse)


def _concat(L, **kw):
    a = dict(qn=0x1000, qn_t=512, qn_h=512, qp=0x2000, qp_t=64, qp_h=64, kc=0x3000, kc_t=512, kp=0x4000, kp_t=64,
             slot=0x5000, T=2, H=1, qo=0x6000, qo_t=576, cache=0x7000, nslots=16, err=None)
    a.update(kw)
    return L.dcp_decode_concat_cache(a["qn"], a["qn_t"], a["qn_h"], a["qp"], a["qp_t"], a["qp_h"], a["kc"], a["kc_t"],
                                     a["kp"], a["kp_t"], a["slot"], a["T"], a["H"], a["qo"], a["qo_t"], a["cache"],
                                     a["nslots"], a["err"], None)


def test_concat_cache_validation_returns_before_launch(L):
    assert _concat(L, T=0) == 0
    assert _concat(L, T=-1) == 1 and _concat(L, H=0) == 1 and _concat(L, nslots=0) == 1
    assert _concat(L, slot=None) == 1 and _concat(L, qo=None) == 1
    assert _concat(L, qo_t=575) == 1                  # output rows narrower than H * 576
    assert _concat(L, qn=0x1008) == 3                 # 16-byte rule
    assert _concat(L, kc_t=516) == 3                  # strides in whole 16-byte units
    assert _concat(L, cache=0x7004) == 3
