"""The integer check of tests/position_code.py is sharp: a simulated device
that reads exactly the oracle's rows passes it, and simulated devices with a
plausible indexing mistake (an off-by-one in the local -> global position
formula, a wrong offset inside the block, the next table column, interleave
ignored) fail it.  CPU only: the simulation gathers planted rows with numpy
and forms what the decode returns at scale 0 (the mean of the rows read, and
ln of their count)."""
import numpy as np
import pytest

import workloads as wl
from tests import position_code as PC

pytestmark = pytest.mark.cpu

SPECS = [
    wl.DecodeSpec("pc_d8_i1", seed=51, B=2, seq_lens=(700, 2049), H=4, block_size=64, D=8, interleave=1),
    wl.DecodeSpec("pc_d4_i3", seed=52, B=2, seq_lens=(250, 40), H=4, block_size=16, D=4, interleave=3),
    wl.DecodeSpec("pc_d8_i64_q4", seed=53, B=3, seq_lens=(0, 1500, 333), q_len=4, H=4, block_size=64, D=8,
                  interleave=64, extra_rows=1),
]


def _local_to_global(j, d, D, I):
    return (j // I) * (D * I) + d * I + j % I


def _simulate(inp, pos_fn=_local_to_global, row_fn=None):
    """What a decode with the given mapping returns at scale 0."""
    D, I, T, H, bs = inp["D"], inp["interleave"], inp["T"], inp["H"], inp["block_size"]
    kv = inp["kv_cache"].reshape(-1, 576)
    seq, qsl = inp["seq_lens"], inp["query_start_loc"]
    O = np.zeros((D, T, H, 512))
    lse = np.full((D, T, H), -np.inf)
    for b in range(inp["B"]):
        q_len = int(qsl[b + 1] - qsl[b])
        for i in range(q_len):
            r = int(qsl[b]) + i
            if seq[b] == 0:
                continue
            L = int(seq[b]) - (q_len - 1 - i)
            for d in range(D):
                n = (L // (I * D)) * I + min(max(L % (I * D) - d * I, 0), I)
                if n == 0:
                    continue
                p = pos_fn(np.arange(n), d, D, I)
                if row_fn is None:
                    rows = inp["block_table"][b, p // bs].astype(np.int64) * bs + p % bs
                else:
                    rows = row_fn(b, p)
                bits = kv[np.clip(rows, 0, kv.shape[0] - 1)].astype(np.uint32) << np.uint32(16)
                v = bits.view(np.float32).astype(np.float64)
                O[d, r, :, :] = v[:, :512].mean(axis=0)
                lse[d, r, :] = np.log(n)
    return O, lse


@pytest.fixture(scope="module", params=SPECS, ids=lambda s: s.name)
def planted(request):
    inp = wl.make_decode_inputs(request.param, kv_rows=PC.kv_rows)
    n, E, rows = PC.expected(inp)
    return inp, n, E


def test_exact_rows_pass(planted):
    inp, n, E = planted
    O, lse = _simulate(inp)
    PC.check(O.astype(np.float32), lse.astype(np.float32), n, E, inp["name"])


def test_off_by_one_in_position_formula_fails(planted):
    inp, n, E = planted
    O, lse = _simulate(inp, pos_fn=lambda j, d, D, I: _local_to_global(j, d, D, I) + 1)
    with pytest.raises(AssertionError):
        PC.check(O, lse, n, E, inp["name"])


def test_interleave_ignored_fails(planted):
    inp, n, E = planted
    if inp["interleave"] == 1:
        pytest.skip("interleave 1: the mistake is invisible")
    O, lse = _simulate(inp, pos_fn=lambda j, d, D, I: j * D + d)
    with pytest.raises(AssertionError):
        PC.check(O, lse, n, E, inp["name"])


def test_wrong_offset_in_block_fails(planted):
    inp, n, E = planted
    bs = inp["block_size"]
    tab = inp["block_table"]
    # the walker's offset taken from the local index instead of the position
    O, lse = _simulate(inp, row_fn=lambda b, p: tab[b, p // bs].astype(np.int64) * bs + (p + 1) % bs)
    with pytest.raises(AssertionError):
        PC.check(O, lse, n, E, inp["name"])


def test_next_table_column_fails(planted):
    inp, n, E = planted
    W = inp["block_table"].shape[1]
    bsz = inp["block_size"]

    def rows(b, p):
        col = np.minimum(p // bsz + 1, W - 1)
        return inp["block_table"][b, col].astype(np.int64) * bsz + p % bsz
    O, lse = _simulate(inp, row_fn=rows)
    with pytest.raises(AssertionError):
        PC.check(O, lse, n, E, inp["name"])
