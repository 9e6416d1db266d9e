"""Bit-exact check of the device's token -> shard mapper and block-table
walker, through the attention arithmetic itself.

With ``scale = 0`` every live token of a (row, shard) gets score 0, hence
weight exactly 1, so the decode's partial output is the plain mean of the
value rows it read and its LSE is ln(count).  The cache rows are planted so
that the row holding logical position p carries small integers derived from
p (base-4 digits of p and of a 16-bit multiplicative hash of p) in its first
value dims, zeros elsewhere.  Small integers are exact in bf16, their sums
stay far below 2^24 (exact in fp32 whatever the summation order), and the
one division by the count, plus the split merge, perturb the mean by about
1e-6 relative.  So ``round(n_d * O_d[k])`` recovers the integer digit sum
over the exact token set the kernel read, and ``round(exp(lse_d))`` the
count: both compared exactly with the oracle's sets (``shard_positions``
over the row's own length; the value at position p is placed by the paged
layout, so a wrong block, a wrong offset or a wrong shard token changes a
sum).  A row that the kernel reads but no position owns holds NaN (the
generator's poison) and fails the check too.

The statement that the mapping and the indexing are bit-exact comes from the
decode-context-parallel pages' interleave rule ("[Kimi-K3] DCP support"
summary on prhub.com.cn, implementation step 3: runs of
cp_kv_cache_interleave_size dealt round-robin over the DCP ranks) and the
block-table contract of "perf(mla): fuse K3 DCP verification queries"
(review follow-up).
"""
from __future__ import annotations

import numpy as np

import oracle
from oracle.dcp_oracle import KDIM

POS_DIGITS = 10    # base-4 digits of p: positions below 4^10 = 1,048,576
HASH_DIGITS = 8    # base-4 digits of (p * 40503) mod 2^16
CODED = POS_DIGITS + HASH_DIGITS
HASH_MUL = 40503
_BF16_OF_SMALL_INT = {v: np.uint16(np.float32(v).view(np.uint32) >> 16) for v in range(4)}


def digits(p: np.ndarray) -> np.ndarray:
    """int64 [len(p), CODED]: base-4 digits of p, then of its hash."""
    p = np.asarray(p, dtype=np.int64)
    assert (p < 4 ** POS_DIGITS).all()
    h = (p * HASH_MUL) % (1 << 16)
    out = np.empty((p.size, CODED), dtype=np.int64)
    for k in range(POS_DIGITS):
        out[:, k] = (p >> (2 * k)) & 3
    for k in range(HASH_DIGITS):
        out[:, POS_DIGITS + k] = (h >> (2 * k)) & 3
    return out


def kv_rows(b: int, positions: np.ndarray) -> np.ndarray:
    """bf16 bits of the planted latent rows (the generator's ``kv_rows`` hook):
    the digits of the position in dims [0, CODED), zeros elsewhere."""
    dg = digits(positions)
    rows = np.zeros((dg.shape[0], KDIM), dtype=np.uint16)
    lut = np.array([_BF16_OF_SMALL_INT[v] for v in range(4)], dtype=np.uint16)
    rows[:, :CODED] = lut[dg]
    return rows


def expected(inp: dict, rows=None):
    """For each listed row r and shard d: the oracle's token count n[d, r]
    and integer digit sums E[d, r, k] over its shard set."""
    D, I = inp["D"], inp["interleave"]
    _, L, pad = oracle.row_lengths(inp["seq_lens"], inp["query_start_loc"], inp["T"])
    rows = np.arange(inp["T"]) if rows is None else np.asarray(rows)
    n = np.zeros((D, len(rows)), dtype=np.int64)
    E = np.zeros((D, len(rows), CODED), dtype=np.int64)
    for j, r in enumerate(rows):
        if pad[r]:
            continue
        for d in range(D):
            pos = oracle.shard_positions(int(L[r]), d, D, I)
            n[d, j] = pos.size
            if pos.size:
                E[d, j] = digits(pos).sum(axis=0)
    return n, E, rows


def check(O: np.ndarray, lse: np.ndarray, n: np.ndarray, E: np.ndarray, what: str = "") -> None:
    """O [D, R, H, 512] and lse [D, R, H] (fp32, from the device) against the
    oracle's counts and digit sums; raises AssertionError on any mismatch."""
    O = np.asarray(O, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    assert not np.isnan(O).any() and not np.isnan(lse).any(), what + ": NaN (a poisoned row was read)"
    empty = n == 0
    assert (lse[empty] == -np.inf).all(), what + ": an empty shard has a finite LSE"
    assert (O[empty] == 0).all(), what + ": an empty shard has a nonzero output"
    live = ~empty
    if not live.any():
        return
    # every head saw the same scores (all zero) and the same rows
    assert (O == O[:, :, :1]).all() and (lse == lse[:, :, :1]).all(), what + ": heads differ"
    Ol, ll, nl, El = O[live][:, 0], lse[live][:, 0], n[live], E[live]
    count = np.rint(np.exp(ll)).astype(np.int64)
    assert np.array_equal(count, nl), what + ": token counts differ: %s" % _first_diff(count, nl)
    assert np.all(np.abs(ll - np.log(nl)) <= 4e-6 * np.maximum(1.0, np.log(nl))), what + ": LSE != ln(count)"
    sums = np.rint(Ol[:, :CODED] * nl[:, None]).astype(np.int64)
    assert np.array_equal(sums, El), what + ": digit sums differ: %s" % _first_diff(sums, El)
    assert np.all(np.abs(Ol[:, :CODED] * nl[:, None] - El) < 0.25), what + ": digit sums not near integers"
    assert (Ol[:, CODED:] == 0).all(), what + ": uncoded value dims are nonzero"


def _first_diff(a, b):
    i = np.argwhere(a != b)
    if i.size == 0:
        return "none"
    k = tuple(i[0])
    return "at %s: got %s, want %s" % (k, a[k], b[k])
