"""Seeded synthetic inputs for the MLA decode-context-parallel (DCP) hot path.

This module is the only code shared by the CPU oracle's tests and the CUDA
path's tests and benchmark.  It draws random numbers and lays them out; it
holds none of the method's arithmetic (no sharding, no attention, no combine).

Recipe (shapes and distributions follow the workloads described for decode
context parallelism on Kimi-K3-style MLA layers: 128 heads, a 576-wide latent
KV row = 512 compressed-KV dims + 64 rope dims, bf16, paged cache):

* ``q`` bf16 ``[T, H, 576]`` and every live KV latent row bf16 ``[576]`` are
  iid N(0, 1) float32 draws rounded to bf16 (round-to-nearest-even).
* KV rows are drawn per request in logical token order, in chunks of
  ``CHUNK`` tokens; chunk ``c`` of request ``b`` of stream ``s`` uses
  ``numpy.random.default_rng([seed, s, b, c])``, so the bytes do not depend on
  the thread count.  The long-context workload draws positions below
  ``prefix_len`` from a "prefix" stream and the rest from a "suffix" stream
  (the pages' 120k workload is a 114k shared prefix plus a 6k suffix).
* The physical block of each logical block comes from a random permutation of
  all blocks; unused block-table columns hold -1 and cache slots past a
  request's length hold bf16 NaN, so that a kernel that touches either shows.
* ``seq_lens`` are explicit or integers uniform on ``[lo, hi]`` inclusive;
  ``query_start_loc`` is the exclusive prefix sum of the per-request query
  lengths.

Combine-sweep inputs (``make_combine_inputs``) are fp32 partial outputs
N(0, 1), partial LSEs N(5, 3), 10 % of (row, shard) pairs empty (LSE -inf,
output NaN), 5 % padding rows (seq_len 0, finite garbage LSE, NaN output),
one request per row.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Optional, Sequence, Tuple, Union

import numpy as np

LATENT = 512          # compressed-KV (kv_c) dims = V dims
ROPE = 64             # k_pe dims
KDIM = LATENT + ROPE  # 576: the width of one latent cache row and of one query head row
CHUNK = 2048          # tokens per independently seeded chunk
BF16_NAN = np.uint16(0x7FC0)
FP8_NAN = np.uint8(0x7F)   # FP8 E4M3 NaN code

# stream tags for default_rng([seed, stream, ...])
_S_SEQ, _S_TABLE, _S_KV, _S_KV_SUFFIX, _S_Q, _S_COMBINE = 0, 1, 2, 3, 4, 5


def quantize_fp8_e4m3(x: np.ndarray):
    """Per-row FP8 E4M3 codes and scales of float32 rows [n, 576]: scale =
    2^ceil(log2(max |x| / 256)) (1 for an all-zero row), codes = x / scale
    rounded to the nearest E4M3 value (ties to even; torch's conversion).
    Power-of-two scales keep x / scale exact before the rounding."""
    import torch
    amax = np.abs(x).max(axis=1)
    e = np.ceil(np.log2(np.where(amax > 0, amax / 256.0, 1.0)))
    sc = np.ldexp(np.float32(1.0), e.astype(np.int32)).astype(np.float32)
    y = torch.from_numpy(np.ascontiguousarray(x / sc[:, None], dtype=np.float32))
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes, sc


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the uint16 bits.

    Inputs are finite normal draws, so no NaN handling is needed here.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


@dataclass(frozen=True)
class DecodeSpec:
    """One decode workload.  ``seq_lens`` is a tuple or ("uniform", lo, hi)."""
    name: str
    seed: int
    B: int
    seq_lens: Union[Tuple[int, ...], Tuple[str, int, int]]
    q_len: Union[int, Tuple[int, ...]] = 1
    H: int = 128
    block_size: int = 64
    D: int = 8
    interleave: int = 1
    scale: float = 1.0 / math.sqrt(192.0)
    prefix_len: Optional[int] = None
    spare_cols: int = 2          # poisoned (-1) block-table columns past the widest request
    extra_rows: int = 0          # rows past query_start_loc[B] (no request: padding)
    tail_fill_nan: bool = True   # cache slots past seq_len hold NaN
    # "global": one block table per request over all positions; "local": the
    # per-shard layout, each shard's tokens stored densely in its own blocks
    # (block_table [D, B, W])
    layout: str = "global"
    # the first prefix_len tokens of every request are the same tokens (drawn
    # once) stored in the same blocks (those holding only prefix tokens)
    shared_prefix: bool = False
    # latent cache format: "bf16", or "fp8_e4m3" codes with one fp32 scale per
    # cache slot (a power of two per token: 2^ceil(log2(max |x| / 256)), so
    # that every code stays within the format's finite range)
    kv_dtype: str = "bf16"

    def q_lens(self) -> Tuple[int, ...]:
        if isinstance(self.q_len, int):
            return (self.q_len,) * self.B
        assert len(self.q_len) == self.B
        return tuple(self.q_len)

    def resolved_seq_lens(self) -> np.ndarray:
        s = self.seq_lens
        if len(s) == 3 and s[0] == "uniform":
            rng = np.random.default_rng([self.seed, _S_SEQ])
            return rng.integers(int(s[1]), int(s[2]) + 1, size=self.B).astype(np.int32)
        assert len(s) == self.B, (self.name, len(s), self.B)
        return np.asarray(s, dtype=np.int32)


# The five workloads.  Names say what they are; the first is small enough for
# the float64 oracle to finish in seconds.
TINY = DecodeSpec("tiny_b2_h16_d4", seed=0, B=2, seq_lens=(3, 37), H=16,
                  block_size=16, D=4, interleave=1)
LONG_120K = DecodeSpec("long_ctx_120k_b1_d8_i1", seed=1, B=1, seq_lens=(120_000,),
                       H=128, block_size=64, D=8, interleave=1, prefix_len=114_000)
BATCHED_B64 = DecodeSpec("batched_b64_d8_i64", seed=2, B=64,
                         seq_lens=("uniform", 1024, 32768), H=128, block_size=64,
                         D=8, interleave=64)
SPEC_VERIFY_B32 = DecodeSpec("spec_verify_b32_q4_d8_i1", seed=3, B=32,
                             seq_lens=("uniform", 8192, 65536), q_len=4, H=128,
                             block_size=64, D=8, interleave=1)
# the 120k workload as two requests sharing the 114,000-token prefix (the
# blocks that hold only prefix tokens are shared), in the global layout and in
# the per-shard (rank-local) layout
LONG_120K_B2_PREFIX = DecodeSpec("long_ctx_120k_b2_shared_prefix_d8_i1", seed=6, B=2, seq_lens=(120_000, 120_000),
                                 H=128, block_size=64, D=8, interleave=1, prefix_len=114_000, shared_prefix=True)
LONG_120K_B2_PREFIX_LOCAL = DecodeSpec("long_ctx_120k_b2_shared_prefix_d8_i1_local", seed=6, B=2,
                                       seq_lens=(120_000, 120_000), H=128, block_size=64, D=8, interleave=1,
                                       prefix_len=114_000, shared_prefix=True, layout="local")
LONG_120K_FP8 = DecodeSpec("long_ctx_120k_b1_d8_i1_fp8", seed=1, B=1, seq_lens=(120_000,), H=128, block_size=64,
                           D=8, interleave=1, prefix_len=114_000, kv_dtype="fp8_e4m3")
BATCHED_B64_LOCAL = DecodeSpec("batched_b64_d8_i64_local", seed=2, B=64, seq_lens=("uniform", 1024, 32768), H=128,
                               block_size=64, D=8, interleave=64, layout="local")
COMBINE_SWEEP = [(D, T) for D in (2, 4, 8) for T in (1, 64, 1024, 4096)]
COMBINE_H = 128

DECODE_WORKLOADS = {s.name: s for s in (TINY, LONG_120K, BATCHED_B64, SPEC_VERIFY_B32, LONG_120K_B2_PREFIX,
                                         LONG_120K_B2_PREFIX_LOCAL, BATCHED_B64_LOCAL, LONG_120K_FP8)}


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _fill_request(store, phys_rows: np.ndarray, spec: DecodeSpec, b: int, L: int) -> None:
    """Draw request b's L latent rows in logical order and store them.  With a
    shared prefix every request draws its prefix from request 0's stream."""
    jobs = []
    if spec.prefix_len is not None and spec.prefix_len < L:
        segs = [(0, spec.prefix_len, _S_KV, 0 if spec.shared_prefix else b), (spec.prefix_len, L, _S_KV_SUFFIX, b)]
    else:
        segs = [(0, L, _S_KV, b)]
    for lo, hi, stream, owner in segs:
        for c, start in enumerate(range(lo, hi, CHUNK)):
            jobs.append((stream, owner, c, start, min(hi, start + CHUNK)))

    def work(job):
        stream, owner, c, start, stop = job
        rng = np.random.default_rng([spec.seed, stream, owner, c])
        x = rng.standard_normal((stop - start, KDIM), dtype=np.float32)
        store(phys_rows[start:stop], x)

    if len(jobs) == 1:
        work(jobs[0])
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, jobs))


def make_decode_inputs(spec: DecodeSpec, kv_rows=None) -> dict:
    """Host (numpy) inputs of one decode workload.

    Returns a dict with ``q`` uint16 [T, H, 576] (bf16 bits), ``kv_cache``
    uint16 [num_blocks, block_size, 576], ``block_table`` int32 [B, W],
    ``seq_lens`` int32 [B], ``query_start_loc`` int32 [B + 1] and the scalar
    parameters (``T``, ``H``, ``D``, ``interleave``, ``block_size``,
    ``scale``, ``max_seq_len``, ``max_q_len``).

    ``kv_rows(b, positions)``, when given, supplies the bf16 bits
    (uint16 [len(positions), 576]) of request b's latent rows at those
    logical positions instead of the seeded normal draws (for tests that
    plant known values, e.g. rows that encode their own position).
    """
    seq = spec.resolved_seq_lens()
    qlens = np.asarray(spec.q_lens(), dtype=np.int32)
    B, bs = spec.B, spec.block_size
    qsl = np.zeros(B + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(qlens)
    T = int(qsl[-1]) + spec.extra_rows
    placement = _place_global if spec.layout == "global" else _place_local
    table, phys_of, num_blocks = placement(spec, seq)

    fp8 = spec.kv_dtype == "fp8_e4m3"
    kv = np.empty((num_blocks, bs, KDIM), dtype=np.uint8 if fp8 else np.uint16)
    if spec.tail_fill_nan:
        kv.fill(FP8_NAN if fp8 else BF16_NAN)
    else:
        kv.fill(0)
    kv_flat = kv.reshape(num_blocks * bs, KDIM)
    kv_scale = np.ones((num_blocks, bs), dtype=np.float32) if fp8 else None

    def store(rows, x):
        if fp8:
            codes, sc = quantize_fp8_e4m3(x)
            kv_flat[rows] = codes
            kv_scale.reshape(-1)[rows] = sc
        else:
            kv_flat[rows] = f32_to_bf16_bits(x)

    for b in range(B):
        L = int(seq[b])
        if L == 0:
            continue
        pos = np.arange(L, dtype=np.int64)
        phys = phys_of(b, pos)
        if kv_rows is None:
            _fill_request(store, phys, spec, b, L)
        else:
            bits = kv_rows(b, pos)
            store(phys, (bits.astype(np.uint32) << np.uint32(16)).view(np.float32))

    q = f32_to_bf16_bits(np.random.default_rng([spec.seed, _S_Q]).standard_normal(
        (T, spec.H, KDIM), dtype=np.float32))
    return dict(
        name=spec.name, q=q, kv_cache=kv, block_table=table, seq_lens=seq,
        query_start_loc=qsl, B=B, T=T, H=spec.H, D=spec.D,
        interleave=spec.interleave, block_size=bs, scale=float(spec.scale),
        max_seq_len=int(seq.max(initial=0)), max_q_len=int(qlens.max(initial=0)),
        num_blocks=num_blocks, layout=spec.layout, kv_dtype=spec.kv_dtype, kv_scale=kv_scale,
    )


def _shared_blocks(spec: DecodeSpec, counts: np.ndarray) -> np.ndarray:
    """Per request, how many leading blocks hold only shared-prefix tokens
    (counts[b] = prefix tokens of request b in the table row's order)."""
    if not spec.shared_prefix or spec.prefix_len is None:
        return np.zeros_like(counts)
    return counts // spec.block_size


def _allocate(spec: DecodeSpec, nblk: np.ndarray, nshared: np.ndarray, W: int, rng_stream: int):
    """Block ids for a set of table rows (nblk[i] blocks each; the first
    nshared[i] of them are the rows' common prefix blocks, allocated once),
    drawn from a random permutation of all blocks.  Returns (table rows
    [len(nblk), W] with -1 in unused columns, number of blocks)."""
    shared = int(nshared.max(initial=0))
    own = nblk - np.minimum(nshared, nblk)
    num_blocks = max(1, shared + int(own.sum()))
    key = [spec.seed, _S_TABLE] if rng_stream == 0 else [spec.seed, _S_TABLE, rng_stream]
    perm = np.random.default_rng(key).permutation(num_blocks).astype(np.int32)
    rows = np.full((len(nblk), max(W, 1)), -1, dtype=np.int32)
    off = shared
    for i in range(len(nblk)):
        ns = int(min(nshared[i], nblk[i]))
        rows[i, :ns] = perm[:ns]
        n = int(nblk[i]) - ns
        rows[i, ns:ns + n] = perm[off:off + n]
        off += n
    return rows, num_blocks


def _place_global(spec: DecodeSpec, seq: np.ndarray):
    """One table row per request: position p of request b lives in row
    table[b, p // bs] * bs + p % bs."""
    bs = spec.block_size
    nblk = (seq.astype(np.int64) + bs - 1) // bs
    pre = np.minimum(seq.astype(np.int64), spec.prefix_len or 0)
    W = int(nblk.max(initial=0)) + spec.spare_cols
    table, num_blocks = _allocate(spec, nblk, _shared_blocks(spec, pre), W, 0)

    def phys_of(b, pos):
        return table[b, pos // bs].astype(np.int64) * bs + pos % bs
    return table, phys_of, num_blocks


def _place_local(spec: DecodeSpec, seq: np.ndarray):
    """The per-shard (DCP rank-local) layout: shard d stores the positions it
    owns, dealt round-robin to the D shards in runs of I, densely in order;
    its j-th token of request b lives in row table[d, b, j // bs] * bs +
    j % bs.  This is how each rank's own cache holds its share of the
    context; the placement is input construction, checked against the global
    layout by the oracle's tests."""
    bs, D, I = spec.block_size, spec.D, spec.interleave
    B = len(seq)
    owners, local_idx, counts = [], [], np.zeros((D, B), dtype=np.int64)
    for b in range(B):
        p = np.arange(int(seq[b]), dtype=np.int64)
        run = p // I
        d = run % D
        j = (run // D) * I + p % I  # rank of p among its shard's positions
        owners.append(d)
        local_idx.append(j)
        for dd in range(D):
            counts[dd, b] = int((d == dd).sum())
    nblk = (counts + bs - 1) // bs
    pre_counts = np.zeros((D, B), dtype=np.int64)
    if spec.shared_prefix and spec.prefix_len:
        for b in range(B):
            k = min(int(seq[b]), spec.prefix_len)
            for dd in range(D):
                pre_counts[dd, b] = int((owners[b][:k] == dd).sum())
    W = int(nblk.max(initial=0)) + spec.spare_cols
    num_blocks = 0
    tables = np.full((D, B, max(W, 1)), -1, dtype=np.int32)
    # each shard's blocks are a contiguous range of one cache (on one GPU the
    # D rank-local caches are partitions of one array), permuted within it
    for dd in range(D):
        r, n = _allocate(spec, nblk[dd], _shared_blocks(spec, pre_counts[dd]), W, 1 + dd)
        tables[dd] = np.where(r >= 0, r + num_blocks, -1)
        num_blocks += n

    def phys_of(b, pos):
        d, j = owners[b][pos], local_idx[b][pos]
        return tables[d, b, j // bs].astype(np.int64) * bs + j % bs
    return tables, phys_of, num_blocks


def combine_masks(D: int, T: int, seed: int, empty_frac: float = 0.10,
                  padding_frac: float = 0.05):
    """(empty[D, T] bool, padding[T] bool) for a combine sweep point.

    Every non-padding row keeps at least one live shard (the rows that drew
    all-empty are given one live shard at random).
    """
    rng = np.random.default_rng([seed, _S_COMBINE])
    padding = rng.random(T) < padding_frac
    empty = rng.random((D, T)) < empty_frac
    dead = empty.all(axis=0) & ~padding
    for r in np.nonzero(dead)[0]:
        empty[rng.integers(0, D), r] = False
    return empty, padding


def make_combine_inputs(D: int, T: int, H: int = COMBINE_H, seed: Optional[int] = None,
                        device=None):
    """Inputs of one combine-sweep point.

    With ``device=None`` returns numpy arrays (O_part float32 [D, T, H, 512],
    lse_part float32 [D, T, H], seq_lens int32 [T], query_start_loc int32
    [T + 1], empty, padding).  With a torch device the two large arrays are
    drawn there by torch's generator seeded with ``seed`` (same recipe, other
    bit stream) and returned as torch tensors; the masks stay numpy.
    """
    if seed is None:
        seed = 4 + COMBINE_SWEEP.index((D, T)) if (D, T) in COMBINE_SWEEP else 4
    empty, padding = combine_masks(D, T, seed)
    seq_lens = np.where(padding, 0, 1 + np.arange(T) % 7).astype(np.int32)
    qsl = np.arange(T + 1, dtype=np.int32)
    if device is None:
        rng = np.random.default_rng([seed, _S_COMBINE, 1])
        O = rng.standard_normal((D, T, H, LATENT), dtype=np.float32)
        lse = (5.0 + 3.0 * rng.standard_normal((D, T, H))).astype(np.float32)
        O[empty] = np.nan
        lse[empty] = -np.inf
        O[:, padding] = np.nan
        return O, lse, seq_lens, qsl, empty, padding
    import torch
    g = torch.Generator(device=device).manual_seed(seed)
    O = torch.randn((D, T, H, LATENT), generator=g, device=device, dtype=torch.float32)
    lse = 5.0 + 3.0 * torch.randn((D, T, H), generator=g, device=device, dtype=torch.float32)
    em = torch.from_numpy(empty).to(device)
    pm = torch.from_numpy(padding).to(device)
    O[em] = float("nan")
    lse[em] = float("-inf")
    O[:, pm] = float("nan")
    return O, lse, seq_lens, qsl, empty, padding


def to_torch(inp: dict, device="cuda") -> dict:
    """Device copies of a decode workload's arrays (bf16 bits viewed as
    torch.bfloat16, int32 tables)."""
    import torch

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)
    if inp.get("kv_dtype", "bf16") == "fp8_e4m3":
        kv = torch.from_numpy(np.ascontiguousarray(inp["kv_cache"])).to(device)
        extra = dict(kv_scale=torch.from_numpy(inp["kv_scale"]).to(device))
    else:
        kv = bf16(inp["kv_cache"])
        extra = {}
    return dict(
        q=bf16(inp["q"]), kv_cache=kv, **extra,
        block_table=torch.from_numpy(inp["block_table"]).to(device),
        seq_lens=torch.from_numpy(inp["seq_lens"]).to(device),
        query_start_loc=torch.from_numpy(inp["query_start_loc"]).to(device),
    )
