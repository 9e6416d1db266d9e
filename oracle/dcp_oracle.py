"""CPU float64 oracle for the MLA decode-context-parallel (DCP) hot path.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
this module.  The CUDA library never calls it and shares no code with it.

It states, as plainly as possible, what the hot path computes:

1. per query row, that row's own context length (speculative-verification
   rows of one request see a causally shorter context);
2. which context shard owns each token position (round-robin in runs of
   ``interleave`` over ``D`` shards);
3. where each token's latent row lives in the paged cache (block table);
4. per (row, head, shard): softmax attention of the 576-wide absorbed query
   against the shard's 576-wide latent rows, values = the first 512 dims,
   returning the normalised partial output O_d and its natural-log LSE L_d;
   a shard with no tokens, or a padding row, gets L_d = -inf and O_d = NaN
   (NaN on purpose: a correct combine never reads it);
5. the LSE-weighted combine over shards with empty-shard and padding-row
   masking;
6. the step before attention: the decode query ``[ql_nope | q_pe]`` and the
   write of this step's latent rows into the paged cache.

Sources (pages on decode context parallelism for MLA):
  [PR50484]  "[Kimi-K3] DCP support", vllm-project/vllm pull request 50484
             (Summary; "CUDA-graph padding follow-up"; the review thread on the
             ``repeat_interleave`` padding-row mask; the merged GLM-5.2 DCP+MTP
             bugfix text on localising per-token seq_lens after MTP expansion).
  [PRHUB]    prhub.com.cn summary of the same pull request (implementation
             breakdown steps 3-4: interleave alignment via lcm, source-side -inf
             masking of empty shards, exp2 LSE-weighted merge, consumer-side
             zero-weight skip; key source snippet "Decode: latent multi-query
             attention", where the cache write precedes ``forward_mqa`` and
             ``combine(latent_out, lse, seq_lens, query_start_loc)`` follows).
  [PR565]    "perf(mla): fuse K3 DCP verification queries",
             local-inference-lab/vllm pull request 565 (Summary: K=3
             verification rows share KV loads; review follow-up on the
             block-table width contract and the 192-wide query row).

Everything is float64.  bf16 inputs are widened exactly.
"""
from __future__ import annotations

import numpy as np

LATENT = 512          # V dims: the compressed-KV part of a latent row
ROPE = 64             # k_pe dims
KDIM = LATENT + ROPE  # 576: query head row = [q absorbed into latent | q_pe]

__all__ = [
    "bf16_to_f64", "row_lengths", "shard_of", "local_len", "shard_positions",
    "physical_rows", "physical_rows_local", "gather_latents", "scores", "shard_partial",
    "decode_partial_row", "decode_partial", "lse_combine", "attention", "concat_cache",
    "fp8_e4m3_to_f64", "kv_rows_f64",
]


# ---------------------------------------------------------------------------
# input decoding
# ---------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) exactly to float64."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# step 1: rows and per-row context length
# ---------------------------------------------------------------------------
def row_lengths(seq_lens: np.ndarray, query_start_loc: np.ndarray, T: int):
    """Per query row: (request index or -1, own context length, padding flag).

    Rows of request b are ``query_start_loc[b] .. query_start_loc[b+1]-1``
    [PRHUB, "Decode" snippet: ``combine(..., seq_lens, query_start_loc)``].
    ``seq_lens[b]`` already counts the request's new tokens, which are written
    to the cache before attention [PRHUB, same snippet: ``_decode_concat_cache``
    runs before ``forward_mqa``], so row i of a request with q_len rows sees
    ``seq_len - (q_len - 1 - i)`` tokens, itself included.  The per-row length
    is formed first and only then split over shards [PR50484, merged bugfix
    text: per-token seq_lens are localised after the MTP expansion].

    A row is padding when its request has ``seq_len == 0`` (a CUDA-graph
    padding request) [PR50484, "CUDA-graph padding follow-up" and the review
    thread on ``repeat_interleave(seq_lens == 0, query_lens, ...)``], or when
    it lies past ``query_start_loc[B]`` (reading: the rows that
    ``output_size=lse.shape[0]`` pads beyond the last request).
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    B = len(seq_lens)
    req = np.full(T, -1, dtype=np.int64)
    L = np.zeros(T, dtype=np.int64)
    padding = np.ones(T, dtype=bool)
    for b in range(B):
        q_len = int(qsl[b + 1] - qsl[b])
        for i in range(q_len):
            r = int(qsl[b]) + i
            if r >= T:
                break
            req[r] = b
            if seq_lens[b] == 0:
                continue  # padding request: stays padding, length 0
            padding[r] = False
            L[r] = max(0, int(seq_lens[b]) - (q_len - 1 - i))
    return req, L, padding


# ---------------------------------------------------------------------------
# step 2: token -> shard
# ---------------------------------------------------------------------------
def shard_of(p, D: int, I: int):
    """Shard owning token position p: positions are dealt to the D shards
    round-robin in runs of I = cp_kv_cache_interleave_size, i.e. runs
    [0, I) -> shard 0, [I, 2I) -> shard 1, ..., wrapping after D runs
    [PRHUB, implementation step 3: the DCP chunk boundary is
    dcp_size * cp_kv_cache_interleave_size]."""
    return (np.asarray(p, dtype=np.int64) // I) % D


def shard_positions(L: int, d: int, D: int, I: int) -> np.ndarray:
    """The set S_d = {p < L : shard_of(p) = d}, in increasing order."""
    p = np.arange(int(L), dtype=np.int64)
    return p[shard_of(p, D, I) == d]


def local_len(L: int, d: int, D: int, I: int) -> int:
    """|S_d|: how many of the first L positions shard d owns (by counting)."""
    return int(shard_positions(L, d, D, I).size)


# ---------------------------------------------------------------------------
# step 3: paged block table
# ---------------------------------------------------------------------------
def physical_rows(table_row: np.ndarray, block_size: int, positions: np.ndarray) -> np.ndarray:
    """Cache row (block * block_size + offset) of each logical position:
    logical block p // block_size is looked up in the request's block-table
    row; only the columns a position refers to are read [PR565, review
    follow-up: the table may be wider than what any sequence references]."""
    positions = np.asarray(positions, dtype=np.int64)
    blocks = np.asarray(table_row, dtype=np.int64)[positions // block_size]
    return blocks * block_size + positions % block_size


def physical_rows_local(shard_table_row: np.ndarray, block_size: int, n: int) -> np.ndarray:
    """Per-shard (DCP rank-local) layout: a shard stores only its own tokens,
    densely and in order, so its j-th token (the j-th position it owns) lives
    in row table[j // block_size] * block_size + j % block_size of its own
    block-table row; that row must cover the shard's local length
    [PR565, review follow-up: the page table must cover the largest local KV
    shard; PR50484, Summary: each DCP rank keeps its own slice of the
    context]."""
    j = np.arange(int(n), dtype=np.int64)
    blocks = np.asarray(shard_table_row, dtype=np.int64)[j // block_size]
    return blocks * block_size + j % block_size


def gather_latents(kv_cache_bits: np.ndarray, table_row: np.ndarray, block_size: int,
                   positions: np.ndarray) -> np.ndarray:
    """float64 [len(positions), 576] latent rows of the given logical positions."""
    nb, bs, kd = kv_cache_bits.shape
    assert bs == block_size and kd == KDIM
    rows = physical_rows(table_row, block_size, positions)
    return bf16_to_f64(kv_cache_bits.reshape(nb * bs, kd)[rows])


# ---------------------------------------------------------------------------
# step 4: per-shard partial attention
# ---------------------------------------------------------------------------
def scores(q_heads: np.ndarray, latents: np.ndarray, scale: float) -> np.ndarray:
    """s[h, t] = scale * sum_{k < 576} q[h, k] * kv[t, k]: the absorbed query
    [ql_nope | q_pe] against the full latent row [kv_c | k_pe]
    [PRHUB, "Decode" snippet: ``mqa_q`` is the concatenation fed to
    ``forward_mqa`` together with the latent cache]."""
    return scale * (np.asarray(q_heads, np.float64) @ np.asarray(latents, np.float64).T)


def shard_partial(s: np.ndarray, values: np.ndarray):
    """Softmax attention over one shard's tokens.

    s: [H, n] scores, values: [n, 512].  Returns (O [H, 512], lse [H]) with
    lse = ln sum_t exp(s_t) and O = sum_t exp(s_t - lse) v_t.  n must be > 0.
    """
    m = s.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(s - m).sum(axis=1))
    p = np.exp(s - lse[:, None])
    return p @ values, lse


def decode_partial_row(q_heads: np.ndarray, kv_cache_bits: np.ndarray, table_row: np.ndarray,
                       block_size: int, L: int, D: int, I: int, scale: float, padding: bool,
                       local: bool = False, rows_f64: np.ndarray = None):
    """(O [D, H, 512], lse [D, H]) of one query row over its own L tokens.
    table_row is the request's block-table row, or with ``local`` its D
    per-shard rows [D, W] (the shard's tokens gathered by local index).
    ``rows_f64`` ([num_blocks * block_size, 576], from kv_rows_f64) replaces
    the bf16 cache bits, e.g. for an fp8 cache.

    Empty shards and padding rows are masked at the source: lse = -inf,
    O = NaN [PR50484, Summary: empty-KV-shard masking; PRHUB, implementation
    step 4: an empty KV shard's LSE is set to -inf at the source]."""
    H = q_heads.shape[0]
    O = np.full((D, H, LATENT), np.nan)
    lse = np.full((D, H), -np.inf)
    if padding or L <= 0:
        return O, lse
    q = bf16_to_f64(q_heads)
    for d in range(D):
        pos = shard_positions(L, d, D, I)
        if pos.size == 0:
            continue
        if local:
            rows = physical_rows_local(table_row[d], block_size, pos.size)
        else:
            rows = physical_rows(table_row, block_size, pos)
        if rows_f64 is not None:
            kv = rows_f64[rows]
        elif local:
            nb, bs, kd = kv_cache_bits.shape
            kv = bf16_to_f64(kv_cache_bits.reshape(nb * bs, kd)[rows])
        else:
            kv = gather_latents(kv_cache_bits, table_row, block_size, pos)
        O[d], lse[d] = shard_partial(scores(q, kv, scale), kv[:, :LATENT])
    return O, lse


def decode_partial(inp: dict, rows=None):
    """Oracle of ``dcp_mla_decode_partial`` on a workload dict from
    ``workloads.make_decode_inputs``, for the listed rows (default all).

    Returns (O_part [D, R, H, 512], lse_part [D, R, H], rows).  With
    ``inp["layout"] == "local"`` the block table is [D, B, W]: each shard's
    own table (the per-shard layout).
    """
    T, H, D = inp["T"], inp["H"], inp["D"]
    local = inp.get("layout", "global") == "local"
    fp8 = inp.get("kv_dtype", "bf16") == "fp8_e4m3"
    rows_f64 = kv_rows_f64(inp) if fp8 else None
    req, L, padding = row_lengths(inp["seq_lens"], inp["query_start_loc"], T)
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    O = np.full((D, len(rows), H, LATENT), np.nan)
    lse = np.full((D, len(rows), H), -np.inf)
    for j, r in enumerate(rows):
        b = req[r]
        if b < 0:
            table_row = None
        else:
            table_row = inp["block_table"][:, b] if local else inp["block_table"][b]
        O[:, j], lse[:, j] = decode_partial_row(
            inp["q"][r], inp["kv_cache"], table_row, inp["block_size"], int(L[r]),
            D, inp["interleave"], inp["scale"], bool(padding[r]), local=local, rows_f64=rows_f64)
    return O, lse, rows


# ---------------------------------------------------------------------------
# step 5: LSE-weighted combine
# ---------------------------------------------------------------------------
def lse_combine(O_part: np.ndarray, lse_part: np.ndarray, padding: np.ndarray):
    """Merge D shard partials.  O_part [D, ..., 512], lse_part [D, ...],
    padding [rows] broadcast over the trailing head axis.

    Per (row, head): E = {d : lse_d != -inf}.  A padding row, or an empty E,
    gives out = 0 and out_lse = -inf.  Otherwise, with M = max_{d in E} lse_d
    and w_d = exp(lse_d - M), out = sum_E w_d O_d / sum_E w_d and
    out_lse = M + ln sum_E w_d.  This is the pages' exp2 weighting
    exp2(lse_d * log2 e - M') written in natural-log form; O_d is never used
    for d outside E (its payload may be stale)
    [PRHUB, implementation step 4 and risk 4: source -inf mask plus
    consumer-side zero-weight skip; PR50484, "CUDA-graph padding follow-up"].
    """
    O_part = np.asarray(O_part, dtype=np.float64)
    lse = np.asarray(lse_part, dtype=np.float64)
    D = lse.shape[0]
    pad = np.asarray(padding, dtype=bool).reshape((-1,) + (1,) * (lse.ndim - 2))
    live = (lse != -np.inf) & ~pad
    M = np.full(lse.shape[1:], -np.inf)
    for d in range(D):
        M = np.where(live[d], np.maximum(M, lse[d]), M)
    anylive = live.any(axis=0)
    Msafe = np.where(anylive, M, 0.0)
    num = np.zeros(O_part.shape[1:])
    den = np.zeros(lse.shape[1:])
    for d in range(D):
        w = np.where(live[d], np.exp(np.where(live[d], lse[d], 0.0) - Msafe), 0.0)
        den += w
        num += np.where(live[d][..., None], w[..., None] * np.where(live[d][..., None], O_part[d], 0.0), 0.0)
    out = np.where(anylive[..., None], num / np.where(anylive, den, 1.0)[..., None], 0.0)
    out_lse = np.where(anylive, Msafe + np.log(np.where(anylive, den, 1.0)), -np.inf)
    return out, out_lse


# ---------------------------------------------------------------------------
# unsharded reference: what sharding + combine must reproduce
# ---------------------------------------------------------------------------
def attention(q_heads_f64: np.ndarray, latents: np.ndarray, scale: float):
    """Plain softmax attention of one row over all its tokens (no shards).
    Returns (out [H, 512], lse [H]); latents [L, 576] float64, L > 0."""
    s = scores(q_heads_f64, latents, scale)
    return shard_partial(s, latents[:, :LATENT])


# ---------------------------------------------------------------------------
# the step before attention: query concat and paged-cache write
# ---------------------------------------------------------------------------
def concat_cache(ql_nope: np.ndarray, q_pe: np.ndarray, kv_c: np.ndarray, k_pe: np.ndarray,
                 slot_mapping: np.ndarray, kv_cache: np.ndarray):
    """The fused decode step that precedes ``forward_mqa`` [PRHUB, snippet
    "Decode: latent multi-query attention": ``_decode_concat_cache`` builds
    the query ``[ql_nope | q_pe]`` and writes this step's ``kv_c_normed`` and
    ``k_pe`` into the paged cache at ``slot_mapping``, in one launch; the
    optional RoPE positions are None].

    Inputs are bf16 bit patterns (uint16): ql_nope [T, H, 512], q_pe
    [T, H, 64], kv_c [T, 512], k_pe [T, 64]; slot_mapping int [T] holds each
    token's cache row (block * block_size + offset), a negative value meaning
    "not written here" (a padding token, or a token another DCP rank owns);
    kv_cache [num_blocks, block_size, 576].  Returns (q [T, H, 576], the new
    cache): a byte copy, so bit-exact.
    """
    ql_nope = np.asarray(ql_nope, dtype=np.uint16)
    q_pe = np.asarray(q_pe, dtype=np.uint16)
    T, H = ql_nope.shape[:2]
    q = np.empty((T, H, KDIM), dtype=np.uint16)
    q[:, :, :LATENT] = ql_nope
    q[:, :, LATENT:] = q_pe
    cache = np.array(kv_cache, dtype=np.uint16, copy=True)
    nb, bs, _ = cache.shape
    flat = cache.reshape(nb * bs, KDIM)
    for t in range(T):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        flat[slot, :LATENT] = kv_c[t]
        flat[slot, LATENT:] = k_pe[t]
    return q, cache


# ---------------------------------------------------------------------------
# fp8 latent KV cache (per-token scale)
# ---------------------------------------------------------------------------
def fp8_e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Widen FP8 E4M3 codes (uint8: 1 sign bit, 4 exponent bits with bias 7,
    3 mantissa bits; exponent 0 is subnormal, 0x7F / 0xFF are NaN, there is no
    infinity) exactly to float64, from the format's definition: a normal code
    is (-1)^s * 2^(e - 7) * (1 + m / 8), a subnormal one (-1)^s * 2^-6 * m / 8.
    [the fp8 KV verify plans of "perf(mla): fuse K3 DCP verification
    queries", review follow-up, store latent KV in this 8-bit format]."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    out = s * mag
    return np.where((c & 0x7F) == 0x7F, np.nan, out)


def kv_rows_f64(inp: dict) -> np.ndarray:
    """All cache rows widened to float64 [num_blocks * block_size, 576]: bf16
    bits, or fp8 E4M3 codes times the slot's fp32 scale when the cache is
    fp8 (``inp["kv_dtype"] == "fp8_e4m3"``, scales in ``inp["kv_scale"]``
    [num_blocks, block_size])."""
    kv = inp["kv_cache"]
    nb, bs, kd = kv.shape
    if inp.get("kv_dtype", "bf16") == "fp8_e4m3":
        scale = np.asarray(inp["kv_scale"], dtype=np.float32).astype(np.float64).reshape(nb * bs, 1)
        return fp8_e4m3_to_f64(kv.reshape(nb * bs, kd)) * scale
    return bf16_to_f64(kv.reshape(nb * bs, kd))
