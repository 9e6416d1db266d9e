"""Pins for the CPU oracle: each check takes the oracle module and raises
AssertionError when the oracle disagrees with what the pages or the
mathematics fix.  The pins never re-type the oracle's own formulas: they use
brute force, closed forms, torch's float64 softmax/logsumexp, independent
scatter/gather, and special cases that reduce to textbook identities.

test_oracle_pins.py runs them against the real oracle; test_oracle_planted.py
plants plausible mistakes in the oracle and checks that a pin fails.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def page_facts() -> dict:
    out = {}
    with open(os.path.join(GOLDEN, "page_facts.txt")) as f:
        for line in f:
            line = line.split("|")[0].strip()
            if not line or line.startswith("#"):
                continue
            k, v = (s.strip() for s in line.split("="))
            out[k] = v
    return out


def _bf16(x: np.ndarray) -> np.ndarray:
    """float64 values exactly representable in bf16 (for hand-made cases)."""
    t = torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# mapper / walker / rows
# ---------------------------------------------------------------------------
def check_mapper(o):
    """Shard sets partition [0, L) and their sizes match the closed form
    n_d = floor(L / (I D)) * I + clamp(L mod (I D) - d I, 0, I)."""
    for D in (1, 2, 3, 4, 8):
        for I in (1, 2, 3, 16, 64):
            for L in list(range(0, 70)) + [127, 128, 129, 1000, 4097]:
                seen = np.zeros(L, dtype=np.int64)
                total = 0
                for d in range(D):
                    pos = o.shard_positions(L, d, D, I)
                    seen[pos] += 1
                    closed = (L // (I * D)) * I + min(max(L % (I * D) - d * I, 0), I)
                    assert len(pos) == closed == o.local_len(L, d, D, I), (D, I, L, d)
                    total += len(pos)
                assert total == L and (seen == 1).all(), (D, I, L)
    # runs of I, wrapping after D runs: position p starts a new run every I
    # tokens and the run index cycles through the shards in order
    for D, I in ((4, 1), (2, 3), (3, 2), (8, 64)):
        p = np.arange(3 * D * I)
        sh = np.asarray(o.shard_of(p, D, I))
        expect = np.concatenate([np.full(I, d) for _ in range(3) for d in range(D)])
        assert (sh == expect).all(), (D, I)


def check_tiny_empty_shard(o):
    facts = page_facts()
    L = int(facts["tiny_request0_seq_len"])
    d_empty = int(facts["tiny_request0_empty_shard"])
    lens = [o.local_len(L, d, 4, 1) for d in range(4)]
    assert lens[d_empty] == 0 and sum(lens) == L and all(n == 1 for i, n in enumerate(lens) if i != d_empty)


def check_block_alignment(o):
    """With block_size a multiple of D*I every block holds block_size/D tokens
    of each shard; with I a multiple of block_size a block lies in one shard
    (the lcm(block_size, D*I) alignment of the chunked-context workspace)."""
    for bs, D, I in ((64, 8, 1), (16, 4, 1), (64, 4, 8), (64, 8, 8)):
        for blk in range(5):
            p = np.arange(blk * bs, (blk + 1) * bs)
            counts = np.bincount(np.asarray(o.shard_of(p, D, I)), minlength=D)
            assert (counts == bs // D).all(), (bs, D, I, blk)
    for bs, D, I in ((64, 8, 64), (16, 4, 32)):
        for blk in range(40):
            p = np.arange(blk * bs, (blk + 1) * bs)
            sh = np.unique(np.asarray(o.shard_of(p, D, I)))
            assert len(sh) == 1 and sh[0] == (blk * bs // I) % D


def check_walker(o):
    """Scatter a logical latent sequence into permuted blocks (independently)
    and gather it back through the block table."""
    rng = np.random.default_rng(7)
    for bs in (1, 16, 64):
        L = 5 * bs + 3
        nblk = (L + bs - 1) // bs
        nb_total = nblk + 4
        perm = rng.permutation(nb_total)[:nblk]
        table = np.concatenate([perm, np.full(3, -1)]).astype(np.int32)
        logical = rng.standard_normal((L, 576)).astype(np.float32)
        bits = _bf16(logical)
        cache = np.zeros((nb_total, bs, 576), dtype=np.uint16)
        for t in range(L):
            cache[perm[t // bs], t % bs] = bits[t]
        pos = np.arange(L)
        got = o.gather_latents(cache, table, bs, pos)
        want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
        assert np.array_equal(got, want)
        sub = pos[rng.permutation(L)[:17]]
        assert np.array_equal(o.gather_latents(cache, table, bs, sub), want[sub])


def check_row_lengths(o):
    """Padding rows follow repeating (seq_len == 0) once per query row of each
    request (numpy's repeat), rows past the last request are padding, and row i
    of a q_len-row request sees seq_len - (q_len - 1 - i) tokens."""
    seq = np.array([5, 0, 7, 0, 2, 9], dtype=np.int32)
    ql = np.array([1, 2, 1, 3, 4, 4], dtype=np.int32)
    qsl = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    T = int(qsl[-1]) + 2
    req, L, pad = o.row_lengths(seq, qsl, T)
    expect_pad = np.concatenate([np.repeat(seq == 0, ql), [True, True]])
    assert (pad == expect_pad).all()
    assert list(req) == [0, 1, 1, 2, 3, 3, 3, 4, 4, 4, 4, 5, 5, 5, 5, -1, -1]
    # request 4: seq 2, q_len 4 -> rows see 2-3, 2-2, 2-1, 2 tokens, clamped at 0
    assert list(L[7:11]) == [0, 0, 1, 2]
    assert list(L[11:15]) == [6, 7, 8, 9]
    assert L[0] == 5 and L[5] == 0 and L[3] == 7


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------
def _torch_attention(q: np.ndarray, kv: np.ndarray, scale: float):
    qt, kt = torch.from_numpy(q), torch.from_numpy(kv)
    s = scale * (qt @ kt.T)
    return (torch.softmax(s, dim=-1) @ kt[:, :512]).numpy(), torch.logsumexp(s, dim=-1).numpy()


def check_attention_closed_forms(o):
    rng = np.random.default_rng(11)
    H = 3
    q = rng.standard_normal((H, 576))
    kv = rng.standard_normal((5, 576))
    sc = 0.3
    # one token: output is that token's value row, lse is its score
    out, lse = o.attention(q, kv[:1], sc)
    s0 = sc * np.array([math.fsum(q[h] * kv[0]) for h in range(H)])
    assert np.allclose(out, np.broadcast_to(kv[0, :512], (H, 512)), rtol=0, atol=1e-14)
    assert np.allclose(lse, s0, rtol=0, atol=1e-12)
    # zero query: uniform weights -> mean of values, lse = ln L
    out, lse = o.attention(np.zeros((H, 576)), kv, sc)
    assert np.allclose(out, np.broadcast_to(kv[:, :512].mean(0), (H, 512)), atol=1e-14)
    assert np.allclose(lse, math.log(5), atol=1e-14)
    # two tokens: weights are logistic functions of the score difference
    out, lse = o.attention(q, kv[:2], sc)
    for h in range(H):
        a = sc * math.fsum(q[h] * kv[0])
        b = sc * math.fsum(q[h] * kv[1])
        w0 = 1.0 / (1.0 + math.exp(b - a))
        assert np.allclose(out[h], w0 * kv[0, :512] + (1 - w0) * kv[1, :512], atol=1e-13)
        assert abs(lse[h] - (max(a, b) + math.log1p(math.exp(-abs(a - b))))) < 1e-12
    # the rope dims take part in the score, not in the value
    kv2 = kv.copy()
    kv2[:, 512:] = 0.0
    q2 = q.copy()
    q2[:, 512:] = 0.0
    out_a, lse_a = o.attention(q2, kv, sc)
    out_b, lse_b = o.attention(q2, kv2, sc)
    assert np.allclose(out_a, out_b, atol=1e-14) and np.allclose(lse_a, lse_b, atol=1e-14)


def check_attention_vs_torch(o):
    rng = np.random.default_rng(12)
    for H, L in ((1, 1), (4, 7), (16, 37), (8, 300)):
        q = rng.standard_normal((H, 576))
        kv = rng.standard_normal((L, 576))
        out, lse = o.attention(q, kv, 1 / math.sqrt(192))
        ref_out, ref_lse = _torch_attention(q, kv, 1 / math.sqrt(192))
        assert np.allclose(out, ref_out, rtol=0, atol=1e-12), (H, L)
        assert np.allclose(lse, ref_lse, rtol=0, atol=1e-12), (H, L)


def _logical_latents(inp, b, L):
    """Request b's first L latent rows, gathered with torch indexing (not the
    oracle's walker)."""
    bs = inp["block_size"]
    cache = torch.from_numpy(inp["kv_cache"].view(np.int16)).view(torch.bfloat16)
    flat = cache.reshape(-1, 576)
    table = torch.from_numpy(inp["block_table"][b].astype(np.int64))
    p = torch.arange(L)
    return flat[table[p // bs] * bs + p % bs].double().numpy()


def check_decode_rows_vs_torch(o, inp, rows=None):
    """Per row, per shard: the oracle's partials equal torch softmax attention
    over the shard's positions (chosen by a plain Python loop over the
    round-robin runs), and the combine equals unsharded attention."""
    D, I, sc = inp["D"], inp["interleave"], inp["scale"]
    qsl, seq = inp["query_start_loc"], inp["seq_lens"]
    O, lse, rows = o.decode_partial(inp, rows)
    req, Lr, pad = o.row_lengths(seq, qsl, inp["T"])
    out, out_lse = o.lse_combine(O, lse, pad[rows])
    for j, r in enumerate(rows):
        b = int(req[r])
        qh = torch.from_numpy(inp["q"][r].view(np.int16)).view(torch.bfloat16).double().numpy()
        if pad[r] or Lr[r] == 0:
            assert (lse[:, j] == -np.inf).all()
            assert (out[j] == 0).all() and (out_lse[j] == -np.inf).all()
            continue
        L = int(Lr[r])
        kv = _logical_latents(inp, b, L)
        for d in range(D):
            pos = [p for p in range(L) if (p // I) % D == d]
            if not pos:
                assert (lse[d, j] == -np.inf).all() and np.isnan(O[d, j]).all()
                continue
            ro, rl = _torch_attention(qh, kv[pos], sc)
            assert np.allclose(O[d, j], ro, rtol=0, atol=1e-12), (r, d)
            assert np.allclose(lse[d, j], rl, rtol=0, atol=1e-12), (r, d)
        ro, rl = _torch_attention(qh, kv, sc)
        assert np.allclose(out[j], ro, rtol=0, atol=1e-12), r
        assert np.allclose(out_lse[j], rl, rtol=0, atol=1e-12), r


# ---------------------------------------------------------------------------
# combine
# ---------------------------------------------------------------------------
def check_combine_special_cases(o):
    rng = np.random.default_rng(13)
    R, H = 5, 3
    pad = np.zeros(R, dtype=bool)
    # D = 1: identity
    O1 = rng.standard_normal((1, R, H, 512))
    l1 = rng.standard_normal((1, R, H))
    out, ol = o.lse_combine(O1, l1, pad)
    assert np.array_equal(ol, l1[0]) and np.allclose(out, O1[0], rtol=0, atol=1e-15)
    # D = 2: the two-way merge weights are logistic functions of lse_0 - lse_1
    O2 = rng.standard_normal((2, R, H, 512))
    l2 = 3 * rng.standard_normal((2, R, H))
    out, ol = o.lse_combine(O2, l2, pad)
    w0 = 1.0 / (1.0 + np.exp(l2[1] - l2[0]))
    assert np.allclose(out, w0[..., None] * O2[0] + (1 - w0[..., None]) * O2[1], atol=1e-13)
    assert np.allclose(ol, np.logaddexp(l2[0], l2[1]), atol=1e-13)
    # the pages' base-2 weighting gives the same result
    log2e = 1.0 / math.log(2.0)
    M2 = np.maximum(l2[0], l2[1]) * log2e
    w = [np.exp2(l2[d] * log2e - M2) for d in range(2)]
    ref = (w[0][..., None] * O2[0] + w[1][..., None] * O2[1]) / (w[0] + w[1])[..., None]
    assert np.allclose(out, ref, atol=1e-13)
    # exactly one live shard: that shard, weight one; the others may hold NaN
    D = 4
    O4 = rng.standard_normal((D, R, H, 512))
    l4 = rng.standard_normal((D, R, H))
    l4[[0, 1, 3]] = -np.inf
    O4[[0, 1, 3]] = np.nan
    out, ol = o.lse_combine(O4, l4, pad)
    assert np.array_equal(out, O4[2]) and np.array_equal(ol, l4[2])
    # equal LSEs: plain mean, lse + ln D
    O4 = rng.standard_normal((D, R, H, 512))
    l4 = np.full((D, R, H), 1.25)
    out, ol = o.lse_combine(O4, l4, pad)
    assert np.allclose(out, O4.mean(0), atol=1e-14) and np.allclose(ol, 1.25 + math.log(D), atol=1e-14)
    # padding rows: zeros and -inf whatever the LSEs and payloads hold
    pad2 = np.array([False, True, False, True, False])
    O4[:, pad2] = np.nan
    l4 = rng.standard_normal((D, R, H))
    out, ol = o.lse_combine(O4, l4, pad2)
    assert (out[pad2] == 0).all() and (ol[pad2] == -np.inf).all()
    assert np.isfinite(out[~pad2]).all() and np.isfinite(ol[~pad2]).all()
    # every shard empty on a live row: zeros and -inf, no NaN
    l4[:, 0] = -np.inf
    O4[:, 0] = np.nan
    out, ol = o.lse_combine(O4, l4, pad2)
    assert (out[0] == 0).all() and (ol[0] == -np.inf).all()


def check_combine_permutation(o):
    rng = np.random.default_rng(14)
    D, R, H = 8, 6, 4
    O = rng.standard_normal((D, R, H, 512))
    l = 5 + 3 * rng.standard_normal((D, R, H))
    empty = rng.random((D, R, H)) < 0.2
    l[empty] = -np.inf
    O[np.broadcast_to(empty[..., None], O.shape)] = np.nan
    pad = np.zeros(R, dtype=bool)
    base, bl = o.lse_combine(O, l, pad)
    for _ in range(4):
        p = rng.permutation(D)
        out, ol = o.lse_combine(O[p], l[p], pad)
        assert np.allclose(out, base, rtol=1e-12, atol=1e-12)
        assert np.allclose(ol, bl, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# the step before attention: query concat + paged-cache write
# ---------------------------------------------------------------------------
def concat_cache_case(seed: int = 7, T: int = 6, H: int = 3, nb: int = 5, bs: int = 4):
    """Small random bf16 inputs for concat_cache: slots include a padding
    token (-1) and tokens scattered over permuted blocks."""
    rng = np.random.default_rng(seed)
    bits = lambda *shape: rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[1] = -1
    return dict(ql_nope=bits(T, H, 512), q_pe=bits(T, H, 64), kv_c=bits(T, 512), k_pe=bits(T, 64),
                slot_mapping=slots, kv_cache=bits(nb, bs, 576))


def check_concat_cache(o):
    """The query is torch.cat of the two parts; the cache equals the old cache
    with exactly the rows of non-negative slots replaced by torch.cat of the
    latent and rope parts (torch index_copy_), every other byte unchanged."""
    c = concat_cache_case()
    q, cache = o.concat_cache(c["ql_nope"], c["q_pe"], c["kv_c"], c["k_pe"], c["slot_mapping"], c["kv_cache"])
    tq = lambda a: torch.from_numpy(np.asarray(a).astype(np.int32))
    want_q = torch.cat([tq(c["ql_nope"]), tq(c["q_pe"])], dim=-1).numpy().astype(np.uint16)
    assert q.shape == want_q.shape and np.array_equal(q, want_q)
    nb, bs, _ = c["kv_cache"].shape
    keep = c["slot_mapping"] >= 0
    idx = torch.from_numpy(c["slot_mapping"][keep])
    rows = torch.cat([tq(c["kv_c"]), tq(c["k_pe"])], dim=-1)[torch.from_numpy(keep)]
    want = tq(c["kv_cache"]).reshape(nb * bs, 576).index_copy_(0, idx, rows)
    assert np.array_equal(cache.reshape(nb * bs, 576), want.numpy().astype(np.uint16))
    # the input cache is not modified in place
    assert not np.shares_memory(cache, c["kv_cache"])


def check_concat_cache_feeds_the_walker(o):
    """A token written at the slot of logical position p of a request (its
    block-table entry) is what the block-table walker reads back at p."""
    rng = np.random.default_rng(11)
    nb, bs, L = 6, 4, 13
    table = rng.permutation(nb).astype(np.int64)
    cache = np.zeros((nb, bs, 576), dtype=np.uint16)
    kv_c = rng.integers(0, 0x7000, size=(1, 512), dtype=np.uint16)  # finite bf16 patterns
    k_pe = rng.integers(0, 0x7000, size=(1, 64), dtype=np.uint16)
    slot = np.array([table[L // bs] * bs + L % bs])
    _, cache = o.concat_cache(np.zeros((1, 1, 512), np.uint16), np.zeros((1, 1, 64), np.uint16), kv_c, k_pe,
                              slot, cache)
    got = o.gather_latents(cache, table, bs, np.array([L]))
    want = o.bf16_to_f64(np.concatenate([kv_c, k_pe], axis=-1))
    assert np.array_equal(got, want)


# ---------------------------------------------------------------------------
# per-shard (rank-local) block tables and shared prefixes
# ---------------------------------------------------------------------------
LAYOUT_CASES = [
    dict(B=2, seq_lens=(300, 77), H=4, block_size=16, D=4, interleave=3),
    dict(B=3, seq_lens=(130, 1, 64), q_len=2, H=2, block_size=8, D=2, interleave=4, extra_rows=1),
    dict(B=2, seq_lens=(200, 150), H=2, block_size=16, D=8, interleave=1, prefix_len=100, shared_prefix=True),
]


def check_local_layout_matches_global(o):
    """The same logical context stored in the per-shard layout or in the
    global layout gives the same partials: the local walker reads exactly the
    positions each shard owns, in the same order as the global one."""
    import workloads as wl
    for i, kw in enumerate(LAYOUT_CASES):
        g = wl.make_decode_inputs(wl.DecodeSpec("g%d" % i, seed=80 + i, layout="global", **kw))
        l = wl.make_decode_inputs(wl.DecodeSpec("l%d" % i, seed=80 + i, layout="local", **kw))
        assert l["block_table"].shape[:2] == (kw["D"], kw["B"])
        Og, lg, _ = o.decode_partial(g)
        Ol, ll, _ = o.decode_partial(l)
        assert np.array_equal(lg, ll), i
        assert np.array_equal(np.isnan(Og), np.isnan(Ol)), i
        live = ~np.isnan(Og)
        assert np.array_equal(Og[live], Ol[live]), i


def check_shared_prefix(o):
    """Two requests sharing a prefix: the prefix tokens are the same values in
    both, the blocks that hold only prefix tokens are the same blocks, and
    shard partials over a context of exactly the prefix agree between them."""
    import workloads as wl
    spec = wl.DecodeSpec("sp", seed=90, B=2, seq_lens=(200, 150), H=3, block_size=16, D=4, interleave=1,
                         prefix_len=96, shared_prefix=True, q_len=1)
    inp = wl.make_decode_inputs(spec)
    t = inp["block_table"]
    assert np.array_equal(t[0, :6], t[1, :6]) and not np.intersect1d(t[0, 6:13], t[1, 6:10]).size
    pos = np.arange(96)
    a = o.gather_latents(inp["kv_cache"], t[0], 16, pos)
    b = o.gather_latents(inp["kv_cache"], t[1], 16, pos)
    assert np.array_equal(a, b)
    # the suffixes differ
    assert not np.array_equal(o.gather_latents(inp["kv_cache"], t[0], 16, np.arange(96, 150)),
                              o.gather_latents(inp["kv_cache"], t[1], 16, np.arange(96, 150)))


# ---------------------------------------------------------------------------
# fp8 latent KV
# ---------------------------------------------------------------------------
def fp8_table() -> dict:
    out = {}
    with open(os.path.join(GOLDEN, "fp8_e4m3_table.txt")) as f:
        for line in f:
            line = line.split("|")[0].strip()
            if not line or line.startswith("#"):
                continue
            k, v = (x.strip() for x in line.split("="))
            out[int(k, 16)] = float(v)
    return out


def check_fp8_widening(o):
    """The hand-decoded E4M3 table, and every one of the 256 codes against
    torch's float8_e4m3fn -> float conversion (NaN codes alike)."""
    tab = fp8_table()
    codes = np.array(sorted(tab), dtype=np.uint8)
    got = o.fp8_e4m3_to_f64(codes)
    want = np.array([tab[c] for c in sorted(tab)])
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok]) and np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))
    allc = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(allc).view(torch.float8_e4m3fn).double().numpy()
    g = o.fp8_e4m3_to_f64(allc)
    assert np.array_equal(np.isnan(g), np.isnan(ref))
    assert np.array_equal(g[~np.isnan(g)], ref[~np.isnan(ref)])


def check_fp8_decode_matches_bf16_twin(o):
    """An fp8 cache with power-of-two per-token scales holds values that bf16
    represents exactly; the oracle's decode over the fp8 cache equals its
    decode over the bf16 cache of the same values (the fp8 path changes only
    the storage)."""
    import workloads as wl
    spec = wl.DecodeSpec("f8", seed=131, B=3, seq_lens=(70, 5, 0), q_len=2, H=3, block_size=16, D=4, interleave=2,
                         kv_dtype="fp8_e4m3")
    f = wl.make_decode_inputs(spec)
    # the twin's values come from torch's own E4M3 conversion times the stored
    # per-slot scale, independently of the oracle's widening
    nb, bs, kd = f["kv_cache"].shape
    codes = torch.from_numpy(f["kv_cache"].reshape(nb * bs, kd)).view(torch.float8_e4m3fn).double()
    vals = (codes * torch.from_numpy(f["kv_scale"].reshape(nb * bs, 1)).double()).numpy()
    live = ~np.isnan(vals).any(axis=1)
    t32 = torch.from_numpy(vals[live].astype(np.float32))
    assert torch.equal(t32.to(torch.bfloat16).float(), t32)  # exact in bf16
    bits = np.full(vals.shape, 0x7FC0, dtype=np.uint16)
    bits[live] = t32.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    twin = dict(f, kv_dtype="bf16", kv_cache=bits.reshape(f["kv_cache"].shape), kv_scale=None)
    Of, lf, _ = o.decode_partial(f)
    Ob, lb, _ = o.decode_partial(twin)
    assert np.array_equal(lf, lb)
    m = ~np.isnan(Ob)
    assert np.array_equal(np.isnan(Of), ~m) and np.array_equal(Of[m], Ob[m])
