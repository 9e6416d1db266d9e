"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin
catches each one.  A pin that passes a wrong oracle pins nothing."""
import numpy as np
import pytest

from oracle import dcp_oracle as O
import workloads as wl
from tests import oracle_checks as C

pytestmark = pytest.mark.cpu


def _fails(check, *args):
    with pytest.raises((AssertionError, ValueError, IndexError)):
        check(O, *args)


def test_shard_ignoring_interleave_is_caught(monkeypatch):
    monkeypatch.setattr(O, "shard_of", lambda p, D, I: np.asarray(p, dtype=np.int64) % D)
    _fails(C.check_mapper)


def test_shard_runs_not_wrapping_is_caught(monkeypatch):
    monkeypatch.setattr(O, "shard_of", lambda p, D, I: np.minimum(np.asarray(p, dtype=np.int64) // I, D - 1))
    _fails(C.check_mapper)


def test_causal_offset_off_by_one_is_caught(monkeypatch):
    real = O.row_lengths

    def shifted(seq_lens, qsl, T):
        req, L, pad = real(seq_lens, qsl, T)
        return req, np.maximum(L - 1, 0) * (~pad), pad
    monkeypatch.setattr(O, "row_lengths", shifted)
    _fails(C.check_row_lengths)


def test_scores_without_rope_dims_are_caught(monkeypatch):
    monkeypatch.setattr(O, "scores", lambda q, kv, s: s * (np.asarray(q)[:, :512] @ np.asarray(kv)[:, :512].T))
    _fails(C.check_attention_vs_torch)


def test_log2_lse_is_caught(monkeypatch):
    def bad(s, v):
        m = s.max(axis=1, keepdims=True)
        lse = m[:, 0] + np.log2(np.exp(s - m).sum(axis=1))
        return np.exp(s - lse[:, None]) @ v, lse
    monkeypatch.setattr(O, "shard_partial", bad)
    _fails(C.check_attention_vs_torch)


def test_unnormalised_partial_is_caught(monkeypatch):
    def bad(s, v):
        m = s.max(axis=1, keepdims=True)
        lse = m[:, 0] + np.log(np.exp(s - m).sum(axis=1))
        return np.exp(s - m) @ v, lse
    monkeypatch.setattr(O, "shard_partial", bad)
    _fails(C.check_attention_closed_forms)


def test_combine_ignoring_padding_is_caught(monkeypatch):
    real = O.lse_combine
    monkeypatch.setattr(O, "lse_combine", lambda Op, lp, pad: real(Op, lp, np.zeros_like(pad)))
    _fails(C.check_combine_special_cases)


def test_combine_multiplying_by_zero_weight_is_caught(monkeypatch):
    def bad(Op, lp, pad):
        Op = np.asarray(Op, np.float64)
        lp = np.asarray(lp, np.float64)
        padb = np.asarray(pad, bool).reshape((-1,) + (1,) * (lp.ndim - 2))
        M = np.max(np.where(padb, -np.inf, lp), axis=0)
        w = np.exp(lp - np.where(np.isfinite(M), M, 0))
        out = (w[..., None] * Op).sum(0) / w.sum(0)[..., None]  # NaN * 0 leaks
        return np.where(padb[..., None], 0, out), np.where(padb, -np.inf, M + np.log(w.sum(0)))
    monkeypatch.setattr(O, "lse_combine", bad)
    _fails(C.check_combine_special_cases)


def test_transposed_block_lookup_is_caught(monkeypatch):
    def bad(table_row, bs, positions):
        positions = np.asarray(positions, dtype=np.int64)
        return np.asarray(table_row, np.int64)[positions % bs] * bs + positions // bs
    monkeypatch.setattr(O, "physical_rows", bad)
    _fails(C.check_walker)


def test_values_from_wrong_dims_are_caught(monkeypatch):
    real = O.shard_partial
    monkeypatch.setattr(O, "shard_partial", lambda s, v: real(s, np.roll(v, 64, axis=1)))
    inp = wl.make_decode_inputs(wl.TINY)
    _fails(C.check_decode_rows_vs_torch, inp)


def _concat_variant(swap=False, neg_wraps=False, drop_pe=False):
    def f(ql_nope, q_pe, kv_c, k_pe, slot_mapping, kv_cache):
        T, H = ql_nope.shape[:2]
        q = np.empty((T, H, 576), dtype=np.uint16)
        q[:, :, :512] = ql_nope
        q[:, :, 512:] = 0 if drop_pe else q_pe
        cache = np.array(kv_cache, copy=True)
        flat = cache.reshape(-1, 576)
        for t in range(T):
            s = int(slot_mapping[t])
            if s < 0 and not neg_wraps:
                continue
            row = np.concatenate([k_pe[t], kv_c[t]]) if swap else np.concatenate([kv_c[t], k_pe[t]])
            flat[s] = row
        return q, cache
    return f


def test_concat_cache_rope_first_is_caught(monkeypatch):
    monkeypatch.setattr(O, "concat_cache", _concat_variant(swap=True))
    _fails(C.check_concat_cache)


def test_concat_cache_negative_slot_written_is_caught(monkeypatch):
    monkeypatch.setattr(O, "concat_cache", _concat_variant(neg_wraps=True))
    _fails(C.check_concat_cache)


def test_concat_cache_dropped_q_pe_is_caught(monkeypatch):
    monkeypatch.setattr(O, "concat_cache", _concat_variant(drop_pe=True))
    _fails(C.check_concat_cache)


def test_local_walker_by_position_is_caught(monkeypatch):
    # a local walker that indexes the shard's table by global position
    def bad(shard_table_row, block_size, n):
        j = np.arange(int(n), dtype=np.int64) * 2
        blocks = np.asarray(shard_table_row, dtype=np.int64)[np.minimum(j // block_size, len(shard_table_row) - 1)]
        return blocks * block_size + j % block_size
    monkeypatch.setattr(O, "physical_rows_local", bad)
    _fails(C.check_local_layout_matches_global)


def test_fp8_bias_8_is_caught(monkeypatch):
    real = O.fp8_e4m3_to_f64
    monkeypatch.setattr(O, "fp8_e4m3_to_f64", lambda c: real(c) / 2.0)  # exponent bias 8 instead of 7
    _fails(C.check_fp8_widening)


def test_fp8_scale_ignored_is_caught(monkeypatch):
    def bad(inp):
        kv = inp["kv_cache"]
        nb, bs, kd = kv.shape
        if inp.get("kv_dtype", "bf16") == "fp8_e4m3":
            return O.fp8_e4m3_to_f64(kv.reshape(nb * bs, kd))
        return O.bf16_to_f64(kv.reshape(nb * bs, kd))
    monkeypatch.setattr(O, "kv_rows_f64", bad)
    _fails(C.check_fp8_decode_matches_bf16_twin)
