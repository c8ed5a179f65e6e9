"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each pin takes an `oracle.Oracle` instance and raises AssertionError when the oracle disagrees with
  * a library routine (torch.nn.functional.scaled_dot_product_attention in float64, numpy fancy
    indexing for the scatter and the gather),
  * a closed form (one key, zero query, equal keys, a dominant logit, the hand-derived three-block
    example under tests/golden/),
  * an invariant of paging (block placement, block sharing, block size, padding).
The same pins run against deliberately mutated copies of the oracle (test_oracle_mutants.py) to show
that a plausible mistake anywhere in it is caught.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
TOL = 1e-12


def _f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def _close(a, b, tol=TOL, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    assert np.all(np.isfinite(a)), f"{what}: non-finite oracle output"
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol:.1e}"


def sdpa(q, k, v, scale, mask=None, causal=False):
    """torch SDPA in float64. q [Hq, Lq, D], k/v [Hkv, Lk, D]; GQA by contiguous head groups."""
    G = q.shape[0] // k.shape[0]
    qt = torch.from_numpy(np.ascontiguousarray(q))[None]
    kt = torch.from_numpy(np.ascontiguousarray(k)).repeat_interleave(G, dim=0)[None]
    vt = torch.from_numpy(np.ascontiguousarray(v)).repeat_interleave(G, dim=0)[None]
    m = None if mask is None else torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m,
                                                         is_causal=causal, scale=scale)
    return o[0].numpy()


def contiguous_kv(case: W.DecodeCase, kc, vc, b):
    """Sequence b's K, V [ctx, Hkv, D] as float64, read with numpy indexing (no oracle code)."""
    ctx = int(case.context_lens[b])
    pos = np.arange(ctx)
    rows = case.block_tables[b, pos // case.block_size].astype(np.int64) * case.block_size \
        + pos % case.block_size
    K = _f64(kc.reshape(-1, case.num_kv_heads, case.head_dim)[rows])
    V = _f64(vc.reshape(-1, case.num_kv_heads, case.head_dim)[rows])
    return K, V


def numpy_store(case: W.DecodeCase):
    """The scatter with numpy fancy indexing: the library reading of 'write row t at slot[t]'."""
    kc = case.k_cache.copy()
    vc = case.v_cache.copy()
    sm = case.slot_mapping
    ok = sm >= 0
    flat_k = kc.reshape(-1, case.num_kv_heads, case.head_dim)
    flat_v = vc.reshape(-1, case.num_kv_heads, case.head_dim)
    flat_k[sm[ok]] = case.k_new[ok]
    flat_v[sm[ok]] = case.v_new[ok]
    return kc, vc


# ------------------------------------------------------------------------------------------------
# KV store
# ------------------------------------------------------------------------------------------------


def pin_store_matches_numpy_scatter(orc):
    for seed in range(3):
        case = W.tiny_decode_case(seed=seed + 1)
        kc, vc, bad = orc.kv_store(case.k_new, case.v_new, case.slot_mapping, case.k_cache,
                                   case.v_cache)
        rk, rv = numpy_store(case)
        assert bad == 0
        assert np.array_equal(kc, rk) and np.array_equal(vc, rv), "store differs from scatter"


def pin_store_padding_and_invalid(orc):
    rng = W.rng_for(7, 0)
    NB, BS, Hkv, D = 6, 4, 2, 8
    sentinel = np.full((NB, BS, Hkv, D), 0x7FC1, dtype=np.uint16)
    slots = np.array([-1, 5, -1, 0, 23, -2, 24, 7, -1], dtype=np.int32)
    T = len(slots)
    k = W.normal_bf16(rng, (T, Hkv, D))
    v = W.normal_bf16(rng, (T, Hkv, D))
    kc, vc, bad = orc.kv_store(k, v, slots, sentinel, sentinel)
    assert bad == 2, f"expected 2 invalid slots (-2 and 24), got {bad}"
    changed = np.any(kc.reshape(NB * BS, -1) != 0x7FC1, axis=1)
    assert set(np.nonzero(changed)[0]) == {5, 0, 23, 7}, "padding or invalid slot wrote a row"
    for t, s in enumerate(slots):
        if 0 <= s < NB * BS:
            assert np.array_equal(kc[s // BS, s % BS], k[t]), "K row not at (slot/BS, slot%BS)"
            assert np.array_equal(vc[s // BS, s % BS], v[t]), "V row not at (slot/BS, slot%BS)"


def pin_store_round_trip(orc):
    case = W.random_decode_case(11, 5, 4, 2, 32, 8, 1, 40, pad_slots=3)
    kc, vc, _ = orc.kv_store(case.k_new, case.v_new, case.slot_mapping, case.k_cache, case.v_cache)
    sm = case.slot_mapping
    ok = sm >= 0
    back_k = kc.reshape(-1, case.num_kv_heads, case.head_dim)[sm[ok]]
    back_v = vc.reshape(-1, case.num_kv_heads, case.head_dim)[sm[ok]]
    assert np.array_equal(back_k, case.k_new[ok]) and np.array_equal(back_v, case.v_new[ok])
    n_changed = int(np.sum(np.any((kc != case.k_cache).reshape(-1, case.num_kv_heads *
                                                                  case.head_dim), axis=1)))
    assert n_changed <= int(ok.sum())


# ------------------------------------------------------------------------------------------------
# Block-table walk
# ------------------------------------------------------------------------------------------------


def pin_gather_identity_and_permuted(orc):
    rng = W.rng_for(3, 0)
    BS, Hkv, D, ctx = 4, 3, 8, 13
    nb = 4
    logical = W.normal_bf16(rng, (nb * BS, Hkv, D))
    perm = rng.permutation(nb).astype(np.int32)
    cache = np.zeros((nb, BS, Hkv, D), dtype=np.uint16)
    for i, p in enumerate(perm):
        cache[p] = logical[i * BS:(i + 1) * BS]
    for g in range(Hkv):
        got = orc.gather_head(cache, perm, ctx, g)
        _close(got, _f64(logical[:ctx, g]), 0.0, "gather through a permuted table")
        ident = orc.gather_head(logical.reshape(nb, BS, Hkv, D), np.arange(nb, dtype=np.int32),
                                ctx, g)
        _close(ident, _f64(logical[:ctx, g]), 0.0, "gather through the identity table")


# ------------------------------------------------------------------------------------------------
# Decode
# ------------------------------------------------------------------------------------------------

DECODE_SHAPES = [  # (B, Hq, Hkv, D, BS, ctx_lo, ctx_hi)
    (4, 4, 2, 64, 16, 1, 64),
    (3, 8, 2, 16, 4, 1, 21),
    (2, 2, 2, 8, 8, 7, 17),
    (3, 6, 1, 32, 16, 15, 33),
]


def _stored_decode_case(shape, seed, q_scale=1.0):
    B, Hq, Hkv, D, BS, lo, hi = shape
    case = W.random_decode_case(seed, B, Hq, Hkv, D, BS, lo, hi, extra_pool=2, q_scale=q_scale)
    kc, vc = numpy_store(case)
    return case, kc, vc


def pin_decode_matches_sdpa(orc):
    for i, shape in enumerate(DECODE_SHAPES):
        for q_scale in (1.0, 8.0):
            case, kc, vc = _stored_decode_case(shape, 100 + i, q_scale)
            out = orc.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens,
                                   case.scale)
            for b in range(case.num_seqs):
                K, V = contiguous_kv(case, kc, vc, b)
                ref = sdpa(_f64(case.q[b])[:, None, :], K.transpose(1, 0, 2),
                           V.transpose(1, 0, 2), case.scale)[:, 0, :]
                _close(out[b], ref, TOL, f"decode vs SDPA shape={shape} q_scale={q_scale}")


def _single_seq_case(K, V, q, BS, scale, rng, Hkv=1):
    """Place one sequence's rows [ctx, Hkv, D] into shuffled blocks; return decode inputs."""
    ctx = K.shape[0]
    nb = max(1, -(-ctx // BS))
    perm = rng.permutation(nb + 2).astype(np.int32)[:nb]
    D = K.shape[-1]
    kc = np.zeros((nb + 2, BS, Hkv, D), dtype=np.uint16)
    vc = np.zeros_like(kc)
    for p in range(ctx):
        kc[perm[p // BS], p % BS] = K[p]
        vc[perm[p // BS], p % BS] = V[p]
    return q[None], kc, vc, perm[None], np.array([ctx], dtype=np.int32), scale


def pin_decode_closed_forms(orc):
    rng = W.rng_for(5, 0)
    D, BS = 16, 4
    # one key: the output is that key's value row, exactly
    K = W.normal_bf16(rng, (1, 1, D))
    V = W.normal_bf16(rng, (1, 1, D))
    q = W.normal_bf16(rng, (1, D))
    out = orc.paged_decode(*_single_seq_case(K, V, q, BS, 0.25, rng))
    _close(out[0, 0], _f64(V[0, 0]), 0.0, "ctx=1 gives V0")
    # zero query: uniform weights, the output is the mean of the value rows
    ctx = 11
    K = W.normal_bf16(rng, (ctx, 1, D))
    V = W.normal_bf16(rng, (ctx, 1, D))
    zq = np.zeros((1, D), dtype=np.uint16)
    out = orc.paged_decode(*_single_seq_case(K, V, zq, BS, 0.3, rng))
    _close(out[0, 0], _f64(V[:, 0]).mean(axis=0), TOL, "q=0 gives mean V")
    # identical keys: uniform weights again, whatever the query
    Keq = np.repeat(K[:1], ctx, axis=0)
    out = orc.paged_decode(*_single_seq_case(Keq, V, q, BS, 0.3, rng))
    _close(out[0, 0], _f64(V[:, 0]).mean(axis=0), TOL, "equal keys give mean V")
    # one dominant logit (margin 40 after scaling): the output is that value row
    Kd = np.zeros((ctx, 1, D), dtype=np.uint16)
    qd = np.zeros((1, D), dtype=np.uint16)
    qd[0, 0] = W.f32_to_bf16_bits(np.array([1.0], dtype=np.float32))[0]
    Kd[6, 0, 0] = W.f32_to_bf16_bits(np.array([40.0], dtype=np.float32))[0]
    out = orc.paged_decode(*_single_seq_case(Kd, V, qd, BS, 1.0, rng))
    _close(out[0, 0], _f64(V[6, 0]), 1e-12, "dominant logit selects its V row")
    # weights e^0 and e^1 on two keys: out = (v0 + e v1) / (1 + e)
    K2 = np.zeros((2, 1, D), dtype=np.uint16)
    K2[1, 0, 0] = W.f32_to_bf16_bits(np.array([1.0], dtype=np.float32))[0]
    out = orc.paged_decode(*_single_seq_case(K2, V[:2], qd, BS, 1.0, rng))
    want = (_f64(V[0, 0]) + math.e * _f64(V[1, 0])) / (1.0 + math.e)
    _close(out[0, 0], want, TOL, "two keys, logits 0 and 1")


def pin_decode_golden_three_blocks(orc):
    with open(os.path.join(GOLDEN, "three_block_decode.json")) as f:
        g = json.load(f)
    BS, NB, D = g["block_size"], g["num_blocks"], g["head_dim"]
    keys = np.array(g["keys"], dtype=np.float32)
    vals = np.array(g["values"], dtype=np.float32)
    kc = np.full((NB, BS, 1, D), W.f32_to_bf16_bits(np.array([99.0], np.float32))[0], np.uint16)
    vc = kc.copy()
    for p in range(g["context_len"]):
        blk = g["block_table"][p // BS]
        kc[blk, p % BS, 0] = W.f32_to_bf16_bits(keys[p])
        vc[blk, p % BS, 0] = W.f32_to_bf16_bits(vals[p])
    q = W.f32_to_bf16_bits(np.array(g["q"], dtype=np.float32))[None, None, :]
    out = orc.paged_decode(q, kc, vc, np.array([g["block_table"]], np.int32),
                           np.array([g["context_len"]], np.int32), g["scale"])
    e = math.e
    den = [c0 + c1 * e + c2 * e * e for c0, c1, c2 in [g["expected_denominator_coefficients"]]][0]
    want = [(a + b * e + c * e * e) / den for a, b, c in g["expected_numerator_coefficients"]]
    _close(out[0, 0], want, TOL, "three-block worked example")


def pin_decode_placement_invariance(orc):
    """Permuting physical block placement (and the tables with it) leaves outputs unchanged."""
    case, kc, vc = _stored_decode_case((3, 4, 2, 32, 8, 5, 40), 21)
    out = orc.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, case.scale)
    rng = W.rng_for(21, 9)
    perm = rng.permutation(case.num_blocks)
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(case.block_tables >= 0, perm[np.maximum(case.block_tables, 0)], -1)
    out2 = orc.paged_decode(case.q, kc2, vc2, bt2.astype(np.int32), case.context_lens, case.scale)
    assert np.array_equal(out, out2), "block placement changed the result"


def pin_decode_shared_vs_duplicated(orc):
    """Two sequences reading the same physical blocks equal two sequences reading copies."""
    rng = W.rng_for(22, 0)
    BS, Hkv, D, ctx = 8, 2, 16, 29
    nb = -(-ctx // BS)
    kc = W.normal_bf16(rng, (2 * nb, BS, Hkv, D))
    vc = W.normal_bf16(rng, (2 * nb, BS, Hkv, D))
    kc[nb:] = kc[:nb]
    vc[nb:] = vc[:nb]
    q = W.normal_bf16(rng, (2, 4, D))
    cl = np.array([ctx, ctx], np.int32)
    shared = np.array([np.arange(nb), np.arange(nb)], np.int32)
    dup = np.array([np.arange(nb), np.arange(nb, 2 * nb)], np.int32)
    o1 = orc.paged_decode(q, kc, vc, shared, cl, 0.25)
    o2 = orc.paged_decode(q, kc, vc, dup, cl, 0.25)
    assert np.array_equal(o1, o2), "shared and duplicated blocks differ"


def pin_decode_block_size_invariance(orc):
    """The same logical K/V laid out with block size 4 and 16 gives the same output."""
    rng = W.rng_for(23, 0)
    Hkv, D, ctx = 2, 16, 37
    K = W.normal_bf16(rng, (ctx, Hkv, D))
    V = W.normal_bf16(rng, (ctx, Hkv, D))
    q = W.normal_bf16(rng, (4, D))
    outs = []
    for BS in (4, 16):
        args = _single_seq_case(K, V, q, BS, 0.2, W.rng_for(BS, 1), Hkv=Hkv)
        outs.append(orc.paged_decode(*args))
    assert np.array_equal(outs[0], outs[1]), "block size changed the result"


def pin_decode_zero_context(orc):
    case, kc, vc = _stored_decode_case((3, 4, 2, 16, 8, 3, 9), 24)
    cl = case.context_lens.copy()
    cl[1] = 0
    out = orc.paged_decode(case.q, kc, vc, case.block_tables, cl, case.scale)
    assert np.all(out[1] == 0.0), "context 0 must give zeros"
    full = orc.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, case.scale)
    assert np.array_equal(out[[0, 2]], full[[0, 2]])


# ------------------------------------------------------------------------------------------------
# Prefill
# ------------------------------------------------------------------------------------------------


def _prefill_keys(case: W.PrefillCase, b):
    """Sequence b's keys/values [k_len, Hkv, D] float64: prefix via numpy indexing, then new rows."""
    P = int(case.k_lens[b] - case.q_lens[b])
    pos = np.arange(P)
    rows = case.block_tables[b, pos // case.block_size].astype(np.int64) * case.block_size \
        + pos % case.block_size
    kp = case.k_cache.reshape(-1, case.num_kv_heads, case.head_dim)[rows]
    vp = case.v_cache.reshape(-1, case.num_kv_heads, case.head_dim)[rows]
    r0, r1 = case.cu_seqlens_q[b], case.cu_seqlens_q[b + 1]
    K = _f64(np.concatenate([kp, case.k[r0:r1]]))
    V = _f64(np.concatenate([vp, case.v[r0:r1]]))
    return K, V, P


def pin_prefill_no_prefix_matches_causal_sdpa(orc):
    for q_scale in (1.0, 8.0):
        rng = W.rng_for(31, 0)
        Hq, Hkv, D = 4, 2, 16
        ql = np.array([1, 7, 19, 33], np.int32)
        T = int(ql.sum())
        cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
        q = W.normal_bf16(rng, (T, Hq, D), q_scale)
        k = W.normal_bf16(rng, (T, Hkv, D))
        v = W.normal_bf16(rng, (T, Hkv, D))
        empty = np.zeros((1, 16, Hkv, D), np.uint16)
        out = orc.paged_prefill(q, k, v, cu, cu, None, empty, empty, 0.25)
        for b in range(len(ql)):
            r = slice(cu[b], cu[b + 1])
            ref = sdpa(_f64(q[r]).transpose(1, 0, 2), _f64(k[r]).transpose(1, 0, 2),
                       _f64(v[r]).transpose(1, 0, 2), 0.25, causal=True)
            _close(out[r], ref.transpose(1, 0, 2), TOL, "prefill vs causal SDPA")


def pin_prefill_prefix_matches_masked_sdpa(orc):
    for q_scale in (1.0, 8.0):
        case = W.prefix_prefill_case(32, 3, 16, 1, 21, 4, 2, 16, 8, q_scale=q_scale,
                                     suffix_lens=np.array([1, 9, 21]))
        out = orc.paged_prefill(case.q, case.k, case.v, case.cu_seqlens_q, case.cu_seqlens_k,
                                case.block_tables, case.k_cache, case.v_cache, case.scale)
        for b in range(case.num_seqs):
            K, V, P = _prefill_keys(case, b)
            qlen = int(case.q_lens[b])
            mask = np.tril(np.ones((qlen, qlen + P), dtype=bool), k=P)
            r = slice(case.cu_seqlens_q[b], case.cu_seqlens_q[b + 1])
            ref = sdpa(_f64(case.q[r]).transpose(1, 0, 2), K.transpose(1, 0, 2),
                       V.transpose(1, 0, 2), case.scale, mask=mask)
            _close(out[r], ref.transpose(1, 0, 2), TOL, "prefix prefill vs masked SDPA")


def pin_prefill_row_equals_decode(orc):
    """Prefill query i equals decode over the first P + i + 1 keys once the new rows are stored."""
    case = W.prefix_prefill_case(33, 2, 16, 3, 12, 4, 2, 16, 8)
    out = orc.paged_prefill(case.q, case.k, case.v, case.cu_seqlens_q, case.cu_seqlens_k,
                            case.block_tables, case.k_cache, case.v_cache, case.scale)
    kc = case.k_cache.copy()
    vc = case.v_cache.copy()
    kc.reshape(-1, case.num_kv_heads, case.head_dim)[case.slot_mapping] = case.k
    vc.reshape(-1, case.num_kv_heads, case.head_dim)[case.slot_mapping] = case.v
    for b in range(case.num_seqs):
        P = int(case.k_lens[b] - case.q_lens[b])
        for i in range(int(case.q_lens[b])):
            row = case.cu_seqlens_q[b] + i
            d = orc.paged_decode(case.q[row:row + 1], kc, vc, case.block_tables[b:b + 1],
                                 np.array([P + i + 1], np.int32), case.scale)
            _close(out[row], d[0], TOL, "prefill row vs decode")


def pin_prefill_shared_vs_duplicated_prefix(orc):
    a = W.prefix_prefill_case(34, 3, 16, 2, 11, 4, 2, 16, 8, shared=True)
    b = W.prefix_prefill_case(34, 3, 16, 2, 11, 4, 2, 16, 8, shared=False)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.k, b.k)
    oa = orc.paged_prefill(a.q, a.k, a.v, a.cu_seqlens_q, a.cu_seqlens_k, a.block_tables,
                           a.k_cache, a.v_cache, a.scale)
    ob = orc.paged_prefill(b.q, b.k, b.v, b.cu_seqlens_q, b.cu_seqlens_k, b.block_tables,
                           b.k_cache, b.v_cache, b.scale)
    assert np.array_equal(oa, ob), "shared prefix blocks and duplicated copies differ"


# ------------------------------------------------------------------------------------------------
# Whole-block moves
# ------------------------------------------------------------------------------------------------


def pin_block_moves_match_numpy(orc):
    rng = W.rng_for(41, 0)
    NB, BS, Hkv, D = 12, 4, 2, 8
    kc = W.normal_bf16(rng, (NB, BS, Hkv, D))
    vc = W.normal_bf16(rng, (NB, BS, Hkv, D))
    pairs = np.array([[3, 7], [0, 11], [5, 2], [-1, 4], [6, 12]], np.int32)
    k2, v2, bad = orc.copy_blocks(kc, vc, pairs)
    assert bad == 2, "two pairs leave the pool"
    rk, rv = kc.copy(), vc.copy()
    ok = pairs[:3]
    rk[ok[:, 1]] = kc[ok[:, 0]]
    rv[ok[:, 1]] = vc[ok[:, 0]]
    assert np.array_equal(k2, rk) and np.array_equal(v2, rv), "copy-on-write differs"
    ids = np.array([9, 1, 4, 4], np.int32)
    gk, gv, bad = orc.gather_blocks(kc, vc, ids)
    assert bad == 0 and np.array_equal(gk, kc[ids]) and np.array_equal(gv, vc[ids])
    dst = np.array([0, 2, 10, 6], np.int32)
    sk, sv, bad = orc.scatter_blocks(gk, gv, dst, kc, vc)
    rk, rv = kc.copy(), vc.copy()
    rk[dst] = gk
    rv[dst] = gv
    assert bad == 0 and np.array_equal(sk, rk) and np.array_equal(sv, rv), "scatter differs"
    # swap out then swap in elsewhere is a permutation of placement: gathering again gives back
    back, _, _ = orc.gather_blocks(sk, sv, dst)
    assert np.array_equal(back, kc[ids])


# ------------------------------------------------------------------------------------------------
# Chained block hashes (prefix caching)
# ------------------------------------------------------------------------------------------------


def pin_xxh64_published_vectors(orc):
    with open(os.path.join(GOLDEN, "xxh64_vectors.json")) as f:
        g = json.load(f)
    for v in g["vectors"]:
        got = orc.xxh64(v["input"].encode(), v["seed"])
        assert got == int(v["xxh64"], 16), f"XXH64({v['input']!r}) = {got:016x}"


def pin_block_hash_chain(orc):
    import struct
    rng = W.rng_for(42, 0)
    BS = 16
    toks = rng.integers(0, 151936, size=5 * BS + 7, dtype=np.int64).astype(np.int32)
    out, clamped = orc.block_hashes(toks, np.array([0, len(toks)], np.int32), BS, 8)
    assert clamped == 0 and np.all(out[0, 5:] == 0), "only the 5 full blocks are hashed"
    parent = None
    for i in range(5):
        blk = struct.pack("<%di" % BS, *toks[i * BS:(i + 1) * BS].tolist())
        data = (b"" if parent is None else struct.pack("<Q", parent)) + blk
        parent = orc.xxh64(data, 0)
        assert int(out[0, i]) == parent, f"block {i}: chain or byte layout differs"


def pin_block_hash_prefix_semantics(orc):
    rng = W.rng_for(43, 0)
    BS = 16
    shared = rng.integers(0, 1000, size=3 * BS, dtype=np.int64).astype(np.int32)
    a = np.concatenate([shared, rng.integers(0, 1000, size=2 * BS).astype(np.int32)])
    b = np.concatenate([shared, rng.integers(0, 1000, size=2 * BS).astype(np.int32)])
    same = np.tile(shared[:BS], 2)  # the same block content at positions 0 and 1
    toks = np.concatenate([a, b, same]).astype(np.int32)
    cu = np.array([0, len(a), len(a) + len(b), len(toks)], np.int32)
    out, _ = orc.block_hashes(toks, cu, BS, 5)
    assert np.array_equal(out[0, :3], out[1, :3]), "a shared prefix must hash identically"
    assert np.all(out[0, 3:5] != out[1, 3:5]), "different continuations must differ"
    assert out[2, 0] != out[2, 1], "equal blocks at different positions must differ"
    assert out[2, 0] == out[0, 0], "block 0 depends only on its own tokens"
    _, clamped = orc.block_hashes(toks, cu, BS, 2)
    assert clamped == 2  # a and b have 5 full blocks; the third has exactly 2


ALL_PINS = [
    pin_store_matches_numpy_scatter,
    pin_store_padding_and_invalid,
    pin_store_round_trip,
    pin_gather_identity_and_permuted,
    pin_decode_matches_sdpa,
    pin_decode_closed_forms,
    pin_decode_golden_three_blocks,
    pin_decode_placement_invariance,
    pin_decode_shared_vs_duplicated,
    pin_decode_block_size_invariance,
    pin_decode_zero_context,
    pin_prefill_no_prefix_matches_causal_sdpa,
    pin_prefill_prefix_matches_masked_sdpa,
    pin_prefill_row_equals_decode,
    pin_prefill_shared_vs_duplicated_prefix,
    pin_block_moves_match_numpy,
    pin_xxh64_published_vectors,
    pin_block_hash_chain,
    pin_block_hash_prefix_semantics,
]
