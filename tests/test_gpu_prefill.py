"""GPU parity: varlen causal paged prefill (tcgen05) through the C ABI against the fp64 oracle.

The new tokens are stored with kv_store first (as the engine does); the kernel then reads every key
through the block table. The oracle reads the cached prefix through the table and the new keys from
k/v directly, so the two share no step. Bar: max-abs error <= 2e-2 on N(0,1) inputs.
"""
import dataclasses

import numpy as np
import pytest
import torch

import paged_kv_cache_496_b300 as pk
import workloads as W
from tests.gpu_util import TOL, assert_attn_close, dev_bf16, dev_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pk.get_device_error()
    yield
    assert pk.get_device_error() == 0


def _run_paged(case: W.PrefillCase):
    kc, vc = dev_bf16(case.k_cache), dev_bf16(case.v_cache)
    k, v = dev_bf16(case.k), dev_bf16(case.v)
    if len(case.slot_mapping):
        pk.kv_store(k, v, dev_i32(case.slot_mapping), kc, vc)
    out = pk.paged_prefill(dev_bf16(case.q), k, v, dev_i32(case.cu_seqlens_q),
                           dev_i32(case.cu_seqlens_k), dev_i32(case.block_tables), case.scale,
                           k_cache=kc, v_cache=vc,
                           max_seqlen_q=int(case.q_lens.max(initial=0)))
    assert pk.get_device_error() == 0
    return out, kc, vc


def _oracle(orc, case):
    return orc.paged_prefill(case.q, case.k, case.v, case.cu_seqlens_q, case.cu_seqlens_k,
                             case.block_tables, case.k_cache, case.v_cache, case.scale)


def test_prefill_single_tile_no_prefix(orc):
    """One sequence, one CTA tile, keys read from k/v directly (no block table)."""
    rng = W.rng_for(61, 0)
    Hq, Hkv, D = 32, 8, 128
    ql = np.array([20], np.int32)
    cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    T = int(ql.sum())
    q, k, v = (W.normal_bf16(rng, (T, Hq, D)), W.normal_bf16(rng, (T, Hkv, D)),
               W.normal_bf16(rng, (T, Hkv, D)))
    out = pk.paged_prefill(dev_bf16(q), dev_bf16(k), dev_bf16(v), dev_i32(cu), dev_i32(cu), None,
                           1 / np.sqrt(D), max_seqlen_q=int(ql.max()))
    assert pk.get_device_error() == 0
    empty = np.zeros((1, 16, Hkv, D), np.uint16)
    ref = orc.paged_prefill(q, k, v, cu, cu, None, empty, empty, 1 / np.sqrt(D))
    assert_attn_close(out, ref, what="single tile")


@pytest.mark.parametrize("qlens", [[1, 37, 130], [64, 65, 200, 0, 3]], ids=["a", "b"])
def test_prefill_no_prefix_varlen(orc, qlens):
    rng = W.rng_for(62, len(qlens))
    Hq, Hkv, D = 32, 8, 128
    ql = np.array(qlens, np.int32)
    cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    T = int(ql.sum())
    q, k, v = (W.normal_bf16(rng, (T, Hq, D)), W.normal_bf16(rng, (T, Hkv, D)),
               W.normal_bf16(rng, (T, Hkv, D)))
    out = pk.paged_prefill(dev_bf16(q), dev_bf16(k), dev_bf16(v), dev_i32(cu), dev_i32(cu), None,
                           1 / np.sqrt(D), max_seqlen_q=int(ql.max()))
    assert pk.get_device_error() == 0
    empty = np.zeros((1, 16, Hkv, D), np.uint16)
    ref = orc.paged_prefill(q, k, v, cu, cu, None, empty, empty, 1 / np.sqrt(D))
    assert_attn_close(out, ref, what=f"no prefix {qlens}")


@pytest.mark.parametrize("BS", [256, 128, 64, 32, 16])
@pytest.mark.parametrize("q_scale", [1.0, 8.0], ids=["normal", "sharp"])
def test_prefill_shared_prefix(orc, BS, q_scale):
    case = W.prefix_prefill_case(63, 4, 256, 1, 300, 32, 8, 128, BS, q_scale=q_scale,
                                 suffix_lens=np.array([1, 63, 64, 300]))
    out, _, _ = _run_paged(case)
    assert_attn_close(out, _oracle(orc, case), what=f"prefix BS={BS} q_scale={q_scale}")


@pytest.mark.parametrize("scale", [-0.0884, 0.0, 0.25], ids=["negative", "zero", "large"])
def test_prefill_scale_sign(orc, scale):
    """Any scale is a valid input. With scale <= 0 every tile takes the masked path, which
    scales before the max (the full-tile path takes the max of raw scores, correct only for a
    positive scale). Scale 0 gives uniform weights over each row's visible keys."""
    case = dataclasses.replace(
        W.prefix_prefill_case(65, 3, 256, 1, 200, 32, 8, 128, 64,
                              suffix_lens=np.array([1, 70, 200])), scale=scale)
    out, _, _ = _run_paged(case)
    assert_attn_close(out, _oracle(orc, case), what=f"scale={scale}")


@pytest.mark.parametrize("Hq", [8, 16, 64], ids=["G1", "G2", "G8"])
def test_prefill_group_sizes(orc, Hq):
    case = W.prefix_prefill_case(64, 3, 128, 1, 200, Hq, 8, 128, 64,
                                 suffix_lens=np.array([5, 129, 200]))
    out, _, _ = _run_paged(case)
    assert_attn_close(out, _oracle(orc, case), what=f"Hq={Hq}")


def test_prefill_row_equals_decode():
    """Prefill query i equals decode over the first P + i + 1 keys of the same cache."""
    case = W.prefix_prefill_case(65, 2, 256, 40, 90, 32, 8, 128, 256)
    out, kc, vc = _run_paged(case)
    for b in range(case.num_seqs):
        P = int(case.k_lens[b] - case.q_lens[b])
        rows = np.arange(case.cu_seqlens_q[b], case.cu_seqlens_q[b + 1])
        ctx = P + 1 + np.arange(len(rows))
        bt = np.repeat(case.block_tables[b:b + 1], len(rows), axis=0)
        q = dev_bf16(case.q[rows])
        d = pk.paged_decode(q, kc, vc, dev_i32(bt), dev_i32(ctx), case.scale,
                            max_context_len=int(ctx.max()))
        err = (d.float() - out[torch.as_tensor(rows, device="cuda")].float()).abs().max().item()
        assert err <= TOL, err


def test_prefill_bad_lengths_flagged():
    case = W.prefix_prefill_case(66, 2, 256, 10, 20, 32, 8, 128, 256)
    cu_k = case.cu_seqlens_k.copy()
    cu_k[1] = cu_k[0] + int(case.q_lens[0]) - 1  # k_len < q_len for sequence 0
    kc, vc = dev_bf16(case.k_cache), dev_bf16(case.v_cache)
    k, v = dev_bf16(case.k), dev_bf16(case.v)
    pk.get_device_error()
    pk.paged_prefill(dev_bf16(case.q), k, v, dev_i32(case.cu_seqlens_q), dev_i32(cu_k),
                     dev_i32(case.block_tables), case.scale, k_cache=kc, v_cache=vc)
    assert pk.get_device_error() & pk.DEVERR_BAD_LENGTHS


def test_prefill_bad_block_flagged_not_faulted():
    case = W.prefix_prefill_case(67, 2, 256, 10, 20, 32, 8, 128, 256)
    bt = case.block_tables.copy()
    bt[0, 0] = case.num_blocks + 3
    kc, vc = dev_bf16(case.k_cache), dev_bf16(case.v_cache)
    pk.get_device_error()
    pk.paged_prefill(dev_bf16(case.q), dev_bf16(case.k), dev_bf16(case.v),
                     dev_i32(case.cu_seqlens_q), dev_i32(case.cu_seqlens_k), dev_i32(bt),
                     case.scale, k_cache=kc, v_cache=vc)
    assert pk.get_device_error() & pk.DEVERR_BAD_BLOCK


def _head_subcase(case: W.PrefillCase, seqs, g: int) -> W.PrefillCase:
    """The sub-problem of sequences `seqs` restricted to kv head g and its G query heads (heads are
    independent, so this is the same attention on fewer heads)."""
    G = case.num_q_heads // case.num_kv_heads
    rows = np.concatenate([np.arange(case.cu_seqlens_q[b], case.cu_seqlens_q[b + 1])
                           for b in seqs]).astype(np.int64)
    ql, kl = case.q_lens[seqs], case.k_lens[seqs]
    return W.PrefillCase(
        case.num_blocks, case.block_size, 1, case.head_dim, G,
        np.ascontiguousarray(case.k_cache[:, :, g:g + 1]),
        np.ascontiguousarray(case.v_cache[:, :, g:g + 1]),
        np.ascontiguousarray(case.q[rows, g * G:(g + 1) * G]),
        np.ascontiguousarray(case.k[rows, g:g + 1]), np.ascontiguousarray(case.v[rows, g:g + 1]),
        np.concatenate([[0], np.cumsum(ql)]).astype(np.int32),
        np.concatenate([[0], np.cumsum(kl)]).astype(np.int32),
        np.ascontiguousarray(case.block_tables[seqs]), case.slot_mapping[:0], case.scale)


@pytest.mark.slow
def test_full_prefix_prefill_workload(orc):
    """64 sequences sharing a 1024-token prefix (4 blocks of 256), U{100..1024} new tokens each,
    in the launch configuration the benchmark times. Every sequence is compared with the oracle
    on one kv head (all G query heads of it; sequence b on kv head b % 8, so every head and every
    item ordering of the persistent grid is covered), and three sequences (longest, shortest,
    index 17) on all heads."""
    ql = W.prefix_prefill_suffix_lengths()
    case = W.prefix_prefill_case(4, 64, 1024, 100, 1024, 32, 8, 128, 256, suffix_lens=ql)
    out, _, _ = _run_paged(case)
    assert torch.isfinite(out.float()).all()
    G = case.num_q_heads // case.num_kv_heads
    for g in range(case.num_kv_heads):
        seqs = np.arange(g, case.num_seqs, case.num_kv_heads)
        ref = _oracle(orc, _head_subcase(case, seqs, g))
        rows = np.concatenate([np.arange(case.cu_seqlens_q[b], case.cu_seqlens_q[b + 1])
                               for b in seqs])
        got = out[torch.as_tensor(rows, device=out.device), g * G:(g + 1) * G]
        assert_attn_close(got, ref, what=f"full workload kv head {g}, sequences {list(seqs)}")
    for b in (int(np.argmax(ql)), int(np.argmin(ql)), 17):
        sub = W.PrefillCase(case.num_blocks, 256, 8, 128, 32, case.k_cache, case.v_cache,
                            case.q[case.cu_seqlens_q[b]:case.cu_seqlens_q[b + 1]],
                            case.k[case.cu_seqlens_q[b]:case.cu_seqlens_q[b + 1]],
                            case.v[case.cu_seqlens_q[b]:case.cu_seqlens_q[b + 1]],
                            np.array([0, ql[b]], np.int32),
                            np.array([0, ql[b] + 1024], np.int32), case.block_tables[b:b + 1],
                            case.slot_mapping[:0], case.scale)
        ref = _oracle(orc, sub)
        rows = slice(int(case.cu_seqlens_q[b]), int(case.cu_seqlens_q[b + 1]))
        assert_attn_close(out[rows], ref, what=f"full workload seq {b}")


def _prefill_call(q, k, v, cu_q, cu_k, bt, scale, kc, vc):
    out = pk.paged_prefill(dev_bf16(q), dev_bf16(k), dev_bf16(v), dev_i32(cu_q), dev_i32(cu_k),
                           dev_i32(bt), scale, k_cache=kc, v_cache=vc)
    assert pk.get_device_error() == 0
    return out


def test_chunked_prefill_equals_one_shot(orc):
    """A prompt prefilled in two chunks (the second sees the first as cached prefix) gives the
    same rows as one prefill of the whole prompt."""
    case = W.prefix_prefill_case(68, 1, 256, 0, 0, 32, 8, 128, 64, suffix_lens=np.array([300]))
    kc, vc = dev_bf16(case.k_cache), dev_bf16(case.v_cache)
    pk.kv_store(dev_bf16(case.k), dev_bf16(case.v), dev_i32(case.slot_mapping), kc, vc)
    whole = _prefill_call(case.q, case.k, case.v, case.cu_seqlens_q, case.cu_seqlens_k,
                          case.block_tables, case.scale, kc, vc)
    a = 120
    first = _prefill_call(case.q[:a], case.k[:a], case.v[:a], np.array([0, a]),
                          np.array([0, 256 + a]), case.block_tables, case.scale, kc, vc)
    second = _prefill_call(case.q[a:], case.k[a:], case.v[a:], np.array([0, 300 - a]),
                           np.array([0, 556]), case.block_tables, case.scale, kc, vc)
    chunked = torch.cat([first, second])
    assert (chunked.float() - whole.float()).abs().max().item() <= TOL
    assert_attn_close(chunked, _oracle(orc, case), what="chunked prefill")


def test_mixed_decode_and_prefill_batch(orc):
    """Decode rows (one new token) and prefill chunks in one varlen call."""
    rng = W.rng_for(69, 0)
    ql = np.array([1, 1, 200, 1, 64, 1, 129], np.int32)
    prefix = np.array([300, 1000, 0, 17, 512, 1, 255], np.int32)
    BS, Hq, Hkv, D = 16, 32, 8, 128
    kl = ql + prefix
    bt, nb = W.place_blocks(rng, kl, BS)
    kc = W.normal_bf16(rng, (nb, BS, Hkv, D))
    vc = W.normal_bf16(rng, (nb, BS, Hkv, D))
    T = int(ql.sum())
    q = W.normal_bf16(rng, (T, Hq, D))
    k = W.normal_bf16(rng, (T, Hkv, D))
    v = W.normal_bf16(rng, (T, Hkv, D))
    cu_q = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(kl)]).astype(np.int32)
    seq = np.concatenate([np.full(n, b) for b, n in enumerate(ql)])
    pos = np.concatenate([prefix[b] + np.arange(n) for b, n in enumerate(ql)])
    slots = W.slots_for_positions(bt, seq, pos, BS)
    kcd, vcd = dev_bf16(kc), dev_bf16(vc)
    pk.kv_store(dev_bf16(k), dev_bf16(v), dev_i32(slots), kcd, vcd)
    out = _prefill_call(q, k, v, cu_q, cu_k, bt, 1 / np.sqrt(D), kcd, vcd)
    ref = orc.paged_prefill(q, k, v, cu_q, cu_k, bt, kc, vc, 1 / np.sqrt(D))
    assert_attn_close(out, ref, what="mixed batch")


def _mixed_case(seed, ql, prefix, BS, Hq, Hkv=8, D=128):
    rng = W.rng_for(seed, 0)
    ql = np.asarray(ql, np.int32)
    prefix = np.asarray(prefix, np.int32)
    kl = ql + prefix
    bt, nb = W.place_blocks(rng, kl, BS)
    kc = W.normal_bf16(rng, (nb, BS, Hkv, D))
    vc = W.normal_bf16(rng, (nb, BS, Hkv, D))
    T = int(ql.sum())
    q, k, v = (W.normal_bf16(rng, (T, Hq, D)), W.normal_bf16(rng, (T, Hkv, D)),
               W.normal_bf16(rng, (T, Hkv, D)))
    cu_q = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(kl)]).astype(np.int32)
    seq = np.concatenate([np.full(n, b) for b, n in enumerate(ql)])
    pos = np.concatenate([prefix[b] + np.arange(n) for b, n in enumerate(ql)])
    slots = W.slots_for_positions(bt, seq, pos, BS)
    return dict(q=q, k=k, v=v, kc=kc, vc=vc, bt=bt, cu_q=cu_q, cu_k=cu_k, slots=slots, ql=ql,
                kl=kl, scale=1 / np.sqrt(D))


@pytest.mark.parametrize("BS,Hq", [(16, 32), (256, 32), (64, 64), (32, 16)],
                         ids=["BS16_G4", "BS256_G4", "BS64_G8", "BS32_G2"])
def test_mixed_batch_decode_rows_match_decode(orc, BS, Hq):
    """A paged varlen call mixing decode rows (q_len == 1, long and short contexts) with prefill
    chunks matches the oracle, and its decode rows match the decode kernel on the same
    sequences within the tolerance."""
    c = _mixed_case(70 + BS + Hq, [1, 1, 200, 1, 64, 1, 129, 1, 1],
                    [300, 1000, 0, 17, 512, 1, 255, 2047, 63], BS, Hq)
    kcd, vcd = dev_bf16(c["kc"]), dev_bf16(c["vc"])
    q, k, v = dev_bf16(c["q"]), dev_bf16(c["k"]), dev_bf16(c["v"])
    pk.kv_store(k, v, dev_i32(c["slots"]), kcd, vcd)
    out = pk.paged_prefill(q, k, v, dev_i32(c["cu_q"]), dev_i32(c["cu_k"]), dev_i32(c["bt"]),
                           c["scale"], k_cache=kcd, v_cache=vcd, max_seqlen_q=int(c["ql"].max()))
    assert pk.get_device_error() == 0
    ref = orc.paged_prefill(c["q"], c["k"], c["v"], c["cu_q"], c["cu_k"], c["bt"], c["kc"],
                            c["vc"], c["scale"])
    assert_attn_close(out, ref, what=f"mixed BS={BS} Hq={Hq}")
    dec = np.nonzero(c["ql"] == 1)[0]
    rows = torch.as_tensor(c["cu_q"][dec], device="cuda")
    d = pk.paged_decode(q[rows], kcd, vcd, dev_i32(c["bt"][dec]), dev_i32(c["kl"][dec]),
                        c["scale"], max_context_len=int(c["kl"].max()))
    assert (out[rows].float() - d.float()).abs().max().item() <= TOL


def test_all_decode_rows_batch(orc):
    """Every sequence of a varlen call a decode row (q_len == 1)."""
    ql = np.ones(37, np.int32)
    prefix = W.uniform_int(W.rng_for(71, 1), 1, 900, 37).astype(np.int32)
    c = _mixed_case(71, ql, prefix, 16, 32)
    kcd, vcd = dev_bf16(c["kc"]), dev_bf16(c["vc"])
    k, v = dev_bf16(c["k"]), dev_bf16(c["v"])
    pk.kv_store(k, v, dev_i32(c["slots"]), kcd, vcd)
    out = pk.paged_prefill(dev_bf16(c["q"]), k, v, dev_i32(c["cu_q"]), dev_i32(c["cu_k"]),
                           dev_i32(c["bt"]), c["scale"], k_cache=kcd, v_cache=vcd,
                           max_seqlen_q=1)
    assert pk.get_device_error() == 0
    ref = orc.paged_prefill(c["q"], c["k"], c["v"], c["cu_q"], c["cu_k"], c["bt"], c["kc"],
                            c["vc"], c["scale"])
    assert_attn_close(out, ref, what="all decode rows")


def test_dense_numbering_many_sequences(orc):
    """400 sequences (some without new tokens, every fifth a prefill chunk of 16-80 tokens): the
    dense lookup's search takes two rounds of probes, and the heavy (prefill) and light
    sequences sit in two queues, so positions are permuted. The output equals the sparse
    numbering's bit for bit and the oracle's."""
    B = 400
    ql = W.uniform_int(W.rng_for(75, 1), 0, 5, B).astype(np.int32)
    ql[::5] = W.uniform_int(W.rng_for(75, 3), 16, 80, len(ql[::5]))
    prefix = W.uniform_int(W.rng_for(75, 2), 0, 200, B).astype(np.int32)
    c = _mixed_case(75, ql, prefix, 16, 32)
    kc, vc = dev_bf16(c["kc"]), dev_bf16(c["vc"])
    pk.kv_store(dev_bf16(c["k"]), dev_bf16(c["v"]), dev_i32(c["slots"]), kc, vc)
    args = (dev_bf16(c["q"]), dev_bf16(c["k"]), dev_bf16(c["v"]), dev_i32(c["cu_q"]),
            dev_i32(c["cu_k"]), dev_i32(c["bt"]), c["scale"])
    kw = dict(k_cache=kc, v_cache=vc, max_seqlen_q=int(ql.max()))
    dense_ws = torch.empty(pk.prefill_workspace_bytes(B), dtype=torch.uint8, device="cuda")
    sparse_ws = torch.empty(pk.PREFILL_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    a = pk.paged_prefill(*args, workspace=dense_ws, **kw)
    b = pk.paged_prefill(*args, workspace=sparse_ws, **kw)
    assert pk.get_device_error() == 0
    assert torch.equal(a, b)
    ref = orc.paged_prefill(c["q"], c["k"], c["v"], c["cu_q"], c["cu_k"], c["bt"], c["kc"],
                            c["vc"], c["scale"])
    assert_attn_close(a, ref, what="400 sequences")


def test_dense_numbering_more_sequences_than_plan_threads(orc):
    """2,500 sequences (more than the plan CTA's 1,024 threads, so each thread places three):
    decode rows with short contexts and every 25th a prefill chunk, merged into one claim order.
    Equal to the sparse numbering bit for bit, and to the oracle on a sample of sequences."""
    B = 2500
    ql = np.ones(B, np.int32)
    ql[::25] = W.uniform_int(W.rng_for(76, 1), 16, 48, len(ql[::25]))
    prefix = W.uniform_int(W.rng_for(76, 2), 0, 60, B).astype(np.int32)
    c = _mixed_case(76, ql, prefix, 16, 32)
    kc, vc = dev_bf16(c["kc"]), dev_bf16(c["vc"])
    pk.kv_store(dev_bf16(c["k"]), dev_bf16(c["v"]), dev_i32(c["slots"]), kc, vc)
    args = (dev_bf16(c["q"]), dev_bf16(c["k"]), dev_bf16(c["v"]), dev_i32(c["cu_q"]),
            dev_i32(c["cu_k"]), dev_i32(c["bt"]), c["scale"])
    kw = dict(k_cache=kc, v_cache=vc, max_seqlen_q=int(ql.max()))
    dense_ws = torch.empty(pk.prefill_workspace_bytes(B), dtype=torch.uint8, device="cuda")
    sparse_ws = torch.empty(pk.PREFILL_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    a = pk.paged_prefill(*args, workspace=dense_ws, **kw)
    b = pk.paged_prefill(*args, workspace=sparse_ws, **kw)
    assert pk.get_device_error() == 0
    assert torch.equal(a, b)
    for s in (0, 1, 1023, 1024, 1025, 1250, 2047, 2048, 2475, 2499):
        q0, q1 = int(c["cu_q"][s]), int(c["cu_q"][s + 1])
        k0, k1 = int(c["cu_k"][s]), int(c["cu_k"][s + 1])
        ref = orc.paged_prefill(c["q"][q0:q1], c["k"][q0:q1], c["v"][q0:q1],
                                np.array([0, q1 - q0], np.int32), np.array([0, k1 - k0], np.int32),
                                c["bt"][s:s + 1], c["kc"], c["vc"], c["scale"])
        assert_attn_close(a[q0:q1], ref, what=f"sequence {s} of {B}")


@pytest.mark.parametrize("which", ["mixed", "no_prefix", "prefix"])
def test_dense_and_sparse_item_numbering_agree(which):
    """With a workspace of pkv_prefill_workspace_bytes(num_seqs) the work is numbered densely
    (a plan kernel lists only the query tiles each sequence has); with PREFILL_WORKSPACE_BYTES
    the grid skips the ids of missing tiles. Every item is computed the same way, so the outputs
    are bit-identical."""
    if which == "mixed":
        c = _mixed_case(72, [1, 1, 300, 1, 64, 0, 129, 1], [300, 1000, 0, 17, 512, 3, 255, 63],
                        16, 32)
        bt, kc, vc = dev_i32(c["bt"]), dev_bf16(c["kc"]), dev_bf16(c["vc"])
        pk.kv_store(dev_bf16(c["k"]), dev_bf16(c["v"]), dev_i32(c["slots"]), kc, vc)
        args = (dev_bf16(c["q"]), dev_bf16(c["k"]), dev_bf16(c["v"]), dev_i32(c["cu_q"]),
                dev_i32(c["cu_k"]), bt, c["scale"])
        kw = dict(k_cache=kc, v_cache=vc, max_seqlen_q=300)
        B = len(c["ql"])
    elif which == "no_prefix":
        rng = W.rng_for(73, 0)
        ql = np.array([64, 1, 200, 0, 3, 130], np.int32)
        cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
        T = int(ql.sum())
        args = (dev_bf16(W.normal_bf16(rng, (T, 32, 128))), dev_bf16(W.normal_bf16(rng, (T, 8, 128))),
                dev_bf16(W.normal_bf16(rng, (T, 8, 128))), dev_i32(cu), dev_i32(cu), None,
                1 / np.sqrt(128))
        kw = dict(max_seqlen_q=200)
        B = len(ql)
    else:
        case = W.prefix_prefill_case(74, 5, 256, 1, 300, 32, 8, 128, 64)
        kc, vc = dev_bf16(case.k_cache), dev_bf16(case.v_cache)
        k, v = dev_bf16(case.k), dev_bf16(case.v)
        pk.kv_store(k, v, dev_i32(case.slot_mapping), kc, vc)
        args = (dev_bf16(case.q), k, v, dev_i32(case.cu_seqlens_q), dev_i32(case.cu_seqlens_k),
                dev_i32(case.block_tables), case.scale)
        kw = dict(k_cache=kc, v_cache=vc, max_seqlen_q=int(case.q_lens.max()))
        B = case.num_seqs
    dense_ws = torch.empty(pk.prefill_workspace_bytes(B), dtype=torch.uint8, device="cuda")
    sparse_ws = torch.empty(pk.PREFILL_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    a = pk.paged_prefill(*args, workspace=dense_ws, **kw)
    b = pk.paged_prefill(*args, workspace=sparse_ws, **kw)
    assert pk.get_device_error() == 0
    assert torch.equal(a, b)
