"""GPU parity: decode on the tensor-core engine (tcgen05 MMAs with 128 keys on the M dimension
and a kv head's query heads on N) through the C ABI against the fp64 oracle, and against the
CUDA-core engine.

Bars as for the CUDA-core engine: outputs within max-abs 2e-2 of the oracle on N(0,1) inputs,
exactly bf16(V0) for a one-token context, zeros for a padded (context 0) row, and the store of a
decode step bit-exact in the cache.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_496_b300 as pk
import workloads as W
from tests.gpu_util import TOL, assert_attn_close, dev_bf16, dev_i32, host_bits

pytestmark = pytest.mark.gpu
TC, CC = pk.DECODE_ENGINE_TENSOR_CORE, pk.DECODE_ENGINE_CUDA_CORE


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pk.get_device_error()
    yield
    assert pk.get_device_error() == 0


def _upload(case):
    return dict(kc=dev_bf16(case.k_cache), vc=dev_bf16(case.v_cache), k=dev_bf16(case.k_new),
                v=dev_bf16(case.v_new), slots=dev_i32(case.slot_mapping), q=dev_bf16(case.q),
                bt=dev_i32(case.block_tables), ctx=dev_i32(case.context_lens))


def _decode(case, engine, split_tokens=0, stored=None):
    d = stored or _upload(case)
    if stored is None:
        pk.kv_store(d["k"], d["v"], d["slots"], d["kc"], d["vc"])
    out = pk.paged_decode(d["q"], d["kc"], d["vc"], d["bt"], d["ctx"], case.scale,
                          max_context_len=max(case.max_context_len, 1),
                          split_tokens=split_tokens, engine=engine)
    assert pk.get_device_error() == 0
    return out, d


def _oracle(orc, case):
    kc, vc, _ = orc.kv_store(case.k_new, case.v_new, case.slot_mapping, case.k_cache,
                             case.v_cache)
    return orc.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, case.scale)


TC_SHAPES = [  # (B, Hq, Hkv, BS, ctx_lo, ctx_hi): head_dim 128, group sizes 1, 2, 4 and 8
    (6, 32, 8, 256, 100, 900),
    (9, 32, 8, 16, 1, 700),
    (5, 64, 8, 32, 1, 500),
    (7, 16, 4, 64, 30, 1300),
    (4, 32, 4, 128, 60, 1100),
    (3, 8, 1, 16, 1, 4000),
    (8, 16, 8, 256, 1, 1024),
    (5, 8, 8, 64, 100, 2000),
    (6, 4, 2, 128, 1, 3000),
]


@pytest.mark.parametrize("shape", TC_SHAPES, ids=lambda s: "B%d_H%d-%d_BS%d" % s[:4])
@pytest.mark.parametrize("q_scale", [1.0, 8.0], ids=["normal", "sharp"])
def test_tc_decode_shapes(orc, shape, q_scale):
    B, Hq, Hkv, BS, lo, hi = shape
    case = W.random_decode_case(4000 + B + Hq + BS, B, Hq, Hkv, 128, BS, lo, hi, extra_pool=3,
                                pad_slots=2, q_scale=q_scale)
    out, d = _decode(case, TC)
    assert_attn_close(out, _oracle(orc, case), what=f"tensor-core decode {shape}")
    cc, _ = _decode(case, CC, stored=d)
    assert (out.float() - cc.float()).abs().max().item() <= TOL


@pytest.mark.parametrize("split", [128, 256, 512, -1, 0], ids=lambda s: f"split{s}")
@pytest.mark.parametrize("hq", [32, 16, 64], ids=lambda h: f"Hq{h}")
def test_tc_decode_split(orc, split, hq):
    """Chunked contexts (flash-decoding split) merged in the kernel: against the oracle, and the
    split result against the unsplit one."""
    case = W.random_decode_case(4050 + hq, 7, hq, 8, 128, 16, 1, 3000, extra_pool=2)
    out, d = _decode(case, TC, split_tokens=split)
    assert_attn_close(out, _oracle(orc, case), what=f"tensor-core split={split} Hq={hq}")
    whole, _ = _decode(case, TC, split_tokens=-1, stored=d)
    assert (out.float() - whole.float()).abs().max().item() <= TOL


def test_tc_decode_ragged_edges(orc):
    """Contexts at and around the 128-key tile and block boundaries, and a single token."""
    ctx = np.array([1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 512, 513],
                   np.int32)
    for Hq, BS in ((32, 16), (64, 256), (32, 64), (16, 128), (8, 32)):
        case = W.random_decode_case(4100 + Hq + BS, len(ctx), Hq, 8, 128, BS, 0, 0,
                                    context_lens=ctx)
        out, _ = _decode(case, TC)
        assert_attn_close(out, _oracle(orc, case), what=f"ragged Hq={Hq} BS={BS}")


@pytest.mark.parametrize("scale", [-0.0884, 0.0], ids=["negative", "zero"])
def test_tc_decode_scale_sign(orc, scale):
    import dataclasses
    case = dataclasses.replace(W.random_decode_case(4150, 6, 32, 8, 128, 16, 1, 700), scale=scale)
    out, _ = _decode(case, TC)
    assert_attn_close(out, _oracle(orc, case), what=f"tensor-core scale={scale}")


def test_tc_decode_single_token_is_exact():
    """ctx = 1: P is exactly 1 for the one key, so the output is bf16(V0) bit for bit."""
    case = W.random_decode_case(4200, 6, 32, 8, 128, 16, 1, 1)
    out, d = _decode(case, TC)
    for b in range(case.num_seqs):
        v0 = host_bits(d["vc"])[case.block_tables[b, 0], 0]
        assert np.array_equal(host_bits(out[b]), np.repeat(v0, 4, axis=0))


def test_tc_decode_zero_context_rows_are_zero(orc):
    ctx = np.array([300, 0, 17, 0, 1, 999, 0], np.int32)
    case = W.random_decode_case(4300, len(ctx), 32, 8, 128, 16, 0, 0, context_lens=ctx,
                                pad_slots=3)
    d = _upload(case)
    pk.kv_store(d["k"], d["v"], d["slots"], d["kc"], d["vc"])
    d["q"] = d["q"].clone()
    out = torch.full_like(d["q"], float("nan"))
    pk.paged_decode(d["q"], d["kc"], d["vc"], d["bt"], d["ctx"], case.scale, out=out,
                    max_context_len=999, engine=TC)
    assert pk.get_device_error() == 0
    for b in (1, 3, 6):
        assert torch.count_nonzero(out[b]) == 0
    assert_attn_close(out, _oracle(orc, case), what="tensor-core zero-context rows")


def test_tc_decode_placement_invariance():
    """Permuting physical blocks (tables permuted alike) gives bit-identical outputs."""
    case = W.random_decode_case(4400, 6, 32, 8, 128, 16, 50, 700)
    a, _ = _decode(case, TC)
    perm = W.rng_for(4400, 7).permutation(case.num_blocks)
    kc2, vc2 = np.empty_like(case.k_cache), np.empty_like(case.v_cache)
    kc2[perm], vc2[perm] = case.k_cache, case.v_cache
    bt2 = np.where(case.block_tables >= 0, perm[np.maximum(case.block_tables, 0)], -1)
    sl2 = np.where(case.slot_mapping >= 0,
                   perm[np.maximum(case.slot_mapping, 0) // 16] * 16 + case.slot_mapping % 16, -1)
    case2 = W.DecodeCase(case.num_blocks, 16, 8, 128, 32, kc2, vc2, case.k_new, case.v_new,
                         sl2.astype(np.int32), case.q, bt2.astype(np.int32), case.context_lens,
                         case.scale)
    b, _ = _decode(case2, TC)
    assert torch.equal(a, b)


def test_tc_decode_flags_bad_blocks_and_clamps():
    case = W.random_decode_case(4500, 3, 32, 8, 128, 16, 40, 60)
    d = _upload(case)
    pk.kv_store(d["k"], d["v"], d["slots"], d["kc"], d["vc"])
    pk.get_device_error()
    bt = d["bt"].clone()
    bt[1, 1] = case.num_blocks + 5
    pk.paged_decode(d["q"], d["kc"], d["vc"], bt, d["ctx"], case.scale, max_context_len=60,
                    engine=TC)
    assert pk.get_device_error() & pk.DEVERR_BAD_BLOCK
    ctx = d["ctx"].clone()
    ctx[0] = case.block_tables.shape[1] * 16 + 100
    pk.paged_decode(d["q"], d["kc"], d["vc"], d["bt"], ctx, case.scale, max_context_len=2000,
                    engine=TC)
    assert pk.get_device_error() & pk.DEVERR_CTX_CLAMPED


def test_tc_decode_store_equals_store_then_decode(orc):
    """The decode step with its store, on the tensor-core engine: the caches equal kv_store's
    bit for bit and the output equals store-then-decode bit for bit."""
    rng = W.rng_for(4600, 7)
    B, Hq, Hkv, D, BS = 9, 32, 8, 128, 16
    ctx = W.uniform_int(rng, 1, 700, B)
    ctx[[2, 6]] = 0
    bt, nb = W.place_blocks(rng, ctx, BS, pool_blocks=int(W.blocks_needed(ctx, BS).sum()) + 2)
    slots = np.full(B, -1, np.int32)
    live = np.nonzero(ctx > 0)[0]
    slots[live] = W.slots_for_positions(bt, live, ctx[live] - 1, BS)
    kc0, vc0 = W.normal_bf16(rng, (nb, BS, Hkv, D)), W.normal_bf16(rng, (nb, BS, Hkv, D))
    k, v, q = (W.normal_bf16(rng, (B, Hkv, D)), W.normal_bf16(rng, (B, Hkv, D)),
               W.normal_bf16(rng, (B, Hq, D)))
    scale = 1 / np.sqrt(D)
    kd, vd, qd = dev_bf16(k), dev_bf16(v), dev_bf16(q)
    btd, cd, sd = dev_i32(bt), dev_i32(ctx), dev_i32(slots)
    kc1, vc1 = dev_bf16(kc0), dev_bf16(vc0)
    pk.kv_store(kd, vd, sd, kc1, vc1)
    ref = pk.paged_decode(qd, kc1, vc1, btd, cd, scale, max_context_len=700, engine=TC)
    kc2, vc2 = dev_bf16(kc0), dev_bf16(vc0)
    out = pk.paged_decode_store(qd, kd, vd, sd, kc2, vc2, btd, cd, scale, max_context_len=700,
                                engine=TC)
    assert pk.get_device_error() == 0
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2)
    assert torch.equal(out, ref)
    rk, rv, _ = orc.kv_store(k, v, slots, kc0, vc0)
    assert_attn_close(out, orc.paged_decode(q, rk, rv, bt, ctx, scale), what="tc decode store")


def test_tc_decode_graph_capture_matches_eager():
    case = W.random_decode_case(4700, 8, 32, 8, 128, 16, 10, 1500)
    d = _upload(case)
    plan = pk.decode_plan(case.num_seqs, 32, d["kc"], case.max_context_len, 0, TC)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d["q"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            pk.kv_store(d["k"], d["v"], d["slots"], d["kc"], d["vc"])
            pk.paged_decode(d["q"], d["kc"], d["vc"], d["bt"], d["ctx"], case.scale, out=out,
                            plan=plan, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    ref = pk.paged_decode(d["q"], d["kc"], d["vc"], d["bt"], d["ctx"], case.scale, plan=plan,
                          workspace=ws)
    assert torch.equal(out, ref)
