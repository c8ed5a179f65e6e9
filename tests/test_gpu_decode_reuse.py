"""GPU parity: decode calls that reuse the device plan of the previous call (PKV_DECODE_PLAN_REUSE),
as every layer of a decode step after the first can: same outputs as planning every call, bit for
bit, on both engines, split and unsplit; the store variant keeps the cache bit-exact."""
import numpy as np
import pytest
import torch

import paged_kv_cache_496_b300 as pk
import workloads as W
from tests.gpu_util import assert_attn_close, dev_bf16, dev_i32

pytestmark = pytest.mark.gpu
ENGINES = [pk.DECODE_ENGINE_CUDA_CORE, pk.DECODE_ENGINE_TENSOR_CORE]
ENGINE_IDS = ["cuda_core", "tensor_core"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pk.get_device_error()
    yield
    assert pk.get_device_error() == 0


def _layers(seed, n_layers, B, Hq, Hkv, BS, lo, hi):
    """One batch (lengths, tables, slots) and n_layers of (q, k_new, v_new, caches)."""
    case = W.random_decode_case(seed, B, Hq, Hkv, 128, BS, lo, hi, extra_pool=2, pad_slots=1)
    layers = []
    for l in range(n_layers):
        if l == 0:
            kc, vc, q = dev_bf16(case.k_cache), dev_bf16(case.v_cache), dev_bf16(case.q)
            kn, vn = dev_bf16(case.k_new), dev_bf16(case.v_new)
        else:
            mk = lambda t, s: W.fill_normal_bf16_(torch.empty_like(t), seed, 10 * l + s)  # noqa
            kc, vc = mk(layers[0]["kc0"], 1), mk(layers[0]["vc0"], 2)
            q, kn, vn = mk(layers[0]["q"], 3), mk(layers[0]["kn"], 4), mk(layers[0]["vn"], 5)
        layers.append(dict(kc0=kc, vc0=vc, q=q, kn=kn, vn=vn))
    return case, layers


@pytest.mark.parametrize("engine", ENGINES, ids=ENGINE_IDS)
@pytest.mark.parametrize("split", [0, 256, -1], ids=["auto", "split256", "unsplit"])
def test_reused_plan_equals_fresh_plan(orc, engine, split):
    case, layers = _layers(5100 + split % 7, 3, 9, 32, 8, 128, 1, 3000)
    bt, ctx, slots = dev_i32(case.block_tables), dev_i32(case.context_lens), dev_i32(
        case.slot_mapping)
    plan = pk.decode_plan(case.num_seqs, 32, layers[0]["kc0"], case.max_context_len, split, engine)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    ws_fresh = torch.empty_like(ws)
    for l, d in enumerate(layers):
        kc, vc = d["kc0"].clone(), d["vc0"].clone()
        pk.kv_store(d["kn"], d["vn"], slots, kc, vc)
        reused = pk.paged_decode(d["q"], kc, vc, bt, ctx, case.scale, plan=plan, workspace=ws,
                                 reuse_plan=l > 0)
        fresh = pk.paged_decode(d["q"], kc, vc, bt, ctx, case.scale, plan=plan,
                                workspace=ws_fresh)
        assert pk.get_device_error() == 0
        assert torch.equal(reused, fresh), f"layer {l}"
    # the last reused layer against the oracle
    host = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    ref = orc.paged_decode(host(d["q"]), host(kc), host(vc), case.block_tables, case.context_lens,
                           case.scale)
    assert_attn_close(reused, ref, what=f"reused plan engine={engine} split={split}")


@pytest.mark.parametrize("engine", ENGINES, ids=ENGINE_IDS)
def test_reused_plan_with_store(engine):
    """paged_decode_store on a reused plan: the store runs in its own grid; caches and outputs
    equal the call that plans (whose plan grid stores)."""
    rng = W.rng_for(5200, 7)
    B, Hq, Hkv, D, BS = 9, 32, 8, 128, 128
    ctx = W.uniform_int(rng, 1, 2500, B)
    ctx[[2, 6]] = 0
    bt, nb = W.place_blocks(rng, ctx, BS, pool_blocks=int(W.blocks_needed(ctx, BS).sum()) + 2)
    slots = np.full(B, -1, np.int32)
    live = np.nonzero(ctx > 0)[0]
    slots[live] = W.slots_for_positions(bt, live, ctx[live] - 1, BS)
    btd, cd, sd = dev_i32(bt), dev_i32(ctx), dev_i32(slots)
    plan = pk.decode_plan(B, Hq, torch.empty((nb, BS, Hkv, D), dtype=torch.bfloat16, device="meta"), 2500, 0,
                          engine)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    ws_fresh = torch.empty_like(ws)
    for l in range(3):
        kc0, vc0 = W.normal_bf16(rng, (nb, BS, Hkv, D)), W.normal_bf16(rng, (nb, BS, Hkv, D))
        k, v, q = (W.normal_bf16(rng, (B, Hkv, D)), W.normal_bf16(rng, (B, Hkv, D)),
                   W.normal_bf16(rng, (B, Hq, D)))
        kd, vd, qd = dev_bf16(k), dev_bf16(v), dev_bf16(q)
        kc1, vc1 = dev_bf16(kc0), dev_bf16(vc0)
        out1 = pk.paged_decode_store(qd, kd, vd, sd, kc1, vc1, btd, cd, D ** -0.5, plan=plan,
                                     workspace=ws, reuse_plan=l > 0)
        kc2, vc2 = dev_bf16(kc0), dev_bf16(vc0)
        out2 = pk.paged_decode_store(qd, kd, vd, sd, kc2, vc2, btd, cd, D ** -0.5, plan=plan,
                                     workspace=ws_fresh)
        assert pk.get_device_error() == 0
        assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2), f"layer {l} cache"
        assert torch.equal(out1, out2), f"layer {l} output"


@pytest.mark.parametrize("engine", ENGINES, ids=ENGINE_IDS)
def test_reused_plan_in_a_captured_step(engine):
    """A step captured as one CUDA graph (store + decode for three layers, the first planning and
    the others reusing its plan, split contexts): replaying it equals the eager step."""
    case, layers = _layers(5300, 3, 7, 32, 8, 128, 1, 3000)
    bt, ctx, slots = dev_i32(case.block_tables), dev_i32(case.context_lens), dev_i32(
        case.slot_mapping)
    plan = pk.decode_plan(case.num_seqs, 32, layers[0]["kc0"], case.max_context_len, 256, engine)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    caches = [(d["kc0"].clone(), d["vc0"].clone()) for d in layers]
    outs = [torch.empty_like(d["q"]) for d in layers]

    def step():
        for l, d in enumerate(layers):
            kc, vc = caches[l]
            pk.kv_store(d["kn"], d["vn"], slots, kc, vc)
            pk.paged_decode(d["q"], kc, vc, bt, ctx, case.scale, out=outs[l], plan=plan,
                            workspace=ws, reuse_plan=l > 0)

    step()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for o in outs:
        o.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert pk.get_device_error() == 0
    for l in range(3):
        assert torch.equal(outs[l], eager[l]), f"layer {l}"


@pytest.mark.parametrize("engine", ENGINES, ids=ENGINE_IDS)
def test_reuse_on_a_foreign_workspace_is_bounded(engine):
    """A reuse on a workspace that never held this call's plan stays inside its buffers: a work
    list longer than the batch allows is dropped (0xff-filled workspace) and a list from a larger
    batch has its extra sequences skipped, both flagged; a planning call on the same workspace
    then gives the fresh plan's output again."""
    case, layers = _layers(5400, 1, 9, 32, 8, 128, 1, 2000)
    d = layers[0]
    kc, vc = d["kc0"].clone(), d["vc0"].clone()
    bt, ctx, slots = dev_i32(case.block_tables), dev_i32(case.context_lens), dev_i32(
        case.slot_mapping)
    pk.kv_store(d["kn"], d["vn"], slots, kc, vc)
    plan = pk.decode_plan(case.num_seqs, 32, kc, case.max_context_len, 256, engine)
    fresh = pk.paged_decode(d["q"], kc, vc, bt, ctx, case.scale, plan=plan)
    ws = torch.full((plan.workspace_bytes,), 0xff, dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(d["q"])
    pk.paged_decode(d["q"], kc, vc, bt, ctx, case.scale, out=out, plan=plan, workspace=ws,
                    reuse_plan=True)
    torch.cuda.synchronize()
    assert pk.get_device_error() & pk.DEVERR_INTERNAL
    assert torch.count_nonzero(out) == 0
    again = pk.paged_decode(d["q"], kc, vc, bt, ctx, case.scale, plan=plan, workspace=ws)
    assert pk.get_device_error() == 0
    assert torch.equal(again, fresh)
    # the workspace now holds the plan of the 9-sequence batch; reuse it for the first 4
    small = pk.decode_plan(4, 32, kc, case.max_context_len, 256, engine)
    ws2 = torch.empty(max(plan.workspace_bytes, small.workspace_bytes), dtype=torch.uint8,
                      device="cuda")
    pk.paged_decode(d["q"], kc, vc, bt, ctx, case.scale, plan=plan, workspace=ws2)
    part = torch.zeros_like(d["q"][:4])
    pk.paged_decode(d["q"][:4], kc, vc, bt[:4], ctx[:4], case.scale, out=part, plan=small,
                    workspace=ws2, reuse_plan=True)
    torch.cuda.synchronize()
    assert pk.get_device_error() & pk.DEVERR_INTERNAL
    pk.paged_decode(d["q"][:4], kc, vc, bt[:4], ctx[:4], case.scale, out=part, plan=small,
                    workspace=ws2)
    assert pk.get_device_error() == 0
    assert torch.equal(part, pk.paged_decode(d["q"][:4], kc, vc, bt[:4], ctx[:4], case.scale,
                                             plan=small))


def test_reuse_needs_a_plan():
    with pytest.raises(ValueError):
        pk._reused(None)
