"""GPU: the decode step with the KV store fused in equals kv_store followed by paged_decode,
bit for bit (outputs and caches), and agrees with the oracle."""
import numpy as np
import pytest
import torch

import paged_kv_cache_496_b300 as pk
import workloads as W
from tests.gpu_util import assert_attn_close, dev_bf16, dev_i32, host_bits

pytestmark = pytest.mark.gpu


def _step_case(seed, B, Hq, Hkv, D, BS, lo, hi, zero_rows=()):
    """One decode step in engine form: row b of k_new / v_new / slot_mapping is sequence b."""
    rng = W.rng_for(seed, 7)
    ctx = W.uniform_int(rng, lo, hi, B)
    ctx[list(zero_rows)] = 0
    bt, nb = W.place_blocks(rng, ctx, BS, pool_blocks=int(W.blocks_needed(ctx, BS).sum()) + 2)
    slots = np.full(B, -1, np.int32)
    live = np.nonzero(ctx > 0)[0]
    slots[live] = W.slots_for_positions(bt, live, ctx[live] - 1, BS)
    shape = (nb, BS, Hkv, D)
    return dict(kc=W.normal_bf16(rng, shape), vc=W.normal_bf16(rng, shape),
                k=W.normal_bf16(rng, (B, Hkv, D)), v=W.normal_bf16(rng, (B, Hkv, D)),
                q=W.normal_bf16(rng, (B, Hq, D)), bt=bt, ctx=ctx.astype(np.int32), slots=slots,
                scale=1.0 / np.sqrt(D))


CASES = [  # (B, Hq, Hkv, D, BS, lo, hi, zero_rows, split)
    (6, 32, 8, 128, 256, 100, 900, (), 0),
    (7, 32, 8, 128, 16, 1, 700, (2, 5), 0),
    (5, 16, 8, 128, 64, 1, 400, (), -1),
    (4, 64, 8, 128, 16, 10, 3000, (1,), 256),   # G = 8, split
    (6, 8, 2, 64, 16, 1, 200, (0,), 0),        # D = 64
    (5, 8, 8, 128, 32, 1, 500, (), 0),         # G = 1 (one CTA per SM instance)
    (4, 8, 4, 64, 128, 5, 300, (3,), -1),      # D = 64, G = 2, auto split
    # the tensor-core engine (D = 128, block size >= 128, G >= 4) stores inside its own grid
    (8, 32, 8, 128, 128, 100, 900, (), 0),
    (5, 32, 8, 128, 256, 1, 300, (0, 3), -1),  # contexts of 0 and 1
    (4, 64, 8, 128, 128, 10, 3000, (1,), 256),  # G = 8, split: the last chunk stores
    (6, 32, 8, 128, 128, 120, 140, (), 0),     # ctx - 1 in a context's only tile
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B%d_H%d-%d_D%d_BS%d" % c[:5])
def test_fused_store_equals_store_then_decode(orc, case):
    B, Hq, Hkv, D, BS, lo, hi, zeros, split = case
    c = _step_case(11 + B + Hq, B, Hq, Hkv, D, BS, lo, hi, zeros)
    q, k, v = dev_bf16(c["q"]), dev_bf16(c["k"]), dev_bf16(c["v"])
    bt, ctx, slots = dev_i32(c["bt"]), dev_i32(c["ctx"]), dev_i32(c["slots"])
    mx = int(c["ctx"].max())
    # reference path: separate store, then decode
    kc1, vc1 = dev_bf16(c["kc"]), dev_bf16(c["vc"])
    pk.kv_store(k, v, slots, kc1, vc1)
    ref = pk.paged_decode(q, kc1, vc1, bt, ctx, c["scale"], max_context_len=mx, split_tokens=split)
    # fused
    kc2, vc2 = dev_bf16(c["kc"]), dev_bf16(c["vc"])
    out = pk.paged_decode_store(q, k, v, slots, kc2, vc2, bt, ctx, c["scale"], max_context_len=mx,
                                split_tokens=split)
    assert pk.get_device_error() == 0
    assert torch.equal(out, ref)
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2)
    rk, rv, _ = orc.kv_store(c["k"], c["v"], c["slots"], c["kc"], c["vc"])
    assert np.array_equal(host_bits(kc2), rk) and np.array_equal(host_bits(vc2), rv)
    want = orc.paged_decode(c["q"], rk, rv, c["bt"], c["ctx"], c["scale"])
    assert_attn_close(out, want, what=f"fused {case}")


@pytest.mark.parametrize("BS", [16, 128], ids=["cuda_core", "tensor_core"])
def test_fused_store_flags_a_slot_off_the_table(BS):
    c = _step_case(5, 3, 32, 8, 128, BS, 20, 40)
    slots = c["slots"].copy()
    slots[1] = (slots[1] + 1) % (c["kc"].shape[0] * BS)  # not the slot of position ctx-1
    kc, vc = dev_bf16(c["kc"]), dev_bf16(c["vc"])
    pk.get_device_error()
    pk.paged_decode_store(dev_bf16(c["q"]), dev_bf16(c["k"]), dev_bf16(c["v"]), dev_i32(slots), kc,
                          vc, dev_i32(c["bt"]), dev_i32(c["ctx"]), c["scale"], max_context_len=40)
    assert pk.get_device_error() & pk.DEVERR_BAD_SLOT
