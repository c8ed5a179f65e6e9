"""GPU parity: copy-on-write block copies and swap gather/scatter, bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import paged_kv_cache_496_b300 as pk
import workloads as W
from tests.gpu_util import dev_bf16, dev_i32, host_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("BS,Hkv,D", [(256, 8, 128), (16, 8, 128), (16, 2, 64)])
def test_block_moves_bit_exact(orc, BS, Hkv, D):
    rng = W.rng_for(81, BS, D)
    NB = 40
    kc = W.normal_bf16(rng, (NB, BS, Hkv, D))
    vc = W.normal_bf16(rng, (NB, BS, Hkv, D))
    perm = rng.permutation(NB).astype(np.int32)
    pairs = np.stack([perm[:12], perm[12:24]], axis=1).astype(np.int32)  # disjoint src / dst
    kd, vd = dev_bf16(kc), dev_bf16(vc)
    pk.copy_blocks(kd, vd, dev_i32(pairs))
    rk, rv, bad = orc.copy_blocks(kc, vc, pairs)
    assert bad == 0
    assert np.array_equal(host_bits(kd), rk) and np.array_equal(host_bits(vd), rv)
    ids = perm[24:34]
    gk, gv = pk.gather_blocks(kd, vd, dev_i32(ids))
    ok, ov, _ = orc.gather_blocks(rk, rv, ids)
    assert np.array_equal(host_bits(gk), ok) and np.array_equal(host_bits(gv), ov)
    dst = perm[34:40].copy()
    pk.scatter_blocks(gk[:6].contiguous(), gv[:6].contiguous(), dev_i32(dst), kd, vd)
    sk, sv, _ = orc.scatter_blocks(ok[:6], ov[:6], dst, rk, rv)
    assert np.array_equal(host_bits(kd), sk) and np.array_equal(host_bits(vd), sv)
    assert pk.get_device_error() == 0


def test_block_moves_flag_bad_ids():
    kd = torch.zeros((4, 16, 2, 64), dtype=torch.bfloat16, device="cuda")
    vd = torch.zeros_like(kd)
    pk.get_device_error()
    pk.copy_blocks(kd, vd, dev_i32(np.array([[0, 9], [1, 2]], np.int32)))
    assert pk.get_device_error() == pk.DEVERR_BAD_BLOCK
    pk.gather_blocks(kd, vd, dev_i32(np.array([-1, 3], np.int32)))
    assert pk.get_device_error() == pk.DEVERR_BAD_BLOCK


def test_swap_out_and_in_preserves_decode():
    """Swapping a sequence's blocks out and back into other physical blocks (tables updated)
    leaves its decode output bit-identical."""
    case = W.random_decode_case(82, 3, 32, 8, 128, 16, 100, 200, extra_pool=40)
    kd, vd = dev_bf16(case.k_cache), dev_bf16(case.v_cache)
    pk.kv_store(dev_bf16(case.k_new), dev_bf16(case.v_new), dev_i32(case.slot_mapping), kd, vd)
    q, ctx = dev_bf16(case.q), dev_i32(case.context_lens)
    a = pk.paged_decode(q, kd, vd, dev_i32(case.block_tables), ctx, case.scale,
                        max_context_len=case.max_context_len, split_tokens=-1)
    used = np.unique(case.block_tables[case.block_tables >= 0])
    free = np.setdiff1d(np.arange(case.num_blocks), used)
    b = 1
    n = int(W.blocks_needed(case.context_lens[b:b + 1], 16)[0])
    old = case.block_tables[b, :n].copy()
    new = free[:n].astype(np.int32)
    gk, gv = pk.gather_blocks(kd, vd, dev_i32(old))
    pk.scatter_blocks(gk, gv, dev_i32(new), kd, vd)
    bt = case.block_tables.copy()
    bt[b, :n] = new
    c = pk.paged_decode(q, kd, vd, dev_i32(bt), ctx, case.scale,
                        max_context_len=case.max_context_len, split_tokens=-1)
    assert torch.equal(a, c)
    assert pk.get_device_error() == 0
