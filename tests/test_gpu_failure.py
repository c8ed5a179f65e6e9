"""Failure detection on the GPU without faulting it: a pipeline wait that can never complete gives
up after its limit, reports PKV_DEVERR_TIMEOUT through the device error word, and the context keeps
working (a decode right after is still correct)."""
import time

import pytest
import torch

import paged_kv_cache_496_b300 as pk
import workloads as W
from tests.gpu_util import assert_attn_close, dev_bf16, dev_i32

pytestmark = pytest.mark.gpu


def test_stuck_wait_times_out_and_context_survives(orc):
    assert torch.cuda.is_available()
    pk.get_device_error()
    t0 = time.time()
    flags = pk.selftest_bounded_wait()
    elapsed = time.time() - t0
    assert flags == pk.DEVERR_TIMEOUT
    assert 0.5 < elapsed < 30.0
    case = W.random_decode_case(71, 4, 32, 8, 128, 16, 10, 300)
    kc, vc = dev_bf16(case.k_cache), dev_bf16(case.v_cache)
    pk.kv_store(dev_bf16(case.k_new), dev_bf16(case.v_new), dev_i32(case.slot_mapping), kc, vc)
    out = pk.paged_decode(dev_bf16(case.q), kc, vc, dev_i32(case.block_tables),
                          dev_i32(case.context_lens), case.scale,
                          max_context_len=case.max_context_len)
    assert pk.get_device_error() == 0
    rk, rv, _ = orc.kv_store(case.k_new, case.v_new, case.slot_mapping, case.k_cache,
                             case.v_cache)
    ref = orc.paged_decode(case.q, rk, rv, case.block_tables, case.context_lens, case.scale)
    assert_attn_close(out, ref, what="decode after a timed-out wait")
