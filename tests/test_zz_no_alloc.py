"""The allocation-free decode entry point (pkv_paged_decode_static_ws), called through the C ABI.

It serves callers that cannot allocate device memory for the decode workspace (a process whose
GPU memory all belongs to its own pool allocator, or code that must not enter an allocator where
attention runs). Its workspace is a fixed array inside the library. This file is collected last so
that a run stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_496_b300 as pk
import workloads as W
from tests.gpu_util import TOL, dev_bf16, dev_i32

pytestmark = pytest.mark.gpu

_fn = pk.lib.pkv_paged_decode_static_ws
_fn.restype = ctypes.c_int
_fn.argtypes = [ctypes.c_void_p] * 3 + [pk.CacheDesc, ctypes.c_void_p, ctypes.c_int32,
                                         ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_float, ctypes.POINTER(pk.DecodePlan),
                                         ctypes.c_void_p, ctypes.c_void_p]


def _call(d, plan, out, case):
    return _fn(d["q"].data_ptr(), d["kc"].data_ptr(), d["vc"].data_ptr(),
               pk.CacheDesc(*d["kc"].shape), d["bt"].data_ptr(), d["bt"].shape[1],
               d["ctx"].data_ptr(), case.num_seqs, case.num_q_heads, case.scale,
               ctypes.byref(plan), out.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("split", [-1, 256], ids=["unsplit", "split"])
def test_static_workspace_decode_matches_workspace_decode(split):
    assert torch.cuda.is_available()
    case = W.random_decode_case(91, 6, 32, 8, 128, 16, 1, 2000)
    d = dict(kc=dev_bf16(case.k_cache), vc=dev_bf16(case.v_cache), q=dev_bf16(case.q),
             bt=dev_i32(case.block_tables), ctx=dev_i32(case.context_lens))
    pk.kv_store(dev_bf16(case.k_new), dev_bf16(case.v_new), dev_i32(case.slot_mapping),
                d["kc"], d["vc"])
    plan = pk.decode_plan(case.num_seqs, case.num_q_heads, d["kc"], case.max_context_len, split)
    assert plan.workspace_bytes <= 8 << 20  # PKV_STATIC_WS_BYTES
    ref = pk.paged_decode(d["q"], d["kc"], d["vc"], d["bt"], d["ctx"], case.scale, plan=plan)
    for _ in range(2):  # the second call reuses the array the first one left behind
        out = torch.full_like(d["q"], float("nan"))
        assert _call(d, plan, out, case) == 0, pk.lib.pkv_last_error()
        torch.cuda.synchronize()
        err = (out.float() - ref.float()).abs().max().item()
        assert err <= TOL, err
    assert pk.get_device_error() == 0


def test_static_workspace_rejects_an_oversized_plan():
    case = W.random_decode_case(92, 2, 32, 8, 128, 16, 10, 20)
    d = dict(kc=dev_bf16(case.k_cache), vc=dev_bf16(case.v_cache), q=dev_bf16(case.q),
             bt=dev_i32(case.block_tables), ctx=dev_i32(case.context_lens))
    big = pk.decode_plan(4096, 32, d["kc"], 65536, 128)  # ~2 GB of chunk partials
    assert big.workspace_bytes > 8 << 20
    out = torch.zeros_like(d["q"])
    assert _call(d, big, out, case) == pk.PKV_ERR_WORKSPACE_TOO_SMALL
    assert b"workspace" in pk.lib.pkv_last_error()
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
