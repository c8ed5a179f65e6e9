"""The allocation-free decode entry point (pkv_paged_decode_static_ws), called through the C ABI.

It serves callers that cannot allocate device memory for the decode workspace (a process whose
GPU memory all belongs to its own pool allocator, or code that must not enter an allocator where
attention runs). Its workspace is a fixed array inside the library, shared by every call in a
CUDA context. This file is collected last so that a run stopping at the first failure has already
run every other test.
"""
import ctypes

import pytest
import torch

import paged_kv_cache_496_b300 as pk
import workloads as W
from tests.gpu_util import TOL, assert_attn_close, dev_bf16, dev_i32

pytestmark = pytest.mark.gpu

STATIC_WS_BYTES = 8 << 20  # PKV_STATIC_WS_BYTES

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


def _layer(case):
    """Device copies of a decode layer, with the new token stored through the workspace-free
    kv_store (it needs no workspace either)."""
    d = dict(kc=dev_bf16(case.k_cache), vc=dev_bf16(case.v_cache), q=dev_bf16(case.q),
             bt=dev_i32(case.block_tables), ctx=dev_i32(case.context_lens))
    pk.kv_store(dev_bf16(case.k_new), dev_bf16(case.v_new), dev_i32(case.slot_mapping),
                d["kc"], d["vc"])
    return d


def _oracle(orc, case):
    kc, vc, bad = orc.kv_store(case.k_new, case.v_new, case.slot_mapping, case.k_cache,
                               case.v_cache)
    assert bad == 0
    return orc.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, case.scale)


def test_static_workspace_calls_in_a_row(orc):
    """A sequence of calls on one stream with different batch sizes and plans: split (B=6), then
    unsplit with another batch (B=3), then split again with finer chunks (B=9). Each call runs
    twice in a row on the array the previous call left behind; each output is compared with the
    fp64 oracle and with the decode that takes a caller workspace."""
    assert torch.cuda.is_available()
    cases = [(W.random_decode_case(91, 6, 32, 8, 128, 16, 1, 2000), 256),
             (W.random_decode_case(93, 3, 32, 8, 128, 256, 100, 700), -1),
             (W.random_decode_case(94, 9, 16, 8, 128, 32, 300, 1500), 128)]
    pk.get_device_error()
    for case, split in cases:
        d = _layer(case)
        plan = pk.decode_plan(case.num_seqs, case.num_q_heads, d["kc"], case.max_context_len,
                              split)
        assert plan.workspace_bytes <= STATIC_WS_BYTES
        assert (plan.max_splits > 1) == (split > 0)
        ref = _oracle(orc, case)
        with_ws = pk.paged_decode(d["q"], d["kc"], d["vc"], d["bt"], d["ctx"], case.scale,
                                  plan=plan)
        for _ in range(2):
            out = torch.full_like(d["q"], float("nan"))
            assert _call(d, plan, out, case) == 0, pk.lib.pkv_last_error()
            torch.cuda.synchronize()
            assert_attn_close(out, ref, what=f"static workspace B={case.num_seqs} split={split}")
            err = (out.float() - with_ws.float()).abs().max().item()
            assert err <= TOL, err
        assert pk.get_device_error() == 0


def test_static_workspace_rejects_an_oversized_plan():
    case = W.random_decode_case(92, 2, 32, 8, 128, 16, 10, 20)
    d = dict(kc=dev_bf16(case.k_cache), vc=dev_bf16(case.v_cache), q=dev_bf16(case.q),
             bt=dev_i32(case.block_tables), ctx=dev_i32(case.context_lens))
    big = pk.decode_plan(4096, 32, d["kc"], 65536, 128)  # ~2 GB of chunk partials
    assert big.workspace_bytes > STATIC_WS_BYTES
    out = torch.zeros_like(d["q"])
    assert _call(d, big, out, case) == pk.PKV_ERR_WORKSPACE_TOO_SMALL
    assert b"workspace" in pk.lib.pkv_last_error()
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
