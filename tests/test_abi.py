"""The C-ABI library on the CPU: it loads, exports every symbol the header declares, and its
host-side logic (decode plan, argument validation) behaves as documented. No kernel is launched:
every call here fails validation (or is a no-op) before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


@pytest.fixture(scope="module")
def pk():
    import paged_kv_cache_496_b300 as pk
    return pk


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"PKV_API\s+[\w\s\*]+?\b(pkv_\w+)\s*\(", text)


def test_header_declares_the_three_operations():
    names = declared_symbols()
    for n in ("pkv_kv_store", "pkv_paged_decode", "pkv_paged_prefill", "pkv_decode_plan_make",
              "pkv_get_device_error", "pkv_status_string", "pkv_last_error", "pkv_version"):
        assert n in names


def test_library_exports_every_declared_symbol(pk):
    out = subprocess.run(["nm", "-D", "--defined-only", pk.LIBRARY], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(pkv_\w+)", out))
    for n in declared_symbols():
        assert n in exported, f"{n} not exported"
        assert getattr(pk.lib, n) is not None


def test_status_strings_and_version(pk):
    assert pk.lib.pkv_version() == pk.ABI_VERSION == 202
    assert pk.lib.pkv_status_string(0) == b"ok"
    assert pk.lib.pkv_status_string(-3) == b"workspace too small"
    assert pk.lib.pkv_status_string(12345) == b"unknown status"


def _desc(pk, nb=64, bs=16, hkv=8, d=128):
    return pk.CacheDesc(nb, bs, hkv, d)


def test_decode_plan_no_split_for_short_contexts(pk):
    plan = pk.DecodePlan()
    assert pk.lib.pkv_decode_plan_make(1024, 32, _desc(pk, 5000, 256), 400, 0,
                                       ctypes.byref(plan)) == 0
    assert plan.max_splits == 1 and plan.auto_split == 0 and plan.split_tokens == 512
    assert plan.workspace_bytes >= 256 + 1024 * 8


@pytest.mark.parametrize("bs,hkv,d,hq,engine", [
    (256, 8, 128, 32, "TENSOR_CORE"),   # Qwen3-8B shape
    (256, 8, 128, 64, "TENSOR_CORE"),   # G = 8
    (128, 4, 128, 16, "TENSOR_CORE"),
    (256, 8, 128, 16, "CUDA_CORE"),     # G = 2 (Qwen3-0.6B shape)
    (256, 8, 128, 8, "CUDA_CORE"),      # G = 1
    (64, 8, 128, 32, "CUDA_CORE"),      # blocks below 128 rows
    (16, 8, 128, 32, "CUDA_CORE"),
    (256, 8, 64, 32, "CUDA_CORE"),      # head_dim 64
])
def test_decode_plan_engine_default(pk, bs, hkv, d, hq, engine):
    """pkv_decode_plan_make picks the tensor-core engine for head_dim 128, block_size >= 128 and
    G >= 4, else the CUDA-core engine; split settings do not change the choice."""
    plan = pk.DecodePlan()
    for B, ctx, hint in ((1024, 2048, 0), (1024, 2048, -1), (64, 32768, 0), (8, 100, 256)):
        assert pk.lib.pkv_decode_plan_make(B, hq, _desc(pk, 5000, bs, hkv, d), ctx, hint,
                                           ctypes.byref(plan)) == 0
        assert plan.engine == getattr(pk, "DECODE_ENGINE_" + engine)
    assert pk.decode_plan.__defaults__[-1] is None


def test_decode_plan_auto_and_fixed(pk):
    plan = pk.DecodePlan()
    assert pk.lib.pkv_decode_plan_make(64, 32, _desc(pk, 9000, 16), 32768, 0,
                                       ctypes.byref(plan)) == 0
    assert plan.auto_split == 1 and plan.split_tokens == 512 and plan.max_splits == 64
    # partials: [B, splits, Hq, D] fp32 + (m, l) per 64-dim slice + counters + items + header
    assert plan.workspace_bytes >= 64 * 64 * 32 * 128 * 4
    assert pk.lib.pkv_decode_plan_make(64, 32, _desc(pk, 9000, 16), 32768, 1000,
                                       ctypes.byref(plan)) == 0
    assert plan.auto_split == 0 and plan.split_tokens == 1024 and plan.max_splits == 32
    assert pk.lib.pkv_decode_plan_make(64, 32, _desc(pk, 9000, 16), 32768, -1,
                                       ctypes.byref(plan)) == 0
    assert plan.max_splits == 1 and plan.split_tokens == 32768


@pytest.mark.parametrize("desc,hq,status", [
    ((64, 16, 8, 96), 32, -2),    # head_dim 96 unsupported
    ((64, 24, 8, 128), 32, -2),   # block size not a power of two
    ((64, 512, 8, 128), 32, -2),  # block size above 256
    ((64, 16, 8, 128), 12, -1),   # Hq not a multiple of Hkv
    ((64, 16, 2, 128), 32, -2),   # group size 16 unsupported
    ((0, 16, 8, 128), 32, -1),    # empty pool
])
def test_decode_plan_rejects_shapes(pk, desc, hq, status):
    plan = pk.DecodePlan()
    assert pk.lib.pkv_decode_plan_make(4, hq, pk.CacheDesc(*desc), 100, 0,
                                       ctypes.byref(plan)) == status
    assert pk.lib.pkv_last_error() != b""


def test_kv_store_validation_without_launch(pk):
    d = _desc(pk)
    assert pk.lib.pkv_kv_store(None, None, None, 0, None, None, d, None) == 0  # no-op
    assert pk.lib.pkv_kv_store(None, None, None, 5, None, None, d, None) == -1
    assert pk.lib.pkv_kv_store(256, 256, 256, -1, 256, 256, d, None) == -1
    assert pk.lib.pkv_kv_store(256, 256, 256, 5, 264, 256, d, None) == -1  # misaligned cache
    assert pk.lib.pkv_kv_store(256, 256, 256, 5, 256, 256, _desc(pk, d=80), None) == -2


def test_decode_validation_without_launch(pk):
    d = _desc(pk)
    plan = pk.DecodePlan()
    assert pk.lib.pkv_decode_plan_make(4, 32, d, 100, 0, ctypes.byref(plan)) == 0
    args = dict(q=256, kc=256, vc=256, bt=256, mb=8, cl=256, B=4, Hq=32, scale=0.1,
                out=256, ws=4096, wsb=plan.workspace_bytes)

    def call(**kw):
        a = dict(args, **kw)
        return pk.lib.pkv_paged_decode(a["q"], a["kc"], a["vc"], d, a["bt"], a["mb"], a["cl"],
                                       a["B"], a["Hq"], a["scale"], ctypes.byref(plan),
                                       a["out"], a["ws"], a["wsb"], None)

    assert call(B=0) == 0                       # empty batch: no-op
    assert call(q=None) == -1                   # null pointer
    assert call(ws=4096 + 16) == -1             # workspace not 256-byte aligned
    assert call(mb=0) == -1                     # empty block table rows
    assert call(scale=float("nan")) == -1       # non-finite scale
    assert call(wsb=plan.workspace_bytes - 1) == -3
    assert b"workspace" in pk.lib.pkv_last_error()
    assert call(Hq=12) == -1
    plan.engine = 7                               # no such engine
    assert call() == -1
    plan.engine = pk.DECODE_ENGINE_TENSOR_CORE    # head_dim 64: no tensor-core instance
    d64 = _desc(pk, d=64)
    assert pk.lib.pkv_paged_decode(256, 256, 256, d64, 256, 8, 256, 4, 32, 0.1, ctypes.byref(plan),
                                   256, 4096, plan.workspace_bytes, None) == -2
    assert b"tensor-core" in pk.lib.pkv_last_error()


def test_prefill_validation_without_launch(pk):
    d = _desc(pk)
    ws, wsb = 4096, pk.PREFILL_WORKSPACE_BYTES
    assert pk.lib.pkv_paged_prefill(None, None, None, None, None, 0, 0, 0, None, 0, None, None,
                                    d, 32, 0.1, None, None, 0, None) in (0, -2)
    assert pk.lib.pkv_paged_prefill(None, 256, 256, 256, 256, 2, 10, 5, None, 0, None, None,
                                    d, 32, 0.1, 256, ws, wsb, None) in (-1, -2)
    # a missing, misaligned or short workspace is refused before anything is launched
    assert pk.lib.pkv_paged_prefill(256, 256, 256, 256, 256, 2, 10, 5, None, 0, None, None,
                                    d, 32, 0.1, 256, None, wsb, None) == -1
    assert b"workspace" in pk.lib.pkv_last_error()
    assert pk.lib.pkv_paged_prefill(256, 256, 256, 256, 256, 2, 10, 5, None, 0, None, None,
                                    d, 32, 0.1, 256, ws + 8, wsb, None) == -1
    assert pk.lib.pkv_paged_prefill(256, 256, 256, 256, 256, 2, 10, 5, None, 0, None, None,
                                    d, 32, 0.1, 256, ws, wsb - 1, None) == -3
    assert b"workspace_bytes" in pk.lib.pkv_last_error()


def test_prefill_workspace_bytes_for_dense_numbering(pk):
    """The prefill counters (256 B), then two ints per sequence (first item id, sequence at each
    position) and one more, rounded to 256 B."""
    f = pk.lib.pkv_prefill_workspace_bytes
    assert f(-1) == 256
    assert f(0) == 512
    assert f(31) == 512
    assert f(32) == 768
    assert f(64) == 1024
    assert f(1000) == 256 + 8192
    assert pk.prefill_workspace_bytes(64) == f(64)


def test_binding_refuses_cpu_tensors(pk):
    import torch
    k = torch.zeros(4, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pk.kv_store(k, k, torch.zeros(4, dtype=torch.int32), torch.zeros(2, 16, 8, 128,
                    dtype=torch.bfloat16), torch.zeros(2, 16, 8, 128, dtype=torch.bfloat16))
