"""GPU parity: chained xxhash64 block hashes, bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import paged_kv_cache_496_b300 as pk
import workloads as W
from tests.gpu_util import dev_i32

pytestmark = pytest.mark.gpu


def _gpu(tokens, cu, BS, max_blocks):
    out = pk.block_hashes(dev_i32(tokens), dev_i32(cu), BS, max_blocks)
    return out.cpu().numpy().view(np.uint64)


@pytest.mark.parametrize("BS", [256, 16, 2, 6])
def test_block_hashes_bit_exact(orc, BS):
    rng = W.rng_for(91, BS)
    lens = np.concatenate([[0, 1, BS - 1, BS, BS + 1, 3 * BS], rng.integers(1, 9 * BS, 40)])
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    tokens = rng.integers(0, 151936, size=int(cu[-1]), dtype=np.int64).astype(np.int32)
    max_blocks = int(lens.max() // BS)
    got = _gpu(tokens, cu, BS, max_blocks)
    ref, _ = orc.block_hashes(tokens, cu, BS, max_blocks)
    assert np.array_equal(got, ref)
    assert pk.get_device_error() == 0


def test_block_hashes_shared_prefix_and_clamp(orc):
    rng = W.rng_for(92, 0)
    BS = 256
    prefix = rng.integers(0, 1000, size=4 * BS).astype(np.int32)
    seqs = [np.concatenate([prefix, rng.integers(0, 1000, size=n).astype(np.int32)])
            for n in (300, 700, 1024)]
    tokens = np.concatenate(seqs)
    cu = np.concatenate([[0], np.cumsum([len(x) for x in seqs])]).astype(np.int32)
    got = _gpu(tokens, cu, BS, 4)
    assert (got == got[0]).all(), "the shared 4-block prefix hashes identically in every sequence"
    assert pk.get_device_error() == pk.DEVERR_CTX_CLAMPED
    ref, clamped = orc.block_hashes(tokens, cu, BS, 4)
    assert clamped == 3 and np.array_equal(got, ref)
