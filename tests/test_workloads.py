"""Seeded input generators: ranges, block placement and bf16 rounding."""
import numpy as np
import torch

import workloads as W


def test_bf16_rounding_matches_torch():
    rng = W.rng_for(0, 0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -0.0, 65504.0], np.float32)])
    ours = W.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_decode_lengths_ranges():
    for name in ("qwen3_0p6b_decode", "qwen3_8b_decode"):
        ctx = W.decode_lengths(name)
        assert len(ctx) == W.WORKLOADS[name].num_seqs
        assert ctx.min() >= 200 and ctx.max() <= 2048
        assert abs(ctx.mean() - 1124) < 4 * 378 / np.sqrt(len(ctx))  # 4 standard errors
    long = W.decode_lengths("long_splitk_decode")
    assert (long[:4] == 32768).all() and long[4:].min() >= 100 and long[4:].max() <= 1024
    tiny = W.decode_lengths("tiny_decode")
    assert tiny.min() >= 1 and tiny.max() <= 64


def test_block_placement_is_a_partition():
    rng = W.rng_for(1, 2)
    ctx = W.decode_context_lengths(rng, 300)
    bt, nb = W.place_blocks(rng, ctx, 256)
    used = bt[bt >= 0]
    assert len(used) == nb == int(W.blocks_needed(ctx, 256).sum())
    assert len(np.unique(used)) == nb and used.min() == 0 and used.max() == nb - 1
    for b in range(len(ctx)):
        n = int(W.blocks_needed(ctx[b:b + 1], 256)[0])
        assert (bt[b, :n] >= 0).all() and (bt[b, n:] == -1).all()


def test_tiny_case_slots():
    c = W.tiny_decode_case()
    assert c.num_blocks == 32 and c.slot_mapping.shape[0] == int(c.context_lens.sum()) + 2
    assert (c.slot_mapping[-2:] == -1).all()
    valid = c.slot_mapping[c.slot_mapping >= 0]
    assert len(np.unique(valid)) == len(valid)


def test_ladder():
    assert W.GRAPH_LADDER == [1, 2, 4, 8, 16, 32, 64, 128, 256, 512]
    assert W.ladder_bucket(1) == 1 and W.ladder_bucket(17) == 32 and W.ladder_bucket(512) == 512
    assert W.ladder_padded_size(1024) == 1024 and W.ladder_padded_size(700) == 768
    n = W.live_batch_size("qwen3_8b_decode")
    assert 513 <= n <= 1023


def test_prefix_case_shares_blocks():
    c = W.prefix_prefill_case(4, 8, 512, 100, 300, 4, 2, 16, 256)
    assert (c.block_tables[:, :2] == c.block_tables[0, :2]).all()
    assert (np.diff(c.cu_seqlens_k) - np.diff(c.cu_seqlens_q) == 512).all()
    rows = c.slot_mapping
    assert len(np.unique(rows)) == len(rows)
    prefix_rows = (c.block_tables[0, :2, None] * 256 + np.arange(256)).ravel()
    assert not np.isin(rows, prefix_rows).any()
