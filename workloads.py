"""Seeded synthetic inputs for the paged KV-cache hot path.

This module is shared by the CPU oracle tests, the CUDA parity tests and the benchmark. It holds
none of the method's arithmetic: it only draws lengths, block placements and N(0,1) values, and
rounds them to bf16 bit patterns (round-to-nearest-even) so that every consumer sees the same bytes.

Workload shapes follow the benchmarks described on the source pages:
  * "DeepSeek研究员1200行代码复刻vLLM，H800硬件实测性能反超原版" (QbitAI), benchmark paragraphs:
    RTX 4070 with Qwen3-0.6B, 256 sequences; H800 with Qwen3-8B, 1024 sequences; input and output
    lengths each drawn at random from 100-1024 tokens.
  * "nano-vllm 深度分析报告", table "关键设计决策": block_size 256 (vLLM uses 16);
    section "创新之处": CUDA graphs captured for batch sizes [1, 2, 4, 8, 16, ..., 512], the live
    batch is rounded up; table "可复用的模式与技巧": padded slots carry slot_mapping -1.
  * same page, "创新之处": prefix-cache hits reuse (share) physical blocks across sequences.

Readings taken where the pages leave a step open (each one is listed in the design notes):
  * "random in 100-1024" is the discrete uniform distribution on {100, ..., 1024}, drawn
    independently for the input length and for the number of tokens generated so far.
  * the CUDA-graph ladder "[1,2,4,8,16,...,512]" is the powers of two up to 512.
  * physical blocks are placed by a seeded random permutation of a pool sized exactly to fit.
  * a decode step stores the newest token (position ctx-1) through slot_mapping and then attends
    over all ctx tokens.

Host arrays are numpy (bf16 as uint16 bit patterns). Device-sized pools for the large decode
workloads are drawn on the GPU with a seeded torch generator (`fill_normal_bf16_`), because a
189 GB cache cannot be drawn on the host; the oracle then reads back only sampled blocks.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

# ----------------------------------------------------------------------------------------------
# Workload definitions
# ----------------------------------------------------------------------------------------------


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "decode" or "prefill"
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_layers: int
    seed: int
    description: str

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def kv_bytes_per_token(self) -> int:
        """K and V bytes one token occupies in one layer's cache (bf16)."""
        return 2 * self.num_kv_heads * self.head_dim * 2


WORKLOADS = {
    "tiny_decode": Workload(
        "tiny_decode", "decode", 4, 4, 2, 64, 16, 1, 1,
        "4 sequences, context U{1..64}, 4 q heads / 2 kv heads, head_dim 64, block_size 16, "
        "pool of 32 blocks, every token written through slot_mapping with 2 extra -1 slots"),
    "qwen3_0p6b_decode": Workload(
        "qwen3_0p6b_decode", "decode", 256, 16, 8, 128, 256, 28, 2,
        "256 sequences, context = input U{100..1024} + generated U{100..1024}, 16/8 heads, "
        "head_dim 128, block_size 256, 28 layer caches, one new token stored per sequence"),
    "qwen3_8b_decode": Workload(
        "qwen3_8b_decode", "decode", 1024, 32, 8, 128, 256, 36, 3,
        "1024 sequences, context = input U{100..1024} + generated U{100..1024}, 32/8 heads, "
        "head_dim 128, block_size 256, 36 layer caches, one new token stored per sequence"),
    "prefix_prefill": Workload(
        "prefix_prefill", "prefill", 64, 32, 8, 128, 256, 1, 4,
        "64 sequences sharing one 1024-token prefix (4 shared blocks of 256), each followed by "
        "U{100..1024} new tokens, 32/8 heads, head_dim 128, varlen causal prefill"),
    "long_splitk_decode": Workload(
        "long_splitk_decode", "decode", 64, 32, 8, 128, 16, 1, 5,
        "4 sequences of context 32768 plus 60 of context U{100..1024}, 32/8 heads, head_dim 128, "
        "block_size 16, random block placement"),
}

GRAPH_LADDER = [1 << i for i in range(10)]  # 1, 2, 4, ..., 512


# ----------------------------------------------------------------------------------------------
# Elementary draws
# ----------------------------------------------------------------------------------------------


def rng_for(seed: int, *stream: int) -> np.random.Generator:
    """A PCG64 generator for (seed, sub-stream ...); sub-streams separate layers and roles."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *stream])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + bias) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    """N(0, scale^2) values rounded to bf16 bit patterns."""
    return f32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32) * np.float32(scale))


def uniform_int(rng: np.random.Generator, lo: int, hi: int, n: int) -> np.ndarray:
    """n draws from the discrete uniform distribution on {lo, ..., hi} (inclusive)."""
    return rng.integers(lo, hi + 1, size=n, dtype=np.int64).astype(np.int32)


def decode_context_lengths(rng: np.random.Generator, n: int) -> np.ndarray:
    """Context = input length + tokens generated so far, each U{100..1024}."""
    return (uniform_int(rng, 100, 1024, n) + uniform_int(rng, 100, 1024, n)).astype(np.int32)


def blocks_needed(lengths: np.ndarray, block_size: int) -> np.ndarray:
    return ((np.asarray(lengths, dtype=np.int64) + block_size - 1) // block_size).astype(np.int64)


def place_blocks(rng: np.random.Generator, lengths: np.ndarray, block_size: int,
                 pool_blocks: Optional[int] = None, max_blocks: Optional[int] = None):
    """Assign physical blocks by a seeded random permutation of the pool, in sequence order.

    Returns (block_tables [B, max_blocks] int32 padded with -1, pool_blocks).
    """
    need = blocks_needed(lengths, block_size)
    total = int(need.sum())
    if pool_blocks is None:
        pool_blocks = max(total, 1)
    if pool_blocks < total:
        raise ValueError("pool too small")
    if max_blocks is None:
        max_blocks = int(max(need.max(initial=0), 1))
    perm = rng.permutation(pool_blocks).astype(np.int32)
    bt = np.full((len(lengths), max_blocks), -1, dtype=np.int32)
    pos = 0
    for b, nb in enumerate(need):
        bt[b, :nb] = perm[pos:pos + nb]
        pos += nb
    return bt, pool_blocks


def slots_for_positions(block_tables: np.ndarray, seq: np.ndarray, pos: np.ndarray,
                        block_size: int) -> np.ndarray:
    """Slot of logical position pos of sequence seq: physical block * block_size + offset."""
    seq = np.asarray(seq, dtype=np.int64)
    pos = np.asarray(pos, dtype=np.int64)
    blk = block_tables[seq, pos // block_size].astype(np.int64)
    return (blk * block_size + pos % block_size).astype(np.int32)


def ladder_bucket(n: int) -> int:
    """Smallest CUDA-graph batch size of the ladder that holds n (n <= 512)."""
    for b in GRAPH_LADDER:
        if b >= n:
            return b
    raise ValueError("batch larger than the largest graph size")


def ladder_padded_size(n: int) -> int:
    """Batch size after splitting into chunks of at most 512 and rounding the last one up."""
    full, rest = divmod(n, GRAPH_LADDER[-1])
    return full * GRAPH_LADDER[-1] + (ladder_bucket(rest) if rest else 0)


# ----------------------------------------------------------------------------------------------
# Host cases (numpy), small enough for the oracle
# ----------------------------------------------------------------------------------------------


@dataclasses.dataclass
class DecodeCase:
    """One layer of a decode step. bf16 arrays hold uint16 bit patterns."""
    num_blocks: int
    block_size: int
    num_kv_heads: int
    head_dim: int
    num_q_heads: int
    k_cache: np.ndarray      # [NB, BS, Hkv, D] uint16, content before the store
    v_cache: np.ndarray
    k_new: np.ndarray        # [T, Hkv, D] uint16, rows to store
    v_new: np.ndarray
    slot_mapping: np.ndarray  # [T] int32, -1 = padding
    q: np.ndarray            # [B, Hq, D] uint16
    block_tables: np.ndarray  # [B, max_blocks] int32
    context_lens: np.ndarray  # [B] int32
    scale: float

    @property
    def num_seqs(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max(initial=0))


def tiny_decode_case(seed: int = 1, q_scale: float = 1.0) -> DecodeCase:
    """Tiny decode check: every token of 4 sequences is written through slot_mapping."""
    w = WORKLOADS["tiny_decode"]
    rng = rng_for(seed, 0)
    B, Hq, Hkv, D, BS = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
    ctx = uniform_int(rng, 1, 64, B)
    bt, nb = place_blocks(rng, ctx, BS, pool_blocks=32, max_blocks=64 // BS)
    seq = np.concatenate([np.full(c, b) for b, c in enumerate(ctx)])
    pos = np.concatenate([np.arange(c) for c in ctx])
    slots = np.concatenate([slots_for_positions(bt, seq, pos, BS),
                            np.full(2, -1, dtype=np.int32)]).astype(np.int32)
    T = len(slots)
    return DecodeCase(
        num_blocks=nb, block_size=BS, num_kv_heads=Hkv, head_dim=D, num_q_heads=Hq,
        k_cache=normal_bf16(rng, (nb, BS, Hkv, D)), v_cache=normal_bf16(rng, (nb, BS, Hkv, D)),
        k_new=normal_bf16(rng, (T, Hkv, D)), v_new=normal_bf16(rng, (T, Hkv, D)),
        slot_mapping=slots, q=normal_bf16(rng, (B, Hq, D), q_scale), block_tables=bt,
        context_lens=ctx.astype(np.int32), scale=1.0 / math.sqrt(D))


def random_decode_case(seed: int, num_seqs: int, num_q_heads: int, num_kv_heads: int,
                       head_dim: int, block_size: int, ctx_lo: int, ctx_hi: int,
                       extra_pool: int = 0, pad_slots: int = 0, q_scale: float = 1.0,
                       context_lens: Optional[np.ndarray] = None) -> DecodeCase:
    """A decode layer: the pool holds positions 0..ctx-2, the new token (ctx-1) is stored."""
    rng = rng_for(seed, 1)
    if context_lens is None:
        context_lens = uniform_int(rng, ctx_lo, ctx_hi, num_seqs)
    ctx = np.asarray(context_lens, dtype=np.int32)
    need = int(blocks_needed(ctx, block_size).sum())
    bt, nb = place_blocks(rng, ctx, block_size, pool_blocks=need + extra_pool)
    live = np.nonzero(ctx > 0)[0]
    slots = slots_for_positions(bt, live, ctx[live] - 1, block_size)
    slots = np.concatenate([slots, np.full(pad_slots, -1, dtype=np.int32)]).astype(np.int32)
    T = len(slots)
    shape = (nb, block_size, num_kv_heads, head_dim)
    return DecodeCase(
        num_blocks=nb, block_size=block_size, num_kv_heads=num_kv_heads, head_dim=head_dim,
        num_q_heads=num_q_heads, k_cache=normal_bf16(rng, shape), v_cache=normal_bf16(rng, shape),
        k_new=normal_bf16(rng, (T, num_kv_heads, head_dim)),
        v_new=normal_bf16(rng, (T, num_kv_heads, head_dim)), slot_mapping=slots,
        q=normal_bf16(rng, (num_seqs, num_q_heads, head_dim), q_scale), block_tables=bt,
        context_lens=ctx, scale=1.0 / math.sqrt(head_dim))


def decode_lengths(workload: str, live: Optional[int] = None) -> np.ndarray:
    """Context lengths of a decode workload (seeded by the workload's seed)."""
    w = WORKLOADS[workload]
    rng = rng_for(w.seed, 100)
    if workload == "long_splitk_decode":
        return np.concatenate([np.full(4, 32768, dtype=np.int32),
                               uniform_int(rng, 100, 1024, 60)]).astype(np.int32)
    if workload == "tiny_decode":
        return uniform_int(rng, 1, 64, w.num_seqs)
    n = w.num_seqs if live is None else live
    return decode_context_lengths(rng, n)


def live_batch_size(workload: str) -> int:
    """A seeded live batch below the full size (sequences finish at different times)."""
    w = WORKLOADS[workload]
    rng = rng_for(w.seed, 101)
    return int(w.num_seqs - uniform_int(rng, 1, 511, 1)[0])


@dataclasses.dataclass
class PrefillCase:
    num_blocks: int
    block_size: int
    num_kv_heads: int
    head_dim: int
    num_q_heads: int
    k_cache: np.ndarray      # [NB, BS, Hkv, D] uint16, holds the shared prefix before the store
    v_cache: np.ndarray
    q: np.ndarray            # [Tq, Hq, D]
    k: np.ndarray            # [Tq, Hkv, D] new tokens
    v: np.ndarray
    cu_seqlens_q: np.ndarray  # [B+1] int32
    cu_seqlens_k: np.ndarray  # [B+1] int32
    block_tables: np.ndarray  # [B, max_blocks] int32 (prefix blocks shared by every row)
    slot_mapping: np.ndarray  # [Tq] int32, slots of the new tokens
    scale: float

    @property
    def num_seqs(self) -> int:
        return len(self.cu_seqlens_q) - 1

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q)

    @property
    def k_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_k)


def prefix_prefill_case(seed: int, num_seqs: int, prefix_len: int, suffix_lo: int, suffix_hi: int,
                        num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                        q_scale: float = 1.0, suffix_lens: Optional[np.ndarray] = None,
                        shared: bool = True) -> PrefillCase:
    """Varlen prefill where every sequence starts with the same cached prefix.

    With shared=True the prefix occupies the same physical blocks in every block table (a
    prefix-cache hit); with shared=False each sequence holds its own copy of the prefix bytes in
    distinct blocks. prefix_len must be a multiple of block_size (hits cover whole blocks).
    """
    if prefix_len % block_size:
        raise ValueError("prefix must cover whole blocks")
    rng = rng_for(seed, 2)       # lengths and values
    place = rng_for(seed, 3)     # physical placement and background cache content
    B = num_seqs
    ql = (np.asarray(suffix_lens, dtype=np.int32) if suffix_lens is not None
          else uniform_int(rng, suffix_lo, suffix_hi, B))
    kl = ql + prefix_len
    pb = prefix_len // block_size
    suffix_blocks = blocks_needed(ql, block_size)
    n_prefix_phys = pb if shared else pb * B
    nb = int(n_prefix_phys + suffix_blocks.sum())
    perm = place.permutation(nb).astype(np.int32)
    max_blocks = int(pb + suffix_blocks.max(initial=0))
    bt = np.full((B, max(max_blocks, 1)), -1, dtype=np.int32)
    prefix_phys = perm[:n_prefix_phys]
    pos = n_prefix_phys
    for b in range(B):
        bt[b, :pb] = prefix_phys if shared else prefix_phys[b * pb:(b + 1) * pb]
        bt[b, pb:pb + suffix_blocks[b]] = perm[pos:pos + suffix_blocks[b]]
        pos += suffix_blocks[b]
    shape = (nb, block_size, num_kv_heads, head_dim)
    k_cache = normal_bf16(place, shape)
    v_cache = normal_bf16(place, shape)
    prefix_k = normal_bf16(rng, (prefix_len, num_kv_heads, head_dim))
    prefix_v = normal_bf16(rng, (prefix_len, num_kv_heads, head_dim))
    for b in range(B if not shared else 1):
        rows = slots_for_positions(bt, np.full(prefix_len, b), np.arange(prefix_len), block_size)
        k_cache.reshape(-1, num_kv_heads, head_dim)[rows] = prefix_k
        v_cache.reshape(-1, num_kv_heads, head_dim)[rows] = prefix_v
    Tq = int(ql.sum())
    cu_q = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(kl)]).astype(np.int32)
    seq = np.concatenate([np.full(n, b) for b, n in enumerate(ql)]) if B else np.zeros(0)
    posn = np.concatenate([prefix_len + np.arange(n) for n in ql]) if B else np.zeros(0)
    slots = slots_for_positions(bt, seq, posn, block_size) if Tq else np.zeros(0, np.int32)
    return PrefillCase(
        num_blocks=nb, block_size=block_size, num_kv_heads=num_kv_heads, head_dim=head_dim,
        num_q_heads=num_q_heads, k_cache=k_cache, v_cache=v_cache,
        q=normal_bf16(rng, (Tq, num_q_heads, head_dim), q_scale),
        k=normal_bf16(rng, (Tq, num_kv_heads, head_dim)),
        v=normal_bf16(rng, (Tq, num_kv_heads, head_dim)),
        cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, block_tables=bt, slot_mapping=slots.astype(np.int32),
        scale=1.0 / math.sqrt(head_dim))


def prefix_prefill_suffix_lengths(num_seqs: int = 64, seed: Optional[int] = None) -> np.ndarray:
    w = WORKLOADS["prefix_prefill"]
    rng = rng_for(w.seed if seed is None else seed, 100)
    return uniform_int(rng, 100, 1024, num_seqs)


# ----------------------------------------------------------------------------------------------
# Device fill for the large pools (torch, seeded)
# ----------------------------------------------------------------------------------------------


def fill_normal_bf16_(t, seed: int, *stream: int):
    """Fill a bf16 torch tensor in place with N(0,1) from a seeded generator on its device."""
    import torch
    g = torch.Generator(device=t.device)
    s = np.random.SeedSequence([seed, *stream]).generate_state(1, dtype=np.uint64)[0]
    g.manual_seed(int(s) & ((1 << 63) - 1))
    t.normal_(generator=g)
    return t
