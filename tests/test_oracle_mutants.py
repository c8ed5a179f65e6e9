"""Plant plausible mistakes in copies of the oracle and check that the pins catch every one.

Each mutant is a one-line textual change to oracle.c (a dropped term, a wrong index, a transposed
operand, an off-by-one), compiled to a temporary library on the CPU. The real oracle source is
never modified. Mutants are chosen so that none of them can read or write out of bounds.
"""
import os

import pytest

import oracle
from oracle import build as obuild
from tests import oracle_pins as pins

MUTANTS = {
    "gqa_interleaved_heads": (
        "for (int32_t h = g * G; h < (g + 1) * G; ++h) {\n      double *o = out + ((int64_t)b",
        "for (int32_t h = g; h < num_q_heads; h += num_kv_heads) {\n      double *o = out + ((int64_t)b"),
    "scale_dropped": ("s[j] = scale * dot;", "s[j] = dot;"),
    "offset_from_block_index": ("const int64_t offset = p % block_size;\n    if (block < 0",
                                "const int64_t offset = (p / block_size) % block_size;\n    if (block < 0"),
    "causal_off_by_one": ("(int64_t)P + i + 1, head_dim", "(int64_t)P + i, head_dim"),
    "value_reads_key": ("num += s[j] * V[j * head_dim + d];", "num += s[j] * K[j * head_dim + d];"),
    "denominator_dropped": ("out[d] = num / den;", "out[d] = num;"),
    "store_v_from_k": ("memcpy(v_cache + dst, v + t * row", "memcpy(v_cache + dst, k + t * row"),
    "store_counts_no_invalid": ("if (s == -1) continue;", "if (s < 0) continue;"),
    "bf16_widening_shift": ("(uint32_t)bits << 16", "(uint32_t)bits << 15"),
    "decode_drops_last_token": ("const int64_t n = ctx > 0 ? ctx : 0;",
                                "const int64_t n = ctx > 1 ? ctx - 1 : 0;"),
    "prefix_keys_from_new_rows": ("bad |= oracle_gather_head(k_cache, num_blocks, block_size, num_kv_heads, head_dim, bt_row,\n                                P, g, K);",
                                  "bad |= oracle_gather_head(v_cache, num_blocks, block_size, num_kv_heads, head_dim, bt_row,\n                                P, g, K);"),
    "max_not_tracked": ("if (s[j] > m) m = s[j];", "if (s[j] < m) m = s[j];"),
    "xxh64_wrong_round_rotation": ("  acc = rotl64(acc, 31);\n  return acc * XXP1;",
                                   "  acc = rotl64(acc, 33);\n  return acc * XXP1;"),
    "xxh64_tail8_rotation": ("acc = rotl64(acc, 27) * XXP1 + XXP4;",
                             "acc = rotl64(acc, 29) * XXP1 + XXP4;"),
    "chain_parent_big_endian": ("buf[n++] = (uint8_t)(parent >> (8 * k));",
                                "buf[n++] = (uint8_t)(parent >> (56 - 8 * k));"),
    "chain_hashes_partial_block": ("int32_t nfull = len / block_size;",
                                   "int32_t nfull = (len + block_size - 1) / block_size;"),
    "cow_copies_backwards": ("memcpy(k_cache + dst * block_elems, k_cache + src * block_elems,",
                             "memcpy(k_cache + src * block_elems, k_cache + dst * block_elems,"),
    "gather_reads_v_for_k": ("memcpy(out_k + i * block_elems, k_cache + blk * block_elems,",
                             "memcpy(out_k + i * block_elems, v_cache + blk * block_elems,"),
}


@pytest.fixture(scope="module")
def source():
    with open(obuild.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) >= 1, f"mutation site for {name} not found in oracle.c"
    mutated = source.replace(old, new, 1)
    src = tmp_path / "mutant.c"
    src.write_text(mutated)
    lib = obuild.build(str(src), str(tmp_path / "libmutant.so"), quiet=True)
    orc = oracle.Oracle(lib)
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, IndexError, ValueError) as e:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
