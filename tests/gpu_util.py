"""Helpers for the GPU parity tests: host <-> device conversion and oracle sampling.

Expected values always come from the oracle on host copies of the inputs; the CUDA path's outputs
are only ever compared, never fed back into the oracle.
"""
from __future__ import annotations

import numpy as np
import torch

import workloads as W

TOL = 2e-2  # max-abs attention error bound for N(0,1) inputs


def dev_bf16(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16).to(device)


def dev_i32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def max_abs(gpu: torch.Tensor, ref: np.ndarray) -> float:
    g = to_f64(gpu)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), "non-finite GPU output"
    return float(np.max(np.abs(g - ref))) if g.size else 0.0


def assert_attn_close(gpu: torch.Tensor, ref: np.ndarray, tol: float = TOL, what: str = ""):
    err = max_abs(gpu, ref)
    assert err <= tol, f"{what}: max abs error {err:.3e} > {tol}"
    return err


class DeviceDecodeLayer:
    """One decode layer drawn on the device: a pool holding positions 0..ctx-2 of each sequence,
    the new token's K/V and slot, and q. Large pools are drawn with the seeded torch generator."""

    def __init__(self, ctx: np.ndarray, Hq: int, Hkv: int, D: int, BS: int, seed: int,
                 layer: int = 0, pad_to: int = 0, device="cuda"):
        rng = W.rng_for(seed, 10, layer)
        self.ctx = np.asarray(ctx, dtype=np.int32)
        B = len(self.ctx)
        self.bt, self.nb = W.place_blocks(rng, self.ctx, BS)
        live = np.nonzero(self.ctx > 0)[0]
        slots = W.slots_for_positions(self.bt, live, self.ctx[live] - 1, BS)
        npad = max(0, pad_to - len(slots))
        self.slots = np.concatenate([slots, np.full(npad, -1, np.int32)]).astype(np.int32)
        self.Hq, self.Hkv, self.D, self.BS = Hq, Hkv, D, BS
        shape = (self.nb, BS, Hkv, D)
        self.k_cache = torch.empty(shape, dtype=torch.bfloat16, device=device)
        self.v_cache = torch.empty(shape, dtype=torch.bfloat16, device=device)
        W.fill_normal_bf16_(self.k_cache, seed, layer, 1)
        W.fill_normal_bf16_(self.v_cache, seed, layer, 2)
        T = len(self.slots)
        self.k_new = W.fill_normal_bf16_(torch.empty((T, Hkv, D), dtype=torch.bfloat16,
                                                     device=device), seed, layer, 3)
        self.v_new = W.fill_normal_bf16_(torch.empty((T, Hkv, D), dtype=torch.bfloat16,
                                                     device=device), seed, layer, 4)
        self.q = W.fill_normal_bf16_(torch.empty((B, Hq, D), dtype=torch.bfloat16,
                                                 device=device), seed, layer, 5)
        self.bt_dev = dev_i32(self.bt, device)
        self.ctx_dev = dev_i32(self.ctx, device)
        self.slots_dev = dev_i32(self.slots, device)
        self.scale = 1.0 / np.sqrt(D)

    def snapshot(self, seqs):
        """Host copy (taken now) of everything the oracle needs for the sampled sequences, with
        the sequences' blocks renumbered into a compact pool (a placement permutation)."""
        BS = self.BS
        need = W.blocks_needed(self.ctx[seqs], BS)
        used = np.unique(np.concatenate([self.bt[b, :n] for b, n in zip(seqs, need)] +
                                        [np.zeros(0, np.int32)]))
        remap = {int(b): i for i, b in enumerate(used)}
        idx = torch.from_numpy(used.astype(np.int64)).to(self.k_cache.device)
        snap = dict(
            blocks=used,
            k_cache=host_bits(self.k_cache.index_select(0, idx)) if len(used) else
            np.zeros((1, BS, self.Hkv, self.D), np.uint16),
            v_cache=host_bits(self.v_cache.index_select(0, idx)) if len(used) else
            np.zeros((1, BS, self.Hkv, self.D), np.uint16),
            q=host_bits(self.q[torch.as_tensor(seqs, device=self.q.device)]),
            ctx=self.ctx[seqs].copy(),
        )
        bt = np.full((len(seqs), max(1, self.bt.shape[1])), -1, np.int32)
        for i, (b, n) in enumerate(zip(seqs, need)):
            bt[i, :n] = [remap[int(x)] for x in self.bt[b, :n]]
        snap["bt"] = bt
        # the new rows of the sampled sequences, with slots in the compact numbering
        live = np.nonzero(self.ctx > 0)[0]
        row_of = {int(b): i for i, b in enumerate(live)}
        rows, slots = [], []
        for i, b in enumerate(seqs):
            if self.ctx[b] > 0:
                p = int(self.ctx[b]) - 1
                rows.append(row_of[int(b)])
                slots.append(bt[i, p // BS] * BS + p % BS)
        rows_t = torch.as_tensor(rows, dtype=torch.long, device=self.q.device)
        snap["k_new"] = host_bits(self.k_new[rows_t]) if rows else np.zeros((0, self.Hkv, self.D),
                                                                            np.uint16)
        snap["v_new"] = host_bits(self.v_new[rows_t]) if rows else np.zeros((0, self.Hkv, self.D),
                                                                            np.uint16)
        snap["slots"] = np.asarray(slots, np.int32)
        return snap


def oracle_decode_from_snapshot(orc, snap, scale, num_q_heads):
    kc, vc, bad = orc.kv_store(snap["k_new"], snap["v_new"], snap["slots"], snap["k_cache"],
                               snap["v_cache"])
    assert bad == 0
    out = orc.paged_decode(snap["q"], kc, vc, snap["bt"], snap["ctx"], scale)
    return out, kc, vc
