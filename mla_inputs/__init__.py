"""Seeded synthetic inputs for the MLA latent-cache decode step.

This module is the one thing the oracle and the CUDA path share: it draws the
inputs and lays them out (paged cache, block tables, slot mappings).  It holds
none of the method's arithmetic: no scores, softmax, weighted sums or merges.

Workloads (shapes from the pages' DeepSeek-V3 numbers: 128 heads, 512 kv_c +
64 k_rope latent per token, 61 layers):

  1 tiny         B=4, lengths {1,17,64,200} then +1 appended, page 16, 1 layer
  2 layer        B=64 x 4096, page 64, 1 layer
  3 dp_rank      B=20 x 4096, page 64, 61 layers each with its own cache,
                 one appended row per sequence per layer (the data-parallel
                 attention rank's share of a 159 x 4096 node batch)
  4 skewed       B=8: one 131072-token sequence and seven of 1024, page 64
  5 mixed        B=256, lengths uniform in [512, 8192], page 64, 4 layers,
                 fragmented pool (1.25x the blocks needed, drawn at random)

Values: latent rows ~ N(0,1) rounded to bfloat16 (round to nearest even);
queries ~ N(0,1)/sqrt(576) ("normal") or N(0,1) ("sharp"); softmax scale
1/sqrt(192).  Rows past a sequence's end inside its last block, and every block
no sequence owns, hold a bfloat16 NaN so that a stray read shows in the output.
For configs 2-5 the context length includes the row appended this step: L-1
rows are pre-filled, the slot of token L-1 is poisoned, and the append writes it.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

ROW = 576
KV_LORA_RANK = 512
ROPE_DIM = 64
NUM_HEADS = 128
SOFTMAX_SCALE = 1.0 / math.sqrt(192.0)
BF16_NAN = 0x7FC0
BASE_SEED = 20261202


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round fp32 values to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class Workload:
    config_id: int
    name: str
    seq_lens: list                 # context length decoded over (after the append)
    block_size: int
    layers: int
    append: bool                   # one new row per sequence per layer
    pool_factor: float = 1.0       # blocks in the pool / blocks needed
    extra: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.seq_lens)

    def blocks_needed(self) -> int:
        return sum(-(-L // self.block_size) for L in self.seq_lens)

    def num_blocks(self) -> int:
        return max(1, int(math.ceil(self.blocks_needed() * self.pool_factor)))

    def max_blocks_per_seq(self) -> int:
        return max(1, max((-(-L // self.block_size) for L in self.seq_lens), default=1))

    def cache_bytes_per_layer_read(self) -> int:
        """Bytes of latent rows one decode pass reads (every context row once)."""
        return sum(self.seq_lens) * ROW * 2


def workload(config_id: int, seed: int | None = None) -> Workload:
    if config_id == 1:
        return Workload(1, "tiny_b4_L1-200_page16", [2, 18, 65, 201], 16, 1, True, 2.0,
                        {"pre_append_lens": [1, 17, 64, 200]})
    if config_id == 2:
        return Workload(2, "layer_b64x4096_page64", [4096] * 64, 64, 1, True)
    if config_id == 3:
        return Workload(3, "dp_rank_b20x4096_61layers_page64", [4096] * 20, 64, 61, True)
    if config_id == 4:
        return Workload(4, "skewed_1x131072_7x1024_page64", [131072] + [1024] * 7, 64, 1, True)
    if config_id == 5:
        rng = np.random.default_rng(BASE_SEED + 5 if seed is None else seed)
        lens = rng.integers(512, 8192, size=256, endpoint=True).tolist()
        return Workload(5, "mixed_b256_U512-8192_4layers_page64", lens, 64, 4, True, 1.25)
    raise ValueError(f"unknown config {config_id}")


def custom_workload(seq_lens, block_size=64, layers=1, append=True, pool_factor=1.0,
                    name="custom") -> Workload:
    return Workload(0, name, list(seq_lens), block_size, layers, append, pool_factor)


# ----------------------------------------------------------------------------- host (numpy)

def make_block_table(rng, seq_lens, block_size, num_blocks):
    """Random distinct physical blocks for every logical block (shuffled pool).

    Returns int32 [B, max_blocks]; entries past a sequence's last block are -1.
    """
    need = [-(-L // block_size) for L in seq_lens]
    total = sum(need)
    assert total <= num_blocks
    phys = rng.permutation(num_blocks)[:total].astype(np.int32)
    mb = max(1, max(need, default=1))
    bt = np.full((len(seq_lens), mb), -1, np.int32)
    o = 0
    for b, n in enumerate(need):
        bt[b, :n] = phys[o:o + n]
        o += n
    return bt


def poison_unused(cache, block_table, seq_lens, block_size):
    """Fill every row no sequence owns (free blocks, tails) with bfloat16 NaN."""
    owned = np.zeros(cache.shape[:2], bool)
    for b, L in enumerate(seq_lens):
        for t in range(0, L, block_size):
            n = min(block_size, L - t)
            owned[block_table[b, t // block_size], :n] = True
    cache[~owned] = BF16_NAN
    return cache


def gather_rows(cache, block_table, b, L, block_size):
    """Logical rows 0..L-1 of request b (uint16 [L, 576]) by the table; no arithmetic."""
    idx = np.arange(L)
    blk = block_table[b, idx // block_size]
    return cache[blk, idx % block_size]


def slot_of(block_table, b, t, block_size) -> int:
    return int(block_table[b, t // block_size]) * block_size + t % block_size


def make_queries(rng, batch, num_heads=NUM_HEADS, kind="normal"):
    x = rng.standard_normal((batch, num_heads, ROW), dtype=np.float32)
    if kind == "normal":
        x /= np.float32(math.sqrt(ROW))
    elif kind != "sharp":
        raise ValueError(kind)
    return f32_to_bf16_bits(x)


def make_host_layer(w: Workload, rng, q_kind="normal", num_heads=NUM_HEADS):
    """One layer's host inputs for workload w (numpy; small configs only).

    Returns dict: q [B,H,576] u16, cache [NB,BS,576] u16 (pre-append, appended
    slots poisoned), block_table [B,max_blocks] i32, seq_lens [B] i32 (after the
    append), kv_new [B,576] u16, slot_mapping [B] i64 (slot of token L-1).
    """
    NB, BS = w.num_blocks(), w.block_size
    bt = make_block_table(rng, w.seq_lens, BS, NB)
    cache = f32_to_bf16_bits(rng.standard_normal((NB, BS, ROW), dtype=np.float32))
    poison_unused(cache, bt, w.seq_lens, BS)
    seq = np.asarray(w.seq_lens, np.int32)
    kv_new = f32_to_bf16_bits(rng.standard_normal((w.batch, ROW), dtype=np.float32))
    slots = np.array([slot_of(bt, b, int(L) - 1, BS) for b, L in enumerate(seq)], np.int64)
    if w.append:
        blk, row = slots // BS, slots % BS
        cache[blk, row] = BF16_NAN
    q = make_queries(rng, w.batch, num_heads, q_kind)
    return dict(q=q, cache=cache, block_table=bt, seq_lens=seq, kv_new=kv_new,
                slot_mapping=slots, softmax_scale=SOFTMAX_SCALE)


def rng_for(config_id: int, layer: int = 0, salt: int = 0):
    return np.random.default_rng([BASE_SEED + config_id, layer, salt])


# ----------------------------------------------------------------------------- device (torch)

def make_device_layer(w: Workload, layer: int, device, q_kind="normal", num_heads=NUM_HEADS,
                      block_table=None):
    """One layer's inputs generated directly on `device` with a seeded torch generator.

    Same recipe as make_host_layer (shuffled or fragmented pool, NaN poison in
    unowned rows and in the slot the append will write), drawn on the GPU so the
    61-layer workload does not have to be built on the host.  The block table is
    drawn on the host (numpy) so the tests can rebuild it; pass `block_table` to
    share one table between layers.
    """
    import torch
    NB, BS = w.num_blocks(), w.block_size
    if block_table is None:
        block_table = make_block_table(rng_for(w.config_id, layer, 1), w.seq_lens, BS, NB)
    g = torch.Generator(device=device)
    g.manual_seed(BASE_SEED * 1000 + w.config_id * 100 + layer)
    cache = torch.randn((NB, BS, ROW), generator=g, device=device, dtype=torch.float32)
    cache = cache.to(torch.bfloat16)
    seq = np.asarray(w.seq_lens, np.int64)
    owned = torch.zeros((NB, BS), dtype=torch.bool, device=device)
    bt_t = torch.as_tensor(block_table, device=device).long()
    for b, L in enumerate(seq.tolist()):
        nfull, tail = divmod(L, BS)
        if nfull:
            owned[bt_t[b, :nfull]] = True
        if tail:
            owned[bt_t[b, nfull], :tail] = True
    nanv = torch.tensor(float("nan"), dtype=torch.bfloat16, device=device)
    cache[~owned] = nanv
    slots = np.array([slot_of(block_table, b, int(L) - 1, BS) for b, L in enumerate(seq)], np.int64)
    slots_t = torch.as_tensor(slots, device=device)
    if w.append:
        cache.view(NB * BS, ROW)[slots_t] = nanv
    q = torch.randn((w.batch, num_heads, ROW), generator=g, device=device, dtype=torch.float32)
    if q_kind == "normal":
        q = q / math.sqrt(ROW)
    q = q.to(torch.bfloat16)
    kv_new = torch.randn((w.batch, ROW), generator=g, device=device, dtype=torch.float32)
    kv_new = kv_new.to(torch.bfloat16)
    return dict(q=q, cache=cache, block_table=torch.as_tensor(block_table, device=device),
                block_table_host=block_table,
                seq_lens=torch.as_tensor(seq.astype(np.int32), device=device),
                kv_new=kv_new, slot_mapping=slots_t, softmax_scale=SOFTMAX_SCALE)


# ----------------------------------------------------------------------------- FP8 cache

def e4m3_codes(x) -> np.ndarray:
    """E4M3 byte codes of fp32 samples, drawn by torch's float8_e4m3fn cast
    (an input-drawing step like the bf16 rounding above; NaN stays NaN)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def make_host_layer_fp8(w: Workload, rng, q_kind="normal", num_heads=NUM_HEADS):
    """make_host_layer with the cache as E4M3 codes (uint8 [NB, BS, 576]) of
    the same N(0,1) rows; unowned rows and the slot the append will write
    hold the NaN code."""
    d = make_host_layer(w, rng, q_kind, num_heads)
    d["cache8"] = e4m3_codes(bf16_bits_to_f32(d["cache"]))
    return d


def make_device_layer_fp8(w: Workload, layer: int, device, q_kind="normal", block_table=None):
    """make_device_layer with the cache as E4M3 codes (torch uint8), drawn on the device."""
    import torch
    d = make_device_layer(w, layer, device, q_kind=q_kind, block_table=block_table)
    d["cache8"] = d.pop("cache").float().to(torch.float8_e4m3fn).view(torch.uint8)
    return d


def to_bits(t) -> np.ndarray:
    """Host uint16 bit patterns of a bfloat16 torch tensor."""
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
