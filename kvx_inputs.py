"""Seeded synthetic workloads for kvx: block-id lists, request lengths, token streams, residency masks.

This module is shared by the tests, the smoke check and the benchmark. It holds none of the method's
arithmetic: it never merges runs, maps tokens to rows, hashes or matches anything. It only draws
numbers from seeded generators (numpy PCG64 for ids and tokens; a seeded torch generator for values)
and describes the shapes of the five workloads:

  1 tiny            2 layers x {K,V}, 2 heads x 64 bf16, block 16, pools of 256 blocks, 4 requests of
                    U[100,300] tokens; src ids contiguous, dst ids a chunked permutation (~50 % of blocks
                    in multi-block runs, run length mean 4), dst canary 0xDEAD per bf16 element.
  2 qwen3_32b_single   64 layers x {K,V}, 8 KV heads x 128 bf16, block 16, one 8192-token prompt
                    (512 blocks), pools of 615 blocks, src ids 0..511, dst ids chunked as in 1.
  3 qwen3_32b_batched  same token shape, 16 requests of U[1024,8192] tokens, pools 1.2x the live blocks,
                    both id sides fragmented (chunk length geometric, mean 2).
  4 tp4_to_tp1_remap   producer: 4 head-shard buffers (2 heads each), block 16; consumer: 1 buffer with
                    all 8 heads, block 64; 64 layers, 8 requests of U[2048,16384] tokens, fragmented ids.
  5 bidir_mla_fp8   48 layers, 1 latent head of 576 fp8 bytes, block 64; 256 sessions = shared 1024-token
                    system prompt + U[2048,32768] history tokens from a 151936-token vocabulary; the
                    prefill side holds a seeded Bernoulli(0.4) subset of each session's blocks.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

VOCAB = 151936          # token-id range of the bidirectional workload
CANARY_BF16 = 0xDEAD    # fill of every untouched consumer bf16 element
CANARY_FP8 = 0x7F       # fill of the prefill pool in the fp8 workload: an e4m3 NaN code, never pushed


LAYOUT_NHD, LAYOUT_HND = 0, 1


@dataclasses.dataclass
class PoolGeom:
    """Shape of one side's paged pool: n_layers*n_planes*n_shards dense buffers, each
    [n_blocks][block_size][heads_per_shard][head_dim] (layout NHD) or
    [n_blocks][heads_per_shard][block_size][head_dim] (layout HND) elements of elem_bytes."""
    n_layers: int
    n_planes: int
    n_shards: int
    heads_per_shard: int
    head_dim: int
    elem_bytes: int
    block_size: int
    n_blocks: int
    layout: int = LAYOUT_NHD

    @property
    def n_buffers(self) -> int:
        return self.n_layers * self.n_planes * self.n_shards

    @property
    def row_bytes(self) -> int:
        return self.heads_per_shard * self.head_dim * self.elem_bytes

    @property
    def buffer_bytes(self) -> int:
        return self.n_blocks * self.block_size * self.row_bytes

    def replace(self, **kw) -> "PoolGeom":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass
class Request:
    n_tokens: int
    src_ids: np.ndarray   # int32, at least ceil(n_tokens / src.block_size) entries
    dst_ids: np.ndarray   # int32, at least ceil(n_tokens / dst.block_size) entries


@dataclasses.dataclass
class PushWorkload:
    name: str
    src: PoolGeom
    dst: PoolGeom
    requests: List[Request]
    seed: int
    values: str           # "bf16_normal" or "fp8_bytes"


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def chunked_order(rng: np.random.Generator, n_pool: int, *, p_single: Optional[float] = None,
                  mean_multi: float = 4.0, mean: float = 2.0) -> np.ndarray:
    """A permutation of range(n_pool) made of shuffled ascending chunks.

    With p_single set: a chunk is a single block with probability p_single, else 1 + Geometric with
    mean mean_multi - 1 (so multi-block chunks have mean length mean_multi). Without it: chunk length
    is Geometric on {1, 2, ...} with the given mean. Chunks are carved from 0 upwards, shuffled with
    the same generator and concatenated.
    """
    if n_pool <= 0:
        return np.zeros(0, np.int32)
    lengths: list = []
    total = 0
    while total < n_pool:
        k = max(16, (n_pool - total) // 2)
        if p_single is not None:
            single = rng.random(k) < p_single
            multi = 1 + rng.geometric(1.0 / (mean_multi - 1.0), k)
            draw = np.where(single, 1, multi)
        else:
            draw = rng.geometric(1.0 / mean, k)
        for length in draw.tolist():
            if total >= n_pool:
                break
            length = min(int(length), n_pool - total)
            lengths.append(length)
            total += length
    starts = np.concatenate([[0], np.cumsum(lengths)[:-1]])
    order = rng.permutation(len(lengths))
    return np.concatenate([np.arange(starts[i], starts[i] + lengths[i]) for i in order]).astype(np.int32)


def _slice_per_request(order: np.ndarray, counts: List[int]) -> List[np.ndarray]:
    out, pos = [], 0
    for c in counts:
        out.append(np.ascontiguousarray(order[pos:pos + c], dtype=np.int32))
        pos += c
    return out


def _qwen3_32b_geom(n_layers: int, n_blocks: int) -> PoolGeom:
    return PoolGeom(n_layers=n_layers, n_planes=2, n_shards=1, heads_per_shard=8, head_dim=128,
                    elem_bytes=2, block_size=16, n_blocks=n_blocks)


def tiny(seed: int = 1) -> PushWorkload:
    rng = np.random.default_rng(seed)
    geom = PoolGeom(2, 2, 1, 2, 64, 2, 16, 256)
    lens = rng.integers(100, 301, 4).tolist()
    need = [_ceil_div(n, 16) for n in lens]
    src = _slice_per_request(np.arange(256, dtype=np.int32), need)
    dst = _slice_per_request(chunked_order(rng, 256, p_single=0.8, mean_multi=4.0), need)
    reqs = [Request(n, s, d) for n, s, d in zip(lens, src, dst)]
    return PushWorkload("tiny", geom, geom.replace(), reqs, seed, "bf16_normal")


def qwen3_32b_single(seed: int = 2, n_layers: int = 64) -> PushWorkload:
    rng = np.random.default_rng(seed)
    n_tok, n_blk, pool = 8192, 512, 615
    geom = _qwen3_32b_geom(n_layers, pool)
    src = np.arange(n_blk, dtype=np.int32)
    dst = chunked_order(rng, pool, p_single=0.8, mean_multi=4.0)[:n_blk].copy()
    return PushWorkload("qwen3_32b_single", geom, geom.replace(), [Request(n_tok, src, dst)], seed,
                        "bf16_normal")


def qwen3_32b_batched(seed: int = 3, n_layers: int = 64, n_requests: int = 16,
                      len_range=(1024, 8192), layout: int = LAYOUT_NHD) -> PushWorkload:
    rng = np.random.default_rng(seed)
    lens = rng.integers(len_range[0], len_range[1] + 1, n_requests).tolist()
    need = [_ceil_div(n, 16) for n in lens]
    pool = math.ceil(1.2 * sum(need))
    geom = _qwen3_32b_geom(n_layers, pool).replace(layout=layout)
    src = _slice_per_request(chunked_order(rng, pool, mean=2.0), need)
    dst = _slice_per_request(chunked_order(rng, pool, mean=2.0), need)
    reqs = [Request(n, s, d) for n, s, d in zip(lens, src, dst)]
    return PushWorkload("qwen3_32b_batched", geom, geom.replace(), reqs, seed, "bf16_normal")


def tp4_to_tp1_remap(seed: int = 4, n_layers: int = 64, n_requests: int = 8,
                     len_range=(2048, 16384)) -> PushWorkload:
    rng = np.random.default_rng(seed)
    lens = rng.integers(len_range[0], len_range[1] + 1, n_requests).tolist()
    need_s = [_ceil_div(n, 16) for n in lens]
    need_d = [_ceil_div(n, 64) for n in lens]
    pool_s = math.ceil(1.2 * sum(need_s))
    pool_d = math.ceil(1.2 * sum(need_d))
    src_geom = PoolGeom(n_layers, 2, 4, 2, 128, 2, 16, pool_s)
    dst_geom = PoolGeom(n_layers, 2, 1, 8, 128, 2, 64, pool_d)
    src = _slice_per_request(chunked_order(rng, pool_s, mean=2.0), need_s)
    dst = _slice_per_request(chunked_order(rng, pool_d, mean=2.0), need_d)
    reqs = [Request(n, s, d) for n, s, d in zip(lens, src, dst)]
    return PushWorkload("tp4_to_tp1_remap", src_geom, dst_geom, reqs, seed, "bf16_normal")


def qwen3_32b_batched_hnd(seed: int = 3, n_layers: int = 64) -> PushWorkload:
    """The batched workload with both pools head-major ([block][head][slot][dim])."""
    w = qwen3_32b_batched(seed=seed, n_layers=n_layers, layout=LAYOUT_HND)
    w.name = "qwen3_32b_batched_hnd"
    return w


def qwen3_32b_batched_nhd_to_hnd(seed: int = 3, n_layers: int = 64) -> PushWorkload:
    """The batched workload from a token-major producer ([block][slot][head][dim]) into a head-major
    consumer ([block][head][slot][dim]): each block is transposed at head granularity."""
    w = qwen3_32b_batched(seed=seed, n_layers=n_layers)
    w.dst = w.dst.replace(layout=LAYOUT_HND)
    w.name = "qwen3_32b_batched_nhd_to_hnd"
    return w


def qwen3_32b_single_nhd_to_hnd(seed: int = 2, n_layers: int = 64) -> PushWorkload:
    """The single-request workload (one 8192-token prompt, 32 MiB per layer read) from a token-major
    producer into a head-major consumer: a head-layout change at per-layer push sizes."""
    w = qwen3_32b_single(seed=seed, n_layers=n_layers)
    w.dst = w.dst.replace(layout=LAYOUT_HND)
    w.name = "qwen3_32b_single_nhd_to_hnd"
    return w


def qwen3_32b_single_hnd_to_nhd(seed: int = 2, n_layers: int = 64) -> PushWorkload:
    """The single-request workload from a head-major producer into a token-major consumer."""
    w = qwen3_32b_single(seed=seed, n_layers=n_layers)
    w.src = w.src.replace(layout=LAYOUT_HND)
    w.name = "qwen3_32b_single_hnd_to_nhd"
    return w


PUSH_WORKLOADS = {
    "tiny": tiny,
    "qwen3_32b_single": qwen3_32b_single,
    "qwen3_32b_batched": qwen3_32b_batched,
    "tp4_to_tp1_remap": tp4_to_tp1_remap,
    "qwen3_32b_batched_hnd": qwen3_32b_batched_hnd,
    "qwen3_32b_batched_nhd_to_hnd": qwen3_32b_batched_nhd_to_hnd,
    "qwen3_32b_single_nhd_to_hnd": qwen3_32b_single_nhd_to_hnd,
    "qwen3_32b_single_hnd_to_nhd": qwen3_32b_single_hnd_to_nhd,
}


# ----------------------------------------------------------------------------------------------
# Bidirectional (decode -> prefill) workload
# ----------------------------------------------------------------------------------------------

@dataclasses.dataclass
class BidirWorkload:
    """Token streams and block placement of the multi-turn reuse workload.

    tokens/tok_off: CSR of each session's context (uint32 ids); block_size tokens per block.
    remote_blk/rem_off: CSR of the decode block holding each *full* block of each session's context
    (decode retains prompt and response blocks). resident: CSR mask (same offsets as remote_blk) of
    which of a session's blocks the prefill side holds locally. free_blocks: prefill blocks a
    decode->prefill push may fill, in the order they are handed out.
    """
    n_sessions: int
    block_size: int
    tokens: np.ndarray        # uint32 [sum lengths]
    tok_off: np.ndarray       # int64 [n_sessions + 1]
    remote_blk: np.ndarray    # int32 [sum full blocks]
    rem_off: np.ndarray       # int64 [n_sessions + 1]
    resident: np.ndarray      # bool  [sum full blocks]
    decode: PoolGeom
    prefill: PoolGeom
    resident_blk: np.ndarray  # int32 prefill block id for each resident entry (same index as resident)
    free_blocks: np.ndarray   # int32, the prefill free region in hand-out order
    threshold: int
    seed: int


def bidir_mla_fp8(seed: int = 5, n_sessions: int = 256, n_layers: int = 48, system_tokens: int = 1024,
                  hist_range=(2048, 32768), resident_p: float = 0.4, threshold: int = 512,
                  free_blocks: Optional[int] = None) -> BidirWorkload:
    """Sessions = one shared system prompt + per-session history; each session's full blocks sit in
    fragmented decode blocks; the prefill pool holds a Bernoulli(resident_p) subset of each session's
    blocks plus a free region (default: room for the largest push any single wave of 64 sessions needs
    is left to the caller; here the free region holds all full blocks of all sessions unless given)."""
    bs = 64
    rng = np.random.default_rng(seed)
    system = rng.integers(0, VOCAB, system_tokens, dtype=np.int64)
    hist = rng.integers(hist_range[0], hist_range[1] + 1, n_sessions).tolist()
    parts, offs = [], [0]
    for h in hist:
        parts.append(system)
        parts.append(rng.integers(0, VOCAB, h, dtype=np.int64))
        offs.append(offs[-1] + system_tokens + h)
    tokens = np.concatenate(parts).astype(np.uint32) if parts else np.zeros(0, np.uint32)
    tok_off = np.asarray(offs, np.int64)
    n_full = [(system_tokens + h) // bs for h in hist]
    rem_off = np.concatenate([[0], np.cumsum(n_full)]).astype(np.int64)
    total = int(rem_off[-1])
    decode_pool = total
    remote_blk = chunked_order(rng, decode_pool, mean=2.0)[:total].copy()
    resident = rng.random(total) < resident_p
    n_res = int(resident.sum())
    resident_blk = np.full(total, -1, np.int32)
    resident_blk[resident] = np.arange(n_res, dtype=np.int32)
    n_free = total if free_blocks is None else int(free_blocks)
    free = (n_res + chunked_order(rng, n_free, mean=2.0)).astype(np.int32)
    decode = PoolGeom(n_layers, 1, 1, 1, 576, 1, bs, decode_pool)
    prefill = PoolGeom(n_layers, 1, 1, 1, 576, 1, bs, n_res + n_free)
    return BidirWorkload(n_sessions, bs, tokens, tok_off, remote_blk, rem_off, resident, decode,
                         prefill, resident_blk, free, threshold, seed)


# ----------------------------------------------------------------------------------------------
# Value fills (bytes only; the path never interprets them)
# ----------------------------------------------------------------------------------------------

def host_random_bytes(n: int, seed: int) -> np.ndarray:
    """Uniform random bytes on the host (CPU-only tests)."""
    return np.random.default_rng(seed).integers(0, 256, n, dtype=np.uint8)


def fill_bf16_normal(t, seed: int) -> None:
    """Fill a torch tensor's storage with bf16 N(0,1) values from a seeded generator on its device."""
    import torch
    gen = torch.Generator(device=t.device)
    gen.manual_seed(seed)
    flat = t.view(torch.bfloat16).view(-1) if t.dtype != torch.bfloat16 else t.view(-1)
    flat.normal_(0.0, 1.0, generator=gen)


def fill_fp8_bytes(t, seed: int, chunk: int = 1 << 30) -> None:
    """Fill a torch uint8 tensor with bytes uniform over 0x00..0xFE minus 0x7F (no e4m3 NaN codes),
    a chunk at a time so that no temporary is as large as the tensor."""
    import torch
    gen = torch.Generator(device=t.device)
    gen.manual_seed(seed)
    flat = t.view(-1)
    for i in range(0, flat.numel(), chunk):
        c = flat[i:i + chunk]
        c.random_(0, 254, generator=gen)
        c.add_((c >= 0x7F).to(torch.uint8))


def fill_canary(t, kind: str) -> None:
    """Fill a consumer buffer with the canary of its workload."""
    import torch
    if kind == "bf16_normal":
        t.view(torch.int16).fill_(CANARY_BF16 - 0x10000)
    else:
        t.view(torch.uint8).fill_(CANARY_FP8)
