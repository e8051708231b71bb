"""Seeded synthetic inputs for paged KV-cache attention.

This module only draws inputs: random bf16 tensors, a physical block layout
and the per-sequence metadata (block tables, context lengths, slot mapping,
cumulative query lengths).  It holds none of the attention arithmetic, so the
CUDA path and the CPU oracle can both consume what it produces without sharing
any of the computation being checked.

Every tensor is created on the CPU from a seeded ``torch.Generator``; callers
copy it to the device themselves.  bf16 values are fp32 N(0, 1) draws rounded
to nearest-even by ``Tensor.to(torch.bfloat16)``.

Cache layout (fixed by the library): ``k_cache`` and ``v_cache`` are bf16
``[num_blocks, 256, num_kv_heads, head_dim]``; token slot
``s = block_id * 256 + offset`` is one ``num_kv_heads * head_dim`` row.
Block tables are int32 ``[num_seqs, max_blocks]`` padded with -1.

The five workloads follow the shapes of the nano-vllm pages: 256-token cache
blocks (tuning guide "Nano-vLLM性能调优实战", §1.1), up to 128 concurrent
sequences and 4096 batched tokens per step (same guide, §3.2), fixed-size
blocks reached through a block table with shared prefix blocks (ocdem.com
nano-vllm article, §2.1 "基石PagedAttention 与 vLLM 的精髓"), and a
Qwen3-0.6B-like head geometry (16 query heads, 8 KV heads, head_dim 128).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

BLOCK_SIZE = 256


def _gen(seed: int) -> torch.Generator:
    return torch.Generator().manual_seed(int(seed))


def randn_bf16(shape, gen: torch.Generator, scale: float = 1.0,
               chunk: int = 1 << 26) -> torch.Tensor:
    """fp32 N(0,1) * scale rounded to bf16, drawn in chunks to bound memory."""
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=torch.bfloat16)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        x = torch.randn(hi - lo, generator=gen, dtype=torch.float32)
        if scale != 1.0:
            x.mul_(scale)
        out[lo:hi] = x.to(torch.bfloat16)
    return out.view(*shape)


@dataclass
class PagedCache:
    k_cache: torch.Tensor          # bf16 [NB, 256, Hkv, D]
    v_cache: torch.Tensor          # bf16 [NB, 256, Hkv, D]
    block_tables: torch.Tensor     # int32 [B, max_blocks], -1 padded
    context_lens: torch.Tensor     # int32 [B]

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])


@dataclass
class DecodeCase:
    """One decode step: store one new K/V row per sequence, then attend."""
    name: str
    q: torch.Tensor                # bf16 [B, Hq, D]
    k_new: torch.Tensor            # bf16 [B, Hkv, D]
    v_new: torch.Tensor            # bf16 [B, Hkv, D]
    slot_mapping: torch.Tensor     # int32 [B]
    cache: PagedCache
    scale: float
    shared_prefix_blocks: int = 0

    @property
    def num_seqs(self) -> int:
        return int(self.q.shape[0])


@dataclass
class PrefillCase:
    """One chunked-prefill step: store the chunk's K/V rows, then attend."""
    name: str
    q: torch.Tensor                # bf16 [T, Hq, D], T = sum of chunk lengths
    k_new: torch.Tensor            # bf16 [T, Hkv, D]
    v_new: torch.Tensor            # bf16 [T, Hkv, D]
    slot_mapping: torch.Tensor     # int32 [T], -1 = do not store
    cu_seqlens_q: torch.Tensor     # int32 [B + 1]
    cache: PagedCache
    scale: float

    @property
    def num_seqs(self) -> int:
        return int(self.cu_seqlens_q.numel() - 1)


def allocate_block_tables(context_lens: Sequence[int], num_blocks: int,
                          gen: torch.Generator, shared_prefix_blocks: int = 0,
                          max_blocks: Optional[int] = None) -> torch.Tensor:
    """Assign physical blocks to sequences from a seeded shuffle of the pool.

    The first ``shared_prefix_blocks`` logical blocks of every sequence map to
    the same physical blocks (a prefix shared by reference, as the ocdem.com
    article's §2.1 describes for common system prompts); the rest are private.
    Unused table entries are -1.
    """
    need = [int(math.ceil(c / BLOCK_SIZE)) for c in context_lens]
    width = max([1] + need) if max_blocks is None else int(max_blocks)
    perm = torch.randperm(num_blocks, generator=gen).tolist()
    shared = perm[:shared_prefix_blocks]
    pos = shared_prefix_blocks
    table = torch.full((len(context_lens), width), -1, dtype=torch.int32)
    for s, n in enumerate(need):
        if n > width:
            raise ValueError("context needs more blocks than the table width")
        ids = list(shared[:min(n, shared_prefix_blocks)])
        for _ in range(n - len(ids)):
            if pos >= num_blocks:
                raise ValueError("block pool exhausted")
            ids.append(perm[pos])
            pos += 1
        if ids:
            table[s, :n] = torch.tensor(ids, dtype=torch.int32)
    return table


def slots_for_positions(block_table_row: torch.Tensor, positions: Sequence[int]) -> List[int]:
    """Cache slot of each logical token position of one sequence.

    This is the allocator's side of the bookkeeping (it hands the step its
    slot_mapping); the kernels and the oracle receive the result as input.
    """
    row = block_table_row.tolist()
    return [int(row[p // BLOCK_SIZE]) * BLOCK_SIZE + p % BLOCK_SIZE for p in positions]


def make_cache(context_lens: Sequence[int], num_blocks: int, num_kv_heads: int,
               head_dim: int, gen: torch.Generator, k_scale: float = 1.0,
               shared_prefix_blocks: int = 0,
               max_blocks: Optional[int] = None) -> PagedCache:
    tables = allocate_block_tables(context_lens, num_blocks, gen,
                                   shared_prefix_blocks, max_blocks)
    shape = (num_blocks, BLOCK_SIZE, num_kv_heads, head_dim)
    k_cache = randn_bf16(shape, gen, k_scale)
    v_cache = randn_bf16(shape, gen)
    return PagedCache(k_cache, v_cache, tables,
                      torch.tensor(list(context_lens), dtype=torch.int32))


def make_decode_case(name: str, context_lens: Sequence[int], num_q_heads: int,
                     num_kv_heads: int, head_dim: int, num_blocks: int, seed: int,
                     k_scale: float = 1.0, shared_prefix_blocks: int = 0,
                     scale: Optional[float] = None,
                     max_blocks: Optional[int] = None) -> DecodeCase:
    """Decode step; ``context_lens`` already count the token being stored."""
    gen = _gen(seed)
    cache = make_cache(context_lens, num_blocks, num_kv_heads, head_dim, gen,
                       k_scale, shared_prefix_blocks, max_blocks)
    b = len(context_lens)
    q = randn_bf16((b, num_q_heads, head_dim), gen)
    k_new = randn_bf16((b, num_kv_heads, head_dim), gen, k_scale)
    v_new = randn_bf16((b, num_kv_heads, head_dim), gen)
    slots = []
    for s, c in enumerate(context_lens):
        slots.append(slots_for_positions(cache.block_tables[s], [c - 1])[0] if c > 0 else -1)
    return DecodeCase(name, q, k_new, v_new, torch.tensor(slots, dtype=torch.int32),
                      cache, float(scale if scale is not None else 1.0 / math.sqrt(head_dim)),
                      shared_prefix_blocks)


def make_prefill_case(name: str, cached_lens: Sequence[int], chunk_lens: Sequence[int],
                      num_q_heads: int, num_kv_heads: int, head_dim: int,
                      num_blocks: int, seed: int, skip_prob: float = 0.0,
                      scale: Optional[float] = None,
                      max_blocks: Optional[int] = None) -> PrefillCase:
    """Chunked prefill; chunk i of sequence s sits at positions cached+i."""
    gen = _gen(seed)
    ctx = [int(a) + int(b) for a, b in zip(cached_lens, chunk_lens)]
    cache = make_cache(ctx, num_blocks, num_kv_heads, head_dim, gen,
                       max_blocks=max_blocks)
    total = int(sum(chunk_lens))
    q = randn_bf16((total, num_q_heads, head_dim), gen)
    k_new = randn_bf16((total, num_kv_heads, head_dim), gen)
    v_new = randn_bf16((total, num_kv_heads, head_dim), gen)
    slots: List[int] = []
    for s, (c0, lq) in enumerate(zip(cached_lens, chunk_lens)):
        slots += slots_for_positions(cache.block_tables[s], range(c0, c0 + lq))
    slot_mapping = torch.tensor(slots, dtype=torch.int32)
    if skip_prob > 0 and total > 0:
        drop = torch.rand(total, generator=gen) < skip_prob
        slot_mapping[drop] = -1
    cu = [0]
    for lq in chunk_lens:
        cu.append(cu[-1] + int(lq))
    return PrefillCase(name, q, k_new, v_new, slot_mapping,
                       torch.tensor(cu, dtype=torch.int32), cache,
                       float(scale if scale is not None else 1.0 / math.sqrt(head_dim)))


# ---------------------------------------------------------------------------
# The five named workloads (seed = 1000 + workload number).
# ---------------------------------------------------------------------------

def tiny_decode(seed: int = 1001) -> DecodeCase:
    """4 seqs, contexts {1, 37, 256, 300}, 4 q / 2 KV heads, head_dim 64, 8-block pool."""
    return make_decode_case("tiny_decode", [1, 37, 256, 300], 4, 2, 64, 8, seed)


def qwen_decode(seed: int = 1002, num_seqs: int = 128) -> DecodeCase:
    """128 seqs, contexts ~U[100, 1024], 16 q / 8 KV heads, head_dim 128, 1024-block pool."""
    g = _gen(seed + 10_000)
    lens = torch.randint(100, 1025, (num_seqs,), generator=g).tolist()
    return make_decode_case("qwen_decode_b128", lens, 16, 8, 128, 1024, seed,
                            max_blocks=4)


def long_decode(seed: int = 1003, num_seqs: int = 16, context_len: int = 32768,
                num_blocks: int = 2048) -> DecodeCase:
    """16 seqs x 32768 tokens over a fully used 2048-block pool, K scaled x3."""
    return make_decode_case("long_decode_32k", [context_len] * num_seqs, 16, 8, 128,
                            num_blocks, seed, k_scale=3.0)


def prefix_decode(seed: int = 1004, num_seqs: int = 64) -> DecodeCase:
    """64 seqs sharing 8 prefix blocks (2048 tokens) + private U[0,512] + 1 new token."""
    g = _gen(seed + 10_000)
    suffix = torch.randint(0, 513, (num_seqs,), generator=g).tolist()
    lens = [2048 + s + 1 for s in suffix]
    return make_decode_case("prefix_decode_b64", lens, 16, 8, 128, 1024, seed,
                            shared_prefix_blocks=8, max_blocks=11)


def chunked_prefill(seed: int = 1005, num_seqs: int = 8, cached: int = 4096,
                    chunk: int = 512, num_blocks: int = 256) -> PrefillCase:
    """8 seqs x 512-token chunk on 4096 cached tokens; ~5% of slots are -1."""
    return make_prefill_case("chunked_prefill_8x512", [cached] * num_seqs,
                             [chunk] * num_seqs, 16, 8, 128, num_blocks, seed,
                             skip_prob=0.05)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "qwen_decode_b128": qwen_decode,
    "long_decode_32k": long_decode,
    "prefix_decode_b64": prefix_decode,
    "chunked_prefill_8x512": chunked_prefill,
}


def block_manager_trace(seed: int, num_ops: int, num_prefixes: int = 4, vocab: int = 64,
                        max_live: int = 24, invalid_prob: float = 0.03) -> List[tuple]:
    """A seeded sequence of block-manager calls with a serving-like structure.

    Each new request's prompt is one of a few shared "system" prefixes (some a
    whole number of 256-token blocks, some not), or none, followed by its own
    tokens; live sequences grow by prefill chunks and single decoded tokens and
    are freed at random.  The ops are tuples:

      ("allocate", seq_id, tokens)   ("append", seq_id, tokens)
      ("free", seq_id)               ("slots", seq_id, begin, end)
      ("tables", [seq_id, ...], max_blocks)
      ("decode", [seq_id, ...], tokens)   (one token for each sequence)
      ("step", [seq_id, ...], tokens, max_blocks)   (the same, with the step's tables)

    A small share of ops is invalid on purpose (unknown or repeated sequence
    ids, a token range past the end, a table narrower than a sequence, a
    decode step naming a sequence twice).  Only
    token ids and op choices are drawn here: which blocks the calls hand out
    is for the manager under test to decide.
    """
    g = _gen(seed)

    def randint(lo: int, hi: int) -> int:  # inclusive
        return int(torch.randint(lo, hi + 1, (1,), generator=g))

    def tokens(n: int) -> List[int]:
        return torch.randint(0, vocab, (n,), generator=g).tolist() if n else []

    prefix_lens = [256, 512, 300, 700, 1024, 130][:num_prefixes]
    prefixes = [tokens(n) for n in prefix_lens]
    live = {}  # seq id -> token count
    next_id = 0
    ops: List[tuple] = []
    for _ in range(num_ops):
        r = float(torch.rand((), generator=g))
        if r < invalid_prob:
            kind = randint(0, 4)
            if kind == 0:
                ops.append(("free", next_id + 1000))
            elif kind == 1 and live:
                ops.append(("allocate", list(live)[0], tokens(3)))
            elif kind == 2 and live:
                s = list(live)[randint(0, len(live) - 1)]
                ops.append(("slots", s, 0, live[s] + 1))
            elif kind == 3 and live:
                s = max(live, key=live.get)
                ops.append(("tables", [s], max(live[s] - 1, 0) // BLOCK_SIZE))
            elif live:
                s = list(live)[0]
                ops.append(("decode", [s, s], tokens(2)))
            continue
        if not live or (len(live) < max_live and r < 0.30):
            pick = randint(0, len(prefixes))
            prompt = (prefixes[pick] if pick < len(prefixes) else []) + tokens(randint(0, 600))
            ops.append(("allocate", next_id, prompt))
            live[next_id] = len(prompt)
            next_id += 1
        elif r < 0.45:
            s = list(live)[randint(0, len(live) - 1)]
            ops.append(("free", s))
            del live[s]
        elif r < 0.55:
            s = list(live)[randint(0, len(live) - 1)]
            chunk = tokens(randint(1, 400))
            ops.append(("append", s, chunk))
            live[s] += len(chunk)
        elif r < 0.70:
            s = list(live)[randint(0, len(live) - 1)]
            ops.append(("append", s, tokens(1)))
            live[s] += 1
        elif r < 0.85:
            ids = [s for s in torch.randperm(len(live), generator=g).tolist()]
            ids = [list(live)[i] for i in ids[:randint(1, len(live))]]
            if randint(0, 1):
                ops.append(("decode", ids, tokens(len(ids))))
            else:  # a table width that sometimes cannot hold the step
                width = max(-(-(live[s] + 1) // BLOCK_SIZE) for s in ids) + randint(-1, 1)
                ops.append(("step", ids, tokens(len(ids)), max(width, 0)))
            for s in ids:
                live[s] += 1
        elif r < 0.93:
            s = list(live)[randint(0, len(live) - 1)]
            b = randint(0, live[s])
            ops.append(("slots", s, b, randint(b, live[s])))
        else:
            ids = list(live)
            width = max(-(-n // BLOCK_SIZE) for n in live.values()) + randint(0, 2)
            ops.append(("tables", ids, width))
    return ops


def shared_prefix_prompts(seed: int = 1006, num_seqs: int = 128, prefix_len: int = 2048,
                          prompt_len: int = 4096, vocab: int = 32000) -> List[torch.Tensor]:
    """num_seqs int32 prompts of prompt_len token ids: one shared system prefix
    of prefix_len ids, then each prompt's own ids (uniform over the vocab)."""
    g = _gen(seed)
    prefix = torch.randint(0, vocab, (prefix_len,), generator=g, dtype=torch.int32)
    return [torch.cat([prefix, torch.randint(0, vocab, (prompt_len - prefix_len,), generator=g,
                                             dtype=torch.int32)]) for _ in range(num_seqs)]
