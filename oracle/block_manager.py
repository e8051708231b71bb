"""Plain model of the host block manager.

TEST INFRASTRUCTURE ONLY: imported by the tests, never by the library.  It
is a slow, direct statement of what the manager does, with exact token
prefixes (Python tuples) where the library uses chained 64-bit keys:

- A pool of 256-token blocks; new blocks come from the front of a free list,
  ceil(tokens / 256) per sequence (intelliparadigm.com Nano-vLLM article,
  §2.1 动态分块内存管理, DynamicMemoryPool).
- Each block has a reference count, the number of live sequences whose table
  holds it (blog.hotdry.top "1200行代码挑战vLLM", §2 内存管理策略: direct
  reference counting).
- The prefix cache (same article, §性能优化 1 前缀缓存): a full block is
  remembered under the whole token prefix that ends with it; a new prompt
  reuses the leading blocks whose prefixes it starts with, and those
  sequences share the physical blocks (ocdem.com nano-vllm article, §2.1
  "基石PagedAttention": 块表, 高效的内存共享).
- Delayed release (intelliparadigm.com article, §7.2 延迟释放策略): a block
  whose count drops to zero goes to the back of the free list and keeps its
  cached prefix until it is handed out again.

Readings taken where the pages are silent (the library takes the same ones):
only full blocks are cached; a prefix already cached in another block is not
registered again; a freed sequence releases its blocks from last to first;
an allocation or append that does not fit raises and changes nothing.

Errors raise ``BlockManagerError`` with ``kind`` "invalid" or "no_memory".
"""
from __future__ import annotations

BLOCK = 256


class BlockManagerError(Exception):
    def __init__(self, kind: str, msg: str = ""):
        super().__init__(f"{kind}: {msg}" if msg else kind)
        self.kind = kind


class BlockManagerModel:
    def __init__(self, num_blocks: int):
        if num_blocks <= 0:
            raise BlockManagerError("invalid", "num_blocks must be positive")
        self.free = list(range(num_blocks))  # index 0 is the front
        self.ref = [0] * num_blocks
        self.prefix_of = {}                  # block -> the prefix tuple it caches
        self.block_of = {}                   # prefix tuple -> block
        self.seqs = {}                       # seq id -> {"table": [...], "tokens": [...]}

    # -- block moves -------------------------------------------------------
    def _take_front(self) -> int:
        b = self.free.pop(0)
        if b in self.prefix_of:              # handed out again: its cached prefix is gone
            del self.block_of[self.prefix_of.pop(b)]
        self.ref[b] = 1
        return b

    def _register(self, b: int, prefix: tuple) -> None:
        if prefix not in self.block_of:
            self.block_of[prefix] = b
            self.prefix_of[b] = prefix

    def _release(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    # -- calls ---------------------------------------------------------------
    def num_free_blocks(self) -> int:
        return len(self.free)

    def ref_count(self, b: int) -> int:
        return self.ref[b] if 0 <= b < len(self.ref) else -1

    def allocate(self, seq_id: int, tokens) -> int:
        tokens = list(tokens)
        if seq_id in self.seqs:
            raise BlockManagerError("invalid", "sequence exists")
        n = len(tokens)
        n_blocks = -(-n // BLOCK)
        n_full = n // BLOCK
        hits = []
        for i in range(n_full):
            b = self.block_of.get(tuple(tokens[:(i + 1) * BLOCK]))
            if b is None:
                break
            hits.append(b)
        revived = sum(1 for b in hits if self.ref[b] == 0)
        if n_blocks - len(hits) + revived > len(self.free):
            raise BlockManagerError("no_memory")
        table = []
        for b in hits:
            if self.ref[b] == 0:
                self.free.remove(b)
            self.ref[b] += 1
            table.append(b)
        for i in range(len(hits), n_blocks):
            b = self._take_front()
            table.append(b)
            if i < n_full:
                self._register(b, tuple(tokens[:(i + 1) * BLOCK]))
        self.seqs[seq_id] = {"table": table, "tokens": tokens}
        return len(hits) * BLOCK

    def append(self, seq_id: int, new_tokens) -> list:
        seq = self._seq(seq_id)
        new_tokens = list(new_tokens)
        table, tokens = seq["table"], seq["tokens"]
        if -(-(len(tokens) + len(new_tokens)) // BLOCK) - len(table) > len(self.free):
            raise BlockManagerError("no_memory")
        slots = []
        for tok in new_tokens:
            if len(tokens) % BLOCK == 0:
                table.append(self._take_front())
            slots.append(table[-1] * BLOCK + len(tokens) % BLOCK)
            tokens.append(tok)
            if len(tokens) % BLOCK == 0:
                self._register(table[-1], tuple(tokens))
        return slots

    def append_decode(self, seq_ids, tokens) -> list:
        """One token for each of several distinct sequences, all or nothing."""
        seq_ids, tokens = list(seq_ids), list(tokens)
        if len(seq_ids) != len(tokens) or len(set(seq_ids)) != len(seq_ids):
            raise BlockManagerError("invalid", "sequence ids must be distinct, one token each")
        seqs = [self._seq(s) for s in seq_ids]
        if sum(1 for q in seqs if len(q["tokens"]) % BLOCK == 0) > len(self.free):
            raise BlockManagerError("no_memory")
        return [self.append(s, [tok])[0] for s, tok in zip(seq_ids, tokens)]

    def decode_step(self, seq_ids, tokens, max_blocks: int):
        """append_decode, then the step's tables; nothing changes on failure."""
        seq_ids = list(seq_ids)
        if len(set(seq_ids)) != len(seq_ids):
            raise BlockManagerError("invalid", "repeated sequence")
        for s in seq_ids:
            q = self._seq(s)
            if len(q["table"]) + (1 if len(q["tokens"]) % BLOCK == 0 else 0) > max_blocks:
                raise BlockManagerError("invalid", "table would outgrow max_blocks")
        slots = self.append_decode(seq_ids, tokens)
        rows, lens = self.block_tables(seq_ids, max_blocks)
        return slots, rows, lens

    def free_seq(self, seq_id: int) -> None:
        seq = self._seq(seq_id)
        for b in reversed(seq["table"]):
            self._release(b)
        del self.seqs[seq_id]

    def slots(self, seq_id: int, begin: int, end: int) -> list:
        seq = self._seq(seq_id)
        if begin < 0 or end < begin or end > len(seq["tokens"]):
            raise BlockManagerError("invalid", "token range")
        return [seq["table"][t // BLOCK] * BLOCK + t % BLOCK for t in range(begin, end)]

    def block_tables(self, seq_ids, max_blocks: int):
        rows, lens = [], []
        for s in seq_ids:
            seq = self._seq(s)
            if len(seq["table"]) > max_blocks:
                raise BlockManagerError("invalid", "table longer than max_blocks")
            rows.append(seq["table"] + [-1] * (max_blocks - len(seq["table"])))
            lens.append(len(seq["tokens"]))
        return rows, lens

    def _seq(self, seq_id: int):
        if seq_id not in self.seqs:
            raise BlockManagerError("invalid", "unknown sequence")
        return self.seqs[seq_id]
