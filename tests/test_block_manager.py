"""Host block manager: pins, parity with the plain model, ABI error handling.

The pins state what the pages fix (256-token blocks from the front of a free
deque, reference counts, prefix reuse of full blocks, delayed release) as
hand-worked expected values, plus the property that defines a correct
manager: every live sequence's block table leads, token by token, to a slot
whose K/V was written for exactly that sequence's prefix.  They run on both
the plain model in ``oracle/block_manager.py`` and the library, so the model
is pinned by them and not only by agreement with the library.  The parity
test then replays seeded serving-like traces through both and compares every
result and the whole pool state after every call.  No GPU is used.
"""
import ctypes
import inspect
import random

import pytest

import paged_kv_cache_493_b300 as pkv
from oracle.block_manager import BLOCK, BlockManagerError, BlockManagerModel
from paged_kv_cache_493_b300 import _build
from paged_kv_cache_493_b300.workloads import block_manager_trace


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


class Lib:
    """The library's manager behind the model's method names and errors."""

    KINDS = {pkv.PKV_ERR_INVALID_ARG: "invalid", pkv.PKV_ERR_NO_MEMORY: "no_memory"}

    def __init__(self, num_blocks: int):
        self.bm = pkv.BlockManager(num_blocks)
        self.num_blocks = num_blocks

    def _call(self, fn, *args):
        try:
            return fn(*args)
        except pkv.PkvError as e:
            raise BlockManagerError(self.KINDS.get(e.status, str(e.status))) from None

    def allocate(self, s, tokens):
        return self._call(self.bm.allocate, s, tokens)

    def append(self, s, tokens):
        return self._call(self.bm.append, s, tokens)

    def append_decode(self, ids, tokens):
        return self._call(self.bm.append_decode, ids, tokens)

    def decode_step(self, ids, tokens, max_blocks):
        return self._call(self.bm.decode_step, ids, tokens, max_blocks)

    def free_seq(self, s):
        return self._call(self.bm.free, s)

    def slots(self, s, b, e):
        return self._call(self.bm.slots, s, b, e)

    def block_tables(self, ids, mb):
        return self._call(self.bm.block_tables, ids, mb)

    def num_free_blocks(self):
        return self.bm.num_free_blocks()

    def ref_count(self, b):
        return self.bm.ref_count(b)


IMPLS = {"model": BlockManagerModel, "library": Lib}


@pytest.fixture(params=sorted(IMPLS))
def make(request):
    return IMPLS[request.param]


def toks(seed, n, vocab=1000):
    r = random.Random(seed)
    return [r.randrange(vocab) for _ in range(n)]


class CacheSim:
    """What the device cache holds: slot -> the token prefix whose K/V was
    last written there.  The caller writes the slots of tokens that are not
    already cached (as an engine would with pkv_store_kvcache).  A prefix is
    named by an interned id: (id of the prefix one token shorter, token) ->
    id, so equal ids mean equal prefixes exactly."""

    def __init__(self):
        self.content = {}
        self.tokens = {}
        self.chain = {}    # seq -> ids of its prefixes tokens[:1], tokens[:2], ...
        self.intern = {}

    def _extend(self, s, new):
        chain = self.chain.setdefault(s, [])
        for tok in new:
            key = (chain[-1] if chain else -1, tok)
            chain.append(self.intern.setdefault(key, len(self.intern)))

    def allocate(self, bm, s, tokens):
        cached = bm.allocate(s, tokens)
        assert cached % BLOCK == 0 and 0 <= cached <= len(tokens)
        self.tokens[s] = list(tokens)
        self._extend(s, tokens)
        for t, slot in enumerate(bm.slots(s, cached, len(tokens)), start=cached):
            self.content[slot] = self.chain[s][t]
        return cached

    def append(self, bm, s, new):
        start = len(self.tokens[s])
        slots = bm.append(s, new)
        self.tokens[s] += list(new)
        self._extend(s, new)
        for i, slot in enumerate(slots):
            self.content[slot] = self.chain[s][start + i]
        return slots

    def append_decode(self, bm, ids, new):
        starts = [len(self.tokens[s]) for s in ids]
        slots = bm.append_decode(ids, new)
        for s, tok, start, slot in zip(ids, new, starts, slots):
            self.tokens[s].append(tok)
            self._extend(s, [tok])
            self.content[slot] = self.chain[s][start]
        return slots

    def free(self, bm, s):
        bm.free_seq(s)
        del self.tokens[s]
        del self.chain[s]

    def check(self, bm, num_blocks):
        """Every live sequence reads its own prefix at every position; counts
        and the free pool agree with the tables."""
        ids = list(self.tokens)
        width = max([-(-len(t) // BLOCK) for t in self.tokens.values()] + [0])
        tables, lens = bm.block_tables(ids, width)
        refs = [0] * num_blocks
        for s, row, n in zip(ids, tables, lens):
            assert n == len(self.tokens[s])
            used = -(-n // BLOCK)
            assert all(b >= 0 for b in row[:used]) and all(b == -1 for b in row[used:])
            for b in row[:used]:
                refs[b] += 1
            slots = bm.slots(s, 0, n)
            assert slots == [row[t // BLOCK] * BLOCK + t % BLOCK for t in range(n)]
            assert [self.content.get(x) for x in slots] == self.chain[s], s
        assert [bm.ref_count(b) for b in range(num_blocks)] == refs
        assert bm.num_free_blocks() == refs.count(0)


# ---------------------------------------------------------------------------
# Pins (hand-worked values from the pages' rules), on both implementations.
# ---------------------------------------------------------------------------

def test_fresh_pool_hands_out_ceil_blocks_from_the_front(make):
    bm = make(10)
    assert bm.allocate(7, toks(1, 600)) == 0
    assert bm.block_tables([7], 4) == ([[0, 1, 2, -1]], [600])
    assert bm.num_free_blocks() == 7
    assert bm.slots(7, 254, 258) == [254, 255, 256, 257]
    assert bm.slots(7, 599, 600) == [2 * BLOCK + 87]
    assert bm.allocate(8, toks(2, 1)) == 0          # next block is the front one
    assert bm.block_tables([8], 1) == ([[3]], [1])
    assert bm.allocate(9, []) == 0                  # an empty prompt holds no block
    assert bm.block_tables([9], 0) == ([[]], [0])
    assert bm.num_free_blocks() == 6


def test_append_opens_a_block_only_at_a_boundary(make):
    bm = make(6)
    bm.allocate(0, toks(1, 255))
    assert bm.append(0, [5]) == [255]
    assert bm.append(0, [6, 7]) == [BLOCK, BLOCK + 1]
    assert bm.block_tables([0], 2) == ([[0, 1]], [258])
    bm.allocate(1, [])
    assert bm.append(1, [1]) == [2 * BLOCK]


def test_common_prefix_blocks_are_shared_and_counted(make):
    bm = make(10)
    system = toks(3, 512)
    assert bm.allocate(0, system + toks(4, 40)) == 0
    assert bm.allocate(1, system + toks(5, 300)) == 512
    (t0, t1), _ = bm.block_tables([0, 1], 4)
    assert t0[:2] == t1[:2] == [0, 1]
    assert t1[2:] == [3, 4] and t0[2] == 2
    assert [bm.ref_count(b) for b in range(5)] == [2, 2, 1, 1, 1]
    bm.free_seq(0)
    assert [bm.ref_count(b) for b in range(5)] == [1, 1, 0, 1, 1]


def test_only_the_leading_run_of_cached_blocks_is_reused(make):
    a, b, c = toks(6, BLOCK), toks(7, BLOCK), toks(8, BLOCK)
    bm = make(8)
    bm.allocate(0, a + b + c)
    assert bm.allocate(1, a + toks(9, BLOCK) + c) == BLOCK   # third block differs by prefix
    assert bm.allocate(2, b + c) == 0                        # same blocks, other prefix
    assert bm.allocate(3, a + b) == 2 * BLOCK


def test_a_partial_block_is_never_shared(make):
    bm = make(8)
    prompt = toks(10, 300)
    bm.allocate(0, prompt)
    assert bm.allocate(1, prompt) == BLOCK
    (t0, t1), _ = bm.block_tables([0, 1], 2)
    assert t0[0] == t1[0] and t0[1] != t1[1]


def test_a_block_filled_by_appends_enters_the_cache(make):
    bm = make(8)
    head = toks(11, 200)
    rest = toks(12, 56)
    bm.allocate(0, head)
    bm.append(0, rest[:50])
    bm.append(0, rest[50:])                      # block 0 is now full
    assert bm.allocate(1, head + rest + [1, 2]) == BLOCK
    assert bm.block_tables([1], 2)[0][0][0] == bm.block_tables([0], 1)[0][0][0]


def test_delayed_release_keeps_a_freed_prefix_until_reuse(make):
    bm = make(4)
    system = toks(13, 512)
    bm.allocate(0, system + toks(14, 10))        # blocks 0, 1, 2
    bm.free_seq(0)                               # free deque: 3, 2, 1, 0
    assert bm.num_free_blocks() == 4
    assert bm.allocate(1, system + toks(15, 5)) == 512
    assert bm.block_tables([1], 3) == ([[0, 1, 3]], [517])
    assert bm.num_free_blocks() == 1


def test_release_goes_last_block_first_to_the_back(make):
    bm = make(4)
    a, b = toks(16, BLOCK), toks(17, BLOCK)
    bm.allocate(0, a + b)                        # blocks 0, 1
    bm.free_seq(0)                               # free deque: 2, 3, 1, 0
    bm.allocate(1, toks(18, 1))                  # takes 2
    bm.allocate(2, toks(19, 1))                  # takes 3
    bm.allocate(3, toks(20, 1))                  # takes 1: the block of a + b is handed out
    assert bm.block_tables([1, 2, 3], 1)[0] == [[2], [3], [1]]
    assert bm.allocate(4, a) == BLOCK            # block 0 still holds a
    assert bm.block_tables([4], 1)[0] == [[0]]
    bm.free_seq(1)
    assert bm.allocate(5, a + b) == BLOCK        # a shared with sequence 4, b gone
    assert bm.block_tables([5], 2)[0] == [[0, 2]]
    assert bm.ref_count(0) == 2 and bm.num_free_blocks() == 0


def test_a_reused_block_forgets_its_old_prefix(make):
    bm = make(3)
    a = toks(22, BLOCK)
    bm.allocate(0, a)
    bm.free_seq(0)
    bm.allocate(1, toks(23, 3 * BLOCK))          # takes every block, 0 last
    bm.free_seq(1)
    assert bm.allocate(2, a) == 0


def test_not_enough_blocks_fails_and_changes_nothing(make):
    bm = make(3)
    x = toks(24, BLOCK)
    bm.allocate(0, x)
    bm.free_seq(0)                               # block 0 free but caching x
    bm.allocate(1, toks(25, 2 * BLOCK))          # takes 1, 2; free: 0
    with pytest.raises(BlockManagerError) as e:
        bm.allocate(2, x + toks(26, 5))          # needs 0 back + one fresh block
    assert e.value.kind == "no_memory"
    assert bm.num_free_blocks() == 1 and bm.ref_count(0) == 0
    assert bm.allocate(2, x) == BLOCK            # the cached block alone does fit
    assert bm.block_tables([2], 1)[0] == [[0]]


def test_append_that_does_not_fit_changes_nothing(make):
    bm = make(2)
    bm.allocate(0, toks(28, BLOCK))
    with pytest.raises(BlockManagerError) as e:
        bm.append(0, toks(29, BLOCK + 1))        # needs two more blocks, one is free
    assert e.value.kind == "no_memory"
    assert bm.block_tables([0], 2) == ([[0, -1]], [BLOCK])
    assert bm.num_free_blocks() == 1
    assert bm.append(0, [1]) == [BLOCK]


def test_decode_step_appends_one_token_per_sequence(make):
    bm = make(3)
    bm.allocate(0, toks(31, BLOCK))              # block 0, full
    bm.allocate(1, toks(32, 10))                 # block 1
    assert bm.append_decode([1, 0], [5, 6]) == [BLOCK + 10, 2 * BLOCK]
    assert bm.block_tables([0, 1], 2) == ([[0, 2], [1, -1]], [BLOCK + 1, 11])
    assert bm.append_decode([], []) == []
    with pytest.raises(BlockManagerError) as e:
        bm.append_decode([0, 0], [1, 2])
    assert e.value.kind == "invalid"
    with pytest.raises(BlockManagerError) as e:
        bm.append_decode([1, 7], [1, 2])
    assert e.value.kind == "invalid"
    assert bm.block_tables([0, 1], 2) == ([[0, 2], [1, -1]], [BLOCK + 1, 11])


def test_decode_step_that_does_not_fit_changes_nothing(make):
    bm = make(3)
    bm.allocate(0, toks(33, BLOCK))
    bm.allocate(1, toks(34, BLOCK))
    bm.allocate(2, toks(35, 5))                  # no block left
    with pytest.raises(BlockManagerError) as e:
        bm.append_decode([2, 0], [1, 2])         # sequence 0 needs a block
    assert e.value.kind == "no_memory"
    assert bm.block_tables([0, 1, 2], 1) == ([[0], [1], [2]], [BLOCK, BLOCK, 5])
    assert bm.append_decode([2], [9]) == [2 * BLOCK + 5]


def test_decode_step_gives_slots_tables_and_lengths(make):
    bm = make(3)
    bm.allocate(0, toks(36, BLOCK))              # block 0, full
    bm.allocate(1, toks(37, 10))                 # block 1
    assert bm.decode_step([1, 0], [5, 6], 2) == ([BLOCK + 10, 2 * BLOCK], [[1, -1], [0, 2]],
                                                  [11, BLOCK + 1])


def test_decode_step_that_outgrows_the_table_changes_nothing(make):
    bm = make(3)
    bm.allocate(0, toks(38, BLOCK))              # a full block: the next token opens another
    bm.allocate(1, toks(39, 3))
    with pytest.raises(BlockManagerError) as e:
        bm.decode_step([1, 0], [1, 2], 1)
    assert e.value.kind == "invalid"
    assert bm.block_tables([0, 1], 1) == ([[0], [1]], [BLOCK, 3])
    assert bm.num_free_blocks() == 1


def test_invalid_calls_raise_and_change_nothing(make):
    bm = make(4)
    bm.allocate(0, toks(30, 300))
    for call in (lambda: bm.allocate(0, [1]), lambda: bm.free_seq(5), lambda: bm.append(5, [1]),
                 lambda: bm.slots(0, 0, 301), lambda: bm.slots(0, 5, 4),
                 lambda: bm.block_tables([0], 1), lambda: bm.block_tables([0, 9], 2)):
        with pytest.raises(BlockManagerError) as e:
            call()
        assert e.value.kind == "invalid"
    assert bm.block_tables([0], 2) == ([[0, 1]], [300])
    assert bm.num_free_blocks() == 2


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_every_sequence_reads_its_own_prefix(make, seed):
    """Random shared-prefix traffic on a small pool (so blocks are evicted and
    reused): after every call each live sequence's slots hold its own K/V."""
    num_blocks = 20
    bm, sim = make(num_blocks), CacheSim()
    for op in block_manager_trace(seed, 400, max_live=10, invalid_prob=0.0):
        try:
            if op[0] == "allocate":
                sim.allocate(bm, op[1], op[2])
            elif op[0] == "append" and op[1] in sim.tokens:
                sim.append(bm, op[1], op[2])
            elif op[0] == "free" and op[1] in sim.tokens:
                sim.free(bm, op[1])
            elif op[0] in ("decode", "step") and all(x in sim.tokens for x in op[1]):
                sim.append_decode(bm, op[1], op[2])
        except BlockManagerError as e:
            assert e.kind == "no_memory"
        sim.check(bm, num_blocks)


# ---------------------------------------------------------------------------
# Parity: the library against the model on seeded traces, call by call.
# ---------------------------------------------------------------------------

def run_op(bm, op):
    """The op's result, or ("error", kind)."""
    try:
        if op[0] == "allocate":
            return bm.allocate(op[1], op[2])
        if op[0] == "append":
            return bm.append(op[1], op[2])
        if op[0] == "free":
            return bm.free_seq(op[1])
        if op[0] == "slots":
            return bm.slots(op[1], op[2], op[3])
        if op[0] == "decode":
            return bm.append_decode(op[1], op[2])
        if op[0] == "step":
            return bm.decode_step(op[1], op[2], op[3])
        return bm.block_tables(op[1], op[2])
    except BlockManagerError as e:
        return ("error", e.kind)


@pytest.mark.parametrize("seed,num_blocks,num_ops,max_live", [
    (10, 16, 800, 8), (11, 40, 1500, 24), (12, 96, 1500, 48), (13, 7, 600, 6)])
def test_library_matches_model_call_by_call(seed, num_blocks, num_ops, max_live):
    model, lib = BlockManagerModel(num_blocks), Lib(num_blocks)
    live = set()
    outcomes = set()
    for i, op in enumerate(block_manager_trace(seed, num_ops, max_live=max_live)):
        want, got = run_op(model, op), run_op(lib, op)
        assert got == want, (i, op[0])
        failed = isinstance(want, tuple) and want[:1] == ("error",)
        outcomes.add(want if failed else op[0])
        if op[0] == "allocate" and not failed:
            live.add(op[1])
        elif op[0] == "free" and not failed:
            live.discard(op[1])
        assert lib.num_free_blocks() == model.num_free_blocks(), i
        assert [lib.ref_count(b) for b in range(num_blocks)] == model.ref, i
        width = max([len(model.seqs[s]["table"]) for s in live] + [0])
        assert lib.block_tables(sorted(live), width) == model.block_tables(sorted(live), width), i
    assert {("error", "invalid"), ("error", "no_memory"), "allocate", "append", "free", "slots",
            "tables", "decode", "step"} <= outcomes


def test_block_tables_into_fills_host_tensors():
    import torch
    bm = pkv.BlockManager(16)
    bm.allocate(3, toks(40, 700))
    bm.allocate(5, toks(40, 512) + [1])
    tables = torch.full((2, 4), 77, dtype=torch.int32)
    lens = torch.zeros(2, dtype=torch.int32)
    bm.block_tables_into([5, 3], tables, lens)
    assert tables.tolist() == [[0, 1, 3, -1], [0, 1, 2, -1]]
    assert lens.tolist() == [513, 700]


def test_binding_takes_tensors_and_arrays_in_place():
    import numpy as np
    import torch
    prompt = toks(41, 300)
    bm, model = pkv.BlockManager(8), BlockManagerModel(8)
    assert bm.allocate(0, torch.tensor(prompt, dtype=torch.int32)) == model.allocate(0, prompt)
    assert bm.allocate(1, np.array(prompt, dtype=np.int32)) == model.allocate(1, prompt)
    assert bm.append(0, np.array([3, 4], dtype=np.int32)) == model.append(0, [3, 4])
    ids = torch.tensor([1, 0], dtype=torch.int64)
    slots = torch.empty(2, dtype=torch.int32)
    bm.append_decode_into(ids, torch.tensor([8, 9], dtype=torch.int32), slots)
    assert slots.tolist() == model.append_decode([1, 0], [8, 9])
    with pytest.raises(pkv.PkvError):
        bm.allocate(2, torch.tensor(prompt, dtype=torch.int64))   # wrong dtype
    with pytest.raises(pkv.PkvError):
        bm.append_decode_into(ids, torch.tensor([1], dtype=torch.int32), slots)


# ---------------------------------------------------------------------------
# The C ABI itself: argument checks, nothing written on failure.
# ---------------------------------------------------------------------------

def test_abi_rejects_bad_arguments():
    lib = pkv.load_library()
    h = ctypes.c_void_p()
    I32 = ctypes.c_int32
    assert lib.pkv_bm_create(0, ctypes.byref(h)) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_bm_create(2 ** 31 // 256, ctypes.byref(h)) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_bm_create(4, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.pkv_bm_num_free_blocks(None) == 0
    assert lib.pkv_bm_ref_count(None, 0) == -1
    lib.pkv_bm_destroy(None)
    assert lib.pkv_bm_create(4, ctypes.byref(h)) == pkv.PKV_OK
    try:
        three = (I32 * 3)(1, 2, 3)
        assert lib.pkv_bm_allocate(None, 0, three, 3, None) == pkv.PKV_ERR_INVALID_ARG
        assert lib.pkv_bm_allocate(h, 0, None, 3, None) == pkv.PKV_ERR_INVALID_ARG
        assert lib.pkv_bm_allocate(h, 0, three, -1, None) == pkv.PKV_ERR_INVALID_ARG
        assert lib.pkv_bm_allocate(h, 0, None, 0, None) == pkv.PKV_OK      # empty prompt
        assert lib.pkv_bm_append(h, 0, three, 3, None) == pkv.PKV_OK       # slots optional
        assert lib.pkv_bm_append(h, 0, None, 1, None) == pkv.PKV_ERR_INVALID_ARG
        assert lib.pkv_bm_append(h, 0, three, -2, None) == pkv.PKV_ERR_INVALID_ARG
        assert lib.pkv_bm_ref_count(h, 4) == -1 and lib.pkv_bm_ref_count(h, -1) == -1
        ids = (ctypes.c_int64 * 2)(0, 9)
        table = (I32 * 4)(55, 55, 55, 55)
        lens = (I32 * 2)(55, 55)
        assert lib.pkv_bm_block_tables(h, ids, 2, 2, table, lens) == pkv.PKV_ERR_INVALID_ARG
        assert list(table) == [55] * 4 and list(lens) == [55, 55]       # nothing written
        assert lib.pkv_bm_block_tables(h, ids, 1, 2, None, lens) == pkv.PKV_ERR_INVALID_ARG
        assert lib.pkv_bm_block_tables(h, ids, -1, 2, table, lens) == pkv.PKV_ERR_INVALID_ARG
        assert lib.pkv_bm_block_tables(h, ids, 1, 2, table, lens) == pkv.PKV_OK
        assert list(table[:2]) == [0, -1] and lens[0] == 3
        out = (I32 * 3)()
        assert lib.pkv_bm_slots(h, 0, 0, 3, out) == pkv.PKV_OK and list(out) == [0, 1, 2]
        assert lib.pkv_bm_slots(h, 0, 0, 3, None) == pkv.PKV_ERR_INVALID_ARG
        assert lib.pkv_bm_slots(h, 0, -1, 2, out) == pkv.PKV_ERR_INVALID_ARG
        assert lib.pkv_bm_slots(h, 0, 2, 4, out) == pkv.PKV_ERR_INVALID_ARG
        assert lib.pkv_bm_free(h, 1) == pkv.PKV_ERR_INVALID_ARG
        assert lib.pkv_bm_free(h, 0) == pkv.PKV_OK
        assert lib.pkv_bm_num_free_blocks(h) == 4
    finally:
        lib.pkv_bm_destroy(h)


# ---------------------------------------------------------------------------
# The pins catch plausible mistakes planted in the model.
# ---------------------------------------------------------------------------

MODEL_SRC = open(inspect.getsourcefile(BlockManagerModel)).read()

MUTANTS = {
    "release_to_front": ("self.free.append(b)", "self.free.insert(0, b)"),
    "release_first_to_last": ('for b in reversed(seq["table"]):', 'for b in seq["table"]:'),
    "key_is_the_block_alone": ("self.block_of.get(tuple(tokens[:(i + 1) * BLOCK]))",
                               "self.block_of.get(tuple(tokens[i * BLOCK:(i + 1) * BLOCK]))"),
    "appended_key_is_the_block_alone": ("self._register(table[-1], tuple(tokens))",
                                        "self._register(table[-1], tuple(tokens[-BLOCK:]))"),
    "hits_skip_a_miss": ("                break\n            hits.append(b)",
                         "                continue\n            hits.append(b)"),
    "shared_count_reset": ("            self.ref[b] += 1\n", "            self.ref[b] = 1\n"),
    "reuse_keeps_old_prefix": ("            del self.block_of[self.prefix_of.pop(b)]",
                               "            pass"),
    "revived_blocks_not_counted": ("n_blocks - len(hits) + revived", "n_blocks - len(hits)"),
    "slot_without_block_size": ('["table"][t // BLOCK] * BLOCK + t % BLOCK',
                                '["table"][t // BLOCK] + t % BLOCK'),
    "new_block_one_late": ("            if len(tokens) % BLOCK == 0:\n                table.append",
                           "            if len(tokens) % BLOCK == 1 or not table:\n                table.append"),
    "register_overwrites": ("        if prefix not in self.block_of:\n",
                            "        if True:\n"),
    "free_check_ignores_table": ("- len(table) > len(self.free)", "> len(self.free)"),
    "decode_counts_every_sequence": ('len(q["tokens"]) % BLOCK == 0)', 'len(q["tokens"]) % BLOCK >= 0)'),
    "decode_allows_repeats": ("or len(set(seq_ids)) != len(seq_ids)", ""),
    "step_width_off_by_one": ("if len(q[\"table\"]) + (1 if len(q[\"tokens\"]) % BLOCK == 0 else 0) > max_blocks:",
                              "if len(q[\"table\"]) > max_blocks:"),
}

PIN_TESTS = [
    test_fresh_pool_hands_out_ceil_blocks_from_the_front,
    test_append_opens_a_block_only_at_a_boundary,
    test_common_prefix_blocks_are_shared_and_counted,
    test_only_the_leading_run_of_cached_blocks_is_reused,
    test_a_partial_block_is_never_shared,
    test_a_block_filled_by_appends_enters_the_cache,
    test_delayed_release_keeps_a_freed_prefix_until_reuse,
    test_release_goes_last_block_first_to_the_back,
    test_a_reused_block_forgets_its_old_prefix,
    test_not_enough_blocks_fails_and_changes_nothing,
    test_append_that_does_not_fit_changes_nothing,
    test_invalid_calls_raise_and_change_nothing,
    test_decode_step_appends_one_token_per_sequence,
    test_decode_step_that_does_not_fit_changes_nothing,
    test_decode_step_gives_slots_tables_and_lengths,
    test_decode_step_that_outgrows_the_table_changes_nothing,
    lambda make: test_every_sequence_reads_its_own_prefix(make, 0),
    lambda make: test_every_sequence_reads_its_own_prefix(make, 1),
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mistakes_planted_in_the_model(name):
    old, new = MUTANTS[name]
    assert MODEL_SRC.count(old) == 1, f"mutation site for {name} not found once"
    ns = {}
    exec(compile(MODEL_SRC.replace(old, new), f"<mutant {name}>", "exec"), ns)
    mutant = ns["BlockManagerModel"]
    caught = None
    for pin in PIN_TESTS:
        try:
            pin(mutant)
        except Exception as e:  # an assertion, or the mutant crashing
            caught = e
            break
    assert caught is not None, f"no pin caught mutant {name}"
