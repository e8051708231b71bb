"""Pins of the fp64 CPU oracle against things other than itself.

Each pin fixes something a plausible oracle bug would break:
  * hand-worked closed forms (tests/golden/hand_examples.json): addressing
    across a block boundary, the bottom-right causal rule, GQA grouping,
    the store's slot arithmetic;
  * the host library's fp64 scaled-dot-product attention in the special case
    of contiguous blocks (decode, prefill with a cached prefix through
    ``causal_lower_right``, prefill with no prefix through ``is_causal``);
  * brute force written as direct per-key loops on tiny inputs;
  * closed forms: one key, zero query, equal keys, a dominant key;
  * invariances the pages fix: relabelling physical blocks, shared prefix
    blocks versus private copies, softmax rows summing to one;
  * the store against the library's own indexed assignment.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from torch.nn.attention.bias import causal_lower_right

import oracle
from paged_kv_cache_493_b300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore")

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")))
BS = W.BLOCK_SIZE


def bf(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)


def f64(t):
    return t.to(torch.float64)


# ---------------------------------------------------------------------------
# Hand-worked closed forms
# ---------------------------------------------------------------------------

def _boundary_cache():
    g = GOLDEN["decode_block_boundary"]
    nb, d = g["num_blocks"], g["head_dim"]
    k = torch.empty(nb, BS, 1, d)
    v = torch.empty(nb, BS, 1, d)
    k[:] = torch.tensor(g["filler"], dtype=torch.float32)
    v[:] = torch.tensor(g["filler"], dtype=torch.float32)
    table = g["block_table"]
    for t in range(g["context_len"]):
        blk, off = table[t // BS], t % BS
        last = t == g["context_len"] - 1
        k[blk, off, 0] = torch.tensor(g["key_last"] if last else g["key_low"], dtype=torch.float32)
        v[blk, off, 0] = torch.tensor(g["value_last"] if last else g["value_low"], dtype=torch.float32)
    return g, k.to(torch.bfloat16), v.to(torch.bfloat16)


def test_golden_decode_block_boundary():
    g, kc, vc = _boundary_cache()
    q = bf([[g["q"]]])
    out = oracle.decode(q, kc, vc, torch.tensor([g["block_table"]]), [g["context_len"]],
                        math.log(g["scale_ln"]))
    np.testing.assert_allclose(out[0, 0], g["expected"], rtol=0, atol=1e-12)


def test_golden_prefill_bottom_right():
    g, kc, vc = _boundary_cache()
    p = GOLDEN["prefill_bottom_right"]
    q = bf([[g["q"]], [g["q"]]])
    out = oracle.prefill(q, kc, vc, torch.tensor([g["block_table"]]), p["cu_seqlens_q"],
                         [g["context_len"]], math.log(g["scale_ln"]))
    np.testing.assert_allclose(out[:, 0], p["expected"], rtol=0, atol=1e-12)


def test_golden_gqa_grouping():
    g = GOLDEN["gqa_grouping"]
    kc = torch.zeros(1, BS, g["num_kv_heads"], g["head_dim"])
    vc = torch.zeros_like(kc)
    for t in range(g["context_len"]):
        kc[0, t] = torch.tensor(g["keys"][t], dtype=torch.float32)
        vc[0, t] = torch.tensor(g["values"][t], dtype=torch.float32)
    q = bf([[[1, 0]] * g["num_q_heads"]])
    out = oracle.decode(q, kc.to(torch.bfloat16), vc.to(torch.bfloat16), torch.tensor([[0]]),
                        [g["context_len"]], math.log(g["scale_ln"]))
    np.testing.assert_allclose(out[0], g["expected"], rtol=0, atol=1e-12)


def test_golden_store_rows():
    g = GOLDEN["store_rows"]
    kc = torch.zeros(g["num_blocks"], BS, 1, 2, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    k, v = bf(g["k"]).view(3, 1, 2), bf(g["v"]).view(3, 1, 2)
    nk, nv = oracle.store_kvcache(k, v, g["slot_mapping"], kc, vc)
    ek = torch.zeros_like(kc, dtype=torch.float32)
    ev = torch.zeros_like(ek)
    for key, val in g["expected_k"].items():
        b, o = map(int, key.split(","))
        ek[b, o, 0] = torch.tensor(val, dtype=torch.float32)
    for key, val in g["expected_v"].items():
        b, o = map(int, key.split(","))
        ev[b, o, 0] = torch.tensor(val, dtype=torch.float32)
    assert torch.equal(nk.float(), ek) and torch.equal(nv.float(), ev)


# ---------------------------------------------------------------------------
# Library routine in the contiguous special case
# ---------------------------------------------------------------------------

def contiguous_case(ctx, hq, hkv, d, seed, extra_blocks=0):
    """Sequence s owns physical blocks s*n .. s*n+n-1 in order (identity paging)."""
    gen = torch.Generator().manual_seed(seed)
    n = max(1, max(math.ceil(c / BS) for c in ctx))
    nb = n * len(ctx) + extra_blocks
    kc = W.randn_bf16((nb, BS, hkv, d), gen, 2.0)
    vc = W.randn_bf16((nb, BS, hkv, d), gen)
    tables = torch.tensor([[s * n + j for j in range(n)] for s in range(len(ctx))], dtype=torch.int32)
    return kc, vc, tables, n, gen


def seq_kv(kc, vc, s, n, c):
    K = f64(kc[s * n:(s + 1) * n].reshape(-1, kc.shape[2], kc.shape[3])[:c])
    V = f64(vc[s * n:(s + 1) * n].reshape(-1, vc.shape[2], vc.shape[3])[:c])
    return K.permute(1, 0, 2).unsqueeze(0), V.permute(1, 0, 2).unsqueeze(0)  # [1, Hkv, C, D]


@pytest.mark.parametrize("hq,hkv,d", [(4, 2, 64), (16, 8, 128), (8, 1, 32), (6, 6, 16)])
def test_decode_matches_library_sdpa(hq, hkv, d):
    ctx = [1, 37, 255, 256, 257, 600]
    kc, vc, tables, n, gen = contiguous_case(ctx, hq, hkv, d, seed=11 + d)
    q = W.randn_bf16((len(ctx), hq, d), gen)
    scale = 1 / math.sqrt(d)
    out = oracle.decode(q, kc, vc, tables, ctx, scale)
    for s, c in enumerate(ctx):
        K, V = seq_kv(kc, vc, s, n, c)
        ref = F.scaled_dot_product_attention(f64(q[s]).unsqueeze(0).unsqueeze(2), K, V,
                                             scale=scale, enable_gqa=True)
        np.testing.assert_allclose(out[s], ref[0, :, 0].numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("cached,lq", [(0, 1), (0, 37), (200, 100), (256, 1), (511, 3), (300, 300)])
def test_prefill_matches_library_sdpa_lower_right(cached, lq):
    hq, hkv, d = 4, 2, 32
    ctx = [cached + lq, cached + lq + 5]
    lqs = [lq, lq + 5]
    kc, vc, tables, n, gen = contiguous_case(ctx, hq, hkv, d, seed=cached * 7 + lq)
    total = sum(lqs)
    q = W.randn_bf16((total, hq, d), gen)
    cu = [0, lqs[0], total]
    scale = 0.125
    out = oracle.prefill(q, kc, vc, tables, cu, ctx, scale)
    for s in range(2):
        K, V = seq_kv(kc, vc, s, n, ctx[s])
        qs = f64(q[cu[s]:cu[s + 1]]).permute(1, 0, 2).unsqueeze(0)
        mask = causal_lower_right(lqs[s], ctx[s])._materialize()
        ref = F.scaled_dot_product_attention(qs, K, V, attn_mask=mask, scale=scale, enable_gqa=True)
        np.testing.assert_allclose(out[cu[s]:cu[s + 1]], ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_prefill_without_prefix_is_plain_causal():
    hq, hkv, d = 4, 4, 16
    ctx = [40, 300]
    kc, vc, tables, n, gen = contiguous_case(ctx, hq, hkv, d, seed=5)
    q = W.randn_bf16((sum(ctx), hq, d), gen)
    cu = [0, 40, 340]
    out = oracle.prefill(q, kc, vc, tables, cu, ctx, 0.3)
    for s in range(2):
        K, V = seq_kv(kc, vc, s, n, ctx[s])
        qs = f64(q[cu[s]:cu[s + 1]]).permute(1, 0, 2).unsqueeze(0)
        ref = F.scaled_dot_product_attention(qs, K, V, is_causal=True, scale=0.3)
        np.testing.assert_allclose(out[cu[s]:cu[s + 1]], ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Brute force: per-key loops straight from the definition, no gather helper
# ---------------------------------------------------------------------------

def brute_decode_row(q, kc, vc, table_row, c, h, group, scale):
    kh = h // group
    logits = []
    for t in range(c):
        blk = int(table_row[t // BS])
        k = kc[blk, t % BS, kh].double().tolist()
        logits.append(scale * math.fsum(a * b for a, b in zip(q, k)))
    m = max(logits)
    w = [math.exp(x - m) for x in logits]
    z = math.fsum(w)
    out = []
    for dd in range(len(q)):
        out.append(math.fsum(w[t] / z * float(vc[int(table_row[t // BS]), t % BS, kh, dd]) for t in range(c)))
    return out


def test_brute_force_tiny_decode():
    case = W.make_decode_case("t", [1, 5, 257, 300], 4, 2, 4, 6, seed=3)
    c = case.cache
    out = oracle.decode(case.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, case.scale)
    for s in range(4):
        for h in range(4):
            ref = brute_decode_row(case.q[s, h].double().tolist(), c.k_cache, c.v_cache,
                                   c.block_tables[s], int(c.context_lens[s]), h, 2, case.scale)
            np.testing.assert_allclose(out[s, h], ref, rtol=0, atol=1e-12)


def test_brute_force_tiny_prefill():
    case = W.make_prefill_case("t", [3, 250], [4, 9], 2, 1, 4, 4, seed=8)
    c = case.cache
    cu = case.cu_seqlens_q.tolist()
    out = oracle.prefill(case.q, c.k_cache, c.v_cache, c.block_tables, cu, c.context_lens, case.scale)
    for s in range(2):
        ctx = int(c.context_lens[s])
        lq = cu[s + 1] - cu[s]
        for i in range(lq):
            for h in range(2):
                ref = brute_decode_row(case.q[cu[s] + i, h].double().tolist(), c.k_cache, c.v_cache,
                                       c.block_tables[s], ctx - lq + i + 1, h, 2, case.scale)
                np.testing.assert_allclose(out[cu[s] + i, h], ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------

def test_single_key_returns_its_value_exactly():
    case = W.tiny_decode()
    c = case.cache
    out = oracle.decode(case.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, case.scale)
    assert int(c.context_lens[0]) == 1
    blk = int(c.block_tables[0, 0])
    for h in range(4):
        assert np.array_equal(out[0, h], f64(c.v_cache[blk, 0, h // 2]).numpy())


def test_zero_query_gives_mean_value():
    case = W.make_decode_case("t", [37, 513], 4, 2, 8, 6, seed=4)
    c = case.cache
    q = torch.zeros_like(case.q)
    out = oracle.decode(q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, case.scale)
    for s in range(2):
        K, V = oracle.gather(c.k_cache, c.v_cache, c.block_tables[s], int(c.context_lens[s]))
        for h in range(4):
            np.testing.assert_allclose(out[s, h], V[:, h // 2].mean(axis=0), rtol=0, atol=1e-12)


def test_equal_keys_give_mean_value():
    case = W.make_decode_case("t", [300], 2, 1, 8, 4, seed=6)
    c = case.cache
    kc = c.k_cache.clone()
    kc[:] = kc[0, 0, 0]
    out = oracle.decode(case.q, kc, c.v_cache, c.block_tables, c.context_lens, case.scale)
    table = c.block_tables[0].tolist()
    vals = torch.stack([c.v_cache[table[t // BS], t % BS, 0] for t in range(300)])
    np.testing.assert_allclose(out[0, 0], f64(vals).mean(0).numpy(), rtol=0, atol=1e-12)


def test_dominant_key_selects_its_value():
    case = W.make_decode_case("t", [700], 2, 1, 16, 4, seed=9)
    c = case.cache
    kc = c.k_cache.clone()
    q = torch.zeros_like(case.q)
    q[0, :, 0] = 1.0
    kc[..., 0] = 0.0
    t_star = 421
    blk = int(c.block_tables[0, t_star // BS])
    kc[blk, t_star % BS, 0, 0] = 256.0        # logit gap 256 * scale = 64 nats
    out = oracle.decode(q, kc, c.v_cache, c.block_tables, c.context_lens, 0.25)
    np.testing.assert_allclose(out[0, 0], f64(c.v_cache[blk, t_star % BS, 0]).numpy(), rtol=0, atol=1e-12)


def test_empty_context_gives_zeros():
    case = W.make_decode_case("t", [0, 3], 2, 1, 8, 4, seed=2)
    c = case.cache
    out = oracle.decode(case.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, case.scale)
    assert np.all(out[0] == 0) and np.all(np.isfinite(out))


# ---------------------------------------------------------------------------
# Invariances the pages fix
# ---------------------------------------------------------------------------

def relabel_blocks(kc, vc, tables, perm):
    """Move physical block b to perm[b] and rewrite the tables accordingly."""
    nk = torch.empty_like(kc)
    nv = torch.empty_like(vc)
    nk[perm] = kc
    nv[perm] = vc
    nt = tables.clone()
    valid = tables >= 0
    nt[valid] = torch.as_tensor(perm, dtype=torch.int32)[tables[valid].long()]
    return nk, nv, nt


def test_block_relabelling_is_invisible():
    case = W.make_decode_case("t", [1, 255, 256, 257, 700], 4, 2, 16, 16, seed=12)
    c = case.cache
    ref = oracle.decode(case.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, case.scale)
    perm = torch.randperm(c.num_blocks, generator=torch.Generator().manual_seed(1))
    nk, nv, nt = relabel_blocks(c.k_cache, c.v_cache, c.block_tables, perm)
    assert not torch.equal(nt, c.block_tables)
    out = oracle.decode(case.q, nk, nv, nt, c.context_lens, case.scale)
    assert np.array_equal(out, ref)


def test_shared_prefix_equals_private_copies():
    case = W.make_decode_case("t", [2 * BS + 5, 2 * BS + 300, 2 * BS + 1], 4, 2, 16, 16, seed=13,
                              shared_prefix_blocks=2)
    c = case.cache
    tb = c.block_tables
    assert torch.equal(tb[0, :2], tb[1, :2]) and torch.equal(tb[0, :2], tb[2, :2])
    ref = oracle.decode(case.q, c.k_cache, c.v_cache, tb, c.context_lens, case.scale)
    # Give sequences 1 and 2 private copies of the two shared blocks.
    used = set(int(x) for x in tb.flatten().tolist() if x >= 0)
    free = [b for b in range(c.num_blocks) if b not in used]
    kc, vc, nt = c.k_cache.clone(), c.v_cache.clone(), tb.clone()
    for s in (1, 2):
        for j in range(2):
            dst = free.pop()
            kc[dst] = c.k_cache[int(tb[s, j])]
            vc[dst] = c.v_cache[int(tb[s, j])]
            nt[s, j] = dst
    out = oracle.decode(case.q, kc, vc, nt, c.context_lens, case.scale)
    assert np.array_equal(out, ref)


def test_softmax_rows_sum_to_one():
    case = W.make_decode_case("t", [1, 700], 2, 1, 32, 8, seed=14, k_scale=3.0)
    c = case.cache
    for s in range(2):
        n = int(c.context_lens[s])
        K, V = oracle.gather(c.k_cache, c.v_cache, c.block_tables[s], n)
        out, p = oracle.attend(f64(case.q[s, 0]).numpy(), K, V, 0, n, case.scale)
        assert p.shape == (n,) and np.all(p >= 0)
        assert abs(math.fsum(p) - 1.0) <= 1e-12
        np.testing.assert_allclose(out, p @ V[:, 0], rtol=0, atol=1e-12)


def test_prefill_of_one_query_equals_decode():
    case = W.make_decode_case("t", [1, 256, 257, 513], 4, 2, 16, 12, seed=15)
    c = case.cache
    dec = oracle.decode(case.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, case.scale)
    pre = oracle.prefill(case.q, c.k_cache, c.v_cache, c.block_tables, [0, 1, 2, 3, 4],
                         c.context_lens, case.scale)
    assert np.array_equal(dec, pre)


def test_sampled_rows_equal_full_output():
    case = W.make_prefill_case("t", [10, 300], [20, 7], 4, 2, 16, 8, seed=16)
    c = case.cache
    full = oracle.prefill(case.q, c.k_cache, c.v_cache, c.block_tables, case.cu_seqlens_q,
                          c.context_lens, case.scale)
    rows = [(0, 0), (19, 3), (20, 1), (26, 2), (0, 0), (19, 3)]   # repeats allowed
    part = oracle.prefill(case.q, c.k_cache, c.v_cache, c.block_tables, case.cu_seqlens_q,
                          c.context_lens, case.scale, rows=rows)
    for i, (t, h) in enumerate(rows):
        assert np.array_equal(part[i], full[t, h])
    dcase = W.tiny_decode()
    dc = dcase.cache
    dfull = oracle.decode(dcase.q, dc.k_cache, dc.v_cache, dc.block_tables, dc.context_lens, dcase.scale)
    drows = [(3, 1), (0, 2), (3, 1)]
    dpart = oracle.decode(dcase.q, dc.k_cache, dc.v_cache, dc.block_tables, dc.context_lens,
                          dcase.scale, rows=drows)
    for i, (s, h) in enumerate(drows):
        assert np.array_equal(dpart[i], dfull[s, h])


# ---------------------------------------------------------------------------
# Store
# ---------------------------------------------------------------------------

def test_store_matches_indexed_assignment():
    case = W.chunked_prefill(num_seqs=2, cached=300, chunk=100, num_blocks=8)
    c = case.cache
    nk, nv = oracle.store_kvcache(case.k_new, case.v_new, case.slot_mapping, c.k_cache, c.v_cache)
    sm = case.slot_mapping.long()
    keep = sm >= 0
    assert 0 < int((~keep).sum()) < sm.numel()
    rk = c.k_cache.clone().view(-1, *c.k_cache.shape[2:])
    rv = c.v_cache.clone().view(-1, *c.v_cache.shape[2:])
    rk[sm[keep]] = case.k_new[keep]
    rv[sm[keep]] = case.v_new[keep]
    assert torch.equal(nk.view(torch.int16), rk.view_as(nk).view(torch.int16))
    assert torch.equal(nv.view(torch.int16), rv.view_as(nv).view(torch.int16))
    # Slots that no row maps to keep their bits; skipped rows leave no trace.
    touched = torch.zeros(c.k_cache.shape[0] * BS, dtype=torch.bool)
    touched[sm[keep]] = True
    flat_old = c.k_cache.view(-1, *c.k_cache.shape[2:])
    flat_new = nk.view(-1, *nk.shape[2:])
    assert torch.equal(flat_old[~touched].view(torch.int16), flat_new[~touched].view(torch.int16))


def test_store_rejects_out_of_range_slot():
    case = W.tiny_decode()
    c = case.cache
    for bad in (8 * BS, -2):
        sm = case.slot_mapping.clone()
        sm[1] = bad
        with pytest.raises(oracle.OracleError):
            oracle.store_kvcache(case.k_new, case.v_new, sm, c.k_cache, c.v_cache)


def test_invalid_inputs_are_rejected():
    case = W.tiny_decode()
    c = case.cache
    bad_table = c.block_tables.clone()
    bad_table[3, 1] = 8
    with pytest.raises(oracle.OracleError):
        oracle.decode(case.q, c.k_cache, c.v_cache, bad_table, c.context_lens, case.scale)
    with pytest.raises(oracle.OracleError):   # context beyond the table width
        oracle.decode(case.q, c.k_cache, c.v_cache, c.block_tables, [1, 37, 256, 513], case.scale)
    with pytest.raises(oracle.OracleError):   # chunk longer than its context
        oracle.prefill(case.q, c.k_cache, c.v_cache, c.block_tables, [0, 2, 3, 4, 4],
                       c.context_lens, case.scale)
    q3 = W.randn_bf16((4, 3, 64), torch.Generator().manual_seed(0))
    with pytest.raises(oracle.OracleError):   # 3 q heads over 2 KV heads
        oracle.decode(q3, c.k_cache, c.v_cache, c.block_tables, c.context_lens, case.scale)


# ---------------------------------------------------------------------------
# The named workloads have the stated structure
# ---------------------------------------------------------------------------

def test_workload_structure():
    t = W.tiny_decode()
    assert t.cache.context_lens.tolist() == [1, 37, 256, 300]
    used = [int(x) for x in t.cache.block_tables.flatten().tolist() if x >= 0]
    assert len(used) == 5 and len(set(used)) == 5 and max(used) < 8
    p = W.prefix_decode()
    tb = p.cache.block_tables
    assert torch.equal(tb[:, :8], tb[:1, :8].expand(64, 8))
    assert all(2049 <= c <= 2561 for c in p.cache.context_lens.tolist())
    private = tb[:, 8:][tb[:, 8:] >= 0].tolist()
    assert len(private) == len(set(private)) and not set(private) & set(tb[0, :8].tolist())
    f = W.make_prefill_case("f", [4096] * 8, [512] * 8, 16, 8, 128, 256, seed=1005, skip_prob=0.05)
    frac = float((f.slot_mapping == -1).float().mean())
    assert 0.03 < frac < 0.07
    assert f.cu_seqlens_q.tolist() == list(range(0, 4097, 512))
