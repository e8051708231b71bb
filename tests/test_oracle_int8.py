"""Pins of the oracle's INT8 KV cache (quantise, store, gather, decode).

Against what the reading of the pages and the mathematics fix: hand-worked
codes and scales (tests/golden/int8_examples.json), the round-to-nearest
error bound |code * scale - x| <= scale / 2, the largest magnitude mapping to
+-127, and the special case in which quantisation is exact (integer rows
whose largest magnitude is 127: scale 1), where the INT8 decode must equal
the bf16 decode of the same values bit for bit.  Planted mistakes in a copy
of the oracle's C source must each fail one of these pins.
"""
import json
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_493_b300 import workloads as W

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "int8_examples.json")))


def nearest_binary32(fr: Fraction) -> np.float32:
    """The binary32 value nearest to a rational (ties to even), by exact search."""
    f = np.float32(float(fr))
    for cand in (np.nextafter(f, np.float32(-np.inf)), np.nextafter(f, np.float32(np.inf))):
        if abs(Fraction(float(cand)) - fr) < abs(Fraction(float(f)) - fr):
            f = cand
    return f


def test_golden_quantised_rows():
    for row in GOLDEN["rows"]:
        x = torch.tensor([row["x"]], dtype=torch.bfloat16)
        codes, scales = oracle.quantize_rows(x)
        assert codes[0].tolist() == row["codes"], row["derivation"]
        want = nearest_binary32(Fraction(row["scale_num"], row["scale_den"]))
        assert scales[0] == want, (float(scales[0]), float(want))


def random_rows(n, d, seed, spread=3.0):
    g = torch.Generator().manual_seed(seed)
    mag = torch.exp(torch.randn(n, 1, generator=g) * spread)  # rows over many magnitudes
    return (torch.randn(n, d, generator=g) * mag).to(torch.bfloat16)


@pytest.mark.parametrize("d", [64, 128])
def test_round_to_nearest_bound_and_range(d):
    x = random_rows(300, d, seed=d)
    codes, scales = oracle.quantize_rows(x)
    xf = x.float().numpy().astype(np.float64)
    s = scales.astype(np.float64)[:, None]
    assert codes.min() >= -127 and codes.max() <= 127
    # The code of x is nearest(x / s) with x / s rounded once in binary32:
    # |x / s - code| <= 1/2 + 127 * 2^-24.
    assert np.all(np.abs(codes * s - xf) <= s * (0.5 + 127 * 2.0 ** -24))
    amax = np.abs(xf).max(axis=1)
    i = np.abs(xf).argmax(axis=1)
    assert np.all(np.abs(codes[np.arange(len(i)), i]) == 127)
    assert np.all(np.sign(codes) * np.sign(xf) >= 0)  # no sign flips
    np.testing.assert_allclose(s[:, 0], amax / 127, rtol=2.0 ** -23)


def int8_cache_of(case):
    """Quantise a case's bf16 pools row by row (the INT8 cache holding the same
    tokens, codes [NB, Hkv, 256, D], scales [NB, Hkv, 256])."""
    c = case.cache
    kc, ks = oracle.quantize_pool(c.k_cache)
    vc, vs = oracle.quantize_pool(c.v_cache)
    return kc, vc, ks, vs


def test_gather_recovers_rows_within_half_a_step():
    case = W.make_decode_case("g8", [300, 40], 4, 2, 64, 4, seed=5)
    kc, vc, ks, vs = int8_cache_of(case)
    c = case.cache
    for s in range(2):
        ctx = int(c.context_lens[s])
        K, V = oracle.gather_int8(kc, vc, ks, vs, c.block_tables[s], ctx)
        Kb, Vb = oracle.gather(c.k_cache, c.v_cache, c.block_tables[s], ctx)
        for got, ref, sc in ((K, Kb, ks), (V, Vb, vs)):
            step = np.zeros(got.shape[:2])
            for t in range(ctx):
                blk = int(c.block_tables[s, t // 256])
                step[t] = sc[blk, :, t % 256].numpy()
            assert np.all(np.abs(got - ref) <= step[:, :, None] * (0.5 + 127 * 2.0 ** -24))


def integer_case(seed):
    """A decode case whose K/V rows are integers in [-127, 127] with one
    +-127 per row: every scale is 1 and quantisation is exact."""
    case = W.make_decode_case("exact", [1, 37, 256, 300], 4, 2, 64, 8, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    for t in (case.cache.k_cache, case.cache.v_cache):
        ints = torch.randint(-126, 127, t.shape, generator=g).float()
        ints[..., 0] = torch.where(torch.rand(t.shape[:-1], generator=g) < 0.5, 127.0, -127.0)
        t.copy_(ints.to(torch.bfloat16))
    case.q.copy_((case.q.float() / 64).to(torch.bfloat16))  # keep softmax away from one-hot
    return case


def test_int8_decode_is_bf16_decode_when_quantisation_is_exact():
    case = integer_case(7)
    kc, vc, ks, vs = int8_cache_of(case)
    assert torch.all(ks == 1) and torch.all(vs == 1)
    c = case.cache
    want = oracle.decode(case.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, case.scale)
    got = oracle.decode_int8(case.q, kc, vc, ks, vs, c.block_tables, c.context_lens, case.scale)
    assert np.array_equal(got, want)


def integer_prefill_case(seed):
    """A chunked-prefill case with the same integer K/V rows (every scale 1)."""
    case = W.make_prefill_case("exact_p", [0, 37, 250, 300], [5, 30, 9, 40], 4, 2, 64, 8,
                               seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    for t in (case.cache.k_cache, case.cache.v_cache):
        ints = torch.randint(-126, 127, t.shape, generator=g).float()
        ints[..., 0] = torch.where(torch.rand(t.shape[:-1], generator=g) < 0.5, 127.0, -127.0)
        t.copy_(ints.to(torch.bfloat16))
    case.q.copy_((case.q.float() / 64).to(torch.bfloat16))
    return case


def test_int8_prefill_is_bf16_prefill_when_quantisation_is_exact():
    case = integer_prefill_case(9)
    kc, vc, ks, vs = int8_cache_of(case)
    assert torch.all(ks == 1) and torch.all(vs == 1)
    c = case.cache
    want = oracle.prefill(case.q, c.k_cache, c.v_cache, c.block_tables, case.cu_seqlens_q,
                          c.context_lens, case.scale)
    got = oracle.prefill_int8(case.q, kc, vc, ks, vs, c.block_tables, case.cu_seqlens_q,
                              c.context_lens, case.scale)
    assert np.array_equal(got, want)


def test_int8_prefill_last_row_is_int8_decode():
    """The last query of a chunk sees the whole context, as a decode query
    does: on general (scaled) rows the two give the same numbers."""
    case = W.make_prefill_case("last", [0, 37, 250, 300], [5, 30, 9, 40], 4, 2, 64, 8, seed=10)
    kc, vc, ks, vs = int8_cache_of(case)
    assert not torch.all(ks == 1)
    c = case.cache
    cu = case.cu_seqlens_q.tolist()
    got = oracle.prefill_int8(case.q, kc, vc, ks, vs, c.block_tables, case.cu_seqlens_q,
                              c.context_lens, case.scale)
    last = torch.stack([case.q[cu[s + 1] - 1] for s in range(len(cu) - 1)])
    dec = oracle.decode_int8(last, kc, vc, ks, vs, c.block_tables, c.context_lens, case.scale)
    for s in range(len(cu) - 1):
        assert np.array_equal(got[cu[s + 1] - 1], dec[s]), s


def test_int8_decode_stays_close_to_bf16_decode():
    """Quantisation noise (relative 1/254 per element at worst) moves the
    attention output little: a sanity bound, not a tolerance of the kernels."""
    case = W.make_decode_case("noise", [1, 37, 256, 300], 4, 2, 64, 8, seed=8)
    kc, vc, ks, vs = int8_cache_of(case)
    c = case.cache
    want = oracle.decode(case.q, c.k_cache, c.v_cache, c.block_tables, c.context_lens, case.scale)
    got = oracle.decode_int8(case.q, kc, vc, ks, vs, c.block_tables, c.context_lens, case.scale)
    assert np.abs(got - want).max() < 0.05


def test_store_int8_writes_quantised_rows_and_skips_minus_one():
    nb, hkv, d = 2, 2, 64
    g = torch.Generator().manual_seed(3)
    k = torch.randn(3, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(3, hkv, d, generator=g).to(torch.bfloat16)
    kc = torch.full((nb, hkv, 256, d), 5, dtype=torch.int8)  # head-major blocks
    vc = kc.clone()
    ks = torch.full((nb, hkv, 256), 9.0)
    vs = ks.clone()
    nkc, nvc, nks, nvs = oracle.store_kvcache_int8(k, v, [5, -1, 258], kc, vc, ks, vs)
    qk, sk = oracle.quantize_rows(k)
    qv, sv = oracle.quantize_rows(v)
    for i, slot in ((0, 5), (2, 258)):
        b, o = divmod(slot, 256)
        assert np.array_equal(nkc[b, :, o].numpy(), qk[i]) and np.array_equal(nvc[b, :, o].numpy(), qv[i])
        assert np.array_equal(nks[b, :, o].numpy(), sk[i]) and np.array_equal(nvs[b, :, o].numpy(), sv[i])
    untouched = torch.ones(nb, hkv, 256, dtype=torch.bool)
    untouched[0, :, 5] = untouched[1, :, 2] = False
    assert torch.all(nkc[untouched] == 5) and torch.all(nks[untouched] == 9.0)
    with pytest.raises(oracle.OracleError):
        oracle.store_kvcache_int8(k, v, [5, -2, 258], kc, vc, ks, vs)
    with pytest.raises(oracle.OracleError):
        oracle.store_kvcache_int8(k, v, [5, 512, 0], kc, vc, ks, vs)


SRC = open(os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.c")).read()

MUTANTS = {
    "round_half_away_from_zero": ("c = lrintf((float)widen_bf16(x[d]) / s);",
                                  "c = (long)roundf((float)widen_bf16(x[d]) / s);"),
    "truncate_toward_zero": ("c = lrintf((float)widen_bf16(x[d]) / s);",
                             "c = (long)((float)widen_bf16(x[d]) / s);"),
    "divide_by_128": ("const float s = amax / 127.0f;", "const float s = amax / 128.0f;"),
    "max_without_abs": ("const float a = fabsf((float)widen_bf16(x[d]));",
                        "const float a = (float)widen_bf16(x[d]);"),
    "dequantise_by_division": ("K[(int64_t)t * row + (int64_t)h * head_dim + d] = (double)k_codes[r * head_dim + d] * ks;",
                               "K[(int64_t)t * row + (int64_t)h * head_dim + d] = (double)k_codes[r * head_dim + d] / (ks > 0 ? ks : 1);"),
    "v_uses_k_scale": ("const double ks = (double)k_scales[r], vs = (double)v_scales[r];",
                       "const double ks = (double)k_scales[r], vs = (double)k_scales[r];"),
    "store_v_codes_from_k": ("oracle_quantize_row(v + i * v_row_stride + (int64_t)h * head_dim, head_dim,",
                             "oracle_quantize_row(k + i * k_row_stride + (int64_t)h * head_dim, head_dim,"),
    "store_head_offset_dropped": ("oracle_quantize_row(k + i * k_row_stride + (int64_t)h * head_dim, head_dim,",
                                  "oracle_quantize_row(k + i * k_row_stride, head_dim,"),
    "prefill_int8_scales_swapped": (
        "const CacheSource c = {NULL, NULL, k_codes, v_codes, k_scales, v_scales};\n  return prefill_from(",
        "const CacheSource c = {NULL, NULL, k_codes, v_codes, v_scales, k_scales};\n  return prefill_from("),
    "prefill_int8_codes_swapped": (
        "const CacheSource c = {NULL, NULL, k_codes, v_codes, k_scales, v_scales};\n  return prefill_from(",
        "const CacheSource c = {NULL, NULL, v_codes, k_codes, k_scales, v_scales};\n  return prefill_from("),
    "slot_major_rows": ("return ((slot / ORACLE_BLOCK) * num_kv_heads + h) * ORACLE_BLOCK + slot % ORACLE_BLOCK;",
                        "return slot * num_kv_heads + h;"),
}

PINS = [
    test_golden_quantised_rows,
    lambda: test_round_to_nearest_bound_and_range(64),
    test_gather_recovers_rows_within_half_a_step,
    test_int8_decode_is_bf16_decode_when_quantisation_is_exact,
    test_store_int8_writes_quantised_rows_and_skips_minus_one,
    test_int8_prefill_is_bf16_prefill_when_quantisation_is_exact,
    test_int8_prefill_last_row_is_int8_decode,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_int8_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation site for {name} not found once"
    src = tmp_path / "mutant.c"
    src.write_text(SRC.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                           "-ffp-contract=off", str(src), "-o", str(so), "-lm"])
    saved, real_build = oracle._lib, oracle.build
    try:
        oracle._lib = None
        oracle.build = lambda force=False: str(so)
        oracle.lib()
        caught = None
        for pin in PINS:
            try:
                pin()
            except (Exception, pytest.fail.Exception):
                caught = pin
                break
        assert caught is not None, f"no pin caught mutant {name}"
    finally:
        oracle.build = real_build
        oracle._lib = saved
