"""Shared helpers of the GPU tests: device copies of seeded cases, running the
CUDA path through the binding, and the tolerance check against the oracle."""
import numpy as np
import torch

import oracle
import oracle.parallel as oracle_parallel
import paged_kv_cache_493_b300 as pkv

# bf16-in / fp32-accumulate attention against the fp64 oracle.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def dev(t):
    return t.to("cuda", non_blocking=False)


def cache_to_device(cache):
    return (dev(cache.k_cache), dev(cache.v_cache), dev(cache.block_tables),
            dev(cache.context_lens))


def assert_close(gpu_out, ref, what=""):
    got = gpu_out.detach().to("cpu", torch.float64).numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max abs {mx:.3e}, mean abs {mean:.3e}"
    return mx, mean


def run_decode_step(case, stream=None):
    """store_kvcache of the new rows, then decode; returns (out, k_cache, v_cache) on device."""
    kc, vc, bt, cl = cache_to_device(case.cache)
    pkv.pkv_store_kvcache(dev(case.k_new), dev(case.v_new), dev(case.slot_mapping), kc, vc, stream)
    q = dev(case.q)
    out = torch.empty_like(q)
    pkv.pkv_decode_attention(q, kc, vc, bt, cl, case.scale, out, stream)
    torch.cuda.synchronize()
    return out, kc, vc


def run_prefill_step(case, stream=None):
    kc, vc, bt, cl = cache_to_device(case.cache)
    pkv.pkv_store_kvcache(dev(case.k_new), dev(case.v_new), dev(case.slot_mapping), kc, vc, stream)
    q = dev(case.q)
    out = torch.empty_like(q)
    pkv.pkv_prefill_attention(q, kc, vc, bt, dev(case.cu_seqlens_q), cl, case.scale, out, stream)
    torch.cuda.synchronize()
    return out, kc, vc


def oracle_decode_after_store(case, rows=None):
    """The oracle's store, then its decode: the full output on every host core
    (oracle.parallel, bit-identical to the single-threaded call), or the
    listed (sequence, head) rows."""
    c = case.cache
    kc, vc = oracle.store_kvcache(case.k_new, case.v_new, case.slot_mapping, c.k_cache, c.v_cache)
    if rows is None:
        return oracle_parallel.decode(case.q, kc, vc, c.block_tables, c.context_lens, case.scale)
    return oracle.decode(case.q, kc, vc, c.block_tables, c.context_lens, case.scale, rows=rows)


def oracle_prefill_after_store(case, rows=None):
    c = case.cache
    kc, vc = oracle.store_kvcache(case.k_new, case.v_new, case.slot_mapping, c.k_cache, c.v_cache)
    if rows is None:
        return oracle_parallel.prefill(case.q, kc, vc, c.block_tables, case.cu_seqlens_q,
                                       c.context_lens, case.scale)
    return oracle.prefill(case.q, kc, vc, c.block_tables, case.cu_seqlens_q, c.context_lens,
                          case.scale, rows=rows)


def no_device_error():
    code, site = pkv.pkv_get_device_error()
    assert code == 0, f"device error {pkv.STATUS.get(code, code)} at site {site}"
