"""pkv_decode_attention_noalloc: decode with its split-K scratch in the
library's static device array instead of a cudaMalloc'ed workspace.

Some callers cannot let a library allocate device memory: an engine that gave
nearly all free memory to its KV block pool at start-up, or code running while
a stream is captured into a CUDA graph.  This entry point serves them; its
results must agree with pkv_decode_attention's on the same inputs, call after
call, although every call reuses (and leaves behind) the same scratch array.

This file is collected last on purpose: it is run alone in a fresh process
as well as after every other test.
"""
import pytest
import torch

import paged_kv_cache_493_b300 as pkv
from paged_kv_cache_493_b300 import workloads as W
from helpers import MAX_ABS, MEAN_ABS, cache_to_device, dev

pytestmark = pytest.mark.gpu


def _stored_case(case):
    """Device copies of a decode case with this step's K/V rows stored."""
    kc, vc, bt, cl = cache_to_device(case.cache)
    pkv.pkv_store_kvcache(dev(case.k_new), dev(case.v_new), dev(case.slot_mapping), kc, vc)
    return dev(case.q), kc, vc, bt, cl


def _within_tolerance(got, ref, what):
    assert torch.isfinite(got.float()).all(), what
    err = (got.double() - ref.double()).abs()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, (
        f"{what}: max abs {err.max().item():.3e}, mean abs {err.mean().item():.3e}")


def test_noalloc_matches_decode_on_two_calls_in_a_row(cuda_device):
    pkv.pkv_set_max_splits(0)
    pkv.pkv_set_wait_limit_ns(1_000_000_000)
    # First call: a few long contexts (each cut into many pieces); second
    # call: the 128-sequence batch (another grid cut and partial layout), so
    # the second call runs over what the first left in the scratch.
    cases = [W.make_decode_case("na", [1, 300, 1500, 4000, 9000], 16, 8, 128, 64, seed=404,
                                k_scale=3.0),
             W.qwen_decode()]
    results = []
    for case in cases:
        q, kc, vc, bt, cl = _stored_case(case)
        out_na = torch.full_like(q, float("nan"))
        pkv.pkv_decode_attention_noalloc(q, kc, vc, bt, cl, case.scale, out_na)
        out_ref = torch.empty_like(q)
        pkv.pkv_decode_attention(q, kc, vc, bt, cl, case.scale, out_ref)
        torch.cuda.synchronize()
        results.append((out_na, out_ref, case.num_seqs))
    for i, (out_na, out_ref, b) in enumerate(results):
        _within_tolerance(out_na, out_ref, f"call {i + 1} ({b} sequences)")
    assert pkv.pkv_get_device_error()[0] == 0


def test_noalloc_rejects_a_batch_beyond_its_scratch(cuda_device):
    """16400 sequences x 16 KV heads (head_dim 64, one query head per KV
    head): 262400 (sequence, KV head) pairs, each needing an 8-byte arrival
    counter, more than the array's 2 MiB counter region holds (262144).  The
    call must refuse with PKV_ERR_UNSUPPORTED and launch nothing."""
    pkv.pkv_set_max_splits(0)
    b, hq, hkv, d, mb = 16400, 16, 16, 64, 1
    kc = torch.zeros(1, 256, hkv, d, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    q = torch.zeros(b, hq, d, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(b, mb, dtype=torch.int32, device="cuda")
    cl = torch.ones(b, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 3.0)
    with pytest.raises(pkv.PkvError) as exc:
        pkv.pkv_decode_attention_noalloc(q, kc, vc, bt, cl, 1.0 / d ** 0.5, out)
    assert exc.value.status == pkv.PKV_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)  # nothing ran
