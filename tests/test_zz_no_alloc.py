"""pkv_decode_attention_noalloc: decode with its split-K scratch in the
library's static device array instead of a cudaMalloc'ed workspace.

Some callers cannot let a library allocate device memory: an engine that gave
nearly all free memory to its KV block pool at start-up, or a process whose
device memory must all come from one caching allocator.  This entry point
serves them.  Its results must match the fp64 oracle on the same inputs, call
after call, although every call reuses (and leaves behind) the same scratch
array; it must allocate nothing; and its device-side check failures must reach
pkv_get_device_error like those of every other call.

This file is collected last on purpose: it is run alone in a fresh process
as well as after every other test.
"""
import pytest
import torch

import paged_kv_cache_493_b300 as pkv
from paged_kv_cache_493_b300 import workloads as W
from helpers import assert_close, cache_to_device, dev, oracle_decode_after_store

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def clean_state(cuda_device):
    pkv.pkv_set_max_splits(0)
    pkv.pkv_set_wait_limit_ns(1_000_000_000)
    pkv.pkv_get_device_error()
    yield
    pkv.pkv_get_device_error()


def _stored_case(case):
    """Device copies of a decode case with this step's K/V rows stored."""
    kc, vc, bt, cl = cache_to_device(case.cache)
    pkv.pkv_store_kvcache(dev(case.k_new), dev(case.v_new), dev(case.slot_mapping), kc, vc)
    return dev(case.q), kc, vc, bt, cl


def test_noalloc_matches_oracle_on_two_calls_in_a_row(cuda_device):
    # First call: a few long contexts (each cut into many pieces); second
    # call: the 128-sequence batch (another grid cut and partial layout), so
    # the second call runs over what the first left in the scratch.
    cases = [W.make_decode_case("na", [1, 300, 1500, 4000, 9000], 16, 8, 128, 64, seed=404,
                                k_scale=3.0),
             W.qwen_decode()]
    outs = []
    for case in cases:
        q, kc, vc, bt, cl = _stored_case(case)
        out = torch.full_like(q, float("nan"))
        pkv.pkv_decode_attention_noalloc(q, kc, vc, bt, cl, case.scale, out)
        torch.cuda.synchronize()
        outs.append(out)
    for i, (case, out) in enumerate(zip(cases, outs)):
        assert_close(out, oracle_decode_after_store(case), f"call {i + 1} ({case.num_seqs} seqs)")
    assert pkv.pkv_get_device_error()[0] == 0


def test_noalloc_allocates_no_device_memory(cuda_device):
    """After one call (which loads the library's device image and looks up the
    array), further calls leave the device's free memory unchanged."""
    case = W.make_decode_case("nm", [700, 2000, 33], 16, 8, 128, 32, seed=405)
    q, kc, vc, bt, cl = _stored_case(case)
    out = torch.empty_like(q)
    pkv.pkv_decode_attention_noalloc(q, kc, vc, bt, cl, case.scale, out)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        pkv.pkv_decode_attention_noalloc(q, kc, vc, bt, cl, case.scale, out)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert_close(out, oracle_decode_after_store(case), "after repeated calls")


def test_noalloc_reports_a_bad_block_id(cuda_device):
    """An out-of-range block id is skipped (zero output for its sequence) and
    pkv_get_device_error returns PKV_ERR_DEVICE_CHECK; the next good call is
    right again and clean."""
    case = W.make_decode_case("nb", [300, 600, 40], 16, 8, 128, 16, seed=406)
    good = oracle_decode_after_store(case)
    q, kc, vc, bt, cl = _stored_case(case)
    bad_bt = bt.clone()
    bad_bt[1, 1] = 16  # == num_blocks: out of range
    out = torch.full_like(q, 7.0)
    pkv.pkv_decode_attention_noalloc(q, kc, vc, bad_bt, cl, case.scale, out)
    code, _ = pkv.pkv_get_device_error()
    assert code == pkv.PKV_ERR_DEVICE_CHECK
    assert torch.all(out[1] == 0)
    assert_close(out[[0, 2]], good[[0, 2]], "unaffected sequences")
    pkv.pkv_decode_attention_noalloc(q, kc, vc, bt, cl, case.scale, out)
    assert pkv.pkv_get_device_error()[0] == 0
    assert_close(out, good, "the next call")


def test_noalloc_rejects_a_batch_beyond_its_scratch(cuda_device):
    """16400 sequences x 16 KV heads (head_dim 64, one query head per KV
    head): 262400 (sequence, KV head) pairs, each needing an 8-byte arrival
    counter, more than the array's 2 MiB counter region holds (262144).  The
    call must refuse with PKV_ERR_UNSUPPORTED and launch nothing."""
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
