"""store_kvcache on the GPU against the oracle: bit-exact over the whole pool."""
import pytest
import torch

import oracle
import paged_kv_cache_493_b300 as pkv
from paged_kv_cache_493_b300 import workloads as W
from helpers import dev, no_device_error

pytestmark = pytest.mark.gpu


def _store_and_compare(k, v, slots, k_cache, v_cache):
    kc, vc = dev(k_cache), dev(v_cache)
    pkv.pkv_store_kvcache(dev(k), dev(v), dev(slots), kc, vc)
    torch.cuda.synchronize()
    rk, rv = oracle.store_kvcache(k, v, slots, k_cache, v_cache)
    assert torch.equal(kc.cpu().view(torch.int16), rk.view(torch.int16))
    assert torch.equal(vc.cpu().view(torch.int16), rv.view(torch.int16))
    no_device_error()


@pytest.mark.parametrize("make", [W.tiny_decode, W.qwen_decode, W.prefix_decode])
def test_store_decode_workloads_bit_exact(cuda_device, make):
    c = make()
    _store_and_compare(c.k_new, c.v_new, c.slot_mapping, c.cache.k_cache, c.cache.v_cache)


def test_store_chunked_prefill_bit_exact(cuda_device):
    c = W.chunked_prefill()
    assert int((c.slot_mapping == -1).sum()) > 0
    _store_and_compare(c.k_new, c.v_new, c.slot_mapping, c.cache.k_cache, c.cache.v_cache)


@pytest.mark.parametrize("n,hkv,d", [(0, 8, 128), (1, 1, 64), (7, 2, 64), (333, 8, 128), (1000, 4, 64)])
def test_store_ragged_sizes(cuda_device, n, hkv, d):
    g = torch.Generator().manual_seed(n + hkv + d)
    nb = 16
    kc = W.randn_bf16((nb, 256, hkv, d), g)
    vc = W.randn_bf16((nb, 256, hkv, d), g)
    k = W.randn_bf16((n, hkv, d), g)
    v = W.randn_bf16((n, hkv, d), g)
    slots = torch.randperm(nb * 256, generator=g)[:n].to(torch.int32)
    if n > 2:
        slots[::3] = -1
    _store_and_compare(k, v, slots, kc, vc)


def test_store_strided_rows(cuda_device):
    """k and v as views into a fused qkv projection (row stride > Hkv * D)."""
    g = torch.Generator().manual_seed(3)
    n, hq, hkv, d, nb = 50, 16, 8, 128, 8
    qkv = W.randn_bf16((n, hq + 2 * hkv, d), g)
    k, v = qkv[:, hq:hq + hkv], qkv[:, hq + hkv:]
    kc = W.randn_bf16((nb, 256, hkv, d), g)
    vc = W.randn_bf16((nb, 256, hkv, d), g)
    slots = torch.randperm(nb * 256, generator=g)[:n].to(torch.int32)
    dq = dev(qkv)
    kcd, vcd = dev(kc), dev(vc)
    pkv.pkv_store_kvcache(dq[:, hq:hq + hkv], dq[:, hq + hkv:], dev(slots), kcd, vcd)
    torch.cuda.synchronize()
    rk, rv = oracle.store_kvcache(k.contiguous(), v.contiguous(), slots, kc, vc)
    assert torch.equal(kcd.cpu().view(torch.int16), rk.view(torch.int16))
    assert torch.equal(vcd.cpu().view(torch.int16), rv.view(torch.int16))
