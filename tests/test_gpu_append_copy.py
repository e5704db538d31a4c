"""GPU: kv_append and kv_copy_blocks through the C ABI, bit-exact against the oracle's
array-copy model (and, for FP8, the oracle's E4M3 quantiser)."""

import numpy as np
import pytest
import torch

from oracle import cache as OC
from oracle import fp8 as OF
from paged_kv_cache_169_gb300 import abi
from paged_kv_cache_169_gb300.cache import PagedKVCache

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> np.ndarray:
    a = t.cpu().numpy()
    return a.view({4: np.uint32, 2: np.uint16, 1: np.uint8}[a.itemsize])


@pytest.mark.parametrize("dtype,B,H,d", [("f32", 16, 2, 64), ("f16", 16, 32, 128), ("f16", 8, 3, 64),
                                         ("f32", 32, 4, 128), ("f16", 32, 40, 128)])
def test_append_bit_exact(dtype, B, H, d):
    rng = np.random.default_rng(21)
    nb = 23
    cache = PagedKVCache(1, nb, B, H, d, dtype)
    npdt = np.float32 if dtype == "f32" else np.float16
    kp = np.full((nb, H, B, d), np.nan, dtype=npdt)
    vp = np.full((nb, H, B, d), np.nan, dtype=npdt)
    cache.k[0].copy_(torch.from_numpy(kp))
    cache.v[0].copy_(torch.from_numpy(vp))
    n = 150
    slots = rng.permutation(nb * B)[:n].astype(np.int64)
    slots[::7] = -1                                   # padding tokens are skipped
    k = rng.standard_normal((n, H, d)).astype(npdt)
    v = rng.standard_normal((n, H, d)).astype(npdt)
    cache.append(0, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                 torch.from_numpy(slots).cuda())
    OC.append(kp, vp, k, v, slots, B)
    assert np.array_equal(_bits(cache.k[0]), kp.view(_bits(cache.k[0]).dtype))
    assert np.array_equal(_bits(cache.v[0]), vp.view(_bits(cache.v[0]).dtype))
    assert cache.device_error() == 0
    cache.close()


@pytest.mark.parametrize("in_dtype,B,d", [("f16", 16, 128), ("f32", 8, 64), ("f16", 32, 64)])
def test_fp8_append_bit_exact(in_dtype, B, d):
    rng = np.random.default_rng(22)
    nb, H = 13, 5
    cache = PagedKVCache(1, nb, B, H, d, "fp8")
    cache.k[0].fill_(0)
    cache.v[0].fill_(0)
    ks = rng.uniform(0.002, 0.05, nb).astype(np.float32)
    vs = rng.uniform(0.002, 0.05, nb).astype(np.float32)
    ks[3] = 1.0
    vs[4] = 2.0 ** -12                                 # forces saturation at +-448
    cache.k_scale[0][:nb].copy_(torch.from_numpy(ks))
    cache.v_scale[0][:nb].copy_(torch.from_numpy(vs))
    npdt = np.float16 if in_dtype == "f16" else np.float32
    n = 60
    slots = rng.permutation(nb * B)[:n].astype(np.int64)
    k = (rng.standard_normal((n, H, d)) * 3).astype(npdt)
    v = (rng.standard_normal((n, H, d)) * 3).astype(npdt)
    k[0, 0, :4] = [0.0, -0.0, 1e-7, -1e-7]             # zero signs and underflow to zero
    cache.append(0, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), torch.from_numpy(slots).cuda())
    kc = np.zeros((nb, H, B, d), dtype=np.uint8)
    vc = np.zeros((nb, H, B, d), dtype=np.uint8)
    OC.append_fp8(kc, vc, k, v, slots, B, ks, vs, OF.quantize)
    assert np.array_equal(cache.k[0].cpu().numpy(), kc)
    assert np.array_equal(cache.v[0].cpu().numpy(), vc)
    cache.close()


def test_append_out_of_range_slot_sets_error_and_skips():
    cache = PagedKVCache(1, 4, 16, 2, 64, "f16")
    cache.k[0].fill_(0)
    cache.v[0].fill_(0)
    k = torch.ones((2, 2, 64), dtype=torch.float16, device="cuda")
    slots = torch.tensor([4 * 16, 5], dtype=torch.int64, device="cuda")
    cache.append(0, k, k, slots)
    assert cache.device_error() == abi.KV_DEVERR_SLOT
    assert cache.device_error() == 0                   # cleared
    assert float(cache.k[0][0, :, 5].float().sum()) == 2 * 64   # the valid token landed
    assert float(cache.k[0].float().sum()) == 2 * 64
    cache.close()


@pytest.mark.parametrize("dtype", ["f16", "fp8", "f32"])
def test_copy_blocks_bit_exact_all_layers(dtype):
    rng = np.random.default_rng(23)
    L, nb, B, H, d = 3, 20, 16, 4, 128
    cache = PagedKVCache(L, nb, B, H, d, dtype)
    host = []
    for t in cache.k + cache.v:
        if t.dtype == torch.uint8:
            a = rng.integers(0, 256, t.shape, dtype=np.uint8)
        else:
            a = rng.standard_normal(t.shape).astype(np.float16 if t.dtype == torch.float16 else np.float32)
            a[:, :, 5:] = np.nan                        # unused slots are copied too
        t.copy_(torch.from_numpy(a))
        host.append(a)
    scales = []
    if dtype == "fp8":
        for t in cache.k_scale + cache.v_scale:
            a = rng.uniform(0.01, 1.0, t.shape).astype(np.float32)
            t.copy_(torch.from_numpy(a))
            scales.append(a)
    pairs = np.array([[2, 11], [7, 3], [0, 19], [2, 12]], dtype=np.int32)
    cache.copy_blocks(torch.from_numpy(pairs).cuda(), 1, 3)          # layers 1..2 only
    for l in range(L):
        arrays = [host[l], host[L + l]]
        sc = [scales[l], scales[L + l]] if scales else []
        if l >= 1:
            OC.copy_blocks(arrays, pairs, sc)
        for t, a in zip([cache.k[l], cache.v[l]], arrays):
            assert np.array_equal(_bits(t), a.view(_bits(t).dtype))
        if scales:
            for t, a in zip([cache.k_scale[l], cache.v_scale[l]], sc):
                assert np.array_equal(t.cpu().numpy().view(np.uint32), a.view(np.uint32))
    assert cache.device_error() == 0
    bad = torch.tensor([[1, 2], [0, nb]], dtype=torch.int32, device="cuda")
    cache.copy_blocks(bad)
    assert cache.device_error() == abi.KV_DEVERR_BLOCK_ID
    cache.close()
