"""WeightCache: one quantization per weight version, the same buffers reused."""
import numpy as np
import pytest
import torch

from tensor_quantization_gb300 import nvfp4
from tensor_quantization_gb300.weight_cache import WeightCache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_quantization_gb300 import build
    build.build()
    nvfp4.load()


def _codes(q):
    return q.codes_row.cpu().numpy(), q.codes_col.cpu().numpy(), q.scales_row.cpu().numpy()


def test_cache_quantizes_once_per_step_and_matches_a_fresh_quantize():
    g = torch.Generator().manual_seed(1)
    w = (torch.randn(256, 512, generator=g) * 0.02).to(torch.bfloat16).cuda()
    cache = WeightCache(block2d=True)
    q1 = cache.get(w, step=0)
    for _ in range(3):  # micro-batches of the same step
        assert cache.get(w, step=0) is q1
    assert cache.quantizations == 1
    fresh = nvfp4.quantize(w, mode="rne", colwise=True, block2d=True, swizzled=True)
    torch.cuda.synchronize()
    for a, b in zip(_codes(q1), _codes(fresh)):
        assert np.array_equal(a, b)
    # the optimizer steps: new values, new step number -> re-quantized into the same buffers
    with torch.no_grad():
        w.add_(torch.randn(256, 512, generator=g).to(torch.bfloat16).cuda() * 0.01)
    q2 = cache.get(w, step=1)
    assert cache.quantizations == 2 and q2.codes_row.data_ptr() == q1.codes_row.data_ptr()
    fresh = nvfp4.quantize(w, mode="rne", colwise=True, block2d=True, swizzled=True)
    torch.cuda.synchronize()
    for a, b in zip(_codes(q2), _codes(fresh)):
        assert np.array_equal(a, b)


def test_cache_without_step_follows_in_place_updates():
    w = torch.randn(128, 256, device="cuda").to(torch.bfloat16)
    cache = WeightCache(mode="sr", block2d=False, swizzled=False)
    q = cache.get(w)
    assert cache.get(w) is q and cache.quantizations == 1
    with torch.no_grad():
        w.mul_(2)  # bumps w._version
    cache.get(w)
    assert cache.quantizations == 2
    cache.drop(w)
    assert len(cache) == 0


def test_mark_step_invalidates_every_weight():
    ws = [torch.randn(64, 128, device="cuda").to(torch.bfloat16) for _ in range(3)]
    cache = WeightCache()
    cache.mark_step()
    qs = [cache.get(w) for w in ws]
    assert [cache.get(w) for w in ws] == qs and cache.quantizations == 3
    fresh = nvfp4.quantize(ws[1], mode="rne", colwise=True, swizzled=True)
    torch.cuda.synchronize()
    for a, b in zip(_codes(qs[1]), _codes(fresh)):
        assert np.array_equal(a, b)
    cache.mark_step()
    for w in ws:
        cache.get(w)
    assert cache.quantizations == 6
