"""WeightCache on the GPU: one quantization per weight version, the same
buffers reused, and every cached orientation equal to the CPU oracle's
quantization of that version ("nvfp4-sm120" README, section "Results":
quant(w) and quant(w^T) cached once per optimizer step)."""
import numpy as np
import pytest
import torch

import oracle
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


def _bits(w: torch.Tensor) -> np.ndarray:
    return w.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_matches_oracle(q, w, cache: WeightCache, offset: int = 0):
    """Both cached orientations against the oracle's quantize of w's current values."""
    torch.cuda.synchronize()
    xb = _bits(w)
    for colwise, codes, scales in ((False, q.codes_row, q.scales_row), (True, q.codes_col, q.scales_col)):
        o = oracle.quantize(xb, colwise=colwise, mode=cache.mode, block2d=cache.block2d,
                            swizzled=cache.swizzled, seed=cache.seed, offset=offset)
        assert np.array_equal(codes.cpu().numpy(), o["codes"]), f"codes (colwise={colwise})"
        assert np.array_equal(scales.cpu().numpy().ravel(), o["scales"].ravel()), f"scales (colwise={colwise})"
        assert q.global_scale.cpu().numpy()[:1].view(np.uint32)[0] == o["global_scale"].view(np.uint32)[0]


@pytest.mark.parametrize("block2d", [False, True])
def test_cached_orientations_equal_the_oracle_per_version(block2d):
    g = torch.Generator().manual_seed(1)
    w = (torch.randn(256, 512, generator=g) * 0.02).to(torch.bfloat16).cuda()
    cache = WeightCache(block2d=block2d)
    q1 = cache.get(w, step=0)
    for _ in range(3):  # micro-batches of the same step
        assert cache.get(w, step=0) is q1
    assert cache.quantizations == 1
    assert_matches_oracle(q1, w, cache)
    # the optimizer steps: new values, new step number -> re-quantized into the same buffers
    with torch.no_grad():
        w.add_(torch.randn(256, 512, generator=g).to(torch.bfloat16).cuda() * 0.01)
    q2 = cache.get(w, step=1)
    assert cache.quantizations == 2 and q2.codes_row.data_ptr() == q1.codes_row.data_ptr()
    assert_matches_oracle(q2, w, cache)


def test_stochastic_cache_uses_a_fresh_stream_per_version():
    g = torch.Generator().manual_seed(2)
    a = torch.randn(128, 256, generator=g).to(torch.bfloat16).cuda()
    b = torch.randn(128, 256, generator=g).to(torch.bfloat16).cuda()
    cache = WeightCache(mode="sr", swizzled=False, seed=11)
    qa = cache.get(a, step=0)
    assert_matches_oracle(qa, a, cache, offset=0)
    codes0 = qa.codes_row.clone()
    qb = cache.get(b, step=0)
    assert_matches_oracle(qb, b, cache, offset=1 << 32)  # the second weight's stream
    qa = cache.get(a, step=1)  # same values, next version: new random bytes
    assert_matches_oracle(qa, a, cache, offset=1)
    assert not torch.equal(qa.codes_row, codes0)


def test_cache_without_step_follows_in_place_updates():
    w = torch.randn(128, 256, device="cuda").to(torch.bfloat16)
    cache = WeightCache(mode="sr", block2d=False, swizzled=False)
    q = cache.get(w)
    assert cache.get(w) is q and cache.quantizations == 1
    with torch.no_grad():
        w.mul_(2)  # bumps w._version
    q = cache.get(w)
    assert cache.quantizations == 2
    assert_matches_oracle(q, w, cache, offset=1)
    cache.drop(w)
    assert len(cache) == 0


def test_mark_step_invalidates_every_weight():
    ws = [torch.randn(64, 128, device="cuda").to(torch.bfloat16) for _ in range(3)]
    cache = WeightCache()
    cache.mark_step()
    qs = [cache.get(w) for w in ws]
    assert [cache.get(w) for w in ws] == qs and cache.quantizations == 3
    assert_matches_oracle(qs[1], ws[1], cache)
    cache.mark_step()
    for w in ws:
        cache.get(w)
    assert cache.quantizations == 6
