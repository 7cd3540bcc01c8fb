"""WeightCache's host-side bookkeeping on the CPU, with the quantize call
replaced by a recorder: one quantization per weight version, keyed on the
step counter when there is one, else on the tensor's in-place version; the
previous buffers handed to the re-quantization."""
import torch

from tensor_quantization_gb300 import weight_cache as wc


class Recorder:
    def __init__(self):
        self.calls = []

    def __call__(self, w, **kw):
        self.calls.append((w.data_ptr(), kw))
        return ("q", len(self.calls))


def test_one_quantization_per_step(monkeypatch):
    rec = Recorder()
    monkeypatch.setattr(wc.nvfp4, "quantize", rec)
    cache = wc.WeightCache(block2d=True)
    w = torch.zeros(32, 64)
    q0 = cache.get(w, step=0)
    assert cache.get(w, step=0) is q0 and cache.get(w, step=0) is q0  # micro-batches of one step
    assert len(rec.calls) == 1 and cache.quantizations == 1
    kw = rec.calls[0][1]
    assert kw["rowwise"] and kw["colwise"] and kw["block2d"] and kw["mode"] == "rne" and kw["out"] is None
    q1 = cache.get(w, step=1)
    assert q1 != q0 and len(rec.calls) == 2
    assert rec.calls[1][1]["out"] == q0  # the old buffers are reused


def test_mark_step_and_in_place_versions(monkeypatch):
    rec = Recorder()
    monkeypatch.setattr(wc.nvfp4, "quantize", rec)
    cache = wc.WeightCache()
    w = torch.zeros(16, 32)
    cache.get(w)
    cache.get(w)
    assert len(rec.calls) == 1
    w.add_(1.0)  # an optimizer update bumps the in-place version
    cache.get(w)
    assert len(rec.calls) == 2
    cache.mark_step()  # from now on the step counter is the key
    cache.get(w)
    cache.get(w)
    assert len(rec.calls) == 3
    w.add_(1.0)  # ignored while a step counter is in use
    cache.get(w)
    assert len(rec.calls) == 3
    cache.mark_step()
    cache.get(w)
    assert len(rec.calls) == 4


def test_weights_are_keyed_apart_and_dropped(monkeypatch):
    rec = Recorder()
    monkeypatch.setattr(wc.nvfp4, "quantize", rec)
    cache = wc.WeightCache()
    a, b = torch.zeros(16, 32), torch.zeros(16, 32)
    cache.get(a, step=0)
    cache.get(b, step=0)
    cache.get(a, step=0)
    assert len(cache) == 2 and len(rec.calls) == 2
    cache.drop(a)
    assert len(cache) == 1
    cache.get(a, step=0)
    assert len(rec.calls) == 3 and rec.calls[-1][1]["out"] is None  # a fresh entry


def test_a_new_tensor_at_a_freed_weights_address_is_a_miss(monkeypatch):
    rec = Recorder()
    monkeypatch.setattr(wc.nvfp4, "quantize", rec)
    cache = wc.WeightCache()
    base = torch.zeros(16 * 32)
    w1 = base.view(16, 32)
    cache.get(w1, step=0)
    # another tensor object with the same address, shape and dtype (what the
    # caching allocator produces when it hands a freed weight's block to a new
    # tensor): never the old codes
    w2 = base.view(16, 32)
    assert w2.data_ptr() == w1.data_ptr() and w2 is not w1
    cache.get(w2, step=0)
    assert len(rec.calls) == 2
    assert rec.calls[1][1]["out"] is None  # w1 is alive: its buffers are not rewritten
    cache.get(w2, step=0)
    assert len(rec.calls) == 2  # w2's own entry now hits


def test_entries_die_with_their_weight(monkeypatch):
    import gc
    rec = Recorder()
    monkeypatch.setattr(wc.nvfp4, "quantize", rec)
    cache = wc.WeightCache()
    w = torch.zeros(16, 32)
    cache.get(w, step=0)
    assert len(cache) == 1
    del w
    gc.collect()
    assert len(cache) == 0


def test_stochastic_rounding_draws_a_new_stream_per_quantization(monkeypatch):
    rec = Recorder()
    monkeypatch.setattr(wc.nvfp4, "quantize", rec)
    cache = wc.WeightCache(mode="sr", seed=7)
    a, b = torch.zeros(16, 32), torch.zeros(16, 64)
    cache.get(a, step=0)
    cache.get(b, step=0)
    cache.get(a, step=1)
    cache.get(a, step=2)
    cache.get(b, step=2)
    streams = [(kw["seed"], kw["offset"]) for _, kw in rec.calls]
    assert all(kw["mode"] == "sr" for _, kw in rec.calls)
    assert len(set(streams)) == len(streams) == 5
    assert all(s == 7 for s, _ in streams)
    # offset = weight number << 32 | that weight's quantization count
    assert [o for _, o in streams] == [0, 1 << 32, 1, 2, (1 << 32) | 1]
