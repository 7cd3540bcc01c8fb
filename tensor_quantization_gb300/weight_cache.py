"""Quantized weights reused until the weight changes.

A weight is read by several GEMMs per optimizer step (forward, and the
transposed orientation for the input gradient; every micro-batch of gradient
accumulation), but it changes only when the optimizer steps.  WeightCache
quantizes each weight once per change, into both orientations, and hands the
same device buffers back until then.  ("nvfp4-sm120" README, section
"Results": caching the weight's two round-to-nearest orientations once per
optimizer step, keyed on a counter bumped after the optimizer step, took a
micro-batched FFN step from 437 ms to 122 ms.)

An entry belongs to one tensor object: it is looked up by (storage address,
shape, dtype, device), holds a weak reference to the tensor it was made for,
and is dropped when that tensor is garbage collected.  A lookup whose entry
was made for another object (a tensor that now occupies a freed weight's
address, or a fresh ``.data`` alias) re-quantizes, so stale codes are never
returned; callers pass the same object every time (e.g. the
``nn.Parameter``).  The version is an optimizer-step counter (passed to
``get``, or bumped with ``mark_step`` after each optimizer step) when there is
one, else the tensor's in-place modification counter
(``torch.Tensor._version``), which every optimizer update also bumps.

With stochastic rounding every quantization draws its own Philox stream: the
cache's ``seed`` is the key, and the counter offset packs a per-weight number
(assigned on the weight's first lookup) in its high 32 bits and that weight's
quantization count in its low 32 bits, so neither successive versions of a
weight nor different weights reuse random bytes.  Host-side bookkeeping only:
every quantization runs through ``nvfp4.quantize``.
"""
from __future__ import annotations

import weakref
from dataclasses import dataclass, field

import torch

from . import nvfp4


@dataclass
class _Entry:
    ref: weakref.ref
    version: object
    q: nvfp4.Quantized
    weight_id: int
    count: int  # quantizations of this weight so far (the SR offset's low half)
    hits: int = 0


@dataclass
class WeightCache:
    """Per-weight NVFP4 copies in both orientations (defaults: 1x16 blocks with
    round-to-nearest and swizzled scales, so both orientations are
    deterministic; block2d=True gives 16x16 tiles; mode="sr" rounds
    stochastically with a fresh Philox stream per quantization)."""
    mode: str = "rne"
    block2d: bool = False
    swizzled: bool = True
    seed: int = 0
    step: int | None = None
    _entries: dict = field(default_factory=dict)
    _next_id: int = 0
    quantizations: int = 0

    def mark_step(self) -> None:
        """Call after each optimizer step: every weight is re-quantized on its next get."""
        self.step = 0 if self.step is None else self.step + 1

    @staticmethod
    def _key(w: torch.Tensor):
        return (w.data_ptr(), tuple(w.shape), w.dtype, w.device)

    def _expire(self, key, ref) -> None:
        e = self._entries.get(key)
        if e is not None and e.ref is ref:
            del self._entries[key]

    def get(self, w: torch.Tensor, step: int | None = None, stream=None) -> nvfp4.Quantized:
        """The quantized weight for this version of w (quantized now if it changed)."""
        key = self._key(w)
        if step is None:
            step = self.step
        version = ("step", step) if step is not None else ("version", w._version)
        e = self._entries.get(key)
        if e is not None and e.ref() is w and e.version == version:
            e.hits += 1
            return e.q
        if e is not None and e.ref() is w:
            wid, count = e.weight_id, e.count
        else:  # a weight not seen before (or a new object at a freed weight's address)
            wid, count = self._next_id, 0
            self._next_id += 1
        offset = ((wid & 0xFFFFFFFF) << 32) | (count & 0xFFFFFFFF)
        # the old buffers are rewritten only when no other live tensor owns them
        owner = e.ref() if e is not None else None
        reuse = e is not None and (owner is w or owner is None)
        q = nvfp4.quantize(w, mode=self.mode, rowwise=True, colwise=True, block2d=self.block2d,
                           swizzled=self.swizzled, seed=self.seed, offset=offset, stream=stream,
                           out=e.q if reuse else None)
        self.quantizations += 1
        cache_ref = weakref.ref(self)

        def expire(r, key=key, cache_ref=cache_ref):
            c = cache_ref()
            if c is not None:
                c._expire(key, r)

        self._entries[key] = _Entry(weakref.ref(w, expire), version, q, wid, count + 1)
        return q

    def drop(self, w: torch.Tensor) -> None:
        """Forget w's copy (its buffers are released with the last reference)."""
        self._entries.pop(self._key(w), None)

    def __len__(self) -> int:
        return len(self._entries)
