"""Inputs that drive the online-softmax rescale and merge paths.

With N(0, 1) inputs at scale 1/sqrt(d) the running max of a long softmax
settles after its first chunk, so a lazily rescaled online softmax (the
running max is only moved when a chunk beats it by more than 2^8) never
rescales a non-empty partial, and split-KV partials never differ by enough
for exp2(m_p - M) to underflow. These cases change that, each in its own way:

* ``scale``: the softmax scale raised to 8/sqrt(d), so that scores spread
  over tens of powers of two;
* ``drift``: keys carry a component that grows with their position
  (synth ``key_drift``): the max of one head in three climbs all along the
  sequence, so it is moved again and again while earlier keys still carry
  weight;
* ``steep``: the same with a drift so steep that every move makes the
  earlier partial underflow to zero, in a chunk, in a merge of two prefill
  partials and in the split-KV combine;
* ``spike``: one key near the end of each decode context outweighs all the
  others by hundreds of powers of two (synth ``spike``), so every split-KV
  piece that does not hold it gets weight exactly zero.

Every case is a seeded ``synth.make_step``; the GPU parity tests and the CPU
restatement of the kernels' update rules take the same inputs.
"""

import math

import numpy as np

from paged_kv_cache_hkv_gb300.synth import RequestSpec, make_step


def _decode_specs(rng, n, lo, hi):
    return [RequestSpec(int(L) - 1, 1) for L in rng.integers(lo, hi, size=n, endpoint=True)]


def _prefill_specs(rng):
    """Chunks over a cached prefix (items of many key tiles), fresh prompts
    (one-tile items and longer ones) and a few decodes."""
    specs = [RequestSpec(int(rng.integers(200, 1500)), int(rng.integers(100, 300)))
             for _ in range(3)]
    specs += [RequestSpec(0, int(rng.integers(2, 60))) for _ in range(4)]
    specs += [RequestSpec(0, int(rng.integers(130, 400)))]
    specs += _decode_specs(rng, 4, 100, 1200)
    return specs


def drift_for(growth, D):
    """key_drift that makes a rising head's score grow by about ``growth``
    powers of two per key at scale 1/sqrt(D): the q components that meet the
    drift average +1, so the score moves by key_drift * D/2 * scale * log2(e)
    per position."""
    return growth * 2.0 * math.sqrt(D) / (D * math.log2(math.e))


def case(name, Hq=32, Hkv=8, D=128, B=16, seed=0):
    """One seeded step of the named case (see the module docstring)."""
    rng = np.random.default_rng(1000 + seed)
    shape = dict(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=B)
    if name == "decode_scale":
        return make_step(_decode_specs(rng, 12, 200, 3000), scale=8 / math.sqrt(D), seed=seed,
                         **shape)
    if name == "decode_drift":
        # a rising head gains ~1 power of two per 16-key chunk: its max is
        # moved every ~8 chunks while the keys before still carry weight
        return make_step(_decode_specs(rng, 12, 200, 3000), key_drift=drift_for(0.06, D),
                         seed=seed, **shape)
    if name == "decode_steep":
        return make_step(_decode_specs(rng, 12, 200, 3000), key_drift=drift_for(1.5, D),
                         seed=seed, **shape)
    if name == "decode_spike":
        return make_step(_decode_specs(rng, 12, 200, 3000), spike=16.0, seed=seed, **shape)
    if name == "prefill_scale":
        return make_step(_prefill_specs(rng), scale=8 / math.sqrt(D), seed=seed, **shape)
    if name == "prefill_drift":
        # ~2.5 powers of two per 256 keys: a softmax warpgroup, which holds
        # every other 128-key tile, moves its max every few of its tiles
        return make_step(_prefill_specs(rng), key_drift=drift_for(0.01, D), seed=seed,
                         **shape)
    if name == "prefill_steep":
        return make_step(_prefill_specs(rng), key_drift=drift_for(1.5, D), seed=seed,
                         **shape)
    raise KeyError(name)


DECODE_CASES = ["decode_scale", "decode_drift", "decode_steep", "decode_spike"]
PREFILL_CASES = ["prefill_scale", "prefill_drift", "prefill_steep"]
