"""CUDA path vs the CPU oracle on the GPU (through the C ABI).

Slot mapping and the cache write must be bit-exact (the whole pool is
compared, so untouched slots must be unchanged too); attention must be within
|gpu - oracle| <= max(2e-2, 1e-2 * |oracle|) per element.
"""

import math

import numpy as np
import pytest

import rescale_cases
from parity import assert_close, oracle_step

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU containers
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from paged_kv_cache_hkv_gb300 import binding, synth  # noqa: E402
from paged_kv_cache_hkv_gb300.runner import DeviceStep  # noqa: E402
from paged_kv_cache_hkv_gb300.synth import RequestSpec, make_step  # noqa: E402


@pytest.fixture(autouse=True)
def _clear_errors():
    binding.pkv_get_device_errors(clear=True)
    yield


WRITE_PATHS = {"separate": {}, "fused": {"fused_write": True},
               "attention": {"write_in_attention": True}}


def run_and_check(step, decode_splits=None, rows=None, check_pool=True, shared_prefix=None,
                  expect_flags=0, write="separate"):
    """One step through the library -- slot mapping, write, attention made as
    three calls (separate), as the fused write plus attention (fused), or as
    the one call with the write inside (attention) -- against the oracle."""
    ds = DeviceStep(step, decode_splits=decode_splits, shared_prefix=shared_prefix,
                    **WRITE_PATHS[write])
    ds.run()
    torch.cuda.synchronize()
    assert binding.pkv_get_device_errors(clear=True) == expect_flags
    slots, pool, ref = oracle_step(step, rows=rows)
    assert np.array_equal(ds.slots_host(), slots)
    if check_pool:
        assert np.array_equal(ds.pool_host(), pool)
    return assert_close(ds.out_host(), ref, rows=rows)


# ---------------------------------------------------------------- workloads
DECODE_WORKLOADS = ["tiny_decode", "llama_decode", "prefix_sharing", "long_context"]


@pytest.mark.parametrize("name", DECODE_WORKLOADS)
def test_decode_workload_parity(name):
    step = synth.WORKLOADS[name]()
    run_and_check(step, check_pool=(name != "long_context"))


def test_long_context_pool_written_exactly():
    step = synth.long_context()
    ds = DeviceStep(step)
    ds.slot_map()
    ds.write()
    slots, _, _ = oracle_step(step, rows=[])
    assert np.array_equal(ds.slots_host(), slots)
    pool = ds.pool_host()
    # every written row is the input row; compare all blocks the step touches
    blocks = np.unique(step.block_table[step.block_table >= 0])
    expect = step.kv_cache[blocks].copy()
    for t, s in enumerate(slots):
        bi = np.searchsorted(blocks, s // 16)
        expect[bi, 0, s % 16] = step.k[t]
        expect[bi, 1, s % 16] = step.v[t]
    assert np.array_equal(pool[blocks], expect)


def test_long_prefill_sampled_rows():
    """Chunks of 2048 new tokens over 6144 cached ones (keys up to 8192):
    sampled rows from every chunk, both ends of each included."""
    step = synth.long_prefill()
    rng = np.random.default_rng(6)
    rows = set(rng.choice(step.num_tokens, size=200, replace=False).tolist())
    for r in range(step.num_reqs):
        rows.update({int(step.query_start_loc[r]), int(step.query_start_loc[r + 1]) - 1})
    run_and_check(step, rows=sorted(rows), check_pool=False)


def test_mixed_step_parity():
    step = synth.mixed_step()
    run_and_check(step)


# ---------------------------------------------------------------- split-KV
@pytest.mark.parametrize("splits", [1, 3, 7, 64, 1000, 5000])
def test_split_kv_partitionings(splits):
    step = make_step([RequestSpec(L - 1, 1) for L in (1, 2, 15, 16, 17, 33, 100, 257, 1000,
                                                       3001)],
                     num_q_heads=8, num_kv_heads=2, head_dim=128, seed=40 + splits)
    run_and_check(step, decode_splits=splits)


@pytest.mark.parametrize("Hq,Hkv,D", [(4, 4, 128), (8, 4, 128), (16, 4, 128), (32, 4, 128),
                                      (4, 4, 64), (8, 4, 64), (16, 4, 64), (64, 8, 64),
                                      (12, 3, 128)])
def test_decode_head_shapes(Hq, Hkv, D):
    rng = np.random.default_rng(Hq * 100 + D)
    lens = rng.integers(1, 700, size=23)
    step = make_step([RequestSpec(int(L) - 1, 1) for L in lens], num_q_heads=Hq,
                     num_kv_heads=Hkv, head_dim=D, seed=int(Hq + D))
    run_and_check(step)
    run_and_check(step, decode_splits=37)


def test_decode_shuffled_order_same_rows():
    rng = np.random.default_rng(7)
    lens = rng.integers(20, 900, size=17)
    specs = [RequestSpec(int(L) - 1, 1) for L in lens]
    a = make_step(specs, num_q_heads=32, num_kv_heads=8, head_dim=128, seed=9)
    run_and_check(a, decode_splits=50)


def test_padding_rows_and_empty_requests():
    # a request with no new tokens and trailing padding rows past the batch
    specs = [RequestSpec(30, 1), RequestSpec(12, 0), RequestSpec(64, 1)]
    step = make_step(specs, num_q_heads=8, num_kv_heads=2, head_dim=64, seed=5)
    ds = DeviceStep(step)
    T = step.num_tokens
    pad = 3
    # grow the token arrays by padding rows
    ds.q = torch.cat([ds.q, torch.zeros((pad,) + tuple(ds.q.shape[1:]), dtype=ds.q.dtype,
                                        device=ds.q.device)])
    ds.out = torch.full((T + pad, 8, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    ds.slot_mapping = torch.empty(T + pad, dtype=torch.int64, device="cuda")
    ds.k = torch.cat([ds.k, torch.zeros((pad, 2, 64), dtype=ds.k.dtype, device="cuda")])
    ds.v = torch.cat([ds.v, torch.zeros((pad, 2, 64), dtype=ds.v.dtype, device="cuda")])
    ds.run()
    torch.cuda.synchronize()
    assert binding.pkv_get_device_errors(clear=True) == 0
    slots = ds.slots_host()
    assert (slots[T:] == -1).all()
    ref_slots, pool, ref = oracle_step(step)
    assert np.array_equal(slots[:T], ref_slots)
    assert np.array_equal(ds.pool_host(), pool)
    out = ds.out_host()
    assert_close(out[:T], ref)
    assert (out[T:] == 0x40E0).all()  # padding rows untouched (7.0 in bf16)


def test_empty_batch_is_a_no_op():
    step = make_step([RequestSpec(5, 1)], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=1)
    ds = DeviceStep(step)
    lay = ds.layout
    lib = binding.load()
    assert lib.pkv_paged_attention(None, None, 0, None, None, 0, None, None, None, 0, 0, 0, 0,
                                   4, 1.0, lay, None, 0, None, None) == 0
    assert lib.pkv_paged_kv_write(None, None, None, 0, 0, None, 0, lay, None) == 0


# ---------------------------------------------------------------- bad data
def test_out_of_range_slot_is_skipped_and_flagged():
    step = make_step([RequestSpec(3, 2)], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=2)
    ds = DeviceStep(step)
    before = ds.pool_host()
    bad = torch.tensor([step.num_blocks * 16 + 5, -1], dtype=torch.int64, device="cuda")
    binding.pkv_paged_kv_write(ds.kv_cache, ds.k, ds.v, bad)
    flags = binding.pkv_get_device_errors(clear=True)
    assert flags & binding.DEVERR_SLOT_RANGE
    assert np.array_equal(ds.pool_host(), before)


def test_bad_block_id_is_masked_and_flagged():
    step = make_step([RequestSpec(40, 1), RequestSpec(20, 1)], num_q_heads=4, num_kv_heads=2,
                     head_dim=64, seed=3)
    ds = DeviceStep(step)
    ds.slot_map()
    ds.write()
    bt = ds.block_table.clone()
    bt[0, 0] = step.num_blocks + 100  # outside the pool
    ds.block_table = bt
    ds.attend()
    flags = binding.pkv_get_device_errors(clear=True)
    assert flags & binding.DEVERR_BLOCK_RANGE
    # request 1 is untouched by the bad entry of request 0
    _, _, ref = oracle_step(step)
    assert_close(ds.out_host()[1:], ref[1:])


def test_rows_of_a_request_with_bad_lengths_get_no_slot():
    """A request whose lengths are inconsistent gets -1 in every row, so
    nothing the slot buffer held before the call (here: valid slots of
    other blocks) can steer this step's K/V into the pool."""
    specs = [RequestSpec(40, 3), RequestSpec(70, 5), RequestSpec(9, 1)]
    step = make_step(specs, num_q_heads=8, num_kv_heads=2, head_dim=64, seed=12)
    ds = DeviceStep(step)
    before = ds.pool_host()
    nc = ds.num_computed.clone()
    nc[1] = -1  # request 1: rows 3..7
    ds.slot_mapping.copy_(torch.arange(step.num_tokens, dtype=torch.int64, device="cuda") + 16)
    binding.pkv_slot_mapping(ds.slot_mapping, ds.block_table, ds.query_start_loc, nc,
                             step.num_blocks, step.block_size)
    binding.pkv_paged_kv_write(ds.kv_cache, ds.k, ds.v, ds.slot_mapping)
    assert binding.pkv_get_device_errors(clear=True) & binding.DEVERR_LENGTHS
    slots = ds.slots_host()
    ref = oracle_step(step, rows=[])[0]
    assert (slots[3:8] == -1).all()
    assert np.array_equal(slots[:3], ref[:3]) and np.array_equal(slots[8:], ref[8:])
    # the pool holds exactly the other requests' rows
    kept = ref.copy()
    kept[3:8] = -1
    import oracle
    assert np.array_equal(ds.pool_host(), oracle.kv_write(before, step.k, step.v, kept))


def test_rows_before_a_bad_first_request_get_no_slot():
    specs = [RequestSpec(5, 2), RequestSpec(30, 4)]
    step = make_step(specs, num_q_heads=8, num_kv_heads=2, head_dim=64, seed=13)
    ds = DeviceStep(step)
    qsl = torch.tensor([1, 2, 6], dtype=torch.int32, device="cuda")  # [0] must be 0
    ds.slot_mapping.fill_(5)
    binding.pkv_slot_mapping(ds.slot_mapping, ds.block_table, qsl, ds.num_computed,
                             step.num_blocks, step.block_size)
    assert binding.pkv_get_device_errors(clear=True) & binding.DEVERR_LENGTHS
    slots = ds.slots_host()
    assert (slots[:2] == -1).all()  # request 0 and the row before it
    assert np.array_equal(slots[2:], oracle_step(step, rows=[])[0][2:])


def test_inconsistent_lengths_are_flagged():
    step = make_step([RequestSpec(10, 1)], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=4)
    ds = DeviceStep(step)
    ds.slot_map()
    ds.write()
    ds.seq_lens = ds.seq_lens + 1  # no longer num_computed + query_len
    ds.attend()
    assert binding.pkv_get_device_errors(clear=True) & binding.DEVERR_LENGTHS


# ---------------------------------------------------------------- prefill (tensor cores)
PREFILL_SPECS = [RequestSpec(0, 2), RequestSpec(15, 3), RequestSpec(16, 17), RequestSpec(17, 100),
                 RequestSpec(200, 129), RequestSpec(1, 1), RequestSpec(33, 300),
                 RequestSpec(127, 1), RequestSpec(0, 128), RequestSpec(250, 64)]


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (8, 8, 128), (16, 8, 128), (64, 8, 128),
                                      (8, 4, 64), (8, 8, 64), (16, 2, 64), (32, 4, 64)])
def test_prefill_mixed_shapes(Hq, Hkv, D):
    step = make_step(PREFILL_SPECS, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                     seed=Hq * 7 + D)
    run_and_check(step)


@pytest.mark.parametrize("n_prefill", [127, 128, 129, 300])
def test_many_prefill_requests(n_prefill):
    """More prefill requests than a CTA keeps in shared memory (128) take the
    global-memory metadata path; thousands of small items cycle the CTAs'
    item queues many times. Decodes are interleaved between them."""
    rng = np.random.default_rng(n_prefill)
    specs = []
    for i in range(n_prefill):
        specs.append(RequestSpec(int(rng.integers(0, 300)), int(rng.integers(2, 40))))
        if i % 3 == 0:
            specs.append(RequestSpec(int(rng.integers(0, 500)), 1))
    step = make_step(specs, num_q_heads=16, num_kv_heads=4, head_dim=128, seed=n_prefill)
    rows = rng.choice(step.num_tokens, size=min(step.num_tokens, 1500), replace=False)
    run_and_check(step, rows=np.sort(rows))


def test_prefill_is_deterministic_across_runs():
    """Thousands of items of 1-3 key tiles are claimed by the CTAs in a
    different order every run (a work counter), so each CTA's tile parity,
    and with it which softmax warpgroup holds which tiles, changes from run
    to run; the output must still be the same bits."""
    rng = np.random.default_rng(77)
    specs = [RequestSpec(int(rng.integers(0, 300)), int(rng.integers(2, 60))) for _ in range(200)]
    specs += [RequestSpec(int(rng.integers(1000, 3000)), int(rng.integers(100, 300))) for _ in range(6)]
    step = make_step(specs, num_q_heads=32, num_kv_heads=8, head_dim=128, seed=77)
    ds = DeviceStep(step)
    outs = []
    for _ in range(4):
        ds.run()
        torch.cuda.synchronize()
        outs.append(ds.out.clone())
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    assert binding.pkv_get_device_errors(clear=True) == 0


def test_prefill_chunks_match_one_shot_on_gpu():
    """A prompt split into chunks over three steps gives the rows of the
    one-shot prefill (each chunk attends the cached prefix plus itself)."""
    full = make_step([RequestSpec(0, 400)], num_q_heads=32, num_kv_heads=8, head_dim=128,
                     seed=77, shuffle_pool=True)
    ds = DeviceStep(full)
    ds.run()
    torch.cuda.synchronize()
    one_shot = ds.out_host().copy()
    _, _, ref = oracle_step(full)
    assert_close(one_shot, ref)  # the one-shot prefill against the oracle
    for c, n in ((0, 150), (150, 131), (281, 119)):
        step = make_step([RequestSpec(c, n)], num_q_heads=32, num_kv_heads=8, head_dim=128,
                         seed=77)
        # reuse the one-shot pool, table and rows: the cache already holds
        # every token of the prompt after the one-shot write
        q = ds.q[c:c + n].contiguous()
        out = torch.zeros_like(q)
        qsl = torch.tensor([0, n], dtype=torch.int32, device="cuda")
        sl = torch.tensor([c + n], dtype=torch.int32, device="cuda")
        nc = torch.tensor([c], dtype=torch.int32, device="cuda")
        ws = torch.empty(binding.pkv_attention_workspace_size(1, 32, ds.layout), dtype=torch.uint8,
                         device="cuda")
        binding.pkv_paged_attention(out, q, ds.kv_cache, ds.block_table, sl, qsl, nc,
                                    max_query_len=n, max_seq_len=c + n, scale=step.scale,
                                    workspace=ws)
        torch.cuda.synchronize()
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        # each chunk's rows against the oracle's one-shot rows (a chunk over a
        # cached prefix is the same attention), and against the GPU one-shot
        assert_close(got, ref[c:c + n], what=f"chunk ({c}, {n})")
        a = got.view(np.uint16).astype(np.uint32) << 16
        b = one_shot[c:c + n].astype(np.uint32) << 16
        diff = np.abs(a.view(np.float32) - b.view(np.float32))
        assert diff.max() <= 2e-2, diff.max()
    assert binding.pkv_get_device_errors(clear=True) == 0


def test_mixed_batch_order_independence():
    specs = [RequestSpec(40, 24), RequestSpec(300, 1), RequestSpec(0, 37), RequestSpec(17, 1),
             RequestSpec(5, 200), RequestSpec(999, 1)]
    step = make_step(specs, num_q_heads=32, num_kv_heads=8, head_dim=128, seed=61)
    run_and_check(step)
    rev = make_step(specs[::-1], num_q_heads=32, num_kv_heads=8, head_dim=128, seed=61)
    run_and_check(rev, decode_splits=9)


# ---------------------------------------------------------------- block sizes
# Lengths around every multiple of 8 up to 33 (a chunk of 16 keys ends inside
# an 8-token block, on a block edge, in the first or second half of a
# 32-token block), long contexts, fresh prefills, chunks over a cached prefix
# and a chunk shorter than one block.
BLOCK_SPECS = ([RequestSpec(L - 1, 1) for L in (1, 7, 8, 9, 15, 16, 17, 24, 25, 31, 32, 33,
                                               100, 1000, 3001)]
               + [RequestSpec(0, 37), RequestSpec(41, 200), RequestSpec(500, 129),
                  RequestSpec(9, 8), RequestSpec(24, 300)])


@pytest.mark.parametrize("B", [8, 32])
@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (8, 4, 64), (16, 2, 64)])
def test_block_sizes_mixed_step(B, Hq, Hkv, D):
    step = make_step(BLOCK_SPECS, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=B,
                     seed=B * 10 + Hq + D)
    run_and_check(step)
    run_and_check(step, decode_splits=29)


@pytest.mark.parametrize("B", [8, 16, 32])
def test_block_size_leaves_the_result_unchanged_on_gpu(B):
    """One logical batch stored with 8-, 16- or 32-token blocks: the same
    output rows (the pool layout is the only difference)."""
    specs = [RequestSpec(700, 1), RequestSpec(33, 1), RequestSpec(120, 90), RequestSpec(0, 1)]
    step = make_step(specs, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=B, seed=88)
    ds = DeviceStep(step)
    ds.run()
    torch.cuda.synchronize()
    assert binding.pkv_get_device_errors(clear=True) == 0
    ref16 = make_step(specs, num_q_heads=32, num_kv_heads=8, head_dim=128, seed=88)
    assert np.array_equal(step.q, ref16.q)
    _, _, ref = oracle_step(ref16)
    assert_close(ds.out_host(), ref)


@pytest.mark.parametrize("B", [8, 32])
def test_block_sizes_mixed_workload(B):
    run_and_check(synth.mixed_step(block_size=B, num_decodes=200), rows=None)


@pytest.mark.parametrize("B", [8, 32])
def test_block_sizes_bad_block_id_is_masked_and_flagged(B):
    specs = [RequestSpec(60, 1), RequestSpec(100, 1), RequestSpec(40, 30)]
    step = make_step(specs, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=B, seed=3)
    # an entry inside the used range of request 1 points past the pool
    step.block_table[1, 1] = step.num_blocks + 5
    ds = DeviceStep(step)
    ds.run()
    torch.cuda.synchronize()
    assert binding.pkv_get_device_errors(clear=True) & binding.DEVERR_BLOCK_RANGE
    # the other requests are untouched by it
    _, _, ref = oracle_step(step, rows=[0] + list(range(2, step.num_tokens)))
    assert_close(ds.out_host(), ref, rows=[0] + list(range(2, step.num_tokens)))


# ---------------------------------------------------------------- block copies
def _rand_pool(nb, hkv=8, d=128, seed=0, device="cuda", pinned=False, block_size=16):
    g = torch.Generator().manual_seed(seed)
    t = torch.randn((nb, 2, block_size, hkv, d), generator=g).to(torch.bfloat16)
    if pinned:
        return t.pin_memory()
    return t.to(device)


def _host_bits(t):
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def test_copy_blocks_copy_on_write_in_pool():
    import oracle
    pool = _rand_pool(300, seed=1)
    before = _host_bits(pool)
    rng = np.random.default_rng(5)
    ids = rng.permutation(300)
    pairs = np.stack([ids[:60], ids[60:120]], axis=1).astype(np.int32)  # disjoint src / dst
    binding.pkv_copy_blocks(pool, pool, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    assert binding.pkv_get_device_errors(clear=True) == 0
    assert np.array_equal(_host_bits(pool), oracle.copy_blocks(before, before, pairs))


@pytest.mark.parametrize("B", [8, 32])
def test_copy_blocks_other_block_sizes(B):
    import oracle
    pool = _rand_pool(100, hkv=4, d=128, seed=6, block_size=B)
    before = _host_bits(pool)
    pairs = np.array([[3, 90], [50, 7], [99, 0]], np.int32)
    binding.pkv_copy_blocks(pool, pool, torch.from_numpy(pairs).cuda())
    torch.cuda.synchronize()
    assert binding.pkv_get_device_errors(clear=True) == 0
    assert np.array_equal(_host_bits(pool), oracle.copy_blocks(before, before, pairs))


def test_copy_blocks_swap_out_and_in_with_pinned_host_pool():
    import oracle
    dev = _rand_pool(200, hkv=4, d=64, seed=2)
    host = _rand_pool(50, hkv=4, d=64, seed=3, pinned=True)
    dev_bits, host_bits = _host_bits(dev), _host_bits(host)
    out_pairs = np.array([[17, 0], [150, 1], [3, 49], [199, 20]], np.int32)
    binding.pkv_copy_blocks(host, dev, torch.from_numpy(out_pairs).cuda())
    torch.cuda.synchronize()
    host_after = oracle.copy_blocks(host_bits, dev_bits, out_pairs)
    assert np.array_equal(_host_bits(host), host_after)
    in_pairs = np.array([[0, 5], [49, 6], [20, 7]], np.int32)
    binding.pkv_copy_blocks(dev, host, torch.from_numpy(in_pairs).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(_host_bits(dev), oracle.copy_blocks(dev_bits, host_after, in_pairs))
    assert binding.pkv_get_device_errors(clear=True) == 0


def test_copy_blocks_out_of_range_pair_is_skipped_and_flagged():
    pool = _rand_pool(10, hkv=2, d=64, seed=4)
    before = _host_bits(pool)
    pairs = torch.tensor([[2, 10], [-1, 3]], dtype=torch.int32, device="cuda")
    binding.pkv_copy_blocks(pool, pool, pairs)
    assert binding.pkv_get_device_errors(clear=True) & binding.DEVERR_BLOCK_RANGE
    assert np.array_equal(_host_bits(pool), before)


# ---------------------------------------------------------------- online-softmax edge paths
# Inputs whose scores move far along the sequence (raised scale, keys that
# drift with their position, one dominant key): the decode's per-chunk and
# the prefill's per-tile lazy rescale of a non-empty partial, alphas and
# merge weights that underflow to zero, and split-KV pieces of weight zero in
# the combine (rescale_cases; the CPU restatement of the same update rules
# runs on the same inputs in test_online_softmax_logic.py).
@pytest.mark.parametrize("B", [8, 16, 32])
@pytest.mark.parametrize("name", rescale_cases.DECODE_CASES + rescale_cases.PREFILL_CASES)
def test_rescale_paths_llama_shape(name, B):
    step = rescale_cases.case(name, B=B, seed=B)
    run_and_check(step)
    run_and_check(step, decode_splits=1)    # whole requests in one CTA
    run_and_check(step, decode_splits=400)  # pieces of a few chunks each


@pytest.mark.parametrize("Hq,Hkv,D", [(16, 4, 64), (8, 8, 64), (16, 8, 128), (64, 8, 128)])
@pytest.mark.parametrize("name", rescale_cases.DECODE_CASES + rescale_cases.PREFILL_CASES)
def test_rescale_paths_head_shapes(name, Hq, Hkv, D):
    step = rescale_cases.case(name, Hq=Hq, Hkv=Hkv, D=D, seed=Hq + D)
    run_and_check(step, decode_splits=97)


def test_mixed_step_with_raised_scale():
    """The bench workload at 8/sqrt(d): the 512-token chunk's 15-16 key
    tiles per item rescale along the way; sampled rows of every class."""
    step = synth.mixed_step(scale=8 / math.sqrt(128))
    rng = np.random.default_rng(8)
    rows = np.sort(np.concatenate([np.arange(0, 1024, 3),
                                   rng.choice(np.arange(1024, step.num_tokens), 400,
                                              replace=False)]))
    run_and_check(step, rows=rows)


# ---------------------------------------------------------------- shared prefix
# A run of decode requests whose tables start with the same blocks (prefix
# caching, ref_cnt > 1): with the shared-prefix hint the call attends the
# shared keys once per group on the tensor cores and each decode only its own
# keys past them. The result must be the oracle's (shared blocks behave as
# private copies).
def test_prefix_sharing_workload_with_the_shared_prefix_hint():
    step = synth.prefix_sharing()
    from paged_kv_cache_hkv_gb300.runner import shared_prefix_of
    assert shared_prefix_of(step) == (1024, 0, 128)
    run_and_check(step, shared_prefix="auto")
    run_and_check(step, shared_prefix="auto", decode_splits=1)
    run_and_check(step, shared_prefix="auto", decode_splits=600)


def _partly_shared_specs(rng, prefix, n_shared=37):
    specs = [RequestSpec(int(rng.integers(100, 700)), int(rng.integers(40, 200)))]  # a chunk
    specs += [RequestSpec(0, int(rng.integers(2, 80))) for _ in range(3)]             # prompts
    specs += [RequestSpec(int(L) - 1, 1) for L in rng.integers(1, 900, size=9)]        # decodes
    specs += [RequestSpec(prefix + int(x), 1, shares_prefix=True)                     # the run
              for x in rng.integers(0, 300, size=n_shared)]
    specs += [RequestSpec(int(L) - 1, 1) for L in rng.integers(1, 900, size=5)]
    return specs


@pytest.mark.parametrize("B", [8, 16, 32])
@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (16, 4, 64), (8, 8, 128), (64, 8, 128),
                                      (8, 2, 64)])
def test_shared_prefix_in_a_mixed_batch(B, Hq, Hkv, D):
    rng = np.random.default_rng(B * 100 + Hq + D)
    prefix = {8: 96, 16: 800, 32: 512}[B]  # under one key tile, 6.25 tiles, 4 tiles
    step = make_step(_partly_shared_specs(rng, prefix), num_q_heads=Hq, num_kv_heads=Hkv,
                     head_dim=D, block_size=B, prefix_tokens=prefix, seed=B + Hq + D)
    hint = (prefix, 13, 37)
    from paged_kv_cache_hkv_gb300.runner import shared_prefix_of
    assert shared_prefix_of(step) == hint
    run_and_check(step, shared_prefix=hint)
    run_and_check(step, shared_prefix=hint, decode_splits=23)


def test_shared_prefix_hint_is_checked_per_request():
    """Requests of the declared run that do not share the prefix (their own
    tables, or a context not past the prefix) are attended without the hint;
    the run's other requests still use it. The flag says so."""
    rng = np.random.default_rng(5)
    specs = [RequestSpec(512 + int(x), 1, shares_prefix=True) for x in rng.integers(0, 200, 20)]
    specs[7] = RequestSpec(700, 1)    # private table inside the run
    specs[12] = RequestSpec(300, 1)   # shorter than the prefix
    step = make_step(specs, num_q_heads=32, num_kv_heads=8, head_dim=128, prefix_tokens=512,
                     seed=5)
    run_and_check(step, shared_prefix=(512, 0, 20), expect_flags=binding.DEVERR_SHARED)


def test_shared_prefix_hint_over_a_prefill_turns_the_run_off():
    rng = np.random.default_rng(6)
    specs = [RequestSpec(512 + int(x), 1, shares_prefix=True) for x in rng.integers(0, 200, 9)]
    specs.insert(4, RequestSpec(600, 30))  # a chunk inside the declared run
    step = make_step(specs, num_q_heads=32, num_kv_heads=8, head_dim=128, prefix_tokens=512,
                     seed=6)
    run_and_check(step, shared_prefix=(512, 0, 10), expect_flags=binding.DEVERR_SHARED)


@pytest.mark.parametrize("name", ["drift", "steep", "scale"])
def test_shared_prefix_on_the_rescale_paths(name):
    """Keys that drift with their position (the shared items' running max
    moves, their pieces' partials differ by up to thousands of powers of
    two, and the decode continues from the merged partial), or a raised
    scale."""
    rng = np.random.default_rng(7)
    specs = [RequestSpec(1024 + int(x), 1, shares_prefix=True) for x in rng.integers(0, 300, 64)]
    kw = {"drift": dict(key_drift=rescale_cases.drift_for(0.01, 128)),
          "steep": dict(key_drift=rescale_cases.drift_for(1.5, 128)),
          "scale": dict(scale=8 / math.sqrt(128))}[name]
    step = make_step(specs, num_q_heads=32, num_kv_heads=8, head_dim=128, prefix_tokens=1024,
                     seed=8, **kw)
    run_and_check(step, shared_prefix="auto")
    run_and_check(step, shared_prefix="auto", decode_splits=300)


# ---------------------------------------------------------------- CUDA graphs
def test_mixed_step_replays_in_a_cuda_graph():
    specs = [RequestSpec(300, 45), RequestSpec(0, 17), RequestSpec(1000, 1), RequestSpec(63, 1),
             RequestSpec(4000, 1)]
    step = make_step(specs, num_q_heads=32, num_kv_heads=8, head_dim=128, seed=131)
    ds = DeviceStep(step)
    ds.run()
    torch.cuda.synchronize()
    eager = ds.out_host().copy()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ds.run()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ds.run()
    slots, pool, ref = oracle_step(step)
    for _ in range(2):
        ds.out.zero_()
        ds.slot_mapping.fill_(-7)
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(ds.out_host(), eager)
        # the replayed step itself against the oracle: slots, pool, output
        assert np.array_equal(ds.slots_host(), slots)
        assert np.array_equal(ds.pool_host(), pool)
        assert_close(ds.out_host(), ref)
    assert binding.pkv_get_device_errors(clear=True) == 0


# ---------------------------------------------------------------- seeded fuzz
FUZZ_SHAPES = [(4, 4, 64), (8, 4, 64), (16, 4, 64), (32, 4, 64), (8, 8, 128), (16, 8, 128),
               (32, 8, 128), (64, 8, 128), (8, 2, 128), (4, 1, 128), (16, 2, 64), (12, 3, 128)]


@pytest.mark.parametrize("trial", range(36))
def test_seeded_fuzz(trial):
    """Random shapes, block sizes, request mixes (decodes, fresh prefills,
    chunks over a cached prefix, empty requests), split-KV CTA counts and the
    three ways to make a step's calls; the slots, the whole pool and sampled
    rows are checked, and a second run of the step must give the same bits."""
    rng = np.random.default_rng(9000 + trial)
    Hq, Hkv, D = FUZZ_SHAPES[trial % len(FUZZ_SHAPES)]
    B = int(rng.choice([8, 16, 32]))
    specs = []
    for _ in range(int(rng.integers(1, 40))):
        kind = rng.choice(["decode", "decode", "prefill", "chunk", "empty"])
        if kind == "decode":
            specs.append(RequestSpec(int(rng.integers(0, 2000)), 1))
        elif kind == "prefill":
            specs.append(RequestSpec(0, int(rng.integers(2, 300))))
        elif kind == "chunk":
            specs.append(RequestSpec(int(rng.integers(1, 1500)), int(rng.integers(2, 400))))
        else:
            specs.append(RequestSpec(int(rng.integers(0, 500)), 0))
    if all(s.query_len == 0 for s in specs):
        specs.append(RequestSpec(10, 1))
    step = make_step(specs, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=B,
                     seed=trial)
    splits = None if trial % 3 == 0 else int(rng.integers(1, 3000))
    rows = rng.choice(step.num_tokens, size=min(step.num_tokens, 400), replace=False)
    write = ("separate", "fused", "attention")[(trial + trial // len(FUZZ_SHAPES)) % 3]  # each shape: all three
    run_and_check(step, decode_splits=splits, rows=np.sort(rows), write=write)
    # the same step again gives the same bits, whatever the CTAs' schedule
    ds = DeviceStep(step, decode_splits=splits, **WRITE_PATHS[write])
    outs = []
    for _ in range(2):
        ds.run()
        torch.cuda.synchronize()
        outs.append(ds.out.clone())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


@pytest.mark.parametrize("trial", range(40))
def test_wide_fuzz(trial):
    """Wider random steps: up to ~90 requests with chunks of up to 1200 new
    tokens over 4000 cached and decodes over up to 5000 keys; in two steps of
    five, a run of decodes over one shared prefix (a multiple of 16 and of
    B), attended with the shared-prefix hint in most of them; keys that
    drift along the sequence or one key that dwarfs the others (the
    online-softmax rescale paths); a random split-KV CTA count and one of the
    three ways to make the step's calls. Slots, the whole pool and sampled
    rows against the oracle."""
    from paged_kv_cache_hkv_gb300.runner import shared_prefix_of
    rng = np.random.default_rng(77000 + trial)
    Hq, Hkv, D = FUZZ_SHAPES[int(rng.integers(0, len(FUZZ_SHAPES)))]
    B = int(rng.choice([8, 16, 32]))
    specs = []
    for _ in range(int(rng.integers(1, 90))):
        kind = rng.choice(["decode", "decode", "decode", "prefill", "chunk", "empty"])
        if kind == "decode":
            specs.append(RequestSpec(int(rng.integers(0, 5000)), 1))
        elif kind == "prefill":
            specs.append(RequestSpec(0, int(rng.integers(2, 700))))
        elif kind == "chunk":
            specs.append(RequestSpec(int(rng.integers(1, 4000)), int(rng.integers(2, 1200))))
        else:
            specs.append(RequestSpec(int(rng.integers(0, 500)), 0))
    prefix = 0
    if rng.random() < 0.4:
        prefix = max(B, 16) * int(rng.integers(1, 48))
        run = [RequestSpec(prefix + int(rng.integers(0, 600)), 1, shares_prefix=True)
               for _ in range(int(rng.integers(2, 70)))]
        at = int(rng.integers(0, len(specs) + 1))
        specs = specs[:at] + run + specs[at:]
    if all(s.query_len == 0 for s in specs):
        specs.append(RequestSpec(10, 1))
    drift = float(rng.choice([0.0, 0.0, 0.03, 0.08]))
    spike = float(rng.choice([0.0, 0.0, 25.0]))
    step = make_step(specs, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=B,
                     seed=trial, prefix_tokens=prefix, key_drift=drift, spike=spike)
    hint = shared_prefix_of(step) if rng.random() < 0.8 else None
    splits = None if rng.random() < 0.5 else int(rng.integers(1, 4000))
    write = ("separate", "fused", "attention")[int(rng.integers(0, 3))]
    rows = np.sort(rng.choice(step.num_tokens, size=min(step.num_tokens, 250), replace=False))
    run_and_check(step, decode_splits=splits, rows=rows, write=write, shared_prefix=hint)
