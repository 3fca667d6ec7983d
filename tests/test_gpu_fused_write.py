"""pkv_slot_mapping_and_write (the slot mapping fused into the cache write) and
pkv_paged_attention_with_write (the whole step of a layer in one call)
against the oracle on the GPU: slots and the whole pool bit-exact, the same
handling of padding rows and inconsistent lengths as the two separate calls.
"""

import numpy as np
import pytest

from parity import assert_close, oracle_step

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU containers
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
from paged_kv_cache_hkv_gb300 import binding, synth  # noqa: E402
from paged_kv_cache_hkv_gb300.runner import DeviceStep  # noqa: E402
from paged_kv_cache_hkv_gb300.synth import RequestSpec, make_step  # noqa: E402


@pytest.fixture(autouse=True)
def _clear_errors():
    binding.pkv_get_device_errors(clear=True)
    yield


def fused_write_matches_oracle(step):
    ds = DeviceStep(step, fused_write=True)
    ds.slot_mapping.fill_(12345)
    ds.slot_map_and_write()
    torch.cuda.synchronize()
    assert binding.pkv_get_device_errors(clear=True) == 0
    slots, pool, _ = oracle_step(step, rows=[])
    assert np.array_equal(ds.slots_host(), slots)
    assert np.array_equal(ds.pool_host(), pool)
    return ds


@pytest.mark.parametrize("name", ["tiny_decode", "llama_decode", "prefix_sharing", "prefill_rows"])
def test_fused_write_workloads(name):
    fused_write_matches_oracle(synth.WORKLOADS[name]())


@pytest.mark.parametrize("B", [8, 16, 32])
def test_fused_write_block_sizes_and_the_mixed_step(B):
    """The whole mixed step through run() with the fused write, at every block
    size: slots and pool exact, attention within the tolerance."""
    step = synth.mixed_step(block_size=B)
    ds = DeviceStep(step, fused_write=True)
    ds.run()
    torch.cuda.synchronize()
    assert binding.pkv_get_device_errors(clear=True) == 0
    slots, pool, ref = oracle_step(step)
    assert np.array_equal(ds.slots_host(), slots)
    assert np.array_equal(ds.pool_host(), pool)
    assert_close(ds.out_host(), ref)


@pytest.mark.parametrize("Hq,Hkv,D", [(4, 2, 64), (8, 8, 128), (64, 32, 128)])
def test_fused_write_row_widths(Hq, Hkv, D):
    """Rows of 256 B to 8 KB: the widest take the path past the words a lane
    loads before its slot is known."""
    rng = np.random.default_rng(Hkv * 7 + D)
    specs = [RequestSpec(int(c), int(n)) for c, n in zip(rng.integers(0, 300, 9),
                                                          rng.integers(1, 40, 9))]
    fused_write_matches_oracle(make_step(specs, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                                         seed=int(Hq + D)))


def test_fused_write_without_a_slot_buffer():
    step = synth.tiny_decode()
    ds = DeviceStep(step)
    binding.pkv_slot_mapping_and_write(ds.kv_cache, ds.k, ds.v, ds.block_table,
                                       ds.query_start_loc, ds.num_computed, slot_mapping=None)
    torch.cuda.synchronize()
    assert binding.pkv_get_device_errors(clear=True) == 0
    _, pool, _ = oracle_step(step, rows=[])
    assert np.array_equal(ds.pool_host(), pool)


def test_fused_write_padding_rows_and_empty_requests():
    specs = [RequestSpec(30, 1), RequestSpec(12, 0), RequestSpec(64, 3)]
    step = make_step(specs, num_q_heads=8, num_kv_heads=2, head_dim=64, seed=5)
    ds = DeviceStep(step)
    T, pad = step.num_tokens, 3
    k = torch.cat([ds.k, torch.zeros((pad, 2, 64), dtype=ds.k.dtype, device="cuda")])
    v = torch.cat([ds.v, torch.ones((pad, 2, 64), dtype=ds.v.dtype, device="cuda")])
    slots = torch.full((T + pad,), 777, dtype=torch.int64, device="cuda")
    binding.pkv_slot_mapping_and_write(ds.kv_cache, k, v, ds.block_table, ds.query_start_loc,
                                       ds.num_computed, slot_mapping=slots)
    torch.cuda.synchronize()
    assert binding.pkv_get_device_errors(clear=True) == 0
    got = slots.cpu().numpy()
    ref_slots, pool, _ = oracle_step(step, rows=[])
    assert (got[T:] == -1).all()
    assert np.array_equal(got[:T], ref_slots)
    assert np.array_equal(ds.pool_host(), pool)


def test_fused_write_rows_of_a_request_with_bad_lengths_get_no_slot():
    specs = [RequestSpec(40, 3), RequestSpec(70, 5), RequestSpec(9, 1)]
    step = make_step(specs, num_q_heads=8, num_kv_heads=2, head_dim=64, seed=12)
    ds = DeviceStep(step)
    before = ds.pool_host()
    nc = ds.num_computed.clone()
    nc[1] = -1  # request 1: rows 3..7
    ds.slot_mapping.copy_(torch.arange(step.num_tokens, dtype=torch.int64, device="cuda") + 16)
    binding.pkv_slot_mapping_and_write(ds.kv_cache, ds.k, ds.v, ds.block_table,
                                       ds.query_start_loc, nc, slot_mapping=ds.slot_mapping)
    assert binding.pkv_get_device_errors(clear=True) & binding.DEVERR_LENGTHS
    slots = ds.slots_host()
    ref = oracle_step(step, rows=[])[0]
    assert (slots[3:8] == -1).all()
    assert np.array_equal(slots[:3], ref[:3]) and np.array_equal(slots[8:], ref[8:])
    kept = ref.copy()
    kept[3:8] = -1
    assert np.array_equal(ds.pool_host(), oracle.kv_write(before, step.k, step.v, kept))


def test_fused_write_rows_before_a_bad_first_request_get_no_slot():
    specs = [RequestSpec(5, 2), RequestSpec(30, 4)]
    step = make_step(specs, num_q_heads=8, num_kv_heads=2, head_dim=64, seed=13)
    ds = DeviceStep(step)
    qsl = torch.tensor([1, 2, 6], dtype=torch.int32, device="cuda")  # [0] must be 0
    ds.slot_mapping.fill_(5)
    binding.pkv_slot_mapping_and_write(ds.kv_cache, ds.k, ds.v, ds.block_table, qsl,
                                       ds.num_computed, slot_mapping=ds.slot_mapping)
    assert binding.pkv_get_device_errors(clear=True) & binding.DEVERR_LENGTHS
    slots = ds.slots_host()
    assert (slots[:2] == -1).all()  # request 0 and the row before it
    assert np.array_equal(slots[2:], oracle_step(step, rows=[])[0][2:])


def test_fused_write_agrees_with_the_two_calls_on_random_batches():
    rng = np.random.default_rng(21)
    for trial in range(6):
        n = int(rng.integers(1, 40))
        specs = [RequestSpec(int(rng.integers(0, 500)), int(rng.choice([0, 1, 1, 1, 7, 33])))
                 for _ in range(n)]
        specs[0] = RequestSpec(specs[0].num_computed, max(1, specs[0].query_len))
        B = int(rng.choice([8, 16, 32]))
        step = make_step(specs, num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=B,
                         seed=100 + trial)
        a = DeviceStep(step)
        a.slot_map()
        a.write()
        b = DeviceStep(step, fused_write=True)
        b.slot_map_and_write()
        torch.cuda.synchronize()
        assert binding.pkv_get_device_errors(clear=True) == 0
        assert np.array_equal(a.slots_host(), b.slots_host())
        assert np.array_equal(a.pool_host(), b.pool_host())


# ------------------------------------------------- the one-call step (write + attention)
def one_call_step_matches_oracle(step, shared_prefix=None, expect_flags=0, rows=None):
    ds = DeviceStep(step, write_in_attention=True, shared_prefix=shared_prefix)
    ds.slot_mapping.fill_(12345)
    ds.run()
    torch.cuda.synchronize()
    assert binding.pkv_get_device_errors(clear=True) == expect_flags
    slots, pool, ref = oracle_step(step, rows=rows)
    assert np.array_equal(ds.slots_host(), slots)
    assert np.array_equal(ds.pool_host(), pool)
    assert_close(ds.out_host(), ref, rows=rows)


@pytest.mark.parametrize("B", [8, 16, 32])
def test_one_call_mixed_step(B):
    one_call_step_matches_oracle(synth.mixed_step(block_size=B))


@pytest.mark.parametrize("name", ["tiny_decode", "llama_decode", "prefill_rows"])
def test_one_call_workloads(name):
    one_call_step_matches_oracle(synth.WORKLOADS[name]())


def test_one_call_with_the_shared_prefix_hint():
    from paged_kv_cache_hkv_gb300.runner import shared_prefix_of
    step = synth.prefix_sharing()
    one_call_step_matches_oracle(step, shared_prefix=shared_prefix_of(step))


@pytest.mark.parametrize("Hq,Hkv,D", [(12, 3, 128), (8, 8, 64), (16, 2, 64)])
def test_one_call_head_shapes_with_chunks(Hq, Hkv, D):
    """Chunked prefills and decodes in one batch at group sizes 4, 1 and 8:
    the prefill's query tile is 128 / G queries."""
    specs = [RequestSpec(40, 70), RequestSpec(300, 1), RequestSpec(0, 33), RequestSpec(129, 1),
             RequestSpec(17, 200)]
    one_call_step_matches_oracle(make_step(specs, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                                           seed=Hq * 10 + D))


def test_one_call_without_attention_still_writes():
    """max_query_len 0 leaves the attention out; the slots and rows are
    still mapped and written."""
    step = synth.tiny_decode()
    ds = DeviceStep(step)
    ds.out.fill_(3.0)
    s = step
    binding.pkv_paged_attention_with_write(
        ds.out, ds.q, ds.kv_cache, ds.k, ds.v, ds.block_table, ds.seq_lens, ds.query_start_loc,
        ds.num_computed, max_query_len=0, max_seq_len=s.max_seq_len, scale=s.scale,
        workspace=ds.workspace, slot_mapping=ds.slot_mapping)
    torch.cuda.synchronize()
    assert binding.pkv_get_device_errors(clear=True) == 0
    slots, pool, _ = oracle_step(step, rows=[])
    assert np.array_equal(ds.slots_host(), slots)
    assert np.array_equal(ds.pool_host(), pool)
    assert (ds.out_host() == 0x4040).all()  # untouched (3.0 in bf16)


def test_one_call_bad_lengths_flagged_and_not_written():
    specs = [RequestSpec(40, 3), RequestSpec(70, 5), RequestSpec(9, 1)]
    step = make_step(specs, num_q_heads=8, num_kv_heads=2, head_dim=64, seed=12)
    ds = DeviceStep(step)
    before = ds.pool_host()
    nc = ds.num_computed.clone()
    nc[1] = -1  # request 1: rows 3..7
    s = step
    binding.pkv_paged_attention_with_write(
        ds.out, ds.q, ds.kv_cache, ds.k, ds.v, ds.block_table, ds.seq_lens, ds.query_start_loc,
        nc, max_query_len=s.max_query_len, max_seq_len=s.max_seq_len, scale=s.scale,
        workspace=ds.workspace, slot_mapping=ds.slot_mapping)
    assert binding.pkv_get_device_errors(clear=True) & binding.DEVERR_LENGTHS
    slots = ds.slots_host()
    ref = oracle_step(step, rows=[])[0]
    assert (slots[3:8] == -1).all()
    kept = ref.copy()
    kept[3:8] = -1
    assert np.array_equal(ds.pool_host(), oracle.kv_write(before, step.k, step.v, kept))
