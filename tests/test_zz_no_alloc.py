"""The attention entry point that allocates nothing, against the normal one.

pkv_paged_attention_static_workspace serves callers that cannot allocate
device memory -- a server whose memory all went to its own allocator and KV
pool at start-up, a plugin whose host framework forbids raw cudaMalloc, a
plain C caller with no allocator. It runs the same kernels on a scratch array
built into the library, so its output must be the same bits as the normal
call's, and both must match the oracle. This file is collected last so that
a failure here leaves every other test already run; it passes alone in a
fresh process and after the rest of the suite.
"""

import ctypes

import numpy as np
import pytest

from parity import assert_close, oracle_step

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU containers
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from paged_kv_cache_hkv_gb300 import binding  # noqa: E402
from paged_kv_cache_hkv_gb300.runner import DeviceStep, bf16_to_numpy  # noqa: E402
from paged_kv_cache_hkv_gb300.synth import RequestSpec, make_step  # noqa: E402


def _static_call(ds, out):
    s = ds.step
    binding.pkv_paged_attention_static_workspace(
        out, ds.q, ds.kv_cache, ds.block_table, ds.seq_lens, ds.query_start_loc,
        ds.num_computed, max_query_len=s.max_query_len, max_seq_len=s.max_seq_len,
        scale=s.scale)
    torch.cuda.synchronize()


def _memory():
    torch.cuda.synchronize()
    return torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]


def test_static_workspace_matches_the_workspace_entry_point_twice():
    steps = [
        # chunked prefill + decodes, Llama layer shape
        make_step([RequestSpec(300, 45), RequestSpec(0, 17), RequestSpec(1000, 1),
                   RequestSpec(63, 1), RequestSpec(4000, 1)],
                  num_q_heads=32, num_kv_heads=8, head_dim=128, seed=101),
        # a different shape right after: nothing left over from the first call may leak in
        make_step([RequestSpec(L - 1, 1) for L in (5, 16, 17, 40, 2049, 300)] +
                  [RequestSpec(20, 30)],
                  num_q_heads=8, num_kv_heads=2, head_dim=64, seed=102),
    ]
    outs = []
    for step in steps:
        ds = DeviceStep(step)
        ds.run()  # normal entry point with a torch-allocated workspace
        torch.cuda.synchronize()
        ref_bits = ds.out_host().copy()
        out = torch.full_like(ds.out, float("nan"))
        outs.append((ds, out, ref_bits))
    # first static call: the library looks up its scratch array's address
    _static_call(outs[0][0], outs[0][1])
    for rnd in range(2):  # two calls in a row per step, alternating shapes
        for ds, out, ref_bits in outs:
            out.fill_(float("nan"))
            before = _memory()
            _static_call(ds, out)
            # nothing was allocated: neither torch's allocator nor the device
            assert _memory() == before
            got = bf16_to_numpy(out)
            # the same kernels on the same inputs: the same bits
            assert np.array_equal(got, ref_bits), f"round {rnd}: differs from the workspace call"
            if rnd == 0:
                _, _, ref = oracle_step(ds.step)
                assert_close(got, ref)
    assert binding.pkv_get_device_errors(clear=True) == 0


def test_static_workspace_rejects_calls_beyond_its_size():
    lib = binding.load()
    lay = binding.pkv_cache_layout(1000, 16, 8, 128)
    huge = 200000  # requests: needs far more than the built-in array
    assert lib.pkv_attention_workspace_size(huge, 32, lay, None) > \
        int(ctypes.c_uint32(32 << 20).value)
    st = lib.pkv_paged_attention_static_workspace(
        None, None, 0, None, None, 0, None, None, None, huge, 1, 1, 16, 32, 0.1, lay, None, None)
    assert st == binding.PKV_ERR_SCRATCH_LIMIT
