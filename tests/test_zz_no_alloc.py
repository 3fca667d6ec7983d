"""The attention entry point that allocates nothing, against the normal one.

pkv_paged_attention_static_workspace serves callers that cannot allocate
device memory -- a server whose memory all went to its own allocator and KV
pool at start-up, a plugin whose host framework forbids raw cudaMalloc, a
plain C caller with no allocator. It runs the same kernels on a scratch array
built into the library. This file is collected last so that a failure here
leaves every other test already run; it passes alone in a fresh process and
after the rest of the suite.
"""

import ctypes

import numpy as np
import pytest

from parity import ABS_TOL, REL_TOL, bits_to_f64

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU containers
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from paged_kv_cache_hkv_gb300 import binding  # noqa: E402
from paged_kv_cache_hkv_gb300.runner import DeviceStep  # noqa: E402
from paged_kv_cache_hkv_gb300.synth import RequestSpec, make_step  # noqa: E402


def _static_call(ds):
    s = ds.step
    out = torch.full_like(ds.out, float("nan"))
    binding.pkv_paged_attention_static_workspace(
        out, ds.q, ds.kv_cache, ds.block_table, ds.seq_lens, ds.query_start_loc,
        ds.num_computed, max_query_len=s.max_query_len, max_seq_len=s.max_seq_len,
        scale=s.scale)
    torch.cuda.synchronize()
    return bits_to_f64(out.view(torch.int16).cpu().numpy().view(np.uint16))


def _check_against(ref_bits, got):
    ref = bits_to_f64(ref_bits)
    err = np.abs(got - ref)
    assert (err <= np.maximum(ABS_TOL, REL_TOL * np.abs(ref))).all(), float(np.nanmax(err))


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
    for step in steps:
        ds = DeviceStep(step)
        ds.run()  # normal entry point with a torch-allocated workspace
        torch.cuda.synchronize()
        ref_bits = ds.out_host().copy()
        got = _static_call(ds)
        _check_against(ref_bits, got)
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
