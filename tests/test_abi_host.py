"""The C ABI library on a machine without a GPU: it builds, loads, exports
every symbol the header declares, and rejects bad arguments on the host
before touching CUDA."""

import ctypes
import os
import re

import pytest

from paged_kv_cache_hkv_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


def header_text():
    with open(HEADER) as f:
        return f.read()


def declared_functions():
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(pkv_\w+)\(", header_text(), re.M)))


def header_define(name):
    m = re.search(rf"#define {name} \(?(-?\w+)\)?", header_text())
    return int(m.group(1).rstrip("u"), 0)


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return binding.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(binding._SIGNATURES)


def test_version_and_status_strings(lib):
    assert lib.pkv_abi_version() == header_define("PKV_ABI_VERSION")
    for code in range(-8, 1):
        assert lib.pkv_status_string(code)


def _layout(nb=8, bs=16, hkv=2, d=64):
    return binding.pkv_cache_layout(nb, bs, hkv, d)


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: checks fail before any use
MISALIGNED = ctypes.c_void_p(0x10008)


def test_write_rejects_bad_arguments(lib):
    ok = header_define("PKV_OK")
    assert ok == 0
    W = lib.pkv_paged_kv_write
    for bs in (4, 24, 64):   # blocks of 8, 16 or 32 tokens only
        assert W(FAKE, FAKE, FAKE, 0, 0, FAKE, 4, _layout(bs=bs), None) == header_define("PKV_ERR_UNSUPPORTED")
    for bs in (8, 32):       # accepted: the next check (a null pointer) decides
        assert W(None, FAKE, FAKE, 0, 0, FAKE, 4, _layout(bs=bs), None) == header_define("PKV_ERR_NULL_POINTER")
    assert W(FAKE, FAKE, FAKE, 0, 0, FAKE, 4, _layout(bs=0), None) == header_define("PKV_ERR_BAD_SHAPE")
    assert W(FAKE, FAKE, FAKE, 0, 0, FAKE, 4, _layout(d=96), None) == header_define("PKV_ERR_UNSUPPORTED")
    assert W(FAKE, FAKE, FAKE, 0, 0, FAKE, -1, _layout(), None) == header_define("PKV_ERR_BAD_SHAPE")
    assert W(FAKE, FAKE, FAKE, 0, 0, FAKE, 4, _layout(nb=0), None) == header_define("PKV_ERR_BAD_SHAPE")
    assert W(None, FAKE, FAKE, 0, 0, FAKE, 4, _layout(), None) == header_define("PKV_ERR_NULL_POINTER")
    assert W(FAKE, MISALIGNED, FAKE, 0, 0, FAKE, 4, _layout(), None) == header_define("PKV_ERR_MISALIGNED")
    assert W(FAKE, FAKE, FAKE, 130, 0, FAKE, 4, _layout(), None) == header_define("PKV_ERR_MISALIGNED")
    assert W(FAKE, FAKE, FAKE, 64, 0, FAKE, 4, _layout(), None) == header_define("PKV_ERR_BAD_SHAPE")
    # nothing to do: OK without touching the device
    assert W(None, None, None, 0, 0, None, 0, _layout(), None) == ok


def _attn(lib, **kw):
    a = dict(out=FAKE, q=FAKE, qs=0, kv=FAKE, bt=FAKE, maxb=8, sl=FAKE, qsl=FAKE, nc=FAKE, R=2,
             T=2, mq=1, ms=100, Hq=4, scale=0.125, lay=_layout(), ws=ctypes.c_void_p(0x10000),
             wsb=1 << 20, opt=None)
    a.update(kw)
    return lib.pkv_paged_attention(a["out"], a["q"], a["qs"], a["kv"], a["bt"], a["maxb"],
                                   a["sl"], a["qsl"], a["nc"], a["R"], a["T"], a["mq"], a["ms"],
                                   a["Hq"], a["scale"], a["lay"], a["ws"], a["wsb"], a["opt"],
                                   None)


def test_attention_rejects_bad_arguments(lib):
    E = header_define
    assert _attn(lib, Hq=3) == E("PKV_ERR_BAD_SHAPE")          # not a multiple of Hkv
    assert _attn(lib, Hq=6) == E("PKV_ERR_UNSUPPORTED")        # group of 3
    assert _attn(lib, lay=_layout(d=80)) == E("PKV_ERR_UNSUPPORTED")
    assert _attn(lib, R=-1) == E("PKV_ERR_BAD_SHAPE")
    assert _attn(lib, ms=200) == E("PKV_ERR_BAD_SHAPE")        # 200 > 8 blocks * 16
    assert _attn(lib, ms=100, lay=_layout(bs=8)) == E("PKV_ERR_BAD_SHAPE")   # 100 > 8 * 8
    assert _attn(lib, ms=200, lay=_layout(bs=32), bt=None) == E("PKV_ERR_NULL_POINTER")  # 200 <= 8 * 32
    assert _attn(lib, lay=_layout(bs=12)) == E("PKV_ERR_UNSUPPORTED")
    # pool rows (block * 2 + k|v) * B must stay below 2^31
    assert _attn(lib, lay=_layout(nb=1 << 25, bs=32)) == E("PKV_ERR_BAD_SHAPE")
    assert _attn(lib, scale=float("nan")) == E("PKV_ERR_BAD_SHAPE")
    assert _attn(lib, scale=-0.5) == E("PKV_ERR_BAD_SHAPE")
    assert _attn(lib, scale=float("inf")) == E("PKV_ERR_BAD_SHAPE")
    assert _attn(lib, qs=100) == E("PKV_ERR_BAD_SHAPE")        # row stride < Hq * D
    assert _attn(lib, bt=None) == E("PKV_ERR_NULL_POINTER")
    assert _attn(lib, q=MISALIGNED) == E("PKV_ERR_MISALIGNED")
    assert _attn(lib, ws=None) == E("PKV_ERR_WORKSPACE")
    assert _attn(lib, ws=ctypes.c_void_p(0x10010)) == E("PKV_ERR_WORKSPACE")
    assert _attn(lib, R=0) == E("PKV_OK")                      # empty batch
    opt = binding.pkv_attention_options()
    opt.reserved[3] = 1
    assert _attn(lib, opt=ctypes.pointer(opt)) < 0


def test_slot_mapping_and_errors_reject_bad_arguments(lib):
    E = header_define
    S = lib.pkv_slot_mapping
    assert S(FAKE, FAKE, 4, FAKE, FAKE, 2, 3, 10, 12, None) == E("PKV_ERR_UNSUPPORTED")
    assert S(FAKE, FAKE, 4, FAKE, FAKE, 2, 3, 10, 0, None) == E("PKV_ERR_BAD_SHAPE")
    for bs in (8, 32):
        assert S(None, FAKE, 4, FAKE, FAKE, 2, 3, 10, bs, None) == E("PKV_ERR_NULL_POINTER")
    assert S(FAKE, FAKE, 4, FAKE, FAKE, 2, -3, 10, 16, None) == E("PKV_ERR_BAD_SHAPE")
    assert S(None, FAKE, 4, FAKE, FAKE, 2, 3, 10, 16, None) == E("PKV_ERR_NULL_POINTER")
    assert S(None, None, 4, None, None, 2, 0, 10, 16, None) == E("PKV_OK")
    assert lib.pkv_get_device_errors(None, 0, None) == E("PKV_ERR_NULL_POINTER")


def test_slot_mapping_and_write_rejects_bad_arguments(lib):
    E = header_define

    def SW(**kw):
        a = dict(kv=FAKE, k=FAKE, v=FAKE, ks=0, vs=0, slots=FAKE, bt=FAKE, maxb=8, qsl=FAKE,
                 nc=FAKE, R=2, T=4, lay=_layout())
        a.update(kw)
        return lib.pkv_slot_mapping_and_write(a["kv"], a["k"], a["v"], a["ks"], a["vs"],
                                              a["slots"], a["bt"], a["maxb"], a["qsl"], a["nc"],
                                              a["R"], a["T"], a["lay"], None)

    assert SW(lay=_layout(bs=12)) == E("PKV_ERR_UNSUPPORTED")
    assert SW(lay=_layout(bs=0)) == E("PKV_ERR_BAD_SHAPE")
    assert SW(lay=_layout(d=96)) == E("PKV_ERR_UNSUPPORTED")
    assert SW(lay=_layout(nb=0)) == E("PKV_ERR_BAD_SHAPE")
    assert SW(T=-1) == E("PKV_ERR_BAD_SHAPE")
    assert SW(R=-1) == E("PKV_ERR_BAD_SHAPE")
    assert SW(maxb=-1) == E("PKV_ERR_BAD_SHAPE")
    assert SW(ks=64) == E("PKV_ERR_BAD_SHAPE")       # row stride < Hkv * D = 128
    assert SW(vs=130) == E("PKV_ERR_MISALIGNED")     # not a whole number of 16-byte words
    assert SW(kv=None) == E("PKV_ERR_NULL_POINTER")
    assert SW(qsl=None) == E("PKV_ERR_NULL_POINTER")
    assert SW(bt=None) == E("PKV_ERR_NULL_POINTER")
    assert SW(nc=None) == E("PKV_ERR_NULL_POINTER")
    assert SW(k=MISALIGNED) == E("PKV_ERR_MISALIGNED")
    assert SW(kv=MISALIGNED) == E("PKV_ERR_MISALIGNED")
    # nothing to write: OK without touching the device
    assert SW(kv=None, k=None, v=None, slots=None, bt=None, qsl=None, nc=None, T=0) == E("PKV_OK")


def test_attention_with_write_rejects_bad_arguments(lib):
    E = header_define

    def AW(**kw):
        a = dict(out=FAKE, q=FAKE, qs=0, kv=FAKE, k=FAKE, v=FAKE, ks=0, vs=0, slots=FAKE, bt=FAKE,
                 maxb=8, sl=FAKE, qsl=FAKE, nc=FAKE, R=2, T=2, mq=1, ms=100, Hq=4, scale=0.125,
                 lay=_layout(), ws=ctypes.c_void_p(0x10000), wsb=1 << 20, opt=None)
        a.update(kw)
        return lib.pkv_paged_attention_with_write(
            a["out"], a["q"], a["qs"], a["kv"], a["k"], a["v"], a["ks"], a["vs"], a["slots"],
            a["bt"], a["maxb"], a["sl"], a["qsl"], a["nc"], a["R"], a["T"], a["mq"], a["ms"],
            a["Hq"], a["scale"], a["lay"], a["ws"], a["wsb"], a["opt"], None)

    # the write's arguments
    assert AW(lay=_layout(bs=12)) == E("PKV_ERR_UNSUPPORTED")
    assert AW(T=-1) == E("PKV_ERR_BAD_SHAPE")
    assert AW(ks=64) == E("PKV_ERR_BAD_SHAPE")
    assert AW(ks=130) == E("PKV_ERR_MISALIGNED")
    assert AW(k=None) == E("PKV_ERR_NULL_POINTER")
    assert AW(v=MISALIGNED) == E("PKV_ERR_MISALIGNED")
    assert AW(nc=None) == E("PKV_ERR_NULL_POINTER")
    # then the attention's: nothing is launched when either part is bad
    assert AW(Hq=3) == E("PKV_ERR_BAD_SHAPE")
    assert AW(Hq=6) == E("PKV_ERR_UNSUPPORTED")
    assert AW(scale=float("nan")) == E("PKV_ERR_BAD_SHAPE")
    assert AW(ms=200) == E("PKV_ERR_BAD_SHAPE")
    assert AW(qs=100) == E("PKV_ERR_BAD_SHAPE")
    assert AW(sl=None) == E("PKV_ERR_NULL_POINTER")
    assert AW(out=MISALIGNED) == E("PKV_ERR_MISALIGNED")
    assert AW(ws=None) == E("PKV_ERR_WORKSPACE")
    assert AW(ws=ctypes.c_void_p(0x10010)) == E("PKV_ERR_WORKSPACE")
    # no tokens and no requests: OK without touching the device
    none = dict(out=None, q=None, kv=None, k=None, v=None, slots=None, bt=None, sl=None, qsl=None,
                nc=None, ws=None)
    assert AW(R=0, T=0, **none) == E("PKV_OK")


def test_copy_blocks_rejects_bad_arguments(lib):
    E = header_define
    C = lib.pkv_copy_blocks
    assert C(FAKE, 4, FAKE, 4, FAKE, 2, _layout(bs=48), None) == E("PKV_ERR_UNSUPPORTED")
    assert C(FAKE, 4, None, 4, FAKE, 2, _layout(bs=8), None) == E("PKV_ERR_NULL_POINTER")
    assert C(FAKE, 0, FAKE, 4, FAKE, 2, _layout(), None) == E("PKV_ERR_BAD_SHAPE")
    assert C(FAKE, 4, FAKE, 4, FAKE, -1, _layout(), None) == E("PKV_ERR_BAD_SHAPE")
    assert C(FAKE, 4, None, 4, FAKE, 2, _layout(), None) == E("PKV_ERR_NULL_POINTER")
    assert C(FAKE, 4, MISALIGNED, 4, FAKE, 2, _layout(), None) == E("PKV_ERR_MISALIGNED")
    assert C(None, 4, None, 4, None, 0, _layout(), None) == E("PKV_OK")


def test_no_gpu_means_an_error_not_a_fallback(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    n = lib.pkv_attention_workspace_size(4, 4, _layout(), None)
    assert n < 0
    assert _attn(lib) < 0  # valid arguments, but no sm_103 device to run on
