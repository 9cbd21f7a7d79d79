"""The C-ABI library builds, loads without a GPU, exports every entry point that
include/inkling.h declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "inkling.h")


@pytest.fixture(scope="module")
def lib():
    from relative_position_gqa_gb300 import build, _lib
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(inkling_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("inkling_sconv_kv", "inkling_rel_attn_prefill", "inkling_rel_attn_decode",
              "inkling_rel_attn_decode_workspace_size", "inkling_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from relative_position_gqa_gb300 import _lib
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    from relative_position_gqa_gb300 import _lib
    assert _lib.status_string(0) == "ok"
    assert "page" in _lib.status_string(5)
    assert _lib.status_string(12345) == "unknown status"


FAKE = 0x10000  # a 16-byte aligned non-null value: the checks below fail before any use


def _prefill(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, maxb=4, cu=FAKE, sl=FAKE, bias=FAKE, R=64,
             scale=0.1, window=0, out=FAKE, odt=0, lse=None, B=1, T=10, Hq=4, Hkv=2, nb=4,
             mq=10, st=None, stream=None)
    a.update(over)
    return lib.inkling_rel_attn_prefill(*a.values())


@pytest.mark.parametrize("over", [dict(window=-1), dict(Hq=5), dict(R=0), dict(odt=3),
                                  dict(q=None), dict(out=FAKE + 2), dict(B=-1), dict(nb=0)])
def test_prefill_host_checks(lib, over):
    assert _prefill(lib, **over) == 1


def _decode(lib, **over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, maxb=4, cu=FAKE, sl=FAKE, bias=FAKE, R=64,
             scale=0.1, window=0, out=FAKE, odt=0, lse=None, B=1, T=10, Hq=8, Hkv=1, nb=4,
             mq=9, msl=500, ns=2, ws=None, wsb=0, st=None, stream=None)
    a.update(over)
    return lib.inkling_rel_attn_decode(*a.values())


def test_decode_host_checks(lib):
    assert _decode(lib, mq=10) == 1              # more than 9 tokens
    assert _decode(lib, Hq=32, Hkv=1) == 2       # G = 32: packed rows exceed one tile
    assert _decode(lib, ns=-1) == 1
    assert _decode(lib, ws=None, wsb=0) == 7     # two splits need a workspace


def _decode_sconv(lib, **over):
    a = dict(q=FAKE, kr=FAKE, vr=FAKE, wk=FAKE, wv=FAKE, state=FAKE, k=FAKE, v=FAKE, bt=FAKE,
             maxb=4, cu=FAKE, sl=FAKE, bias=FAKE, R=64, scale=0.1, window=0, out=FAKE, odt=0,
             lse=None, B=1, T=10, Hq=8, Hkv=1, nb=4, mq=9, msl=500, ns=2, ws=None, wsb=0,
             st=None, stream=None)
    a.update(over)
    return lib.inkling_rel_attn_decode_sconv(*a.values())


def test_decode_sconv_host_checks(lib):
    assert _decode_sconv(lib, kr=None) == 1          # the conv's inputs are required
    assert _decode_sconv(lib, state=FAKE + 8) == 1   # and 16-byte aligned
    assert _decode_sconv(lib, mq=10) == 1            # the decode's own checks follow
    assert _decode_sconv(lib, Hq=32, Hkv=1) == 2
    assert _decode_sconv(lib, ws=None, wsb=0) == 7


def test_sconv_host_checks(lib):
    f = lib.inkling_sconv_kv
    assert f(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, 4, 4, None, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 0, 4, 4, None, None) == 1
    assert f(FAKE + 8, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, 4, 4, None, None) == 1
    # nothing to do is not an error
    assert f(None, None, None, None, None, None, None, None, None, 0, 0, 1, 4, 0, None, None) == 0


def test_workspace_size_rule(lib):
    ws = lib.inkling_rel_attn_decode_workspace_size
    assert ws(1, 8, 1, 9, 100000, 0, 1) == 0
    two = ws(1, 8, 1, 9, 100000, 0, 2)
    assert two >= 2 * 72 * 130 * 4
    assert ws(1, 8, 1, 9, 100000, 0, 8) > two


def test_decode_plan_rule(lib):
    """The plan query follows the split rule: 8 pages in 3 splits are ranges of 3 pages
    (3 + 3 + 2), 6 CTAs for 2 sequences; one split needs no merge."""
    from relative_position_gqa_gb300 import _lib
    assert _lib.decode_plan(2, 8, 1, 9, 1000, 0, 3) == [3, 6, 3, 1]
    assert _lib.decode_plan(2, 8, 1, 9, 1000, 0, 1) == [1, 2, 8, 0]
    # a 300-token window bounds the visible range to (300 + 8 + 127) // 128 + 1 = 4 pages
    assert _lib.decode_plan(64, 32, 4, 9, 131072, 300, 2) == [2, 512, 2, 1]
    for bad in (dict(mq=10), dict(ns=-1), dict(B=0)):
        a = dict(B=2, Hq=8, Hkv=1, mq=9, msl=1000, w=0, ns=3)
        a.update(bad)
        with pytest.raises(_lib.InklingError) as e:
            _lib.decode_plan(*a.values())
        assert e.value.code == 1


def test_dense_sconv_host_checks(lib):
    f = lib.inkling_sconv
    ok = dict(x=FAKE, w=FAKE, st=FAKE, cu=FAKE, y=FAKE + 4096, B=1, T=4, C=64, mq=4, ds=None, s=None)

    def call(**over):
        a = dict(ok)
        a.update(over)
        return f(*a.values())
    assert call(C=12) == 1            # not a multiple of 8 channels
    assert call(C=0) == 1
    assert call(y=FAKE) == 1          # output aliases the input
    assert call(x=FAKE + 8) == 1      # misaligned
    assert call(w=None) == 1
    assert call(B=0, T=0, x=None, w=None, st=None, cu=None, y=None) == 0


def test_rollback_host_checks(lib):
    f = lib.inkling_sconv_state_rollback
    ok = dict(sb=FAKE, x0=FAKE, x1=FAKE, cu=FAKE, acc=FAKE, sa=FAKE, B=2, T=18, C=256, streams=2,
              ds=None, s=None)

    def call(**over):
        a = dict(ok)
        a.update(over)
        return f(*a.values())
    assert call(streams=3) == 1
    assert call(streams=2, x1=None) == 1  # the K/V pair needs both raw streams
    assert call(acc=None) == 1
    assert call(sa=FAKE + 2) == 1
    assert call(C=4) == 1
    assert call(B=0) == 0


def _step(lib, name, **over):
    cu = (ctypes.c_int32 * 3)(0, 5, 10)  # the host copy of cu_q_lens is read by the checks
    a = dict(qh=FAKE, kh=FAKE, vh=FAKE, oh=FAKE, qd=FAKE, kd=FAKE, vd=FAKE, od=FAKE,
             cu_h=ctypes.cast(cu, ctypes.c_void_p), wk=FAKE, wv=FAKE, st=FAKE, cu=FAKE,
             slot=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, maxb=4, sl=FAKE, bias=FAKE, R=64, scale=0.1,
             window=0, odt=0, lse=None, B=2, T=10, Hq=4, Hkv=2, nb=4, mq=5)
    if name == "inkling_decode_step_host":
        a.update(msl=500, ns=0, ws=None, wsb=0, chunks=2)
    else:
        a.update(chunks=2, scratch=None)
    a.update(ds=None, s=None, up=0x20000, down=0x30000)
    a.update(over)
    rc = getattr(lib, name)(*a.values())
    del cu
    return rc


@pytest.mark.parametrize("name", ["inkling_prefill_step_host", "inkling_decode_step_host"])
@pytest.mark.parametrize("over", [dict(chunks=0), dict(up=0x30000), dict(down=None),
                                  dict(qh=None), dict(od=None), dict(odt=3), dict(mq=4),
                                  dict(T=11), dict(Hq=5), dict(wk=None), dict(B=-1)])
def test_step_host_checks(lib, name, over):
    """Host-buffer steps reject bad arguments before enqueueing anything: missing buffers,
    chunks < 1, copy streams that coincide, lengths that disagree with cu_q_lens_host."""
    assert _step(lib, name, **over) == 1


def _step_fp8(lib, name, **over):
    cu = (ctypes.c_int32 * 3)(0, 5, 10)
    a = dict(qh=FAKE, kh=FAKE, vh=FAKE, oh=FAKE, qd=FAKE, kd=FAKE, vd=FAKE, od=FAKE,
             cu_h=ctypes.cast(cu, ctypes.c_void_p), wk=FAKE, wv=FAKE, st=FAKE, cu=FAKE,
             slot=FAKE, kc=FAKE, vc=FAKE, ks=0.5, vs=0.25, bt=FAKE, maxb=4, sl=FAKE, bias=FAKE,
             R=64, scale=0.1, window=0, odt=0, lse=None, B=2, T=10, Hq=4, Hkv=2, nb=4, mq=5,
             msl=500)
    if name == "inkling_decode_step_host_fp8":
        a.update(ns=0, ws=None, wsb=0, chunks=2)
    else:
        a.update(ws=None, wsb=0, chunks=2, scratch=None)
    a.update(ds=None, s=None, up=0x20000, down=0x30000)
    a.update(over)
    rc = getattr(lib, name)(*a.values())
    del cu
    return rc


@pytest.mark.parametrize("name", ["inkling_prefill_step_host_fp8", "inkling_decode_step_host_fp8"])
@pytest.mark.parametrize("over", [dict(chunks=0), dict(up=0x30000), dict(qh=None), dict(odt=3),
                                  dict(mq=4), dict(T=11), dict(wk=None), dict(ks=0.0),
                                  dict(vs=float("inf")), dict(ks=-1.0), dict(msl=-1)])
def test_step_host_fp8_checks(lib, name, over):
    """The FP8 step forms reject what the bf16 forms reject, and scales that are not
    positive and finite, before enqueueing anything."""
    assert _step_fp8(lib, name, **over) == 1


def test_prefill_step_host_fp8_needs_workspace(lib):
    """The whole step's widening workspace is checked before any group is enqueued."""
    need = lib.inkling_rel_attn_prefill_fp8_workspace_size(2, 2, 4, 5, 500, 0)
    assert need > 0
    assert _step_fp8(lib, "inkling_prefill_step_host_fp8") == 7          # INKLING_ERR_WORKSPACE
    assert _step_fp8(lib, "inkling_prefill_step_host_fp8", ws=FAKE, wsb=need - 16) == 7


def test_decode_step_host_checks(lib):
    assert _step(lib, "inkling_decode_step_host", mq=10) == 1   # more than 9 tokens
    assert _step(lib, "inkling_decode_step_host", ns=-1) == 1


def test_prefill_fp8_host_checks(lib):
    ws = lib.inkling_rel_attn_prefill_fp8_workspace_size
    one = ws(1, 2, 4, 100, 500, 0)
    assert one >= 2 * 4 * 2 * 128 * 128 * 2          # four visible pages of K and V, 2 heads
    assert ws(1, 2, 4, 100, 500, 100) < one          # a window bounds the visible pages
    f = lib.inkling_rel_attn_prefill_fp8
    ok = dict(q=FAKE, k=FAKE, v=FAKE, ks=0.5, vs=0.5, bt=FAKE, maxb=4, cu=FAKE, sl=FAKE,
              bias=FAKE, R=64, scale=0.1, window=0, out=FAKE, odt=0, lse=None, B=1, T=10, Hq=4,
              Hkv=2, nb=4, mq=10, msl=500, ws=None, wsb=0, st=None, stream=None)

    def call(**over):
        a = dict(ok)
        a.update(over)
        return f(*a.values())
    assert call(ks=0.0) == 1
    assert call(vs=float("inf")) == 1
    assert call(Hq=5) == 1
    assert call() == 7                                # no workspace
    assert call(ws=FAKE, wsb=16) == 7


def test_selftest_host_checks(lib):
    f = lib.inkling_selftest_bounded_wait
    assert f(2, 1, FAKE, FAKE, None) == 1
    assert f(0, 0, FAKE, FAKE, None) == 1
    assert f(0, 1, None, FAKE, None) == 1
