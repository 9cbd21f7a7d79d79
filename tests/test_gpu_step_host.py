"""GPU: the host-buffer step entry points (inkling_prefill_step_host /
inkling_decode_step_host) launch the same kernels as the separate calls, one group of
sequences at a time, so their outputs, caches and sconv states are bit-identical to
sconv_kv followed by the attention call on device buffers, for any number of groups."""
import pytest
import torch

import workloads as W
from harness import gpu_attn, gpu_sconv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ink():
    import relative_position_gqa_gb300 as m
    m._lib.load()
    return m


def _host_step(ink, g, *, decode, out_dtype, chunks, num_splits=0):
    spec = g.spec
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    host = [t.cpu().pin_memory() for t in (g.q, g.k_raw, g.v_raw)]
    out_h = torch.full((spec.total_q, spec.hq, 128), float("nan"), dtype=out_dtype).pin_memory()
    staging = (torch.empty_like(g.q), torch.empty_like(g.k_raw), torch.empty_like(g.v_raw),
               torch.empty(out_h.shape, dtype=out_dtype, device="cuda"))
    lse = torch.full((spec.total_q, spec.hq), float("nan"), dtype=torch.float32, device="cuda")
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    args = (host[0], host[1], host[2], out_h, staging, g.cu_q_lens.cpu(), g.w_k, g.w_v, g.state,
            g.cu_q_lens, g.slot_mapping, g.k_cache, g.v_cache, g.block_table, g.seq_lens, g.bias)
    if decode:
        ink.decode_step_host(*args, scale=spec.scale, window=spec.window,
                             max_q_len=spec.max_q_len, max_seq_len=spec.max_seq_len,
                             num_splits=num_splits, h2d_stream=up, d2h_stream=down,
                             chunks=chunks, lse=lse, dev_status=st)
    else:
        ink.prefill_step_host(*args, scale=spec.scale, window=spec.window,
                              max_q_len=spec.max_q_len, h2d_stream=up, d2h_stream=down,
                              chunks=chunks, lse=lse, dev_status=st)
    torch.cuda.current_stream().synchronize()
    assert int(st.item()) == 0, ink.status_string(int(st.item()))
    return out_h, lse


def _device_step(ink, g, *, decode, out_dtype, num_splits=0):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_sconv(ink, g, st)
    out, lse = gpu_attn(ink, g, st, decode=decode, out_dtype=out_dtype, num_splits=num_splits)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, ink.status_string(int(st.item()))
    return out.cpu(), lse


PREFILL = W.small(q_lens=(150, 37, 0, 300, 9), seq_lens=(150, 200, 40, 300, 600), hq=4, hkv=2,
                  r=64, window=100)
DECODE = W.small(q_lens=(9, 9, 3, 1), seq_lens=(500, 700, 129, 1000), hq=8, hkv=1, r=64)


@pytest.mark.parametrize("chunks", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_prefill_step_host_bit_identical(ink, chunks, out_dtype):
    """With 3, 8 or 16 groups the 150- and 300-token sequences are cut into pieces of whole
    query tiles (chunked prefills of one sequence; 16 asks for more pieces than the query
    tiles allow); the bits must not change."""
    a = W.make_case(PREFILL, seed=5, device="cuda")
    b = W.make_case(PREFILL, seed=5, device="cuda")
    ref, ref_lse = _device_step(ink, a, decode=False, out_dtype=out_dtype)
    got, got_lse = _host_step(ink, b, decode=False, out_dtype=out_dtype, chunks=chunks)
    assert torch.equal(got.view(torch.uint8), ref.view(torch.uint8))
    assert torch.equal(got_lse.view(torch.int32), ref_lse.view(torch.int32))
    assert torch.equal(b.k_cache, a.k_cache) and torch.equal(b.v_cache, a.v_cache)
    assert torch.equal(b.state, a.state)


@pytest.mark.parametrize("chunks", [1, 2, 4])
def test_decode_step_host_bit_identical(ink, chunks):
    a = W.make_case(DECODE, seed=6, device="cuda")
    b = W.make_case(DECODE, seed=6, device="cuda")
    ref, ref_lse = _device_step(ink, a, decode=True, out_dtype=torch.float32, num_splits=2)
    got, got_lse = _host_step(ink, b, decode=True, out_dtype=torch.float32, chunks=chunks,
                              num_splits=2)
    assert torch.equal(got.view(torch.uint8), ref.view(torch.uint8))
    assert torch.equal(got_lse.view(torch.int32), ref_lse.view(torch.int32))
    assert torch.equal(b.state, a.state)


K_SCALE, V_SCALE = 0.0625, 0.03125


def _fp8_case(spec, seed):
    g = W.make_case(spec, seed=seed, device="cuda")
    g.k_cache = W.fp8_history(g.k_cache, K_SCALE)
    g.v_cache = W.fp8_history(g.v_cache, V_SCALE)
    return g


def _device_step_fp8(ink, g, *, decode, out_dtype, num_splits=0):
    spec = g.spec
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ink.sconv_kv_fp8(g.k_raw, g.v_raw, g.w_k, g.w_v, g.state, g.cu_q_lens, g.slot_mapping,
                     g.k_cache, g.v_cache, k_scale=K_SCALE, v_scale=V_SCALE,
                     max_q_len=spec.max_q_len, dev_status=st)
    out = torch.empty(spec.total_q, spec.hq, 128, dtype=out_dtype, device="cuda")
    lse = torch.empty(spec.total_q, spec.hq, dtype=torch.float32, device="cuda")
    kw = dict(k_scale=K_SCALE, v_scale=V_SCALE, scale=spec.scale, window=spec.window,
              max_q_len=spec.max_q_len, max_seq_len=spec.max_seq_len, out=out, lse=lse,
              dev_status=st)
    args = (g.q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens, g.seq_lens, g.bias)
    if decode:
        ink.rel_attn_decode_fp8(*args, num_splits=num_splits, **kw)
    else:
        ink.rel_attn_prefill_fp8(*args, **kw)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, ink.status_string(int(st.item()))
    return out.cpu(), lse


def _host_step_fp8(ink, g, *, decode, out_dtype, chunks, num_splits=0):
    spec = g.spec
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    host = [t.cpu().pin_memory() for t in (g.q, g.k_raw, g.v_raw)]
    out_h = torch.full((spec.total_q, spec.hq, 128), float("nan"), dtype=out_dtype).pin_memory()
    staging = (torch.empty_like(g.q), torch.empty_like(g.k_raw), torch.empty_like(g.v_raw),
               torch.empty(out_h.shape, dtype=out_dtype, device="cuda"))
    lse = torch.full((spec.total_q, spec.hq), float("nan"), dtype=torch.float32, device="cuda")
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    args = (host[0], host[1], host[2], out_h, staging, g.cu_q_lens.cpu(), g.w_k, g.w_v, g.state,
            g.cu_q_lens, g.slot_mapping, g.k_cache, g.v_cache, g.block_table, g.seq_lens, g.bias)
    kw = dict(k_scale=K_SCALE, v_scale=V_SCALE, scale=spec.scale, window=spec.window,
              max_q_len=spec.max_q_len, max_seq_len=spec.max_seq_len, h2d_stream=up,
              d2h_stream=down, chunks=chunks, lse=lse, dev_status=st)
    if decode:
        ink.decode_step_host_fp8(*args, num_splits=num_splits, **kw)
    else:
        ink.prefill_step_host_fp8(*args, **kw)
    torch.cuda.current_stream().synchronize()
    assert int(st.item()) == 0, ink.status_string(int(st.item()))
    return out_h, lse


@pytest.mark.parametrize("chunks", [1, 3, 8])
def test_prefill_step_host_fp8_bit_identical(ink, chunks):
    """E4M3 caches: the groups (and the pieces of whole query tiles that 3 and 8 groups cut
    the long sequences into) reuse one widening workspace; outputs, codes and states are
    those of sconv_kv_fp8 followed by rel_attn_prefill_fp8."""
    a = _fp8_case(PREFILL, seed=7)
    b = _fp8_case(PREFILL, seed=7)
    ref, ref_lse = _device_step_fp8(ink, a, decode=False, out_dtype=torch.bfloat16)
    got, got_lse = _host_step_fp8(ink, b, decode=False, out_dtype=torch.bfloat16, chunks=chunks)
    assert torch.equal(got.view(torch.uint8), ref.view(torch.uint8))
    assert torch.equal(got_lse.view(torch.int32), ref_lse.view(torch.int32))
    assert torch.equal(b.k_cache, a.k_cache) and torch.equal(b.v_cache, a.v_cache)
    assert torch.equal(b.state, a.state)


@pytest.mark.parametrize("chunks", [1, 2, 4])
def test_decode_step_host_fp8_bit_identical(ink, chunks):
    a = _fp8_case(DECODE, seed=8)
    b = _fp8_case(DECODE, seed=8)
    ref, ref_lse = _device_step_fp8(ink, a, decode=True, out_dtype=torch.float32, num_splits=2)
    got, got_lse = _host_step_fp8(ink, b, decode=True, out_dtype=torch.float32, chunks=chunks,
                                  num_splits=2)
    assert torch.equal(got.view(torch.uint8), ref.view(torch.uint8))
    assert torch.equal(got_lse.view(torch.int32), ref_lse.view(torch.int32))
    assert torch.equal(b.k_cache, a.k_cache) and torch.equal(b.v_cache, a.v_cache)
    assert torch.equal(b.state, a.state)
