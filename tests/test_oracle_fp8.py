"""Pins for the oracle's FP8 KV cache: the E4M3 codec, the conv written as E4M3 codes, and
attention over an E4M3 cache (vLLM Day-0 Inkling blog, "Roadmap": FP8 for the global-attention
layers).  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_golden():
    n = 0
    for line in open(os.path.join(GOLDEN, "e4m3.txt")):
        if line.startswith("#") or not line.strip():
            continue
        val, want = line.split()[:2]
        assert oracle.e4m3_round(float.fromhex(val)) == int(want, 16), line
        n += 1
    assert n >= 20


def test_e4m3_decode_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.uint8)
    want = codes.view(torch.float8_e4m3fn).float().tolist()
    for c, w in zip(range(256), want):
        got = oracle.e4m3_to_float(c)
        assert (math.isnan(got) and math.isnan(w)) or got == w, (hex(c), got, w)


def test_e4m3_round_trips_every_finite_code():
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        assert oracle.e4m3_round(oracle.e4m3_to_float(c)) == c


def test_e4m3_round_matches_torch_in_range():
    """torch's float32 -> float8_e4m3fn conversion rounds to nearest even; on binary32
    inputs inside the finite range the oracle must agree bit for bit."""
    g = torch.Generator().manual_seed(3)
    x = torch.randn(20000, generator=g) * torch.exp2(torch.randint(-12, 9, (20000,), generator=g).float())
    x = x[x.abs() < 448]
    want = x.to(torch.float8_e4m3fn).view(torch.uint8).tolist()
    got = [oracle.e4m3_round(v) for v in x.tolist()]
    assert got == want


def test_e4m3_round_is_nearest():
    """For random doubles, the chosen code is at least as near as both neighbours."""
    g = np.random.default_rng(4)
    for y in g.standard_normal(3000) * 50:
        c = oracle.e4m3_round(y)
        v = oracle.e4m3_to_float(c)
        if abs(y) >= 448:
            assert abs(v) == 448
            continue
        for nb in (c - 1, c + 1):
            if 0 <= (nb & 0x7F) <= 0x7E and (nb & 0x80) == (c & 0x80):
                assert abs(v - y) <= abs(oracle.e4m3_to_float(nb) - y)


def _fp8_case(q_lens=(7, 2, 19), hkv=2, seed=71):
    spec = W.small(q_lens=q_lens, seq_lens=[n + 5 for n in q_lens], hq=2 * hkv, hkv=hkv,
                   history_random=True, state_random=True)
    return W.make_case(spec, seed=seed)


def _u8_cache_like(c):
    return torch.zeros(c.k_cache.shape, dtype=torch.uint8)


@pytest.mark.parametrize("scale", [1.0, 0.25, 3.0])
def test_fp8_conv_one_hot_taps_store_the_rounded_raw_row(scale):
    """With the current-row tap 1 and the others 0, each code is e4m3(x / scale) of the
    raw bf16 value (exact conv sum), so the cache is the codec applied to the raw rows."""
    c = _fp8_case()
    C = c.spec.channels
    w = torch.tensor([0, 0, 0, 1], dtype=torch.float32).repeat(C, 1)
    kc, vc = _u8_cache_like(c), _u8_cache_like(c)
    oracle.sconv_kv_fp8(c.k_raw, c.v_raw, w, w, c.state.clone(), c.cu_q_lens, c.slot_mapping,
                        kc, vc, scale, scale)
    slots = c.slot_mapping
    got = kc[slots // 128, :, slots % 128, :].reshape(len(slots), -1)
    want = torch.tensor([[oracle.e4m3_round(v / scale) for v in row]
                         for row in c.k_raw.double().tolist()], dtype=torch.uint8)
    assert torch.equal(got, want)


def test_fp8_conv_state_equals_bf16_conv_state():
    c = _fp8_case(seed=72)
    st8, st16 = c.state.clone(), c.state.clone()
    oracle.sconv_kv_fp8(c.k_raw, c.v_raw, c.w_k, c.w_v, st8, c.cu_q_lens, c.slot_mapping,
                        _u8_cache_like(c), _u8_cache_like(c), 0.5, 2.0)
    oracle.sconv_kv(c.k_raw, c.v_raw, c.w_k, c.w_v, st16, c.cu_q_lens, c.slot_mapping,
                    c.k_cache.clone(), c.v_cache.clone())
    assert torch.equal(st8.view(torch.int16), st16.view(torch.int16))


def test_fp8_conv_exact_when_sums_are_representable():
    """Small integers, dyadic taps and a power-of-two scale: every y / scale is exactly an
    E4M3 value, so the stored code decodes to the brute-force sum."""
    c = _fp8_case(seed=73)
    g = torch.Generator().manual_seed(8)
    c.k_raw = torch.randint(-2, 3, c.k_raw.shape, generator=g).to(torch.bfloat16)
    c.v_raw = torch.randint(-2, 3, c.v_raw.shape, generator=g).to(torch.bfloat16)
    c.state = torch.randint(-2, 3, c.state.shape, generator=g).to(torch.bfloat16)
    C = c.spec.channels
    choices = torch.tensor([-1.0, -0.5, 0.0, 0.5, 1.0])
    w = choices[torch.randint(0, 5, (C, 4), generator=g)]
    kc, vc = _u8_cache_like(c), _u8_cache_like(c)
    oracle.sconv_kv_fp8(c.k_raw, c.v_raw, w, w, c.state.clone(), c.cu_q_lens, c.slot_mapping,
                        kc, vc, 0.5, 0.5)
    cu = c.cu_q_lens.tolist()
    for b in range(c.spec.batch):
        ext = torch.cat([c.state[b, 0].float(), c.k_raw[cu[b]:cu[b + 1]].float()])
        n = cu[b + 1] - cu[b]
        y = sum(w[:, j] * ext[j:j + n] for j in range(4))  # |y| <= 8: exact in fp32
        slots = c.slot_mapping[cu[b]:cu[b + 1]]
        got = kc[slots // 128, :, slots % 128, :].reshape(n, -1)
        dec = torch.tensor([[oracle.e4m3_to_float(v) for v in row] for row in got.tolist()])
        assert torch.equal(dec * 0.5, y)


def test_fp8_attention_equals_bf16_attention_on_representable_caches():
    """An E4M3 code times a power-of-two scale has at most 4 significant bits, so it is
    exact in bf16: the FP8 attention must equal the bf16 attention over the decoded
    cache, bit for bit (same fp64 arithmetic)."""
    spec = W.small(q_lens=(9, 3), seq_lens=(300, 140), hq=8, hkv=2, window=0, r=64,
                   history_random=True, state_random=True)
    c = W.make_case(spec, seed=74)
    g = torch.Generator().manual_seed(9)
    k8 = torch.randint(0, 256, c.k_cache.shape, generator=g, dtype=torch.int32).to(torch.uint8)
    v8 = torch.randint(0, 256, c.v_cache.shape, generator=g, dtype=torch.int32).to(torch.uint8)
    k8[(k8 & 0x7F) == 0x7F] = 0x30  # no NaN codes
    v8[(v8 & 0x7F) == 0x7F] = 0x30
    ks, vs = 0.25, 2.0
    kb = (k8.view(torch.float8_e4m3fn).float() * ks).to(torch.bfloat16)
    vb = (v8.view(torch.float8_e4m3fn).float() * vs).to(torch.bfloat16)
    assert torch.equal(kb.float(), k8.view(torch.float8_e4m3fn).float() * ks)
    for window in (0, 100):
        o8, l8 = oracle.rel_attn_fp8(c.q, k8, v8, ks, vs, c.block_table, c.cu_q_lens, c.seq_lens,
                                     c.bias, scale=spec.scale, window=window)
        o16, l16 = oracle.rel_attn(c.q, kb, vb, c.block_table, c.cu_q_lens, c.seq_lens, c.bias,
                                   scale=spec.scale, window=window)
        assert np.array_equal(o8, o16) and np.array_equal(l8, l16)
