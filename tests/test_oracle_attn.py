"""Pins for the oracle's relative-bias GQA attention (vLLM Day-0 Inkling blog, "Model
Architecture / Attention": GQA with head size 128, full and sliding-window layers, a
learned relative-position term on the pre-softmax logits; "Model Architecture / MTP": up
to 9 query tokens per decode step).  CPU only.

Each pin comes from outside the oracle: a pure-Python brute force over logical keys,
torch's own scaled_dot_product_attention in float64 with an explicit additive mask,
closed forms, and invariants of softmax (shift invariance, one-key rows)."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import brute
import workloads as W


def _logical_kv(case):
    """Per sequence: K, V as [L, Hkv, 128] float64, gathered with torch indexing."""
    out = []
    for b in range(case.spec.batch):
        L = int(case.seq_lens[b])
        pos = torch.arange(L)
        blk = case.block_table[b].long()[pos // 128]
        k = case.k_cache[blk, :, pos % 128, :].double()
        v = case.v_cache[blk, :, pos % 128, :].double()
        out.append((k, v))
    return out


def _sdpa_reference(case, bias=None):
    """torch SDPA (float64, CPU) with a dense additive mask built from the table."""
    spec = case.spec
    bias = case.bias if bias is None else bias
    G = spec.group
    cu = case.cu_q_lens.tolist()
    outs, lses = [], []
    for b, (k, v) in enumerate(_logical_kv(case)):
        n, L = cu[b + 1] - cu[b], int(case.seq_lens[b])
        q = case.q[cu[b]:cu[b + 1]].double()                  # [n, Hq, D]
        pq = torch.arange(L - n, L)[:, None]
        pk = torch.arange(L)[None, :]
        dist = pq - pk
        allowed = dist >= 0
        if spec.window:
            allowed &= dist <= spec.window - 1
        bidx = dist.clamp(0, spec.r - 1)
        add = bias.double()[:, bidx]                          # [Hq, n, L]
        add = add.masked_fill(~allowed, float("-inf"))
        kk = k.repeat_interleave(G, dim=1).permute(1, 0, 2)  # [Hq, L, D]
        vv = v.repeat_interleave(G, dim=1).permute(1, 0, 2)
        qq = q.permute(1, 0, 2)                               # [Hq, n, D]
        o = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=add, scale=spec.scale)
        logits = spec.scale * qq @ kk.transpose(1, 2) + add
        outs.append(o.permute(1, 0, 2))
        lses.append(torch.logsumexp(logits, dim=-1).permute(1, 0))
    return torch.cat(outs).numpy(), torch.cat(lses).numpy()


def _oracle(case, rows=None, bias=None, window=None):
    return oracle.rel_attn(case.q, case.k_cache, case.v_cache, case.block_table,
                           case.cu_q_lens, case.seq_lens,
                           case.bias if bias is None else bias, scale=case.spec.scale,
                           window=case.spec.window if window is None else window, rows=rows)


CASES = [
    dict(q_lens=(150, 37), seq_lens=None, hq=4, hkv=2, r=64, window=0),
    dict(q_lens=(150, 37), seq_lens=None, hq=4, hkv=2, r=64, window=40),
    dict(q_lens=(9, 1, 5), seq_lens=(300, 129, 128), hq=8, hkv=1, r=200, window=0),
    dict(q_lens=(9, 3), seq_lens=(400, 50), hq=6, hkv=3, r=16, window=100),
    dict(q_lens=(64,), seq_lens=(64,), hq=2, hkv=2, r=1, window=0),
]


@pytest.mark.parametrize("kw", CASES)
def test_matches_torch_sdpa_float64(kw):
    case = W.make_case(W.small(**kw), seed=21)
    out, lse = _oracle(case)
    ref, ref_lse = _sdpa_reference(case)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-11)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-11)


@pytest.mark.parametrize("r,window", [(1, 0), (3, 0), (64, 0), (4, 0), (3, 1), (64, 2), (5, 5), (64, 7)])
def test_matches_pure_python_brute_force(r, window):
    """Per-logit enumeration over logical keys on a tiny case (S <= 16, Hq=4, Hkv=2)."""
    spec = W.small(q_lens=(11, 5), seq_lens=(16, 5), hq=4, hkv=2, r=r, window=window,
                   bias_std=1.0)
    case = W.make_case(spec, seed=22)
    case.bias = torch.arange(4 * r, dtype=torch.float32).reshape(4, r) * 0.37 - 1.0  # distinct entries
    out, lse = _oracle(case)
    kv = _logical_kv(case)
    cu = case.cu_q_lens.tolist()
    G = spec.group
    for b in range(spec.batch):
        n, L = cu[b + 1] - cu[b], int(case.seq_lens[b])
        k, v = kv[b]
        for t in range(n):
            for h in range(spec.hq):
                o, l = brute.attention_row(case.q[cu[b] + t, h].double().tolist(),
                                           k[:, h // G].tolist(), v[:, h // G].tolist(),
                                           case.bias[h].double().tolist(), L - n + t,
                                           spec.scale, window)
                np.testing.assert_allclose(out[cu[b] + t, h], o, rtol=0, atol=1e-12)
                assert abs(lse[cu[b] + t, h] - l) < 1e-12


def test_closed_form_two_keys():
    """Query at position 1 with keys 0 and 1: o = (e^s0 v0 + e^s1 v1) / (e^s0 + e^s1),
    s0 = scale q.k0 + b[1], s1 = scale q.k1 + b[0]."""
    spec = W.small(q_lens=(2,), seq_lens=(2,), hq=1, hkv=1, r=4, scale=0.5)
    case = W.make_case(spec, seed=23)
    q = torch.zeros(2, 1, 128); q[1, 0, 0] = 2.0; q[1, 0, 1] = -1.0
    case.q = q.to(torch.bfloat16)
    k0 = torch.zeros(128); k0[0] = 1.0
    k1 = torch.zeros(128); k1[1] = 3.0
    v0 = torch.arange(128.0) / 64
    v1 = -torch.ones(128)
    blk = int(case.block_table[0, 0])
    case.k_cache[blk, 0, 0] = k0.bfloat16(); case.k_cache[blk, 0, 1] = k1.bfloat16()
    case.v_cache[blk, 0, 0] = v0.bfloat16(); case.v_cache[blk, 0, 1] = v1.bfloat16()
    case.bias = torch.tensor([[0.5, -0.25, 7.0, 7.0]])
    out, lse = _oracle(case, rows=[1])
    s0 = 0.5 * 2.0 + (-0.25)
    s1 = 0.5 * (-3.0) + 0.5
    e0, e1 = math.exp(s0), math.exp(s1)
    want = (e0 * v0.double() + e1 * v1.double()) / (e0 + e1)
    np.testing.assert_allclose(out[0, 0], want.numpy(), rtol=0, atol=1e-14)
    assert abs(lse[0, 0] - math.log(e0 + e1)) < 1e-14


def test_window_one_returns_own_value_row():
    case = W.make_case(W.small(q_lens=(40, 3), seq_lens=(40, 200), window=1), seed=24)
    out, _ = _oracle(case)
    kv = _logical_kv(case)
    cu = case.cu_q_lens.tolist()
    for b in range(2):
        n, L = cu[b + 1] - cu[b], int(case.seq_lens[b])
        v = kv[b][1]
        for t in range(n):
            for h in range(case.spec.hq):
                assert np.array_equal(out[cu[b] + t, h], v[L - n + t, h // case.spec.group].numpy())


def test_first_row_returns_first_value_row():
    case = W.make_case(W.small(q_lens=(20,)), seed=25)
    out, _ = _oracle(case, rows=[0])
    v = _logical_kv(case)[0][1]
    for h in range(case.spec.hq):
        assert np.array_equal(out[0, h], v[0, h // case.spec.group].numpy())


def test_zero_and_row_constant_bias_give_plain_attention():
    case = W.make_case(W.small(q_lens=(130, 9), seq_lens=(130, 140)), seed=26)
    hq, r = case.bias.shape
    plain, plain_lse = _oracle(case, bias=torch.zeros(hq, r))
    # plain softmax attention from torch, no bias at all
    ref, _ = _sdpa_reference(case, bias=torch.zeros(hq, r))
    np.testing.assert_allclose(plain, ref, rtol=0, atol=1e-11)
    const = torch.linspace(-3, 5, hq)[:, None].expand(hq, r).contiguous()
    out, lse = _oracle(case, bias=const)
    np.testing.assert_allclose(out, plain, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse - plain_lse, const[:, 0].double().numpy()[None, :].repeat(lse.shape[0], 0), atol=1e-11)


def test_per_head_shift_of_table_leaves_output_unchanged():
    case = W.make_case(W.small(q_lens=(70, 20), window=33), seed=27)
    out, _ = _oracle(case)
    shifted = case.bias + torch.linspace(-2, 2, case.spec.hq)[:, None]
    out2, _ = _oracle(case, bias=shifted)
    np.testing.assert_allclose(out, out2, rtol=0, atol=1e-12)


def test_r_equal_one_is_plain_attention():
    case = W.make_case(W.small(q_lens=(90,), r=1), seed=28)
    out, _ = _oracle(case)
    plain, _ = _oracle(case, bias=torch.zeros_like(case.bias))
    np.testing.assert_allclose(out, plain, rtol=0, atol=1e-12)


def test_window_at_least_length_equals_full():
    case = W.make_case(W.small(q_lens=(100, 7), seq_lens=(100, 180)), seed=29)
    full, _ = _oracle(case, window=0)
    for w in (180, 181, 10_000):
        out, _ = _oracle(case, window=w)
        assert np.array_equal(out, full)
    out, _ = _oracle(case, window=150)
    assert not np.allclose(out, full)


def test_shuffled_pages_equal_identity_pages():
    spec = W.small(q_lens=(200, 9), seq_lens=(300, 129))
    a = W.make_case(spec, seed=30, identity_table=True)
    b = W.make_case(spec, seed=30, table_seed=777)
    # same logical contents: re-scatter a's pages into b's physical layout
    for s in range(spec.batch):
        for lp in range((int(a.seq_lens[s]) + 127) // 128):
            b.k_cache[int(b.block_table[s, lp])] = a.k_cache[int(a.block_table[s, lp])]
            b.v_cache[int(b.block_table[s, lp])] = a.v_cache[int(a.block_table[s, lp])]
    assert not torch.equal(a.block_table, b.block_table)
    oa, la = _oracle(a)
    ob, lb = _oracle(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_gqa_equals_repeated_kv_heads():
    """G = 2 with Hkv = 1 equals G = 1 with the single KV head copied to two heads."""
    spec = W.small(q_lens=(50,), hq=2, hkv=1)
    a = W.make_case(spec, seed=31)
    spec2 = W.small(q_lens=(50,), hq=2, hkv=2)
    b = W.make_case(spec2, seed=31)
    b.q, b.bias = a.q, a.bias
    b.block_table = a.block_table
    b.k_cache = a.k_cache.expand(-1, 2, -1, -1).contiguous()
    b.v_cache = a.v_cache.expand(-1, 2, -1, -1).contiguous()
    oa, _ = _oracle(a)
    ob, _ = _oracle(b)
    assert np.array_equal(oa, ob)


def test_token_by_token_decode_equals_one_shot_prefill():
    """Carry the sconv state and the paged cache through 100 + 1 + 1 + 9 + 9 tokens and
    compare every step's attention rows with one prefill over all 120 tokens."""
    Lt = 120
    spec = W.small(q_lens=(Lt,), seq_lens=(Lt,), hq=4, hkv=2, r=50, window=37)
    full = W.make_case(spec, seed=32)
    kc, vc, st = full.k_cache.clone(), full.v_cache.clone(), full.state.clone()
    oracle.sconv_kv(full.k_raw, full.v_raw, full.w_k, full.w_v, st, full.cu_q_lens,
                    full.slot_mapping, kc, vc)
    ref, ref_lse = oracle.rel_attn(full.q, kc, vc, full.block_table, full.cu_q_lens,
                                   full.seq_lens, full.bias, scale=spec.scale, window=spec.window)

    kc2, vc2, st2 = full.k_cache.clone(), full.v_cache.clone(), full.state.clone()
    start = 0
    for n in (100, 1, 1, 9, 9):
        sl = slice(start, start + n)
        cu = torch.tensor([0, n], dtype=torch.int32)
        oracle.sconv_kv(full.k_raw[sl], full.v_raw[sl], full.w_k, full.w_v, st2, cu,
                        full.slot_mapping[sl], kc2, vc2)
        out, lse = oracle.rel_attn(full.q[sl], kc2, vc2, full.block_table, cu,
                                   torch.tensor([start + n], dtype=torch.int32), full.bias,
                                   scale=spec.scale, window=spec.window)
        assert np.array_equal(out, ref[sl]) and np.array_equal(lse, ref_lse[sl])
        start += n
    assert start == Lt
    assert torch.equal(kc.view(torch.int16), kc2.view(torch.int16))
    assert torch.equal(st.view(torch.int16), st2.view(torch.int16))


def test_bad_block_id_is_reported():
    case = W.make_case(W.small(q_lens=(10,)), seed=33)
    case.block_table = case.block_table.clone()
    case.block_table[0, 0] = case.k_cache.shape[0]
    with pytest.raises(RuntimeError, match="block id"):
        _oracle(case)
