"""Pins for the oracle's sconv (window-4 causal depthwise conv on K and V, with a cache of
the last 3 raw rows; vLLM Day-0 Inkling blog, "Model Architecture / Sconv" and
"vLLM Integration & Optimization / Managing the sconv cache").  CPU only."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_bf16_rounding_golden():
    """Hand-derived bf16 round-to-nearest-even cases, incl. a double-rounding trap."""
    n = 0
    for line in open(os.path.join(GOLDEN, "bf16_round.txt")):
        if line.startswith("#") or not line.strip():
            continue
        val, want = line.split()[:2]
        assert oracle.bf16_round(float.fromhex(val)) == int(want, 16), line
        n += 1
    assert n >= 15


def test_bf16_rounding_matches_torch_on_binary32_values():
    """For inputs that are exact binary32 values, one-step rounding equals torch's own
    float32 -> bfloat16 conversion (round to nearest even)."""
    g = torch.Generator().manual_seed(0)
    x = torch.randn(4000, generator=g) * torch.exp2(torch.randint(-40, 40, (4000,), generator=g).float())
    want = _bits(x.to(torch.bfloat16))
    got = np.array([oracle.bf16_round(float(v)) for v in x.tolist()], dtype=np.uint16)
    assert np.array_equal(got, want)


def _run(case, k_cache=None, v_cache=None, state=None):
    kc = case.k_cache.clone() if k_cache is None else k_cache
    vc = case.v_cache.clone() if v_cache is None else v_cache
    st = case.state.clone() if state is None else state
    oracle.sconv_kv(case.k_raw, case.v_raw, case.w_k, case.w_v, st, case.cu_q_lens,
                    case.slot_mapping, kc, vc)
    return kc, vc, st


def _gather_new(cache, case):
    """The cache rows at the new tokens' slots, [T, C] (page math written with torch)."""
    slots = case.slot_mapping
    blk, off = slots // 128, slots % 128
    rows = cache[blk, :, off, :]              # [T, Hkv, 128]
    return rows.reshape(rows.shape[0], -1)


def _spec(q_lens=(7, 2, 19), hkv=2, state_random=True):
    return W.small(q_lens=q_lens, seq_lens=[n + 5 for n in q_lens], hq=2 * hkv, hkv=hkv,
                   state_random=state_random, history_random=True)


@pytest.mark.parametrize("taps,shift", [([0, 0, 0, 1], 0), ([0, 0, 1, 0], 1),
                                        ([0, 1, 0, 0], 2), ([1, 0, 0, 0], 3)])
def test_one_hot_taps_select_rows(taps, shift):
    """w[c,3] multiplies the current raw row, w[c,0] the row three back; rows before the
    new tokens come from the state, oldest first.  Bit-exact."""
    case = W.make_case(_spec(), seed=11)
    C = case.spec.channels
    w = torch.tensor(taps, dtype=torch.float32).repeat(C, 1)
    case.w_k, case.w_v = w.clone(), w.clone()
    kc, vc, _ = _run(case)
    for which, cache, raw in ((0, kc, case.k_raw), (1, vc, case.v_raw)):
        got = _gather_new(cache, case)
        cu = case.cu_q_lens.tolist()
        for b in range(case.spec.batch):
            ext = torch.cat([case.state[b, which], raw[cu[b]:cu[b + 1]]])   # [3+n, C]
            n = cu[b + 1] - cu[b]
            want = ext[3 - shift: 3 - shift + n]
            assert torch.equal(got[cu[b]:cu[b + 1]].view(torch.int16), want.view(torch.int16))


def test_state_becomes_last_three_raw_rows():
    case = W.make_case(_spec(q_lens=(7, 2, 1, 0, 3)), seed=12)
    _, _, st = _run(case)
    cu = case.cu_q_lens.tolist()
    for b in range(case.spec.batch):
        for which, raw in ((0, case.k_raw), (1, case.v_raw)):
            ext = torch.cat([case.state[b, which], raw[cu[b]:cu[b + 1]]])
            assert torch.equal(st[b, which].view(torch.int16), ext[-3:].view(torch.int16))


def test_small_integer_inputs_are_exact():
    """Small integers and dyadic taps: every sum is exact in bf16, so the conv must equal
    the brute-force sum bit for bit."""
    case = W.make_case(_spec(), seed=13)
    g = torch.Generator().manual_seed(5)
    for name in ("k_raw", "v_raw"):
        setattr(case, name, torch.randint(-3, 4, getattr(case, name).shape, generator=g).to(torch.bfloat16))
    case.state = torch.randint(-3, 4, case.state.shape, generator=g).to(torch.bfloat16)
    choices = torch.tensor([-1.0, -0.5, 0.0, 0.25, 0.5, 1.0, 2.0])
    C = case.spec.channels
    case.w_k = choices[torch.randint(0, 7, (C, 4), generator=g)]
    case.w_v = choices[torch.randint(0, 7, (C, 4), generator=g)]
    kc, vc, _ = _run(case)
    cu = case.cu_q_lens.tolist()
    for which, cache, raw, w in ((0, kc, case.k_raw, case.w_k), (1, vc, case.v_raw, case.w_v)):
        got = _gather_new(cache, case).float()
        for b in range(case.spec.batch):
            y = brute.sconv_rows(case.state[b, which].float().tolist(),
                                 raw[cu[b]:cu[b + 1]].float().tolist(), w.tolist())
            if y:
                assert torch.equal(got[cu[b]:cu[b + 1]], torch.tensor(y, dtype=torch.float32))


def test_random_inputs_within_half_ulp_of_brute_force():
    case = W.make_case(_spec(q_lens=(33, 4)), seed=14)
    kc, vc, _ = _run(case)
    cu = case.cu_q_lens.tolist()
    for which, cache, raw, w in ((0, kc, case.k_raw, case.w_k), (1, vc, case.v_raw, case.w_v)):
        got = _gather_new(cache, case).double()
        for b in range(case.spec.batch):
            y = torch.tensor(brute.sconv_rows(case.state[b, which].double().tolist(),
                                              raw[cu[b]:cu[b + 1]].double().tolist(),
                                              w.double().tolist()), dtype=torch.float64)
            # half a bf16 ulp of |y|: 2^(floor(log2|y|) - 8)
            half_ulp = torch.exp2(torch.floor(torch.log2(y.abs().clamp_min(2.0 ** -126))) - 8)
            assert (got[cu[b]:cu[b + 1]] - y).abs().le(half_ulp).all()


def test_chunked_calls_equal_one_call():
    """256 new tokens as one call, or as 100 + 1 + 155 carried through the state."""
    spec = W.small(q_lens=(256,), seq_lens=(256,), hq=2, hkv=1)
    case = W.make_case(spec, seed=15)
    kc1, vc1, st1 = _run(case)
    kc, vc, st = case.k_cache.clone(), case.v_cache.clone(), case.state.clone()
    start = 0
    for n in (100, 1, 155):
        sl = slice(start, start + n)
        oracle.sconv_kv(case.k_raw[sl], case.v_raw[sl], case.w_k, case.w_v, st,
                        torch.tensor([0, n], dtype=torch.int32), case.slot_mapping[sl], kc, vc)
        start += n
    assert torch.equal(kc.view(torch.int16), kc1.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vc1.view(torch.int16))
    assert torch.equal(st.view(torch.int16), st1.view(torch.int16))


def test_slot_minus_one_is_not_stored():
    case = W.make_case(_spec(q_lens=(5,)), seed=16)
    case.slot_mapping = case.slot_mapping.clone()
    skipped = int(case.slot_mapping[2])
    case.slot_mapping[2] = -1
    kc, _, _ = _run(case)
    blk, off = skipped // 128, skipped % 128
    assert torch.equal(kc[blk, :, off].view(torch.int16), case.k_cache[blk, :, off].view(torch.int16))


def test_linearity_in_taps():
    """conv(w1 + w2) == conv(w1) + conv(w2) before rounding; with small-integer data and
    dyadic taps the rounding is exact, so the identity holds bit for bit."""
    case = W.make_case(_spec(q_lens=(9,)), seed=17)
    g = torch.Generator().manual_seed(9)
    case.k_raw = torch.randint(-2, 3, case.k_raw.shape, generator=g).to(torch.bfloat16)
    case.state = torch.randint(-2, 3, case.state.shape, generator=g).to(torch.bfloat16)
    C = case.spec.channels
    w1 = torch.randint(-2, 3, (C, 4), generator=g).float()
    w2 = torch.randint(-2, 3, (C, 4), generator=g).float() * 0.5
    outs = []
    for w in (w1, w2, w1 + w2):
        case.w_k = w
        kc, _, _ = _run(case)
        outs.append(_gather_new(kc, case).double())
    assert torch.equal(outs[0] + outs[1], outs[2])


# ------------------------------------------------ dense stream and MTP rollback ----

def _dense_case(q_lens=(7, 2, 40), C=64, seed=18, state_random=True):
    g = torch.Generator().manual_seed(seed)
    T = sum(q_lens)
    x = torch.randn(T, C, generator=g).to(torch.bfloat16)
    w = (torch.randn(C, 4, generator=g) * 0.5).float()
    st = (torch.randn(len(q_lens), 3, C, generator=g) if state_random
          else torch.zeros(len(q_lens), 3, C)).to(torch.bfloat16)
    cu = torch.tensor([0] + list(np.cumsum(q_lens)), dtype=torch.int32)
    return x, w, st, cu


def test_dense_sconv_equals_the_k_stream_of_sconv_kv():
    """The dense-stream conv and the paged K/V conv are the same definition."""
    case = W.make_case(_spec(q_lens=(7, 2, 19)), seed=19)
    kc, _, st = _run(case)
    st_d = case.state[:, 0].clone().contiguous()
    y = oracle.sconv_dense(case.k_raw, case.w_k, st_d, case.cu_q_lens)
    assert torch.equal(_gather_new(kc, case).view(torch.int16), y.view(torch.int16))
    assert torch.equal(st[:, 0].contiguous().view(torch.int16), st_d.view(torch.int16))


@pytest.mark.parametrize("taps,shift", [([0, 0, 0, 1], 0), ([1, 0, 0, 0], 3), ([0, 0, 1, 0], 1)])
def test_dense_sconv_one_hot_taps(taps, shift):
    x, _, st, cu = _dense_case()
    w = torch.tensor(taps, dtype=torch.float32).repeat(x.shape[1], 1)
    y = oracle.sconv_dense(x, w, st.clone(), cu)
    c = cu.tolist()
    for b in range(len(c) - 1):
        ext = torch.cat([st[b], x[c[b]:c[b + 1]]])
        n = c[b + 1] - c[b]
        assert torch.equal(y[c[b]:c[b + 1]].view(torch.int16), ext[3 - shift:3 - shift + n].view(torch.int16))


def test_dense_sconv_within_half_ulp_of_brute_force():
    x, w, st, cu = _dense_case(q_lens=(11, 5), C=32)
    y = oracle.sconv_dense(x, w, st.clone(), cu).double()
    c = cu.tolist()
    for b in range(len(c) - 1):
        ref = torch.tensor(brute.sconv_rows(st[b].double().tolist(), x[c[b]:c[b + 1]].double().tolist(),
                                            w.double().tolist()), dtype=torch.float64)
        half_ulp = torch.exp2(torch.floor(torch.log2(ref.abs().clamp_min(2.0 ** -126))) - 8)
        assert (y[c[b]:c[b + 1]] - ref).abs().le(half_ulp).all()


@pytest.mark.parametrize("accepted", [[7, 2, 40], [0, 0, 0], [3, 1, 17], [1, 2, 2]])
def test_rollback_equals_running_only_the_kept_tokens(accepted):
    """After a step of n_b tokens of which only the first a_b are kept, the cache must be
    what a step of just those a_b tokens would have left (rows of the conv are causal)."""
    x, w, st0, cu = _dense_case(q_lens=(7, 2, 40))
    st_full = st0.clone()
    oracle.sconv_dense(x, w, st_full, cu)
    rolled = oracle.sconv_rollback(st0, x, None, cu, torch.tensor(accepted, dtype=torch.int32))
    c = cu.tolist()
    keep = torch.cat([torch.arange(c[b], c[b] + a) for b, a in enumerate(accepted)])
    cu_keep = torch.tensor([0] + list(np.cumsum(accepted)), dtype=torch.int32)
    st_keep = st0.clone()
    oracle.sconv_dense(x[keep], w, st_keep, cu_keep)
    assert torch.equal(rolled.view(torch.int16), st_keep.view(torch.int16))
    if accepted == [7, 2, 40]:
        assert torch.equal(rolled.view(torch.int16), st_full.view(torch.int16))
    if accepted == [0, 0, 0]:
        assert torch.equal(rolled.view(torch.int16), st0.view(torch.int16))


def test_rollback_kv_pair_layout():
    case = W.make_case(_spec(q_lens=(9, 9, 4)), seed=20)
    acc = torch.tensor([4, 9, 0], dtype=torch.int32)
    rolled = oracle.sconv_rollback(case.state, case.k_raw, case.v_raw, case.cu_q_lens, acc)
    c = case.cu_q_lens.tolist()
    for b in range(3):
        for which, raw in ((0, case.k_raw), (1, case.v_raw)):
            ext = torch.cat([case.state[b, which], raw[c[b]:c[b] + int(acc[b])]])
            assert torch.equal(rolled[b, which].view(torch.int16), ext[-3:].view(torch.int16))
