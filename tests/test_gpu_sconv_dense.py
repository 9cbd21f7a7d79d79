"""GPU parity of the conv on a dense stream (inkling_sconv) and of the sconv-state rollback
after a speculative step (inkling_sconv_state_rollback) against the oracle (vLLM Day-0
Inkling blog, "Model Architecture / Sconv" and "Model Architecture / MTP",
"Re-computing MTP KV cache")."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from harness import bf16_bits, gpu_sconv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ink():
    import relative_position_gqa_gb300 as m
    m._lib.load()
    return m


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _magnitude(x, w, state, cu):
    """S[t, c] = sum_j |w[c, j]| |x~[t + j, c]|: the scale of the fp32 rounding error."""
    cu = cu.tolist()
    out = []
    for b in range(len(cu) - 1):
        n = cu[b + 1] - cu[b]
        ext = torch.cat([state[b].float().abs(), x[cu[b]:cu[b + 1]].float().abs()])
        acc = torch.zeros(n, x.shape[1])
        for j in range(4):
            acc += w[:, j].abs() * ext[j:j + n]
        out.append(acc)
    return torch.cat(out).double()


def _assert_conv_close(y_gpu, y_ora, S):
    """|gpu - oracle| <= ulp_bf16(oracle) + 2^-21 S (four fp32 roundings vs one fp64 sum,
    each rounded once to bf16), and almost all outputs identical."""
    g, o = y_gpu.cpu().double(), y_ora.double()
    ulp = torch.exp2(torch.floor(torch.log2(o.abs().clamp_min(2.0 ** -126))) - 7)
    bad = (g - o).abs() > ulp + 2.0 ** -21 * S
    assert not bad.any(), f"{int(bad.sum())} conv outputs outside the fp32 rounding bound"
    if g.numel():
        assert float((g != o).double().mean()) < 1e-3


CASES = [((1, 2, 3, 0, 33, 64, 65, 200), 128), ((256,), 1024), ((9,) * 7, 4096),
         ((31, 32, 97), 8), ((5, 0, 1), 24)]


@pytest.mark.parametrize("q_lens,C", CASES)
def test_dense_sconv_matches_oracle(ink, q_lens, C):
    c = W.make_dense(q_lens, C, seed=61)
    g = W.make_dense(q_lens, C, seed=61, device="cuda")
    st = _status()
    y = ink.sconv(g.x, g.w, g.state, g.cu_q_lens, max_q_len=c.max_q_len, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    S = _magnitude(c.x, c.w, c.state, c.cu_q_lens)
    state_ora = c.state.clone()
    y_ora = oracle.sconv_dense(c.x, c.w, state_ora, c.cu_q_lens)
    _assert_conv_close(y, y_ora, S)
    assert np.array_equal(bf16_bits(g.state), bf16_bits(state_ora))


@pytest.mark.parametrize("taps,shift", [([0, 0, 0, 1], 0), ([1, 0, 0, 0], 3), ([0, 0, 1, 0], 1)])
def test_dense_one_hot_taps_bit_exact(ink, taps, shift):
    g = W.make_dense((70, 2, 33), 256, seed=62, device="cuda")
    w = torch.tensor(taps, dtype=torch.float32, device="cuda").repeat(256, 1).contiguous()
    state0 = g.state.clone()
    y = ink.sconv(g.x, w, g.state, g.cu_q_lens, max_q_len=g.max_q_len)
    torch.cuda.synchronize()
    cu = g.cu_q_lens.tolist()
    for b in range(len(cu) - 1):
        ext = torch.cat([state0[b], g.x[cu[b]:cu[b + 1]]])
        n = cu[b + 1] - cu[b]
        assert np.array_equal(bf16_bits(y[cu[b]:cu[b + 1]]), bf16_bits(ext[3 - shift:3 - shift + n]))


def test_dense_chunked_calls_bit_identical_to_one_call(ink):
    a = W.make_dense((256,), 512, seed=63, device="cuda")
    b = W.make_dense((256,), 512, seed=63, device="cuda")
    y1 = ink.sconv(a.x, a.w, a.state, a.cu_q_lens, max_q_len=256)
    parts, start = [], 0
    for n in (100, 1, 155):
        parts.append(ink.sconv(b.x[start:start + n], b.w, b.state,
                               torch.tensor([0, n], dtype=torch.int32, device="cuda"), max_q_len=n))
        start += n
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), torch.cat(parts).view(torch.int16))
    assert torch.equal(a.state.view(torch.int16), b.state.view(torch.int16))


def test_dense_bad_lengths_reported(ink):
    g = W.make_dense((20, 4), 64, seed=64, device="cuda")
    st = _status()
    ink.sconv(g.x, g.w, g.state, g.cu_q_lens, max_q_len=8, dev_status=st)  # n = 20 > 8
    torch.cuda.synchronize()
    assert int(st.item()) == 6  # INKLING_ERR_BAD_INPUT


def test_dense_rejects_aliased_output(ink):
    g = W.make_dense((4,), 64, seed=65, device="cuda")
    with pytest.raises(ink.InklingError):
        ink.sconv(g.x, g.w, g.state, g.cu_q_lens, max_q_len=4, y=g.x)


ACCEPTED = [[0, 1, 2, 3, 9, 9, 5, 7], [9] * 8, [0] * 8, [1, 0, 2, 2, 8, 3, 4, 6]]


@pytest.mark.parametrize("accepted", ACCEPTED)
@pytest.mark.parametrize("in_place", [False, True])
def test_rollback_kv_pair_matches_oracle(ink, accepted, in_place):
    spec = W.small(q_lens=(9,) * 8, seq_lens=(9, 20, 130, 300, 9, 12, 128, 129), hq=8, hkv=4,
                   history_random=True, state_random=True)
    g = W.make_case(spec, seed=66, device="cuda")
    before = g.state.clone()
    acc = torch.tensor(accepted, dtype=torch.int32)
    want = oracle.sconv_rollback(before.cpu(), g.k_raw.cpu(), g.v_raw.cpu(), g.cu_q_lens.cpu(), acc)
    st = _status()
    gpu_sconv(ink, g, st)  # the verify step moves the state past all 9 tokens
    torch.cuda.synchronize()
    after_all = g.state.clone()
    if in_place:
        g.state.copy_(before)
        out = ink.sconv_state_rollback(g.state, g.k_raw, g.v_raw, g.cu_q_lens, acc.cuda(),
                                       g.state, dev_status=st)
    else:
        out = ink.sconv_state_rollback(before, g.k_raw, g.v_raw, g.cu_q_lens, acc.cuda(),
                                       dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(bf16_bits(out), bf16_bits(want))
    if accepted == [9] * 8:  # keeping everything reproduces the conv call's own update
        assert np.array_equal(bf16_bits(out), bf16_bits(after_all))


@pytest.mark.parametrize("accepted", [[0, 4, 1], [3, 4, 2], [2, 1, 0]])
def test_rollback_dense_matches_oracle(ink, accepted):
    c = W.make_dense((3, 4, 2), 1024, seed=67)
    g = W.make_dense((3, 4, 2), 1024, seed=67, device="cuda")
    acc = torch.tensor(accepted, dtype=torch.int32)
    want = oracle.sconv_rollback(c.state, c.x, None, c.cu_q_lens, acc)
    out = ink.sconv_state_rollback(g.state, g.x, None, g.cu_q_lens, acc.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(out), bf16_bits(want))


def test_rollback_bad_accept_count_reported_and_state_untouched(ink):
    g = W.make_dense((3, 4), 64, seed=68, device="cuda")
    out = torch.full_like(g.state, 7.0)
    st = _status()
    ink.sconv_state_rollback(g.state, g.x, None, g.cu_q_lens,
                             torch.tensor([2, 5], dtype=torch.int32, device="cuda"), out,
                             dev_status=st)  # 5 > n_1 = 4
    torch.cuda.synchronize()
    assert int(st.item()) == 6
    assert torch.equal(out[1], torch.full_like(out[1], 7.0))
    assert not torch.equal(out[0], torch.full_like(out[0], 7.0))


def test_speculative_steps_equal_running_only_accepted_tokens(ink):
    """Three MTP verify steps of 9 tokens each with partial acceptance, the state rolled
    back after each: the K/V pages of the accepted tokens and the final state equal a run
    that saw only the accepted tokens (the oracle, one call per step)."""
    B, hkv = 4, 2
    C = hkv * 128
    gen = torch.Generator().manual_seed(69)
    state0 = torch.randn(B, 2, 3, C, generator=gen).to(torch.bfloat16)
    w_k = (torch.randn(C, 4, generator=gen) * 0.5).contiguous()
    w_v = (torch.randn(C, 4, generator=gen) * 0.5).contiguous()
    steps = [torch.tensor(a, dtype=torch.int32) for a in ([9, 0, 3, 1], [2, 9, 0, 5], [9, 9, 9, 9])]
    NB = 4 * B
    kc = torch.zeros(NB, hkv, 128, 128, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    kc_o, vc_o = kc.clone(), vc.clone()
    gk, gv = kc.cuda(), vc.cuda()
    g_state = state0.cuda()
    o_state = state0.clone()
    pos = [0] * B
    cu = torch.arange(0, 9 * B + 1, 9, dtype=torch.int32)
    st = _status()
    for acc in steps:
        k_raw = torch.randn(9 * B, C, generator=gen).to(torch.bfloat16)
        v_raw = torch.randn(9 * B, C, generator=gen).to(torch.bfloat16)
        slots = torch.tensor([b * 4 * 128 + pos[b] + i for b in range(B) for i in range(9)],
                             dtype=torch.int64)
        before = g_state.clone()
        ink.sconv_kv(k_raw.cuda(), v_raw.cuda(), w_k.cuda(), w_v.cuda(), g_state, cu.cuda(),
                     slots.cuda(), gk, gv, max_q_len=9, dev_status=st)
        ink.sconv_state_rollback(before, k_raw.cuda(), v_raw.cuda(), cu.cuda(), acc.cuda(),
                                 g_state, dev_status=st)
        # the oracle only ever sees the accepted tokens
        keep = torch.cat([torch.arange(9 * b, 9 * b + int(acc[b])) for b in range(B)])
        cu_keep = torch.zeros(B + 1, dtype=torch.int32)
        cu_keep[1:] = torch.cumsum(acc, 0)
        oracle.sconv_kv(k_raw[keep], v_raw[keep], w_k, w_v, o_state, cu_keep, slots[keep], kc_o, vc_o)
        for b in range(B):
            pos[b] += int(acc[b])
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(bf16_bits(g_state), bf16_bits(o_state))
    for b in range(B):  # accepted slots only (rejected drafts leave stale rows past pos[b])
        for cache_g, cache_o in ((gk, kc_o), (gv, vc_o)):
            g = cache_g[4 * b:4 * b + 4].cpu().permute(0, 2, 1, 3).reshape(4 * 128, C)[:pos[b]]
            o = cache_o[4 * b:4 * b + 4].permute(0, 2, 1, 3).reshape(4 * 128, C)[:pos[b]]
            # the paged conv's fp32-vs-fp64 bound, ulp + 2^-21 S, with S = sum |w x| < 64
            # for these N(0,1) rows and N(0, 0.5) taps
            ulp = torch.exp2(torch.floor(torch.log2(o.double().abs().clamp_min(2.0 ** -126))) - 7)
            assert ((g.double() - o.double()).abs() <= ulp + 2.0 ** -21 * 64.0).all()
            assert float((g != o).double().mean()) < 1e-2
