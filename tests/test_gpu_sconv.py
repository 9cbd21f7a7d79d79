"""GPU parity of inkling_sconv_kv against the oracle (sconv on K/V into the paged cache and
the sconv-state update; vLLM Day-0 Inkling blog, "Model Architecture / Sconv" and
"Managing the sconv cache")."""
import numpy as np
import pytest
import torch

import workloads as W
from harness import (assert_cache_matches, assert_state_matches, bf16_bits, gpu_sconv,
                     run_oracle, snapshot)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ink():
    import relative_position_gqa_gb300 as m
    m._lib.load()
    return m


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


CASES = [
    dict(q_lens=(1, 2, 3, 0, 33, 64, 65, 200), seq_lens=(5, 2, 130, 7, 33, 300, 65, 260), hkv=2),
    dict(q_lens=(256,), seq_lens=(256,), hkv=1),
    dict(q_lens=(9,) * 5, seq_lens=(4096, 10, 129, 128, 127), hkv=8),
    dict(q_lens=(31, 32, 97), seq_lens=(31, 40, 1000), hkv=4),
]


@pytest.mark.parametrize("kw", CASES)
def test_sconv_matches_oracle(ink, kw):
    spec = W.small(q_lens=kw["q_lens"], seq_lens=kw["seq_lens"], hq=kw["hkv"], hkv=kw["hkv"],
                   history_random=True, state_random=True)
    g = W.make_case(spec, seed=41, device="cuda")
    snap = snapshot(g)
    st = _status()
    gpu_sconv(ink, g, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    kc, vc, state, _, _ = run_oracle(snap, rows=[])
    assert_cache_matches(g.k_cache, kc, snap, 0)
    assert_cache_matches(g.v_cache, vc, snap, 1)
    assert_state_matches(g.state, state, snap)


@pytest.mark.parametrize("taps,shift", [([0, 0, 0, 1], 0), ([1, 0, 0, 0], 3), ([0, 1, 0, 0], 2)])
def test_one_hot_taps_bit_exact(ink, taps, shift):
    spec = W.small(q_lens=(70, 2), seq_lens=(80, 2), hq=2, hkv=2, history_random=True,
                   state_random=True)
    g = W.make_case(spec, seed=42, device="cuda")
    w = torch.tensor(taps, dtype=torch.float32, device="cuda").repeat(spec.channels, 1).contiguous()
    g.w_k, g.w_v = w, w.clone()
    state0 = g.state.clone()
    st = _status()
    gpu_sconv(ink, g, st)
    torch.cuda.synchronize()
    cu = g.cu_q_lens.tolist()
    for b in range(spec.batch):
        for which, raw, cache in ((0, g.k_raw, g.k_cache), (1, g.v_raw, g.v_cache)):
            ext = torch.cat([state0[b, which], raw[cu[b]:cu[b + 1]]])
            slots = g.slot_mapping[cu[b]:cu[b + 1]]
            got = cache[slots // 128, :, slots % 128, :].reshape(len(slots), -1)
            want = ext[3 - shift: 3 - shift + len(slots)]
            assert np.array_equal(bf16_bits(got), bf16_bits(want))


def test_chunked_calls_bit_identical_to_one_call(ink):
    spec = W.small(q_lens=(256,), seq_lens=(256,), hq=4, hkv=4)
    a = W.make_case(spec, seed=43, device="cuda")
    b = W.make_case(spec, seed=43, device="cuda")
    st = _status()
    gpu_sconv(ink, a, st)
    start = 0
    for n in (100, 1, 155):
        sl = slice(start, start + n)
        ink.sconv_kv(b.k_raw[sl], b.v_raw[sl], b.w_k, b.w_v, b.state,
                     torch.tensor([0, n], dtype=torch.int32, device="cuda"), b.slot_mapping[sl],
                     b.k_cache, b.v_cache, max_q_len=n, dev_status=st)
        start += n
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for x, y in ((a.k_cache, b.k_cache), (a.v_cache, b.v_cache), (a.state, b.state)):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_skip_slot_and_bad_slot(ink):
    spec = W.small(q_lens=(5,), seq_lens=(5,), hq=2, hkv=2)
    g = W.make_case(spec, seed=44, device="cuda")
    before = g.k_cache.clone()
    g.slot_mapping = g.slot_mapping.clone()
    s2 = int(g.slot_mapping[2])
    g.slot_mapping[2] = -1
    st = _status()
    gpu_sconv(ink, g, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(g.k_cache[s2 // 128, :, s2 % 128], before[s2 // 128, :, s2 % 128])
    g.slot_mapping[3] = g.num_blocks * 128  # one past the last slot: reported, not written
    gpu_sconv(ink, g, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 5  # INKLING_ERR_BAD_BLOCK


def test_step_form_bit_identical_to_run_form(ink):
    """A host bound max_q_len <= 16 selects the step form of the kernel (one thread takes
    all of its sequence's new rows, loads issued in two rounds); a larger bound selects the
    run form.  They do the same arithmetic in the same order: caches and state agree bit
    for bit."""
    spec = W.small(q_lens=(9, 3, 0, 16, 1, 2), seq_lens=(100, 3, 5, 400, 129, 2), hq=2, hkv=2,
                   history_random=True, state_random=True)
    out = []
    for bound in (16, 64):
        g = W.make_case(spec, seed=43, device="cuda")
        st = _status()
        ink.sconv_kv(g.k_raw, g.v_raw, g.w_k, g.w_v, g.state, g.cu_q_lens, g.slot_mapping,
                     g.k_cache, g.v_cache, max_q_len=bound, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        out.append(g)
    a, b = out
    assert torch.equal(a.k_cache, b.k_cache) and torch.equal(a.v_cache, b.v_cache)
    assert torch.equal(a.state, b.state)
