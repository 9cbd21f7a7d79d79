"""GPU parity of inkling_rel_attn_decode_sconv, the decode step with the sconv of its new
tokens fused into the decode kernel's prologue (vLLM Day-0 Inkling blog, "vLLM
Integration & Optimization": kernel fusion; "Managing the sconv cache").  Against the two
separate calls (inkling_sconv_kv, then inkling_rel_attn_decode) on the same inputs the
caches, the sconv state, the output and the LSE must be bit-identical, and against the
fp64 oracle the output must meet the parity bar.  The cases put a step's new rows in one
page and across two, across two splits of the keys (so that two CTAs convolve parts of
one step and the merge kernel writes the state), fewer than three rows (the old state
feeds the new one), and sequences with no new token."""
import pytest
import torch

import workloads as W
from harness import compare_out, gpu_attn, gpu_sconv, run_oracle, snapshot

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ink():
    import relative_position_gqa_gb300 as m
    m._lib.load()
    return m


CASES = {
    # 251..259 straddle pages 1 and 2, which three splits of one page each separate
    "straddle_3_splits": (W.small(q_lens=(9, 9), seq_lens=(260, 130), hq=8, hkv=2, r=300), 3),
    "mtp9_auto": (W.small(q_lens=(9, 9, 9), seq_lens=(6000, 129, 9), hq=8, hkv=1, r=300), 0),
    "mixed_n_one_split": (W.small(q_lens=(1, 5, 9, 2, 0), seq_lens=(700, 5, 300, 1200, 40),
                                  hq=8, hkv=2, r=1000), 1),
    "mixed_n_4_splits": (W.small(q_lens=(1, 5, 9, 2, 0), seq_lens=(700, 5, 300, 1200, 40),
                                 hq=8, hkv=2, r=1000), 4),
    "window_300": (W.small(q_lens=(9, 3, 9), seq_lens=(1500, 200, 301), hq=8, hkv=1, r=2000,
                           window=300), 0),
    "n1_g16": (W.small(q_lens=(1, 1, 2), seq_lens=(2000, 128, 257), hq=16, hkv=1, r=500), 2),
}


def _fused(ink, g, num_splits, st):
    spec = g.spec
    out = torch.full((spec.total_q, spec.hq, 128), float("nan"), device="cuda")
    lse = torch.full((spec.total_q, spec.hq), float("nan"), device="cuda")
    ink.rel_attn_decode_sconv(g.q, g.k_raw, g.v_raw, g.w_k, g.w_v, g.state, g.k_cache,
                              g.v_cache, g.block_table, g.cu_q_lens, g.seq_lens, g.bias,
                              scale=spec.scale, window=spec.window, max_q_len=spec.max_q_len,
                              max_seq_len=spec.max_seq_len, num_splits=num_splits, out=out,
                              lse=lse, dev_status=st)
    return out, lse


def _both(ink, spec, seed, num_splits):
    sep = W.make_case(spec, seed=seed, device="cuda")
    fus = W.make_case(spec, seed=seed, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_sconv(ink, sep, st)
    ref, ref_lse = gpu_attn(ink, sep, st, decode=True, num_splits=num_splits)
    out, lse = _fused(ink, fus, num_splits, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, ink.status_string(int(st.item()))
    assert torch.equal(fus.k_cache.view(torch.int16), sep.k_cache.view(torch.int16))
    assert torch.equal(fus.v_cache.view(torch.int16), sep.v_cache.view(torch.int16))
    assert torch.equal(fus.state.view(torch.int16), sep.state.view(torch.int16))
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
    return fus, out, lse


@pytest.mark.parametrize("name", sorted(CASES))
def test_fused_decode_bit_identical_to_separate_calls_and_matches_oracle(ink, name):
    spec, num_splits = CASES[name]
    _, out, lse = _both(ink, spec, seed=71, num_splits=num_splits)
    snap = snapshot(W.make_case(spec, seed=71, device="cuda"))
    _, _, _, ref, ref_lse = run_oracle(snap)
    compare_out(out, lse, ref, ref_lse, snap.tok_index)


def test_fused_decode_steps_carry_the_state(ink):
    """Decode steps of 9, 1, 2, 9 tokens through the fused call, each step's state feeding
    the next, equal the same steps through the separate calls, bit for bit."""
    total = 21
    spec = W.small(q_lens=(total,), seq_lens=(600,), hq=8, hkv=1, r=150, window=0)
    sep = W.make_case(spec, seed=72, device="cuda")
    fus = W.make_case(spec, seed=72, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    start = 600 - total
    done = 0
    for n in (9, 1, 2, 9):
        sl = slice(done, done + n)
        cu = torch.tensor([0, n], dtype=torch.int32, device="cuda")
        L = torch.tensor([start + done + n], dtype=torch.int32, device="cuda")
        outs = []
        for g, fused in ((sep, False), (fus, True)):
            out = torch.empty(n, spec.hq, 128, device="cuda")
            kw = dict(scale=spec.scale, window=0, max_q_len=n, max_seq_len=start + done + n,
                      num_splits=2, out=out, dev_status=st)
            if fused:
                ink.rel_attn_decode_sconv(g.q[sl], g.k_raw[sl], g.v_raw[sl], g.w_k, g.w_v,
                                          g.state, g.k_cache, g.v_cache, g.block_table, cu, L,
                                          g.bias, **kw)
            else:
                ink.sconv_kv(g.k_raw[sl], g.v_raw[sl], g.w_k, g.w_v, g.state, cu,
                             g.slot_mapping[sl], g.k_cache, g.v_cache, max_q_len=n,
                             dev_status=st)
                ink.rel_attn_decode(g.q[sl], g.k_cache, g.v_cache, g.block_table, cu, L, g.bias,
                                    **kw)
            outs.append(out)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(outs[0], outs[1])
        assert torch.equal(fus.state.view(torch.int16), sep.state.view(torch.int16))
        done += n
    assert torch.equal(fus.k_cache.view(torch.int16), sep.k_cache.view(torch.int16))
    assert torch.equal(fus.v_cache.view(torch.int16), sep.v_cache.view(torch.int16))


@pytest.mark.parametrize("wl,variant", [(4, "swa"), (4, "full"), (5, "n9")])
def test_fused_decode_full_size_bit_identical(ink, wl, variant):
    """The MTP decode (both layer kinds) and the 1M-token 9-token decode at full size."""
    _both(ink, W.config(wl, variant=variant), seed=wl, num_splits=0)
