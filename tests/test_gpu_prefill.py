"""GPU parity of inkling_rel_attn_prefill (relative-bias GQA over full or sliding windows;
vLLM Day-0 Inkling blog, "Model Architecture / Attention") against the fp64 oracle, at
sizes the oracle finishes in seconds that still span several tiles and ragged tails."""
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


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _run(ink, spec, seed, out_dtype=torch.float32, **kw):
    g = W.make_case(spec, seed=seed, device="cuda", **kw)
    snap = snapshot(g)
    st = _status()
    gpu_sconv(ink, g, st)
    out, lse = gpu_attn(ink, g, st, decode=False, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, ink.status_string(int(st.item()))
    _, _, _, ref, ref_lse = run_oracle(snap)
    return compare_out(out, lse, ref, ref_lse, snap.tok_index), g, out


CASES = {
    "tiny_prefill": W.config(1),
    "ragged_two_seqs": W.small(q_lens=(150, 37), hq=4, hkv=2, r=64),
    "chunked_prefix": W.small(q_lens=(200, 9, 130), seq_lens=(457, 300, 130), hq=4, hkv=2, r=100),
    "window_5": W.small(q_lens=(300,), hq=2, hkv=1, r=64, window=5),
    "window_1": W.small(q_lens=(140,), hq=2, hkv=2, r=16, window=1),
    "window_130": W.small(q_lens=(400, 129), seq_lens=(600, 129), hq=4, hkv=1, r=256, window=130),
    "window_ge_len": W.small(q_lens=(260,), hq=2, hkv=1, r=64, window=4096),
    "r1_plain": W.small(q_lens=(190,), hq=2, hkv=1, r=1),
    "r3_clamped": W.small(q_lens=(300,), hq=4, hkv=4, r=3),
    "gqa3_odd": W.small(q_lens=(129, 1), seq_lens=(129, 1), hq=6, hkv=2, r=80),
    "gqa8": W.small(q_lens=(384,), hq=8, hkv=1, r=200, window=256),
    "empty_seq": W.small(q_lens=(0, 70, 0, 5), seq_lens=(10, 70, 0, 300), hq=2, hkv=1, r=32),
    "bias_r_mid_tile": W.small(q_lens=(513,), hq=2, hkv=1, r=300),
    # tables long enough that interior tiles fetch their bias run with one bulk copy,
    # mixed with diagonal and clamped tiles that take the per-element path
    "bulk_bias_full": W.small(q_lens=(900,), hq=4, hkv=2, r=1024),
    "bulk_bias_window": W.small(q_lens=(1000, 300), seq_lens=(1200, 300), hq=2, hkv=1, r=2048,
                                window=420),
    "bulk_bias_clamp_edge": W.small(q_lens=(700,), hq=2, hkv=1, r=520),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_matches_oracle(ink, name):
    (mx, mean), _, _ = _run(ink, CASES[name], seed=51)
    assert mx <= 1e-2


@pytest.mark.parametrize("name", ["ragged_two_seqs", "chunked_prefix", "gqa8"])
def test_prefill_bf16_output(ink, name):
    _run(ink, CASES[name], seed=52, out_dtype=torch.bfloat16)


def test_prefill_deterministic_and_page_order_free(ink):
    """Run twice: bit-identical.  Same logical K/V on shuffled pages: bit-identical."""
    spec = W.small(q_lens=(300, 100), hq=4, hkv=2, r=128, window=200)  # no random history
    st = _status()
    outs = []
    for identity in (True, False, False):
        g = W.make_case(spec, seed=53, device="cuda", identity_table=identity)
        gpu_sconv(ink, g, st)
        out, lse = gpu_attn(ink, g, st, decode=False)
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


def test_prefill_bad_block_reported(ink):
    spec = W.small(q_lens=(150,), hq=2, hkv=1)
    g = W.make_case(spec, seed=54, device="cuda")
    g.block_table = g.block_table.clone()
    g.block_table[0, 1] = g.num_blocks + 7
    st = _status()
    gpu_attn(ink, g, st, decode=False)
    torch.cuda.synchronize()
    assert int(st.item()) == 5  # INKLING_ERR_BAD_BLOCK


def test_prefill_host_argument_errors(ink):
    spec = W.small(q_lens=(10,), hq=4, hkv=2)
    g = W.make_case(spec, seed=55, device="cuda")
    out = torch.empty(10, 4, 128, device="cuda")
    with pytest.raises(ink.InklingError) as e:
        ink.rel_attn_prefill(g.q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens, g.seq_lens,
                             g.bias, scale=1.0, window=-1, max_q_len=10, out=out)
    assert e.value.code == 1
