"""GPU parity of inkling_rel_attn_decode: paged KV, up to 9 query tokens per sequence (MTP
verify, vLLM Day-0 Inkling blog "Model Architecture / MTP"), split over pages and merged
("FA4 with sheared bias": num_splits), full or sliding window."""
import pytest
import torch

import workloads as W
from harness import compare_out, gpu_attn, gpu_sconv, permute_pages, run_oracle, snapshot

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ink():
    import relative_position_gqa_gb300 as m
    m._lib.load()
    return m


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


CASES = {
    "mtp9_gqa8": W.small(q_lens=(9, 9, 9), seq_lens=(1000, 129, 9), hq=8, hkv=1, r=300),
    "n1_gqa8": W.small(q_lens=(1, 1, 1, 1), seq_lens=(2000, 1, 128, 129), hq=16, hkv=2, r=500),
    "mixed_n": W.small(q_lens=(1, 5, 9, 2, 0), seq_lens=(700, 5, 300, 1200, 40), hq=8, hkv=2, r=1000),
    "window_300": W.small(q_lens=(9, 3, 9), seq_lens=(1500, 200, 301), hq=8, hkv=1, r=2000, window=300),
    "window_1": W.small(q_lens=(9, 4), seq_lens=(500, 4), hq=4, hkv=2, r=64, window=1),
    "g16_n8": W.small(q_lens=(8, 8), seq_lens=(900, 8), hq=16, hkv=1, r=128),
    "g1_n9": W.small(q_lens=(9,), seq_lens=(777,), hq=2, hkv=2, r=50),
    "g3_odd": W.small(q_lens=(7, 9), seq_lens=(400, 260), hq=9, hkv=3, r=8192),
}


def _run(ink, spec, seed, num_splits=0, out_dtype=torch.float32):
    g = W.make_case(spec, seed=seed, device="cuda")
    snap = snapshot(g)
    st = _status()
    gpu_sconv(ink, g, st)
    out, lse = gpu_attn(ink, g, st, decode=True, num_splits=num_splits, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, ink.status_string(int(st.item()))
    _, _, _, ref, ref_lse = run_oracle(snap)
    return compare_out(out, lse, ref, ref_lse, snap.tok_index), out


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_decode_matches_oracle(ink, name, num_splits):
    _run(ink, CASES[name], seed=61, num_splits=num_splits)


def test_decode_bf16_output(ink):
    _run(ink, CASES["mixed_n"], seed=62, out_dtype=torch.bfloat16, num_splits=2)


def test_split_count_invariance(ink):
    spec = W.small(q_lens=(9, 1), seq_lens=(3000, 2500), hq=8, hkv=1, r=4000)
    outs = [_run(ink, spec, seed=63, num_splits=n)[1] for n in (1, 2, 5, 24, 0)]
    for o in outs[1:]:
        d = (o - outs[0]).abs()
        assert d.max().item() <= 1e-2 and d.mean().item() <= 1e-3


def test_token_by_token_decode_equals_prefill(ink):
    """Prefill 200 tokens, then decode steps of 1, 9, 9, 1, 5 tokens (sconv each step)
    against one prefill of all 225 tokens."""
    total = 225
    spec = W.small(q_lens=(total,), seq_lens=(total,), hq=8, hkv=1, r=150, window=100)
    full = W.make_case(spec, seed=64, device="cuda")
    st = _status()
    ref_case = W.make_case(spec, seed=64, device="cuda")
    gpu_sconv(ink, ref_case, st)
    ref, ref_lse = gpu_attn(ink, ref_case, st, decode=False)
    start = 0
    for n in (200, 1, 9, 9, 1, 5):
        sl = slice(start, start + n)
        cu = torch.tensor([0, n], dtype=torch.int32, device="cuda")
        L = torch.tensor([start + n], dtype=torch.int32, device="cuda")
        ink.sconv_kv(full.k_raw[sl], full.v_raw[sl], full.w_k, full.w_v, full.state, cu,
                     full.slot_mapping[sl], full.k_cache, full.v_cache, max_q_len=n, dev_status=st)
        out = torch.empty(n, spec.hq, 128, device="cuda")
        lse = torch.empty(n, spec.hq, device="cuda")
        if n <= 9:
            ink.rel_attn_decode(full.q[sl], full.k_cache, full.v_cache, full.block_table, cu, L,
                                full.bias, scale=spec.scale, window=spec.window, max_q_len=n,
                                max_seq_len=start + n, out=out, lse=lse, dev_status=st)
        else:
            ink.rel_attn_prefill(full.q[sl], full.k_cache, full.v_cache, full.block_table, cu, L,
                                 full.bias, scale=spec.scale, window=spec.window, max_q_len=n,
                                 out=out, lse=lse, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        # both sides carry their own bf16 rounding of P: hold them to the parity bar
        d = (out - ref[sl]).abs()
        assert d.max().item() <= 1e-2 and d.mean().item() <= 1e-3
        assert (lse - ref_lse[sl]).abs().max().item() <= 1e-3
        start += n
    assert torch.equal(full.k_cache.view(torch.int16), ref_case.k_cache.view(torch.int16))
    # and the one-shot rows against the oracle
    snap = snapshot(W.make_case(spec, seed=64, device="cuda"))
    _, _, _, o_ref, o_lse = run_oracle(snap)
    compare_out(ref, ref_lse, o_ref, o_lse, snap.tok_index)


def test_decode_workspace_too_small(ink):
    spec = CASES["mtp9_gqa8"]
    g = W.make_case(spec, seed=65, device="cuda")
    need = ink.decode_workspace_size(spec.batch, spec.hq, spec.hkv, 9, spec.max_seq_len, 0, 4)
    assert need > 0
    ws = torch.empty(need - 1, dtype=torch.uint8, device="cuda")
    out = torch.empty(spec.total_q, spec.hq, 128, device="cuda")
    with pytest.raises(ink.InklingError) as e:
        ink.rel_attn_decode(g.q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens, g.seq_lens,
                            g.bias, scale=spec.scale, window=0, max_q_len=9,
                            max_seq_len=spec.max_seq_len, num_splits=4, out=out, workspace=ws)
    assert e.value.code == 7


def test_decode_rejects_more_than_nine_tokens(ink):
    spec = W.small(q_lens=(10,), seq_lens=(100,), hq=2, hkv=1)
    g = W.make_case(spec, seed=66, device="cuda")
    out = torch.empty(10, 2, 128, device="cuda")
    with pytest.raises(ink.InklingError) as e:
        ink.rel_attn_decode(g.q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens, g.seq_lens,
                            g.bias, scale=spec.scale, window=0, max_q_len=10, max_seq_len=100,
                            out=out)
    assert e.value.code == 1


@pytest.mark.parametrize("num_splits", [1, 3])
def test_decode_bad_block_reported(ink, num_splits):
    """A page id past the cache in a sequence's visible range comes back as
    INKLING_ERR_BAD_BLOCK, with no access made through it."""
    spec = CASES["mixed_n"]
    g = W.make_case(spec, seed=31, device="cuda")
    st = _status()
    gpu_sconv(ink, g, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    L = spec.seq_lens[3]
    g.block_table[3, (L - 1) // 128 - 2] = g.num_blocks  # inside sequence 3's range
    gpu_attn(ink, g, st, decode=True, num_splits=num_splits)
    torch.cuda.synchronize()
    assert int(st.item()) == 5  # INKLING_ERR_BAD_BLOCK


@pytest.mark.parametrize("name,num_splits", [("mixed_n", 0), ("mixed_n", 3), ("window_300", 0),
                                             ("g16_n8", 2)])
def test_decode_plan_matches_launch(ink, name, num_splits):
    """decode_plan's merge flag agrees with the workspace the call needs, and its split
    count with the split rule: ceil(pages / pages_per_split) splits cover the visible range."""
    spec = CASES[name]
    plan = ink.decode_plan(spec.batch, spec.hq, spec.hkv, spec.max_q_len, spec.max_seq_len,
                           spec.window, num_splits)
    need = ink.decode_workspace_size(spec.batch, spec.hq, spec.hkv, spec.max_q_len,
                                     spec.max_seq_len, spec.window, num_splits)
    assert plan["merge"] == (need > 0) == (plan["num_splits"] > 1)
    assert plan["ctas"] == plan["num_splits"] * spec.hkv * spec.batch
    if num_splits > 0:
        assert plan["num_splits"] <= num_splits
    pages = -(-spec.max_seq_len // 128)
    if spec.window > 0:
        pages = min(pages, (spec.window + spec.max_q_len - 1 + 127) // 128 + 1)
    assert plan["num_splits"] * plan["pages_per_split"] >= pages
    assert (plan["num_splits"] - 1) * plan["pages_per_split"] < pages


# long enough that the automatic rule splits (num_splits 0), with ragged page tails
ORDER_SPEC = {
    0: W.small(q_lens=(9, 1, 9, 5), seq_lens=(6000, 300, 4500, 129), hq=8, hkv=2, r=2000),
    1000: W.small(q_lens=(9, 1, 9, 5), seq_lens=(6000, 300, 4500, 129), hq=8, hkv=2, r=2000,
                  window=1000),
}


@pytest.mark.parametrize("window", sorted(ORDER_SPEC))
@pytest.mark.parametrize("num_splits", [1, 3, 0])
def test_decode_page_order_free_and_deterministic(ink, num_splits, window):
    """The same logical K/V on shuffled physical pages gives bit-identical outputs and
    LSE, and so does running the same call again (a race in the split or merge path
    would show up as a difference)."""
    spec = ORDER_SPEC[window]
    plan = ink.decode_plan(spec.batch, spec.hq, spec.hkv, spec.max_q_len, spec.max_seq_len,
                           window, num_splits)
    if num_splits != 1 and window == 0:
        assert plan["num_splits"] > 1
    base = W.make_case(spec, seed=67, device="cuda", identity_table=True)
    st = _status()
    results = []
    for g in (base, permute_pages(base, seed=5), permute_pages(base, seed=6)):
        gpu_sconv(ink, g, st)
        for _ in range(2):
            results.append(gpu_attn(ink, g, st, decode=True, num_splits=num_splits))
    torch.cuda.synchronize()
    assert int(st.item()) == 0, ink.status_string(int(st.item()))
    out0, lse0 = results[0]
    assert torch.isfinite(out0).all()
    for out, lse in results[1:]:
        assert torch.equal(out, out0) and torch.equal(lse, lse0)
