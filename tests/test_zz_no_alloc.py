"""The allocation-free decode entry point, for callers that cannot allocate device memory
while they run (a runtime that reserves all device memory at start-up, or code called
from inside another framework's allocator).  Its split partials live in the library's
static device scratch; its output must match the workspace-based decode call's within
the parity tolerance, and the fp64 oracle's, on two calls in a row (the second reuses the
scratch the first left behind).  Collected last on purpose: it also runs after every
other GPU test."""
import pytest
import torch

import workloads as W
from harness import MAX_ABS, MEAN_ABS, LSE_ABS, compare_out, gpu_sconv, run_oracle, snapshot

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ink():
    import relative_position_gqa_gb300 as m
    m._lib.load()
    return m


# (q_lens, seq_lens, Hq, Hkv, R, window, num_splits): an explicit split count; the
# automatic split rule (the size query and the call's own plan must agree); and a sliding
# window wide enough that the automatic rule splits it too
CASES = {
    "explicit_5": ((9, 1, 9), (3000, 700, 2200), 8, 2, 1000, 0, 5),
    "auto": ((9, 1, 9), (9000, 700, 5000), 8, 2, 1000, 0, 0),
    "auto_window": ((9, 3, 9), (9000, 700, 5000), 8, 1, 6000, 4100, 0),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_noalloc_decode_matches_workspace_decode_and_oracle_twice(ink, name):
    q_lens, seq_lens, hq, hkv, r, window, splits = CASES[name]
    dev = torch.device("cuda")
    spec = W.small(q_lens=q_lens, seq_lens=seq_lens, hq=hq, hkv=hkv, r=r, window=window,
                   history_random=True, state_random=True)
    g = W.make_case(spec, seed=91, device=dev)
    snap = snapshot(g)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    gpu_sconv(ink, g, st)
    plan = ink.decode_plan(spec.batch, spec.hq, spec.hkv, 9, spec.max_seq_len, window, splits)
    assert plan["num_splits"] > 1  # the partials really pass through the scratch
    need = ink.decode_workspace_size(spec.batch, spec.hq, spec.hkv, 9, spec.max_seq_len,
                                     window, splits)
    assert 0 < need <= ink.decode_noalloc_capacity()
    kw = dict(scale=spec.scale, window=window, max_q_len=9, max_seq_len=spec.max_seq_len,
              num_splits=splits, dev_status=st)
    ref = torch.empty(spec.total_q, spec.hq, 128, device=dev)
    ref_lse = torch.empty(spec.total_q, spec.hq, device=dev)
    ink.rel_attn_decode(g.q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens, g.seq_lens,
                        g.bias, out=ref, lse=ref_lse, **kw)
    _, _, _, o_ref, o_lse = run_oracle(snap)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        ink.rel_attn_decode_noalloc(g.q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens,
                                    g.seq_lens, g.bias, out=out, lse=lse, **kw)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, ink.status_string(int(st.item()))
        assert torch.isfinite(out).all()
        d = (out - ref).abs()
        assert d.max().item() <= MAX_ABS and d.mean().item() <= MEAN_ABS
        assert (lse - ref_lse).abs().max().item() <= LSE_ABS
        compare_out(out, lse, o_ref, o_lse, snap.tok_index)


def test_noalloc_decode_rejects_requests_beyond_capacity(ink):
    dev = torch.device("cuda")
    spec = W.small(q_lens=(9,), seq_lens=(200,), hq=8, hkv=1, history_random=True)
    g = W.make_case(spec, seed=92, device=dev)
    cap = ink.decode_noalloc_capacity()
    # enough sequences x splits that the partials exceed the static scratch
    big_b = cap // (2 * 72 * 130 * 4) + 1
    need = ink.decode_workspace_size(big_b, 8, 1, 9, 1 << 20, 0, 2)
    assert need > cap
    cu = torch.arange(0, 9 * big_b + 1, 9, dtype=torch.int32, device=dev)[:big_b + 1]
    q = torch.zeros(9 * big_b, 8, 128, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ink.InklingError) as e:
        ink.rel_attn_decode_noalloc(q, g.k_cache, g.v_cache, g.block_table, cu,
                                    g.seq_lens.repeat(big_b), g.bias, scale=spec.scale,
                                    window=0, max_q_len=9, max_seq_len=1 << 20, num_splits=2,
                                    out=torch.empty(9 * big_b, 8, 128, device=dev))
    assert e.value.code == 7  # INKLING_ERR_WORKSPACE
    # the argument checks come before the capacity: a bad argument on the same oversized
    # request reports that argument, as the workspace entry point does
    with pytest.raises(ink.InklingError) as e:
        ink.rel_attn_decode_noalloc(q, g.k_cache, g.v_cache, g.block_table, cu,
                                    g.seq_lens.repeat(big_b), g.bias, scale=spec.scale,
                                    window=-1, max_q_len=9, max_seq_len=1 << 20, num_splits=2,
                                    out=torch.empty(9 * big_b, 8, 128, device=dev))
    assert e.value.code == 1  # INKLING_ERR_INVALID_ARG


def test_noalloc_decode_graph_replay(ink):
    """Captured into a CUDA graph (no allocation during the capture), the allocation-free
    decode replays bit-identically to the eager call, and a replay after new Q values are
    written into the captured buffer gives the eager call's new output."""
    spec = W.small(q_lens=(9, 9, 3, 1), seq_lens=(500, 700, 129, 1000), hq=8, hkv=1, r=64)
    c = W.make_case(spec, seed=23, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_sconv(ink, c, st)
    out = torch.empty(spec.total_q, spec.hq, 128, device="cuda")
    lse = torch.empty(spec.total_q, spec.hq, device="cuda")

    def call():
        ink.rel_attn_decode_noalloc(c.q, c.k_cache, c.v_cache, c.block_table, c.cu_q_lens,
                                    c.seq_lens, c.bias, scale=spec.scale, window=spec.window,
                                    max_q_len=spec.max_q_len, max_seq_len=spec.max_seq_len,
                                    out=out, lse=lse, num_splits=3, dev_status=st)
    call()
    torch.cuda.synchronize()
    ref, ref_lse = out.clone(), lse.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for _ in range(2):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32))
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
    gen = torch.Generator(device="cuda").manual_seed(98)
    c.q.copy_(torch.randn(c.q.shape, generator=gen, device="cuda").to(torch.bfloat16))
    call()
    torch.cuda.synchronize()
    ref2 = out.clone()
    out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int32), ref2.view(torch.int32))
