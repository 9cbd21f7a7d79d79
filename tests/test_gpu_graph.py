"""GPU: the attention calls captured into a CUDA graph replay bit-identically to the same
calls made eagerly.  Every launch of the library is a programmatic dependent launch, which
stream capture turns into graph edges; the graph reads the buffers it was captured with, so
new inputs written into them before a replay give the new outputs."""
import pytest
import torch

import workloads as W
from harness import gpu_sconv

pytestmark = pytest.mark.gpu

PREFILL = W.small(q_lens=(150, 37, 300), seq_lens=(150, 200, 600), hq=4, hkv=2, r=64,
                  window=100)
DECODE = W.small(q_lens=(9, 9, 3, 1), seq_lens=(500, 700, 129, 1000), hq=8, hkv=1, r=64)


@pytest.fixture(scope="module")
def ink():
    import relative_position_gqa_gb300 as m
    m._lib.load()
    return m


def _capture(fn):
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    return graph


def _replay_matches_eager(c, call, out, lse, st):
    """Eager result, then the captured call's replays: on the same inputs, and after new
    Q values are written into the captured buffer."""
    call()
    torch.cuda.synchronize()
    ref, ref_lse = out.clone(), lse.clone()
    graph = _capture(call)
    for _ in range(2):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32))
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
    gen = torch.Generator(device="cuda").manual_seed(99)
    c.q.copy_(torch.randn(c.q.shape, generator=gen, device="cuda").to(torch.bfloat16))
    call()
    torch.cuda.synchronize()
    ref2 = out.clone()
    assert not torch.equal(ref2, ref)
    out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out.view(torch.int32), ref2.view(torch.int32))


def test_prefill_graph_replay(ink):
    c = W.make_case(PREFILL, seed=21, device="cuda")
    spec = c.spec
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_sconv(ink, c, st)
    out = torch.empty(spec.total_q, spec.hq, 128, device="cuda")
    lse = torch.empty(spec.total_q, spec.hq, device="cuda")

    def call():
        ink.rel_attn_prefill(c.q, c.k_cache, c.v_cache, c.block_table, c.cu_q_lens, c.seq_lens,
                             c.bias, scale=spec.scale, window=spec.window,
                             max_q_len=spec.max_q_len, out=out, lse=lse, dev_status=st)
    _replay_matches_eager(c, call, out, lse, st)


def test_decode_graph_replay(ink):
    """The split decode (merge kernel included), with a workspace allocated before the
    capture."""
    c = W.make_case(DECODE, seed=22, device="cuda")
    spec = c.spec
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_sconv(ink, c, st)
    out = torch.empty(spec.total_q, spec.hq, 128, device="cuda")
    lse = torch.empty(spec.total_q, spec.hq, device="cuda")
    kw = dict(scale=spec.scale, window=spec.window, max_q_len=spec.max_q_len,
              max_seq_len=spec.max_seq_len, out=out, lse=lse, num_splits=3, dev_status=st)
    args = (c.q, c.k_cache, c.v_cache, c.block_table, c.cu_q_lens, c.seq_lens, c.bias)
    need = ink.decode_workspace_size(spec.batch, spec.hq, spec.hkv, spec.max_q_len,
                                     spec.max_seq_len, spec.window, 3)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")

    def call():
        ink.rel_attn_decode(*args, workspace=ws, **kw)
    _replay_matches_eager(c, call, out, lse, st)
