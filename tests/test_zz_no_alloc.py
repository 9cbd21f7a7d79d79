"""The allocation-free decode entry point, for callers that cannot allocate device memory
while they run (a runtime that reserves all device memory at start-up, or code called
from inside another framework's allocator).  Its split partials live in the library's
static device scratch; its output must match the workspace-based decode call's within
the parity tolerance, on two calls in a row (the second reuses the scratch the first left
behind).  Collected last on purpose: it also runs after every other GPU test."""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def test_noalloc_decode_matches_workspace_decode_twice():
    import relative_position_gqa_gb300 as ink
    ink._lib.load()
    dev = torch.device("cuda")
    spec = W.small(q_lens=(9, 1, 9), seq_lens=(3000, 700, 2200), hq=8, hkv=2, r=1000,
                   history_random=True, state_random=True)
    g = W.make_case(spec, seed=91, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ink.sconv_kv(g.k_raw, g.v_raw, g.w_k, g.w_v, g.state, g.cu_q_lens, g.slot_mapping,
                 g.k_cache, g.v_cache, max_q_len=9, dev_status=st)
    splits = 5  # several splits, so the partials really pass through the scratch
    need = ink.decode_workspace_size(spec.batch, spec.hq, spec.hkv, 9, spec.max_seq_len, 0,
                                     splits)
    assert 0 < need <= ink.decode_noalloc_capacity()
    kw = dict(scale=spec.scale, window=0, max_q_len=9, max_seq_len=spec.max_seq_len,
              num_splits=splits, dev_status=st)
    ref = torch.empty(spec.total_q, spec.hq, 128, device=dev)
    ref_lse = torch.empty(spec.total_q, spec.hq, device=dev)
    ink.rel_attn_decode(g.q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens, g.seq_lens,
                        g.bias, out=ref, lse=ref_lse, **kw)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        ink.rel_attn_decode_noalloc(g.q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens,
                                    g.seq_lens, g.bias, out=out, lse=lse, **kw)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, ink.status_string(int(st.item()))
        d = (out - ref).abs()
        assert torch.isfinite(out).all()
        assert d.max().item() <= 1e-2 and d.mean().item() <= 1e-3
        assert (lse - ref_lse).abs().max().item() <= 1e-3


def test_noalloc_decode_rejects_requests_beyond_capacity():
    import relative_position_gqa_gb300 as ink
    ink._lib.load()
    dev = torch.device("cuda")
    spec = W.small(q_lens=(9,), seq_lens=(200,), hq=8, hkv=1, history_random=True)
    g = W.make_case(spec, seed=92, device=dev)
    cap = ink.decode_noalloc_capacity()
    # enough sequences x splits that the partials exceed the static scratch
    big_b = cap // (2 * 72 * 130 * 4) + 1
    need = ink.decode_workspace_size(big_b, 8, 1, 9, 1 << 20, 0, 2)
    assert need > cap
    out = torch.empty(9, 8, 128, device=dev)
    cu = torch.arange(0, 9 * big_b + 1, 9, dtype=torch.int32, device=dev)[:big_b + 1]
    q = torch.zeros(9 * big_b, 8, 128, dtype=torch.bfloat16, device=dev)
    with pytest.raises(ink.InklingError) as e:
        ink.rel_attn_decode_noalloc(q, g.k_cache, g.v_cache, g.block_table, cu,
                                    g.seq_lens.repeat(big_b), g.bias, scale=spec.scale,
                                    window=0, max_q_len=9, max_seq_len=1 << 20, num_splits=2,
                                    out=torch.empty(9 * big_b, 8, 128, device=dev))
    assert e.value.code == 7  # INKLING_ERR_WORKSPACE
