"""Parity at the five workloads' full sizes, through the same calls the benchmark times
(sconv into the paged cache, then prefill or split-KV decode), on sampled query rows the
fp64 oracle computes one by one: the first and last rows of a sequence, rows around the
window edge and around distance R (where the bias table starts to clamp), and seeded
random rows.  The cache pages and sconv state of the sampled sequences are compared in
full."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from harness import (assert_cache_matches, assert_state_matches, compare_out, gpu_attn,
                     gpu_sconv, run_oracle, snapshot)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ink():
    import relative_position_gqa_gb300 as m
    m._lib.load()
    return m


def _rows(snap, per_seq):
    """Snapshot token indices: per_seq(b_index, n) -> local rows of that sequence."""
    cu = snap.case.cu_q_lens.tolist()
    rows = []
    for i in range(len(snap.seqs)):
        n = cu[i + 1] - cu[i]
        rows += sorted({cu[i] + r for r in per_seq(i, n) if 0 <= r < n})
    return rows


def _check(ink, wl, seqs, per_seq, *, decode, variant=None, out_dtype=torch.float32, seed=None):
    spec = W.config(wl, variant=variant)
    g = W.make_case(spec, seed=wl if seed is None else seed, device="cuda")
    snap = snapshot(g, seqs)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_sconv(ink, g, st)
    out, lse = gpu_attn(ink, g, st, decode=decode, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, ink.status_string(int(st.item()))
    rows = _rows(snap, per_seq)
    kc, vc, state, ref, ref_lse = run_oracle(snap, rows=rows)
    assert_cache_matches(g.k_cache, kc, snap, 0)
    assert_cache_matches(g.v_cache, vc, snap, 1)
    assert_state_matches(g.state, state, snap)
    tok = snap.tok_index[torch.tensor(rows, dtype=torch.long)]
    return compare_out(out, lse, ref, ref_lse, tok)


def _rand(seed, n, k):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, max(n, 1), (k,), generator=g).tolist()


def test_tiny_prefill_all_rows(ink):
    _check(ink, 1, [0], lambda i, n: range(n), decode=False)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_swa_prefill_sampled(ink, out_dtype):
    edge = lambda i, n: (list(range(0, 40)) + list(range(n - 40, n)) +
                         list(range(4096 - 24, 4096 + 24)) + _rand(100 + i, n, 48))
    _check(ink, 2, [0, 3], edge, decode=False, out_dtype=out_dtype)


def test_full_prefill_64k_sampled(ink):
    rows = lambda i, n: (list(range(0, 24)) + list(range(n - 16, n)) +
                         list(range(8192 - 12, 8192 + 12)) + _rand(300, n, 16))
    _check(ink, 3, [0], rows, decode=False)


def _mtp_seqs(variant, k=8):
    """The shortest and the longest sequence and six seeded others (with the full layer's
    automatic split, the short ones run as one split and the long ones are split)."""
    lens = W.config(4, variant=variant).seq_lens
    pick = {min(range(64), key=lambda b: lens[b]), max(range(64), key=lambda b: lens[b])}
    g = torch.Generator().manual_seed(41)
    for b in torch.randperm(64, generator=g).tolist():
        if len(pick) >= k:
            break
        pick.add(b)
    return sorted(pick)


@pytest.mark.parametrize("variant", ["swa", "full", "swa_8k"])
def test_mtp_decode_sampled(ink, variant):
    spec = W.config(4, variant=variant)
    seqs = _mtp_seqs(variant)
    if variant == "full":
        plan = ink.decode_plan(spec.batch, spec.hq, spec.hkv, spec.max_q_len, spec.max_seq_len,
                               spec.window)
        span = plan["pages_per_split"] * 128
        split = [spec.seq_lens[b] > span for b in seqs]
        assert any(split) and not all(split)  # both kinds are checked
    _check(ink, 4, seqs, lambda i, n: range(n), decode=True, variant=variant)


@pytest.mark.parametrize("variant", ["n1", "n9"])
def test_decode_1m_sampled(ink, variant):
    """Every query row of the step (1 or 9 tokens x 64 heads)."""
    _check(ink, 5, [0], lambda i, n: range(n), decode=True, variant=variant)


# ------------------------------------------------------------- FP8 KV cache, full size ----
K_SCALE, V_SCALE = 0.0625, 0.0625  # the benchmark's scales


def _ordinal(codes: torch.Tensor) -> np.ndarray:
    b = codes.numpy().astype(np.int64)
    return np.where(b & 0x80, -(b & 0x7F), b & 0x7F)


def _check_fp8(ink, wl, seqs, per_seq, *, decode, variant=None):
    """The FP8 path at full size: history pages as E4M3 codes, the conv into E4M3 pages,
    then the FP8 decode or prefill.  The snapshot's conv codes are compared with the
    oracle's (adjacent codes only where the fp32 and fp64 sums straddle a midpoint), and
    the sampled rows with the oracle's attention over the GPU's codes."""
    spec = W.config(wl, variant=variant)
    g = W.make_case(spec, seed=wl, device="cuda")
    g.k_cache = W.fp8_history(g.k_cache, K_SCALE)
    g.v_cache = W.fp8_history(g.v_cache, V_SCALE)
    snap = snapshot(g, seqs)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ink.sconv_kv_fp8(g.k_raw, g.v_raw, g.w_k, g.w_v, g.state, g.cu_q_lens, g.slot_mapping,
                     g.k_cache, g.v_cache, k_scale=K_SCALE, v_scale=V_SCALE,
                     max_q_len=spec.max_q_len, dev_status=st)
    out = torch.full((spec.total_q, spec.hq, 128), float("nan"), device="cuda")
    lse = torch.full((spec.total_q, spec.hq), float("nan"), device="cuda")
    kw = dict(k_scale=K_SCALE, v_scale=V_SCALE, scale=spec.scale, window=spec.window,
              max_q_len=spec.max_q_len, max_seq_len=spec.max_seq_len, out=out, lse=lse,
              dev_status=st)
    fn = ink.rel_attn_decode_fp8 if decode else ink.rel_attn_prefill_fp8
    fn(g.q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens, g.seq_lens, g.bias, **kw)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, ink.status_string(int(st.item()))
    c = snap.case
    idx = snap.page_index.to(g.k_cache.device)
    gk, gv = g.k_cache.index_select(0, idx).cpu(), g.v_cache.index_select(0, idx).cpu()
    kc, vc, state = c.k_cache.clone(), c.v_cache.clone(), c.state.clone()
    oracle.sconv_kv_fp8(c.k_raw, c.v_raw, c.w_k, c.w_v, state, c.cu_q_lens, c.slot_mapping,
                        kc, vc, K_SCALE, V_SCALE)
    for got, want in ((gk, kc), (gv, vc)):
        d = np.abs(_ordinal(got) - _ordinal(want))
        assert d.max() <= 1 and (d > 0).mean() < 1e-3
    assert_state_matches(g.state, state, snap)
    rows = _rows(snap, per_seq)
    ref, ref_lse = oracle.rel_attn_fp8(c.q, gk, gv, K_SCALE, V_SCALE, c.block_table,
                                       c.cu_q_lens, c.seq_lens, c.bias, scale=spec.scale,
                                       window=spec.window, rows=rows)
    tok = snap.tok_index[torch.tensor(rows, dtype=torch.long)]
    return compare_out(out, lse, ref, ref_lse, tok)


def test_swa_prefill_fp8_sampled(ink):
    edge = lambda i, n: (list(range(0, 24)) + list(range(n - 24, n)) +
                         list(range(4096 - 16, 4096 + 16)) + _rand(120 + i, n, 32))
    _check_fp8(ink, 2, [0, 3], edge, decode=False)


@pytest.mark.parametrize("variant", ["swa", "full"])
def test_mtp_decode_fp8_sampled(ink, variant):
    _check_fp8(ink, 4, _mtp_seqs(variant), lambda i, n: range(n), decode=True, variant=variant)


@pytest.mark.parametrize("variant", ["n1", "n9"])
def test_decode_1m_fp8_sampled(ink, variant):
    _check_fp8(ink, 5, [0], lambda i, n: range(n), decode=True, variant=variant)
