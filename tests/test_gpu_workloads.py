"""Parity at the five workloads' full sizes, through the same calls the benchmark times
(sconv into the paged cache, then prefill or split-KV decode), on sampled query rows the
fp64 oracle computes one by one: the first and last rows of a sequence, rows around the
window edge and around distance R (where the bias table starts to clamp), and seeded
random rows.  The cache pages and sconv state of the sampled sequences are compared in
full."""
import pytest
import torch

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


@pytest.mark.parametrize("variant", ["swa", "full", "swa_8k"])
def test_mtp_decode_sampled(ink, variant):
    lens = W.config(4, variant=variant).seq_lens
    seqs = sorted({min(range(64), key=lambda b: lens[b]), max(range(64), key=lambda b: lens[b]), 17})
    _check(ink, 4, seqs, lambda i, n: range(n), decode=True, variant=variant)


@pytest.mark.parametrize("variant", ["n1", "n9"])
def test_decode_1m_sampled(ink, variant):
    _check(ink, 5, [0], lambda i, n: [0, n // 2, n - 1], decode=True, variant=variant)
