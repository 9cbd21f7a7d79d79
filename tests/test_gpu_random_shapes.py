"""GPU parity on seeded random shapes: batches of ragged sequences with cached prefixes,
random GQA groupings, bias-table lengths and windows, for the prefill and for the decode
(one to nine new tokens), each against the fp64 oracle.  The shapes stay small enough for
the oracle; the draw is seeded, so a failure names a reproducible case."""
import random

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


def _spec(seed: int, decode: bool) -> W.Spec:
    rnd = random.Random(seed)
    hkv = rnd.choice([1, 2, 3])
    g = rnd.choice([1, 2, 4, 8] if decode else [1, 2, 3, 4, 8])
    B = rnd.randint(1, 6)
    q_lens, seq_lens = [], []
    for _ in range(B):
        n = rnd.randint(0, 9) if decode else rnd.choice([0, 1, 17, 128, 129, 200, 300])
        L = n + rnd.choice([0, 0, 5, 127, 128, 260, 700])
        q_lens.append(n)
        seq_lens.append(max(L, n))
    if decode and g * max(q_lens) > 128:
        g = 8
        q_lens = [min(n, 128 // g) for n in q_lens]
    r = rnd.choice([1, 3, 64, 300, 1024])
    window = rnd.choice([0, 0, 1, 100, 257])
    return W.small(name=f"rand{seed}", q_lens=q_lens, seq_lens=seq_lens, hq=hkv * g, hkv=hkv,
                   r=r, window=window)


def _check(ink, spec, seed, decode, num_splits=0):
    g = W.make_case(spec, seed=seed, device="cuda")
    snap = snapshot(g)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gpu_sconv(ink, g, st)
    out, lse = gpu_attn(ink, g, st, decode=decode, num_splits=num_splits)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, ink.status_string(int(st.item()))
    _, _, _, ref, ref_lse = run_oracle(snap)
    compare_out(out, lse, ref, ref_lse, snap.tok_index)


@pytest.mark.parametrize("seed", range(100, 112))
def test_prefill_random_shapes(ink, seed):
    _check(ink, _spec(seed, decode=False), seed, decode=False)


@pytest.mark.parametrize("seed", range(200, 212))
def test_decode_random_shapes(ink, seed):
    _check(ink, _spec(seed, decode=True), seed, decode=True, num_splits=seed % 4)


def test_many_sequences(ink):
    """Hundreds of sequences in one call (grid dimension over sequences, split partials for
    each): decode with 1-9 new tokens on short histories."""
    rnd = random.Random(7)
    q_lens = [rnd.randint(0, 9) for _ in range(400)]
    seq_lens = [n + rnd.randint(0, 300) for n in q_lens]
    spec = W.small(name="many", q_lens=q_lens, seq_lens=seq_lens, hq=8, hkv=1, r=200)
    _check(ink, spec, 7, decode=True, num_splits=2)
