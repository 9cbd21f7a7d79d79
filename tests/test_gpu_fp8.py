"""GPU parity of the FP8 (E4M3) KV cache: inkling_sconv_kv_fp8 against the oracle's
conv into E4M3 codes, and inkling_rel_attn_decode_fp8 against the oracle's attention over
the same codes (vLLM Day-0 Inkling blog, "Roadmap": FP8 for the global-attention layers)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from harness import LSE_ABS, MAX_ABS, MEAN_ABS

pytestmark = pytest.mark.gpu

K_SCALE, V_SCALE = 0.0625, 0.03125  # powers of two: y * (1/scale) == y / scale exactly


@pytest.fixture(scope="module")
def ink():
    import relative_position_gqa_gb300 as m
    m._lib.load()
    return m


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _fp8_case(spec, seed, ks=K_SCALE, vs=V_SCALE):
    c = W.make_case(spec, seed=seed)  # CPU
    c.k_cache = W.fp8_history(c.k_cache, ks)
    c.v_cache = W.fp8_history(c.v_cache, vs)
    return c


def _ordinal(codes: torch.Tensor) -> np.ndarray:
    """E4M3 codes -> integers ordered like their values (adjacent values differ by 1)."""
    b = codes.numpy().astype(np.int64)
    return np.where(b & 0x80, -(b & 0x7F), b & 0x7F)


def _sconv_both(ink, c, ks=K_SCALE, vs=V_SCALE):
    g = c.to("cuda")
    st = _status()
    ink.sconv_kv_fp8(g.k_raw, g.v_raw, g.w_k, g.w_v, g.state, g.cu_q_lens, g.slot_mapping,
                     g.k_cache, g.v_cache, k_scale=ks, v_scale=vs, max_q_len=c.spec.max_q_len,
                     dev_status=st)
    kc, vc, state = c.k_cache.clone(), c.v_cache.clone(), c.state.clone()
    oracle.sconv_kv_fp8(c.k_raw, c.v_raw, c.w_k, c.w_v, state, c.cu_q_lens, c.slot_mapping,
                        kc, vc, ks, vs)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return g, kc, vc, state


@pytest.mark.parametrize("ks,vs", [(K_SCALE, V_SCALE), (0.1, 0.07)])
def test_sconv_fp8_codes_match_oracle(ink, ks, vs):
    """Codes agree except where the fp32 sum and the fp64 sum straddle a rounding
    midpoint: then they are adjacent codes, and that is rare."""
    spec = W.small(q_lens=(1, 9, 33, 64, 200), seq_lens=(5, 130, 40, 300, 260), hq=4, hkv=2,
                   history_random=True, state_random=True)
    c = _fp8_case(spec, seed=81, ks=ks, vs=vs)
    g, kc, vc, state = _sconv_both(ink, c, ks, vs)
    for got, want in ((g.k_cache.cpu(), kc), (g.v_cache.cpu(), vc)):
        d = np.abs(_ordinal(got) - _ordinal(want))
        assert d.max() <= 1
        assert (d > 0).mean() < 1e-3
    assert torch.equal(g.state.cpu().view(torch.int16), state.view(torch.int16))


def test_sconv_fp8_one_hot_taps_bit_exact(ink):
    spec = W.small(q_lens=(70, 2), seq_lens=(80, 2), hq=2, hkv=2, history_random=True,
                   state_random=True)
    c = _fp8_case(spec, seed=82)
    w = torch.tensor([0, 0, 1, 0], dtype=torch.float32).repeat(spec.channels, 1).contiguous()
    c.w_k, c.w_v = w, w.clone()
    g, kc, vc, _ = _sconv_both(ink, c)
    assert torch.equal(g.k_cache.cpu(), kc) and torch.equal(g.v_cache.cpu(), vc)


CASES = {
    "mtp9_gqa8": W.small(q_lens=(9, 9, 9), seq_lens=(1000, 129, 9), hq=8, hkv=1, r=300),
    "mixed_n": W.small(q_lens=(1, 5, 9, 2, 0), seq_lens=(700, 5, 300, 1200, 40), hq=8, hkv=2, r=1000),
    "window_300": W.small(q_lens=(9, 3, 9), seq_lens=(1500, 200, 301), hq=8, hkv=1, r=2000, window=300),
    "g1_n9": W.small(q_lens=(9,), seq_lens=(777,), hq=2, hkv=2, r=50),
}


def _decode_both(ink, spec, seed, num_splits=0, nan_tail=False):
    c = _fp8_case(spec, seed)
    if nan_tail:
        # stale slots past each sequence's end hold NaN codes: no output may see them
        for b, L in enumerate(spec.seq_lens):
            if L % 128:
                blk = int(c.block_table[b, (L - 1) // 128])
                c.k_cache[blk, :, L % 128:, :] = 0x7F
                c.v_cache[blk, :, L % 128:, :] = 0x7F
    g, kc, vc, _ = _sconv_both(ink, c)
    out = torch.empty(spec.total_q, spec.hq, 128, dtype=torch.float32, device="cuda")
    lse = torch.empty(spec.total_q, spec.hq, dtype=torch.float32, device="cuda")
    st = _status()
    ink.rel_attn_decode_fp8(g.q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens, g.seq_lens,
                            g.bias, k_scale=K_SCALE, v_scale=V_SCALE, scale=spec.scale,
                            window=spec.window, max_q_len=spec.max_q_len,
                            max_seq_len=spec.max_seq_len, out=out, lse=lse,
                            num_splits=num_splits, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, ink.status_string(int(st.item()))
    # the oracle reads the GPU's codes, so that only the attention is compared
    ref, ref_lse = oracle.rel_attn_fp8(c.q, g.k_cache.cpu(), g.v_cache.cpu(), K_SCALE, V_SCALE,
                                       c.block_table, c.cu_q_lens, c.seq_lens, c.bias,
                                       scale=spec.scale, window=spec.window)
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert err.max() <= MAX_ABS, f"max |err| {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"mean |err| {err.mean():.3e}"
    assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= LSE_ABS
    return out


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("num_splits", [0, 1, 3])
def test_decode_fp8_matches_oracle(ink, name, num_splits):
    _decode_both(ink, CASES[name], seed=83, num_splits=num_splits)


def test_decode_fp8_ignores_stale_nan_slots(ink):
    _decode_both(ink, CASES["mixed_n"], seed=84, num_splits=2, nan_tail=True)


@pytest.mark.parametrize("num_splits", [1, 3])
def test_decode_fp8_bad_block_reported(ink, num_splits):
    """A page id past the cache in a sequence's visible range comes back as
    INKLING_ERR_BAD_BLOCK: the converter warps check each id before they read the page."""
    spec = CASES["mixed_n"]
    c = _fp8_case(spec, seed=86)
    g, _, _, _ = _sconv_both(ink, c)
    L = spec.seq_lens[3]
    g.block_table[3, (L - 1) // 128 - 2] = g.k_cache.shape[0]  # inside sequence 3's range
    out = torch.empty(spec.total_q, spec.hq, 128, dtype=torch.float32, device="cuda")
    st = _status()
    ink.rel_attn_decode_fp8(g.q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens, g.seq_lens,
                            g.bias, k_scale=K_SCALE, v_scale=V_SCALE, scale=spec.scale,
                            window=0, max_q_len=spec.max_q_len, max_seq_len=spec.max_seq_len,
                            out=out, num_splits=num_splits, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 5  # INKLING_ERR_BAD_BLOCK


def test_decode_fp8_rejects_bad_scale(ink):
    spec = CASES["g1_n9"]
    c = _fp8_case(spec, seed=85).to("cuda")
    out = torch.empty(spec.total_q, spec.hq, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(ink.InklingError):
        ink.rel_attn_decode_fp8(c.q, c.k_cache, c.v_cache, c.block_table, c.cu_q_lens,
                                c.seq_lens, c.bias, k_scale=0.0, v_scale=1.0, scale=spec.scale,
                                window=0, max_q_len=9, max_seq_len=spec.max_seq_len, out=out)


PREFILL_CASES = {
    "ragged": W.small(q_lens=(150, 37, 0, 300), seq_lens=(150, 200, 40, 300), hq=4, hkv=2, r=64),
    "window_100": W.small(q_lens=(400, 129), seq_lens=(600, 129), hq=4, hkv=1, r=256, window=100),
    "chunked_gqa4": W.small(q_lens=(200, 9, 130), seq_lens=(457, 300, 130), hq=8, hkv=2, r=100),
}


def _prefill_both(ink, spec, seed, ks, vs, nan_tail=False, out_dtype=torch.float32):
    c = _fp8_case(spec, seed, ks, vs)
    if nan_tail:
        for b, L in enumerate(spec.seq_lens):
            if L % 128:
                blk = int(c.block_table[b, (L - 1) // 128])
                c.k_cache[blk, :, L % 128:, :] = 0x7F
                c.v_cache[blk, :, L % 128:, :] = 0x7F
    g, _, _, _ = _sconv_both(ink, c, ks, vs)
    out = torch.empty(spec.total_q, spec.hq, 128, dtype=out_dtype, device="cuda")
    lse = torch.empty(spec.total_q, spec.hq, dtype=torch.float32, device="cuda")
    st = _status()
    ink.rel_attn_prefill_fp8(g.q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens, g.seq_lens,
                             g.bias, k_scale=ks, v_scale=vs, scale=spec.scale,
                             window=spec.window, max_q_len=spec.max_q_len,
                             max_seq_len=spec.max_seq_len, out=out, lse=lse, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, ink.status_string(int(st.item()))
    ref, ref_lse = oracle.rel_attn_fp8(c.q, g.k_cache.cpu(), g.v_cache.cpu(), ks, vs,
                                       c.block_table, c.cu_q_lens, c.seq_lens, c.bias,
                                       scale=spec.scale, window=spec.window)
    return out, lse, ref, ref_lse


@pytest.mark.parametrize("name", sorted(PREFILL_CASES))
@pytest.mark.parametrize("ks,vs", [(K_SCALE, V_SCALE), (0.1, 0.07)])
def test_prefill_fp8_matches_oracle(ink, name, ks, vs):
    """Prefill over E4M3 caches (pages widened to bf16 exactly, k_scale in the logit scale,
    v_scale on the output) against the oracle's attention over the same codes."""
    out, lse, ref, ref_lse = _prefill_both(ink, PREFILL_CASES[name], 87, ks, vs)
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert err.max() <= MAX_ABS, f"max |err| {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"mean |err| {err.mean():.3e}"
    assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= LSE_ABS


def test_prefill_fp8_ignores_stale_nan_slots(ink):
    out, _, ref, _ = _prefill_both(ink, PREFILL_CASES["ragged"], 88, K_SCALE, V_SCALE,
                                   nan_tail=True)
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= MAX_ABS


def test_prefill_fp8_workspace_too_small(ink):
    spec = PREFILL_CASES["ragged"]
    c = _fp8_case(spec, seed=89).to("cuda")
    out = torch.empty(spec.total_q, spec.hq, 128, dtype=torch.float32, device="cuda")
    need = ink.prefill_fp8_workspace_size(spec.batch, spec.hkv, c.block_table.shape[1],
                                          spec.max_q_len, spec.max_seq_len, spec.window)
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ink.InklingError) as e:
        ink.rel_attn_prefill_fp8(c.q, c.k_cache, c.v_cache, c.block_table, c.cu_q_lens,
                                 c.seq_lens, c.bias, k_scale=K_SCALE, v_scale=V_SCALE,
                                 scale=spec.scale, window=0, max_q_len=spec.max_q_len,
                                 max_seq_len=spec.max_seq_len, out=out, workspace=ws)
    assert e.value.code == 7


@pytest.mark.parametrize("seed", range(300, 306))
def test_fp8_random_shapes(ink, seed):
    """Seeded random batches for the FP8 cache: the conv into E4M3 pages, then the decode
    (even seeds) or the prefill (odd seeds) against the oracle over the same codes."""
    import random
    rnd = random.Random(seed)
    decode = seed % 2 == 0
    hkv = rnd.choice([1, 2])
    g = rnd.choice([1, 4, 8])
    B = rnd.randint(1, 4)
    q_lens = [rnd.randint(1, 9) if decode else rnd.choice([1, 60, 130, 257]) for _ in range(B)]
    seq_lens = [n + rnd.choice([0, 3, 128, 400]) for n in q_lens]
    spec = W.small(name=f"fp8rand{seed}", q_lens=q_lens, seq_lens=seq_lens, hq=hkv * g, hkv=hkv,
                   r=rnd.choice([5, 200, 1024]), window=rnd.choice([0, 50]))
    ks, vs = rnd.choice([(K_SCALE, V_SCALE), (0.1, 0.07)])
    if decode:
        c = _fp8_case(spec, seed, ks, vs)
        g_, _, _, _ = _sconv_both(ink, c, ks, vs)
        out = torch.empty(spec.total_q, spec.hq, 128, dtype=torch.float32, device="cuda")
        st = _status()
        ink.rel_attn_decode_fp8(g_.q, g_.k_cache, g_.v_cache, g_.block_table, g_.cu_q_lens,
                                g_.seq_lens, g_.bias, k_scale=ks, v_scale=vs, scale=spec.scale,
                                window=spec.window, max_q_len=spec.max_q_len,
                                max_seq_len=spec.max_seq_len, out=out, num_splits=seed % 3,
                                dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, ink.status_string(int(st.item()))
        ref, _ = oracle.rel_attn_fp8(c.q, g_.k_cache.cpu(), g_.v_cache.cpu(), ks, vs,
                                     c.block_table, c.cu_q_lens, c.seq_lens, c.bias,
                                     scale=spec.scale, window=spec.window)
    else:
        out, _, ref, _ = _prefill_both(ink, spec, seed, ks, vs)
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert err.max() <= MAX_ABS, f"max |err| {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"mean |err| {err.mean():.3e}"


def test_prefill_fp8_bad_block_reported(ink):
    """A page id past the cache stops the widening of that page and is reported; the
    prefill then reads only pages of the pool."""
    spec = PREFILL_CASES["ragged"]
    c = _fp8_case(spec, seed=90).to("cuda")
    c.block_table[0, 0] = c.k_cache.shape[0] + 3
    out = torch.empty(spec.total_q, spec.hq, 128, dtype=torch.float32, device="cuda")
    st = _status()
    ink.rel_attn_prefill_fp8(c.q, c.k_cache, c.v_cache, c.block_table, c.cu_q_lens, c.seq_lens,
                             c.bias, k_scale=K_SCALE, v_scale=V_SCALE, scale=spec.scale,
                             window=0, max_q_len=spec.max_q_len, max_seq_len=spec.max_seq_len,
                             out=out, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 5  # INKLING_ERR_BAD_BLOCK


@pytest.mark.parametrize("num_splits", [1, 3, 0])
def test_decode_fp8_page_order_free_and_deterministic(ink, num_splits):
    """FP8 cache: shuffled physical pages and a second run give bit-identical outputs."""
    from harness import permute_pages
    spec = W.small(q_lens=(9, 1, 9, 5), seq_lens=(6000, 300, 4500, 129), hq=8, hkv=2, r=2000)
    base = W.make_case(spec, seed=87, device="cuda", identity_table=True)
    base.k_cache = W.fp8_history(base.k_cache, K_SCALE)
    base.v_cache = W.fp8_history(base.v_cache, V_SCALE)
    st = _status()
    results = []
    for g in (base, permute_pages(base, seed=5)):
        ink.sconv_kv_fp8(g.k_raw, g.v_raw, g.w_k, g.w_v, g.state, g.cu_q_lens, g.slot_mapping,
                         g.k_cache, g.v_cache, k_scale=K_SCALE, v_scale=V_SCALE,
                         max_q_len=spec.max_q_len, dev_status=st)
        for _ in range(2):
            out = torch.full((spec.total_q, spec.hq, 128), float("nan"), device="cuda")
            lse = torch.full((spec.total_q, spec.hq), float("nan"), device="cuda")
            ink.rel_attn_decode_fp8(g.q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens,
                                    g.seq_lens, g.bias, k_scale=K_SCALE, v_scale=V_SCALE,
                                    scale=spec.scale, window=0, max_q_len=spec.max_q_len,
                                    max_seq_len=spec.max_seq_len, out=out, lse=lse,
                                    num_splits=num_splits, dev_status=st)
            results.append((out, lse))
    torch.cuda.synchronize()
    assert int(st.item()) == 0, ink.status_string(int(st.item()))
    out0, lse0 = results[0]
    assert torch.isfinite(out0).all()
    for out, lse in results[1:]:
        assert torch.equal(out, out0) and torch.equal(lse, lse0)
