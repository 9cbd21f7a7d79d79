"""Shared plumbing for the GPU parity tests: run the CUDA path through the C ABI, run the
fp64 oracle on a CPU copy of the same seeded inputs, and compare.

Parity bars (fixed by the block's specification: bf16 inputs, fp32 accumulation):
  attention output (fp32 out mode): max |err| <= 1e-2 and mean |err| <= 1e-3;
  attention output (bf16 out mode): |err| <= max(1e-2, half a bf16 ulp of the oracle
    value) + 1e-3 (the output rounding alone can exceed 1e-2 for |o| >= 4);
  lse: |err| <= 1e-3;
  sconv output in the cache: |gpu - oracle| <= ulp_bf16(oracle) + 2^-21 * sum_j |w_j x_j|
    (the fp32 sum's rounding error; near-cancelling sums can differ by many ulps of their
    small result); every other cache slot and the sconv state bit-exact.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np
import torch

import oracle
import workloads as W

MAX_ABS = 1e-2
MEAN_ABS = 1e-3
LSE_ABS = 1e-3


@dataclasses.dataclass
class Snapshot:
    case: W.Case                # CPU, restricted to `seqs`, pages gathered in table order
    seqs: List[int]
    tok_index: torch.Tensor     # snapshot token -> original token index
    page_index: torch.Tensor    # snapshot page -> original physical page


def snapshot(case: W.Case, seqs: Optional[Sequence[int]] = None) -> Snapshot:
    """A CPU copy of `case` holding only sequences `seqs` (taken BEFORE the CUDA path
    touches the caches).  Pages are gathered into a compact cache and the block table /
    slot mapping re-pointed at them: storage only, no arithmetic of the block."""
    spec = case.spec
    seqs = list(range(spec.batch)) if seqs is None else list(seqs)
    cu = case.cu_q_lens.cpu().tolist()
    sl = case.seq_lens.cpu().tolist()
    bt = case.block_table.cpu()
    toks, pages, new_cu, tables = [], [], [0], []
    for b in seqs:
        toks.append(torch.arange(cu[b], cu[b + 1]))
        np_ = (sl[b] + 127) // 128
        tables.append(torch.arange(len(pages), len(pages) + np_, dtype=torch.int32))
        pages.extend(bt[b, :np_].tolist())
        new_cu.append(new_cu[-1] + cu[b + 1] - cu[b])
    tok = torch.cat(toks) if toks else torch.zeros(0, dtype=torch.long)
    page_idx = torch.tensor(pages, dtype=torch.long)
    max_blocks = max(1, max(len(t) for t in tables))
    table = torch.full((len(seqs), max_blocks), -1, dtype=torch.int32)
    for i, t in enumerate(tables):
        table[i, :len(t)] = t
    remap = torch.full((case.num_blocks,), -1, dtype=torch.long)
    remap[page_idx] = torch.arange(len(pages))
    dev = case.q.device
    slots = case.slot_mapping.index_select(0, tok.to(dev)).cpu()
    new_slots = torch.where(slots >= 0, remap[slots.clamp_min(0) // 128] * 128 + slots.clamp_min(0) % 128,
                            torch.full_like(slots, -1))
    sub_spec = dataclasses.replace(spec, batch=len(seqs), q_lens=[spec.q_lens[b] for b in seqs],
                                   seq_lens=[spec.seq_lens[b] for b in seqs])
    sel = lambda t: t.index_select(0, tok.to(dev)).cpu()
    pg = lambda t: t.index_select(0, page_idx.to(dev)).cpu()
    sub = W.Case(spec=sub_spec, q=sel(case.q), k_raw=sel(case.k_raw), v_raw=sel(case.v_raw),
                 w_k=case.w_k.cpu(), w_v=case.w_v.cpu(), bias=case.bias.cpu(),
                 state=case.state.index_select(0, torch.tensor(seqs, device=dev)).cpu(),
                 cu_q_lens=torch.tensor(new_cu, dtype=torch.int32),
                 seq_lens=torch.tensor([sl[b] for b in seqs], dtype=torch.int32),
                 block_table=table, slot_mapping=new_slots, k_cache=pg(case.k_cache),
                 v_cache=pg(case.v_cache))
    return Snapshot(case=sub, seqs=seqs, tok_index=tok, page_index=page_idx)


def permute_pages(case: W.Case, seed: int) -> W.Case:
    """The same logical K/V on other physical pages: page j of `case` moves to page
    perm[j], and the block table and slot mapping follow it.  Storage only: every
    sequence sees the same keys and values in the same logical order."""
    dev = case.k_cache.device
    nb = case.num_blocks
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(seed)).to(dev)
    k = torch.empty_like(case.k_cache)
    v = torch.empty_like(case.v_cache)
    k[perm] = case.k_cache
    v[perm] = case.v_cache
    bt = case.block_table
    table = torch.where(bt >= 0, perm[bt.clamp_min(0).long()].to(torch.int32), bt)
    sm = case.slot_mapping
    slots = torch.where(sm >= 0, perm[(sm.clamp_min(0) // 128)] * 128 + sm.clamp_min(0) % 128, sm)
    return dataclasses.replace(case, k_cache=k, v_cache=v, block_table=table.contiguous(),
                               slot_mapping=slots.contiguous(), q=case.q.clone(),
                               k_raw=case.k_raw.clone(), v_raw=case.v_raw.clone(),
                               state=case.state.clone())


def run_oracle(snap: Snapshot, rows: Optional[Sequence[int]] = None):
    """Oracle sconv into the snapshot's caches, then attention rows (snapshot indices)."""
    c = snap.case
    kc, vc, st = c.k_cache.clone(), c.v_cache.clone(), c.state.clone()
    oracle.sconv_kv(c.k_raw, c.v_raw, c.w_k, c.w_v, st, c.cu_q_lens, c.slot_mapping, kc, vc)
    out, lse = oracle.rel_attn(c.q, kc, vc, c.block_table, c.cu_q_lens, c.seq_lens, c.bias,
                               scale=c.spec.scale, window=c.spec.window, rows=rows)
    return kc, vc, st, out, lse


def gpu_sconv(ink, g: W.Case, status):
    ink.sconv_kv(g.k_raw, g.v_raw, g.w_k, g.w_v, g.state, g.cu_q_lens, g.slot_mapping,
                 g.k_cache, g.v_cache, max_q_len=g.spec.max_q_len, dev_status=status)


def gpu_attn(ink, g: W.Case, status, *, decode: bool, out_dtype=torch.float32, lse=True,
             num_splits=0, window=None):
    spec = g.spec
    out = torch.full((spec.total_q, spec.hq, 128), float("nan"), dtype=out_dtype, device=g.q.device)
    lse_t = torch.full((spec.total_q, spec.hq), float("nan"), dtype=torch.float32,
                       device=g.q.device) if lse else None
    w = spec.window if window is None else window
    if decode:
        ink.rel_attn_decode(g.q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens, g.seq_lens,
                            g.bias, scale=spec.scale, window=w, max_q_len=spec.max_q_len,
                            max_seq_len=spec.max_seq_len, num_splits=num_splits, out=out,
                            lse=lse_t, dev_status=status)
    else:
        ink.rel_attn_prefill(g.q, g.k_cache, g.v_cache, g.block_table, g.cu_q_lens,
                             g.seq_lens, g.bias, scale=spec.scale, window=w,
                             max_q_len=spec.max_q_len, out=out, lse=lse_t, dev_status=status)
    return out, lse_t


def _order_key(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> integers ordered like the values (adjacent values differ by 1)."""
    b = bits.astype(np.int64) & 0xFFFF
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _sconv_magnitude(c: W.Case, which: int) -> torch.Tensor:
    """S[t, c] = sum_j |w[c, j]| * |x~[t + j, c]| for every new token (snapshot order):
    the scale of the fp32 rounding error of the conv sum."""
    w = (c.w_k if which == 0 else c.w_v).abs().float()
    raw = (c.k_raw if which == 0 else c.v_raw).float().abs()
    cu = c.cu_q_lens.tolist()
    out = []
    for b in range(len(cu) - 1):
        n = cu[b + 1] - cu[b]
        ext = torch.cat([c.state[b, which].float().abs(), raw[cu[b]:cu[b + 1]]])
        acc = torch.zeros(n, ext.shape[1])
        for j in range(4):
            acc += w[:, j] * ext[j:j + n]
        out.append(acc)
    return torch.cat(out) if out else torch.zeros(0, w.shape[0])


def assert_cache_matches(gpu_cache: torch.Tensor, ora_cache: torch.Tensor, snap: Snapshot,
                         which: int):
    """The snapshot's pages of the GPU cache vs the oracle's.

    Slots of the new tokens hold the conv output: the GPU sums four products in fp32
    (four roundings, |error| <= 4 * 2^-24 * S with S = sum |w x|), the oracle in fp64, and
    each result is rounded once to bf16, so |gpu - oracle| <= ulp_bf16(oracle) + 2^-21 * S.
    Every other slot must be untouched: bit-exact."""
    c = snap.case
    g = gpu_cache.index_select(0, snap.page_index.to(gpu_cache.device)).cpu()
    o = ora_cache.clone()
    slots = c.slot_mapping
    keep = slots >= 0
    blk, off = slots[keep] // 128, slots[keep] % 128
    n = int(keep.sum())
    gv = g[blk, :, off, :].reshape(n, -1).double()
    ov = o[blk, :, off, :].reshape(n, -1).double()
    S = _sconv_magnitude(c, which)[keep].double()
    ulp = torch.exp2(torch.floor(torch.log2(ov.abs().clamp_min(2.0 ** -126))) - 7)
    bad = (gv - ov).abs() > ulp + 2.0 ** -21 * S
    assert not bad.any(), f"{int(bad.sum())} conv outputs outside the fp32 rounding bound"
    differ = float((gv != ov).double().mean()) if n else 0.0
    assert differ < 1e-3, f"{differ:.2e} of conv outputs differ from the oracle"
    # everything that is not a new token's slot: bit-exact
    g[blk, :, off, :] = 0
    o[blk, :, off, :] = 0
    assert torch.equal(g.view(torch.int16), o.view(torch.int16)), "untouched cache slots differ"
    return differ


def assert_state_matches(gpu_state: torch.Tensor, ora_state: torch.Tensor, snap: Snapshot):
    g = gpu_state.index_select(0, torch.tensor(snap.seqs, device=gpu_state.device))
    assert np.array_equal(bf16_bits(g), bf16_bits(ora_state)), "sconv state differs"


def compare_out(gpu_out: torch.Tensor, gpu_lse: Optional[torch.Tensor], ref: np.ndarray,
                ref_lse: np.ndarray, tok: torch.Tensor):
    """gpu_out rows at original token indices `tok` vs the oracle rows."""
    got = gpu_out.index_select(0, tok.to(gpu_out.device)).double().cpu().numpy()
    assert np.isfinite(got).all(), "non-finite output"
    err = np.abs(got - ref)
    if gpu_out.dtype == torch.float32:
        assert err.max() <= MAX_ABS, f"max |err| {err.max():.3e}"
        assert err.mean() <= MEAN_ABS, f"mean |err| {err.mean():.3e}"
    else:
        half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 8)
        bound = np.maximum(MAX_ABS, half_ulp) + 1e-3
        assert (err <= bound).all(), f"bf16 out: worst excess {(err - bound).max():.3e}"
        assert err.mean() <= MEAN_ABS, f"mean |err| {err.mean():.3e}"
    if gpu_lse is not None:
        gl = gpu_lse.index_select(0, tok.to(gpu_lse.device)).double().cpu().numpy()
        lerr = np.abs(gl - ref_lse)
        assert lerr.max() <= LSE_ABS, f"lse max |err| {lerr.max():.3e}"
    return float(err.max()), float(err.mean())
