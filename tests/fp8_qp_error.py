"""How large an error E4M3 tensor-core arithmetic (Q and P in FP8) would put into the
attention output, measured on the CPU against the fp64 oracle.

Test infrastructure, not part of the library: it decides whether an FP8 QK^T / PV kernel
(kind::f8f6f4) could meet the block's parity bar (max |err| <= 1e-2, mean |err| <= 1e-3 on
fp32 outputs).  The vLLM Day-0 Inkling blog's "Roadmap" plans FP8 for the global-attention
layers; this script measures what that costs in accuracy.

Setting: the FP8 KV cache (E4M3 codes, k_scale = v_scale = 0.0625, as the benchmark), so K
and V are exact in any FP8 kernel.  The reference is oracle.rel_attn_fp8 (fp64 over the same
codes).  The emulation follows a tiled FP8 kernel, in fp64 apart from the roundings it
names:
  - Q: one scale per query row and head, s_q = max|q| / 448, codes e4m3(q / s_q);
  - logits x_j = scale * s_q * k_scale * (q8 . k8_j) + b[h, min(p - j, R - 1)] (the FP8 MMA
    accumulates in fp32; its rounding is far below the FP8 input rounding and is left out);
  - online softmax over 128-key tiles from the diagonal backwards; P_j = exp(x_j - m_run);
  - P to E4M3 as e4m3(P * 448) (P <= 1, so the codes span the format's range), PV with
    those codes, O = sum_j (p8_j / 448) V_j / l with l the fp32 sum of P (variant "l=P") or
    of the rounded P (variant "l=p8").
Variants: Q in FP8 only (P kept bf16 as the shipped kernels do), P in FP8 only, both; and
Q and/or P as the sum of two E4M3 terms at one scale, x ~ (e4m3(x/s) + e4m3(x/s - e4m3(x/s))) s,
which two FP8 MMAs would accumulate into one fp32 result (K and V read as E4M3 directly).

python tests/fp8_qp_error.py [--workload 2|3] [--rows N] [--seed S]
"""
from __future__ import annotations

import argparse
import math
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads as W  # noqa: E402

KS = VS = 0.0625


def e4m3(x: np.ndarray) -> np.ndarray:
    """Round to the nearest E4M3 value (ties to even), saturating at +-448."""
    t = torch.from_numpy(np.clip(x, -448.0, 448.0).astype(np.float32))
    return t.to(torch.float8_e4m3fn).to(torch.float64).numpy()


def e4m3_split(x: np.ndarray, s: float) -> np.ndarray:
    """x as the sum of two E4M3 terms at scale s: a leading code and the code of its residual."""
    hi = e4m3(x / s)
    return (hi + e4m3(x / s - hi)) * s


def bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def emulate_row(q, kcodes, vcodes, bias_row, R, p, window, scale, q_fp8, p_fp8, l_from_p8,
                split=False):
    """One query row of one head: q [128] (bf16 values), kcodes/vcodes [L, 128] (E4M3
    values), keys 0..L-1 at positions 0..L-1, the query at position p."""
    lo = 0 if window <= 0 else max(0, p - window + 1)
    if q_fp8:
        s_q = np.abs(q).max() / 448.0
        if s_q <= 0:
            qq = q
        else:
            qq = e4m3_split(q, s_q) if split else e4m3(q / s_q) * s_q
    else:
        qq = q
    m, l = -math.inf, 0.0
    o = np.zeros(128)
    hi_tile = p // 128
    for kt in range(hi_tile, lo // 128 - 1, -1):
        j0, j1 = max(kt * 128, lo), min(kt * 128 + 128, p + 1)
        if j0 >= j1:
            continue
        k = kcodes[j0:j1] * KS
        d = p - np.arange(j0, j1)
        x = scale * (k @ qq) + bias_row[np.minimum(d, R - 1)]
        m_new = max(m, x.max())
        alpha = math.exp(m - m_new) if m > -math.inf else 0.0
        o *= alpha
        l *= alpha
        m = m_new
        pj = np.exp(x - m)
        if p_fp8:
            pq = e4m3_split(pj, 1.0 / 448.0) if split else e4m3(pj * 448.0) / 448.0
        else:
            pq = bf16(pj)
        o += pq @ (vcodes[j0:j1] * VS)
        l += pq.sum() if l_from_p8 else pj.sum()
    return o / l


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", type=int, default=2, choices=[1, 2, 3])
    ap.add_argument("--rows", type=int, default=48, help="sampled query rows (all heads each)")
    ap.add_argument("--heads", type=int, default=8, help="heads per sampled row")
    ap.add_argument("--seed", type=int, default=0)
    args = ap.parse_args()
    spec = W.config(args.workload)
    # one sequence of the workload is enough: every row's keys are its own sequence's
    spec = W.Spec(**{**spec.__dict__, "batch": 1, "q_lens": [spec.q_lens[0]],
                     "seq_lens": [spec.seq_lens[0]]})
    c = W.make_case(spec, seed=args.workload)
    kc = W.fp8_history(c.k_cache, KS)
    vc = W.fp8_history(c.v_cache, VS)
    st = c.state.clone()
    oracle.sconv_kv_fp8(c.k_raw, c.v_raw, c.w_k, c.w_v, st, c.cu_q_lens, c.slot_mapping, kc, vc,
                        KS, VS)
    n = spec.q_lens[0]
    rng = np.random.default_rng(args.seed)
    # rows with few keys (peaked softmax), rows at the window edge, seeded random rows
    rows = sorted(set(list(range(0, 16)) + list(range(n - 8, n)) +
                      ([4096 - 4 + i for i in range(8)] if spec.window else []) +
                      rng.integers(0, n, max(args.rows - 32, 0)).tolist()))
    ref, _ = oracle.rel_attn_fp8(c.q, kc, vc, KS, VS, c.block_table, c.cu_q_lens, c.seq_lens,
                                 c.bias, scale=spec.scale, window=spec.window, rows=rows)
    # logical K/V rows of the sequence, as E4M3 values
    f8 = lambda t: t.view(torch.float8_e4m3fn).to(torch.float64)
    pages = c.block_table[0, : (spec.seq_lens[0] + 127) // 128].long()
    heads = rng.choice(spec.hq, size=min(args.heads, spec.hq), replace=False)
    variants = {"Q fp8, P bf16": (True, False, False), "Q bf16, P fp8 (l=P)": (False, True, False),
                "Q bf16, P fp8 (l=p8)": (False, True, True), "Q fp8, P fp8 (l=p8)": (True, True, True),
                "Q bf16, P bf16 (shipped)": (False, False, False),
                "Q 2xfp8, P bf16": (True, False, False, True),
                "Q bf16, P 2xfp8 (l=P)": (False, True, False, True),
                "Q 2xfp8, P 2xfp8 (l=P)": (True, True, False, True)}
    errs = {k: [] for k in variants}
    qf = c.q.to(torch.float64).numpy()
    bias = c.bias.to(torch.float64).numpy()
    for h in heads:
        kvh = h // spec.group
        kk = f8(kc[pages, kvh]).reshape(-1, 128).numpy()
        vv = f8(vc[pages, kvh]).reshape(-1, 128).numpy()
        for i, t in enumerate(rows):
            p = spec.seq_lens[0] - n + t
            for name, v in variants.items():
                o = emulate_row(qf[t, h], kk, vv, bias[h], spec.r, p, spec.window, spec.scale, *v)
                errs[name].append(np.abs(o - ref[i, h]))
    print(f"workload {args.workload} ({spec.name}): {len(rows)} rows x {len(heads)} heads, "
          f"E4M3 cache, bar max 1e-2 / mean 1e-3")
    for name, e in errs.items():
        e = np.concatenate(e)
        print(f"  {name:26s} max |err| {e.max():.3e}   mean |err| {e.mean():.3e}   "
              f"{'within' if e.max() <= 1e-2 and e.mean() <= 1e-3 else 'OUTSIDE'} the bar")


if __name__ == "__main__":
    main()
