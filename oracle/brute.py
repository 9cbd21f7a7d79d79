"""Pure-Python brute force of the relative-bias GQA attention and the sconv, for tiny
inputs only.  TEST INFRASTRUCTURE ONLY.

A second statement of the same definitions as oracle.c, written with plain loops,
`math.exp` and Python floats, over *logical* (unpaged) keys, so that it shares neither
code nor storage conventions with the C oracle:

  logit(q_row, key j) = scale * <q, k_j> + bias[h][min(p - j, R - 1)]
  allowed iff 0 <= p - j and (window == 0 or p - j <= window - 1)
  out = sum_j exp(logit_j) v_j / sum_j exp(logit_j)

(the learned relative-position term on the pre-softmax logits is the Inkling "relative
attention" of the vLLM Day-0 blog, "Model Architecture / Attention"; the table form is
this library's reading).
"""
from __future__ import annotations

import math
from typing import List, Sequence


def attention_row(q: Sequence[float], keys: Sequence[Sequence[float]],
                  values: Sequence[Sequence[float]], bias_row: Sequence[float], p: int,
                  scale: float, window: int):
    """One query row at absolute position p over logical keys 0..len(keys)-1.

    Returns (out vector, natural-log sum of exp of the allowed logits)."""
    R = len(bias_row)
    logits = []
    for j in range(len(keys)):
        dist = p - j
        if dist < 0:
            continue
        if window and dist > window - 1:
            continue
        dot = 0.0
        for a, b in zip(q, keys[j]):
            dot += a * b
        logits.append((j, scale * dot + bias_row[min(dist, R - 1)]))
    top = max(s for _, s in logits)
    weights = [(j, math.exp(s - top)) for j, s in logits]
    z = sum(w for _, w in weights)
    out = [0.0] * len(values[0])
    for j, w in weights:
        for d, v in enumerate(values[j]):
            out[d] += w * v
    return [o / z for o in out], top + math.log(z)


def sconv_rows(history: Sequence[Sequence[float]], new_rows: Sequence[Sequence[float]],
               taps: Sequence[Sequence[float]]) -> List[List[float]]:
    """Causal depthwise conv, window 4: y[t][c] = sum_j taps[c][j] * x~[t + j][c] with
    x~ = history (3 rows, oldest first) followed by the new rows.  Unrounded."""
    ext = [list(r) for r in history] + [list(r) for r in new_rows]
    out = []
    for t in range(len(new_rows)):
        row = []
        for c in range(len(taps)):
            acc = 0.0
            for j in range(4):
                acc += taps[c][j] * ext[t + j][c]
            row.append(acc)
        out.append(row)
    return out
