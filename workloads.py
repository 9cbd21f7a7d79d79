"""Seeded synthetic inputs for the Inkling attention block.

This module only draws random numbers and lays them out in the storage formats the
library and the oracle both accept (packed query rows, paged K/V cache, block table,
slot mapping).  It holds none of the block's arithmetic: no convolution, no logits,
no softmax.  Both the CUDA path's tests/bench and the fp64 oracle take their inputs
from here.

Shapes follow the five workloads of the attention block (head size 128, paged KV with
128-token pages, a per-head relative-bias table of length R):

  tiny_prefill     B=1,  S=256,    Hq=4,  Hkv=1, full causal,   R=512,  bias N(0,1)
  swa_prefill      B=4,  S=8192,   Hq=32, Hkv=4, window 4096,   R=8192, bias N(0,0.5)
  full_prefill_64k B=1,  S=65536,  Hq=64, Hkv=8, full causal,   R=8192, Q pre-scaled by 1/sqrt(128)
  mtp_decode       B=64, n=9,      Hq=32, Hkv=4, L ~ U[4096, 131072], window 4096 or full, R=8192
  decode_1m        B=1,  n=1 or 9, Hq=64, Hkv=8, L = 1,048,576, full causal, R=8192

Random-number recipe (all normal draws are float32 then rounded to the stored dtype):
  Q, raw K, raw V ~ N(0,1) bf16; sconv taps ~ N(0,0.5) fp32 [C,4] for K and for V;
  bias ~ N(0, bias_std) fp32 [Hq,R]; decode history (already-convolved K/V in the
  pages) ~ N(0,1) bf16; decode sconv state rows ~ N(0,1) bf16; prefill starts from a
  zero sconv state (fresh sequence).  Physical pages are a seeded random permutation.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

HEAD_DIM = 128
BLOCK = 128
SCONV_W = 4


@dataclasses.dataclass
class Spec:
    name: str
    batch: int
    hq: int
    hkv: int
    r: int
    window: int                      # 0 = full causal
    bias_std: float
    q_lens: Sequence[int]            # new (query) tokens per sequence
    seq_lens: Sequence[int]          # KV length per sequence, new tokens included
    q_prescale: float = 1.0          # multiply Q by this before rounding to bf16
    scale: float = 1.0 / math.sqrt(HEAD_DIM)
    w_std: float = 0.5
    history_random: bool = False     # fill pages before the new tokens with N(0,1)
    state_random: bool = False       # random sconv state rows (a continuing sequence)
    spare_blocks: int = 0

    @property
    def group(self) -> int:
        return self.hq // self.hkv

    @property
    def channels(self) -> int:
        return self.hkv * HEAD_DIM

    @property
    def total_q(self) -> int:
        return int(sum(self.q_lens))

    @property
    def max_q_len(self) -> int:
        return int(max(self.q_lens)) if len(self.q_lens) else 0

    @property
    def max_seq_len(self) -> int:
        return int(max(self.seq_lens)) if len(self.seq_lens) else 0


def _prefill(name, B, S, hq, hkv, r, window, bias_std, q_prescale=1.0, scale=None):
    return Spec(name=name, batch=B, hq=hq, hkv=hkv, r=r, window=window, bias_std=bias_std,
                q_lens=[S] * B, seq_lens=[S] * B, q_prescale=q_prescale,
                scale=(1.0 / math.sqrt(HEAD_DIM)) if scale is None else scale)


def config(n: int, *, variant: Optional[str] = None) -> Spec:
    """The five workloads.  `variant` picks the sliding/full half of the MTP decode
    workload ("swa" | "full" | "swa_8k") and the 1- or 9-token form of the 1M decode
    ("n1" | "n9" | "n1_256k" | "n9_256k")."""
    if n == 1:
        return _prefill("tiny_prefill", 1, 256, 4, 1, 512, 0, 1.0)
    if n == 2:
        return _prefill("swa_prefill", 4, 8192, 32, 4, 8192, 4096, 0.5)
    if n == 3:
        return _prefill("full_prefill_64k", 1, 65536, 64, 8, 8192, 0, 0.5,
                        q_prescale=1.0 / math.sqrt(HEAD_DIM), scale=1.0)
    if n == 4:
        # swa_8k: the sliding-window half with contexts in [4096, 8192] (the same 33-34
        # visible pages per sequence, under 1 GB of cache), small enough for multi-pass
        # profiler captures of the same kernel launch
        g = torch.Generator().manual_seed(4)
        hi = 8192 if variant == "swa_8k" else 131072
        lens = torch.randint(4096, hi + 1, (64,), generator=g).tolist()
        window = 0 if variant == "full" else 4096
        tag = "full" if window == 0 else ("swa_8k" if variant == "swa_8k" else "swa")
        return Spec(name=f"mtp_decode_{tag}", batch=64, hq=32,
                    hkv=4, r=8192, window=window, bias_std=0.5, q_lens=[9] * 64,
                    seq_lens=lens, history_random=True, state_random=True)
    if n == 5:
        # n1 / n9: the 1M-token sequence; n1_256k / n9_256k: a quarter of it (1 GB of K/V),
        # small enough for multi-pass profiler captures of the same kernel
        nq = 1 if variant in (None, "n1", "n1_256k") else 9
        L = (1 << 18) if variant in ("n1_256k", "n9_256k") else (1 << 20)
        tag = "256k" if L == (1 << 18) else "1m"
        return Spec(name=f"decode_{tag}_n{nq}", batch=1, hq=64, hkv=8, r=8192, window=0,
                    bias_std=0.5, q_lens=[nq], seq_lens=[L], history_random=True,
                    state_random=True)
    raise ValueError(f"no workload {n}")


@dataclasses.dataclass
class Case:
    spec: Spec
    q: torch.Tensor            # [T, Hq, 128] bf16
    k_raw: torch.Tensor        # [T, C] bf16 (pre-sconv)
    v_raw: torch.Tensor        # [T, C] bf16
    w_k: torch.Tensor          # [C, 4] fp32
    w_v: torch.Tensor          # [C, 4] fp32
    bias: torch.Tensor         # [Hq, R] fp32
    state: torch.Tensor        # [B, 2, 3, C] bf16 (oldest row first; index 0 = K, 1 = V)
    cu_q_lens: torch.Tensor    # [B+1] int32
    seq_lens: torch.Tensor     # [B] int32
    block_table: torch.Tensor  # [B, max_blocks] int32, -1 = unused
    slot_mapping: torch.Tensor # [T] int64
    k_cache: torch.Tensor      # [NB, Hkv, 128, 128] bf16
    v_cache: torch.Tensor      # [NB, Hkv, 128, 128] bf16

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    def to(self, device) -> "Case":
        kw = {f.name: getattr(self, f.name) for f in dataclasses.fields(self)}
        for k, v in kw.items():
            if isinstance(v, torch.Tensor):
                kw[k] = v.to(device)
        return Case(**kw)


def _randn(shape, gen, device, std=1.0, dtype=torch.bfloat16):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def make_case(spec: Spec, seed: int, device="cpu", *, table_seed: Optional[int] = None,
              identity_table: bool = False) -> Case:
    """Draw one seeded input set for `spec` on `device`.

    The page permutation uses its own CPU generator (`table_seed`, default seed+1000),
    so the block table is the same whichever device draws the tensors."""
    device = torch.device(device)
    gen = torch.Generator(device=device).manual_seed(seed)
    B, hq, hkv, C = spec.batch, spec.hq, spec.hkv, spec.channels
    q_lens = [int(x) for x in spec.q_lens]
    seq_lens = [int(x) for x in spec.seq_lens]
    assert len(q_lens) == B and len(seq_lens) == B
    assert all(0 <= n <= L for n, L in zip(q_lens, seq_lens))
    T = sum(q_lens)

    q = _randn((T, hq, HEAD_DIM), gen, device, dtype=torch.float32)
    if spec.q_prescale != 1.0:
        q.mul_(spec.q_prescale)
    q = q.to(torch.bfloat16)
    k_raw = _randn((T, C), gen, device)
    v_raw = _randn((T, C), gen, device)
    w_k = _randn((C, SCONV_W), gen, device, std=spec.w_std, dtype=torch.float32)
    w_v = _randn((C, SCONV_W), gen, device, std=spec.w_std, dtype=torch.float32)
    bias = _randn((hq, spec.r), gen, device, std=spec.bias_std, dtype=torch.float32)
    if spec.state_random:
        state = _randn((B, 2, SCONV_W - 1, C), gen, device)
    else:
        state = torch.zeros((B, 2, SCONV_W - 1, C), dtype=torch.bfloat16, device=device)

    pages = [(L + BLOCK - 1) // BLOCK for L in seq_lens]
    nb = sum(pages) + spec.spare_blocks
    max_blocks = max(max(pages) if pages else 1, 1)
    tgen = torch.Generator().manual_seed(seed + 1000 if table_seed is None else table_seed)
    perm = torch.arange(nb) if identity_table else torch.randperm(nb, generator=tgen)
    table = torch.full((B, max_blocks), -1, dtype=torch.int32)
    off = 0
    for b, p in enumerate(pages):
        table[b, :p] = perm[off:off + p].to(torch.int32)
        off += p

    cu = [0]
    for n in q_lens:
        cu.append(cu[-1] + n)
    slots = torch.empty(T, dtype=torch.int64)
    for b in range(B):
        n, L = q_lens[b], seq_lens[b]
        pos = torch.arange(L - n, L, dtype=torch.int64)
        slots[cu[b]:cu[b + 1]] = table[b].to(torch.int64)[pos // BLOCK] * BLOCK + pos % BLOCK

    if spec.history_random:
        k_cache = _randn((nb, hkv, BLOCK, HEAD_DIM), gen, device)
        v_cache = _randn((nb, hkv, BLOCK, HEAD_DIM), gen, device)
    else:
        k_cache = torch.zeros((nb, hkv, BLOCK, HEAD_DIM), dtype=torch.bfloat16, device=device)
        v_cache = torch.zeros((nb, hkv, BLOCK, HEAD_DIM), dtype=torch.bfloat16, device=device)

    return Case(spec=spec, q=q, k_raw=k_raw, v_raw=v_raw, w_k=w_k, w_v=w_v, bias=bias,
                state=state,
                cu_q_lens=torch.tensor(cu, dtype=torch.int32, device=device),
                seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=device),
                block_table=table.to(device), slot_mapping=slots.to(device),
                k_cache=k_cache, v_cache=v_cache)


def small(name="small", *, B=2, q_lens=(150, 37), seq_lens=None, hq=4, hkv=2, r=64,
          window=0, bias_std=1.0, history_random=None, state_random=None, q_prescale=1.0,
          scale=None, spare_blocks=3) -> Spec:
    """A small spec for tests: several tiles, ragged tails, optional cached prefix."""
    q_lens = list(q_lens)
    seq_lens = list(q_lens) if seq_lens is None else list(seq_lens)
    has_prefix = any(L > n for n, L in zip(q_lens, seq_lens))
    return Spec(name=name, batch=len(q_lens), hq=hq, hkv=hkv, r=r, window=window,
                bias_std=bias_std, q_lens=q_lens, seq_lens=seq_lens, q_prescale=q_prescale,
                scale=(1.0 / math.sqrt(HEAD_DIM)) if scale is None else scale,
                history_random=has_prefix if history_random is None else history_random,
                state_random=has_prefix if state_random is None else state_random,
                spare_blocks=spare_blocks)


@dataclasses.dataclass
class DenseCase:
    """One dense stream for the conv on a [T, C] activation (e.g. the attention output)."""
    x: torch.Tensor            # [T, C] bf16 raw rows
    w: torch.Tensor            # [C, 4] fp32 taps
    state: torch.Tensor        # [B, 3, C] bf16, oldest row first
    cu_q_lens: torch.Tensor    # [B+1] int32

    @property
    def max_q_len(self) -> int:
        cu = self.cu_q_lens.tolist()
        return max([b - a for a, b in zip(cu[:-1], cu[1:])] + [0])


def make_dense(q_lens, C: int, seed: int, device="cpu", w_std: float = 0.5,
               state_random: bool = True) -> DenseCase:
    """Seeded dense-stream inputs: x ~ N(0,1) bf16, taps ~ N(0, w_std) fp32, state ~ N(0,1)
    bf16 (zeros when state_random is False)."""
    g = torch.Generator().manual_seed(seed)
    T = int(sum(q_lens))
    x = torch.randn(T, C, generator=g).to(torch.bfloat16)
    w = torch.randn(C, 4, generator=g) * w_std
    st = torch.randn(len(q_lens), 3, C, generator=g) if state_random else torch.zeros(len(q_lens), 3, C)
    cu = torch.zeros(len(q_lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(list(q_lens), dtype=torch.int64), 0).to(torch.int32)
    return DenseCase(x.to(device), w.float().contiguous().to(device),
                     st.to(torch.bfloat16).contiguous().to(device), cu.to(device))


def fp8_history(cache: torch.Tensor, scale: float) -> torch.Tensor:
    """Seeded FP8 cache contents for tests and benches: the bf16 history pages quantized
    to E4M3 codes of cache / scale with torch's own float8_e4m3fn conversion (input
    generation only: the kernels and the oracle both consume the codes as given)."""
    return (cache.float() / scale).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
