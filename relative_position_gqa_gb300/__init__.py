"""Inkling attention block on GB300: sconv on K/V into a paged cache, and relative-bias
GQA prefill / paged decode, as a C-ABI CUDA library (include/inkling.h) for sm_103a.

This module only marshals torch tensors into the C calls: every step of the computation
runs in the library's CUDA kernels.  It raises if the library has not been built; there
is no CPU or PyTorch fallback.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib

HEAD_DIM = 128
BLOCK_SIZE = 128
MAX_DECODE_Q = 9
OUT_BF16, OUT_F32 = 0, 1

InklingError = _lib.InklingError
status_string = _lib.status_string
library_path = _lib.library_path


def _check_cuda(*ts):
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("all tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("all tensors must be on the same device")
    return dev


def _stream(stream):
    return (stream if stream is not None else torch.cuda.current_stream()).cuda_stream


def sconv_kv(k_raw: torch.Tensor, v_raw: torch.Tensor, w_k: torch.Tensor, w_v: torch.Tensor,
             sconv_state: torch.Tensor, cu_q_lens: torch.Tensor, slot_mapping: torch.Tensor,
             k_cache: torch.Tensor, v_cache: torch.Tensor, *, max_q_len: int,
             dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    """inkling_sconv_kv: conv on the new raw K/V rows straight into the paged caches, and
    the in-place sconv-state update.  Shapes as in include/inkling.h."""
    dev = _check_cuda(k_raw, v_raw, w_k, w_v, sconv_state, cu_q_lens, slot_mapping, k_cache,
                      v_cache, dev_status)
    assert k_raw.dtype == v_raw.dtype == sconv_state.dtype == k_cache.dtype == torch.bfloat16
    assert w_k.dtype == w_v.dtype == torch.float32
    assert cu_q_lens.dtype == torch.int32 and slot_mapping.dtype == torch.int64
    B = cu_q_lens.shape[0] - 1
    T = k_raw.shape[0]
    hkv = k_cache.shape[1]
    with torch.cuda.device(dev):
        _lib.call("inkling_sconv_kv", k_raw, v_raw, w_k, w_v, sconv_state, cu_q_lens,
                  slot_mapping, k_cache, v_cache, B, T, hkv, k_cache.shape[0], int(max_q_len),
                  dev_status, _stream(stream))


def sconv_kv_fp8(k_raw, v_raw, w_k, w_v, sconv_state, cu_q_lens, slot_mapping, k_cache,
                 v_cache, *, k_scale: float, v_scale: float, max_q_len: int,
                 dev_status=None, stream=None) -> None:
    """inkling_sconv_kv_fp8: the conv into FP8 (E4M3, uint8) paged caches,
    code = e4m3(y / scale)."""
    dev = _check_cuda(k_raw, v_raw, w_k, w_v, sconv_state, cu_q_lens, slot_mapping, k_cache,
                      v_cache, dev_status)
    assert k_raw.dtype == v_raw.dtype == sconv_state.dtype == torch.bfloat16
    assert k_cache.dtype == v_cache.dtype == torch.uint8
    with torch.cuda.device(dev):
        _lib.call("inkling_sconv_kv_fp8", k_raw, v_raw, w_k, w_v, sconv_state, cu_q_lens,
                  slot_mapping, k_cache, v_cache, float(k_scale), float(v_scale),
                  cu_q_lens.shape[0] - 1, k_raw.shape[0], k_cache.shape[1], k_cache.shape[0],
                  int(max_q_len), dev_status, _stream(stream))


def sconv(x: torch.Tensor, w: torch.Tensor, sconv_state: torch.Tensor, cu_q_lens: torch.Tensor,
          *, max_q_len: int, y: Optional[torch.Tensor] = None, dev_status=None,
          stream=None) -> torch.Tensor:
    """inkling_sconv: the conv on one dense stream x [T, C] with its own state [B, 3, C]
    (updated in place); returns y [T, C] bf16 (allocated when not given)."""
    if y is None:
        y = torch.empty_like(x)
    dev = _check_cuda(x, w, sconv_state, cu_q_lens, y, dev_status)
    assert x.dtype == sconv_state.dtype == y.dtype == torch.bfloat16 and w.dtype == torch.float32
    assert cu_q_lens.dtype == torch.int32
    with torch.cuda.device(dev):
        _lib.call("inkling_sconv", x, w, sconv_state, cu_q_lens, y, cu_q_lens.shape[0] - 1,
                  x.shape[0], x.shape[1], int(max_q_len), dev_status, _stream(stream))
    return y


def sconv_state_rollback(state_before: torch.Tensor, x0: torch.Tensor,
                         x1: Optional[torch.Tensor], cu_q_lens: torch.Tensor,
                         accepted: torch.Tensor, state_after: Optional[torch.Tensor] = None, *,
                         dev_status=None, stream=None) -> torch.Tensor:
    """inkling_sconv_state_rollback: the sconv state after keeping only the first
    accepted[b] new tokens of a step.  With x1 (v_raw) the state is the K/V pair layout
    [B, 2, 3, C]; without it, one stream [B, 3, C].  state_after may be state_before."""
    if state_after is None:
        state_after = torch.empty_like(state_before)
    dev = _check_cuda(state_before, x0, x1, cu_q_lens, accepted, state_after, dev_status)
    assert state_before.dtype == state_after.dtype == x0.dtype == torch.bfloat16
    assert cu_q_lens.dtype == accepted.dtype == torch.int32
    streams = 2 if x1 is not None else 1
    with torch.cuda.device(dev):
        _lib.call("inkling_sconv_state_rollback", state_before, x0, x1, cu_q_lens, accepted,
                  state_after, cu_q_lens.shape[0] - 1, x0.shape[0], x0.shape[1], streams,
                  dev_status, _stream(stream))
    return state_after


def _attn_common(q, k_cache, v_cache, block_table, cu_q_lens, seq_lens, bias, out, lse,
                 dev_status, cache_dtype=torch.bfloat16):
    dev = _check_cuda(q, k_cache, v_cache, block_table, cu_q_lens, seq_lens, bias, out, lse,
                      dev_status)
    assert q.dtype == torch.bfloat16 and k_cache.dtype == v_cache.dtype == cache_dtype
    assert block_table.dtype == cu_q_lens.dtype == seq_lens.dtype == torch.int32
    assert bias.dtype == torch.float32
    if out.dtype == torch.bfloat16:
        out_dtype = OUT_BF16
    elif out.dtype == torch.float32:
        out_dtype = OUT_F32
    else:
        raise ValueError("out must be bf16 or fp32")
    if lse is not None:
        assert lse.dtype == torch.float32
    return dev, out_dtype


def rel_attn_prefill(q, k_cache, v_cache, block_table, cu_q_lens, seq_lens, bias, *,
                     scale: float, window: int, max_q_len: int, out: torch.Tensor,
                     lse: Optional[torch.Tensor] = None, dev_status=None, stream=None) -> None:
    """inkling_rel_attn_prefill into `out` ([T, Hq, 128], bf16 or fp32)."""
    dev, out_dtype = _attn_common(q, k_cache, v_cache, block_table, cu_q_lens, seq_lens, bias,
                                  out, lse, dev_status)
    T, hq = q.shape[0], q.shape[1]
    with torch.cuda.device(dev):
        _lib.call("inkling_rel_attn_prefill", q, k_cache, v_cache, block_table,
                  block_table.shape[1], cu_q_lens, seq_lens, bias, bias.shape[1], float(scale),
                  int(window), out, out_dtype, lse, cu_q_lens.shape[0] - 1, T, hq,
                  k_cache.shape[1], k_cache.shape[0], int(max_q_len), dev_status,
                  _stream(stream))


def decode_workspace_size(B: int, hq: int, hkv: int, max_q_len: int, max_seq_len: int,
                          window: int, num_splits: int = 0, device=None) -> int:
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return _lib.workspace_size(B, hq, hkv, max_q_len, max_seq_len, window, num_splits)


def decode_plan(B: int, hq: int, hkv: int, max_q_len: int, max_seq_len: int, window: int,
                num_splits: int = 0, device=None) -> dict:
    """inkling_rel_attn_decode_plan: how the decode calls split the keys."""
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        v = _lib.decode_plan(B, hq, hkv, max_q_len, max_seq_len, window, num_splits)
    return {"num_splits": v[0], "ctas": v[1], "pages_per_split": v[2], "merge": bool(v[3])}


def rel_attn_decode(q, k_cache, v_cache, block_table, cu_q_lens, seq_lens, bias, *,
                    scale: float, window: int, max_q_len: int, max_seq_len: int,
                    out: torch.Tensor, lse: Optional[torch.Tensor] = None, num_splits: int = 0,
                    workspace: Optional[torch.Tensor] = None, dev_status=None,
                    stream=None) -> None:
    """inkling_rel_attn_decode into `out`.  `workspace` is a caller-owned device buffer of
    at least decode_workspace_size(...) bytes (allocated here when omitted).  num_splits:
    0 automatic, > 0 equal splits per (sequence, KV head) (decode_plan tells which)."""
    dev, out_dtype = _attn_common(q, k_cache, v_cache, block_table, cu_q_lens, seq_lens, bias,
                                  out, lse, dev_status)
    T, hq = q.shape[0], q.shape[1]
    B = cu_q_lens.shape[0] - 1
    hkv = k_cache.shape[1]
    with torch.cuda.device(dev):
        need = _lib.workspace_size(B, hq, hkv, int(max_q_len), int(max_seq_len), int(window),
                                   int(num_splits))
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _lib.call("inkling_rel_attn_decode", q, k_cache, v_cache, block_table,
                  block_table.shape[1], cu_q_lens, seq_lens, bias, bias.shape[1], float(scale),
                  int(window), out, out_dtype, lse, B, T, hq, hkv, k_cache.shape[0],
                  int(max_q_len), int(max_seq_len), int(num_splits), workspace, ws_bytes,
                  dev_status, _stream(stream))


def rel_attn_decode_sconv(q, k_raw, v_raw, w_k, w_v, sconv_state, k_cache, v_cache,
                          block_table, cu_q_lens, seq_lens, bias, *, scale: float, window: int,
                          max_q_len: int, max_seq_len: int, out: torch.Tensor,
                          lse: Optional[torch.Tensor] = None, num_splits: int = 0,
                          workspace: Optional[torch.Tensor] = None, dev_status=None,
                          stream=None) -> None:
    """inkling_rel_attn_decode_sconv: one decode step with the conv of its new tokens fused
    into the decode kernel (the new K/V rows go into the caches at the slots the block
    table gives their positions; the state is updated in place).  The same results as
    sconv_kv followed by rel_attn_decode."""
    dev, out_dtype = _attn_common(q, k_cache, v_cache, block_table, cu_q_lens, seq_lens, bias,
                                  out, lse, dev_status)
    _check_cuda(k_raw, v_raw, w_k, w_v, sconv_state)
    assert k_raw.dtype == v_raw.dtype == sconv_state.dtype == torch.bfloat16
    assert w_k.dtype == w_v.dtype == torch.float32
    T, hq = q.shape[0], q.shape[1]
    B = cu_q_lens.shape[0] - 1
    hkv = k_cache.shape[1]
    with torch.cuda.device(dev):
        need = _lib.workspace_size(B, hq, hkv, int(max_q_len), int(max_seq_len), int(window),
                                   int(num_splits))
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _lib.call("inkling_rel_attn_decode_sconv", q, k_raw, v_raw, w_k, w_v, sconv_state,
                  k_cache, v_cache, block_table, block_table.shape[1], cu_q_lens, seq_lens, bias,
                  bias.shape[1], float(scale), int(window), out, out_dtype, lse, B, T, hq, hkv,
                  k_cache.shape[0], int(max_q_len), int(max_seq_len), int(num_splits), workspace,
                  ws_bytes, dev_status, _stream(stream))


def rel_attn_decode_fp8(q, k_cache, v_cache, block_table, cu_q_lens, seq_lens, bias, *,
                        k_scale: float, v_scale: float, scale: float, window: int,
                        max_q_len: int, max_seq_len: int, out: torch.Tensor,
                        lse: Optional[torch.Tensor] = None, num_splits: int = 0,
                        workspace: Optional[torch.Tensor] = None, dev_status=None,
                        stream=None) -> None:
    """inkling_rel_attn_decode_fp8: decode over FP8 (E4M3, uint8) caches,
    K = code * k_scale, V = code * v_scale."""
    dev = _check_cuda(q, k_cache, v_cache, block_table, cu_q_lens, seq_lens, bias, out, lse,
                      dev_status)
    assert q.dtype == torch.bfloat16 and k_cache.dtype == v_cache.dtype == torch.uint8
    assert block_table.dtype == cu_q_lens.dtype == seq_lens.dtype == torch.int32
    out_dtype = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
    T, hq = q.shape[0], q.shape[1]
    B = cu_q_lens.shape[0] - 1
    hkv = k_cache.shape[1]
    with torch.cuda.device(dev):
        need = _lib.workspace_size(B, hq, hkv, int(max_q_len), int(max_seq_len), int(window),
                                   int(num_splits))
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _lib.call("inkling_rel_attn_decode_fp8", q, k_cache, v_cache, float(k_scale),
                  float(v_scale), block_table, block_table.shape[1], cu_q_lens, seq_lens, bias,
                  bias.shape[1], float(scale), int(window), out, out_dtype, lse, B, T, hq, hkv,
                  k_cache.shape[0], int(max_q_len), int(max_seq_len), int(num_splits), workspace,
                  ws_bytes, dev_status, _stream(stream))


def prefill_fp8_workspace_size(B: int, hkv: int, max_blocks: int, max_q_len: int,
                               max_seq_len: int, window: int) -> int:
    """Bytes of workspace inkling_rel_attn_prefill_fp8 needs (the widened bf16 pages)."""
    return int(_lib.load().inkling_rel_attn_prefill_fp8_workspace_size(
        int(B), int(hkv), int(max_blocks), int(max_q_len), int(max_seq_len), int(window)))


def rel_attn_prefill_fp8(q, k_cache, v_cache, block_table, cu_q_lens, seq_lens, bias, *,
                         k_scale: float, v_scale: float, scale: float, window: int,
                         max_q_len: int, max_seq_len: int, out: torch.Tensor,
                         lse: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None, dev_status=None,
                         stream=None) -> None:
    """inkling_rel_attn_prefill_fp8: prefill over FP8 (E4M3, uint8) caches, K = code *
    k_scale, V = code * v_scale.  `workspace` holds the widened bf16 pages (allocated here
    when omitted)."""
    dev = _check_cuda(q, k_cache, v_cache, block_table, cu_q_lens, seq_lens, bias, out, lse,
                      dev_status, workspace)
    assert q.dtype == torch.bfloat16 and k_cache.dtype == v_cache.dtype == torch.uint8
    assert block_table.dtype == cu_q_lens.dtype == seq_lens.dtype == torch.int32
    out_dtype = OUT_BF16 if out.dtype == torch.bfloat16 else OUT_F32
    T, hq = q.shape[0], q.shape[1]
    B = cu_q_lens.shape[0] - 1
    hkv = k_cache.shape[1]
    with torch.cuda.device(dev):
        if workspace is None:
            need = prefill_fp8_workspace_size(B, hkv, block_table.shape[1], max_q_len,
                                              max_seq_len, window)
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        ws_bytes = workspace.numel() * workspace.element_size()
        _lib.call("inkling_rel_attn_prefill_fp8", q, k_cache, v_cache, float(k_scale),
                  float(v_scale), block_table, block_table.shape[1], cu_q_lens, seq_lens, bias,
                  bias.shape[1], float(scale), int(window), out, out_dtype, lse, B, T, hq, hkv,
                  k_cache.shape[0], int(max_q_len), int(max_seq_len), workspace, ws_bytes,
                  dev_status, _stream(stream))


def decode_noalloc_capacity() -> int:
    """Bytes of the library's static decode scratch (per device)."""
    return int(_lib.load().inkling_rel_attn_decode_noalloc_capacity())


def rel_attn_decode_noalloc(q, k_cache, v_cache, block_table, cu_q_lens, seq_lens, bias, *,
                            scale: float, window: int, max_q_len: int, max_seq_len: int,
                            out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                            num_splits: int = 0, dev_status=None, stream=None) -> None:
    """inkling_rel_attn_decode_noalloc: the same decode, with its split partials in the
    library's static device scratch instead of a workspace, for callers that cannot
    allocate device memory while they run.  Nothing is allocated here either.  Calls
    that can overlap on the GPU share that scratch and must be serialised."""
    dev, out_dtype = _attn_common(q, k_cache, v_cache, block_table, cu_q_lens, seq_lens, bias,
                                  out, lse, dev_status)
    T, hq = q.shape[0], q.shape[1]
    with torch.cuda.device(dev):
        _lib.call("inkling_rel_attn_decode_noalloc", q, k_cache, v_cache, block_table,
                  block_table.shape[1], cu_q_lens, seq_lens, bias, bias.shape[1], float(scale),
                  int(window), out, out_dtype, lse, cu_q_lens.shape[0] - 1, T, hq,
                  k_cache.shape[1], k_cache.shape[0], int(max_q_len), int(max_seq_len),
                  int(num_splits), dev_status, _stream(stream))


def _check_host(*ts):
    for t in ts:
        if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
            raise ValueError("host buffers must be contiguous page-locked CPU tensors")


def _step_args(q_host, k_raw_host, v_raw_host, out_host, staging, cu_q_lens_host, w_k, w_v,
               sconv_state, cu_q_lens, slot_mapping, k_cache, v_cache, block_table, seq_lens,
               bias, lse, dev_status, cache_dtype=torch.bfloat16):
    q_dev, k_dev, v_dev, out_dev = staging
    _check_host(q_host, k_raw_host, v_raw_host, out_host)
    if cu_q_lens_host.is_cuda or cu_q_lens_host.dtype != torch.int32:
        raise ValueError("cu_q_lens_host must be an int32 CPU tensor")
    cu_host = cu_q_lens_host.contiguous()
    dev, out_dtype = _attn_common(q_dev, k_cache, v_cache, block_table, cu_q_lens, seq_lens,
                                  bias, out_dev, lse, dev_status, cache_dtype)
    _check_cuda(q_dev, k_dev, v_dev, out_dev, w_k, w_v, sconv_state, cu_q_lens, slot_mapping,
                k_cache, v_cache, block_table, seq_lens, bias, lse, dev_status)
    for h, d in ((q_host, q_dev), (k_raw_host, k_dev), (v_raw_host, v_dev), (out_host, out_dev)):
        if h.shape != d.shape or h.dtype != d.dtype:
            raise ValueError("each host buffer must match its device staging buffer")
    return dev, out_dtype, cu_host


def prefill_step_host(q_host, k_raw_host, v_raw_host, out_host, staging, cu_q_lens_host, w_k,
                      w_v, sconv_state, cu_q_lens, slot_mapping, k_cache, v_cache, block_table,
                      seq_lens, bias, *, scale: float, window: int, max_q_len: int,
                      h2d_stream, d2h_stream, chunks: int = 4, split_sequences: bool = True,
                      scratch: Optional[torch.Tensor] = None, lse=None, dev_status=None,
                      stream=None) -> None:
    """inkling_prefill_step_host: sconv_kv + rel_attn_prefill for a step whose Q, raw K/V
    and output live in page-locked host memory.  `staging` = (q_dev, k_raw_dev, v_raw_dev,
    out_dev), device buffers of the host buffers' shapes; the copies of one group of
    sequences run on h2d_stream / d2h_stream while another group is computed.  With
    split_sequences, a long sequence may be cut into pieces of whole query tiles (its
    lengths go to `scratch`, 4 * chunks int32 on the device, allocated when omitted)."""
    dev, out_dtype, cu_host = _step_args(q_host, k_raw_host, v_raw_host, out_host, staging,
                                         cu_q_lens_host, w_k, w_v, sconv_state, cu_q_lens,
                                         slot_mapping, k_cache, v_cache, block_table, seq_lens,
                                         bias, lse, dev_status)
    q_dev, k_dev, v_dev, out_dev = staging
    with torch.cuda.device(dev):
        if split_sequences and scratch is None:
            scratch = torch.empty(4 * max(int(chunks), 1), dtype=torch.int32, device=dev)
        if not split_sequences:
            scratch = None
        _lib.call("inkling_prefill_step_host", q_host, k_raw_host, v_raw_host, out_host, q_dev,
                  k_dev, v_dev, out_dev, cu_host, w_k, w_v, sconv_state, cu_q_lens,
                  slot_mapping, k_cache, v_cache, block_table, block_table.shape[1], seq_lens,
                  bias, bias.shape[1], float(scale), int(window), out_dtype, lse,
                  cu_q_lens.shape[0] - 1, q_dev.shape[0], q_dev.shape[1], k_cache.shape[1],
                  k_cache.shape[0], int(max_q_len), int(chunks), scratch, dev_status,
                  _stream(stream), h2d_stream.cuda_stream, d2h_stream.cuda_stream)


def decode_step_host(q_host, k_raw_host, v_raw_host, out_host, staging, cu_q_lens_host, w_k,
                     w_v, sconv_state, cu_q_lens, slot_mapping, k_cache, v_cache, block_table,
                     seq_lens, bias, *, scale: float, window: int, max_q_len: int,
                     max_seq_len: int, h2d_stream, d2h_stream, num_splits: int = 0,
                     workspace: Optional[torch.Tensor] = None, chunks: int = 1, lse=None,
                     dev_status=None, stream=None) -> None:
    """inkling_decode_step_host: sconv_kv + rel_attn_decode over host buffers, as
    prefill_step_host.  `workspace` is sized for all B sequences (allocated when omitted)."""
    dev, out_dtype, cu_host = _step_args(q_host, k_raw_host, v_raw_host, out_host, staging,
                                         cu_q_lens_host, w_k, w_v, sconv_state, cu_q_lens,
                                         slot_mapping, k_cache, v_cache, block_table, seq_lens,
                                         bias, lse, dev_status)
    q_dev, k_dev, v_dev, out_dev = staging
    B = cu_q_lens.shape[0] - 1
    hkv = k_cache.shape[1]
    with torch.cuda.device(dev):
        need = _lib.workspace_size(B, q_dev.shape[1], hkv, int(max_q_len), int(max_seq_len),
                                   int(window), int(num_splits))
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _lib.call("inkling_decode_step_host", q_host, k_raw_host, v_raw_host, out_host, q_dev,
                  k_dev, v_dev, out_dev, cu_host, w_k, w_v, sconv_state, cu_q_lens,
                  slot_mapping, k_cache, v_cache, block_table, block_table.shape[1], seq_lens,
                  bias, bias.shape[1], float(scale), int(window), out_dtype, lse, B,
                  q_dev.shape[0], q_dev.shape[1], hkv, k_cache.shape[0], int(max_q_len),
                  int(max_seq_len), int(num_splits), workspace, ws_bytes, int(chunks),
                  dev_status, _stream(stream), h2d_stream.cuda_stream, d2h_stream.cuda_stream)


def prefill_step_host_fp8(q_host, k_raw_host, v_raw_host, out_host, staging, cu_q_lens_host,
                          w_k, w_v, sconv_state, cu_q_lens, slot_mapping, k_cache, v_cache,
                          block_table, seq_lens, bias, *, k_scale: float, v_scale: float,
                          scale: float, window: int, max_q_len: int, max_seq_len: int,
                          h2d_stream, d2h_stream, chunks: int = 4, split_sequences: bool = True,
                          scratch: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None, lse=None, dev_status=None,
                          stream=None) -> None:
    """inkling_prefill_step_host_fp8: sconv_kv_fp8 + rel_attn_prefill_fp8 over host buffers,
    as prefill_step_host, for E4M3 (uint8) caches.  `workspace` takes the widened pages
    (prefill_fp8_workspace_size bytes for all B sequences, allocated when omitted)."""
    dev, out_dtype, cu_host = _step_args(q_host, k_raw_host, v_raw_host, out_host, staging,
                                         cu_q_lens_host, w_k, w_v, sconv_state, cu_q_lens,
                                         slot_mapping, k_cache, v_cache, block_table, seq_lens,
                                         bias, lse, dev_status, torch.uint8)
    q_dev, k_dev, v_dev, out_dev = staging
    B = cu_q_lens.shape[0] - 1
    hkv = k_cache.shape[1]
    with torch.cuda.device(dev):
        if split_sequences and scratch is None:
            scratch = torch.empty(4 * max(int(chunks), 1), dtype=torch.int32, device=dev)
        if not split_sequences:
            scratch = None
        if workspace is None:
            need = prefill_fp8_workspace_size(B, hkv, block_table.shape[1], max_q_len,
                                              max_seq_len, window)
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        ws_bytes = workspace.numel() * workspace.element_size()
        _lib.call("inkling_prefill_step_host_fp8", q_host, k_raw_host, v_raw_host, out_host,
                  q_dev, k_dev, v_dev, out_dev, cu_host, w_k, w_v, sconv_state, cu_q_lens,
                  slot_mapping, k_cache, v_cache, float(k_scale), float(v_scale), block_table,
                  block_table.shape[1], seq_lens, bias, bias.shape[1], float(scale), int(window),
                  out_dtype, lse, B, q_dev.shape[0], q_dev.shape[1], hkv, k_cache.shape[0],
                  int(max_q_len), int(max_seq_len), workspace, ws_bytes, int(chunks), scratch,
                  dev_status, _stream(stream), h2d_stream.cuda_stream, d2h_stream.cuda_stream)


def decode_step_host_fp8(q_host, k_raw_host, v_raw_host, out_host, staging, cu_q_lens_host,
                         w_k, w_v, sconv_state, cu_q_lens, slot_mapping, k_cache, v_cache,
                         block_table, seq_lens, bias, *, k_scale: float, v_scale: float,
                         scale: float, window: int, max_q_len: int, max_seq_len: int,
                         h2d_stream, d2h_stream, num_splits: int = 0,
                         workspace: Optional[torch.Tensor] = None, chunks: int = 1, lse=None,
                         dev_status=None, stream=None) -> None:
    """inkling_decode_step_host_fp8: sconv_kv_fp8 + rel_attn_decode_fp8 over host buffers,
    as decode_step_host, for E4M3 (uint8) caches."""
    dev, out_dtype, cu_host = _step_args(q_host, k_raw_host, v_raw_host, out_host, staging,
                                         cu_q_lens_host, w_k, w_v, sconv_state, cu_q_lens,
                                         slot_mapping, k_cache, v_cache, block_table, seq_lens,
                                         bias, lse, dev_status, torch.uint8)
    q_dev, k_dev, v_dev, out_dev = staging
    B = cu_q_lens.shape[0] - 1
    hkv = k_cache.shape[1]
    with torch.cuda.device(dev):
        need = _lib.workspace_size(B, q_dev.shape[1], hkv, int(max_q_len), int(max_seq_len),
                                   int(window), int(num_splits))
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _lib.call("inkling_decode_step_host_fp8", q_host, k_raw_host, v_raw_host, out_host,
                  q_dev, k_dev, v_dev, out_dev, cu_host, w_k, w_v, sconv_state, cu_q_lens,
                  slot_mapping, k_cache, v_cache, float(k_scale), float(v_scale), block_table,
                  block_table.shape[1], seq_lens, bias, bias.shape[1], float(scale), int(window),
                  out_dtype, lse, B, q_dev.shape[0], q_dev.shape[1], hkv, k_cache.shape[0],
                  int(max_q_len), int(max_seq_len), int(num_splits), workspace, ws_bytes,
                  int(chunks), dev_status, _stream(stream), h2d_stream.cuda_stream,
                  d2h_stream.cuda_stream)


def selftest_bounded_wait(mode: int, ctas: int, dev_status: torch.Tensor,
                          gave_up: torch.Tensor, stream=None) -> None:
    """inkling_selftest_bounded_wait: CTAs wait on a barrier nothing arrives on; mode 0
    must time out (about 2 s), mode 1 must stop early on another CTA's error."""
    dev = _check_cuda(dev_status, gave_up)
    with torch.cuda.device(dev):
        _lib.call("inkling_selftest_bounded_wait", int(mode), int(ctas), dev_status, gave_up,
                  _stream(stream))
