// Whole steps (the sconv of the new tokens, then the attention) over page-locked host
// buffers.  The step is cut into groups of whole sequences; the copies of one group cross
// the host link while another group is computed (three streams, events between them).
// The host link of GB300 moves about 200 GB/s each way, so a prefill step whose Q and
// output are a few hundred MB spends longer copying than computing unless the two overlap.
// Host code only: the kernels are the ones the separate calls launch.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <vector>

#include "../../include/inkling.h"
#include "kernels.h"

namespace {

struct Group {
  int b0, b1;      // sequences [b0, b1)
  int64_t t0, t1;  // their new tokens [t0, t1)
  int max_n;       // longest n_b in the group
  bool piece;      // a run of one sequence's new tokens (b1 == b0 + 1), not all of them
};

// Groups of whole sequences with about T / chunks new tokens each: a group closes once the
// tokens seen reach its share of T.  Sequences with no new token join their neighbours.
std::vector<Group> make_groups(const int32_t* cu, int B, int chunks) {
  std::vector<Group> g;
  const int64_t T = cu[B];
  int b0 = 0, max_n = 0;
  for (int b = 0; b < B; ++b) {
    const int n = cu[b + 1] - cu[b];
    if (n > max_n) max_n = n;
    const int k = (int)g.size() + 1;  // this group's index + 1
    const bool last = b + 1 == B;
    if (last || (k < chunks && (int64_t)cu[b + 1] * chunks >= T * k)) {
      g.push_back(Group{b0, b + 1, cu[b0], cu[b + 1], max_n, false});
      b0 = b + 1;
      max_n = 0;
    }
  }
  return g;
}

// Prefill groups that may also cut a sequence: a sequence with more new tokens than a
// group's share becomes pieces of whole 128-token query tiles (so that every query tile,
// and with it the order of its sums, is the one the uncut call computes).  At most
// `chunks` pieces in all (their lengths need one scratch slot each); past that budget a
// long sequence stays whole.
std::vector<Group> make_prefill_groups(const int32_t* cu, int B, int chunks) {
  const int64_t T = cu[B];
  const int64_t share = ((T + chunks - 1) / chunks + 127) / 128 * 128;
  std::vector<Group> g;
  int b0 = -1, max_n = 0, pieces = 0;
  auto flush = [&](int b_end) {
    if (b0 >= 0) g.push_back(Group{b0, b_end, cu[b0], cu[b_end], max_n, false});
    b0 = -1;
    max_n = 0;
  };
  for (int b = 0; b < B; ++b) {
    const int n = cu[b + 1] - cu[b];
    const int need = (int)((n + share - 1) / share);
    if (n > share && pieces + need <= chunks) {
      pieces += need;
      flush(b);
      for (int64_t r = 0; r < n; r += share) {
        const int64_t e = r + share < n ? r + share : n;
        g.push_back(Group{b, b + 1, cu[b] + r, cu[b] + e, (int)(e - r), true});
      }
      continue;
    }
    if (b0 < 0) b0 = b;
    if (n > max_n) max_n = n;
    if ((int64_t)(cu[b + 1] - cu[b0]) >= share) flush(b + 1);
  }
  flush(B);
  return g;
}

// The lengths of a piece of sequence b, as the calls read them: cu = {0, rel1 - rel0} and
// the sequence's length at the piece's last token.
__global__ void piece_lens_kernel(const int32_t* cu_q_lens, const int32_t* seq_lens, int b,
                                  int rel0, int rel1, int32_t* out) {
  if (threadIdx.x == 0) {
    const int n = cu_q_lens[b + 1] - cu_q_lens[b];
    out[0] = 0;
    out[1] = rel1 - rel0;
    out[2] = seq_lens[b] - n + rel1;
    out[3] = 0;
  }
}

struct Events {
  std::vector<cudaEvent_t> ev;
  ~Events() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);  // safe while still pending
  }
  cudaEvent_t make() {
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    ev.push_back(e);
    return e;
  }
};

struct HostRows {
  const uint8_t* q_host;
  const uint8_t* k_host;
  const uint8_t* v_host;
  uint8_t* out_host;
  uint8_t* q_dev;
  uint8_t* k_dev;
  uint8_t* v_dev;
  uint8_t* out_dev;
  size_t q_row, kv_row, out_row;  // bytes per token
};

int copy_rows(void* dst, const void* src, int64_t t0, int64_t t1, size_t row, cudaMemcpyKind kind,
              cudaStream_t st) {
  if (t1 <= t0) return INKLING_OK;
  return cudaMemcpyAsync(static_cast<uint8_t*>(dst) + t0 * row,
                         static_cast<const uint8_t*>(src) + t0 * row, (size_t)(t1 - t0) * row,
                         kind, st) == cudaSuccess
             ? INKLING_OK
             : INKLING_ERR_CUDA;
}

// The pipeline shared by both step forms: `launch(group)` enqueues one group's sconv and
// attention on `s` and returns an inkling status.
template <class Launch>
int run_groups(const HostRows& h, const std::vector<Group>& groups, cudaStream_t s,
               cudaStream_t up, cudaStream_t down, Launch launch) {
  Events evs;
  cudaEvent_t start = evs.make();
  if (!start) return INKLING_ERR_CUDA;
  // the staging buffers may still be read by work already on `s`
  if (cudaEventRecord(start, s) != cudaSuccess || cudaStreamWaitEvent(up, start, 0) != cudaSuccess)
    return INKLING_ERR_CUDA;
  std::vector<cudaEvent_t> landed(groups.size());
  for (size_t i = 0; i < groups.size(); ++i) {
    const Group& g = groups[i];
    int rc = copy_rows(h.q_dev, h.q_host, g.t0, g.t1, h.q_row, cudaMemcpyHostToDevice, up);
    if (rc == INKLING_OK) rc = copy_rows(h.k_dev, h.k_host, g.t0, g.t1, h.kv_row, cudaMemcpyHostToDevice, up);
    if (rc == INKLING_OK) rc = copy_rows(h.v_dev, h.v_host, g.t0, g.t1, h.kv_row, cudaMemcpyHostToDevice, up);
    if (rc != INKLING_OK) return rc;
    landed[i] = evs.make();
    if (!landed[i] || cudaEventRecord(landed[i], up) != cudaSuccess) return INKLING_ERR_CUDA;
  }
  for (size_t i = 0; i < groups.size(); ++i) {
    const Group& g = groups[i];
    if (cudaStreamWaitEvent(s, landed[i], 0) != cudaSuccess) return INKLING_ERR_CUDA;
    const int rc = launch(g);
    if (rc != INKLING_OK) return rc;
    cudaEvent_t done = evs.make();
    if (!done || cudaEventRecord(done, s) != cudaSuccess ||
        cudaStreamWaitEvent(down, done, 0) != cudaSuccess)
      return INKLING_ERR_CUDA;
    const int crc = copy_rows(h.out_host, h.out_dev, g.t0, g.t1, h.out_row, cudaMemcpyDeviceToHost, down);
    if (crc != INKLING_OK) return crc;
  }
  cudaEvent_t end = evs.make();
  if (!end || cudaEventRecord(end, down) != cudaSuccess || cudaStreamWaitEvent(s, end, 0) != cudaSuccess)
    return INKLING_ERR_CUDA;
  return INKLING_OK;
}

// Host-side checks shared by both forms; fills rows and groups.
int prepare(const void* q_host, const void* k_raw_host, const void* v_raw_host, void* out_host,
            void* q_dev, void* k_raw_dev, void* v_raw_dev, void* out_dev,
            const int32_t* cu_host, int32_t out_dtype, int32_t B, int32_t T, int32_t Hq,
            int32_t Hkv, int32_t max_q_len, int32_t chunks, inkling_stream_t stream,
            inkling_stream_t h2d, inkling_stream_t d2h, HostRows* h, std::vector<Group>* groups) {
  if (!q_host || !k_raw_host || !v_raw_host || !out_host || !q_dev || !k_raw_dev || !v_raw_dev ||
      !out_dev || !cu_host)
    return INKLING_ERR_INVALID_ARG;
  if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || chunks < 1 || max_q_len < 0)
    return INKLING_ERR_INVALID_ARG;
  if (out_dtype != INKLING_OUT_BF16 && out_dtype != INKLING_OUT_F32) return INKLING_ERR_INVALID_ARG;
  if (h2d == nullptr || d2h == nullptr || h2d == d2h || h2d == stream || d2h == stream)
    return INKLING_ERR_INVALID_ARG;
  if (cu_host[0] != 0 || (B >= 0 && cu_host[B] != T)) return INKLING_ERR_INVALID_ARG;
  for (int b = 0; b < B; ++b) {
    const int n = cu_host[b + 1] - cu_host[b];
    if (n < 0 || n > max_q_len) return INKLING_ERR_INVALID_ARG;
  }
  h->q_host = static_cast<const uint8_t*>(q_host);
  h->k_host = static_cast<const uint8_t*>(k_raw_host);
  h->v_host = static_cast<const uint8_t*>(v_raw_host);
  h->out_host = static_cast<uint8_t*>(out_host);
  h->q_dev = static_cast<uint8_t*>(q_dev);
  h->k_dev = static_cast<uint8_t*>(k_raw_dev);
  h->v_dev = static_cast<uint8_t*>(v_raw_dev);
  h->out_dev = static_cast<uint8_t*>(out_dev);
  h->q_row = (size_t)Hq * 128 * 2;
  h->kv_row = (size_t)Hkv * 128 * 2;
  h->out_row = (size_t)Hq * 128 * (out_dtype == INKLING_OUT_F32 ? 4 : 2);
  *groups = B > 0 ? make_groups(cu_host, B, chunks < B ? chunks : B) : std::vector<Group>{};
  return INKLING_OK;
}

bool scales_ok(float k_scale, float v_scale) {
  return k_scale > 0.f && v_scale > 0.f && std::isfinite(k_scale) && std::isfinite(v_scale);
}

// One prefill step over a bf16 cache (fp8 false) or an E4M3 cache (fp8 true: the conv
// writes E4M3 codes with k_scale / v_scale, and each group's attention widens the pages it
// reads into `workspace`, which the groups reuse one after another on `stream`).
int prefill_step(bool fp8, float k_scale, float v_scale, const void* q_host,
                 const void* k_raw_host, const void* v_raw_host, void* out_host, void* q_dev,
                 void* k_raw_dev, void* v_raw_dev, void* out_dev, const int32_t* cu_q_lens_host,
                 const float* w_k, const float* w_v, void* sconv_state, const int32_t* cu_q_lens,
                 const int64_t* slot_mapping, void* k_cache, void* v_cache,
                 const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                 const float* bias, int32_t R, float scale, int32_t window, int32_t out_dtype,
                 float* lse, int32_t B, int32_t T, int32_t Hq, int32_t Hkv, int64_t num_blocks,
                 int32_t max_q_len, int32_t max_seq_len, void* workspace, size_t workspace_bytes,
                 int32_t chunks, int32_t* dev_scratch, int32_t* dev_status,
                 inkling_stream_t stream, inkling_stream_t h2d_stream,
                 inkling_stream_t d2h_stream) {
  HostRows h;
  std::vector<Group> groups;
  int rc = prepare(q_host, k_raw_host, v_raw_host, out_host, q_dev, k_raw_dev, v_raw_dev,
                   out_dev, cu_q_lens_host, out_dtype, B, T, Hq, Hkv, max_q_len, chunks, stream,
                   h2d_stream, d2h_stream, &h, &groups);
  if (rc != INKLING_OK) return rc;
  if (!w_k || !w_v || !sconv_state || !cu_q_lens || !slot_mapping || !block_table || !seq_lens)
    return INKLING_ERR_INVALID_ARG;
  if (fp8 && (!scales_ok(k_scale, v_scale) || max_seq_len < 0)) return INKLING_ERR_INVALID_ARG;
  if (B == 0 || T == 0) return INKLING_OK;
  // the widened pages of any group fit in a workspace sized for all B sequences
  if (fp8 && max_q_len > 0 && max_seq_len > 0 &&
      (workspace == nullptr ||
       workspace_bytes < ink::prefill_fp8_workspace_bytes(B, Hkv, max_blocks, max_q_len,
                                                          max_seq_len, window)))
    return INKLING_ERR_WORKSPACE;
  // with scratch for their lengths, long sequences may be cut into pieces
  if (dev_scratch != nullptr) groups = make_prefill_groups(cu_q_lens_host, B, chunks);
  const size_t state_seq = (size_t)2 * 3 * Hkv * 128 * 2;  // bytes of one sequence's state
  const size_t kv_row = (size_t)Hkv * 128 * 2;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  auto conv = [&](const void* k_raw, const void* v_raw, void* state, const int32_t* cu,
                  const int64_t* slots, int nb, int t, int max_n) {
    return fp8 ? inkling_sconv_kv_fp8(k_raw, v_raw, w_k, w_v, state, cu, slots, k_cache, v_cache,
                                      k_scale, v_scale, nb, t, Hkv, num_blocks, max_n, dev_status,
                                      stream)
               : inkling_sconv_kv(k_raw, v_raw, w_k, w_v, state, cu, slots, k_cache, v_cache, nb,
                                  t, Hkv, num_blocks, max_n, dev_status, stream);
  };
  auto attn = [&](const void* q, const int32_t* table, const int32_t* cu, const int32_t* lens,
                  void* out, float* lse_g, int nb, int t, int max_n) {
    return fp8 ? inkling_rel_attn_prefill_fp8(q, k_cache, v_cache, k_scale, v_scale, table,
                                              max_blocks, cu, lens, bias, R, scale, window, out,
                                              out_dtype, lse_g, nb, t, Hq, Hkv, num_blocks, max_n,
                                              max_seq_len, workspace, workspace_bytes, dev_status,
                                              stream)
               : inkling_rel_attn_prefill(q, k_cache, v_cache, table, max_blocks, cu, lens, bias,
                                          R, scale, window, out, out_dtype, lse_g, nb, t, Hq, Hkv,
                                          num_blocks, max_n, dev_status, stream);
  };
  int piece = 0;
  auto launch = [&](const Group& g) {
    if (g.piece) {
      // one run of sequence b's tokens: pointers start at its first row, and the lengths
      // come from a scratch slot (cu = {0, rows}, the sequence's length at its last row)
      int32_t* lens = dev_scratch + 4 * piece++;  // piece < chunks by construction
      const int b = g.b0;
      const int rel0 = (int)(g.t0 - cu_q_lens_host[b]), rel1 = (int)(g.t1 - cu_q_lens_host[b]);
      const int rows = rel1 - rel0;
      piece_lens_kernel<<<1, 32, 0, st>>>(cu_q_lens, seq_lens, b, rel0, rel1, lens);
      if (cudaGetLastError() != cudaSuccess) return (int)INKLING_ERR_CUDA;
      int r = conv(static_cast<uint8_t*>(k_raw_dev) + g.t0 * kv_row,
                   static_cast<uint8_t*>(v_raw_dev) + g.t0 * kv_row,
                   static_cast<uint8_t*>(sconv_state) + b * state_seq, lens, slot_mapping + g.t0,
                   1, rows, rows);
      if (r != INKLING_OK) return r;
      return attn(static_cast<uint8_t*>(q_dev) + g.t0 * h.q_row,
                  block_table + (size_t)b * max_blocks, lens, lens + 2,
                  static_cast<uint8_t*>(out_dev) + g.t0 * h.out_row,
                  lse ? lse + g.t0 * Hq : nullptr, 1, rows, rows);
    }
    const int nb = g.b1 - g.b0;
    int r = conv(k_raw_dev, v_raw_dev, static_cast<uint8_t*>(sconv_state) + g.b0 * state_seq,
                 cu_q_lens + g.b0, slot_mapping, nb, T, g.max_n);
    if (r != INKLING_OK) return r;
    return attn(q_dev, block_table + (size_t)g.b0 * max_blocks, cu_q_lens + g.b0,
                seq_lens + g.b0, out_dev, lse, nb, T, g.max_n);
  };
  return run_groups(h, groups, st, reinterpret_cast<cudaStream_t>(h2d_stream),
                    reinterpret_cast<cudaStream_t>(d2h_stream), launch);
}

// One decode step over a bf16 cache or (fp8 true) an E4M3 cache.
int decode_step(bool fp8, float k_scale, float v_scale, const void* q_host,
                const void* k_raw_host, const void* v_raw_host, void* out_host, void* q_dev,
                void* k_raw_dev, void* v_raw_dev, void* out_dev, const int32_t* cu_q_lens_host,
                const float* w_k, const float* w_v, void* sconv_state, const int32_t* cu_q_lens,
                const int64_t* slot_mapping, void* k_cache, void* v_cache,
                const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                const float* bias, int32_t R, float scale, int32_t window, int32_t out_dtype,
                float* lse, int32_t B, int32_t T, int32_t Hq, int32_t Hkv, int64_t num_blocks,
                int32_t max_q_len, int32_t max_seq_len, int32_t num_splits, void* workspace,
                size_t workspace_bytes, int32_t chunks, int32_t* dev_status,
                inkling_stream_t stream, inkling_stream_t h2d_stream,
                inkling_stream_t d2h_stream) {
  HostRows h;
  std::vector<Group> groups;
  int rc = prepare(q_host, k_raw_host, v_raw_host, out_host, q_dev, k_raw_dev, v_raw_dev,
                   out_dev, cu_q_lens_host, out_dtype, B, T, Hq, Hkv, max_q_len, chunks, stream,
                   h2d_stream, d2h_stream, &h, &groups);
  if (rc != INKLING_OK) return rc;
  if (!w_k || !w_v || !sconv_state || !cu_q_lens || !slot_mapping || !block_table || !seq_lens)
    return INKLING_ERR_INVALID_ARG;
  if (max_q_len > INKLING_MAX_DECODE_Q || num_splits < 0 || max_seq_len < 0)
    return INKLING_ERR_INVALID_ARG;
  if (fp8 && !scales_ok(k_scale, v_scale)) return INKLING_ERR_INVALID_ARG;
  if (B == 0 || T == 0) return INKLING_OK;
  // One split count for every group, the one the whole batch would get: a group's
  // partials then fit in a workspace sized for all B sequences.
  if (num_splits == 0 && groups.size() > 1) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return INKLING_ERR_CUDA;
    num_splits = ink::decode_split(B, Hkv, max_q_len, max_seq_len, window, 0, sms).num_splits;
  }
  const size_t state_seq = (size_t)2 * 3 * Hkv * 128 * 2;
  auto launch = [&](const Group& g) {
    const int nb = g.b1 - g.b0;
    void* state = static_cast<uint8_t*>(sconv_state) + g.b0 * state_seq;
    int r = fp8 ? inkling_sconv_kv_fp8(k_raw_dev, v_raw_dev, w_k, w_v, state, cu_q_lens + g.b0,
                                       slot_mapping, k_cache, v_cache, k_scale, v_scale, nb, T,
                                       Hkv, num_blocks, g.max_n, dev_status, stream)
                : inkling_sconv_kv(k_raw_dev, v_raw_dev, w_k, w_v, state, cu_q_lens + g.b0,
                                   slot_mapping, k_cache, v_cache, nb, T, Hkv, num_blocks,
                                   g.max_n, dev_status, stream);
    if (r != INKLING_OK) return r;
    const int32_t* table = block_table + (size_t)g.b0 * max_blocks;
    return fp8 ? inkling_rel_attn_decode_fp8(q_dev, k_cache, v_cache, k_scale, v_scale, table,
                                             max_blocks, cu_q_lens + g.b0, seq_lens + g.b0, bias,
                                             R, scale, window, out_dev, out_dtype, lse, nb, T, Hq,
                                             Hkv, num_blocks, g.max_n, max_seq_len, num_splits,
                                             workspace, workspace_bytes, dev_status, stream)
               : inkling_rel_attn_decode(q_dev, k_cache, v_cache, table, max_blocks,
                                         cu_q_lens + g.b0, seq_lens + g.b0, bias, R, scale,
                                         window, out_dev, out_dtype, lse, nb, T, Hq, Hkv,
                                         num_blocks, g.max_n, max_seq_len, num_splits, workspace,
                                         workspace_bytes, dev_status, stream);
  };
  return run_groups(h, groups, reinterpret_cast<cudaStream_t>(stream),
                    reinterpret_cast<cudaStream_t>(h2d_stream),
                    reinterpret_cast<cudaStream_t>(d2h_stream), launch);
}

}  // namespace

extern "C" {

int inkling_prefill_step_host(
    const void* q_host, const void* k_raw_host, const void* v_raw_host, void* out_host,
    void* q_dev, void* k_raw_dev, void* v_raw_dev, void* out_dev, const int32_t* cu_q_lens_host,
    const float* w_k, const float* w_v, void* sconv_state, const int32_t* cu_q_lens,
    const int64_t* slot_mapping, void* k_cache, void* v_cache, const int32_t* block_table,
    int32_t max_blocks, const int32_t* seq_lens, const float* bias, int32_t R, float scale,
    int32_t window, int32_t out_dtype, float* lse, int32_t B, int32_t T, int32_t Hq,
    int32_t Hkv, int64_t num_blocks, int32_t max_q_len, int32_t chunks, int32_t* dev_scratch,
    int32_t* dev_status, inkling_stream_t stream, inkling_stream_t h2d_stream,
    inkling_stream_t d2h_stream) {
  return prefill_step(false, 1.f, 1.f, q_host, k_raw_host, v_raw_host, out_host, q_dev,
                      k_raw_dev, v_raw_dev, out_dev, cu_q_lens_host, w_k, w_v, sconv_state,
                      cu_q_lens, slot_mapping, k_cache, v_cache, block_table, max_blocks,
                      seq_lens, bias, R, scale, window, out_dtype, lse, B, T, Hq, Hkv, num_blocks,
                      max_q_len, 0, nullptr, 0, chunks, dev_scratch, dev_status, stream,
                      h2d_stream, d2h_stream);
}

int inkling_prefill_step_host_fp8(
    const void* q_host, const void* k_raw_host, const void* v_raw_host, void* out_host,
    void* q_dev, void* k_raw_dev, void* v_raw_dev, void* out_dev, const int32_t* cu_q_lens_host,
    const float* w_k, const float* w_v, void* sconv_state, const int32_t* cu_q_lens,
    const int64_t* slot_mapping, void* k_cache, void* v_cache, float k_scale, float v_scale,
    const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens, const float* bias,
    int32_t R, float scale, int32_t window, int32_t out_dtype, float* lse, int32_t B, int32_t T,
    int32_t Hq, int32_t Hkv, int64_t num_blocks, int32_t max_q_len, int32_t max_seq_len,
    void* workspace, size_t workspace_bytes, int32_t chunks, int32_t* dev_scratch,
    int32_t* dev_status, inkling_stream_t stream, inkling_stream_t h2d_stream,
    inkling_stream_t d2h_stream) {
  return prefill_step(true, k_scale, v_scale, q_host, k_raw_host, v_raw_host, out_host, q_dev,
                      k_raw_dev, v_raw_dev, out_dev, cu_q_lens_host, w_k, w_v, sconv_state,
                      cu_q_lens, slot_mapping, k_cache, v_cache, block_table, max_blocks,
                      seq_lens, bias, R, scale, window, out_dtype, lse, B, T, Hq, Hkv, num_blocks,
                      max_q_len, max_seq_len, workspace, workspace_bytes, chunks, dev_scratch,
                      dev_status, stream, h2d_stream, d2h_stream);
}

int inkling_decode_step_host(
    const void* q_host, const void* k_raw_host, const void* v_raw_host, void* out_host,
    void* q_dev, void* k_raw_dev, void* v_raw_dev, void* out_dev, const int32_t* cu_q_lens_host,
    const float* w_k, const float* w_v, void* sconv_state, const int32_t* cu_q_lens,
    const int64_t* slot_mapping, void* k_cache, void* v_cache, const int32_t* block_table,
    int32_t max_blocks, const int32_t* seq_lens, const float* bias, int32_t R, float scale,
    int32_t window, int32_t out_dtype, float* lse, int32_t B, int32_t T, int32_t Hq,
    int32_t Hkv, int64_t num_blocks, int32_t max_q_len, int32_t max_seq_len,
    int32_t num_splits, void* workspace, size_t workspace_bytes, int32_t chunks,
    int32_t* dev_status, inkling_stream_t stream, inkling_stream_t h2d_stream,
    inkling_stream_t d2h_stream) {
  return decode_step(false, 1.f, 1.f, q_host, k_raw_host, v_raw_host, out_host, q_dev,
                     k_raw_dev, v_raw_dev, out_dev, cu_q_lens_host, w_k, w_v, sconv_state,
                     cu_q_lens, slot_mapping, k_cache, v_cache, block_table, max_blocks,
                     seq_lens, bias, R, scale, window, out_dtype, lse, B, T, Hq, Hkv, num_blocks,
                     max_q_len, max_seq_len, num_splits, workspace, workspace_bytes, chunks,
                     dev_status, stream, h2d_stream, d2h_stream);
}

int inkling_decode_step_host_fp8(
    const void* q_host, const void* k_raw_host, const void* v_raw_host, void* out_host,
    void* q_dev, void* k_raw_dev, void* v_raw_dev, void* out_dev, const int32_t* cu_q_lens_host,
    const float* w_k, const float* w_v, void* sconv_state, const int32_t* cu_q_lens,
    const int64_t* slot_mapping, void* k_cache, void* v_cache, float k_scale, float v_scale,
    const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens, const float* bias,
    int32_t R, float scale, int32_t window, int32_t out_dtype, float* lse, int32_t B, int32_t T,
    int32_t Hq, int32_t Hkv, int64_t num_blocks, int32_t max_q_len, int32_t max_seq_len,
    int32_t num_splits, void* workspace, size_t workspace_bytes, int32_t chunks,
    int32_t* dev_status, inkling_stream_t stream, inkling_stream_t h2d_stream,
    inkling_stream_t d2h_stream) {
  return decode_step(true, k_scale, v_scale, q_host, k_raw_host, v_raw_host, out_host, q_dev,
                     k_raw_dev, v_raw_dev, out_dev, cu_q_lens_host, w_k, w_v, sconv_state,
                     cu_q_lens, slot_mapping, k_cache, v_cache, block_table, max_blocks,
                     seq_lens, bias, R, scale, window, out_dtype, lse, B, T, Hq, Hkv, num_blocks,
                     max_q_len, max_seq_len, num_splits, workspace, workspace_bytes, chunks,
                     dev_status, stream, h2d_stream, d2h_stream);
}

}  // extern "C"
