// C ABI of libkvq.so: argument checks, rotary frequency tables, launches.
// The operations and their page citations are documented in include/kvq.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "kvq_internal.h"
#include "kvq_prompt.h"

namespace {

thread_local std::string g_last_error;

kvq_status fail(kvq_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
kvq_status fail(kvq_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

kvq_status cuda_fail(cudaError_t e, const char* what) {
  return fail(KVQ_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

// Positions are below 2^24 (exact in fp32); checked before max_pos + 1 is formed.
bool max_pos_ok(int32_t max_pos) { return max_pos >= 0 && max_pos < (1 << 24); }

// theta^(-2j/D) (libm pow, float64) split into three floats that sum to it
// exactly, cached per (theta, D, rope_dims).
const kvq::RopeFreqs& rope_freqs(double theta, int D, int R) {
  static std::mutex mu;
  static std::map<std::tuple<double, int, int>, kvq::RopeFreqs> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto key = std::make_tuple(theta, D, R);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  kvq::RopeFreqs f;
  std::memset(&f, 0, sizeof f);
  for (int j = 0; j < R / 2; ++j) {
    const double v = std::pow(theta, -(2.0 * j) / D);
    const float f1 = (float)v;
    const double r1 = v - (double)f1;      // exact
    const float f2 = (float)r1;
    const double r2 = r1 - (double)f2;     // exact
    f.f[j][0] = f1;
    f.f[j][1] = f2;
    f.f[j][2] = (float)r2;
  }
  return cache.emplace(key, f).first->second;
}

// SM count of the current device, looked up once per device (atomics: host
// threads may make their first call on a device at the same time).
int num_sms_current() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cached[dev].load(std::memory_order_acquire);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev].store(n, std::memory_order_release);
  }
  return n;
}

// kvq_profile_next_read's events for this host thread
thread_local cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;

cudaError_t prof_record(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  // inside a stream capture the record becomes a graph node that times the replay
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal)
                                             : cudaEventRecord(ev, st);
}

kvq_status check_layer(const kvq_layer* L, kvq::LayerArgs* out) {
  if (!L) return fail(KVQ_EINVAL, "layer is NULL");
  if (L->n_kv_heads <= 0 || L->n_q_heads <= 0 || L->n_q_heads % L->n_kv_heads)
    return fail(KVQ_EINVAL, "n_q_heads (%d) must be a positive multiple of n_kv_heads (%d)",
                L->n_q_heads, L->n_kv_heads);
  const int G = L->n_q_heads / L->n_kv_heads;
  if (G > kvq::kMaxG)
    return fail(KVQ_EUNSUPPORTED, "n_q_heads / n_kv_heads = %d exceeds %d", G, kvq::kMaxG);
  if (L->head_dim != 64 && L->head_dim != 128 && L->head_dim != 256 && L->head_dim != 512)
    return fail(KVQ_EUNSUPPORTED, "head_dim %d not in {64, 128, 256, 512}", L->head_dim);
  if (L->group_size != 64) return fail(KVQ_EUNSUPPORTED, "group_size %d != 64", L->group_size);
  if (L->window < 0) return fail(KVQ_EINVAL, "window %d < 0", L->window);
  if (L->rope_dims < 0 || L->rope_dims > L->head_dim || (L->rope_dims & 1))
    return fail(KVQ_EINVAL, "rope_dims %d must be even and in [0, head_dim]", L->rope_dims);
  if (!(L->rope_theta > 0.0) || !std::isfinite(L->rope_theta))
    return fail(KVQ_EINVAL, "rope_theta must be positive and finite");
  if (!(L->rms_eps >= 0.f) || !std::isfinite(L->rms_eps)) return fail(KVQ_EINVAL, "rms_eps must be >= 0");
  if (L->k_eq_v != 0 && L->k_eq_v != 1) return fail(KVQ_EINVAL, "k_eq_v must be 0 or 1");
  out->n_q = L->n_q_heads;
  out->n_kv = L->n_kv_heads;
  out->D = L->head_dim;
  out->G = G;
  out->window = L->window;
  out->rope_dims = L->rope_dims;
  out->k_eq_v = L->k_eq_v;
  out->eps = L->rms_eps;
  out->rot = L->rot_signs;
  out->qk_scale = L->rot_signs ? 1.0f / (float)L->head_dim : 1.0f;
  return KVQ_OK;
}

// A non-NULL pointer aligned to `al` bytes (16 for tensors read with 128-bit
// loads, the element size otherwise, 8 for the descriptor array).
#define REQUIRE_PTR(p, name, al)                                                         \
  do {                                                                                   \
    if (!(p)) return fail(KVQ_EINVAL, "%s is NULL", name);                               \
    if (!aligned(p, al)) return fail(KVQ_EINVAL, "%s is not %d-byte aligned", name, al); \
  } while (0)

// One attention call, checked and planned, ready to launch.
enum class Path { kDecode, kPrefillTc, kPromptTc };
struct Prepared {
  kvq::DecodeArgs a;
  const kvq::RopeFreqs* f;
  bool tc;              // a tensor-core path (launched first among attn_mixed's groups)
  Path path;
  void* workspace;
  size_t workspace_bytes;
  int32_t max_rows_per_seq;
  int32_t max_keys;     // the decode plan's bound on keys per row
  bool fixed_chunks;
  bool empty;
};

// Windows of at most this many rows per sequence (verify windows) are read
// by the decode kernels row by row.  Measured on GB300 (16 sequences of a
// sliding layer, 8q/2kv D256 W512, lengths 1k-8k): the tensor-core prompt
// path takes 42-44 us for 1..16 rows per sequence, the decode kernels 4-33 us
// more than a 48-sequence decode group alone; at 32 rows the tensor cores win
// (46 us against 75 us).
constexpr int kRowPathWindowRows = 16;

// The path of a call: sliding-window prompt rows on the dequantize-once
// tensor-core path, other prompt rows the tensor cores fit on the codes-in-MMA
// tensor-core path, verify windows and the rest on the decode kernels.
Path choose_path(const kvq::LayerArgs& L, bool prompt, int max_rows_per_seq) {
  if (!prompt || max_rows_per_seq <= kRowPathWindowRows) return Path::kDecode;
  if (kvq::prompt_tc_supported(L)) return Path::kPromptTc;
  if (kvq::prefill_tc_supported(L)) return Path::kPrefillTc;
  return Path::kDecode;
}

// Every check of an attention call; enqueues nothing.
kvq_status attention_prepare(const kvq_layer* layer, const kvq_seq_cache* seqs, int32_t n_seqs,
                             const int32_t* row_offsets, const int32_t* pos, int32_t n_rows, int32_t max_keys,
                             bool fixed_chunks, int32_t max_rows_per_seq,
                             const uint16_t* q_raw, const uint16_t* q_norm_w, void* out, int32_t out_is_f32,
                             uint16_t* q_prepped, void* workspace, size_t workspace_bytes, Prepared* p) {
  kvq::LayerArgs L;
  kvq_status st = check_layer(layer, &L);
  if (st != KVQ_OK) return st;
  p->empty = false;
  if (n_seqs < 0 || n_rows < 0) return fail(KVQ_EINVAL, "negative n_seqs or n_rows");
  if (n_rows == 0) {
    p->empty = true;
    return KVQ_OK;
  }
  if (n_seqs == 0) return fail(KVQ_EINVAL, "n_rows > 0 with n_seqs == 0");
  if (max_keys < 1 || max_keys > (1 << 24)) return fail(KVQ_EINVAL, "max position out of range");
  REQUIRE_PTR(seqs, "seqs", 8);
  REQUIRE_PTR(pos, "pos/start_pos", 4);
  REQUIRE_PTR(q_raw, "q_raw", 16);
  REQUIRE_PTR(q_norm_w, "q_norm_w", 2);
  REQUIRE_PTR(out, "out", out_is_f32 ? 4 : 2);
  REQUIRE_PTR(workspace, "workspace", 256);
  if (row_offsets) REQUIRE_PTR(row_offsets, "row_offsets", 4);
  if (q_prepped && !aligned(q_prepped, 2)) return fail(KVQ_EINVAL, "q_prepped is not 2-byte aligned");
  if (out_is_f32 != 0 && out_is_f32 != 1) return fail(KVQ_EINVAL, "out_is_f32 must be 0 or 1");
  // prompt chunks whose head shape fits a tensor-core kernel take it
  const Path path = choose_path(L, row_offsets != nullptr, max_rows_per_seq);
  const bool tc = path != Path::kDecode;
  const kvq::DecodePlan plan = tc ? kvq::DecodePlan{1, 0, 0}
                                  : kvq::decode_plan(L, n_rows, max_keys, num_sms_current(), fixed_chunks);
  const size_t need = path == Path::kPromptTc ? kvq::prompt_tc_ws_bytes(n_seqs, n_rows, max_rows_per_seq, L)
                      : path == Path::kPrefillTc ? kvq::prefill_tc_ws_bytes(n_rows, L)
                                                 : kvq::decode_ws_bytes(n_rows, L.n_kv, L.D, plan);
  if (workspace_bytes < need)
    return fail(KVQ_EWORKSPACE, "workspace %zu bytes < %zu required", workspace_bytes, need);
  kvq::DecodeArgs& a = p->a;
  a = kvq::DecodeArgs{};
  a.L = L;
  a.seqs = seqs;
  a.n_seqs = n_seqs;
  a.n_rows = n_rows;
  a.row_offsets = row_offsets;
  a.pos = pos;
  a.q_raw = q_raw;
  a.q_w = q_norm_w;
  a.out = out;
  a.out_f32 = out_is_f32;
  a.q_prepped = q_prepped;
  a.splits = plan.splits;
  a.chunk_tiles = plan.chunk_tiles;
  a.sk_ctas = plan.sk_ctas;
  if (path == Path::kPromptTc) {
    a.ws = kvq::DecodeWs{};
    a.ws.status = static_cast<uint32_t*>(workspace);
  } else {
    a.ws = tc ? kvq::prefill_tc_ws_carve(workspace, n_rows, L)
              : kvq::decode_ws_carve(workspace, n_rows, L.n_kv, L.D, plan);
  }
  p->f = &rope_freqs(layer->rope_theta, L.D, L.rope_dims);
  p->tc = tc;
  p->path = path;
  p->workspace = workspace;
  p->workspace_bytes = workspace_bytes;
  p->max_rows_per_seq = max_rows_per_seq;
  p->max_keys = max_keys;
  p->fixed_chunks = fixed_chunks;
  return KVQ_OK;
}

// ap: NULL, or the call's K/V append, run in the grid of the tensor-core
// paths' q prep (the row path appends first, then reads)
kvq_status attention_launch(const Prepared& p, cudaStream_t st, const kvq::AppendArgs* ap = nullptr) {
  if (p.empty) return KVQ_OK;
  cudaError_t e = cudaSuccess;
  if (p.path == Path::kPromptTc) {
    e = kvq::launch_prompt_tc(p.a, p.workspace, p.max_rows_per_seq, *p.f, st, ap);
  } else if (p.path == Path::kPrefillTc) {
    e = kvq::launch_prefill_tc(p.a, *p.f, p.max_rows_per_seq, st, ap);
  } else {
    if (ap) e = kvq::launch_append(*ap, *p.f, st);
    if (e == cudaSuccess) e = kvq::launch_decode(p.a, *p.f, num_sms_current(), st);
  }
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  return KVQ_OK;
}

kvq_status attention_common(const kvq_layer* layer, const kvq_seq_cache* seqs, int32_t n_seqs,
                            const int32_t* row_offsets, const int32_t* pos, int32_t n_rows, int32_t max_keys,
                            bool fixed_chunks, int32_t max_rows_per_seq,
                            const uint16_t* q_raw, const uint16_t* q_norm_w, void* out, int32_t out_is_f32,
                            uint16_t* q_prepped, void* workspace, size_t workspace_bytes, void* stream) {
  Prepared p;
  const kvq_status st = attention_prepare(layer, seqs, n_seqs, row_offsets, pos, n_rows, max_keys, fixed_chunks,
                                          max_rows_per_seq, q_raw, q_norm_w, out, out_is_f32, q_prepped, workspace,
                                          workspace_bytes, &p);
  if (st != KVQ_OK) return st;
  return attention_launch(p, static_cast<cudaStream_t>(stream));
}

}  // namespace

namespace kvq {
cudaError_t prof_before(cudaStream_t st) { return g_prof_start ? prof_record(g_prof_start, st) : cudaSuccess; }
cudaError_t prof_after(cudaStream_t st) {
  const cudaEvent_t ev = g_prof_stop;
  g_prof_start = g_prof_stop = nullptr;
  return ev ? prof_record(ev, st) : cudaSuccess;
}
}  // namespace kvq

extern "C" {

kvq_status kv_quant_append(const kvq_layer* layer, const kvq_seq_cache* seqs, int32_t n_seqs,
                           const int32_t* row_offsets, const int32_t* start_pos, int32_t n_rows,
                           const uint16_t* k_raw, const uint16_t* v_raw, const uint16_t* k_norm_w,
                           uint16_t* kv_prepped, void* stream) {
  kvq::LayerArgs L;
  kvq_status st = check_layer(layer, &L);
  if (st != KVQ_OK) return st;
  if (n_seqs < 0 || n_rows < 0) return fail(KVQ_EINVAL, "negative n_seqs or n_rows");
  if (n_rows == 0) return KVQ_OK;
  if (n_seqs == 0) return fail(KVQ_EINVAL, "n_rows > 0 with n_seqs == 0");
  REQUIRE_PTR(seqs, "seqs", 8);
  REQUIRE_PTR(row_offsets, "row_offsets", 4);
  REQUIRE_PTR(start_pos, "start_pos", 4);
  REQUIRE_PTR(k_raw, "k_raw", 16);
  REQUIRE_PTR(k_norm_w, "k_norm_w", 2);
  if (L.k_eq_v) {
    if (v_raw) return fail(KVQ_EINVAL, "v_raw must be NULL when k_eq_v = 1");
  } else {
    REQUIRE_PTR(v_raw, "v_raw", 16);
  }
  if (kv_prepped && !aligned(kv_prepped, 2)) return fail(KVQ_EINVAL, "kv_prepped is not 2-byte aligned");
  kvq::AppendArgs a = {};
  a.L = L;
  a.seqs = seqs;
  a.n_seqs = n_seqs;
  a.row_offsets = row_offsets;
  a.start_pos = start_pos;
  a.n_rows = n_rows;
  a.k_raw = k_raw;
  a.v_raw = v_raw;
  a.k_w = k_norm_w;
  a.prepped = kv_prepped;
  const kvq::RopeFreqs& f = rope_freqs(layer->rope_theta, L.D, L.rope_dims);
  cudaError_t e = kvq::launch_append(a, f, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_quant_append launch");
  return KVQ_OK;
}

kvq_status attn_decode(const kvq_layer* layer, const kvq_seq_cache* seqs, int32_t n_seqs,
                       const int32_t* pos, int32_t max_pos, const uint16_t* q_raw, const uint16_t* q_norm_w,
                       void* out, int32_t out_is_f32, uint16_t* q_prepped, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (!max_pos_ok(max_pos)) return fail(KVQ_EINVAL, "max_pos %d not in [0, 2^24)", max_pos);
  return attention_common(layer, seqs, n_seqs, nullptr, pos, n_seqs, max_pos + 1, true, 0, q_raw, q_norm_w, out,
                          out_is_f32, q_prepped, workspace, workspace_bytes, stream);
}

kvq_status attn_decode_append(const kvq_layer* layer, const kvq_seq_cache* seqs, int32_t n_seqs,
                              const int32_t* pos, int32_t max_pos, const uint16_t* q_raw, const uint16_t* k_raw,
                              const uint16_t* v_raw, const uint16_t* q_norm_w, const uint16_t* k_norm_w,
                              void* out, int32_t out_is_f32, uint16_t* q_prepped, uint16_t* kv_prepped,
                              void* workspace, size_t workspace_bytes, void* stream) {
  if (!max_pos_ok(max_pos)) return fail(KVQ_EINVAL, "max_pos %d not in [0, 2^24)", max_pos);
  Prepared p;
  kvq_status st = attention_prepare(layer, seqs, n_seqs, nullptr, pos, n_seqs, max_pos + 1, true, 0, q_raw,
                                    q_norm_w, out, out_is_f32, q_prepped, workspace, workspace_bytes, &p);
  if (st != KVQ_OK || p.empty) return st;
  // the append's own checks (the layer, sequences and positions passed above)
  REQUIRE_PTR(k_raw, "k_raw", 16);
  REQUIRE_PTR(k_norm_w, "k_norm_w", 2);
  if (p.a.L.k_eq_v) {
    if (v_raw) return fail(KVQ_EINVAL, "v_raw must be NULL when k_eq_v = 1");
  } else {
    REQUIRE_PTR(v_raw, "v_raw", 16);
  }
  if (kv_prepped && !aligned(kv_prepped, 2)) return fail(KVQ_EINVAL, "kv_prepped is not 2-byte aligned");
  kvq::AppendArgs ap = {};
  ap.L = p.a.L;
  ap.seqs = seqs;
  ap.n_seqs = n_seqs;
  ap.row_offsets = nullptr;                 // one row per sequence
  ap.start_pos = pos;
  ap.n_rows = n_seqs;
  ap.k_raw = k_raw;
  ap.v_raw = v_raw;
  ap.k_w = k_norm_w;
  ap.prepped = kv_prepped;
  p.a.fused_append = 1;
  const cudaError_t e = kvq::launch_decode_append(p.a, ap, *p.f, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attn_decode_append launch");
  return KVQ_OK;
}

size_t attn_decode_workspace_bytes(const kvq_layer* layer, int32_t n_seqs, int32_t max_pos) {
  kvq::LayerArgs L;
  if (check_layer(layer, &L) != KVQ_OK || n_seqs < 0 || !max_pos_ok(max_pos)) return 0;
  const kvq::DecodePlan plan = kvq::decode_plan(L, n_seqs, max_pos + 1, num_sms_current(), true);
  return kvq::decode_ws_bytes(n_seqs, L.n_kv, L.D, plan);
}

kvq_status attn_prefill_chunk(const kvq_layer* layer, const kvq_seq_cache* seqs, int32_t n_seqs,
                              const int32_t* row_offsets, const int32_t* start_pos, int32_t n_rows,
                              int32_t max_rows_per_seq, const uint16_t* q_raw, const uint16_t* q_norm_w,
                              void* out, int32_t out_is_f32, uint16_t* q_prepped, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (n_rows > 0 && !row_offsets) return fail(KVQ_EINVAL, "row_offsets is NULL");
  if (max_rows_per_seq < 1 && n_rows > 0) return fail(KVQ_EINVAL, "max_rows_per_seq < 1");
  // each row reads at most window keys (full layers: the caller's positions)
  const int32_t max_keys = layer && layer->window > 0 ? layer->window : (1 << 24);
  return attention_common(layer, seqs, n_seqs, row_offsets, start_pos, n_rows, max_keys, false, max_rows_per_seq,
                          q_raw, q_norm_w, out, out_is_f32, q_prepped, workspace, workspace_bytes, stream);
}

kvq_status attn_prefill_append(const kvq_layer* layer, const kvq_seq_cache* seqs, int32_t n_seqs,
                               const int32_t* row_offsets, const int32_t* start_pos, int32_t n_rows,
                               int32_t max_rows_per_seq, const uint16_t* q_raw, const uint16_t* k_raw,
                               const uint16_t* v_raw, const uint16_t* q_norm_w, const uint16_t* k_norm_w,
                               void* out, int32_t out_is_f32, uint16_t* q_prepped, uint16_t* kv_prepped,
                               void* workspace, size_t workspace_bytes, void* stream) {
  if (n_rows > 0 && !row_offsets) return fail(KVQ_EINVAL, "row_offsets is NULL");
  if (max_rows_per_seq < 1 && n_rows > 0) return fail(KVQ_EINVAL, "max_rows_per_seq < 1");
  const int32_t max_keys = layer && layer->window > 0 ? layer->window : (1 << 24);
  Prepared p;
  kvq_status st = attention_prepare(layer, seqs, n_seqs, row_offsets, start_pos, n_rows, max_keys, false,
                                    max_rows_per_seq, q_raw, q_norm_w, out, out_is_f32, q_prepped, workspace,
                                    workspace_bytes, &p);
  if (st != KVQ_OK || p.empty) return st;
  REQUIRE_PTR(k_raw, "k_raw", 16);
  REQUIRE_PTR(k_norm_w, "k_norm_w", 2);
  if (p.a.L.k_eq_v) {
    if (v_raw) return fail(KVQ_EINVAL, "v_raw must be NULL when k_eq_v = 1");
  } else {
    REQUIRE_PTR(v_raw, "v_raw", 16);
  }
  if (kv_prepped && !aligned(kv_prepped, 2)) return fail(KVQ_EINVAL, "kv_prepped is not 2-byte aligned");
  kvq::AppendArgs ap = {};
  ap.L = p.a.L;
  ap.seqs = seqs;
  ap.n_seqs = n_seqs;
  ap.row_offsets = row_offsets;
  ap.start_pos = start_pos;
  ap.n_rows = n_rows;
  ap.k_raw = k_raw;
  ap.v_raw = v_raw;
  ap.k_w = k_norm_w;
  ap.prepped = kv_prepped;
  return attention_launch(p, static_cast<cudaStream_t>(stream), &ap);
}

size_t attn_prefill_workspace_bytes(const kvq_layer* layer, int32_t n_seqs, int32_t n_rows,
                                    int32_t max_rows_per_seq) {
  kvq::LayerArgs L;
  if (check_layer(layer, &L) != KVQ_OK || n_seqs < 0 || n_rows < 0 || max_rows_per_seq < 0) return 0;
  const Path path = choose_path(L, true, max_rows_per_seq);
  if (path == Path::kPromptTc) return kvq::prompt_tc_ws_bytes(n_seqs, n_rows, max_rows_per_seq, L);
  if (path == Path::kPrefillTc) return kvq::prefill_tc_ws_bytes(n_rows, L);
  const int32_t max_keys = layer->window > 0 ? layer->window : (1 << 24);
  const kvq::DecodePlan plan = kvq::decode_plan(L, n_rows, max_keys, num_sms_current(), false);
  return kvq::decode_ws_bytes(n_rows, L.n_kv, L.D, plan);
}

// ---------------------------------------------------------------------------
// attn_mixed: the groups of one layer checked together; the groups the
// decode kernels serve run as one grouped launch, every other group on its
// own kernels, forked from the caller's stream onto library streams and
// joined back.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace {

// Everything attn_mixed does before it enqueues: every group checked and
// planned (p), the members of the grouped launch (member) and, when two or
// more groups share it, its arguments (*ga non-null).
struct MixedPlan {
  Prepared p[KVQ_MAX_MIXED_GROUPS];
  bool member[KVQ_MAX_MIXED_GROUPS];
  kvq::GroupedDecode ga_buf;
  kvq::GroupedDecode* ga;
  const kvq::RopeFreqs* gf;
};

kvq_status mixed_prepare(const kvq_layer* layer, const kvq_attn_group* groups, int32_t n_groups,
                         const uint16_t* q_norm_w, int32_t out_is_f32, MixedPlan* mp) {
  Prepared* p = mp->p;
  bool* member = mp->member;
  mp->ga = nullptr;
  mp->gf = nullptr;
  if (n_groups < 0 || n_groups > KVQ_MAX_MIXED_GROUPS)
    return fail(KVQ_EINVAL, "n_groups %d not in [0, %d]", n_groups, KVQ_MAX_MIXED_GROUPS);
  if (n_groups == 0) return KVQ_OK;
  if (!groups) return fail(KVQ_EINVAL, "groups is NULL");
  for (int i = 0; i < n_groups; ++i) {
    const kvq_attn_group& g = groups[i];
    kvq_status st;
    if (g.phase == KVQ_PHASE_DECODE) {
      if (!max_pos_ok(g.max_pos)) return fail(KVQ_EINVAL, "group %d: max_pos %d not in [0, 2^24)", i, g.max_pos);
      st = attention_prepare(layer, g.seqs, g.n_seqs, nullptr, g.pos, g.n_seqs, g.max_pos + 1, true, 0, g.q_raw,
                             q_norm_w, g.out, out_is_f32, g.q_prepped, g.workspace, g.workspace_bytes, &p[i]);
    } else if (g.phase == KVQ_PHASE_WINDOW) {
      if (g.n_rows > 0 && !g.row_offsets) return fail(KVQ_EINVAL, "group %d: row_offsets is NULL", i);
      if (g.max_rows_per_seq < 1 && g.n_rows > 0) return fail(KVQ_EINVAL, "group %d: max_rows_per_seq < 1", i);
      const int32_t max_keys = layer && layer->window > 0 ? layer->window : (1 << 24);
      st = attention_prepare(layer, g.seqs, g.n_seqs, g.row_offsets, g.pos, g.n_rows, max_keys, false,
                             g.max_rows_per_seq, g.q_raw, q_norm_w, g.out, out_is_f32, g.q_prepped, g.workspace,
                             g.workspace_bytes, &p[i]);
    } else {
      return fail(KVQ_EINVAL, "group %d: phase %d is neither decode nor window", i, g.phase);
    }
    if (st != KVQ_OK) {
      g_last_error = "group " + std::to_string(i) + ": " + g_last_error;
      return st;
    }
  }
  for (int i = 0; i < n_groups; ++i)
    for (int j = 0; j < i; ++j) {
      if (p[i].empty || p[j].empty) continue;
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(groups[i].workspace), a1 = a0 + groups[i].workspace_bytes;
      const uintptr_t b0 = reinterpret_cast<uintptr_t>(groups[j].workspace), b1 = b0 + groups[j].workspace_bytes;
      if (a0 < b1 && b0 < a1) return fail(KVQ_EINVAL, "groups %d and %d share workspace memory", j, i);
    }
  // The grouped schedule: every group the decode kernels serve (decode
  // groups, verify windows, window groups of shapes the tensor-core kernels
  // do not take) runs in ONE launch of each decode-path kernel -- q prep,
  // attention, merge -- whose grids cover all of them, each group with its own
  // sequences, positions, bits, q, output and workspace.  A group whose
  // workspace cannot hold even one split of the shared plan runs on its own.
  int n_member = 0;
  for (int i = 0; i < n_groups; ++i) {
    member[i] = !p[i].empty && !p[i].tc;
    n_member += member[i];
  }
  const kvq::LayerArgs* Lg = nullptr;
  for (int i = 0; i < n_groups; ++i)
    if (member[i]) Lg = &p[i].a.L;
  while (n_member >= 2) {
    int idx[KVQ_MAX_MIXED_GROUPS], rows[KVQ_MAX_MIXED_GROUPS], mk[KVQ_MAX_MIXED_GROUPS], cap[KVQ_MAX_MIXED_GROUPS];
    bool fx[KVQ_MAX_MIXED_GROUPS];
    int n = 0;
    for (int i = 0; i < n_groups; ++i)
      if (member[i]) {
        idx[n] = i;
        rows[n] = p[i].a.n_rows;
        mk[n] = p[i].max_keys;
        fx[n] = p[i].fixed_chunks;
        cap[n] = kvq::decode_max_splits(rows[n], Lg->n_kv, Lg->D, p[i].workspace_bytes);
        ++n;
      }
    bool dropped = false;
    for (int k = 0; k < n; ++k)
      if (cap[k] < 1) {
        member[idx[k]] = false;
        --n_member;
        dropped = true;
      }
    if (dropped) continue;
    kvq::DecodePlan plans[KVQ_MAX_MIXED_GROUPS];
    kvq::decode_plan_grouped(*Lg, n, rows, mk, fx, cap, num_sms_current(), plans);
    long long total_rows = 0, total_ctas = 0;
    for (int k = 0; k < n; ++k) {
      total_rows += rows[k];
      total_ctas += (long long)rows[k] * Lg->n_kv * plans[k].splits;
    }
    if (total_rows > INT32_MAX || total_ctas > INT32_MAX) break;   // past one 1-D grid: run them apart
    kvq::GroupedDecode* ga = &mp->ga_buf;
    *ga = kvq::GroupedDecode{};
    ga->n = n;
    mp->ga = ga;
    mp->gf = p[idx[0]].f;
    for (int k = 0; k < n; ++k) {
      kvq::DecodeArgs a = p[idx[k]].a;
      a.splits = plans[k].splits;
      a.chunk_tiles = plans[k].chunk_tiles;
      a.sk_ctas = 0;
      a.ws = kvq::decode_ws_carve(p[idx[k]].workspace, rows[k], a.L.n_kv, a.L.D, plans[k]);
      ga->g[k] = a;
      ga->row_base[k + 1] = ga->row_base[k] + rows[k];
      ga->cta_base[k + 1] = ga->cta_base[k] + rows[k] * a.L.n_kv * a.splits;
    }
    break;
  }
  return KVQ_OK;
}

struct MixedPool {
  cudaStream_t s[KVQ_MAX_MIXED_GROUPS];
  cudaEvent_t fork, join[KVQ_MAX_MIXED_GROUPS];
};

// Streams and events of attn_mixed on the current device, created once.
MixedPool* mixed_pool() {
  static std::mutex mu;
  static MixedPool* pools[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cuda_fail(e, "attn_mixed: cudaGetDevice");
    return nullptr;
  }
  if (dev < 0 || dev >= 64) {
    fail(KVQ_EUNSUPPORTED, "attn_mixed: device ordinal %d >= 64", dev);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!pools[dev]) {
    MixedPool* q = new MixedPool();
    e = cudaEventCreateWithFlags(&q->fork, cudaEventDisableTiming);
    for (int i = 0; e == cudaSuccess && i < KVQ_MAX_MIXED_GROUPS; ++i) {
      e = cudaStreamCreateWithFlags(&q->s[i], cudaStreamNonBlocking);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&q->join[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
      cuda_fail(e, "attn_mixed: creating streams and events");
      return nullptr;                     // (the partial pool is not reused)
    }
    pools[dev] = q;
  }
  return pools[dev];
}

}  // namespace

extern "C" {

kvq_status attn_mixed(const kvq_layer* layer, const kvq_attn_group* groups, int32_t n_groups,
                      const uint16_t* q_norm_w, int32_t out_is_f32, void* stream) {
  static thread_local MixedPlan mp;
  g_prof_start = g_prof_stop = nullptr;           // not a call kvq_profile_next_read times
  const kvq_status pst = mixed_prepare(layer, groups, n_groups, q_norm_w, out_is_f32, &mp);
  if (pst != KVQ_OK || n_groups == 0) return pst;
  const Prepared* p = mp.p;
  const bool* member = mp.member;
  const kvq::GroupedDecode* ga = mp.ga;
  // Launch order: the library streams' units are enqueued first and the
  // caller's stream's unit last.  Window groups on the tensor cores go first:
  // their one-wave grids of one CTA per SM then get the SMs, and the short,
  // latency-bound decode kernels fill in around them.  (Measured on GB300, a
  // 48-sequence decode group beside two 256-row prompt chunks of a sliding
  // layer: 0.078 ms per step this way, 0.090 with the decode group first,
  // 0.087 as separate calls.)  Unit -1 is the grouped launch.
  int live[KVQ_MAX_MIXED_GROUPS + 1], n_live = 0;
  if (ga) live[n_live++] = -1;
  for (int i = 0; i < n_groups; ++i)
    if (!p[i].empty && !p[i].tc && !(ga && member[i])) live[n_live++] = i;
  for (int i = 0; i < n_groups; ++i)
    if (!p[i].empty && p[i].tc && !(ga && member[i])) live[n_live++] = i;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  auto launch_unit = [&](int u, cudaStream_t s) -> kvq_status {
    if (u >= 0) return attention_launch(p[u], s);
    const cudaError_t le = kvq::launch_decode_grouped(*ga, *mp.gf, s);
    return le == cudaSuccess ? KVQ_OK : cuda_fail(le, "attn_mixed: grouped launch");
  };
  if (n_live == 0) return KVQ_OK;
  if (n_live == 1) return launch_unit(live[0], st);
  MixedPool* pool = mixed_pool();
  if (!pool) return KVQ_ECUDA;
  cudaError_t e = cudaEventRecord(pool->fork, st);
  if (e != cudaSuccess) return cuda_fail(e, "attn_mixed: fork");
  // live[1..] on the library streams, live[0] on the caller's; every side
  // stream that waited on the fork is joined back, even after a failure
  kvq_status result = KVQ_OK;
  int forked = 0;
  for (int k = 1; k < n_live; ++k) {
    e = cudaStreamWaitEvent(pool->s[k], pool->fork, 0);
    if (e != cudaSuccess) {
      result = cuda_fail(e, "attn_mixed: fork wait");
      break;
    }
    forked = k;
    const kvq_status ls = launch_unit(live[k], pool->s[k]);
    if (ls != KVQ_OK) {
      result = ls;
      break;
    }
  }
  if (result == KVQ_OK) result = launch_unit(live[0], st);
  for (int k = 1; k <= forked; ++k) {
    e = cudaEventRecord(pool->join[k], pool->s[k]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, pool->join[k], 0);
    if (e != cudaSuccess && result == KVQ_OK) result = cuda_fail(e, "attn_mixed: join");
  }
  return result;
}

kvq_status attn_mixed_schedule(const kvq_layer* layer, const kvq_attn_group* groups, int32_t n_groups,
                               const uint16_t* q_norm_w, int32_t out_is_f32, uint32_t* grouped_mask) {
  if (!grouped_mask) return fail(KVQ_EINVAL, "grouped_mask is NULL");
  static thread_local MixedPlan mp;
  const kvq_status st = mixed_prepare(layer, groups, n_groups, q_norm_w, out_is_f32, &mp);
  if (st != KVQ_OK) return st;
  uint32_t m = 0;
  if (mp.ga)
    for (int i = 0; i < n_groups; ++i)
      if (mp.member[i]) m |= 1u << i;
  *grouped_mask = m;
  return KVQ_OK;
}

// ---------------------------------------------------------------------------
// attn_decode_static: attn_decode for callers that cannot allocate device
// memory.  Its scratch is this file-scope array, which every GPU that loads
// the library holds until the process exits.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace {

static __device__ __align__(256) uint8_t g_static_scratch[KVQ_STATIC_SCRATCH_BYTES];

// Device address of g_static_scratch on the current device, looked up once
// per device.  Returns nullptr (and sets the error message) on failure.
void* static_scratch_address(int* dev_out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cuda_fail(e, "attn_decode_static: cudaGetDevice");
    return nullptr;
  }
  if (dev < 0 || dev >= 64) {
    fail(KVQ_EUNSUPPORTED, "attn_decode_static: device ordinal %d >= 64", dev);
    return nullptr;
  }
  *dev_out = dev;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cuda_fail(e, "attn_decode_static: cudaGetSymbolAddress");
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" {

kvq_status attn_decode_static(const kvq_layer* layer, const kvq_seq_cache* seqs, int32_t n_seqs,
                              const int32_t* pos, int32_t max_pos, const uint16_t* q_raw,
                              const uint16_t* q_norm_w, void* out, int32_t out_is_f32, uint16_t* q_prepped,
                              void* stream) {
  if (!max_pos_ok(max_pos)) return fail(KVQ_EINVAL, "max_pos %d not in [0, 2^24)", max_pos);
  kvq::LayerArgs L;
  kvq_status st = check_layer(layer, &L);
  if (st != KVQ_OK) return st;
  if (n_seqs < 0) return fail(KVQ_EINVAL, "negative n_seqs");
  const size_t need = attn_decode_workspace_bytes(layer, n_seqs, max_pos);
  if (need > (size_t)KVQ_STATIC_SCRATCH_BYTES)
    return fail(KVQ_EWORKSPACE,
                "attn_decode_static: this call needs %zu bytes of scratch, more than the %zu-byte "
                "static buffer; use attn_decode with a caller-provided workspace",
                need, (size_t)KVQ_STATIC_SCRATCH_BYTES);
  int dev = 0;
  void* scratch = static_scratch_address(&dev);
  if (!scratch) return KVQ_ECUDA;
  return attention_common(layer, seqs, n_seqs, nullptr, pos, n_seqs, max_pos + 1, true, 0, q_raw, q_norm_w, out,
                          out_is_f32, q_prepped, scratch, (size_t)KVQ_STATIC_SCRATCH_BYTES, stream);
}

kvq_status kvq_static_status(uint32_t* status, void* stream) {
  if (!status || !aligned(status, 4)) return fail(KVQ_EINVAL, "status is NULL or not 4-byte aligned");
  const cudaError_t e = cudaMemcpyFromSymbolAsync(status, g_static_scratch, sizeof(uint32_t), 0, cudaMemcpyDefault,
                                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kvq_static_status copy");
  return KVQ_OK;
}

kvq_status kvq_selftest_wait_timeout(uint32_t* status, uint64_t limit_ns, void* stream) {
  if (!status || !aligned(status, 4)) return fail(KVQ_EINVAL, "status is NULL or not 4-byte aligned");
  if (limit_ns < 1000u || limit_ns > 1000000000u)
    return fail(KVQ_EINVAL, "limit_ns %llu not in [1e3, 1e9]", (unsigned long long)limit_ns);
  const cudaError_t e = kvq::launch_wait_selftest(status, limit_ns, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kvq_selftest_wait_timeout launch");
  return KVQ_OK;
}

// ---------------------------------------------------------------------------
// The training forward's stateless read: plain keys and values of a donor
// layer, then the read of any layer under the prefix-shared block layout.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace {

kvq_status check_layout(int32_t n_blocks, const int32_t* block_offsets, int32_t n_rows) {
  if (n_blocks < 1 || n_blocks > 65535) return fail(KVQ_EINVAL, "n_blocks %d not in [1, 65535]", n_blocks);
  if (n_rows < 0 || n_rows >= (1 << 24)) return fail(KVQ_EINVAL, "n_rows %d not in [0, 2^24)", n_rows);
  REQUIRE_PTR(block_offsets, "block_offsets", 4);
  return KVQ_OK;
}

kvq_status check_train_layer(const kvq_layer* layer, kvq::LayerArgs* L) {
  const kvq_status st = check_layer(layer, L);
  if (st != KVQ_OK) return st;
  if (L->rot) return fail(KVQ_EUNSUPPORTED, "the training read takes plain keys and values (rot_signs must be NULL)");
  return KVQ_OK;
}

}  // namespace

extern "C" {

kvq_status kvq_train_kv_prep(const kvq_layer* layer, int32_t n_blocks, const int32_t* block_offsets, int32_t n_rows,
                             const uint16_t* k_raw, const uint16_t* v_raw, const uint16_t* k_norm_w,
                             uint16_t* k_hat, uint16_t* v_hat, void* stream) {
  kvq::LayerArgs L;
  kvq_status st = check_train_layer(layer, &L);
  if (st != KVQ_OK) return st;
  if ((st = check_layout(n_blocks, block_offsets, n_rows)) != KVQ_OK) return st;
  if (n_rows == 0) return KVQ_OK;
  REQUIRE_PTR(k_raw, "k_raw", 16);
  REQUIRE_PTR(k_norm_w, "k_norm_w", 2);
  if (L.k_eq_v) {
    if (v_raw) return fail(KVQ_EINVAL, "v_raw must be NULL when k_eq_v = 1");
  } else {
    REQUIRE_PTR(v_raw, "v_raw", 16);
  }
  REQUIRE_PTR(k_hat, "k_hat", 16);
  REQUIRE_PTR(v_hat, "v_hat", 16);
  kvq::AppendArgs a = {};
  a.L = L;
  a.seqs = nullptr;
  a.n_seqs = n_blocks;
  a.row_offsets = block_offsets;
  a.start_pos = nullptr;
  a.n_rows = n_rows;
  a.k_raw = k_raw;
  a.v_raw = v_raw;
  a.k_w = k_norm_w;
  a.out_k = k_hat;
  a.out_v = v_hat;
  const kvq::RopeFreqs& f = rope_freqs(layer->rope_theta, L.D, L.rope_dims);
  const cudaError_t e = kvq::launch_append(a, f, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kvq_train_kv_prep launch");
  return KVQ_OK;
}

size_t attn_train_workspace_bytes(const kvq_layer* layer, int32_t n_rows) {
  kvq::LayerArgs L;
  if (check_layer(layer, &L) != KVQ_OK || n_rows < 0 || n_rows >= (1 << 24)) return 0;
  return kvq::train_ws_bytes(n_rows, L);
}

kvq_status attn_train_forward(const kvq_layer* layer, int32_t n_blocks, const int32_t* block_offsets, int32_t n_rows,
                              int32_t max_block_rows, const uint16_t* q_raw, const uint16_t* q_norm_w,
                              const uint16_t* k_hat, const uint16_t* v_hat, void* out, int32_t out_is_f32,
                              uint16_t* q_prepped, void* workspace, size_t workspace_bytes, void* stream) {
  kvq::LayerArgs L;
  kvq_status st = check_train_layer(layer, &L);
  if (st != KVQ_OK) return st;
  if (!kvq::train_supported(L))
    return fail(KVQ_EUNSUPPORTED, "training read: n_q_heads / n_kv_heads = %d must divide 128", L.G);
  if ((st = check_layout(n_blocks, block_offsets, n_rows)) != KVQ_OK) return st;
  if (n_rows == 0) return KVQ_OK;
  if (max_block_rows < 1 || max_block_rows > n_rows)
    return fail(KVQ_EINVAL, "max_block_rows %d not in [1, n_rows]", max_block_rows);
  REQUIRE_PTR(q_raw, "q_raw", 16);
  REQUIRE_PTR(q_norm_w, "q_norm_w", 2);
  REQUIRE_PTR(k_hat, "k_hat", 16);
  REQUIRE_PTR(v_hat, "v_hat", 16);
  REQUIRE_PTR(out, "out", out_is_f32 ? 4 : 2);
  REQUIRE_PTR(workspace, "workspace", 256);
  if (q_prepped && !aligned(q_prepped, 2)) return fail(KVQ_EINVAL, "q_prepped is not 2-byte aligned");
  if (out_is_f32 != 0 && out_is_f32 != 1) return fail(KVQ_EINVAL, "out_is_f32 must be 0 or 1");
  const size_t need = kvq::train_ws_bytes(n_rows, L);
  if (workspace_bytes < need) return fail(KVQ_EWORKSPACE, "workspace %zu bytes < %zu required", workspace_bytes, need);
  kvq::TrainArgs t = {};
  t.L = L;
  t.n_rows = n_rows;
  t.n_blocks = n_blocks;
  t.off = block_offsets;
  t.out = out;
  t.out_f32 = out_is_f32;
  const kvq::RopeFreqs& f = rope_freqs(layer->rope_theta, L.D, L.rope_dims);
  const cudaError_t e = kvq::launch_train(t, q_raw, q_norm_w, k_hat, v_hat, q_prepped, workspace, max_block_rows, f,
                                          static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "attn_train_forward launch");
  return KVQ_OK;
}

kvq_status attn_train_donor_forward(const kvq_layer* layer, int32_t n_blocks, const int32_t* block_offsets,
                                    int32_t n_rows, int32_t max_block_rows, const uint16_t* q_raw,
                                    const uint16_t* k_raw, const uint16_t* v_raw, const uint16_t* q_norm_w,
                                    const uint16_t* k_norm_w, uint16_t* k_hat, uint16_t* v_hat, void* out,
                                    int32_t out_is_f32, uint16_t* q_prepped, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  kvq::LayerArgs L;
  kvq_status st = check_train_layer(layer, &L);
  if (st != KVQ_OK) return st;
  if (!kvq::train_supported(L))
    return fail(KVQ_EUNSUPPORTED, "training read: n_q_heads / n_kv_heads = %d must divide 128", L.G);
  if ((st = check_layout(n_blocks, block_offsets, n_rows)) != KVQ_OK) return st;
  if (n_rows == 0) return KVQ_OK;
  if (max_block_rows < 1 || max_block_rows > n_rows)
    return fail(KVQ_EINVAL, "max_block_rows %d not in [1, n_rows]", max_block_rows);
  REQUIRE_PTR(q_raw, "q_raw", 16);
  REQUIRE_PTR(q_norm_w, "q_norm_w", 2);
  REQUIRE_PTR(k_raw, "k_raw", 16);
  REQUIRE_PTR(k_norm_w, "k_norm_w", 2);
  if (L.k_eq_v) {
    if (v_raw) return fail(KVQ_EINVAL, "v_raw must be NULL when k_eq_v = 1");
  } else {
    REQUIRE_PTR(v_raw, "v_raw", 16);
  }
  REQUIRE_PTR(k_hat, "k_hat", 16);
  REQUIRE_PTR(v_hat, "v_hat", 16);
  REQUIRE_PTR(out, "out", out_is_f32 ? 4 : 2);
  REQUIRE_PTR(workspace, "workspace", 256);
  if (q_prepped && !aligned(q_prepped, 2)) return fail(KVQ_EINVAL, "q_prepped is not 2-byte aligned");
  if (out_is_f32 != 0 && out_is_f32 != 1) return fail(KVQ_EINVAL, "out_is_f32 must be 0 or 1");
  const size_t need = kvq::train_ws_bytes(n_rows, L);
  if (workspace_bytes < need) return fail(KVQ_EWORKSPACE, "workspace %zu bytes < %zu required", workspace_bytes, need);
  kvq::AppendArgs ap = {};
  ap.L = L;
  ap.seqs = nullptr;
  ap.n_seqs = n_blocks;
  ap.row_offsets = block_offsets;
  ap.start_pos = nullptr;
  ap.n_rows = n_rows;
  ap.k_raw = k_raw;
  ap.v_raw = v_raw;
  ap.k_w = k_norm_w;
  ap.out_k = k_hat;
  ap.out_v = v_hat;
  kvq::TrainArgs t = {};
  t.L = L;
  t.n_rows = n_rows;
  t.n_blocks = n_blocks;
  t.off = block_offsets;
  t.out = out;
  t.out_f32 = out_is_f32;
  const kvq::RopeFreqs& f = rope_freqs(layer->rope_theta, L.D, L.rope_dims);
  const cudaError_t e = kvq::launch_train(t, q_raw, q_norm_w, k_hat, v_hat, q_prepped, workspace, max_block_rows, f,
                                          static_cast<cudaStream_t>(stream), &ap);
  if (e != cudaSuccess) return cuda_fail(e, "attn_train_donor_forward launch");
  return KVQ_OK;
}

kvq_status kvq_profile_next_read(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr))
    return fail(KVQ_EINVAL, "give both events or neither");
  g_prof_start = static_cast<cudaEvent_t>(start_event);
  g_prof_stop = static_cast<cudaEvent_t>(stop_event);
  return KVQ_OK;
}

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_EINVAL: return "invalid argument";
    case KVQ_EUNSUPPORTED: return "unsupported shape";
    case KVQ_ECUDA: return "CUDA error";
    case KVQ_EWORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

const char* kvq_last_error(void) { return g_last_error.c_str(); }

int32_t kvq_version(void) { return 130; }

}  // extern "C"
