// Internal launch interfaces between the C ABI (kvq_api.cu) and the kernels.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kMaxRopeHalf = 256;   // head_dim <= 512
constexpr int kTileKeys = 64;       // keys per pipeline tile; capacities are multiples of it
constexpr int kMaxG = 16;           // q heads per kv head handled by one MMA row block

// theta^(-2j/D) for j < rope_dims/2, each as an exact sum of three floats.
struct alignas(16) RopeFreqs {
  float f[kMaxRopeHalf][3];
};

struct LayerArgs {
  int n_q, n_kv, D, G, window, rope_dims, k_eq_v;
  float eps;
  const int8_t* rot;    // signs of the deferred TurboQuant read (device), or nullptr
  float qk_scale;       // score scale: 1, or 1/D on a rotated layer (a power of two)
};

struct AppendArgs {
  LayerArgs L;
  const kvq_seq_cache* seqs;
  int n_seqs;
  const int32_t* row_offsets;   // nullptr: one row per sequence (row s is sequence s)
  const int32_t* start_pos;
  int n_rows;
  const uint16_t* k_raw;
  const uint16_t* v_raw;
  const uint16_t* k_w;
  uint16_t* prepped;
  // training read (seqs == nullptr): the prepped rows are the output, written
  // to out_k / out_v [n_rows][n_kv][D], and nothing is quantized
  uint16_t* out_k;
  uint16_t* out_v;
  // prompt chunks read on the dequantize-once tensor-core path (sk_hi
  // non-null): each stored row's dequantized key (as k_hi + k_lo f16) or
  // value (f16) also goes to the read's scratch [n_seqs * sks][n_kv][D],
  // whose row 0 of sequence s is position max(0, start_pos[s] - window + 1)
  uint16_t* sk_hi;
  uint16_t* sk_lo;
  uint16_t* sv;
  int sks;
};

// Workspace of the attention calls, carved from the caller's buffer.
struct DecodeWs {
  uint32_t* status;     // 1 word (padded to 256 B)
  uint4* qfrag;         // [n_rows][n_kv][NG][4][32] x uint4
  uint4* qbias;         // [n_rows][n_kv][32] x uint4: A fragment of the QK bias term
  float* part_o;        // [n_rows][n_kv][splits][16][D]
  float* part_ml;       // [n_rows][n_kv][splits][2][16]  (m, l)
                        // stream-K: part_o / part_ml hold [ctas][2] pieces instead
  long long* plan;      // stream-K: T, nc, then the row tile prefix [n_rows + 1]
  // prompt-chunk tensor-core path only
  uint16_t* q16;        // [n_rows][n_q][D] q_hat as f16
  float* qsum;          // [n_rows][n_q][D/64] per-group sums of those f16 values
  // training-read path only
  uint16_t* qhat;       // [n_rows][n_q][D] q_hat as bf16
};

// Query rows of an attention call.  Decode: row i is sequence i at position
// pos[i] (row_offsets == nullptr).  Prompt chunk: row i belongs to the
// sequence s with row_offsets[s] <= i < row_offsets[s+1] and sits at position
// pos[s] + (i - row_offsets[s]); the sequence's newest cached position is its
// last row's.  Training read (pos == nullptr): the row_offsets are the blocks
// of a prefix-shared layout, block 0 (the prefix) starting at position 0 and
// every other block at position row_offsets[1].
struct DecodeArgs {
  LayerArgs L;
  const kvq_seq_cache* seqs;
  int n_seqs;
  int n_rows;
  const int32_t* row_offsets;
  const int32_t* pos;
  const uint16_t* q_raw;
  const uint16_t* q_w;
  void* out;
  int out_f32;
  uint16_t* q_prepped;
  int splits;
  int chunk_tiles;      // > 0: every split covers this many tiles; 0: ceil(row tiles / splits)
  int sk_ctas;          // > 0: stream-K schedule over this many CTAs (splits / chunk_tiles unused)
  // 1: the call's first kernel also appends each row's new K/V (the row's
  // position is its newest key), so the tile holding a row's newest key is
  // copied only once that kernel is complete
  int fused_append;
  DecodeWs ws;
};

// Several calls of one layer in one launch of each decode-path kernel (q
// prep, attention, merge): group g's rows are rows [row_base[g],
// row_base[g+1]) of the q prep and merge grids, its fixed-chunk CTAs
// [cta_base[g], cta_base[g+1]) of the attention grid, in (row, kv head,
// split) order.  Every group keeps its own arguments (sequences, positions,
// rows, q, output, workspace, plan); the layer is the same for all.
constexpr int kMaxGroups = KVQ_MAX_MIXED_GROUPS;
struct GroupedDecode {
  int n;
  int row_base[kMaxGroups + 1];
  int cta_base[kMaxGroups + 1];
  DecodeArgs g[kMaxGroups];
};

constexpr int kChunkTiles = 48;   // target tiles per split when the longest row is known
// Stream-K decode: used for decode calls whose longest row spans several
// chunks and whose row count fits the plan held in shared memory.
constexpr int kSkMaxRows = 1024;
constexpr int kSkMinTiles = 16;   // shortest range per CTA
struct DecodePlan { int splits, chunk_tiles, sk_ctas; };
size_t decode_ws_bytes(int n_rows, int n_kv, int D, const DecodePlan& plan);
DecodeWs decode_ws_carve(void* base, int n_rows, int n_kv, int D, const DecodePlan& plan);
DecodePlan decode_plan(const LayerArgs& L, int n_rows, int max_keys, int num_sms, bool fixed_chunks);
// Fixed-chunk plans of the groups of a grouped launch (no stream-K): one
// wave shared by every group's (row, kv head) units.  rows, max_keys and
// fixed_chunks per group as for decode_plan; group g takes at most
// max_splits[g] >= 1 splits (what its workspace holds).
void decode_plan_grouped(const LayerArgs& L, int n, const int* rows, const int* max_keys, const bool* fixed_chunks,
                         const int* max_splits, int num_sms, DecodePlan* plans);
// The most splits of a fixed-chunk plan whose workspace for n_rows rows fits
// in `bytes` (0 when not even one split fits).
int decode_max_splits(int n_rows, int n_kv, int D, size_t bytes);

// Prompt chunks on the tensor cores (tcgen05): head_dim <= 256 and G | 128.
bool prefill_tc_supported(const LayerArgs& L);
size_t prefill_tc_ws_bytes(int n_rows, const LayerArgs& L);
DecodeWs prefill_tc_ws_carve(void* base, int n_rows, const LayerArgs& L);
// ap: NULL, or the rows' K/V append, run in the q prep's grid (the read that
// follows reads the appended rows)
cudaError_t launch_prefill_tc(const DecodeArgs& a, const RopeFreqs& f, int max_rows_per_seq, cudaStream_t st,
                              const AppendArgs* ap = nullptr);

cudaError_t launch_append(const AppendArgs& a, const RopeFreqs& f, cudaStream_t st);

// The training forward's stateless read (tcgen05): q prep, then the read of
// the plain bf16 keys and values under the prefix-shared block mask.
struct TrainArgs {
  LayerArgs L;
  int n_rows, n_blocks;
  const int32_t* off;   // block offsets [n_blocks + 1]
  void* out;
  int out_f32;
};
bool train_supported(const LayerArgs& L);
size_t train_ws_bytes(int n_rows, const LayerArgs& L);
// ap: NULL, or the donor's K/V prep of the pass (writing k_hat / v_hat), run
// in the q prep's grid
cudaError_t launch_train(const TrainArgs& t, const uint16_t* q_raw, const uint16_t* q_w, const uint16_t* k_hat,
                         const uint16_t* v_hat, uint16_t* q_prepped, void* ws, int max_block_rows,
                         const RopeFreqs& f, cudaStream_t st, const AppendArgs* ap = nullptr);
// One CTA whose bounded wait on an mbarrier that nothing completes gives up
// after limit_ns and flags the timeout bit in *status.
cudaError_t launch_wait_selftest(uint32_t* status, unsigned long long limit_ns, cudaStream_t st);
cudaError_t launch_decode(const DecodeArgs& a, const RopeFreqs& f, int num_sms, cudaStream_t st);
// Profiling (kvq_profile_next_read): the events the calling host thread's
// next attention call records on its stream right before and right after
// launching its attention kernel; prof_after also clears them.
cudaError_t prof_before(cudaStream_t st);
cudaError_t prof_after(cudaStream_t st);
// The grouped launch (fixed-chunk plans in every group, ga.n >= 1).
cudaError_t launch_decode_grouped(const GroupedDecode& ga, const RopeFreqs& f, cudaStream_t st);
// attn_decode_append: one kernel preps q and appends each sequence's new K/V
// row (ap: one row per sequence, ap.start_pos == a.pos), then the attention
// and merge kernels of launch_decode (a.fused_append == 1).
cudaError_t launch_decode_append(const DecodeArgs& a, const AppendArgs& ap, const RopeFreqs& f, cudaStream_t st);

}  // namespace kvq
