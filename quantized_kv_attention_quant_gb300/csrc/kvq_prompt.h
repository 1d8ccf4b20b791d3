// Launch interface of the sliding-window prompt path on the tensor cores
// (kvq_prompt.cu): dequantize each visible key once into the workspace, then
// read it with tcgen05 MMAs fed by the tensor memory accelerator.
#pragma once
#include <cstddef>

#include "kvq_internal.h"

namespace kvq {

// Sliding layers (window > 0) with head_dim <= 256, G | 128, no rotation.
bool prompt_tc_supported(const LayerArgs& L);
// Status word, q_hat as f16, and the k_hi / k_lo / v scratch of
// window + max_rows - 1 keys (rounded up to whole tiles) per sequence.
size_t prompt_tc_ws_bytes(int n_seqs, int n_rows, int max_rows_per_seq, const LayerArgs& L);
// ap: NULL, or the rows' K/V append, run in the q prep's grid (the key
// dequantization that follows reads the appended rows)
cudaError_t launch_prompt_tc(const DecodeArgs& a, void* ws, int max_rows_per_seq, const RopeFreqs& f,
                             cudaStream_t st, const AppendArgs* ap = nullptr);

}  // namespace kvq
