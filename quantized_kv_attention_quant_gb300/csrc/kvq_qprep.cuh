// Shared pieces of the attention kernels: descriptor checks, the mapping of
// query rows to sequences and positions, and the q prep kernel (q RMSNorm
// and RoPE, model.ts attentionTraining: qNorm, then RoPE at the cache offset).
#pragma once
#include "kvq_common.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

__device__ __forceinline__ bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

__device__ __forceinline__ bool seq_ok(const kvq_seq_cache& c) {
  return (c.bits == 4 || c.bits == 8) && c.capacity > 0 && (c.capacity % kTileKeys) == 0 &&
         aligned16(c.k_codes) && aligned16(c.v_codes) && aligned16(c.k_scales) &&
         aligned16(c.k_biases) && aligned16(c.v_scales) && aligned16(c.v_biases) &&
         c.k_codes && c.v_codes && c.k_scales && c.k_biases && c.v_scales && c.v_biases;
}

// Dims (relative to the thread's 16-dim slice 16*t4 of a group) that feed A
// fragment registers a0, a1, a4, a5 of k-step ks.  They mirror how the code
// words are split into f16 pairs for the B fragment (nibbles (i, i+4) of a
// 4-bit word, bytes (i, i+2) of an 8-bit word).
__device__ __forceinline__ void qk_dims(int bits, int ks, int (&d)[4]) {
  if (bits == 4) {
    const int base = (ks < 2 ? 0 : 8) + (ks & 1) * 2;
    d[0] = base; d[1] = base + 4; d[2] = base + 1; d[3] = base + 5;
  } else {
    const int base = 4 * ks;
    d[0] = base; d[1] = base + 2; d[2] = base + 1; d[3] = base + 3;
  }
}

struct RowInfo { int s, p, newest; };

__device__ __forceinline__ RowInfo row_info(const DecodeArgs& a, int row) {
  if (a.row_offsets == nullptr) {
    const int p = a.pos[row];
    return {row, p, p};
  }
  int lo = 0, hi = a.n_seqs - 1;           // largest s with row_offsets[s] <= row
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.row_offsets + mid) <= row) lo = mid; else hi = mid - 1;
  }
  const int o0 = __ldg(a.row_offsets + lo), o1 = __ldg(a.row_offsets + lo + 1);
  const int p0 = __ldg(a.pos + lo);
  return {lo, p0 + (row - o0), p0 + (o1 - o0) - 1};
}

// ----------------------------------------------------------------------------
// 1. q prep: one block per (row, kv head, q head slot h < 16), max(32, D/4)
// threads of 4 (or 2) elements.  Writes q_hat (bf16), the head's words of the
// QK A fragments and of the bias-term A fragment (rows >= G are zeros).
// Each 32-bit fragment word holds two dims of ONE row, so blocks of different
// heads write disjoint words.
// ----------------------------------------------------------------------------
template <int D>
struct Qp {
  static constexpr int THREADS = D / 4 >= 32 ? D / 4 : 32;
  static constexpr int E = D / THREADS;
  static constexpr int NWARP = THREADS / 32;
  static constexpr int TPG = 64 / E;
};

// ROWS = false: decode (mma.sync fragments, grid z = 16 head slots);
// ROWS = true: prompt chunk (q_hat as f16 rows and per-group sums of those
// f16 values, grid z = G heads).
template <int D, bool ROWS>
__global__ void __launch_bounds__(Qp<D>::THREADS)
qprep_kernel(const DecodeArgs a, const RopeFreqs freqs) {
  using Q = Qp<D>;
  constexpr int E = Q::E, NG = D / 64;
  __shared__ uint16_t qn[D];               // normed, then q_hat
  __shared__ float4 cs[D / 2];
  __shared__ float freq[D / 2][3];
  __shared__ ff red[Q::NWARP];
  __shared__ float qs[8];                  // per-group sums of the f16 q values
  pdl_launch();
  const int row = blockIdx.x, kvh = blockIdx.y, h = blockIdx.z;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int G = a.L.G, R = a.L.rope_dims, half = R >> 1;
  const RowInfo ri = row_info(a, row);
  const int bits = a.seqs[ri.s].bits;
  uint32_t* frag = ROWS ? nullptr : reinterpret_cast<uint32_t*>(a.ws.qfrag) + ((size_t)row * a.L.n_kv + kvh) * NG * 4 * 32 * 4;
  uint32_t* qb = ROWS ? nullptr : reinterpret_cast<uint32_t*>(a.ws.qbias) + ((size_t)row * a.L.n_kv + kvh) * 128;
  // this row's fragment words: lanes with lane/4 == h % 8, register 0/2 (h < 8) or 1/3
  const int rq = h & 7, reg_lo = h < 8 ? 0 : 1;
  if (ROWS && h >= G) return;
  if (!ROWS && h >= G) {
    for (int i = t; i < NG * 4 * 4 * 2; i += Q::THREADS) {
      const int pair = i & 1, t4 = (i >> 1) & 3, ks = (i >> 3) & 3, g = i >> 5;
      frag[((g * 4 + ks) * 32 + rq * 4 + t4) * 4 + reg_lo + 2 * pair] = 0u;
    }
    if (t < 8) qb[(rq * 4 + (t & 3)) * 4 + reg_lo + 2 * (t >> 2)] = 0u;
    return;
  }
  if (R > 0) stage_freqs(freqs.f, half, freq);
  const int hq = kvh * G + h;
  const int pc = min(max(ri.p, 0), (1 << 24) - 1);
  const uint16_t* src = a.q_raw + ((size_t)row * a.L.n_q + hq) * D + t * E;
  float x[E];
  if constexpr (E == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(src);
    x[0] = bf16lo_to_f(u.x); x[1] = bf16hi_to_f(u.x); x[2] = bf16lo_to_f(u.y); x[3] = bf16hi_to_f(u.y);
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(src);
    x[0] = bf16lo_to_f(u); x[1] = bf16hi_to_f(u);
  }
  ff ss = {0.f, 0.f};
#pragma unroll
  for (int i = 0; i < E; ++i) ff_acc_sq(ss, x[i]);
  ss = ff_warp_sum(ss);
  if constexpr (Q::NWARP > 1) {
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    ss = red[0];
#pragma unroll
    for (int w = 1; w < Q::NWARP; ++w) ss = ff_add(ss, red[w]);
  }
  const ff inv = rms_inv(ss, D, a.L.eps);
  uint16_t y[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    y[i] = norm_scale_bf16(x[i], bf16_to_f(a.q_w[t * E + i]), inv);
    qn[t * E + i] = y[i];
  }
  __syncthreads();                         // freq[] staged, qn[] complete
  if (R > 0) {
    for (int j = t; j < half; j += Q::THREADS) {
      ff cc, sn;
      rope_cos_sin(pc, freq[j][0], freq[j][1], freq[j][2], cc, sn);
      cs[j] = make_float4(cc.hi, cc.lo, sn.hi, sn.lo);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const int e = t * E + i;
      if (e < R) {
        const int j = e < half ? e : e - half;
        const float4 cv = cs[j];
        const ff cc = {cv.x, cv.y};
        y[i] = e < half ? rot_bf16(bf16_to_f(qn[e]), bf16_to_f(qn[e + half]), cc, ff{cv.z, cv.w})
                        : rot_bf16(bf16_to_f(qn[e]), bf16_to_f(qn[j]), cc, ff{-cv.z, -cv.w});
      }
    }
    __syncthreads();                       // every read of the normed row is done
#pragma unroll
    for (int i = 0; i < E; ++i) qn[t * E + i] = y[i];
  }
  float gs = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) gs += __half2float(__float2half_rn(bf16_to_f(y[i])));   // the f16 value the MMA multiplies
#pragma unroll
  for (int m = 1; m < Q::TPG; m <<= 1) gs += __shfl_xor_sync(0xffffffffu, gs, m);
  if (t % Q::TPG == 0) qs[t / Q::TPG] = gs;
  if (a.q_prepped) {
    uint16_t* dst = a.q_prepped + ((size_t)row * a.L.n_q + hq) * D + t * E;
#pragma unroll
    for (int i = 0; i < E; ++i) dst[i] = y[i];
  }
  if constexpr (ROWS) {
    __half* dst = reinterpret_cast<__half*>(a.ws.q16) + ((size_t)row * a.L.n_q + hq) * D + t * E;
#pragma unroll
    for (int i = 0; i < E; ++i) dst[i] = __float2half_rn(bf16_to_f(y[i]));
    if (t % Q::TPG == 0) a.ws.qsum[((size_t)row * a.L.n_q + hq) * NG + t / Q::TPG] = gs;
    return;
  }
  __syncthreads();                         // q_hat and the group sums complete
  // QK A fragment words of row h: for each (group, k-step, t4) two words
  for (int i = t; i < NG * 4 * 4 * 2; i += Q::THREADS) {
    const int pair = i & 1, t4 = (i >> 1) & 3, ks = (i >> 3) & 3, g = i >> 5;
    int d[4];
    qk_dims(bits, ks, d);
    const int base = g * 64 + 16 * t4;
    const int d0 = base + (pair ? d[2] : d[0]), d1 = base + (pair ? d[3] : d[1]);
    // with 4-bit codes the second k-half of every step multiplies codes read
    // from bits 4..7 (16 times too large as f16 subnormals): q/16 there
    const float f = (bits == 4 && pair) ? 0.0625f : 1.f;
    frag[((g * 4 + ks) * 32 + rq * 4 + t4) * 4 + reg_lo + 2 * pair] =
        pack_h2(bf16_to_f(qn[d0]) * f, bf16_to_f(qn[d1]) * f);
  }
  // bias-term A fragment words of row h: k = group (hi part) | 8 + group (lo part)
  if (t < 8) {
    const int t4 = t & 3, lo_part = t >> 2;
    float v[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int g = 2 * t4 + e;
      const float xs = g < NG ? qs[g] : 0.f;
      const float hi = __half2float(__float2half_rn(xs));
      v[e] = lo_part ? xs - hi : hi;
    }
    qb[(rq * 4 + t4) * 4 + reg_lo + 2 * lo_part] = pack_h2(v[0], v[1]);
  }
}

}  // namespace
}  // namespace kvq
