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
  // training read: the prefix starts at 0, every branch continues it
  const int p0 = a.pos ? __ldg(a.pos + lo) : (lo == 0 ? 0 : __ldg(a.row_offsets + 1));
  return {lo, p0 + (row - o0), p0 + (o1 - o0) - 1};
}

// ----------------------------------------------------------------------------
// q prep of the decode kernels: one block per (row, block of heads), laid
// out for latency (few rows per call).  The block first evaluates the row's
// RoPE angles once for all its heads (the float-float sine/cosine is the
// costly part), then each head's TH threads of E elements RMS-normalise and
// rotate it.  Outputs: the mma.sync A fragments of every head slot of the
// row's kv heads (slots >= G are zeros) and the bias-term fragment (each
// 32-bit fragment word holds two dims of ONE head, so heads write disjoint
// words), and q_hat (bf16) in q_prepped when it is given.  Calls with many
// rows use qprep_rows_kernel (kvq_qrows.cuh).
// ----------------------------------------------------------------------------
template <int D>
struct Qp {
  static constexpr int TH = D / 4 >= 32 ? D / 4 : 32;                         // threads per head
  static constexpr int E = D / TH;                                            // elements per thread
  static constexpr int HW = TH / 32;                                          // warps per head
  static constexpr int TPG = 64 / E;                                          // threads per 64-dim group
  static constexpr int HPB = 1024 / TH;                                       // most heads per block
};

// heads per block and blocks per row for n_q heads
template <int D>
inline void qprep_shape(int n_q, int& hpb, int& nblk) {
  hpb = n_q < Qp<D>::HPB ? n_q : Qp<D>::HPB;
  nblk = (n_q + hpb - 1) / hpb;
}

// One block: row `row` of the call `a`, heads hb*hpb .. hb*hpb + hpb - 1.
template <int D>
__device__ __forceinline__ void qprep_block(const DecodeArgs& a, const RopeFreqs& freqs, const int hpb,
                                            const int row, const int hb) {
  using Q = Qp<D>;
  constexpr int E = Q::E, NG = D / 64, TH = Q::TH;
  __shared__ uint16_t qn[Q::HPB * D];      // normed, then q_hat, per head of the block
  __shared__ float4 cs[D / 2];             // (cos.hi, cos.lo, sin.hi, sin.lo) per rotated pair
  __shared__ __align__(16) float freq[D / 2][3];
  __shared__ ff red[Q::HPB][Q::HW];
  __shared__ float qs[Q::HPB][8];          // per-group sums of the f16 q values
  extern __shared__ double rot_rows[];     // [hpb][D], rotated layers only
  const int tid = threadIdx.x, hl = tid / TH, tt = tid % TH, lane = tid & 31;
  const int G = a.L.G, R = a.L.rope_dims, half = R >> 1;
  // Launched as a programmatic dependent of the stream's previous kernel:
  // until that grid is complete only the library's own frequency table is
  // read; every caller buffer (q, positions, descriptors, the workspace) is
  // touched after the wait.  The attention kernel may launch only after it
  // too, so that its ring reads caches an earlier append has finished.
  if (R > 0) stage_freqs(freqs.f, half, freq);
  pdl_wait();
  // the first kernel of an attention call clears its status word; the later
  // kernels flag errors only once this grid is complete
  if (row == 0 && hb == 0 && tid == 0) *a.ws.status = 0u;
  pdl_launch();
  const int hq = hb * hpb + hl;                           // q head of this thread
  const bool active = hl < hpb && hq < a.L.n_q;
  // the raw row and the norm weight first: their latency overlaps the row
  // lookup and the angles
  float x[E], wq[E];
  if (active) {
    const uint16_t* src = a.q_raw + ((size_t)row * a.L.n_q + hq) * D + tt * E;
#pragma unroll
    for (int v = 0; v < E; v += 2) {
      const uint32_t u = *reinterpret_cast<const uint32_t*>(src + v);
      x[v] = bf16lo_to_f(u);
      x[v + 1] = bf16hi_to_f(u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) x[i] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < E; ++i) wq[i] = bf16_to_f(a.q_w[tt * E + i]);
  const RowInfo ri = row_info(a, row);
  const int bits = a.seqs ? a.seqs[ri.s].bits : 8;
  const int pc = min(max(ri.p, 0), (1 << 24) - 1);

  // ---- the row's rotation angles, once for all heads ----
  if (R > 0) {
    __syncthreads();                       // the staged frequencies
    for (int j = tid; j < half; j += blockDim.x) {
      ff cc, sn;
      rope_cos_sin(pc, freq[j][0], freq[j][1], freq[j][2], cc, sn);
      cs[j] = make_float4(cc.hi, cc.lo, sn.hi, sn.lo);
    }
  }

  // ---- RMSNorm of this thread's E elements ----
  uint16_t y[E];
  ff ss = {0.f, 0.f};
#pragma unroll
  for (int i = 0; i < E; ++i) ff_acc_sq(ss, x[i]);
  ss = ff_warp_sum(ss);
  if constexpr (Q::HW > 1) {
    if (lane == 0 && hl < Q::HPB) red[hl][(tt >> 5)] = ss;
    __syncthreads();
    if (hl < Q::HPB) {
      ss = red[hl][0];
#pragma unroll
      for (int w = 1; w < Q::HW; ++w) ss = ff_add(ss, red[hl][w]);
    }
  }
  uint16_t* qh = qn + (hl < Q::HPB ? hl : 0) * D;
  if (active) {
    const ff inv = rms_inv(ss, D, a.L.eps);
#pragma unroll
    for (int i = 0; i < E; ++i) {
      y[i] = norm_scale_bf16(x[i], wq[i], inv);
      qh[tt * E + i] = y[i];
    }
  }
  __syncthreads();                         // angles and normed rows complete

  // ---- RoPE ----
  if (R > 0 && active) {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const int e = tt * E + i;
      if (e < R) {
        // x_e c - x_(e+h) s below half, x_e c + x_(e-h) s above: one call
        const bool lo = e < half;
        const int j = lo ? e : e - half;
        const float4 cv = cs[j];
        y[i] = rot_bf16(bf16_to_f(qh[e]), bf16_to_f(qh[lo ? e + half : j]), ff{cv.x, cv.y},
                        lo ? ff{cv.z, cv.w} : ff{-cv.z, -cv.w});
      }
    }
  }
  __syncthreads();                         // every read of the normed rows is done
  // the deferred TurboQuant read: q_hat R, rounded to bf16 like K and V
  if (a.L.rot) rotate_row_bf16<D, E, TH>(y, a.L.rot, rot_rows + (hl < Q::HPB ? hl : 0) * D, tt, active);
  float gs = 0.f;
  if (active) {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      qh[tt * E + i] = y[i];
      gs += __half2float(__float2half_rn(bf16_to_f(y[i])));   // the f16 value the MMA multiplies
    }
  }
#pragma unroll
  for (int m = 1; m < Q::TPG; m <<= 1) gs += __shfl_xor_sync(0xffffffffu, gs, m);
  if (active) {
    if (tt % Q::TPG == 0) qs[hl][tt / Q::TPG] = gs;
    if (a.q_prepped) {
      uint16_t* dst = a.q_prepped + ((size_t)row * a.L.n_q + hq) * D + tt * E;
#pragma unroll
      for (int i = 0; i < E; ++i) dst[i] = y[i];
    }
  }
  __syncthreads();                         // q_hat and the group sums complete
  if (!active) return;
  const int kvh = hq / G, h = hq % G;
  uint32_t* frag = reinterpret_cast<uint32_t*>(a.ws.qfrag) + ((size_t)row * a.L.n_kv + kvh) * NG * 4 * 32 * 4;
  uint32_t* qb = reinterpret_cast<uint32_t*>(a.ws.qbias) + ((size_t)row * a.L.n_kv + kvh) * 128;
  // fragment words of head slot h: lanes with lane/4 == h % 8, register 0/2 (h < 8) or 1/3
  {
    const int rq = h & 7, reg_lo = h < 8 ? 0 : 1;
    for (int i = tt; i < NG * 4 * 4 * 2; i += TH) {
      const int pair = i & 1, t4 = (i >> 1) & 3, ks = (i >> 3) & 3, g = i >> 5;
      int d[4];
      qk_dims(bits, ks, d);
      const int base = g * 64 + 16 * t4;
      const int d0 = base + (pair ? d[2] : d[0]), d1 = base + (pair ? d[3] : d[1]);
      // with 4-bit codes the second k-half of every step multiplies codes read
      // from bits 4..7 (16 times too large as f16 subnormals): q/16 there
      const float f = (bits == 4 && pair) ? 0.0625f : 1.f;
      frag[((g * 4 + ks) * 32 + rq * 4 + t4) * 4 + reg_lo + 2 * pair] =
          pack_h2(bf16_to_f(qh[d0]) * f, bf16_to_f(qh[d1]) * f);
    }
    // bias-term A fragment words of slot h: k = group (hi part) | 8 + group (lo part)
    if (tt < 8) {
      const int t4 = tt & 3, lo_part = tt >> 2;
      float v[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int g = 2 * t4 + e;
        // the bias term meets the scores' scale (1, or 1/D exactly on a rotated layer)
        const float xs = g < NG ? qs[hl][g] * a.L.qk_scale : 0.f;
        const float hi = __half2float(__float2half_rn(xs));
        v[e] = lo_part ? xs - hi : hi;
      }
      qb[(rq * 4 + t4) * 4 + reg_lo + 2 * lo_part] = pack_h2(v[0], v[1]);
    }
  }
  // the last q head of a kv head also zero-fills the unused slots G .. 15
  if (h == G - 1) {
    for (int hz = G; hz < kMaxG; ++hz) {
      const int rq = hz & 7, reg_lo = hz < 8 ? 0 : 1;
      for (int i = tt; i < NG * 4 * 4 * 2; i += TH) {
        const int pair = i & 1, t4 = (i >> 1) & 3, ks = (i >> 3) & 3, g = i >> 5;
        frag[((g * 4 + ks) * 32 + rq * 4 + t4) * 4 + reg_lo + 2 * pair] = 0u;
      }
      if (tt < 8) qb[(rq * 4 + (tt & 3)) * 4 + reg_lo + 2 * (tt >> 2)] = 0u;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(1024)
qprep_kernel(const DecodeArgs a, const RopeFreqs freqs, const int hpb) {
  qprep_block<D>(a, freqs, hpb, blockIdx.x, blockIdx.y);
}

// The group of block x of a grouped grid whose groups start at base[0..n).
__device__ __forceinline__ int group_of(const int* base, int n, int x) {
  int g = 0;
  for (int i = 1; i < n; ++i)
    if (x >= base[i]) g = i;
  return g;
}

// Grouped schedule: the rows of every group in one grid (rows, head blocks).
template <int D>
__global__ void __launch_bounds__(1024)
qprep_grouped_kernel(const GroupedDecode ga, const RopeFreqs freqs, const int hpb) {
  const int g = group_of(ga.row_base, ga.n, blockIdx.x);
  qprep_block<D>(ga.g[g], freqs, hpb, blockIdx.x - ga.row_base[g], blockIdx.y);
}

}  // namespace
}  // namespace kvq
