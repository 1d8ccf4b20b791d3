// q prep for calls with many query rows (prompt chunks on the tensor cores,
// the training read): q RMSNorm and RoPE (model.ts attentionTraining: qNorm,
// then RoPE at the row's position), the same arithmetic as qprep_kernel in
// kvq_qprep.cuh, laid out for throughput instead of latency:
//   - a block of 8 warps takes `rb` consecutive rows; it stages the rotary
//     frequencies once and evaluates every (row, pair) angle of its rows once,
//     spread over all its threads;
//   - each warp then preps one (row, q head) at a time, D/32 elements per
//     lane: the float-float sum of squares is a warp reduction (no block
//     barrier); under full RoPE the partner of element e (e +- D/2) sits in
//     lane ^ 16 at the same index, one shuffle away; under partial RoPE the
//     rotated dims (a share of the row) are spread over all 32 lanes through
//     a per-warp shared row.
// Outputs: q_hat as bf16 (q_prepped and/or ws.qhat) and, for the prompt
// kernels, q_hat as f16 (ws.q16) with (when ws.qsum is given) the per-group
// sums of those f16 values.  Rotated layers do not come here.
#pragma once
#include <algorithm>

#include "kvq_append.cuh"
#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "kvq_qprep.cuh"

namespace kvq {
namespace {

constexpr int kQrWarps = 8;

// One block: rows bx*rb .. bx*rb + rb - 1 of the call `a`.
template <int D>
__device__ __forceinline__ void qprep_rows_block(const DecodeArgs& a, const RopeFreqs& freqs, const int rb,
                                                 const int bx) {
  constexpr int E = D / 32;                 // elements per lane
  constexpr int NG = D / 64, LPG = 64 / E;  // 64-dim groups; lanes per group
  extern __shared__ __align__(16) uint8_t qr_smem[];
  __shared__ int rpos[16];
  const int R = a.L.rope_dims, half = R >> 1, Hq = a.L.n_q;
  float4* cs = reinterpret_cast<float4*>(qr_smem);                        // [rb][half] (cos, sin) pairs
  // under full RoPE pair j = 16 * (j % E) + j / E of a row's table: the 16
  // lanes of a half read consecutive entries
  float (*freq)[3] = reinterpret_cast<float (*)[3]>(qr_smem + (size_t)rb * half * 16);
  uint16_t* nrm = reinterpret_cast<uint16_t*>(qr_smem + (size_t)rb * half * 16 + 16 * ((3 * half + 3) / 4));
  // per warp: the normed row, then the rotated dims
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row0 = bx * rb;
  // Launched as a programmatic dependent of the stream's previous kernel:
  // until that grid is complete only the library's frequency table is read
  if (R > 0) stage_freqs(freqs.f, half, freq);
  pdl_wait();
  if (bx == 0 && tid == 0) *a.ws.status = 0u;            // the first kernel of the call
  pdl_launch();

  float wq[E];                                          // (the weights are only 2-byte aligned)
#pragma unroll
  for (int i = 0; i < E; ++i) wq[i] = bf16_to_f(__ldg(a.q_w + lane * E + i));
  // ---- the rows' rotation angles, once per (row, pair) ----
  if (R > 0) {
    if (tid < rb) {
      const int row = row0 + tid;
      rpos[tid] = row < a.n_rows ? min(max(row_info(a, row).p, 0), (1 << 24) - 1) : 0;
    }
    __syncthreads();
    for (int idx = tid; idx < rb * half; idx += kQrWarps * 32) {
      const int r = idx / half, j = idx - r * half;
      ff cc, sn;
      rope_cos_sin(rpos[r], freq[j][0], freq[j][1], freq[j][2], cc, sn);
      cs[R == D ? r * half + (j % E) * 16 + j / E : idx] = make_float4(cc.hi, cc.lo, sn.hi, sn.lo);
    }
    __syncthreads();
  }

  // ---- one (row, q head) per warp at a time ----
  uint16_t* nr = nrm + warp * 2 * D;
  uint16_t* rt = nr + D;
  for (int it = warp; it < rb * Hq; it += kQrWarps) {
    const int r = it / Hq, hq = it - r * Hq;
    const int row = row0 + r;
    if (row >= a.n_rows) break;                         // later items are later rows
    const size_t base = ((size_t)row * Hq + hq) * D + lane * E;
    float x[E];
    const uint32_t* src = reinterpret_cast<const uint32_t*>(a.q_raw + base);
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      const uint32_t u = src[i / 2];
      x[i] = bf16lo_to_f(u);
      x[i + 1] = bf16hi_to_f(u);
    }
    // sum of squares in two independent float-float chains (more work in
    // flight per warp), joined before the warp reduction
    ff s0 = {0.f, 0.f}, s1 = {0.f, 0.f};
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      ff_acc_sq(s0, x[i]);
      ff_acc_sq(s1, x[i + 1]);
    }
    const ff ss = ff_warp_sum(ff_add(s0, s1));
    const ff inv = rms_inv(ss, D, a.L.eps);
    uint16_t y[E];
#pragma unroll
    for (int i = 0; i < E; ++i) y[i] = norm_scale_bf16(x[i], wq[i], inv);
    uint32_t yw[E / 2];
#pragma unroll
    for (int i = 0; i < E; i += 2) yw[i / 2] = (uint32_t)y[i] | ((uint32_t)y[i + 1] << 16);
    if (R == D) {
      // x_e c - x_(e+D/2) s in lanes 0..15, x_e c + x_(e-D/2) s in lanes 16..31
      const float4* csr = cs + r * half + (lane & 15);
      const bool upper = lane >= 16;
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const float xe = bf16_to_f(y[i]);
        const float xp = __shfl_xor_sync(0xffffffffu, xe, 16);
        const float4 cv = csr[i * 16];
        y[i] = rot_bf16(xe, xp, ff{cv.x, cv.y}, upper ? ff{-cv.z, -cv.w} : ff{cv.z, cv.w});
      }
#pragma unroll
      for (int i = 0; i < E; i += 2) yw[i / 2] = (uint32_t)y[i] | ((uint32_t)y[i + 1] << 16);
    } else if (R > 0) {
      // the normed row to shared memory; the rotated dims are then spread over
      // all lanes (dim e = lane + 32 k), whatever share of the row they are
      uint32_t* nw = reinterpret_cast<uint32_t*>(nr) + lane * (E / 2);
      if constexpr (E % 8 == 0) {
#pragma unroll
        for (int i = 0; i < E / 2; i += 4)
          *reinterpret_cast<uint4*>(nw + i) = make_uint4(yw[i], yw[i + 1], yw[i + 2], yw[i + 3]);
      } else {
#pragma unroll
        for (int i = 0; i < E / 2; ++i) nw[i] = yw[i];
      }
      __syncwarp();
      const float4* csr = cs + r * half;
      for (int e = lane; e < R; e += 32) {
        const bool lo = e < half;
        const int j = lo ? e : e - half;
        const float4 cv = csr[j];
        rt[e] = rot_bf16(bf16_to_f(nr[e]), bf16_to_f(nr[lo ? e + half : j]), ff{cv.x, cv.y},
                         lo ? ff{cv.z, cv.w} : ff{-cv.z, -cv.w});
      }
      __syncwarp();
      if (lane * E < R) {                               // this lane holds rotated dims
#pragma unroll
        for (int i = 0; i < E; i += 2) {
          const int e = lane * E + i;                   // R is even: e and e + 1 on the same side
          if (e < R) yw[i / 2] = (uint32_t)rt[e] | ((uint32_t)rt[e + 1] << 16);
        }
#pragma unroll
        for (int i = 0; i < E; i += 2) {
          y[i] = uint16_t(yw[i / 2] & 0xFFFFu);
          y[i + 1] = uint16_t(yw[i / 2] >> 16);
        }
      }
      __syncwarp();                                     // both rows read before the next item writes them
    }
    if (a.q_prepped) {                                  // (only 2-byte alignment is asked of it)
      if ((reinterpret_cast<uintptr_t>(a.q_prepped) & 3u) == 0) {
        uint32_t* d = reinterpret_cast<uint32_t*>(a.q_prepped + base);
#pragma unroll
        for (int i = 0; i < E / 2; ++i) d[i] = yw[i];
      } else {
#pragma unroll
        for (int i = 0; i < E; ++i) a.q_prepped[base + i] = y[i];
      }
    }
    if (a.ws.qhat) {
      uint32_t* d = reinterpret_cast<uint32_t*>(a.ws.qhat + base);
#pragma unroll
      for (int i = 0; i < E / 2; ++i) d[i] = yw[i];
    }
    if (a.ws.q16) {
      uint32_t* d = reinterpret_cast<uint32_t*>(a.ws.q16 + base);
      float gs = 0.f;
#pragma unroll
      for (int i = 0; i < E; i += 2) {
        const __half2 h = __floats2half2_rn(bf16_to_f(y[i]), bf16_to_f(y[i + 1]));
        const float2 hf = __half22float2(h);
        gs += hf.x + hf.y;                              // the f16 values the MMA multiplies
        d[i / 2] = *reinterpret_cast<const uint32_t*>(&h);
      }
#pragma unroll
      for (int m = 1; m < LPG; m <<= 1) gs += __shfl_xor_sync(0xffffffffu, gs, m);
      if (a.ws.qsum && lane % LPG == 0) a.ws.qsum[((size_t)row * Hq + hq) * NG + lane / LPG] = gs;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kQrWarps * 32)
qprep_rows_kernel(const DecodeArgs a, const RopeFreqs freqs, const int rb) {
  qprep_rows_block<D>(a, freqs, rb, blockIdx.x);
}

// The q prep of a call together with the K/V prep of its rows (the append of
// attn_prefill_append, the donor's K/V of attn_train_donor_forward) in one
// grid: blocks below nq prep q, the others each take one row's block of ipb
// append items (ablk blocks per row).  The halves share nothing.
template <int D>
__global__ void __launch_bounds__(kQrWarps * 32)
qprep_rows_append_kernel(const DecodeArgs a, const AppendArgs ap, const RopeFreqs freqs, const int rb,
                         const int nq, const int ipb, const int ablk) {
  if ((int)blockIdx.x < nq) {
    qprep_rows_block<D>(a, freqs, rb, blockIdx.x);
  } else {
    const int b = blockIdx.x - nq;
    append_block<D>(ap, freqs, ipb, b / ablk, b % ablk);
  }
}

// rows per block: enough (row, head) items for the 8 warps, angle tables of
// at most 16 KB
inline int qprep_rows_rb(const LayerArgs& L) {
  int rb = std::max(1, std::min(16, 32 / L.n_q));
  const int half = L.rope_dims / 2;
  if (half > 0) rb = std::max(1, std::min(rb, 1024 / half));
  return rb;
}

// dynamic shared memory of a q-prep block of rb rows: the angle table, the
// frequencies, two rows per warp
inline size_t qprep_rows_smem(const LayerArgs& L, int rb) {
  const int half = L.rope_dims / 2;
  return (size_t)rb * half * 16 + 16 * ((3 * half + 3) / 4) + (size_t)kQrWarps * 2 * L.D * 2;
}

// ap: NULL, or the append whose blocks share the q prep's grid (its rows
// need not be the q rows: the training read's K/V rows are those of the pass)
template <int D>
cudaError_t launch_qprep_rows(const DecodeArgs& a, const RopeFreqs& f, cudaStream_t st,
                              const AppendArgs* ap = nullptr) {
  const int rb = qprep_rows_rb(a.L);
  const size_t smem = qprep_rows_smem(a.L, rb);
  const int nq = (a.n_rows + rb - 1) / rb;
  if (!ap || ap->n_rows == 0) return launch_pdl(qprep_rows_kernel<D>, dim3(nq), dim3(kQrWarps * 32), smem, st, a, f, rb);
  const int items = 2 * ap->L.n_kv;
  const int ipb = std::min(items, kQrWarps * 32 / App<D>::TH);
  const int ablk = (items + ipb - 1) / ipb;
  const long long blocks = (long long)nq + (long long)ap->n_rows * ablk;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  return launch_pdl(qprep_rows_append_kernel<D>, dim3((unsigned)blocks), dim3(kQrWarps * 32), smem, st, a, *ap, f,
                    rb, nq, ipb, ablk);
}

}  // namespace
}  // namespace kvq
