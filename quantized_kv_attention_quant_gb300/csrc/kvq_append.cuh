// The append's per-block work (prep, quantize, pack, store of new K/V rows),
// shared by kv_quant_append's kernel and the fused q + K/V prep of
// attn_decode_append.  See kvq_append.cu for the operation.
#pragma once
#include <type_traits>

#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "kvq_qprep.cuh"

namespace kvq {
namespace {


template <int D>
struct App {
  static constexpr int TH = D / 4 >= 32 ? D / 4 : 32;                         // threads per item
  static constexpr int E = D / TH;                 // elements per thread
  static constexpr int HW = TH / 32;               // warps per item
  static constexpr int TPG = 64 / E;               // threads per quantization group
  static constexpr int IPB = 1024 / TH;            // most items per block
};

__device__ __forceinline__ int find_seq(const int32_t* off, int n_seqs, int row) {
  // one row per sequence (decode steps) needs one round trip: off[row] == row
  if (row < n_seqs && __ldg(off + row) == row && __ldg(off + row + 1) > row) return row;
  int lo = 0, hi = n_seqs - 1;          // largest s with off[s] <= row
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(off + mid) <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// rint(fl32(d / s)) for s > 0, bit-identical to the IEEE quotient rounded
// half to even, without an IEEE division per element.  q1 = d * rcp(s)
// (both correctly rounded) is within |d/s| * 2^-23 of d/s and fl32(d/s) within
// |d/s| * 2^-24; for |d/s| <= 256 the two differ by < 5e-5, so their rints
// agree unless q1 lies within 1e-4 of a half-integer, in which case the
// quotient is formed exactly.
__device__ __forceinline__ int quant_code(float d, float s, float rcp) {
  const float q1 = __fmul_rn(d, rcp);
  const float f = q1 - floorf(q1);
  if (fabsf(f - 0.5f) > 1e-4f) return __float2int_rn(q1);
  return __float2int_rn(__fdiv_rn(d, s));
}

// Quantize this thread's E prepped values (one slice of a 64-group), pack the
// codes little-endian and store them, the group's scale and its bias.  With
// shi non-null the dequantized values scale * code + bias (fp32, one
// rounding) also go to shi as f16 and, with slo non-null, their remainders
// v - f16(v) to slo as f16: the prompt read's scratch, as its dequantization
// writes it from the stored codes, scale and bias.
template <int D, int BITS>
__device__ __forceinline__ void quantize_store(const uint16_t (&y)[App<D>::E], const kvq_seq_cache& c,
                                               int kind, int head, int pos, int t, uint16_t* shi,
                                               uint16_t* slo) {
  constexpr int E = App<D>::E;
  constexpr int TPG = App<D>::TPG;
  constexpr int NG = D / 64;
  constexpr int TOP = (1 << BITS) - 1;
  float v[E];
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < E; ++i) { v[i] = bf16_to_f(y[i]); mn = fminf(mn, v[i]); mx = fmaxf(mx, v[i]); }
#pragma unroll
  for (int m = 1; m < TPG; m <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, m));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
  }
  // a zero minimum or maximum is taken as +0 (min/max of -0 and +0 is unordered)
  mn = __fadd_rn(mn, 0.f);
  mx = __fadd_rn(mx, 0.f);
  // scale = bf16((max - min) / (2^bits - 1)), two IEEE fp32 roundings
  const uint16_t sb = f_to_bf16_rn(__fdiv_rn(__fsub_rn(mx, mn), (float)TOP));
  const float sf = bf16_to_f(sb);
  const float rcp = sf != 0.f ? __frcp_rn(sf) : 0.f;
  uint32_t code[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    int q = 0;
    if (sf != 0.f) q = min(max(quant_code(__fsub_rn(v[i], mn), sf, rcp), 0), TOP);
    code[i] = uint32_t(q);
  }
  if (shi) {                              // mn is a bf16 value: the stored bias exactly
#pragma unroll
    for (int i = 0; i < E; i += 2) {
      const float v0 = __fmaf_rn(sf, (float)code[i], mn), v1 = __fmaf_rn(sf, (float)code[i + 1], mn);
      const __half2 h = __floats2half2_rn(v0, v1);
      reinterpret_cast<uint32_t*>(shi)[i / 2] = *reinterpret_cast<const uint32_t*>(&h);
      if (slo) {
        const float2 hf = __half22float2(h);
        const __half2 l = __floats2half2_rn(__fsub_rn(v0, hf.x), __fsub_rn(v1, hf.y));
        reinterpret_cast<uint32_t*>(slo)[i / 2] = *reinterpret_cast<const uint32_t*>(&l);
      }
    }
  }
  const int slot = pos % c.capacity;
  const size_t rowi = (size_t)head * c.capacity + slot;
  uint32_t* codes = kind == 0 ? c.k_codes : c.v_codes;
  constexpr int WPR = D * BITS / 32;       // words per row
  constexpr int LB = E * BITS;             // bits per thread
  if constexpr (LB >= 32) {
    constexpr int NW = LB / 32, PER = 32 / BITS;
    uint32_t* dst = codes + rowi * WPR + t * NW;
#pragma unroll
    for (int wi = 0; wi < NW; ++wi) {
      uint32_t w = 0;
#pragma unroll
      for (int i = 0; i < PER; ++i) w |= code[wi * PER + i] << (i * BITS);
      dst[wi] = w;
    }
  } else {
    constexpr int TPW = 32 / LB;           // threads sharing one word
    uint32_t part = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) part |= code[i] << (i * BITS);
    part <<= (t % TPW) * LB;
#pragma unroll
    for (int m = 1; m < TPW; m <<= 1) part |= __shfl_xor_sync(0xffffffffu, part, m);
    if (t % TPW == 0) codes[rowi * WPR + t / TPW] = part;
  }
  if (t % TPG == 0) {
    const int g = t / TPG;
    uint16_t* sc = kind == 0 ? c.k_scales : c.v_scales;
    uint16_t* bi = kind == 0 ? c.k_biases : c.v_biases;
    sc[rowi * NG + g] = sb;
    bi[rowi * NG + g] = f_to_bf16_rn(mn);            // mn is a bf16 value: exact
  }
}

// One block of the append: row `row`, items by*ipb .. by*ipb + ipb - 1 (item
// 2h is the K row of kv head h, 2h + 1 its V row).  Every thread of the block
// calls it; threads past the last item take part in the block barriers only.
template <int D>
__device__ __forceinline__ void append_block(const AppendArgs& a, const RopeFreqs& freqs, const int ipb,
                                             const int row, const int by) {
  using A = App<D>;
  constexpr int E = A::E, TH = A::TH;
  __shared__ uint16_t normed[A::IPB * D];
  __shared__ float4 cs[D / 2];            // (cos.hi, cos.lo, sin.hi, sin.lo) per pair
  __shared__ __align__(16) float freq[D / 2][3];   // rotary frequency triples
  __shared__ ff red[A::IPB][A::HW];
  extern __shared__ double rot_rows[];    // [ipb][D], rotated layers only
  const int tid = threadIdx.x, il = tid / TH, tt = tid % TH, lane = tid & 31;
  const int R = a.L.rope_dims, half = R >> 1;
  const int Hkv = a.L.n_kv;
  const int item = by * ipb + il;
  const bool active = il < ipb && item < 2 * Hkv;
  const int kind = item & 1;             // 0: K, 1: V
  const int head = item >> 1;

  // Launched as a programmatic dependent of the stream's previous kernel:
  // until that grid is complete only the library's own frequency table is
  // read; every caller buffer is touched after the wait.
  if (R > 0) stage_freqs(freqs.f, half, freq);
  pdl_wait();
  pdl_launch();

  // the raw row and the norm weight first: their latency overlaps the
  // sequence lookup and the angles
  float x[E], wk[E];
  if (active) {
    const uint16_t* src = (kind == 0 || a.L.k_eq_v) ? a.k_raw : a.v_raw;
    src += ((size_t)row * Hkv + head) * D + tt * E;
#pragma unroll
    for (int v = 0; v < E; v += 2) {
      const uint32_t u = __ldg(reinterpret_cast<const uint32_t*>(src + v));
      x[v] = bf16lo_to_f(u);
      x[v + 1] = bf16hi_to_f(u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) x[i] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < E; ++i) wk[i] = kind == 0 ? bf16_to_f(__ldg(a.k_w + tt * E + i)) : 1.f;

  // row_offsets == nullptr: one new row per sequence, row s of sequence s
  int s = row, t_in = 0, rows_s = 1;
  if (a.row_offsets) {
    s = find_seq(a.row_offsets, a.n_seqs, row);
    const int off0 = __ldg(a.row_offsets + s), off1 = __ldg(a.row_offsets + s + 1);
    t_in = row - off0;
    rows_s = off1 - off0;
  }
  // training read (no caches): block 0 of the layout starts at position 0,
  // every later block (a branch) continues the prefix
  const bool train = a.seqs == nullptr;
  const int pos = (train ? (s == 0 ? 0 : __ldg(a.row_offsets + 1)) : __ldg(a.start_pos + s)) + t_in;
  kvq_seq_cache c = {};
  if (!train) c = a.seqs[s];
  const bool ok = (train || ((c.bits == 4 || c.bits == 8) && c.capacity > 0 && (c.capacity % kTileKeys) == 0 &&
                             c.k_codes && c.v_codes && c.k_scales && c.k_biases && c.v_scales && c.v_biases &&
                             aligned16(c.k_codes) && aligned16(c.v_codes) && aligned16(c.k_scales) &&
                             aligned16(c.k_biases) && aligned16(c.v_scales) && aligned16(c.v_biases))) &&
                  pos >= 0 && pos < (1 << 24);
  if (!ok) return;                       // uniform over the block
  // a row whose slot a newer row of this call overwrites is prepped (for
  // kv_prepped) but not stored
  const bool store = !train && t_in >= rows_s - c.capacity;

  // ---- the row's rotation angles, once for all K heads ----
  if (R > 0) {
    __syncthreads();                     // the staged frequencies
    for (int j = tid; j < half; j += blockDim.x) {
      ff cc, sn;
      rope_cos_sin(pos, freq[j][0], freq[j][1], freq[j][2], cc, sn);
      cs[j] = make_float4(cc.hi, cc.lo, sn.hi, sn.lo);
    }
  }

  // ---- RMSNorm (weight on K only) ----
  ff ss = {0.f, 0.f};
#pragma unroll
  for (int i = 0; i < E; ++i) ff_acc_sq(ss, x[i]);
  ss = ff_warp_sum(ss);
  if constexpr (A::HW > 1) {
    if (lane == 0) red[il][tt >> 5] = ss;
    __syncthreads();
    ss = red[il][0];
#pragma unroll
    for (int w = 1; w < A::HW; ++w) ss = ff_add(ss, red[il][w]);
  }
  const ff inv = rms_inv(ss, D, a.L.eps);
  uint16_t y[E];
#pragma unroll
  for (int i = 0; i < E; ++i) y[i] = norm_scale_bf16(x[i], wk[i], inv);

  // ---- RoPE on K ----
  if (R > 0) {
    uint16_t* nr = normed + il * D;
#pragma unroll
    for (int i = 0; i < E; ++i) nr[tt * E + i] = y[i];
    __syncthreads();                     // angles and normed rows complete
    if (active && kind == 0) {
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const int e = tt * E + i;
        if (e < R) {
          // x_j cos - x_{j+h} sin below half, x_{j+h} cos + x_j sin above: one call
          const bool lo = e < half;
          const int j = lo ? e : e - half;
          const float4 cv = cs[j];
          y[i] = rot_bf16(bf16_to_f(nr[e]), bf16_to_f(nr[lo ? e + half : j]), ff{cv.x, cv.y},
                          lo ? ff{cv.z, cv.w} : ff{-cv.z, -cv.w});
        }
      }
    }
  }
  // ---- the deferred TurboQuant read's rotation: bf16((y * s) H) ----
  if (a.L.rot) rotate_row_bf16<D, E, TH>(y, a.L.rot, rot_rows + il * D, tt, active);
  if (!active) return;

  if (a.prepped) {
    uint16_t* dst = a.prepped + (((size_t)kind * a.n_rows + row) * Hkv + head) * D + tt * E;
#pragma unroll
    for (int i = 0; i < E; ++i) dst[i] = y[i];
  }

  if (train) {                           // the plain keys and values are the output
    uint16_t* dst = (kind == 0 ? a.out_k : a.out_v) + ((size_t)row * Hkv + head) * D + tt * E;
#pragma unroll
    for (int i = 0; i < E; ++i) dst[i] = y[i];
    return;
  }

  // ---- quantize the 64-element group, pack, store ----
  if (!store) return;
  // the prompt read's scratch row of this position (rows of a sequence the
  // read flags, and rows past the scratch slot, are not written)
  uint16_t* shi = nullptr;
  uint16_t* slo = nullptr;
  if (a.sk_hi) {
    const int start = pos - t_in, W = a.L.window;
    const int q = pos - (W > 0 ? max(0, start - W + 1) : 0);
    if (start >= 0 && start + rows_s - 1 < (1 << 24) && q < a.sks) {
      const size_t o = (((size_t)s * a.sks + q) * Hkv + head) * D + tt * E;
      if (kind == 0) {
        shi = a.sk_hi + o;
        slo = a.sk_lo + o;
      } else {
        shi = a.sv + o;
      }
    }
  }
  if (c.bits == 4) quantize_store<D, 4>(y, c, kind, head, pos, tt, shi, slo);
  else quantize_store<D, 8>(y, c, kind, head, pos, tt, shi, slo);
}

}  // namespace
}  // namespace kvq
