// attn_decode / attn_prefill_chunk: query rows attend their quantized cache
// (model.ts attentionTraining: qNorm, RoPE at the cache offset,
// read.attend(q, 1.0); "Parity notes": SDPA scale 1.0, K = V full layers,
// GQA over n_kv heads).
//
// Two launches on the caller's stream:
//   1. decode_kernel (rows, n_kv, splits): split-K ("flash decoding") over the
//      keys each query row sees.  One CTA = 16 warps (8 for head_dim 64).
//      Prologue: the first tiles' TMA copies are issued, then the CTA preps
//      its G q heads itself (RMSNorm, RoPE in float-float; correctly rounded
//      bf16) while they land, and every warp builds the f16 A fragments of
//      its own 64-dim group.  64-key tiles (packed codes row by row into
//      padded shared rows, scales and biases) stream through a ring of
//      stages filled by TMA bulk copies and tracked by mbarriers; the warps
//      refill a stage as soon as the first barrier of a tile shows that all
//      of them are done with it.  Per tile:
//        QK, split by head_dim group: warp (g, slice) multiplies the group-g
//          codes of its keys (exact integers in f16) by q on the tensor cores
//          (mma.sync m16n8k16, fp32 accumulate) and writes scale * (q . c) to
//          a per-group partial-score buffer;
//        softmax, one warp per q head: sums the group partials, adds the
//          bias term sum_g bias * sum(q_g), masks the window, and keeps the
//          online max / sum; writes P (f16);
//        PV, split by head_dim slice: O += (P * scale) c + P bias, with the
//          per-key scale folded into the f16 A operand (times a power of two
//          that keeps it clear of f16 subnormals) and the bias as one extra
//          MMA column.
//      Each split writes its (m, l, o) partial.
//   2. combine_kernel (rows, n_q): merges the split partials.
#include "kvq_common.cuh"
#include "kvq_internal.h"

#include <algorithm>

namespace kvq {

namespace {

template <int D>
struct Dec {
  static constexpr int NG = D / 64;                  // 64-dim groups
  static constexpr int NW = NG >= 2 ? 16 : 8;        // warps per CTA
  static constexpr int THREADS = NW * 32;
  static constexpr int WPG = NW / NG;                // warps per group
  static constexpr int KPW = 64 / WPG;               // keys per warp in QK
  static constexpr int NTQ = KPW / 8;                // QK n-tiles per warp
  static constexpr int DPW = 64 / WPG;               // dims per warp in PV
  static constexpr int NTP = DPW / 8;                // PV n-tiles per warp
};

constexpr int kMaxStages = 8;
constexpr int kSPS = 68;      // row stride (floats) of the partial-score buffer

__host__ __device__ constexpr int row_bytes(int D, int bits) { return D * bits / 8; }
__host__ __device__ constexpr int row_stride(int D, int bits) { return D * bits / 8 + 16; }
__host__ __device__ constexpr int sb_bytes(int D) { return 64 * (D / 64) * 2; }
__host__ __device__ constexpr int stage_bytes(int D, int bits) { return 2 * 64 * row_stride(D, bits) + 4 * sb_bytes(D); }
__host__ __device__ constexpr int align128(int x) { return (x + 127) & ~127; }
__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }
// control block: mbarriers (128 B), alpha[16], qsum[16][8] (floats), V scale/bias f16 pairs [2][2][NG][32]
__host__ __device__ constexpr int off_alpha() { return 128; }
__host__ __device__ constexpr int off_qsum() { return 128 + 64; }
__host__ __device__ constexpr int off_vsb() { return 128 + 64 + 512; }
__host__ __device__ constexpr int ctrl_bytes(int D) { return align128(off_vsb() + 2 * 2 * (D / 64) * 32 * 4); }
// scratch: q prep in the prologue, partial scores + P in the tile loop
__host__ __device__ constexpr int scratch_loop(int D) { return (D / 64) * 16 * kSPS * 4 + 16 * 64 * 2; }
__host__ __device__ constexpr int scratch_prep(int D) { return 2 * 16 * D * 2 + (D / 2) * 16; }
__host__ __device__ constexpr int scratch_bytes(int D) { return align128(cmax(scratch_loop(D), scratch_prep(D))); }
__host__ __device__ constexpr int stage0_off(int D) { return ctrl_bytes(D) + scratch_bytes(D); }

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

__device__ __forceinline__ uint32_t bf16_pair_to_h2(uint16_t lo, uint16_t hi) {
  return pack_h2(bf16_to_f(lo), bf16_to_f(hi));
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

struct TileRange {
  int t_begin, n_my, lo, hi;
};

// log2 of the power of two the PV A operand (P * scale) is multiplied by.
template <int BITS> struct PvPrescale { static constexpr int log2 = BITS == 4 ? 2 : 6; };

// q prep of the CTA's G heads into shared memory: bf16 q_hat [16][D] (rows >= G
// zero) and per-group sums of its f16 values [16][8].  Writes q_prepped when
// asked.  Ends with a block barrier.
template <int D>
__device__ __forceinline__ void prep_q_block(const DecodeArgs& a, const RopeFreqs& freqs, int row, int kvh, int p,
                                             uint8_t* scratch, float* qsum_sm, bool write_prepped) {
  using C = Dec<D>;
  constexpr int E = D / 32, LPG = 64 / E;
  uint16_t* qn = reinterpret_cast<uint16_t*>(scratch);            // [16][D] normed
  uint16_t* qh = qn + 16 * D;                                     // [16][D] q_hat
  float4* cs = reinterpret_cast<float4*>(qh + 16 * D);            // [D/2]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.L.G, R = a.L.rope_dims, half = R >> 1;
  const int pc = min(max(p, 0), (1 << 24) - 1);
  for (int j = threadIdx.x; j < half; j += C::THREADS) {
    ff cc, sn;
    rope_cos_sin(pc, freqs.f[j][0], freqs.f[j][1], freqs.f[j][2], cc, sn);
    cs[j] = make_float4(cc.hi, cc.lo, sn.hi, sn.lo);
  }
  for (int h = warp; h < 16; h += C::NW) {
    uint16_t y[E];
    if (h < G) {
      const uint16_t* src = a.q_raw + ((size_t)row * a.L.n_q + kvh * G + h) * D + lane * E;
      float x[E];
      if constexpr (E >= 8) {
#pragma unroll
        for (int v = 0; v < E / 8; ++v) {
          const uint4 u = *reinterpret_cast<const uint4*>(src + 8 * v);
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) { x[8 * v + 2 * i] = bf16lo_to_f(w[i]); x[8 * v + 2 * i + 1] = bf16hi_to_f(w[i]); }
        }
      } else {
#pragma unroll
        for (int i = 0; i < E; ++i) x[i] = bf16_to_f(src[i]);
      }
      ff ss = {0.f, 0.f};
#pragma unroll
      for (int i = 0; i < E; ++i) ff_acc_sq(ss, x[i]);
      ss = ff_warp_sum(ss);
      const ff inv = rms_inv(ss, D, a.L.eps);
#pragma unroll
      for (int i = 0; i < E; ++i) y[i] = norm_scale_bf16(x[i], bf16_to_f(a.q_w[lane * E + i]), inv);
    } else {
#pragma unroll
      for (int i = 0; i < E; ++i) y[i] = 0;
    }
#pragma unroll
    for (int i = 0; i < E; ++i) qn[h * D + lane * E + i] = y[i];
  }
  __syncthreads();                       // cs[] and qn[] complete
  for (int h = warp; h < 16; h += C::NW) {
    uint16_t y[E];
    float gs = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const int e = lane * E + i;
      y[i] = qn[h * D + e];
      if (h < G && e < R) {
        const int j = e < half ? e : e - half;
        const float4 t = cs[j];
        const ff cc = {t.x, t.y};
        y[i] = e < half ? rot_bf16(bf16_to_f(qn[h * D + e]), bf16_to_f(qn[h * D + e + half]), cc, ff{t.z, t.w})
                        : rot_bf16(bf16_to_f(qn[h * D + e]), bf16_to_f(qn[h * D + j]), cc, ff{-t.z, -t.w});
      }
      gs += __half2float(__float2half_rn(bf16_to_f(y[i])));   // the f16 value the MMA multiplies
    }
#pragma unroll
    for (int i = 0; i < E; ++i) qh[h * D + lane * E + i] = y[i];
#pragma unroll
    for (int m = 1; m < LPG; m <<= 1) gs += __shfl_xor_sync(0xffffffffu, gs, m);
    if (lane % LPG == 0) qsum_sm[h * 8 + lane / LPG] = gs;
    if (write_prepped && h < G) {
      uint16_t* dst = a.q_prepped + ((size_t)row * a.L.n_q + kvh * G + h) * D + lane * E;
#pragma unroll
      for (int i = 0; i < E; ++i) dst[i] = y[i];
    }
  }
  __syncthreads();
}

template <int D, int BITS>
__device__ __forceinline__ void decode_body(const DecodeArgs& a, const RopeFreqs& freqs, const kvq_seq_cache& c,
                                            uint8_t* smem, const int nst, const TileRange tr, const int row,
                                            const int kvh, const int split, const int p) {
  using C = Dec<D>;
  constexpr int NG = C::NG, WPG = C::WPG, KPW = C::KPW, NTQ = C::NTQ, DPW = C::DPW, NTP = C::NTP;
  constexpr int RB = row_bytes(D, BITS), RS = row_stride(D, BITS), SB = sb_bytes(D);
  constexpr int STB = stage_bytes(D, BITS);
  constexpr float L2E = 1.4426950408889634f;
  constexpr float PRESCALE = float(1 << PvPrescale<BITS>::log2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t4 = lane & 3, rq = lane >> 2;
  const int G = a.L.G;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  float* alpha_sm = reinterpret_cast<float*>(smem + off_alpha());     // [16]
  float* qsum_sm = reinterpret_cast<float*>(smem + off_qsum());       // [16][8]
  uint32_t* vsb = reinterpret_cast<uint32_t*>(smem + off_vsb());      // [2][2][NG][32]
  uint8_t* scratch = smem + ctrl_bytes(D);
  float* spart = reinterpret_cast<float*>(scratch);                   // [NG][16][kSPS]
  uint8_t* Pb = scratch + NG * 16 * kSPS * 4;                         // [16][64] f16, swizzled
  uint8_t* stages = smem + stage0_off(D);
  const int cap = c.capacity;
  const size_t head_row0 = (size_t)kvh * cap;

  // Issue tile `it` into its stage: 128 code rows and 4 scale/bias blocks,
  // one bulk copy per thread.
  auto issue = [&](int it) {
    const int st = it % nst;
    uint8_t* sb = stages + st * STB;
    const size_t r0 = head_row0 + ((tr.t_begin + it) * kTileKeys) % cap;
    if (threadIdx.x == 0) mbar_arrive_expect_tx(&full[st], 2 * 64 * RB + 4 * SB);
    fence_proxy_async();        // order this CTA's earlier generic reads of the stage before the copies
    for (int j = threadIdx.x; j < 2 * 64 + 4; j += C::THREADS) {
      if (j < 64) {
        bulk_g2s(sb + j * RS, reinterpret_cast<const uint8_t*>(c.k_codes) + (r0 + j) * RB, RB, &full[st]);
      } else if (j < 128) {
        const int r = j - 64;
        bulk_g2s(sb + j * RS, reinterpret_cast<const uint8_t*>(c.v_codes) + (r0 + r) * RB, RB, &full[st]);
      } else {
        const int q = j - 128;
        const uint16_t* src = q == 0 ? c.k_scales : q == 1 ? c.k_biases : q == 2 ? c.v_scales : c.v_biases;
        bulk_g2s(sb + 2 * 64 * RS + q * SB, src + r0 * NG, SB, &full[st]);
      }
    }
  };
  // prologue: fill every stage (the cache was written before this launch)
  for (int it = 0; it < min(nst, tr.n_my); ++it) issue(it);
  int issued = min(nst, tr.n_my);

  // q prep while the first tiles land
  prep_q_block<D>(a, freqs, row, kvh, p, scratch, qsum_sm, split == 0 && a.q_prepped != nullptr);
  const int g_qk = warp / WPG, slice = warp % WPG;
  uint32_t qa[4][4];            // A fragments of group g_qk: 16 rows (q heads) x 64 dims
  {
    const uint16_t* qh = reinterpret_cast<const uint16_t*>(scratch) + 16 * D;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      int d[4];
      qk_dims(BITS, ks, d);
      const int base = g_qk * 64 + 16 * t4;
      qa[ks][0] = bf16_pair_to_h2(qh[rq * D + base + d[0]], qh[rq * D + base + d[1]]);
      qa[ks][1] = bf16_pair_to_h2(qh[(rq + 8) * D + base + d[0]], qh[(rq + 8) * D + base + d[1]]);
      qa[ks][2] = bf16_pair_to_h2(qh[rq * D + base + d[2]], qh[rq * D + base + d[3]]);
      qa[ks][3] = bf16_pair_to_h2(qh[(rq + 8) * D + base + d[2]], qh[(rq + 8) * D + base + d[3]]);
    }
  }
  // softmax warp `warp` owns q head `warp` (when < G): its per-group q sums
  float qs[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) qs[g] = qsum_sm[(warp & 15) * 8 + g];
  if (threadIdx.x < 16) alpha_sm[threadIdx.x] = 1.f;
  __syncthreads();              // the scratch region becomes the partial-score buffer

  float oacc[NTP][4];           // PV accumulator: 16 rows x this warp's DPW dims (permuted)
  float cb[4];                  // sum_j P_j * bias_j of this warp's group (column 0 is used)
#pragma unroll
  for (int i = 0; i < NTP; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  cb[0] = cb[1] = cb[2] = cb[3] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;   // softmax state of head `warp`
  bool dead = false;
  const int g_pv = warp / WPG, dslice = warp % WPG;

  for (int it = 0; it < tr.n_my; ++it) {
    const int st = it % nst, buf = it & 1;
    if (!dead && !mbar_wait(&full[st], (it / nst) & 1)) {
      dead = true;
      flag_error(a.ws.status, KVQ_DEV_TIMEOUT);
    }
    const uint8_t* Ks = stages + st * STB;
    const uint8_t* Vs = Ks + 64 * RS;
    const uint16_t* sks = reinterpret_cast<const uint16_t*>(Ks + 2 * 64 * RS);
    const uint16_t* skb = sks + 64 * NG;
    const uint16_t* svs = skb + 64 * NG;
    const uint16_t* svb = svs + 64 * NG;
    const int tpos0 = (tr.t_begin + it) * kTileKeys;

    // ---- V scale/bias of this tile as f16 pairs (scale pre-multiplied by
    // PRESCALE), zero for keys outside the window ----
    for (int idx = threadIdx.x; idx < NG * 64; idx += C::THREADS) {
      const int which = idx / (NG * 32);                    // 0: scale, 1: bias
      const int rem = idx % (NG * 32);
      const int g = rem % NG, pr = rem / NG;                // consecutive threads: consecutive groups
      const int k0 = 2 * pr;
      const bool v0 = tpos0 + k0 >= tr.lo && tpos0 + k0 <= tr.hi;
      const bool v1 = tpos0 + k0 + 1 >= tr.lo && tpos0 + k0 + 1 <= tr.hi;
      const uint16_t* srcp = which == 0 ? svs : svb;
      const float mul = which == 0 ? PRESCALE : 1.f;
      const float x0 = v0 ? bf16_to_f(srcp[k0 * NG + g]) * mul : 0.f;
      const float x1 = v1 ? bf16_to_f(srcp[(k0 + 1) * NG + g]) * mul : 0.f;
      vsb[((buf * 2 + which) * NG + g) * 32 + pr] = pack_h2(x0, x1);
    }

    // ---- QK partial of group g_qk for this warp's keys ----
#pragma unroll
    for (int nt = 0; nt < NTQ; ++nt) {
      const int kb8 = slice * KPW + nt * 8;
      const int kB = kb8 + rq, kC = kb8 + 2 * t4;
      float acc[4];
      if constexpr (BITS == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(Ks + kB * RS + g_qk * 32 + t4 * 8);
        mma_f16_zc(acc, qa[0], nib_lo(w.x), nib_hi(w.x));
        mma_f16(acc, qa[1], nib_lo(w.x >> 8), nib_hi(w.x >> 8));
        mma_f16(acc, qa[2], nib_lo(w.y), nib_hi(w.y));
        mma_f16(acc, qa[3], nib_lo(w.y >> 8), nib_hi(w.y >> 8));
      } else {
        const uint4 w = *reinterpret_cast<const uint4*>(Ks + kB * RS + g_qk * 64 + t4 * 16);
        mma_f16_zc(acc, qa[0], byte_lo(w.x), byte_lo(w.x >> 8));
        mma_f16(acc, qa[1], byte_lo(w.y), byte_lo(w.y >> 8));
        mma_f16(acc, qa[2], byte_lo(w.z), byte_lo(w.z >> 8));
        mma_f16(acc, qa[3], byte_lo(w.w), byte_lo(w.w >> 8));
      }
      const float s0 = bf16_to_f(sks[kC * NG + g_qk]), s1 = bf16_to_f(sks[(kC + 1) * NG + g_qk]);
      float* sp = spart + (g_qk * 16 + rq) * kSPS + kC;
      *reinterpret_cast<float2*>(sp) = make_float2(s0 * acc[0], s1 * acc[1]);
      *reinterpret_cast<float2*>(sp + 8 * kSPS) = make_float2(s0 * acc[2], s1 * acc[3]);
    }
    named_bar(1, C::THREADS);
    // every warp has finished tile it-1: its stage takes tile it-1+nst
    if (it >= 1 && issued < tr.n_my) {
      issue(issued);
      ++issued;
    }

    // ---- softmax: warp h < G owns q head h; lane l keys 2l, 2l+1 ----
    if (warp < G) {
      const int h = warp, j = 2 * lane;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const float2 v = *reinterpret_cast<const float2*>(spart + (g * 16 + h) * kSPS + j);
        s0 += v.x;
        s1 += v.y;
      }
      {
        uint32_t b0[(NG + 1) / 2], b1[(NG + 1) / 2];
        if constexpr (NG == 8) {
          const uint4 u0 = *reinterpret_cast<const uint4*>(skb + j * NG);
          const uint4 u1 = *reinterpret_cast<const uint4*>(skb + (j + 1) * NG);
          b0[0] = u0.x; b0[1] = u0.y; b0[2] = u0.z; b0[3] = u0.w;
          b1[0] = u1.x; b1[1] = u1.y; b1[2] = u1.z; b1[3] = u1.w;
        } else if constexpr (NG == 4) {
          const uint2 u0 = *reinterpret_cast<const uint2*>(skb + j * NG);
          const uint2 u1 = *reinterpret_cast<const uint2*>(skb + (j + 1) * NG);
          b0[0] = u0.x; b0[1] = u0.y; b1[0] = u1.x; b1[1] = u1.y;
        } else if constexpr (NG == 2) {
          b0[0] = *reinterpret_cast<const uint32_t*>(skb + j * NG);
          b1[0] = *reinterpret_cast<const uint32_t*>(skb + (j + 1) * NG);
        } else {
          b0[0] = skb[j];
          b1[0] = skb[j + 1];
        }
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const float bb0 = (g & 1) ? bf16hi_to_f(b0[g >> 1]) : bf16lo_to_f(b0[g >> 1]);
          const float bb1 = (g & 1) ? bf16hi_to_f(b1[g >> 1]) : bf16lo_to_f(b1[g >> 1]);
          s0 = fmaf(bb0, qs[g], s0);
          s1 = fmaf(bb1, qs[g], s1);
        }
      }
      const int kp = tpos0 + j;
      if (!(kp >= tr.lo && kp <= tr.hi)) s0 = -INFINITY;
      if (!(kp + 1 >= tr.lo && kp + 1 <= tr.hi)) s1 = -INFINITY;
      float mt = fmaxf(s0, s1);
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, m));
      const float m_new = fmaxf(m_run, mt);
      const float alpha = m_new == -INFINITY ? 1.f : exp2f((m_run - m_new) * L2E);
      float p0 = 0.f, p1 = 0.f;
      if (m_new != -INFINITY) {
        p0 = exp2f((s0 - m_new) * L2E);
        p1 = exp2f((s1 - m_new) * L2E);
      }
      const __half2 ph = __floats2half2_rn(p0, p1);
      const float2 pf = __half22float2(ph);
      float ls = pf.x + pf.y;
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, m);
      l_run = l_run * alpha + ls;
      m_run = m_new;
      const int chunk = (j >> 3) ^ (h & 7);
      *reinterpret_cast<__half2*>(Pb + h * 128 + chunk * 16 + (j & 7) * 2) = ph;
      if (lane == 0) alpha_sm[h] = alpha;
    }
    named_bar(1, C::THREADS);

    // ---- PV for this warp's DPW dims of group g_pv ----
    {
      const float a0 = alpha_sm[rq], a1 = alpha_sm[rq + 8];
      if (!__all_sync(0xffffffffu, a0 == 1.f && a1 == 1.f)) {
#pragma unroll
        for (int nt = 0; nt < NTP; ++nt) {
          oacc[nt][0] *= a0; oacc[nt][1] *= a0;
          oacc[nt][2] *= a1; oacc[nt][3] *= a1;
        }
        cb[0] *= a0; cb[1] *= a0; cb[2] *= a1; cb[3] *= a1;
      }
    }
    const uint32_t* vs16 = vsb + ((buf * 2 + 0) * NG + g_pv) * 32;
    const uint32_t* vb16 = vsb + ((buf * 2 + 1) * NG + g_pv) * 32;
    // byte offset of this thread's codes in a V row: dims g*64 + dslice*DPW + rq*NTP ...
    constexpr int CBITS = NTP * BITS;            // code bits per key held by a thread
    const int dim0 = g_pv * 64 + dslice * DPW + rq * NTP;
    const int boff = dim0 * BITS / 8;
    const int nib_shift = (CBITS == 4) ? ((dim0 & 1) * 4) : 0;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      {
        const int mtx = lane >> 3, i = lane & 7;
        const int prow = (mtx & 1) * 8 + i;
        const int chunk = (kk * 2 + (mtx >> 1)) ^ (prow & 7);
        ldmatrix_x4(pa, Pb + prow * 128 + chunk * 16);
      }
      const int ka = kk * 16 + 2 * t4;           // keys ka, ka+1, ka+8, ka+9
      const uint32_t sAB = vs16[kk * 8 + t4], sCD = vs16[kk * 8 + 4 + t4];
      // bias column: only B column 0 (lanes 0..3) is non-zero
      const uint32_t bAB = rq == 0 ? vb16[kk * 8 + t4] : 0u, bCD = rq == 0 ? vb16[kk * 8 + 4 + t4] : 0u;
      mma_f16(cb, pa, bAB, bCD);
      const uint32_t ps[4] = {h2_mul(pa[0], sAB), h2_mul(pa[1], sAB), h2_mul(pa[2], sCD), h2_mul(pa[3], sCD)};
      uint32_t wa, wb, wc, wd;
      const uint8_t* vp = Vs + boff;
      if constexpr (CBITS == 32) {
        wa = *reinterpret_cast<const uint32_t*>(vp + ka * RS);
        wb = *reinterpret_cast<const uint32_t*>(vp + (ka + 1) * RS);
        wc = *reinterpret_cast<const uint32_t*>(vp + (ka + 8) * RS);
        wd = *reinterpret_cast<const uint32_t*>(vp + (ka + 9) * RS);
      } else if constexpr (CBITS == 16) {
        wa = *reinterpret_cast<const uint16_t*>(vp + ka * RS);
        wb = *reinterpret_cast<const uint16_t*>(vp + (ka + 1) * RS);
        wc = *reinterpret_cast<const uint16_t*>(vp + (ka + 8) * RS);
        wd = *reinterpret_cast<const uint16_t*>(vp + (ka + 9) * RS);
      } else {
        wa = vp[ka * RS];
        wb = vp[(ka + 1) * RS];
        wc = vp[(ka + 8) * RS];
        wd = vp[(ka + 9) * RS];
      }
      // pair each code with the same code of the next key: low half <- key a/c, high half <- key b/d
      const uint32_t xab = prmt(wa, wb, 0x5410) >> nib_shift, xcd = prmt(wc, wd, 0x5410) >> nib_shift;
      if constexpr (BITS == 4) {
        // n-tile nt <- nibble nt of the thread's codes
        mma_f16(oacc[0], ps, nib_lo(xab), nib_lo(xcd));
        if constexpr (NTP >= 2) mma_f16(oacc[1], ps, nib_hi(xab), nib_hi(xcd));
        if constexpr (NTP >= 4) {
          mma_f16(oacc[2], ps, nib_lo(xab >> 8), nib_lo(xcd >> 8));
          mma_f16(oacc[3], ps, nib_hi(xab >> 8), nib_hi(xcd >> 8));
        }
      } else {
        // n-tile nt <- byte nt of the thread's codes
        mma_f16(oacc[0], ps, byte_lo(xab), byte_lo(xcd));
        if constexpr (NTP >= 2) mma_f16(oacc[1], ps, byte_lo(xab >> 8), byte_lo(xcd >> 8));
        if constexpr (NTP >= 4) {
          const uint32_t yab = prmt(wa, wb, 0x7632), ycd = prmt(wc, wd, 0x7632);
          mma_f16(oacc[2], ps, byte_lo(yab), byte_lo(ycd));
          mma_f16(oacc[3], ps, byte_lo(yab >> 8), byte_lo(ycd >> 8));
        }
      }
    }
  }
  pdl_launch();
  // a timed-out wait may leave copies in flight: they must land before exit
  if (dead && threadIdx.x == 0)
    for (int it = max(0, issued - nst); it < issued; ++it) mbar_wait(&full[it % nst], (it / nst) & 1);

  // ---- write this split's partial (m, l, o) ----
  const size_t pidx = ((size_t)row * a.L.n_kv + kvh) * a.splits + split;
  float* po = a.ws.part_o + pidx * 16 * D;
  float* ml = a.ws.part_ml + pidx * 32;
  if (warp < G && lane == 0) { ml[warp] = m_run; ml[16 + warp] = l_run; }
  // bias column 0 lives in lanes with t4 == 0 (c0: row rq, c2: row rq + 8)
  const float bias_r = __shfl_sync(0xffffffffu, cb[0], lane & ~3);
  const float bias_r8 = __shfl_sync(0xffffffffu, cb[2], lane & ~3);
  constexpr float UNSCALE = 1.f / PRESCALE;
#pragma unroll
  for (int nt = 0; nt < NTP; ++nt) {
    // column n of n-tile nt is dim g*64 + dslice*DPW + n*NTP + nt
    const int d0 = g_pv * 64 + dslice * DPW + (2 * t4) * NTP + nt, d1 = d0 + NTP;
    if (rq < G) {
      po[rq * D + d0] = fmaf(oacc[nt][0], UNSCALE, bias_r);
      po[rq * D + d1] = fmaf(oacc[nt][1], UNSCALE, bias_r);
    }
    if (rq + 8 < G) {
      po[(rq + 8) * D + d0] = fmaf(oacc[nt][2], UNSCALE, bias_r8);
      po[(rq + 8) * D + d1] = fmaf(oacc[nt][3], UNSCALE, bias_r8);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(Dec<D>::THREADS, 1)
decode_kernel(const DecodeArgs a, const RopeFreqs freqs, const int smem_total) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int row = blockIdx.x, kvh = blockIdx.y, split = blockIdx.z;
  const RowInfo ri = row_info(a, row);
  const kvq_seq_cache c = a.seqs[ri.s];
  const int p = ri.p;
  const int W = a.L.window;
  const int lo = W > 0 ? max(0, p - W + 1) : 0, hi = p;
  // every key from lo up to the newest cached position must own its slot
  const bool ok = seq_ok(c) && p >= 0 && ri.newest < (1 << 24) && p <= ri.newest &&
                  (ri.newest - lo + 1) <= c.capacity;
  const int t_lo = lo / kTileKeys, t_hi = hi / kTileKeys;
  const int ntiles = t_hi - t_lo + 1;
  const int chunk = (ntiles + a.splits - 1) / a.splits;
  const int t_begin = t_lo + split * chunk;
  const int n_my = ok ? max(0, min(chunk, t_hi + 1 - t_begin)) : 0;
  if (n_my == 0) {
    // nothing to read: an empty partial (m = -inf), or NaN for a bad sequence
    if (!ok && split == 0 && kvh == 0 && threadIdx.x == 0) flag_error(a.ws.status, KVQ_DEV_BADSEQ);
    const size_t pidx = ((size_t)row * a.L.n_kv + kvh) * a.splits + split;
    if (threadIdx.x < 16) {
      a.ws.part_ml[pidx * 32 + threadIdx.x] = ok ? -INFINITY : __int_as_float(0x7fc00000);
      a.ws.part_ml[pidx * 32 + 16 + threadIdx.x] = 0.f;
    }
    pdl_launch();
    // q_prepped covers every row, also one whose attention is NaN
    if (split == 0 && a.q_prepped != nullptr)
      prep_q_block<D>(a, freqs, row, kvh, p, smem + ctrl_bytes(D),
                      reinterpret_cast<float*>(smem + off_qsum()), true);
    return;
  }
  const int bits = c.bits;
  const int nst = min(kMaxStages, (smem_total - stage0_off(D)) / stage_bytes(D, bits));
  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) mbar_init(reinterpret_cast<uint64_t*>(smem) + i, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const TileRange tr{t_begin, n_my, lo, hi};
  if (bits == 4) decode_body<D, 4>(a, freqs, c, smem, nst, tr, row, kvh, split, p);
  else decode_body<D, 8>(a, freqs, c, smem, nst, tr, row, kvh, split, p);
}

// ----------------------------------------------------------------------------
// 2. merge split partials: out = sum_i e^(m_i - M) o_i / sum_i e^(m_i - M) l_i
// ----------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128)
combine_kernel(const DecodeArgs a) {
  __shared__ float wsm[256];
  __shared__ float inv_l;
  pdl_wait();
  const int row = blockIdx.x, hq = blockIdx.y;
  const int G = a.L.G, kvh = hq / G, r = hq % G;
  const int S = a.splits;
  const size_t base = ((size_t)row * a.L.n_kv + kvh) * S;
  if (threadIdx.x < 32) {
    float M = -INFINITY;
    bool nan = false;
    for (int i = threadIdx.x; i < S; i += 32) {
      const float m = a.ws.part_ml[(base + i) * 32 + r];
      nan |= m != m;
      M = fmaxf(M, m);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    nan = __any_sync(0xffffffffu, nan);
    float L = 0.f;
    for (int i = threadIdx.x; i < S; i += 32) {
      const float m = a.ws.part_ml[(base + i) * 32 + r];
      const float w = (m == -INFINITY || m != m) ? 0.f : exp2f((m - M) * 1.4426950408889634f);
      wsm[i] = w;
      L += w * a.ws.part_ml[(base + i) * 32 + 16 + r];
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (threadIdx.x == 0) inv_l = nan ? __int_as_float(0x7fc00000) : 1.f / L;
  }
  __syncthreads();
  const float il = inv_l;
  const float* po = a.ws.part_o + (base * 16 + r) * D;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float acc = 0.f;
    int i = 0;
    for (; i + 4 <= S; i += 4) {
      const float o0 = po[(size_t)(i + 0) * 16 * D + d], o1 = po[(size_t)(i + 1) * 16 * D + d];
      const float o2 = po[(size_t)(i + 2) * 16 * D + d], o3 = po[(size_t)(i + 3) * 16 * D + d];
      acc = fmaf(wsm[i], o0, acc);
      acc = fmaf(wsm[i + 1], o1, acc);
      acc = fmaf(wsm[i + 2], o2, acc);
      acc = fmaf(wsm[i + 3], o3, acc);
    }
    for (; i < S; ++i) acc = fmaf(wsm[i], po[(size_t)i * 16 * D + d], acc);
    const float o = acc * il;
    const size_t oi = ((size_t)row * a.L.n_q + hq) * D + d;
    if (a.out_f32) reinterpret_cast<float*>(a.out)[oi] = o;
    else reinterpret_cast<uint16_t*>(a.out)[oi] = f_to_bf16_rn(o);
  }
}

template <int D>
int decode_smem_bytes() {
  return std::min(227 * 1024, stage0_off(D) + kMaxStages * stage_bytes(D, 8));
}

template <int D>
cudaError_t launch_decode_t(const DecodeArgs& a, const RopeFreqs& f, cudaStream_t st) {
  cudaError_t e;
  const int smem = decode_smem_bytes<D>();
  static bool attr_set[64] = {};
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  decode_kernel<D><<<dim3(a.n_rows, a.L.n_kv, a.splits), dim3(Dec<D>::THREADS), smem, st>>>(a, f, smem);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_rows, a.L.n_q);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel<D>, a);
}

}  // namespace

size_t decode_ws_bytes(int n_rows, int n_kv, int D, int splits) {
  const size_t B = (size_t)n_rows * n_kv;
  size_t off = 256;
  off += B * splits * 16 * (size_t)D * 4;      // part_o
  off += B * splits * 32 * 4;                  // part_ml
  return off;
}

DecodeWs decode_ws_carve(void* base, int n_rows, int n_kv, int D, int splits) {
  const size_t B = (size_t)n_rows * n_kv;
  uint8_t* p = static_cast<uint8_t*>(base);
  DecodeWs w;
  w.status = reinterpret_cast<uint32_t*>(p);
  size_t off = 256;
  w.part_o = reinterpret_cast<float*>(p + off);
  off += B * splits * 16 * (size_t)D * 4;
  w.part_ml = reinterpret_cast<float*>(p + off);
  return w;
}

int decode_pick_splits(const LayerArgs& L, int n_rows, int max_keys, int num_sms) {
  const long keys = L.window > 0 ? std::min<long>((long)max_keys, L.window) : (long)max_keys;
  const int tiles = int(keys / kTileKeys) + 2;
  const int per_sm = 1;          // one 16-warp CTA per SM
  const long base = (long)n_rows * L.n_kv;
  long want = ((long)num_sms * per_sm + base - 1) / std::max<long>(base, 1);
  want = std::min<long>(want, std::max(1, tiles / 2));
  return int(std::max<long>(1, std::min<long>(want, 256)));
}

cudaError_t launch_decode(const DecodeArgs& a, const RopeFreqs& f, int /*num_sms*/, cudaStream_t st) {
  if (a.n_rows == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(a.ws.status, 0, 4, st);
  if (e != cudaSuccess) return e;
  switch (a.L.D) {
    case 64: return launch_decode_t<64>(a, f, st);
    case 128: return launch_decode_t<128>(a, f, st);
    case 256: return launch_decode_t<256>(a, f, st);
    case 512: return launch_decode_t<512>(a, f, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
