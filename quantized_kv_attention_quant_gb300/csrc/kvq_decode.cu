// attn_decode: one query token per sequence attends its quantized cache
// (model.ts attentionTraining, decode phase: qNorm, RoPE at the cache offset,
// read.attend(q, 1.0); "Parity notes": SDPA scale 1.0, GQA over n_kv heads).
//
// Three launches on the caller's stream:
//   1. qprep_kernel   (rows, blocks of q heads): q RMSNorm + RoPE, written as
//      ready-made mma.sync A fragments plus per-group sums.
//   2. decode_kernel  programmatic dependent launch: split-K ("flash
//      decoding") over the visible keys, in one of two schedules:
//        fixed chunks (rows of at most 48 tiles): grid (rows, n_kv, splits),
//          split z takes tiles [z*chunk, (z+1)*chunk) of its row;
//        stream-K (longer rows): grid of one wave of CTAs, each taking an
//          equal range of the tiles of all (row, kv head) units in a row and
//          walking it unit by unit (see decode_kernel).
//      64-key tiles (packed codes row by row into padded shared rows, scales
//      and biases) stream through a ring of stages filled by TMA bulk copies
//      and tracked by mbarriers.  There is no producer warp (a 9th warp would
//      share a register sub-partition with two consumers and cap them at 168
//      registers): once a tile's max-exchange barrier shows every warp is done
//      with the previous tile, the warps refill that stage themselves.
//      Warps 0..NW-1 compute
//        QK: warp w takes 64/NW keys, all G heads (M = 16 rows), full head_dim;
//            codes enter the tensor cores exactly as f16 integers, per 64-dim
//            group: S += scale * (q . codes) + bias * sum(q)
//        softmax: online, tile max exchanged through shared memory
//        PV: warp w owns head_dim group w; A = P * scale (f16), B = exact
//            codes, plus one MMA for sum(P * bias).
//      Each run of tiles writes its (m, l, o) partial, or the output itself
//      when it covers its whole row.
//   3. combine_kernel / combine_sk_kernel (rows, n_q): merge the partials.
#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "kvq_append.cuh"
#include "kvq_qprep.cuh"

#include <algorithm>
#include <atomic>
#include <mutex>

namespace kvq {

namespace {

template <int D>
struct Dec {
  static constexpr int NG = D / 64;          // 64-dim groups = consumer warps
  static constexpr int NW = NG;
  static constexpr int KPW = 64 / NW;        // keys per consumer warp in QK
  static constexpr int NTQ = KPW / 8;        // QK n-tiles per warp
  static constexpr int THREADS = NW * 32;      // no dedicated producer warp
  static constexpr int MIN_BLOCKS = D >= 512 ? 1 : (D == 256 ? 2 : 4);
};

constexpr int kMaxStages = 8;

// Shared memory holds a ring of stages; a stage is one 64-key tile, a K slot
// followed by a V slot.  A slot's code rows arrive as 4 chunks of 16
// consecutive keys, each chunk one bulk copy of 16 rows followed by 32 bytes
// of padding (chunk c starts 32*c bytes, mod 128, into the bank space, so rows
// of different chunks fall on different banks), then the 64 x (D/64) bf16
// scale block and the bias block.
__host__ __device__ constexpr int row_bytes(int D, int bits) { return D * bits / 8; }
__host__ __device__ constexpr int chunk_stride(int D, int bits) { return 16 * row_bytes(D, bits) + 32; }
__host__ __device__ constexpr int sb_bytes(int D) { return 64 * (D / 64) * 2; }
__host__ __device__ constexpr int slot_bytes(int D, int bits) { return 4 * chunk_stride(D, bits) + 2 * sb_bytes(D); }
__host__ __device__ constexpr int align128(int x) { return (x + 127) & ~127; }
// control block: kMaxStages mbarriers (16 reserved), max-exchange
// [2][16][NW] and l-exchange [16][NW] (floats)
__host__ __device__ constexpr int ctrl_bytes(int D) { return align128(16 * 8 + (3 * (D / 64) * 16) * 4); }
__host__ __device__ constexpr int slot0_off(int D) { return ctrl_bytes(D) + 2 * 16 * 64 * 2; }
// stages for a given dynamic shared-memory size
__host__ __device__ constexpr int ring_slots(int D, int bits, int smem) {
  return (smem - slot0_off(D)) / (2 * slot_bytes(D, bits)) < kMaxStages
             ? (smem - slot0_off(D)) / (2 * slot_bytes(D, bits)) : kMaxStages;
}

// ----------------------------------------------------------------------------
// 2. split-K attention over the quantized cache
// ----------------------------------------------------------------------------
struct TileRange {
  int t_begin, n_my, lo, hi;
};

// Load NG consecutive bf16 values (16 B for NG = 8) as raw words.
template <int NG>
__device__ __forceinline__ void load_bf16_row(const uint16_t* p, uint32_t (&w)[(NG + 1) / 2]) {
  if constexpr (NG == 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (NG == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x; w[1] = v.y;
  } else if constexpr (NG == 2) {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  } else {
    w[0] = *p;
  }
}
template <int NG>
__device__ __forceinline__ float bf16_word_at(const uint32_t (&w)[(NG + 1) / 2], int g) {
  return (g & 1) ? bf16hi_to_f(w[g >> 1]) : bf16lo_to_f(w[g >> 1]);
}

// The power of two the PV A operand (P * scale) is multiplied by, so that it
// stays clear of the f16 subnormal range; divided out at the end.  V rows are
// RMS-normalised without a weight (|v| <= sqrt(D), a group's range <= 2 sqrt(D)),
// so with P <= e^8: 2^2 at 4 bits and 2^6 at 8 bits keep P * scale * 2^k below
// f16's 65504.  A rotated layer's values v R reach D in size (range <= 2 D):
// 2^-2 and 2^2 there.
template <int BITS, bool ROT>
__host__ __device__ constexpr float pv_prescale() {
  return ROT ? (BITS == 4 ? 0.25f : 4.f) : (BITS == 4 ? 4.f : 64.f);
}

// Key mapping inside a tile (key 16c + s: chunk c < 4, slot s < 16).
//   QK n-tile j (0..7): column n is key 16*(n & 3) + 2j + (n >> 2), so the
//   eight B fragment rows sit in four chunks, two per chunk.
//   PV k-step kk (0..3): MMA k index 2t + b + 8a (t < 4, a, b < 2) is key
//   16t + 4kk + 2a + b, and P is stored in this order (column = 16*kk + k).
__device__ __forceinline__ int qk_key(int n, int j) { return 16 * (n & 3) + 2 * j + (n >> 2); }
__device__ __forceinline__ int pv_col(int key) {
  const int c = key >> 4, s = key & 15;
  return (s >> 2) * 16 + 2 * c + (s & 1) + 8 * ((s >> 1) & 1);
}

template <int NW>
__device__ __forceinline__ float max_over_warps(const float* p) {
  float m;
  if constexpr (NW >= 4) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    m = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
    if constexpr (NW == 8) {
      const float4 u = *reinterpret_cast<const float4*>(p + 4);
      m = fmaxf(m, fmaxf(fmaxf(u.x, u.y), fmaxf(u.z, u.w)));
    }
  } else if constexpr (NW == 2) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    m = fmaxf(v.x, v.y);
  } else {
    m = p[0];
  }
  return m;
}

// One run of consecutive tiles of one (row, kv head): the ring prologue, the
// pipelined loop and the epilogue, which writes the run's (m, l, o) partial
// to po / ml, or, when the run is the whole row (final_out), the normalised
// output.  Returns true when a bounded wait gave up.
template <int D, int BITS, bool ROT>
__device__ __forceinline__ bool decode_body(const DecodeArgs& a, const kvq_seq_cache& c, uint8_t* smem,
                                            const int nst, const TileRange tr, const int row, const int kvh,
                                            float* po, float* ml, const bool final_out) {
  using C = Dec<D>;
  constexpr int NG = C::NG, NW = C::NW, NTQ = C::NTQ;
  static_assert(NW == NG, "one PV warp per 64-dim group");
  constexpr int RB = row_bytes(D, BITS), CS = chunk_stride(D, BITS), SB = sb_bytes(D);
  constexpr int SLB = slot_bytes(D, BITS);
  constexpr uint32_t TX = 64 * RB + 2 * SB;     // bytes of one slot
  constexpr float L2E = 1.4426950408889634f;
  constexpr float PRESCALE = pv_prescale<BITS, ROT>();
  constexpr int GB = NG < 8 ? NG : 8;           // groups whose MMA chains run interleaved
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t4 = lane & 3, rq = lane >> 2;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  float* red = reinterpret_cast<float*>(smem + 16 * 8);     // [2][16][NW] tile max exchange
  float* lred = red + 2 * NW * 16;                          // [16][NW]
  uint8_t* Pbuf = smem + ctrl_bytes(D);                     // [2][16][64] f16, swizzled
  uint8_t* stages = smem + slot0_off(D);                    // stage i: K slot, then V slot
  uint8_t* const slots_base = stages;
  const int cap_tiles = c.capacity / kTileKeys;
  const size_t head_row0 = (size_t)kvh * c.capacity;
  // codes' units times the score scale (1, or 1/D exactly on a rotated layer)
  const float ksc = ROT ? kTwo24 * a.L.qk_scale : kTwo24;

  // Copies of one stage: per side 4 code chunks, the scale block and the bias
  // block; K copies by copy ids 0..5, V copies by 6..11 (copy id j is lane
  // j / NW of warp j % NW).  A stage is refilled only after a block barrier
  // that follows every read of its previous contents.
  const int my_copy = lane * NW + warp;
  auto issue = [&](int st, int slot_tile) {
    if (threadIdx.x == 0) mbar_arrive_expect_tx(&full[st], 2 * TX);
    if (my_copy < 12) {
      const bool v_side = my_copy >= 6;
      const int j = my_copy - (v_side ? 6 : 0);
      uint8_t* sl = stages + (2 * st + (v_side ? 1 : 0)) * SLB;
      const size_t r0 = head_row0 + (size_t)slot_tile * kTileKeys;
      if (j < 4) {
        const uint32_t* src = v_side ? c.v_codes : c.k_codes;
        bulk_g2s(sl + j * CS, reinterpret_cast<const uint8_t*>(src) + (r0 + 16 * j) * RB, 16 * RB, &full[st]);
      } else {
        const uint16_t* src = j == 4 ? (v_side ? c.v_scales : c.k_scales) : (v_side ? c.v_biases : c.k_biases);
        bulk_g2s(sl + 4 * CS + (j - 4) * SB, src + r0 * NG, SB, &full[st]);
      }
    }
  };
  int issued = 0, issue_st = 0, issue_slot = tr.t_begin % cap_tiles;
  auto refill = [&]() {
    if (issued < tr.n_my) {
      // a key the call's first kernel is still appending: wait for that grid
      if (a.fused_append && tr.t_begin + issued == tr.hi / kTileKeys) pdl_wait();
      issue(issue_st, issue_slot);
      if (++issue_st == nst) issue_st = 0;
      if (++issue_slot == cap_tiles) issue_slot = 0;
      ++issued;
    }
  };
  // prologue: fill the ring (the cache was written before this launch, but
  // for the newest keys of an attn_decode_append call: see refill)
  for (int i = 0; i < nst; ++i) refill();

  pdl_wait();                                   // q fragments come from qprep_kernel
  // QK A fragments (q heads x permuted head_dim) and the bias-term A fragment
  // (per-group q sums as f16 hi | lo parts)
  uint32_t qa[NG][4][4];
  uint32_t qb[4];
  {
    const size_t rkv = (size_t)row * a.L.n_kv + kvh;
    const uint4* src = a.ws.qfrag + rkv * NG * 4 * 32;
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint4 v = src[(g * 4 + ks) * 32 + lane];
        qa[g][ks][0] = v.x; qa[g][ks][1] = v.y; qa[g][ks][2] = v.z; qa[g][ks][3] = v.w;
      }
    const uint4 v = a.ws.qbias[rkv * 32 + lane];
    qb[0] = v.x; qb[1] = v.y; qb[2] = v.z; qb[3] = v.w;
  }

  float oacc[8][4];      // PV accumulator of this warp's group: 16 rows x 64 dims (permuted), 2^-24 units
  float cb[4];           // sum_j P_j * bias_j of this warp's group (column 0 is used)
#pragma unroll
  for (int i = 0; i < 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  cb[0] = cb[1] = cb[2] = cb[3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  bool dead = false;
  const int g_pv = warp;                        // PV group of this warp

  // Tiles flow through a two-deep software pipeline: while PV of tile i runs,
  // the same warp already computes QK of tile i+1, so the tensor cores always
  // have two independent streams of MMAs from every warp.
  int cons_st = 0, cons_phase = 0;
  auto wait_stage = [&]() -> const uint8_t* {
    const int stg = cons_st;
    if (!dead && !mbar_wait(&full[stg], cons_phase)) {
      dead = true;
      flag_error(a.ws.status, KVQ_DEV_TIMEOUT);
    }
    if (++cons_st == nst) { cons_st = 0; cons_phase ^= 1; }
    return stages + 2 * stg * SLB;
  };

  // V scale/bias of tile `ti`, this warp's group, as f16 pairs of consecutive
  // keys (scale pre-multiplied by PRESCALE), zero for keys outside the window.
  // Lane l forms pair l (keys 2l, 2l+1); PV lane (rq, t4) needs pairs
  // 8*t4 + m (m < 8), fetched by shuffles: sv[m], bv[m].
  auto build_vsb = [&](const uint8_t* vslot, int ti, uint32_t (&sv)[8], uint32_t (&bv)[8]) {
    const uint16_t* svs = reinterpret_cast<const uint16_t*>(vslot + 4 * CS);
    const uint16_t* svb = svs + 64 * NG;
    const int kp = (tr.t_begin + ti) * kTileKeys + 2 * lane;
    const bool v0 = kp >= tr.lo && kp <= tr.hi, v1 = kp + 1 >= tr.lo && kp + 1 <= tr.hi;
    const int i0 = 2 * lane * NG + g_pv;
    const float s0 = v0 ? bf16_to_f(svs[i0]) * PRESCALE : 0.f, s1 = v1 ? bf16_to_f(svs[i0 + NG]) * PRESCALE : 0.f;
    const float b0 = v0 ? bf16_to_f(svb[i0]) : 0.f, b1 = v1 ? bf16_to_f(svb[i0 + NG]) : 0.f;
    const uint32_t sp = pack_h2(s0, s1), bp = pack_h2(b0, b1);
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      sv[m] = __shfl_sync(0xffffffffu, sp, 8 * t4 + m);
      bv[m] = __shfl_sync(0xffffffffu, bp, 8 * t4 + m);
    }
  };

  // QK of tile `ti`: this warp's NTQ n-tiles (keys of slot j, one per chunk),
  // all q heads, full head_dim; masked keys get -inf.  Returns the row maxima.
  auto qk = [&](const uint8_t* stage, int ti, float (&S)[NTQ][4], float (&tmax)[2]) {
    const uint16_t* sks = reinterpret_cast<const uint16_t*>(stage + 4 * CS);
    const uint16_t* skb = sks + 64 * NG;
    const int tpos0 = (tr.t_begin + ti) * kTileKeys;
    tmax[0] = tmax[1] = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < NTQ; ++nt) {
      const int j = warp * NTQ + nt;
      // bias term: sum_g qsum[h][g] * bias[key][g] as one MMA (k = group for
      // the hi part, 8 + group for the lo part); B column rq is key qk_key(rq, j)
      float Sb[4];
      const int kB = qk_key(rq, j);
      {
        uint32_t bb = 0;
        if constexpr (NG == 1) {       // one group: a single bf16 (2-byte aligned only)
          bb = t4 == 0 ? pack_h2(bf16_to_f(skb[kB]), 0.f) : 0u;
        } else {
          if (2 * t4 < NG) {           // an aligned pair of groups 2*t4, 2*t4+1
            const uint32_t w = *reinterpret_cast<const uint32_t*>(skb + kB * NG + 2 * t4);
            bb = pack_h2(bf16lo_to_f(w), bf16hi_to_f(w));
          }
        }
        mma_f16_zc(Sb, qb, bb, bb);
      }
      // S columns 2*t4 and 2*t4+1
      const int kc0 = qk_key(2 * t4, j), kc1 = qk_key(2 * t4 + 1, j);
      uint32_t sw0[(NG + 1) / 2], sw1[(NG + 1) / 2];
      load_bf16_row<NG>(sks + kc0 * NG, sw0);
      load_bf16_row<NG>(sks + kc1 * NG, sw1);
      const uint8_t* krow = stage + (kB >> 4) * CS + (kB & 15) * RB + t4 * (BITS * 2);
      float T[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int g0 = 0; g0 < NG; g0 += GB) {
        float acc[GB][4];
        if constexpr (BITS == 4) {
          uint2 w[GB];
#pragma unroll
          for (int u = 0; u < GB; ++u) w[u] = *reinterpret_cast<const uint2*>(krow + (g0 + u) * 32);
#pragma unroll
          for (int u = 0; u < GB; ++u) mma_f16_zc(acc[u], qa[g0 + u][0], sub_n0(w[u].x), sub_n1(w[u].x));
#pragma unroll
          for (int u = 0; u < GB; ++u) {
            const uint32_t x = w[u].x >> 8;
            mma_f16(acc[u], qa[g0 + u][1], sub_n0(x), sub_n1(x));
          }
#pragma unroll
          for (int u = 0; u < GB; ++u) mma_f16(acc[u], qa[g0 + u][2], sub_n0(w[u].y), sub_n1(w[u].y));
#pragma unroll
          for (int u = 0; u < GB; ++u) {
            const uint32_t y = w[u].y >> 8;
            mma_f16(acc[u], qa[g0 + u][3], sub_n0(y), sub_n1(y));
          }
        } else {
          uint4 w[GB];
#pragma unroll
          for (int u = 0; u < GB; ++u) w[u] = *reinterpret_cast<const uint4*>(krow + (g0 + u) * 64);
#pragma unroll
          for (int u = 0; u < GB; ++u) mma_f16_zc(acc[u], qa[g0 + u][0], sub_b0(w[u].x), sub_b1(w[u].x));
#pragma unroll
          for (int u = 0; u < GB; ++u) mma_f16(acc[u], qa[g0 + u][1], sub_b0(w[u].y), sub_b1(w[u].y));
#pragma unroll
          for (int u = 0; u < GB; ++u) mma_f16(acc[u], qa[g0 + u][2], sub_b0(w[u].z), sub_b1(w[u].z));
#pragma unroll
          for (int u = 0; u < GB; ++u) mma_f16(acc[u], qa[g0 + u][3], sub_b0(w[u].w), sub_b1(w[u].w));
        }
#pragma unroll
        for (int u = 0; u < GB; ++u) {
          const float s0 = bf16_word_at<NG>(sw0, g0 + u), s1 = bf16_word_at<NG>(sw1, g0 + u);
          T[0] = fmaf(s0, acc[u][0], T[0]);
          T[1] = fmaf(s1, acc[u][1], T[1]);
          T[2] = fmaf(s0, acc[u][2], T[2]);
          T[3] = fmaf(s1, acc[u][3], T[3]);
        }
      }
      // the code products are in units of 2^-24 (times the score scale; the
      // bias term arrives scaled)
      const int kp0 = tpos0 + kc0, kp1 = tpos0 + kc1;
      const bool v0 = kp0 >= tr.lo && kp0 <= tr.hi, v1 = kp1 >= tr.lo && kp1 <= tr.hi;
      S[nt][0] = v0 ? fmaf(T[0], ksc, Sb[0]) : -INFINITY;
      S[nt][1] = v1 ? fmaf(T[1], ksc, Sb[1]) : -INFINITY;
      S[nt][2] = v0 ? fmaf(T[2], ksc, Sb[2]) : -INFINITY;
      S[nt][3] = v1 ? fmaf(T[3], ksc, Sb[3]) : -INFINITY;
      tmax[0] = fmaxf(tmax[0], fmaxf(S[nt][0], S[nt][1]));
      tmax[1] = fmaxf(tmax[1], fmaxf(S[nt][2], S[nt][3]));
    }
#pragma unroll
    for (int m = 1; m <= 2; m <<= 1) {
      tmax[0] = fmaxf(tmax[0], __shfl_xor_sync(0xffffffffu, tmax[0], m));
      tmax[1] = fmaxf(tmax[1], __shfl_xor_sync(0xffffffffu, tmax[1], m));
    }
  };

  auto post_max = [&](const float (&tmax)[2], int bf) {
    float* redb = red + bf * NW * 16;
    if (t4 == 0) { redb[rq * NW + warp] = tmax[0]; redb[(rq + 8) * NW + warp] = tmax[1]; }
  };

  // P (f16) = e^(S - ref) of this warp's keys into the P buffer; returns the
  // row sums of the stored (rounded) values
  auto store_p = [&](const float (&S)[NTQ][4], int bf, const float (&ref)[2], float (&lsum)[2]) {
    uint8_t* Pb = Pbuf + bf * (16 * 64 * 2);
    lsum[0] = lsum[1] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NTQ; ++nt) {
      const int j = warp * NTQ + nt;
      const int col0 = pv_col(qk_key(2 * t4, j)), col1 = pv_col(qk_key(2 * t4 + 1, j));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float p0 = 0.f, p1 = 0.f;
        if (ref[h] != -INFINITY) {
          p0 = exp2f((S[nt][2 * h] - ref[h]) * L2E);
          p1 = exp2f((S[nt][2 * h + 1] - ref[h]) * L2E);
        }
        const __half h0 = __float2half_rn(p0), h1 = __float2half_rn(p1);
        lsum[h] += __half2float(h0) + __half2float(h1);
        const int prow = rq + 8 * h;
        uint8_t* prw = Pb + prow * 128;
        *reinterpret_cast<__half*>(prw + (((col0 >> 3) ^ (prow & 7)) << 4) + (col0 & 7) * 2) = h0;
        *reinterpret_cast<__half*>(prw + (((col1 >> 3) ^ (prow & 7)) << 4) + (col1 & 7) * 2) = h1;
      }
    }
  };

  // after the max exchange: the tile's row maxima (every warp reads the same
  // values, so anything derived from them is uniform over the block)
  auto tile_max = [&](int bf, float (&mt)[2]) {
    const float* redb = red + bf * NW * 16;
#pragma unroll
    for (int h = 0; h < 2; ++h) mt[h] = max_over_warps<NW>(redb + (rq + 8 * h) * NW);
  };

  // exact online-softmax step: new running max, P against it, running sums;
  // returns the rescale factors of the old state
  auto softmax = [&](const float (&S)[NTQ][4], int bf, const float (&mt)[2], float (&alpha)[2]) {
    float m_new[2], lsum[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      m_new[h] = fmaxf(m_run[h], mt[h]);
      alpha[h] = m_new[h] == -INFINITY ? 1.f : exp2f((m_run[h] - m_new[h]) * L2E);
    }
    store_p(S, bf, m_new, lsum);
#pragma unroll
    for (int h = 0; h < 2; ++h) { l_run[h] = l_run[h] * alpha[h] + lsum[h]; m_run[h] = m_new[h]; }
  };

  auto rescale = [&](const float (&alpha)[2]) {
    if (!__all_sync(0xffffffffu, alpha[0] == 1.f && alpha[1] == 1.f)) {
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        oacc[nt][0] *= alpha[0]; oacc[nt][1] *= alpha[0];
        oacc[nt][2] *= alpha[1]; oacc[nt][3] *= alpha[1];
      }
      cb[0] *= alpha[0]; cb[1] *= alpha[0]; cb[2] *= alpha[1]; cb[3] *= alpha[1];
    }
  };

  // PV of one tile for this warp's 64-dim group: O += (P * scale) codes + P bias
  auto pv = [&](const uint8_t* vslot, int bf, const uint32_t (&sv)[8], const uint32_t (&bv)[8]) {
    const uint8_t* Pb = Pbuf + bf * (16 * 64 * 2);
    // this lane's B rows (k = 2*t4 + b + 8a) are keys 16*t4 + 4kk + 2a + b: all in chunk t4
    const uint8_t* vrow = vslot + t4 * CS + (BITS == 4 ? g_pv * 32 + rq * 4 : g_pv * 64 + rq * 8);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      {
        const int mtx = lane >> 3, i = lane & 7;
        const int prow = (mtx & 1) * 8 + i;
        const int chunk = (kk * 2 + (mtx >> 1)) ^ (prow & 7);
        ldmatrix_x4(pa, Pb + prow * 128 + chunk * 16);
      }
      // key pairs (16*t4 + 4kk, +1) and (16*t4 + 4kk + 2, +3): pairs 8*t4 + 2kk, +1
      const uint32_t sAB = sv[2 * kk], sCD = sv[2 * kk + 1];
      // bias column: only B column 0 (lanes 0..3) is non-zero
      const uint32_t bAB = rq == 0 ? bv[2 * kk] : 0u, bCD = rq == 0 ? bv[2 * kk + 1] : 0u;
      mma_f16(cb, pa, bAB, bCD);
      const uint32_t ps[4] = {h2_mul(pa[0], sAB), h2_mul(pa[1], sAB), h2_mul(pa[2], sCD), h2_mul(pa[3], sCD)};
      const uint8_t* vk = vrow + 4 * kk * RB;
      if constexpr (BITS == 4) {
        const uint32_t wa = *reinterpret_cast<const uint32_t*>(vk);
        const uint32_t wb = *reinterpret_cast<const uint32_t*>(vk + RB);
        const uint32_t wc = *reinterpret_cast<const uint32_t*>(vk + 2 * RB);
        const uint32_t wd = *reinterpret_cast<const uint32_t*>(vk + 3 * RB);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          // byte q of both keys into the low byte of each half
          const uint32_t sel = (uint32_t)(q | (q << 4) | ((4 + q) << 8) | ((4 + q) << 12));
          const uint32_t xab = prmt(wa, wb, sel), xcd = prmt(wc, wd, sel);
          mma_f16(oacc[2 * q], ps, sub_n0(xab), sub_n0(xcd));
          mma_f16(oacc[2 * q + 1], ps, sub_n1(xab), sub_n1(xcd));
        }
      } else {
        const uint2 wa = *reinterpret_cast<const uint2*>(vk);
        const uint2 wb = *reinterpret_cast<const uint2*>(vk + RB);
        const uint2 wc = *reinterpret_cast<const uint2*>(vk + 2 * RB);
        const uint2 wd = *reinterpret_cast<const uint2*>(vk + 3 * RB);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int bq = q & 3;
          const uint32_t sel = (uint32_t)(bq | ((4 + bq) << 8));
          const uint32_t xab = prmt(q < 4 ? wa.x : wa.y, q < 4 ? wb.x : wb.y, sel) & 0x00FF00FFu;
          const uint32_t xcd = prmt(q < 4 ? wc.x : wc.y, q < 4 ? wd.x : wd.y, sel) & 0x00FF00FFu;
          mma_f16(oacc[q], ps, xab, xcd);
        }
      }
    }
  };

  // ---- pipeline prologue: scores and P of tile 0 ----
  float S[NTQ][4], tmax[2], alpha[2], mt[2];
  const uint8_t* cur = wait_stage();
  {
    qk(cur, 0, S, tmax);
    post_max(tmax, 0);
    named_bar(1, NW * 32);
    tile_max(0, mt);
    softmax(S, 0, mt, alpha);
    named_bar(1, NW * 32);
  }
  // ---- steady state: QK(it+1) alongside PV(it) ----
  // P of tile it+1 is formed before the max exchange against the running max
  // (the same in every warp).  Scores up to kSlack above it keep P <= e^8,
  // well inside f16 even after the V scale is folded in; then the exchange
  // barrier also publishes P and nothing is rescaled.  A tile that exceeds the
  // running max by more has P redone against its own maximum.
  constexpr float kSlack = 8.f;
  for (int it = 0; it + 1 < tr.n_my; ++it) {
    const int bf = it & 1;
    const uint8_t* nxt = wait_stage();
    uint32_t sv[8], bv[8];
    build_vsb(cur + SLB, it, sv, bv);
    qk(nxt, it + 1, S, tmax);
    float lsum[2];
    store_p(S, bf ^ 1, m_run, lsum);
    pv(cur + SLB, bf, sv, bv);
    post_max(tmax, bf ^ 1);
    named_bar(1, NW * 32);
    refill();                                   // every warp is done with tile it
    tile_max(bf ^ 1, mt);
    if (__any_sync(0xffffffffu, mt[0] > m_run[0] + kSlack || mt[1] > m_run[1] + kSlack)) {
      softmax(S, bf ^ 1, mt, alpha);
      rescale(alpha);
      named_bar(1, NW * 32);
    } else {
      l_run[0] += lsum[0];
      l_run[1] += lsum[1];
    }
    cur = nxt;
  }
  {
    uint32_t sv[8], bv[8];
    build_vsb(cur + SLB, tr.n_my - 1, sv, bv);
    pv(cur + SLB, (tr.n_my - 1) & 1, sv, bv);
  }
  pdl_launch();
  // a timed-out wait may leave copies in flight: they must land before exit
  if (dead && threadIdx.x == 0)
    for (int i = max(0, issued - nst); i < issued; ++i) mbar_wait(&full[i % nst], (i / nst) & 1);

  // ---- write this split's partial (m, l, o) ----
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
  if (t4 == 0) { lred[rq * NW + warp] = l_run[0]; lred[(rq + 8) * NW + warp] = l_run[1]; }
  // bias column 0 lives in lanes with t4 == 0 (c0: row rq, c2: row rq + 8)
  const float bias_r = __shfl_sync(0xffffffffu, cb[0], lane & ~3);
  const float bias_r8 = __shfl_sync(0xffffffffu, cb[2], lane & ~3);
  const bool any_dead = __syncthreads_or(dead);
  const int G = a.L.G;
  float* lfin = red;                            // [16] row sums (final output); the max exchange is done
  if (warp == 0) {
    // every warp holds the same running max; warp 0 writes it
    if (!final_out && t4 == 0) { ml[rq] = m_run[0]; ml[rq + 8] = m_run[1]; }
    if (lane < 16) {
      float l = 0.f;
      for (int w = 0; w < NW; ++w) l += lred[lane * NW + w];
      if (final_out) lfin[lane] = l;
      else ml[16 + lane] = l;
    }
  }
  // the o partial goes through shared memory (the stages are free: every warp
  // passed the barrier above after its last read) so that the global stores
  // are whole 16-byte pieces of rows; rows padded by 4 floats against bank
  // conflicts
  constexpr int PS = D + 4;
  float* ps = reinterpret_cast<float*>(slots_base);
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    // codes were 2^-24 units (2^-20 for 4-bit codes from bits 4..7: odd nt)
    const float uns = (BITS == 4 && (nt & 1) ? kTwo24 / 16.f : kTwo24) / PRESCALE;
    const int d0 = g_pv * 64 + 8 * (2 * t4) + nt, d1 = d0 + 8;
    ps[rq * PS + d0] = fmaf(oacc[nt][0], uns, bias_r);
    ps[rq * PS + d1] = fmaf(oacc[nt][1], uns, bias_r);
    ps[(rq + 8) * PS + d0] = fmaf(oacc[nt][2], uns, bias_r8);
    ps[(rq + 8) * PS + d1] = fmaf(oacc[nt][3], uns, bias_r8);
  }
  named_bar(1, NW * 32);
  if (!final_out) {
    for (int i = threadIdx.x; i < G * (D / 4); i += NW * 32) {
      const int r = i / (D / 4), c4 = i % (D / 4);
      *reinterpret_cast<float4*>(po + r * D + 4 * c4) = *reinterpret_cast<const float4*>(ps + r * PS + 4 * c4);
    }
  } else {
    // the whole row in this run: out = o / l, as the merge of one partial;
    // on a rotated layer the rows are un-rotated first: o R^T / D
    if constexpr (ROT) {
#pragma unroll 1
      for (int h = 1; h < D; h <<= 1) {
        for (int p = threadIdx.x; p < G * (D / 2); p += NW * 32) {
          const int r = p / (D / 2), q = p % (D / 2);
          const int i = r * PS + (q / h) * 2 * h + (q % h);
          const float u = ps[i], v = ps[i + h];
          ps[i] = u + v;
          ps[i + h] = u - v;
        }
        named_bar(1, NW * 32);
      }
    }
    const size_t ob = ((size_t)row * a.L.n_q + (size_t)kvh * G) * D;
    for (int i = threadIdx.x; i < G * D; i += NW * 32) {
      const int r = i / D, d = i % D;
      float o = ps[r * PS + d] * (1.f / lfin[r]);
      if constexpr (ROT) o *= (float)__ldg(a.L.rot + d) * a.L.qk_scale;
      if (a.out_f32) reinterpret_cast<float*>(a.out)[ob + i] = o;
      else reinterpret_cast<uint16_t*>(a.out)[ob + i] = f_to_bf16_rn(o);
    }
  }
  return any_dead;
}

// Visible keys of a row and whether its cache can serve them: every key from
// lo up to the newest cached position must own its slot.
struct RowWin {
  int lo, hi, tiles;     // tiles = 0 for a sequence the kernels skip
  bool ok;
};
__device__ __forceinline__ RowWin row_window(const DecodeArgs& a, const RowInfo& ri, const kvq_seq_cache& c) {
  const int p = ri.p, W = a.L.window;
  const int lo = W > 0 ? max(0, p - W + 1) : 0, hi = p;
  const bool ok = seq_ok(c) && p >= 0 && ri.newest < (1 << 24) && p <= ri.newest &&
                  (ri.newest - lo + 1) <= c.capacity;
  return {lo, hi, ok ? hi / kTileKeys - lo / kTileKeys + 1 : 0, ok};
}

// Stream-K schedule (a.sk_ctas > 0, decode rows only): the tiles of all
// (row, kv head) units, concatenated in unit order (u = row * n_kv + kvh),
// are cut into nc equal ranges, range c = [c*T/nc, (c+1)*T/nc) for CTA c.  A
// CTA walks its range unit by unit; a unit that lies wholly inside the range
// is written as final output, every other piece as a partial in slot 0 (the
// range's first piece) or 1 (its last piece) of the CTA.  With equal rows
// and at least as many CTAs as units, nc is a multiple of the unit count so
// that no range crosses a unit boundary.  Every CTA computes the same plan
// from the rows' positions; CTA 0 also stores it for the merge kernel:
// plan[0] = T, plan[1] = nc, plan[2 + r] = tiles of rows < r (per kv head).
// The walk's state lives in shared memory (it is read only between pieces):
struct SkWalk {
  long long b, e, pos;   // the CTA's range and the next tile to run
  long long next;        // end of the current piece
  int r, kvh;            // unit of tile `pos`
};

__device__ __forceinline__ long long sk_range_start(long long c, long long T, long long nc) { return c * T / nc; }
// shared memory of the plan, at the end of the dynamic allocation: the row
// prefix [n_rows + 1], three control ints, then the walk (8-byte aligned)
__host__ __device__ constexpr int sk_plan_bytes(int n_rows) {
  return (((n_rows + 5) & ~1) * 4 + (int)sizeof(SkWalk) + 127) & ~127;
}

// One CTA of the attention kernel.  Fixed chunks: (bx, by, bz) = (row, kv
// head, split) of the call `a`; stream-K: bx is the CTA's index in the wave.
template <int D, bool SK, bool ROT>
__device__ __forceinline__ void decode_cta(const DecodeArgs& a, const int smem_total, const int bx, const int by,
                                           const int bz) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr bool sk = SK;
  const int ring_smem = sk ? smem_total - sk_plan_bytes(a.n_rows) : smem_total;
  const int n_kv = a.L.n_kv;
  int row, kvh;
  kvq_seq_cache c;
  TileRange tr;
  float* po;
  float* ml;
  bool final_out = false;
  int* pr = reinterpret_cast<int*>(smem + ring_smem);        // [n_rows + 1] row tile prefix (stream-K)
  SkWalk* wk = reinterpret_cast<SkWalk*>(pr + ((a.n_rows + 5) & ~1));
  if constexpr (!SK) {
    row = bx; kvh = by;
    const int split = bz;
    const RowInfo ri = row_info(a, row);
    c = a.seqs[ri.s];
    const RowWin rw = row_window(a, ri, c);
    const int t_lo = rw.lo / kTileKeys;
    const int chunk = a.chunk_tiles > 0 ? a.chunk_tiles : (rw.tiles + a.splits - 1) / a.splits;
    const int t_begin = t_lo + split * chunk;
    const int n_my = rw.ok ? max(0, min(chunk, t_lo + rw.tiles - t_begin)) : 0;
    const size_t pidx = ((size_t)row * n_kv + kvh) * a.splits + split;
    if (n_my == 0) {
      // nothing to read: an empty partial (m = -inf), or NaN for a bad sequence
      if (!rw.ok && split == 0 && kvh == 0 && threadIdx.x == 0) {
        pdl_wait();                                   // after q prep has cleared the status word
        flag_error(a.ws.status, KVQ_DEV_BADSEQ);
      }
      if (threadIdx.x < 16) {
        a.ws.part_ml[pidx * 32 + threadIdx.x] = rw.ok ? -INFINITY : __int_as_float(0x7fc00000);
        a.ws.part_ml[pidx * 32 + 16 + threadIdx.x] = 0.f;
      }
      pdl_launch();
      return;
    }
    tr = TileRange{t_begin, n_my, rw.lo, rw.hi};
    po = a.ws.part_o + pidx * 16 * D;
    ml = a.ws.part_ml + pidx * 32;
  } else {
    // ---- the plan: tiles per row, prefix over rows ----
    const int n_rows = a.n_rows, tid = threadIdx.x, NT = blockDim.x;
    int* ctl = pr + a.n_rows + 1;                            // min tiles, max tiles, any bad row
    if (tid == 0) { ctl[0] = 0x7fffffff; ctl[1] = 0; ctl[2] = 0; }
    __syncthreads();
    int mn = 0x7fffffff, mx = 0, bad = 0;
    for (int r = tid; r < n_rows; r += NT) {
      const RowWin rw = row_window(a, row_info(a, r), a.seqs[r]);
      pr[r + 1] = rw.tiles;
      mn = min(mn, rw.tiles); mx = max(mx, rw.tiles); bad |= !rw.ok;
    }
    atomicMin(ctl, mn); atomicMax(ctl + 1, mx);
    if (bad) atomicOr(ctl + 2, 1);
    __syncthreads();
    if (tid < 32) {                                          // inclusive scan, lane l takes a block of rows
      const int per = (n_rows + 31) / 32, r0 = min(n_rows, tid * per), r1 = min(n_rows, r0 + per);
      int sum = 0;
      for (int r = r0; r < r1; ++r) sum += pr[r + 1];
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += v;
      }
      int run = incl - sum;
      for (int r = r0; r < r1; ++r) { run += pr[r + 1]; pr[r + 1] = run; }
      if (tid == 0) pr[0] = 0;
    }
    __syncthreads();
    const long long T = (long long)n_kv * pr[n_rows];
    const long long U = (long long)n_rows * n_kv;
    long long nc = a.sk_ctas;
    if (ctl[0] == ctl[1] && ctl[0] > 0 && U <= nc) {
      // equal rows: a whole number of ranges per unit, none below kSkMinTiles
      nc = U * max(1LL, min(nc / U, (long long)ctl[0] / kSkMinTiles));
    } else {
      nc = min(nc, max(1LL, T / kSkMinTiles));
    }
    if (bx == 0) {
      long long* plan = a.ws.plan;
      for (int r = tid; r <= n_rows; r += NT) plan[2 + r] = pr[r];
      if (tid == 0) { plan[0] = T; plan[1] = nc; }
      if (ctl[2] && tid == 0) {
        pdl_wait();                                          // after q prep has cleared the status word
        flag_error(a.ws.status, KVQ_DEV_BADSEQ);
      }
    }
    const long long cta = bx;
    const long long b = sk_range_start(cta, T, nc), e = sk_range_start(cta + 1, T, nc);
    if (cta >= nc || b >= e) { pdl_launch(); return; }
    if (tid == 0) {
      // the row holding tile b: the largest r with n_kv * pr[r] <= b (it has tiles)
      int lo_r = 0, hi_r = n_rows - 1;
      while (lo_r < hi_r) {
        const int mid = (lo_r + hi_r + 1) >> 1;
        if ((long long)n_kv * pr[mid] <= b) lo_r = mid; else hi_r = mid - 1;
      }
      wk->b = b; wk->e = e; wk->pos = b;
      wk->r = lo_r;
      wk->kvh = (int)((b - (long long)n_kv * pr[lo_r]) / (pr[lo_r + 1] - pr[lo_r]));
    }
    __syncthreads();
  }
  // stream-K: the piece of the walk's current unit (every thread reads the
  // walk; thread 0 records where the piece ends)
  auto sk_piece = [&]() {
    const int t = pr[wk->r + 1] - pr[wk->r];
    const long long pu = (long long)n_kv * pr[wk->r] + (long long)wk->kvh * t;
    const int s0 = (int)(wk->pos - pu), s1 = (int)(min(wk->e, pu + t) - pu);
    row = wk->r; kvh = wk->kvh;
    const RowInfo ri = row_info(a, row);
    c = a.seqs[ri.s];
    const RowWin rw = row_window(a, ri, c);
    tr = TileRange{rw.lo / kTileKeys + s0, s1 - s0, rw.lo, rw.hi};
    final_out = s0 == 0 && s1 == t;
    const size_t pidx = (size_t)bx * 2 + (pu > wk->b ? 1 : 0);
    po = a.ws.part_o + pidx * 16 * D;
    ml = a.ws.part_ml + pidx * 32;
    if (threadIdx.x == 0) wk->next = pu + s1;
  };
  if constexpr (SK) sk_piece();
  for (;;) {
    if (threadIdx.x == 0) {
      for (int i = 0; i < kMaxStages; ++i) mbar_init(reinterpret_cast<uint64_t*>(smem) + i, 1);
      fence_mbar_init();
    }
    __syncthreads();
    const int nst = ring_slots(D, c.bits, ring_smem);
    const bool dead = c.bits == 4 ? decode_body<D, 4, ROT>(a, c, smem, nst, tr, row, kvh, po, ml, final_out)
                                  : decode_body<D, 8, ROT>(a, c, smem, nst, tr, row, kvh, po, ml, final_out);
    if (!SK || dead) break;
    // every thread is past its reads of the walk (decode_body has block
    // barriers); thread 0 moves it to the next unit with tiles
    if (threadIdx.x == 0) {
      wk->pos = wk->next;
      if (wk->pos < wk->e && ++wk->kvh == n_kv) {
        wk->kvh = 0;
        do { ++wk->r; } while (pr[wk->r + 1] == pr[wk->r]);
      }
    }
    // every read of the ring and of the staged partial is done, and the
    // generic-proxy writes are ordered before the next bulk copies
    fence_proxy_async();
    __syncthreads();
    if (wk->pos >= wk->e) break;
    sk_piece();
  }
}

template <int D, bool SK, bool ROT>
__global__ void __launch_bounds__(Dec<D>::THREADS, Dec<D>::MIN_BLOCKS)
decode_kernel(const DecodeArgs a, const int smem_total) {
  decode_cta<D, SK, ROT>(a, smem_total, blockIdx.x, blockIdx.y, blockIdx.z);
}

// Grouped schedule: the fixed-chunk CTAs of every group in one 1-D grid.
template <int D, bool ROT>
__global__ void __launch_bounds__(Dec<D>::THREADS, Dec<D>::MIN_BLOCKS)
decode_grouped_kernel(const GroupedDecode ga, const int smem_total) {
  const int g = group_of(ga.cta_base, ga.n, blockIdx.x);
  const DecodeArgs& a = ga.g[g];
  const int local = blockIdx.x - ga.cta_base[g];
  const int per_row = a.L.n_kv * a.splits;
  const int row = local / per_row, rem = local - row * per_row;
  decode_cta<D, false, ROT>(a, smem_total, row, rem / a.splits, rem % a.splits);
}

// The output value of dim d = threadIdx.x of a row (blockDim == D) on a
// rotated layer: o R^T / D = s_d (o H)_d / D, H the Sylvester Hadamard matrix,
// by in-place butterflies in `buf` (D floats of shared memory, reused: the
// caller is done with it).  Every thread of the block calls it.
template <int D>
__device__ __forceinline__ float unrotate_dim(float o, const int8_t* signs, float inv_d, float* buf) {
  const int d = threadIdx.x;
  __syncthreads();                               // every earlier read of buf is done
  buf[d] = o;
  __syncthreads();
#pragma unroll 1
  for (int h = 1; h < D; h <<= 1) {
    if ((d & h) == 0) {
      const float u = buf[d], v = buf[d + h];
      buf[d] = u + v;
      buf[d + h] = u - v;
    }
    __syncthreads();
  }
  return buf[d] * (float)__ldg(signs + d) * inv_d;
}

// ----------------------------------------------------------------------------
// 3. merge split partials: out = sum_i e^(m_i - M) o_i / sum_i e^(m_i - M) l_i
// ----------------------------------------------------------------------------
template <int D, bool ROT>
__device__ __forceinline__ void combine_row(const DecodeArgs& a, const int row, const int hq) {
  __shared__ float wsm[D > 256 ? D : 256];   // split weights, then (rotated layers) the output row
  __shared__ float inv_l;
  pdl_launch();                              // the next call's first kernel waits for this grid itself
  pdl_wait();
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
  const int d = threadIdx.x;               // one output dim per thread
  const float* po = a.ws.part_o + (base * 16 + r) * D + d;
  float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
  int i = 0;
  // a split with no keys wrote no o partial (its weight is 0): never touch it
  for (; i + 8 <= S; i += 8) {
    float o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) o[k] = wsm[i + k] != 0.f ? po[(size_t)(i + k) * 16 * D] : 0.f;
    acc0 = fmaf(wsm[i], o[0], acc0); acc1 = fmaf(wsm[i + 1], o[1], acc1);
    acc2 = fmaf(wsm[i + 2], o[2], acc2); acc3 = fmaf(wsm[i + 3], o[3], acc3);
    acc0 = fmaf(wsm[i + 4], o[4], acc0); acc1 = fmaf(wsm[i + 5], o[5], acc1);
    acc2 = fmaf(wsm[i + 6], o[6], acc2); acc3 = fmaf(wsm[i + 7], o[7], acc3);
  }
  for (; i < S; ++i)
    if (wsm[i] != 0.f) acc0 = fmaf(wsm[i], po[(size_t)i * 16 * D], acc0);
  float o = ((acc0 + acc1) + (acc2 + acc3)) * inv_l;
  if constexpr (ROT) o = unrotate_dim<D>(o, a.L.rot, a.L.qk_scale, wsm);
  const size_t oi = ((size_t)row * a.L.n_q + hq) * D + d;
  if (a.out_f32) reinterpret_cast<float*>(a.out)[oi] = o;
  else reinterpret_cast<uint16_t*>(a.out)[oi] = f_to_bf16_rn(o);
}

template <int D, bool ROT>
__global__ void __launch_bounds__(D)
combine_kernel(const DecodeArgs a) {
  combine_row<D, ROT>(a, blockIdx.x, blockIdx.y);
}

template <int D, bool ROT>
__global__ void __launch_bounds__(D)
combine_grouped_kernel(const GroupedDecode ga) {
  const int g = group_of(ga.row_base, ga.n, blockIdx.x);
  combine_row<D, ROT>(ga.g[g], blockIdx.x - ga.row_base[g], blockIdx.y);
}

// Stream-K merge: one block per (row, q head) of a unit whose tiles were
// split between CTAs c_first .. c_last (a unit inside one CTA was written
// by the attention kernel).  CTA c's piece of the unit is its slot 0 unless
// the unit starts after c's range start (slot 1).
__device__ __forceinline__ long long sk_cta_of(long long x, long long T, long long nc) {
  return ((x + 1) * nc - 1) / T;                 // the largest c with c*T/nc <= x
}

template <int D, bool ROT>
__global__ void __launch_bounds__(D)
combine_sk_kernel(const DecodeArgs a) {
  __shared__ float wsm[1024];
  __shared__ int pid[1024];
  __shared__ float inv_l;
  pdl_launch();                              // the next call's first kernel waits for this grid itself
  pdl_wait();
  const int row = blockIdx.x, hq = blockIdx.y;
  const int G = a.L.G, kvh = hq / G, r = hq % G, n_kv = a.L.n_kv;
  const long long* plan = a.ws.plan;
  const long long T = plan[0], nc = plan[1];
  const long long p0 = plan[2 + row], t = plan[3 + row] - p0;
  const size_t oi = ((size_t)row * a.L.n_q + hq) * D + threadIdx.x;
  if (t == 0) {                                  // a skipped sequence
    if (a.out_f32) reinterpret_cast<float*>(a.out)[oi] = __int_as_float(0x7fc00000);
    else reinterpret_cast<uint16_t*>(a.out)[oi] = 0x7fc0u;
    return;
  }
  const long long pu = n_kv * p0 + kvh * t;
  const long long c0 = sk_cta_of(pu, T, nc), c1 = sk_cta_of(pu + t - 1, T, nc);
  if (c0 == c1) return;
  const int S = (int)(c1 - c0 + 1);              // <= nc <= 1024
  for (int i = threadIdx.x; i < S; i += blockDim.x) {
    const long long cc = c0 + i;
    pid[i] = (int)(cc * 2 + (pu > cc * T / nc ? 1 : 0));
  }
  __syncthreads();
  auto piece = [&](int i) -> size_t { return (size_t)pid[i]; };
  if (threadIdx.x < 32) {
    float M = -INFINITY;
    for (int i = threadIdx.x; i < S; i += 32) M = fmaxf(M, a.ws.part_ml[piece(i) * 32 + r]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int i = threadIdx.x; i < S; i += 32) {
      const size_t pi = piece(i);
      const float m = a.ws.part_ml[pi * 32 + r];
      const float w = m == -INFINITY ? 0.f : exp2f((m - M) * 1.4426950408889634f);
      wsm[i] = w;
      L += w * a.ws.part_ml[pi * 32 + 16 + r];
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (threadIdx.x == 0) inv_l = 1.f / L;
  }
  __syncthreads();
  const int d = threadIdx.x;
  float acc0 = 0.f, acc1 = 0.f;
  int i = 0;
  for (; i + 2 <= S; i += 2) {
    const float o0 = a.ws.part_o[(piece(i) * 16 + r) * D + d];
    const float o1 = a.ws.part_o[(piece(i + 1) * 16 + r) * D + d];
    acc0 = fmaf(wsm[i], o0, acc0);
    acc1 = fmaf(wsm[i + 1], o1, acc1);
  }
  if (i < S) acc0 = fmaf(wsm[i], a.ws.part_o[(piece(i) * 16 + r) * D + d], acc0);
  float o = (acc0 + acc1) * inv_l;
  if constexpr (ROT) o = unrotate_dim<D>(o, a.L.rot, a.L.qk_scale, wsm);
  if (a.out_f32) reinterpret_cast<float*>(a.out)[oi] = o;
  else reinterpret_cast<uint16_t*>(a.out)[oi] = f_to_bf16_rn(o);
}

template <int D>
constexpr int decode_smem_bytes() {
  // D = 512: one CTA per SM with the largest shared carve-out; smaller head
  // dims leave room for several CTAs per SM.
  return D >= 512 ? 227 * 1024 : (D == 256 ? 110 * 1024 : 56 * 1024);
}

// attn_decode_append's first kernel: blocks y < nq_blocks prep q (as
// qprep_kernel), the others append the rows' new K/V (as append_kernel); the
// two halves share nothing and run side by side.
template <int D>
__global__ void __launch_bounds__(1024)
prep_append_kernel(const DecodeArgs a, const AppendArgs ap, const RopeFreqs freqs, const int hpb,
                   const int nq_blocks, const int ipb) {
  if ((int)blockIdx.y < nq_blocks) qprep_block<D>(a, freqs, hpb, blockIdx.x, blockIdx.y);
  else append_block<D>(ap, freqs, ipb, blockIdx.x, blockIdx.y - nq_blocks);
}

// The shared-memory opt-in of every attention kernel of head_dim D, once per
// device (a lock: host threads may make their first call on a device at the
// same time).
template <int D>
cudaError_t decode_attrs(int smem) {
  static std::atomic<bool> attr_set[64];
  static std::mutex attr_mu;
  cudaError_t e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(attr_mu);
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
      const void* fns[6] = {
          reinterpret_cast<const void*>(decode_kernel<D, false, false>),
          reinterpret_cast<const void*>(decode_kernel<D, true, false>),
          reinterpret_cast<const void*>(decode_kernel<D, false, true>),
          reinterpret_cast<const void*>(decode_kernel<D, true, true>),
          reinterpret_cast<const void*>(decode_grouped_kernel<D, false>),
          reinterpret_cast<const void*>(decode_grouped_kernel<D, true>)};
      for (const void* fn : fns)
        if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
          return e;
      // the fused q + K/V prep of a rotated layer: one float64 row per head
      // or item beside the static shared memory of both halves
      if ((e = cudaFuncSetAttribute(prep_append_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (1024 / Qp<D>::TH) * D * (int)sizeof(double))) != cudaSuccess)
        return e;
      attr_set[dev].store(true, std::memory_order_release);
    }
  }
  return cudaSuccess;
}

// The attention and merge launches of a call, programmatic dependents of the
// call's first kernel.
template <int D>
cudaError_t launch_read_merge_t(const DecodeArgs& a, cudaStream_t st) {
  const int smem = decode_smem_bytes<D>();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = a.sk_ctas > 0 ? dim3(a.sk_ctas) : dim3(a.n_rows, a.L.n_kv, a.splits);
  cfg.blockDim = dim3(Dec<D>::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if ((e = prof_before(st)) != cudaSuccess) return e;
  if (a.L.rot)       // the deferred TurboQuant read: score scale, PV pre-scale, output un-rotation
    e = a.sk_ctas > 0 ? cudaLaunchKernelEx(&cfg, decode_kernel<D, true, true>, a, smem)
                      : cudaLaunchKernelEx(&cfg, decode_kernel<D, false, true>, a, smem);
  else
    e = a.sk_ctas > 0 ? cudaLaunchKernelEx(&cfg, decode_kernel<D, true, false>, a, smem)
                      : cudaLaunchKernelEx(&cfg, decode_kernel<D, false, false>, a, smem);
  if (e != cudaSuccess) return e;
  if ((e = prof_after(st)) != cudaSuccess) return e;

  cfg.gridDim = dim3(a.n_rows, a.L.n_q);
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  if (a.L.rot)
    e = a.sk_ctas > 0 ? cudaLaunchKernelEx(&cfg, combine_sk_kernel<D, true>, a)
                      : cudaLaunchKernelEx(&cfg, combine_kernel<D, true>, a);
  else
    e = a.sk_ctas > 0 ? cudaLaunchKernelEx(&cfg, combine_sk_kernel<D, false>, a)
                      : cudaLaunchKernelEx(&cfg, combine_kernel<D, false>, a);
  return e;
}

template <int D>
cudaError_t launch_decode_t(const DecodeArgs& a, const RopeFreqs& f, cudaStream_t st) {
  static_assert(D % 64 == 0, "");
  static_assert(ring_slots(D, 8, decode_smem_bytes<D>()) >= 2 && ring_slots(D, 4, decode_smem_bytes<D>()) >= 2,
                "the pipeline needs at least two stages");
  static_assert(ring_slots(D, 8, decode_smem_bytes<D>() - sk_plan_bytes(kSkMaxRows)) >= 2,
                "the stream-K plan leaves two stages");
  cudaError_t e;
  if ((e = decode_attrs<D>(decode_smem_bytes<D>())) != cudaSuccess) return e;
  int hpb = 1, nblk = 1;
  qprep_shape<D>(a.L.n_q, hpb, nblk);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_rows, nblk);
  cfg.blockDim = dim3(hpb * Qp<D>::TH);
  cfg.dynamicSmemBytes = a.L.rot ? (size_t)hpb * D * sizeof(double) : 0;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&cfg, qprep_kernel<D>, a, f, hpb)) != cudaSuccess) return e;
  return launch_read_merge_t<D>(a, st);
}

template <int D>
cudaError_t launch_decode_append_t(const DecodeArgs& a, const AppendArgs& ap, const RopeFreqs& f, cudaStream_t st) {
  cudaError_t e;
  if ((e = decode_attrs<D>(decode_smem_bytes<D>())) != cudaSuccess) return e;
  int hpb = 1, nblk = 1;
  qprep_shape<D>(a.L.n_q, hpb, nblk);
  const int items = 2 * a.L.n_kv;
  const int ipb = std::min(items, App<D>::IPB);
  const int ablk = (items + ipb - 1) / ipb;
  const int per = std::max(hpb, ipb);            // Qp<D>::TH == App<D>::TH threads per head or item
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_rows, nblk + ablk);
  cfg.blockDim = dim3(per * Qp<D>::TH);
  cfg.dynamicSmemBytes = a.L.rot ? (size_t)per * D * sizeof(double) : 0;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&cfg, prep_append_kernel<D>, a, ap, f, hpb, nblk, ipb)) != cudaSuccess) return e;
  return launch_read_merge_t<D>(a, st);
}

// The grouped schedule: the same three kernels, each grid over every group.
template <int D>
cudaError_t launch_decode_grouped_t(const GroupedDecode& ga, const RopeFreqs& f, cudaStream_t st) {
  cudaError_t e;
  const int smem = decode_smem_bytes<D>();
  if ((e = decode_attrs<D>(smem)) != cudaSuccess) return e;
  const LayerArgs& L = ga.g[0].L;
  const int rows = ga.row_base[ga.n], ctas = ga.cta_base[ga.n];
  int hpb = 1, nblk = 1;
  qprep_shape<D>(L.n_q, hpb, nblk);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows, nblk);
  cfg.blockDim = dim3(hpb * Qp<D>::TH);
  cfg.dynamicSmemBytes = L.rot ? (size_t)hpb * D * sizeof(double) : 0;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&cfg, qprep_grouped_kernel<D>, ga, f, hpb)) != cudaSuccess) return e;

  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(Dec<D>::THREADS);
  cfg.dynamicSmemBytes = smem;
  e = L.rot ? cudaLaunchKernelEx(&cfg, decode_grouped_kernel<D, true>, ga, smem)
            : cudaLaunchKernelEx(&cfg, decode_grouped_kernel<D, false>, ga, smem);
  if (e != cudaSuccess) return e;

  cfg.gridDim = dim3(rows, L.n_q);
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  return L.rot ? cudaLaunchKernelEx(&cfg, combine_grouped_kernel<D, true>, ga)
               : cudaLaunchKernelEx(&cfg, combine_grouped_kernel<D, false>, ga);
}

}  // namespace

size_t decode_ws_bytes(int n_rows, int n_kv, int D, const DecodePlan& plan) {
  const size_t NG = D / 64, B = (size_t)n_rows * n_kv;
  // partial pieces: per (row, kv head, split), or two per stream-K CTA
  const size_t pieces = plan.sk_ctas > 0 ? (size_t)plan.sk_ctas * 2 : B * plan.splits;
  size_t off = 256;
  off += B * NG * 4 * 32 * 16;                 // qfrag
  off += B * 32 * 16;                          // qbias
  off = (off + 255) & ~size_t(255);
  off += pieces * 16 * (size_t)D * 4;          // part_o
  off += pieces * 32 * 4;                      // part_ml
  off += ((size_t)n_rows + 3) * 8;             // plan
  return off;
}

DecodeWs decode_ws_carve(void* base, int n_rows, int n_kv, int D, const DecodePlan& plan) {
  const size_t NG = D / 64, B = (size_t)n_rows * n_kv;
  const size_t pieces = plan.sk_ctas > 0 ? (size_t)plan.sk_ctas * 2 : B * plan.splits;
  uint8_t* p = static_cast<uint8_t*>(base);
  DecodeWs w = {};
  w.status = reinterpret_cast<uint32_t*>(p);
  size_t off = 256;
  w.qfrag = reinterpret_cast<uint4*>(p + off);
  off += B * NG * 4 * 32 * 16;
  w.qbias = reinterpret_cast<uint4*>(p + off);
  off += B * 32 * 16;
  off = (off + 255) & ~size_t(255);
  w.part_o = reinterpret_cast<float*>(p + off);
  off += pieces * 16 * (size_t)D * 4;
  w.part_ml = reinterpret_cast<float*>(p + off);
  off += pieces * 32 * 4;
  w.plan = reinterpret_cast<long long*>(p + off);
  return w;
}

namespace {
// The attention kernels' bounded wait, alone: an mbarrier expecting one
// arrival that never comes.  No copy is in flight, so returning is safe.
__global__ void __launch_bounds__(32) wait_selftest_kernel(uint32_t* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const bool ok = mbar_wait_for(&bar, 0, limit_ns);
  if (!ok && threadIdx.x == 0) flag_error(status, KVQ_DEV_TIMEOUT);
}
}  // namespace

cudaError_t launch_wait_selftest(uint32_t* status, unsigned long long limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

DecodePlan decode_plan(const LayerArgs& L, int n_rows, int max_keys, int num_sms, bool fixed_chunks) {
  // tiles one row can touch: keys 0..max_keys-1 when causal, else a window
  // of at most `window` keys starting anywhere inside a tile
  const long full_tiles = ((long)std::max(max_keys, 1) - 1) / kTileKeys + 1;
  const int tiles = int(L.window > 0 ? std::min<long>(full_tiles, (L.window + kTileKeys - 2) / kTileKeys + 1)
                                     : full_tiles);
  const int per_sm = L.D >= 512 ? 1 : (L.D == 256 ? 2 : 4);
  const long base = std::max<long>((long)n_rows * L.n_kv, 1);
  const long wave = std::max<long>(1, ((long)num_sms * per_sm) / base);   // splits that still fit one wave
  DecodePlan plan;
  plan.sk_ctas = 0;
  if (fixed_chunks && n_rows <= kSkMaxRows && tiles > kChunkTiles) {
    // long rows: stream-K over one wave of CTAs
    plan.sk_ctas = std::max(1, std::min(1024, num_sms * per_sm));
    plan.splits = 1;
    plan.chunk_tiles = 0;
  } else if (fixed_chunks) {
    // every split takes the same number of tiles: rows shorter than the
    // longest use fewer splits and their surplus CTAs exit at once, so ragged
    // batches balance through the block scheduler
    long splits = std::max<long>(wave, (tiles + kChunkTiles - 1) / kChunkTiles);
    splits = std::max<long>(1, std::min<long>(splits, 256));
    const int chunk = int((tiles + splits - 1) / splits);
    plan.chunk_tiles = chunk;
    plan.splits = (tiles + chunk - 1) / chunk;
  } else {
    long splits = std::min<long>(wave, std::max(1, tiles / 2));
    plan.splits = int(std::max<long>(1, std::min<long>(splits, 256)));
    plan.chunk_tiles = 0;                                   // per row: ceil(row tiles / splits)
  }
  return plan;
}

void decode_plan_grouped(const LayerArgs& L, int n, const int* rows, const int* max_keys, const bool* fixed_chunks,
                         const int* max_splits, int num_sms, DecodePlan* plans) {
  const int per_sm = L.D >= 512 ? 1 : (L.D == 256 ? 2 : 4);
  long base = 0;
  for (int g = 0; g < n; ++g) base += (long)rows[g] * L.n_kv;
  const long wave = std::max<long>(1, ((long)num_sms * per_sm) / std::max<long>(base, 1));
  for (int g = 0; g < n; ++g) {
    const long full_tiles = ((long)std::max(max_keys[g], 1) - 1) / kTileKeys + 1;
    const int tiles = int(L.window > 0 ? std::min<long>(full_tiles, (L.window + kTileKeys - 2) / kTileKeys + 1)
                                       : full_tiles);
    DecodePlan& p = plans[g];
    p.sk_ctas = 0;
    const long cap = std::max(1, std::min(max_splits[g], 256));
    if (fixed_chunks[g]) {
      long splits = std::max<long>(wave, (tiles + kChunkTiles - 1) / kChunkTiles);
      splits = std::max<long>(1, std::min<long>(splits, cap));
      const int chunk = int((tiles + splits - 1) / splits);
      p.chunk_tiles = chunk;
      p.splits = (tiles + chunk - 1) / chunk;
    } else {
      p.splits = int(std::max<long>(1, std::min<long>(std::min<long>(wave, std::max(1, tiles / 2)), cap)));
      p.chunk_tiles = 0;
    }
  }
}

int decode_max_splits(int n_rows, int n_kv, int D, size_t bytes) {
  const DecodePlan one{1, 0, 0};
  const size_t fixed = decode_ws_bytes(n_rows, n_kv, D, one) - (size_t)n_rows * n_kv * (16 * (size_t)D * 4 + 32 * 4);
  if (bytes < fixed) return 0;
  const size_t per_split = (size_t)n_rows * n_kv * (16 * (size_t)D * 4 + 32 * 4);
  return (int)std::min<size_t>((bytes - fixed) / std::max<size_t>(per_split, 1), 256);
}

cudaError_t launch_decode_grouped(const GroupedDecode& ga, const RopeFreqs& f, cudaStream_t st) {
  if (ga.n < 1 || ga.row_base[ga.n] == 0) return cudaSuccess;
  switch (ga.g[0].L.D) {
    case 64: return launch_decode_grouped_t<64>(ga, f, st);
    case 128: return launch_decode_grouped_t<128>(ga, f, st);
    case 256: return launch_decode_grouped_t<256>(ga, f, st);
    case 512: return launch_decode_grouped_t<512>(ga, f, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_append(const DecodeArgs& a, const AppendArgs& ap, const RopeFreqs& f, cudaStream_t st) {
  if (a.n_rows == 0) return cudaSuccess;
  static_assert(Qp<64>::TH == App<64>::TH && Qp<512>::TH == App<512>::TH, "one block shape for both halves");
  switch (a.L.D) {
    case 64: return launch_decode_append_t<64>(a, ap, f, st);
    case 128: return launch_decode_append_t<128>(a, ap, f, st);
    case 256: return launch_decode_append_t<256>(a, ap, f, st);
    case 512: return launch_decode_append_t<512>(a, ap, f, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode(const DecodeArgs& a, const RopeFreqs& f, int /*num_sms*/, cudaStream_t st) {
  if (a.n_rows == 0) return cudaSuccess;
  // the status word is cleared by q prep, the first kernel of the call
  switch (a.L.D) {
    case 64: return launch_decode_t<64>(a, f, st);
    case 128: return launch_decode_t<128>(a, f, st);
    case 256: return launch_decode_t<256>(a, f, st);
    case 512: return launch_decode_t<512>(a, f, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
