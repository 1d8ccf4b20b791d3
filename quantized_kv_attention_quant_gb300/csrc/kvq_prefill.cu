// attn_prefill_chunk on the tensor cores (tcgen05): the rows of a prompt
// chunk attend the quantized cache (model.ts attentionTraining, prompt phase:
// qNorm, RoPE at the cache offset, read.attend(q, 1.0) under the causal +
// sliding-window mask; "Parity notes": SDPA scale 1.0, GQA).
//
// One CTA takes 128 query rows that share a kv head: 128/G consecutive tokens
// of one sequence times its G q heads (row r = token r / G, head r % G), with
// kNQ threads per row (warps w, w + 4, w + 8, ... reach the same
// tensor-memory lanes; each takes a 1/kNQ share of the row's keys and output
// dims).  It walks the keys its
// rows can see in 64-key tiles:
//   1. TMA bulk copies bring the tile's packed codes and bf16 scale/bias
//      blocks into a staging area (prefetched one tile ahead).
//   2. All threads turn the K codes into f16 integers (exact) and the V codes
//      into v_hat = scale * code + bias, one f16 fma (written transposed with
//      stmatrix so that keys run along the MMA's K).  V is converted while QK
//      runs and the next tile's K while PV runs.
//   3. One thread issues QK as one MMA chain per 64-dim group into tensor
//      memory (M = 128 rows, N = 64 keys): S = sum_g scale_g * (q_g . codes_g)
//      + sum_g bias_g * sum(q_g) keeps the QK product exact up to fp32
//      rounding, as on the decode path.
//   4. Each thread reads its row of the group products, forms the masked
//      scores, and P = e^(S - ref) as f16, where ref is the row's running max;
//      the output accumulator in tensor memory is rescaled only when a tile's
//      max exceeds ref by more than 8 (P <= e^8 stays well inside f16).
//   5. One thread issues PV (M = 128, N = head_dim, K = 64 keys) into the
//      output accumulator.
// The output is O / l per row.  All operands are K-major with the 128-byte
// swizzle; tensor memory holds the NG group products (64 columns each) and
// the output (head_dim columns).
#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "kvq_qprep.cuh"
#include "kvq_qrows.cuh"
#include "kvq_tc.cuh"

#include <algorithm>
#include <atomic>
#include <mutex>

namespace kvq {

namespace {

constexpr int kRows = 128;      // MMA rows per CTA
constexpr int kNQ = 4;                  // threads per row: warps w + 4i share tensor-memory lanes
constexpr int kThreads = kRows * kNQ;
constexpr int kKPT = 64 / kNQ;          // keys of a tile per thread

template <int D>
struct Pf {
  static constexpr int NG = D / 64;
  static constexpr int RB8 = D;                         // code bytes per key row at 8 bits (the larger case)
  static constexpr int SB = 64 * NG * 2;                // one 64 x NG bf16 block
  // byte offsets from the 1024-aligned base
  static constexpr int Q_OFF = 0;                       // NG blocks of [128 rows x 128 B]: q as f16
  static constexpr int K_OFF = Q_OFF + NG * 16384;      // NG blocks of [64 keys x 128 B]: K codes as f16
  static constexpr int V_OFF = K_OFF + NG * 8192;       // [D dims x 128 B]: v_hat as f16, 64 keys per row
  static constexpr int P_OFF = V_OFF + D * 128;         // [128 rows x 128 B]: P as f16
  static constexpr int S_OFF = P_OFF + 16384;           // staging: K codes, V codes, 4 scale/bias blocks
  static constexpr int STAGE = 2 * 64 * RB8 + 4 * SB;
  static constexpr int T_OFF = S_OFF + STAGE;           // K scale, K bias as f32 [2][NG][64]
  static constexpr int X_OFF = T_OFF + 2 * 64 * NG * 4; // row exchange between a row's threads [kNQ][128] f32
  static constexpr int C_OFF = X_OFF + kNQ * 128 * 4;   // 3 mbarriers and the tensor-memory address
  static constexpr int BYTES = C_OFF + 64 + 1024;       // + room to align the base
  static constexpr int TMEM_COLS = 2 * D;               // group products (NG x 64) then the output (D)
};

__device__ __forceinline__ uint32_t h2_fma_u(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b), *reinterpret_cast<__half2*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t h2_sub_u(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
constexpr uint32_t kF16_1024 = 0x64006400u;            // (1024, 1024): OR-ing v < 1024 into the mantissa gives 1024 + v


template <int D, int BITS>
__device__ __forceinline__ void prefill_body(const DecodeArgs& a, uint8_t* sm, const kvq_seq_cache& c,
                                             const int s, const int kvh, const int t0, const int rows_s,
                                             const int start) {
  using P = Pf<D>;
  constexpr int NG = P::NG, SB = P::SB;
  constexpr int RB = D * BITS / 8;
  constexpr float L2E = 1.4426950408889634f;
  constexpr float kSlack = 8.f;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.L.G, TQ = kRows / G, W = a.L.window;
  uint64_t* bar_tma = reinterpret_cast<uint64_t*>(sm + P::C_OFF);
  uint64_t* bar_s = bar_tma + 1;
  uint64_t* bar_o = bar_tma + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + P::C_OFF + 24);
  float* xr = reinterpret_cast<float*>(sm + P::X_OFF);    // [kNQ][128] row exchange
  float* skf = reinterpret_cast<float*>(sm + P::T_OFF);   // [NG][64] K scale as f32
  float* bkf = skf + 64 * NG;                             // [NG][64] K bias as f32
  uint8_t* stg = sm + P::S_OFF;
  const uint8_t* stg_k = stg;
  const uint8_t* stg_v = stg + 64 * RB;
  const uint16_t* stg_ks = reinterpret_cast<const uint16_t*>(stg + 128 * RB);
  const uint16_t* stg_kb = stg_ks + 64 * NG;
  const uint16_t* stg_vs = stg_kb + 64 * NG;
  const uint16_t* stg_vb = stg_vs + 64 * NG;
  const uint32_t base = smem_u32(sm);

  // ---- this thread's row (share hf of its keys and output dims) and the CTA's key range ----
  const int r = 32 * (warp & 3) + lane, hf = warp >> 2;
  constexpr int DPT = D / kNQ;                            // output dims per thread
  const int tq = r / G, h = r % G;
  const int t = t0 + tq;
  const bool row_valid = t < rows_s;
  const int newest = start + rows_s - 1;
  const int cap = c.capacity;
  const int resident_lo = max(0, newest - cap + 1);      // older positions were overwritten
  const int p_r = start + t;
  const int lo_r = W > 0 ? max(0, p_r - W + 1) : 0;
  const bool row_nan = row_valid && lo_r < resident_lo;  // its window reaches an overwritten key
  const bool row_live = row_valid && !row_nan;
  const int p_first = start + t0, p_last = start + min(t0 + TQ, rows_s) - 1;
  const int k_lo = max(W > 0 ? max(0, p_first - W + 1) : 0, resident_lo);
  const int k_hi = p_last;
  const int tile_lo = k_lo / kTileKeys;
  const int n_tiles = k_lo <= k_hi ? k_hi / kTileKeys - tile_lo + 1 : 0;
  const int cap_tiles = cap / kTileKeys;
  const size_t head_row0 = (size_t)kvh * cap;
  const int hq = kvh * G + h;
  const size_t grow = (size_t)__ldg(a.row_offsets + s) + t;     // global query row
  const int kk0 = kKPT * hf;                              // this thread's keys of a tile
  const int dd0 = DPT * hf;                               // this thread's output dims

  // 16-byte stores when the output allows them (the API asks only for element alignment)
  const bool out_vec = (reinterpret_cast<uintptr_t>(a.out) & 15u) == 0;
  auto write_row = [&](const float* v, int d0) {          // 16 values at dims d0..d0+15
    const size_t oi = (grow * a.L.n_q + hq) * D + d0;
    if (!out_vec) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (a.out_f32) reinterpret_cast<float*>(a.out)[oi + i] = v[i];
        else reinterpret_cast<uint16_t*>(a.out)[oi + i] = f_to_bf16_rn(v[i]);
      }
    } else if (a.out_f32) {
      float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.out) + oi);
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = (uint32_t)f_to_bf16_rn(v[2 * i]) | ((uint32_t)f_to_bf16_rn(v[2 * i + 1]) << 16);
      uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + oi);
      o[0] = make_uint4(w[0], w[1], w[2], w[3]);
      o[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  };
  auto write_nan_half = [&]() {
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __int_as_float(0x7fc00000);
    for (int d0 = dd0; d0 < dd0 + DPT; d0 += 16) write_row(v, d0);
  };
  if (n_tiles == 0) {                                     // uniform over the CTA
    if (row_valid) write_nan_half();
    return;
  }

  // ---- setup: barriers, tensor memory, the first tile's copies, Q ----
  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, P::TMEM_COLS);
    tc::tmem_relinquish();
  }
  auto issue_tile = [&](int ti) {                         // thread 0
    const int slot_tile = (tile_lo + ti) % cap_tiles;
    const size_t r0 = head_row0 + (size_t)slot_tile * kTileKeys;
    mbar_arrive_expect_tx(bar_tma, 2 * 64 * RB + 4 * SB);
    bulk_g2s(stg, reinterpret_cast<const uint8_t*>(c.k_codes) + r0 * RB, 64 * RB, bar_tma);
    bulk_g2s(stg + 64 * RB, reinterpret_cast<const uint8_t*>(c.v_codes) + r0 * RB, 64 * RB, bar_tma);
    bulk_g2s(stg + 128 * RB, c.k_scales + r0 * NG, SB, bar_tma);
    bulk_g2s(stg + 128 * RB + SB, c.k_biases + r0 * NG, SB, bar_tma);
    bulk_g2s(stg + 128 * RB + 2 * SB, c.v_scales + r0 * NG, SB, bar_tma);
    bulk_g2s(stg + 128 * RB + 3 * SB, c.v_biases + r0 * NG, SB, bar_tma);
  };
  __syncthreads();                                        // barriers initialised, tensor memory address written
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  if (tid == 0) issue_tile(0);

  // Q rows as f16 (each thread a 1/kNQ share of its row's chunks).  With 4-bit codes
  // the K conversion yields the dims of each 8-dim chunk in the order
  // 0 4 1 5 2 6 3 7; Q uses the same order.
  {
    const uint4* src = reinterpret_cast<const uint4*>(a.ws.q16 + (grow * a.L.n_q + hq) * D);
#pragma unroll 4
#pragma unroll 1
    for (int ch = hf * (D / 8 / kNQ); ch < (hf + 1) * (D / 8 / kNQ); ++ch) {
      uint4 v = row_valid ? src[ch] : make_uint4(0u, 0u, 0u, 0u);
      if (BITS == 4)
        v = make_uint4(prmt(v.x, v.z, 0x5410u), prmt(v.x, v.z, 0x7632u), prmt(v.y, v.w, 0x5410u),
                       prmt(v.y, v.w, 0x7632u));
      *reinterpret_cast<uint4*>(sm + P::Q_OFF + (ch >> 3) * 16384 + tc::sw128_off(r, ch & 7)) = v;
    }
  }
  float qsum[NG];
#pragma unroll
  for (int g = 0; g < NG; ++g) qsum[g] = row_valid ? a.ws.qsum[(grow * a.L.n_q + hq) * NG + g] : 0.f;

  float m_ref = -INFINITY, l_part = 0.f;
  int ph_tma = 0, ph_s = 0, ph_o = 0;
  bool dead = false;
  auto wait = [&](uint64_t* bar, int& ph) {
    if (!dead && !mbar_wait(bar, ph)) {
      dead = true;
      flag_error(a.ws.status, KVQ_DEV_TIMEOUT);
    }
    ph ^= 1;
  };
  const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  constexpr uint32_t ID_QK = tc::idesc_f16_f32(128, 64);
  constexpr uint32_t ID_PV = tc::idesc_f16_f32(128, D);

  // K codes of the staged tile -> f16 integers; K scale/bias -> f32 tables
  auto convert_k = [&]() {
#pragma unroll 1
    for (int i = tid; i < 64 * D / 8; i += kThreads) {
      const int key = i / (D / 8), ch = i % (D / 8);
      uint4 o;
      if constexpr (BITS == 4) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(stg_k + key * RB + ch * 4);
        o.x = h2_sub_u((w & 0x000F000Fu) | kF16_1024, kF16_1024);
        o.y = h2_sub_u(((w >> 4) & 0x000F000Fu) | kF16_1024, kF16_1024);
        o.z = h2_sub_u(((w >> 8) & 0x000F000Fu) | kF16_1024, kF16_1024);
        o.w = h2_sub_u(((w >> 12) & 0x000F000Fu) | kF16_1024, kF16_1024);
      } else {
        const uint2 w = *reinterpret_cast<const uint2*>(stg_k + key * RB + ch * 8);
        o.x = h2_sub_u(prmt(w.x, 0x64646464u, 0x4140u), kF16_1024);
        o.y = h2_sub_u(prmt(w.x, 0x64646464u, 0x4342u), kF16_1024);
        o.z = h2_sub_u(prmt(w.y, 0x64646464u, 0x4140u), kF16_1024);
        o.w = h2_sub_u(prmt(w.y, 0x64646464u, 0x4342u), kF16_1024);
      }
      *reinterpret_cast<uint4*>(sm + P::K_OFF + (ch >> 3) * 8192 + tc::sw128_off(key, ch & 7)) = o;
    }
    for (int i = tid; i < 64 * NG; i += kThreads) {       // [key][g] -> [g][key]
      const int key = i / NG, g = i % NG;
      skf[g * 64 + key] = bf16_to_f(stg_ks[i]);
      bkf[g * 64 + key] = bf16_to_f(stg_kb[i]);
    }
  };
  // V of the staged tile: v_hat = scale * code + bias (one f16 fma), stored
  // transposed (row = dim, 64 keys per row); keys outside the CTA's range are zero
  auto convert_v = [&](int tpos0) {
    for (int task = warp; task < 8 * (D / 32); task += kThreads / 32) {
      const int kb = task & 7, db = task >> 3;
      const int key = 8 * kb + (lane >> 2);
      const int g = db >> 1;
      const int kp = tpos0 + key;
      const bool in = kp >= k_lo && kp <= k_hi;
      const float sc = in ? bf16_to_f(stg_vs[key * NG + g]) : 0.f;
      const float bi = in ? bf16_to_f(stg_vb[key * NG + g]) : 0.f;
      const uint32_t s2 = pack_h2(sc, sc), b2 = pack_h2(bi, bi);
      // each lane loads its key's dims 32 db + 8 (lane & 3) .. +7 (one load per
      // lane); the pair a fragment needs comes from a neighbour by shuffle
      uint32_t rr[4];
      if constexpr (BITS == 4) {
        const uint32_t mine = *reinterpret_cast<const uint32_t*>(stg_v + key * RB + 16 * db + 4 * (lane & 3));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w = __shfl_sync(0xffffffffu, mine, (lane & ~3) + j);   // dims 32 db + 8 j .. +7
          const uint32_t b = (w >> (8 * (lane & 3))) & 0xFFu;                   // dims + 2 (lane & 3), +1
          const uint32_t cp = (b & 0xFu) | ((b & 0xF0u) << 12) | kF16_1024;
          rr[j] = h2_fma_u(h2_sub_u(cp, kF16_1024), s2, b2);
        }
      } else {
        const uint2 mine = *reinterpret_cast<const uint2*>(stg_v + key * RB + 32 * db + 8 * (lane & 3));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t wx = __shfl_sync(0xffffffffu, mine.x, (lane & ~3) + j);
          const uint32_t wy = __shfl_sync(0xffffffffu, mine.y, (lane & ~3) + j);
          const uint32_t w = (lane & 2) ? wy : wx;
          const uint32_t cp = prmt(w >> (16 * (lane & 1)), 0x64646464u, 0x4140u);
          rr[j] = h2_fma_u(h2_sub_u(cp, kF16_1024), s2, b2);
        }
      }
      const int dim = 32 * db + 8 * (lane >> 3) + (lane & 7);
      tc::stmatrix_x4_trans(base + P::V_OFF + tc::sw128_off(dim, kb), rr[0], rr[1], rr[2], rr[3]);
    }
  };

  // prologue: K of tile 0
  wait(bar_tma, ph_tma);
  convert_k();
  for (int ti = 0; ti < n_tiles; ++ti) {
    const int tpos0 = (tile_lo + ti) * kTileKeys;
    fence_proxy_async();
    __syncthreads();                                      // K(ti) and Q written
    if (tid == 0) {
      tc::fence_after_sync();
#pragma unroll
      for (int g = 0; g < NG; ++g)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_f16(tmem + g * 64, tc::desc_kmajor_sw128(base + P::Q_OFF + g * 16384 + 32 * k, 1024),
                      tc::desc_kmajor_sw128(base + P::K_OFF + g * 8192 + 32 * k, 1024), ID_QK, k > 0);
      tc::commit(bar_s);
    }
    // V(ti) while QK(ti) runs; its buffer is free once PV(ti-1) is done
    if (ti > 0) {
      wait(bar_o, ph_o);
      tc::fence_after_sync();
    }
    convert_v(tpos0);
    fence_proxy_async();
    __syncthreads();                                      // staging read completely: prefetch the next tile
    if (tid == 0 && ti + 1 < n_tiles) issue_tile(ti + 1);
    wait(bar_s, ph_s);
    tc::fence_after_sync();

    // ---- scores of this thread's kKPT keys ----
    float S[kKPT];
#pragma unroll
    for (int q4 = 0; q4 < kKPT / 4; ++q4) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const float4 b4 = *reinterpret_cast<const float4*>(bkf + g * 64 + kk0 + 4 * q4);
        acc.x = fmaf(b4.x, qsum[g], acc.x); acc.y = fmaf(b4.y, qsum[g], acc.y);
        acc.z = fmaf(b4.z, qsum[g], acc.z); acc.w = fmaf(b4.w, qsum[g], acc.w);
      }
      S[4 * q4] = acc.x; S[4 * q4 + 1] = acc.y; S[4 * q4 + 2] = acc.z; S[4 * q4 + 3] = acc.w;
    }
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      float v[kKPT / 16][16];
#pragma unroll
      for (int u = 0; u < kKPT / 16; ++u) tc::ld_x16(lane_base + g * 64 + kk0 + 16 * u, v[u]);
      tc::wait_ld();
#pragma unroll
      for (int q4 = 0; q4 < kKPT / 4; ++q4) {
        const float4 s4 = *reinterpret_cast<const float4*>(skf + g * 64 + kk0 + 4 * q4);
        const float* vv = &v[q4 >> 2][4 * (q4 & 3)];
        S[4 * q4] = fmaf(s4.x, vv[0], S[4 * q4]);
        S[4 * q4 + 1] = fmaf(s4.y, vv[1], S[4 * q4 + 1]);
        S[4 * q4 + 2] = fmaf(s4.z, vv[2], S[4 * q4 + 2]);
        S[4 * q4 + 3] = fmaf(s4.w, vv[3], S[4 * q4 + 3]);
      }
    }
    float mt = -INFINITY;
    // keys outside a row's window: only where the thread's keys are not all
    // visible to every row of the warp (interior tiles skip the masks)
    if (__all_sync(0xffffffffu, row_live && tpos0 + kk0 >= lo_r && tpos0 + kk0 + kKPT - 1 <= p_r)) {
#pragma unroll
      for (int j = 0; j < kKPT; ++j) mt = fmaxf(mt, S[j]);
    } else {
#pragma unroll
      for (int j = 0; j < kKPT; ++j) {
        const int kp = tpos0 + kk0 + j;
        S[j] = (row_live && kp >= lo_r && kp <= p_r) ? S[j] : -INFINITY;
        mt = fmaxf(mt, S[j]);
      }
    }
    xr[hf * 128 + r] = mt;
    __syncthreads();                                      // row maxima of every share
#pragma unroll
    for (int i = 1; i < kNQ; ++i) mt = fmaxf(mt, xr[((hf + i) % kNQ) * 128 + r]);
    // a new reference for this row; its output row is rescaled unless it had
    // no visible key before (tensor-memory loads and stores are warp-wide:
    // the whole warp takes part, with factor 1 for rows that keep theirs)
    const bool renew = mt > m_ref + kSlack;
    const bool rescale_o = renew && m_ref != -INFINITY;
    const float alpha = rescale_o ? exp2f((m_ref - mt) * L2E) : 1.f;
    if (renew) {
      l_part *= alpha;
      m_ref = mt;
    }
    if (__any_sync(0xffffffffu, rescale_o)) {
      for (int cc = 0; cc < DPT / 16; ++cc) {
        float v[16];
        tc::ld_x16(lane_base + D + dd0 + 16 * cc, v);
        tc::wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] *= alpha;
        tc::st_x16(lane_base + D + dd0 + 16 * cc, v);
      }
      tc::wait_st();
    }
    // ---- P = e^(S - ref) as f16 ----
#pragma unroll
    for (int ch = 0; ch < kKPT / 8; ++ch) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 8 * ch + 2 * e;
        float p0 = 0.f, p1 = 0.f;
        if (m_ref != -INFINITY) {
          p0 = exp2f((S[j] - m_ref) * L2E);
          p1 = exp2f((S[j + 1] - m_ref) * L2E);
        }
        const __half2 hp = __floats2half2_rn(p0, p1);
        const float2 pf = __half22float2(hp);
        l_part += pf.x + pf.y;
        w[e] = *reinterpret_cast<const uint32_t*>(&hp);
      }
      *reinterpret_cast<uint4*>(sm + P::P_OFF + tc::sw128_off(r, (kKPT / 8) * hf + ch)) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
    fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();                                      // P written, group products read, output rescaled
    if (tid == 0) {
      tc::fence_after_sync();
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tc::mma_f16(tmem + D, tc::desc_kmajor_sw128(base + P::P_OFF + 32 * k, 1024),
                    tc::desc_kmajor_sw128(base + P::V_OFF + 32 * k, 1024), ID_PV, ti > 0 || k > 0);
      tc::commit(bar_o);
    }
    // K(ti+1) while PV(ti) runs (QK(ti) is done, its tables were read above)
    if (ti + 1 < n_tiles) {
      wait(bar_tma, ph_tma);
      convert_k();
    }
  }
  wait(bar_o, ph_o);                                      // the last PV
  tc::fence_after_sync();

  // ---- output: O / l, each thread a 1/kNQ share of its row's dims ----
  xr[hf * 128 + r] = l_part;
  __syncthreads();
  float l_row = l_part;
#pragma unroll
  for (int i = 1; i < kNQ; ++i) l_row += xr[((hf + i) % kNQ) * 128 + r];
  const float inv = 1.f / l_row;
  for (int cc = 0; cc < DPT / 16; ++cc) {
    float v[16];
    tc::ld_x16(lane_base + D + dd0 + 16 * cc, v);
    tc::wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] *= inv;
    if (row_live) write_row(v, dd0 + 16 * cc);
  }
  if (row_nan) write_nan_half();
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, P::TMEM_COLS);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int qb = blockIdx.x, s = blockIdx.y, kvh = blockIdx.z;
  const int G = a.L.G, TQ = kRows / G;
  const int off0 = __ldg(a.row_offsets + s), off1 = __ldg(a.row_offsets + s + 1);
  const int rows_s = off1 - off0;
  const int t0 = qb * TQ;
  if (t0 >= rows_s) return;
  const int start = __ldg(a.pos + s);
  const kvq_seq_cache c = a.seqs[s];
  const bool ok = seq_ok(c) && start >= 0 && start + rows_s - 1 < (1 << 24);
  if (!ok) {
    if (qb == 0 && kvh == 0 && threadIdx.x == 0) flag_error(a.ws.status, KVQ_DEV_BADSEQ);
    const int r = threadIdx.x, t = t0 + r / G;
    if (r < kRows && t < rows_s) {
      const size_t oi = (((size_t)off0 + t) * a.L.n_q + kvh * G + r % G) * D;
      for (int d = 0; d < D; ++d) {
        if (a.out_f32) reinterpret_cast<float*>(a.out)[oi + d] = __int_as_float(0x7fc00000);
        else reinterpret_cast<uint16_t*>(a.out)[oi + d] = 0x7fc0;
      }
    }
    return;
  }
  if (c.bits == 4) prefill_body<D, 4>(a, sm, c, s, kvh, t0, rows_s, start);
  else prefill_body<D, 8>(a, sm, c, s, kvh, t0, rows_s, start);
}

template <int D>
cudaError_t launch_prefill_t(const DecodeArgs& a, const RopeFreqs& f, int max_rows, cudaStream_t st,
                             const AppendArgs* ap) {
  cudaError_t e;
  constexpr int smem = Pf<D>::BYTES;
  static_assert(smem <= 227 * 1024, "shared memory");
  // the shared-memory opt-in, once per device (a lock: host threads may make
  // their first call on a device at the same time)
  static std::atomic<bool> attr_set[64];
  static std::mutex attr_mu;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(attr_mu);
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
      // at most 512 / (2 D) CTAs may share an SM's tensor memory: ask for
      // enough shared memory that no more fit
      const int per_sm = 512 / Pf<D>::TMEM_COLS;
      const int want = per_sm >= 3 ? smem : std::max(smem, (228 * 1024) / (per_sm + 1) + 1024);
      e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
      if (e != cudaSuccess) return e;
      attr_set[dev].store(true, std::memory_order_release);
    }
  }
  const int per_sm = 512 / Pf<D>::TMEM_COLS;
  const int launch_smem = per_sm >= 3 ? smem : std::max(smem, (228 * 1024) / (per_sm + 1) + 1024);
  if ((e = launch_qprep_rows<D>(a, f, st, ap)) != cudaSuccess) return e;
  const int TQ = kRows / a.L.G;
  if (a.n_seqs > 65535 || a.L.n_kv > 65535) return cudaErrorInvalidValue;
  const dim3 grid((max_rows + TQ - 1) / TQ, a.n_seqs, a.L.n_kv);
  if ((e = prof_before(st)) != cudaSuccess) return e;
  prefill_tc_kernel<D><<<grid, kThreads, launch_smem, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return prof_after(st);
}

}  // namespace

bool prefill_tc_supported(const LayerArgs& L) {
  // (a rotated layer takes the row path, whose merge un-rotates the output)
  return (L.D == 64 || L.D == 128 || L.D == 256) && L.G >= 1 && L.G <= kMaxG && (kRows % L.G) == 0 &&
         L.rot == nullptr;
}

size_t prefill_tc_ws_bytes(int n_rows, const LayerArgs& L) {
  size_t off = 256;
  off += (size_t)n_rows * L.n_q * L.D * 2;                 // q16
  off = (off + 255) & ~size_t(255);
  off += (size_t)n_rows * L.n_q * (L.D / 64) * 4;          // qsum
  return off;
}

DecodeWs prefill_tc_ws_carve(void* base, int n_rows, const LayerArgs& L) {
  uint8_t* p = static_cast<uint8_t*>(base);
  DecodeWs w = {};
  w.status = reinterpret_cast<uint32_t*>(p);
  size_t off = 256;
  w.q16 = reinterpret_cast<uint16_t*>(p + off);
  off += (size_t)n_rows * L.n_q * L.D * 2;
  off = (off + 255) & ~size_t(255);
  w.qsum = reinterpret_cast<float*>(p + off);
  return w;
}

cudaError_t launch_prefill_tc(const DecodeArgs& a, const RopeFreqs& f, int max_rows_per_seq, cudaStream_t st,
                              const AppendArgs* ap) {
  if (a.n_rows == 0) return cudaSuccess;
  // the status word is cleared by q prep, the first kernel of the call
  switch (a.L.D) {
    case 64: return launch_prefill_t<64>(a, f, max_rows_per_seq, st, ap);
    case 128: return launch_prefill_t<128>(a, f, max_rows_per_seq, st, ap);
    case 256: return launch_prefill_t<256>(a, f, max_rows_per_seq, st, ap);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
