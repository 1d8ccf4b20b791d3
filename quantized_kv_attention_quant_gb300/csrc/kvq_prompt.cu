// attn_prefill_chunk on sliding-window layers, tensor cores (tcgen05): the
// rows of a prompt chunk or verify window attend the quantized cache (model.ts
// attentionTraining, prompt phase: qNorm, RoPE at the cache offset,
// read.attend(q, 1.0) under the causal + sliding-window mask).
//
// Two steps after q prep:
//   1. Dequantization, once per key: the keys the chunk of a sequence can see
//      (its window before the first row through its last row, at most
//      window + rows - 1) are read from the ring and written in position order
//      to a scratch area of the workspace: k_hat = scale * code + bias in fp32
//      (one rounding), split into two f16 values k_hi + k_lo (the split is
//      exact to ~2^-22 relative), and v_hat = f16(scale * code + bias).
//   2. The read, one CTA per 128 (token, head) rows of a sequence and kv head:
//      the tensor memory accelerator brings q (f16), each 64-key tile's k_hi,
//      k_lo and V rows into shared memory in the 128-byte-swizzled K-major
//      layout the MMA reads; a dedicated MMA warp issues QK as two f16 MMA
//      chains (q k_hi + q k_lo, fp32 accumulation) into one of two score slots
//      of tensor memory, and PV (A = P from tensor memory, B = V^T); 16
//      softmax warps (four threads per row) mask, exchange the row maxima
//      through tensor memory, write P as f16 and transpose the V tile.
// The k_hi / k_lo split keeps the scores within ~2^-22 of the exact dot
// products of the dequantized values (the decode path multiplies the codes
// exactly); PV multiplies the same f16 v_hat as the decode-path row kernel of
// the prompt path did.  Every key tile is dequantized once instead of once
// per 128-row CTA that reads it.
#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "kvq_prompt.h"
#include "kvq_qprep.cuh"
#include "kvq_qrows.cuh"
#include "kvq_tc.cuh"
#include "kvq_tma.cuh"

#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <mutex>

namespace kvq {

namespace {

constexpr int kRows = 128;              // MMA rows per CTA
constexpr int kNQ = 4;                  // threads per row
constexpr int kThreads = kRows * kNQ;   // softmax threads; + one MMA warp
constexpr int kKPT = 64 / kNQ;          // keys of a tile per thread

template <int D>
struct Pr {
  static constexpr int NG = D / 64;                     // 64-dim groups
  static constexpr int KB = D <= 128 ? 2 : 1;           // K buffers (hi and lo each)
  static constexpr int KBYTES = 2 * NG * 8192;          // one K buffer: hi then lo, NG blocks [64 keys x 128 B] each
  // byte offsets from the 1024-aligned base
  static constexpr int Q_OFF = 0;                       // NG blocks [128 rows x 128 B]: q as f16
  static constexpr int K_OFF = Q_OFF + NG * 16384;
  static constexpr int V_OFF = K_OFF + KB * KBYTES;     // [D dims x 128 B]: V^T as f16
  static constexpr int VS_OFF = V_OFF + NG * 8192;      // stage: NG blocks [64 keys x 128 B] of V (f16)
  static constexpr int C_OFF = VS_OFF + NG * 8192;      // mbarriers, tensor-memory address
  static constexpr int BYTES = C_OFF + 128 + 1024;
  // tensor-memory columns
  static constexpr int C_O = 0;                         // output accumulator, D columns
  static constexpr int C_S = D;                         // two score slots of 64 columns
  static constexpr int C_P = D + 128;                   // P as f16 pairs, 32 columns
  static constexpr int C_X = D + 160;                   // row exchange
  static constexpr int TMEM_COLS = C_X + kNQ <= 256 ? 256 : 512;
};

// keys per sequence in the scratch area: the window before the first row of
// the chunk through its last row, in whole tiles
inline int prompt_scratch_keys(int window, int max_rows) {
  return ((window + max_rows - 1 + kTileKeys - 1) / kTileKeys) * kTileKeys;
}

struct PromptArgs {
  LayerArgs L;
  const kvq_seq_cache* seqs;
  int n_seqs, n_rows;
  const int32_t* row_offsets;
  const int32_t* pos;
  void* out;
  int out_f32;
  int ks;               // scratch keys per sequence
  uint32_t* status;
  uint16_t* k_hi;       // scratch [n_seqs * ks][n_kv][D] f16
  uint16_t* k_lo;
  uint16_t* v;
};

// ---------------------------------------------------------------------------
// 1. dequantization into the scratch area
// ---------------------------------------------------------------------------
constexpr int kDqKeys = 16;             // keys per block of the dequantization

// Scratch rows bx * kDqKeys .. + kDqKeys - 1 of sequence s, kv head kvh.
// appended: the call's append writes the rows of its own stored positions
// (the chunk's rows a later row of the chunk does not overwrite) in the same
// grid, so only the older keys are read here; they sit in ring slots the
// append does not write.
template <int D>
__device__ __forceinline__ void prompt_dequant_block(const PromptArgs& a, const int bx, const int s, const int kvh,
                                                     const bool appended) {
  constexpr int NG = D / 64;
  const kvq_seq_cache c = a.seqs[s];
  const int off0 = __ldg(a.row_offsets + s), off1 = __ldg(a.row_offsets + s + 1);
  const int rows_s = off1 - off0;
  const int start = __ldg(a.pos + s), W = a.L.window;
  // an invalid descriptor (the read flags it and writes NaN) or no rows: the
  // slot is only zero-filled
  const bool live = seq_ok(c) && rows_s > 0 && start >= 0 && start + rows_s - 1 < (1 << 24);
  const int newest = start + rows_s - 1;
  const int kbase = live ? max(0, start - W + 1) : 0;
  const int klo = live ? max(kbase, newest - c.capacity + 1) : 1;   // older positions were overwritten
  const int khi = live ? newest : 0;
  const int RW = D * c.bits / 32;                         // code words per cache row
  // one thread per (key, 8-dim chunk) of this block's kDqKeys keys.  Every
  // scratch row of the slot is written: rows no key fills are zeros, so that
  // the tiles that reach them (masked out of the scores) multiply finite values
  for (int i = threadIdx.x; i < kDqKeys * (D / 8); i += blockDim.x) {
    const int key = i / (D / 8), ch = i % (D / 8), g = ch / 8;
    const int q = bx * kDqKeys + key;                     // scratch row in the slot
    const int p = kbase + q;
    const size_t o = (((size_t)s * a.ks + q) * a.L.n_kv + kvh) * D + ch * 8;
    if (appended && p >= start && p >= klo && p <= khi) continue;   // the append's row
    if (p < klo || p > khi) {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(a.k_hi + o) = z;
      *reinterpret_cast<uint4*>(a.k_lo + o) = z;
      *reinterpret_cast<uint4*>(a.v + o) = z;
      continue;
    }
    const size_t crow = (size_t)kvh * c.capacity + (p % c.capacity);
    uint32_t kc[8], vc[8];
    if (c.bits == 4) {
      const uint32_t wk = c.k_codes[crow * RW + ch], wv = c.v_codes[crow * RW + ch];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        kc[e] = (wk >> (4 * e)) & 0xFu;
        vc[e] = (wv >> (4 * e)) & 0xFu;
      }
    } else {
      const uint2 wk = reinterpret_cast<const uint2*>(c.k_codes + crow * RW)[ch];
      const uint2 wv = reinterpret_cast<const uint2*>(c.v_codes + crow * RW)[ch];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kc[e] = (wk.x >> (8 * e)) & 0xFFu;
        kc[e + 4] = (wk.y >> (8 * e)) & 0xFFu;
        vc[e] = (wv.x >> (8 * e)) & 0xFFu;
        vc[e + 4] = (wv.y >> (8 * e)) & 0xFFu;
      }
    }
    const float ks = bf16_to_f(c.k_scales[crow * NG + g]), kb = bf16_to_f(c.k_biases[crow * NG + g]);
    const float vs = bf16_to_f(c.v_scales[crow * NG + g]), vb = bf16_to_f(c.v_biases[crow * NG + g]);
    uint32_t hi[4], lo[4], vv[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const float k0 = __fmaf_rn(ks, (float)kc[e], kb), k1 = __fmaf_rn(ks, (float)kc[e + 1], kb);
      const __half2 h = __floats2half2_rn(k0, k1);
      const float2 hf = __half22float2(h);
      const __half2 l = __floats2half2_rn(k0 - hf.x, k1 - hf.y);          // exact differences
      const __half2 v = __floats2half2_rn(__fmaf_rn(vs, (float)vc[e], vb), __fmaf_rn(vs, (float)vc[e + 1], vb));
      hi[e / 2] = *reinterpret_cast<const uint32_t*>(&h);
      lo[e / 2] = *reinterpret_cast<const uint32_t*>(&l);
      vv[e / 2] = *reinterpret_cast<const uint32_t*>(&v);
    }
    *reinterpret_cast<uint4*>(a.k_hi + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(a.k_lo + o) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    *reinterpret_cast<uint4*>(a.v + o) = make_uint4(vv[0], vv[1], vv[2], vv[3]);
  }
}

// The read's first kernel: the q prep of the chunk's rows (blocks below nq),
// the call's K/V append (the next nap blocks, ablk per row, writing the
// appended rows' scratch too) and the dequantization of the scratch (the
// rest: slot blocks x sequences x kv heads), which share nothing.  (The
// dequantization blocks placed among the others, every other block index,
// made the prompt step slower: 0.093 -> 0.095 ms.)
template <int D, bool APPEND>
__global__ void __launch_bounds__(kQrWarps * 32, APPEND ? 5 : 1)
prompt_prep_kernel(const DecodeArgs a, const AppendArgs ap, const PromptArgs pa, const RopeFreqs freqs,
                   const int rb, const int nq, const int ipb, const int ablk, const int nap) {
  const int b = blockIdx.x;
  if (b < nq) {
    qprep_rows_block<D>(a, freqs, rb, b);
  } else if (APPEND && b < nq + nap) {
    append_block<D>(ap, freqs, ipb, (b - nq) / ablk, (b - nq) % ablk);
  } else {
    pdl_wait();                                           // (launched as a programmatic dependent)
    pdl_launch();
    const int x = b - nq - nap, nx = pa.ks / kDqKeys;
    prompt_dequant_block<D>(pa, x % nx, (x / nx) % pa.n_seqs, x / (nx * pa.n_seqs), APPEND);
  }
}

// ---------------------------------------------------------------------------
// 2. the read
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}
__device__ __forceinline__ void softmax_sync() { named_bar(1, kThreads); }

template <int D>
__global__ void __launch_bounds__(kThreads + 32, 1)
prompt_tc_kernel(const PromptArgs a, const __grid_constant__ CUtensorMap tmq,
                 const __grid_constant__ CUtensorMap tmkh, const __grid_constant__ CUtensorMap tmkl,
                 const __grid_constant__ CUtensorMap tmv) {
  using T = Pr<D>;
  constexpr int NG = T::NG, KB = T::KB;
  constexpr float L2E = 1.4426950408889634f;
  constexpr float kSlack = 8.f;
  constexpr float kHead = 6.f;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.L.G, TQ = kRows / G, W = a.L.window;
  const int s = blockIdx.y, kvh = blockIdx.z;
  const int off0 = __ldg(a.row_offsets + s), off1 = __ldg(a.row_offsets + s + 1);
  const int rows_s = off1 - off0;
  const int t0 = blockIdx.x * TQ;
  pdl_launch();                                           // the next call's first kernel waits for this grid
  if (t0 >= rows_s) return;
  const int start = __ldg(a.pos + s);
  const kvq_seq_cache c = a.seqs[s];
  const bool ok = seq_ok(c) && start >= 0 && start + rows_s - 1 < (1 << 24);
  constexpr int DPT = D / kNQ;                            // output dims per thread
  auto write_nan_rows = [&](bool only_nan_rows, auto is_nan) {
    if (tid >= kThreads) return;
    const int r = 32 * (warp & 3) + lane, hf = warp >> 2, t = t0 + r / G;
    if (t >= rows_s || (only_nan_rows && !is_nan(t))) return;
    const size_t oi = (((size_t)off0 + t) * a.L.n_q + kvh * G + r % G) * D + DPT * hf;
    for (int d = 0; d < DPT; ++d) {
      if (a.out_f32) reinterpret_cast<float*>(a.out)[oi + d] = __int_as_float(0x7fc00000);
      else reinterpret_cast<uint16_t*>(a.out)[oi + d] = 0x7fc0;
    }
  };
  if (!ok) {
    pdl_wait();                                           // the prep grid clears the status word
    if (t0 == 0 && kvh == 0 && tid == 0) flag_error(a.status, KVQ_DEV_BADSEQ);
    write_nan_rows(false, [](int) { return true; });
    return;
  }
  const int newest = start + rows_s - 1;
  const int resident_lo = max(0, newest - c.capacity + 1);   // older positions were overwritten
  const int kbase = max(0, start - W + 1);                    // scratch row 0 of the sequence
  const int p_first = start + t0, p_last = start + min(t0 + TQ, rows_s) - 1;
  const int k_lo = max(max(0, p_first - W + 1), resident_lo), k_hi = p_last;
  const int n_tiles = k_lo <= k_hi ? (k_hi - k_lo) / kTileKeys + 1 : 0;
  // a row whose window reaches an overwritten key returns NaN
  auto row_is_nan = [&](int t) { return max(0, start + t - W + 1) < resident_lo; };
  if (n_tiles == 0) {                                     // uniform: every row of the CTA is such a row
    write_nan_rows(false, [](int) { return true; });
    return;
  }

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + T::C_OFF);
  uint64_t* bar_q = bars;
  uint64_t* bar_k = bars + 1;
  uint64_t* bar_v = bars + 3;
  uint64_t* bar_s = bars + 4;
  uint64_t* bar_sfree = bars + 6;
  uint64_t* bar_pv = bars + 8;
  uint64_t* bar_o = bars + 9;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + T::C_OFF + 96);
  const uint32_t sbase = smem_u32(sm);
  const int srow0 = s * a.ks - kbase;                     // scratch row of position p: srow0 + p
  auto issue_k = [&](int i) {                             // one thread: k_hi and k_lo rows of tile i
    const int p0 = k_lo + kTileKeys * i;
    uint64_t* bk = bar_k + (i % KB);
    const uint32_t dst = sbase + T::K_OFF + (i % KB) * T::KBYTES;
    mbar_arrive_expect_tx(bk, 2 * NG * 8192);
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      tc::tma_load_3d(dst + g * 8192, &tmkh, 64 * g, kvh, srow0 + p0, smem_u32(bk));
      tc::tma_load_3d(dst + (NG + g) * 8192, &tmkl, 64 * g, kvh, srow0 + p0, smem_u32(bk));
    }
  };
  auto issue_v = [&](int i) {                             // one thread: V rows of tile i into the stage
    const int p0 = k_lo + kTileKeys * i;
    mbar_arrive_expect_tx(bar_v, NG * 8192);
#pragma unroll
    for (int g = 0; g < NG; ++g)
      tc::tma_load_3d(sbase + T::VS_OFF + g * 8192, &tmv, 64 * g, kvh, srow0 + p0, smem_u32(bar_v));
  };

  // ---- setup ----
  if (tid == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_k, 1);
    mbar_init(bar_k + 1, 1);
    mbar_init(bar_v, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_s + 1, 1);
    mbar_init(bar_sfree, kThreads / 32);
    mbar_init(bar_sfree + 1, kThreads / 32);
    mbar_init(bar_pv, 1);
    mbar_init(bar_o, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, T::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();                                        // barriers initialised, tensor memory address written
  tc::fence_after_sync();
  const uint32_t tmem = *tslot;
  // launched as a programmatic dependent of the prep grid: q, the scratch and
  // the status word are read or written only after it is complete
  pdl_wait();
  bool dead = false;
  auto wait = [&](uint64_t* bar, int parity) {
    if (!dead && !mbar_wait(bar, parity)) {
      dead = true;
      flag_error(a.status, KVQ_DEV_TIMEOUT);
    }
  };

  if (warp == kThreads / 32) {
    // ================= the MMA warp: copies of q and K, QK and PV =================
    const bool leader = lane == 0;
    constexpr uint32_t ID_QK = tc::idesc_f16_f32(128, 64);
    constexpr uint32_t ID_PV = tc::idesc_f16_f32(128, D);
    if (leader) {
      mbar_arrive_expect_tx(bar_q, NG * 16384);
#pragma unroll
      for (int g = 0; g < NG; ++g)
        tc::tma_load_3d(sbase + T::Q_OFF + g * 16384, &tmq, 64 * g, kvh * G, off0 + t0, smem_u32(bar_q));
      issue_k(0);
      if (KB == 2 && n_tiles > 1) issue_k(1);
    }
    __syncwarp();
    wait(bar_q, 0);
    auto issue_pv = [&](int i) {                          // P(i) and V^T(i) are ready
      wait(bar_pv, i & 1);
      tc::fence_after_sync();
      if (leader) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_f16_ts(tmem + T::C_O, tmem + T::C_P + 8 * k,
                         tc::desc_kmajor_sw128(sbase + T::V_OFF + 32 * k, 1024), ID_PV, i > 0 || k > 0);
        tc::commit(bar_o);
      }
      __syncwarp();
    };
    for (int ti = 0; ti < n_tiles; ++ti) {
      const int slot = ti & 1, kb = ti % KB;
      wait(bar_k + kb, (ti / KB) & 1);                    // K(ti) landed
      if (ti >= 2) wait(bar_sfree + slot, ((ti - 2) >> 1) & 1);   // scores of ti-2 read
      tc::fence_after_sync();
      if (leader) {
        const uint32_t kbuf = sbase + T::K_OFF + kb * T::KBYTES;
#pragma unroll
        for (int part = 0; part < 2; ++part)              // q k_hi, then q k_lo
#pragma unroll
          for (int g = 0; g < NG; ++g)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc::mma_f16(tmem + T::C_S + 64 * slot,
                          tc::desc_kmajor_sw128(sbase + T::Q_OFF + g * 16384 + 32 * k, 1024),
                          tc::desc_kmajor_sw128(kbuf + (part * NG + g) * 8192 + 32 * k, 1024), ID_QK,
                          (part | g | k) != 0);
        tc::commit(bar_s + slot);
      }
      __syncwarp();
      if (ti > 0) issue_pv(ti - 1);
      // K buffer kb is free once QK(ti) is done: the tile KB ahead goes there
      if (ti + KB < n_tiles) {
        wait(bar_s + slot, (ti >> 1) & 1);
        if (leader) issue_k(ti + KB);
        __syncwarp();
      }
    }
    issue_pv(n_tiles - 1);
  } else {
    // ================= the softmax warps =================
    const int r = 32 * (warp & 3) + lane, hf = warp >> 2;
    const int tq = r / G, h = r % G;
    const int t = t0 + tq;
    const bool row_valid = t < rows_s;
    const bool row_nan = row_valid && row_is_nan(t);
    const bool row_live = row_valid && !row_nan;
    const int p_r = start + t;
    const int lo_r = max(0, p_r - W + 1);
    const int hq = kvh * G + h;
    const int kk0 = kKPT * hf;
    const int dd0 = DPT * hf;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    if (tid == 0) issue_v(0);
    float m_ref = -INFINITY, l_part = 0.f;
    for (int ti = 0; ti < n_tiles; ++ti) {
      const int slot = ti & 1;
      const int kp0 = k_lo + kTileKeys * ti;
      wait(bar_s + slot, (ti >> 1) & 1);                  // QK(ti) done
      tc::fence_after_sync();
      __syncwarp();
      float S[kKPT];
      tc::ld_x16(lane_base + T::C_S + 64 * slot + kk0, S);
      tc::wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_sfree + slot);       // this warp's share of the slot is read
      const int kpk = kp0 + kk0;
      float mt = -INFINITY;
      if (__all_sync(0xffffffffu, row_live && kpk >= lo_r && kpk + kKPT - 1 <= p_r)) {
#pragma unroll
        for (int j = 0; j < kKPT; ++j) mt = fmaxf(mt, S[j]);
      } else {
#pragma unroll
        for (int j = 0; j < kKPT; ++j) {
          const bool vis = row_live && kpk + j >= lo_r && kpk + j <= p_r;
          S[j] = vis ? S[j] : -INFINITY;
          mt = fmaxf(mt, S[j]);
        }
      }
      // the row's maximum over its kNQ shares, through tensor memory
      tc::st_x1(lane_base + T::C_X + hf, mt);
      tc::wait_st();
      tc::fence_before_sync();
      softmax_sync();
      tc::fence_after_sync();
      {
        float xm[4];
        tc::ld_x4(lane_base + T::C_X, xm);
        tc::wait_ld();
        mt = fmaxf(fmaxf(xm[0], xm[1]), fmaxf(xm[2], xm[3]));
      }
      // a new reference sits kHead above the tile's maximum, so that a later
      // tile must exceed it by kSlack + kHead before the output is rescaled
      // again (P stays below e^kSlack, the largest P after a renewal is
      // e^-kHead, far from f16's limits at either end)
      const bool renew = mt > m_ref + kSlack;
      const bool rescale_o = renew && m_ref != -INFINITY;
      const float alpha = rescale_o ? exp2f((m_ref - (mt + kHead)) * L2E) : 1.f;
      if (renew) {
        l_part *= alpha;
        m_ref = mt + kHead;
      }
      // PV(ti-1) done: the output is settled, P and V^T are free
      if (ti > 0) {
        wait(bar_o, (ti - 1) & 1);
        tc::fence_after_sync();
        __syncwarp();
      }
      if (__any_sync(0xffffffffu, rescale_o)) {
        for (int cc = 0; cc < DPT / 16; ++cc) {
          float v[16];
          tc::ld_x16(lane_base + T::C_O + dd0 + 16 * cc, v);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] *= alpha;
          tc::st_x16(lane_base + T::C_O + dd0 + 16 * cc, v);
        }
      }
      // ---- P = e^(S - ref) as f16 pairs into tensor memory ----
      {
        uint32_t pw[kKPT / 2];
#pragma unroll
        for (int e = 0; e < kKPT / 2; ++e) {
          float p0 = 0.f, p1 = 0.f;
          if (m_ref != -INFINITY) {
            p0 = exp2f((S[2 * e] - m_ref) * L2E);
            p1 = exp2f((S[2 * e + 1] - m_ref) * L2E);
          }
          const __half2 hp = __floats2half2_rn(p0, p1);
          const float2 pf = __half22float2(hp);
          l_part += pf.x + pf.y;
          pw[e] = *reinterpret_cast<const uint32_t*>(&hp);
        }
        tc::st_x8(lane_base + T::C_P + (kKPT / 2) * hf, pw);
      }

      // ---- V(ti) -> V^T (both f16) ----
      wait(bar_v, ti & 1);
      __syncwarp();
      constexpr int QPK = D / 32;                         // groups of four 8x8 blocks per 8-key row
      uint32_t vr[NG][4];
#pragma unroll
      for (int i = 0; i < NG; ++i) {
        const int qd = warp * NG + i, kb8 = qd / QPK, db0 = 4 * (qd % QPK);
        const int dch = db0 + (lane >> 3);
        ldsm_x4(sbase + T::VS_OFF + (dch >> 3) * 8192 + tc::sw128_off(8 * kb8 + (lane & 7), dch & 7), vr[i]);
      }
#pragma unroll
      for (int i = 0; i < NG; ++i) {
        const int qd = warp * NG + i, kb8 = qd / QPK, db0 = 4 * (qd % QPK);
        const int dim = 8 * (db0 + (lane >> 3)) + (lane & 7);
        tc::stmatrix_x4_trans(sbase + T::V_OFF + tc::sw128_off(dim, kb8), vr[i][0], vr[i][1], vr[i][2], vr[i][3]);
      }
      fence_proxy_async();
      tc::wait_st();                                      // P and the rescaled output written
      tc::fence_before_sync();
      softmax_sync();
      if (tid == 0) {
        mbar_arrive(bar_pv);                              // PV(ti) may go
        if (ti + 1 < n_tiles) issue_v(ti + 1);            // the stage is read
      }
    }
    wait(bar_o, (n_tiles - 1) & 1);                       // the last PV
    tc::fence_after_sync();
    __syncwarp();

    // ---- output: O / l, each thread a quarter of its row's dims ----
    tc::st_x1(lane_base + T::C_X + hf, l_part);
    tc::wait_st();
    tc::fence_before_sync();
    softmax_sync();
    tc::fence_after_sync();
    float l_row;
    {
      float xl[4];
      tc::ld_x4(lane_base + T::C_X, xl);
      tc::wait_ld();
      l_row = (xl[0] + xl[1]) + (xl[2] + xl[3]);
    }
    const float inv = 1.f / l_row;
    const bool out_vec = (reinterpret_cast<uintptr_t>(a.out) & 15u) == 0;
    for (int cc = 0; cc < DPT / 16; ++cc) {
      float v[16];
      tc::ld_x16(lane_base + T::C_O + dd0 + 16 * cc, v);
      tc::wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = row_nan ? __int_as_float(0x7fc00000) : v[i] * inv;
      if (!row_valid) continue;
      const size_t oi = (((size_t)off0 + t) * a.L.n_q + hq) * D + dd0 + 16 * cc;
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
        for (int i = 0; i < 8; ++i)
          w[i] = (uint32_t)f_to_bf16_rn(v[2 * i]) | ((uint32_t)f_to_bf16_rn(v[2 * i + 1]) << 16);
        uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.out) + oi);
        o[0] = make_uint4(w[0], w[1], w[2], w[3]);
        o[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, T::TMEM_COLS);
  }
}

template <int D>
int prompt_launch_smem() {
  // at most 512 / TMEM_COLS CTAs may share an SM's tensor memory: ask for
  // enough shared memory that no more fit
  constexpr int smem = Pr<D>::BYTES;
  const int per_sm = 512 / Pr<D>::TMEM_COLS;
  return per_sm >= 3 ? smem : std::max(smem, (228 * 1024) / (per_sm + 1) + 1024);
}

struct PromptWs {
  uint32_t* status;
  uint16_t* q16;
  uint16_t *k_hi, *k_lo, *v;
  int ks;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

PromptWs prompt_ws_carve(void* base, int n_seqs, int n_rows, int max_rows, const LayerArgs& L) {
  uint8_t* p = static_cast<uint8_t*>(base);
  PromptWs w;
  w.ks = prompt_scratch_keys(L.window, max_rows);
  const size_t scratch = (size_t)n_seqs * w.ks * L.n_kv * L.D * 2;
  size_t off = 0;
  w.status = reinterpret_cast<uint32_t*>(p);
  off = 256;
  w.q16 = reinterpret_cast<uint16_t*>(p + off);
  off = align256(off + (size_t)n_rows * L.n_q * L.D * 2);
  w.k_hi = reinterpret_cast<uint16_t*>(p + off);
  off = align256(off + scratch);
  w.k_lo = reinterpret_cast<uint16_t*>(p + off);
  off = align256(off + scratch);
  w.v = reinterpret_cast<uint16_t*>(p + off);
  return w;
}

template <int D>
cudaError_t launch_prompt_t(const DecodeArgs& a, void* ws, int max_rows, const RopeFreqs& f, cudaStream_t st,
                            const AppendArgs* ap) {
  static_assert(Pr<D>::BYTES <= 227 * 1024, "shared memory");
  cudaError_t e;
  static std::atomic<bool> attr_set[64];
  static std::mutex attr_mu;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int smem = prompt_launch_smem<D>();
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(attr_mu);
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(prompt_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      attr_set[dev].store(true, std::memory_order_release);
    }
  }
  const LayerArgs& L = a.L;
  const PromptWs w = prompt_ws_carve(ws, a.n_seqs, a.n_rows, max_rows, L);
  const int TQ = kRows / L.G;
  const int srows = a.n_seqs * w.ks;
  CUtensorMap mq, mkh, mkl, mv;
  if (!rows_map(&mq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, w.q16, D, L.n_q, a.n_rows, L.G, TQ) ||
      !rows_map(&mkh, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, w.k_hi, D, L.n_kv, srows, 1, kTileKeys) ||
      !rows_map(&mkl, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, w.k_lo, D, L.n_kv, srows, 1, kTileKeys) ||
      !rows_map(&mv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, w.v, D, L.n_kv, srows, 1, kTileKeys))
    return cudaErrorInvalidValue;
  // q prep (q_hat as f16 rows; it also clears the status word), the append
  // and the dequantization in one grid
  DecodeArgs qa = a;
  qa.ws = DecodeWs{};
  qa.ws.status = w.status;
  qa.ws.q16 = w.q16;
  PromptArgs pa;
  pa.L = L;
  pa.seqs = a.seqs;
  pa.n_seqs = a.n_seqs;
  pa.n_rows = a.n_rows;
  pa.row_offsets = a.row_offsets;
  pa.pos = a.pos;
  pa.out = a.out;
  pa.out_f32 = a.out_f32;
  pa.ks = w.ks;
  pa.status = w.status;
  pa.k_hi = w.k_hi;
  pa.k_lo = w.k_lo;
  pa.v = w.v;
  if (a.n_seqs > 65535 || L.n_kv > 65535) return cudaErrorInvalidValue;
  AppendArgs apx = {};
  int ipb = 1, ablk = 1;
  long long nap = 0;
  if (ap && ap->n_rows > 0) {
    apx = *ap;
    apx.sk_hi = w.k_hi;
    apx.sk_lo = w.k_lo;
    apx.sv = w.v;
    apx.sks = w.ks;
    const int items = 2 * L.n_kv;
    ipb = std::min(items, kQrWarps * 32 / App<D>::TH);
    ablk = (items + ipb - 1) / ipb;
    nap = (long long)ap->n_rows * ablk;
  }
  const int rb = qprep_rows_rb(L);
  const long long nq = (a.n_rows + rb - 1) / rb;
  const long long ndq = (long long)(w.ks / kDqKeys) * a.n_seqs * L.n_kv;
  if (nq + nap + ndq > 0x7fffffffLL) return cudaErrorInvalidValue;
  e = nap > 0 ? launch_pdl(prompt_prep_kernel<D, true>, dim3((unsigned)(nq + nap + ndq)), dim3(kQrWarps * 32),
                           qprep_rows_smem(L, rb), st, qa, apx, pa, f, rb, (int)nq, ipb, ablk, (int)nap)
              : launch_pdl(prompt_prep_kernel<D, false>, dim3((unsigned)(nq + ndq)), dim3(kQrWarps * 32),
                           qprep_rows_smem(L, rb), st, qa, apx, pa, f, rb, (int)nq, ipb, ablk, 0);
  if (e != cudaSuccess) return e;
  const dim3 grid((max_rows + TQ - 1) / TQ, a.n_seqs, L.n_kv);
  if ((e = prof_before(st)) != cudaSuccess) return e;
  if ((e = launch_pdl(prompt_tc_kernel<D>, grid, dim3(kThreads + 32), (size_t)smem, st, pa, mq, mkh, mkl, mv)) !=
      cudaSuccess)
    return e;
  return prof_after(st);
}

}  // namespace

bool prompt_tc_supported(const LayerArgs& L) {
  return L.window > 0 && (L.D == 64 || L.D == 128 || L.D == 256) && L.G >= 1 && L.G <= kMaxG &&
         (kRows % L.G) == 0 && L.rot == nullptr;
}

size_t prompt_tc_ws_bytes(int n_seqs, int n_rows, int max_rows, const LayerArgs& L) {
  const size_t scratch = (size_t)n_seqs * prompt_scratch_keys(L.window, max_rows) * L.n_kv * L.D * 2;
  size_t off = 256;
  off = align256(off + (size_t)n_rows * L.n_q * L.D * 2);
  off = align256(off + scratch);
  off = align256(off + scratch);
  return off + scratch;
}

cudaError_t launch_prompt_tc(const DecodeArgs& a, void* ws, int max_rows_per_seq, const RopeFreqs& f,
                             cudaStream_t st, const AppendArgs* ap) {
  if (a.n_rows == 0) return cudaSuccess;
  switch (a.L.D) {
    case 64: return launch_prompt_t<64>(a, ws, max_rows_per_seq, f, st, ap);
    case 128: return launch_prompt_t<128>(a, ws, max_rows_per_seq, f, st, ap);
    case 256: return launch_prompt_t<256>(a, ws, max_rows_per_seq, f, st, ap);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
