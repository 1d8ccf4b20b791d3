// attn_train_forward on the tensor cores (tcgen05): the training forward's
// stateless read (trainable.ts, trainingCaches and
// prefixShared.prefixSharedHidden; model.ts, the attentionTraining comment:
// a training cache stores nothing and reads the plain keys and values handed
// to it under the run's mask -- causal, windowed, or block-sparse with a
// logical-position window under a prefix-shared layout).
//
// Layout: the packed rows of one training sequence are blocks [off[b],
// off[b+1]); block 0 is the prefix (rows at positions 0 ..), every other
// block a branch continuing it (its row j at position off[1] + j).  A row
// sees the prefix and its own block, up to its own position and, on a
// sliding layer, within the window.
//
// One CTA takes 128 query rows of one block that share a kv head (128/G
// consecutive rows times their G q heads, row r = token r / G, head r % G)
// and DO <= 256 of the output dims (head_dim 512: two CTAs per row tile).
// It walks the keys it can see -- the prefix segment, then its own block's
// segment -- in 64-key tiles, with two roles:
//   - one MMA warp: the tensor memory accelerator copies of q (once) and of
//     each tile's K rows (all dims) as bf16 in the 128-byte-swizzled K-major
//     layout the MMA reads (rows past the end of the sequence arrive as
//     zeros); QK (M = 128 rows, N = 64 keys, bf16 operands: the products of
//     bf16 values are exact in fp32) into one of two score slots of tensor
//     memory, so that the next tile's QK runs under this tile's softmax; and
//     PV (A = P from tensor memory, B = V^T, N = DO) into the output
//     accumulator;
//   - 16 softmax warps, four threads per row (warps w, w + 4, w + 8, w + 12
//     reach the same tensor-memory lanes; each takes a quarter of a tile's
//     keys and of the output dims): mask the keys outside a row's view,
//     exchange the row maximum through tensor memory, write P = e^(S - ref)
//     as f16 into tensor memory (ref is a lazily renewed reference: the
//     output is rescaled only when a tile's maximum exceeds it by more than
//     8), and transpose the V tile, staged by the tensor memory accelerator,
//     into (dims x keys) f16 rows (ldmatrix / stmatrix; bf16 -> f16 is exact
//     for |v| in f16's normal range, and v_hat = vNorm(v) is at most
//     sqrt(head_dim)).
// Head_dim <= 256 keeps two K buffers and a V stage; head_dim 512 (128 KB of
// q) has one K buffer and transposes V in place.  The output is O / l per
// row.
#include "kvq_common.cuh"
#include "kvq_internal.h"
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
constexpr int kThreads = kRows * kNQ;
constexpr int kKPT = 64 / kNQ;          // keys of a tile per thread

template <int D>
struct Tr {
  static constexpr int DO = D > 256 ? 256 : D;         // output dims per CTA
  static constexpr int NSPLIT = D / DO;                 // CTAs per row tile
  static constexpr int NG = D / 64;                     // 64-dim groups of q and K
  static constexpr int NO = DO / 64;                    // 64-dim groups of the CTA's output dims
  static constexpr int KB = D <= 256 ? 2 : 1;           // K buffers (head_dim 512: no room for two)
  static constexpr bool VSTAGE = D <= 256;              // V copied into a stage, then transposed apart
  // byte offsets from the 1024-aligned base
  static constexpr int Q_OFF = 0;                       // NG blocks [128 rows x 128 B]: q as bf16
  static constexpr int K_OFF = Q_OFF + NG * 16384;      // KB x NG blocks [64 keys x 128 B]: K as bf16
  static constexpr int V_OFF = K_OFF + KB * NG * 8192;  // [DO dims x 128 B]: V^T as f16 (in place of V
                                                        // when there is no stage)
  static constexpr int VS_OFF = V_OFF + NO * 8192;      // stage: NO blocks [64 keys x 128 B] of V (bf16)
  static constexpr int C_OFF = VS_OFF + (VSTAGE ? NO * 8192 : 0);   // mbarriers, tensor-memory address
  static constexpr int BYTES = C_OFF + 128 + 1024;      // + room to align the base
  // tensor-memory columns
  static constexpr int C_O = 0;                         // output accumulator, DO columns
  static constexpr int C_S = DO;                        // two score slots of 64 columns
  static constexpr int C_P = DO + 128;                  // P as f16 pairs, 32 columns (A of PV)
  static constexpr int C_X = DO + 160;                  // row exchange, one column per share
  static constexpr int TMEM_COLS = C_X + kNQ <= 256 ? 256 : 512;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}

// two bf16 values -> the same two values as f16 (round to nearest)
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w) { return pack_h2(bf16lo_to_f(w), bf16hi_to_f(w)); }

// the 16 softmax warps' own barrier (the MMA warp does not take part)
__device__ __forceinline__ void softmax_sync() { named_bar(1, kThreads); }

template <int D>
__global__ void __launch_bounds__(kThreads + 32, 1)
train_tc_kernel(const TrainArgs a, uint32_t* status, const __grid_constant__ CUtensorMap tmq,
                const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  using T = Tr<D>;
  constexpr int NG = T::NG, NO = T::NO, DO = T::DO, KB = T::KB;
  constexpr float L2E = 1.4426950408889634f;
  constexpr float kSlack = 8.f;
  constexpr float kHead = 6.f;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.L.G, TQ = kRows / G, W = a.L.window;
  const int b = blockIdx.y;
  const int kvh = blockIdx.z / T::NSPLIT, d_base = (blockIdx.z % T::NSPLIT) * DO;
  const int off0 = __ldg(a.off + b), off1 = __ldg(a.off + b + 1);
  const int P = __ldg(a.off + 1);                         // prefix rows
  const int t0 = blockIdx.x * TQ;
  pdl_launch();                                           // the next call's first kernel waits for this grid
  // the layout as the rows of this block need it (uniform over the CTA)
  const bool ok = off0 >= 0 && off0 <= off1 && off1 <= a.n_rows && P >= 0 && P <= a.n_rows &&
                  (b == 0 ? off0 == 0 : off0 >= P) && (b + 1 < a.n_blocks || off1 == a.n_rows);
  if (!ok) {
    pdl_wait();                                           // the q prep clears the status word
    if (blockIdx.x == 0 && blockIdx.z == 0 && tid == 0) flag_error(status, KVQ_DEV_BADSEQ);
    return;
  }
  const int rows_b = off1 - off0;
  if (t0 >= rows_b) return;
  const int base = b == 0 ? 0 : P;                        // position of the block's first row
  // mbarriers: q, K[2], V, S[2] (QK done), Sfree[2] (scores read), PV ready, O (PV done)
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

  // ---- the keys of the CTA: the prefix segment, then its own block's ----
  const int t_last = min(t0 + TQ, rows_b) - 1;
  const int lp_first = base + t0, lp_last = base + t_last;
  const int lo_first = W > 0 ? max(0, lp_first - W + 1) : 0;
  const int a_lo = lo_first, a_hi = b == 0 ? lp_last : P - 1;          // prefix rows (packed = position)
  const int nA = a_hi >= a_lo ? (a_hi - a_lo) / kTileKeys + 1 : 0;
  const int bl_lo = b == 0 ? 1 : max(P, lo_first), bl_hi = b == 0 ? 0 : lp_last;   // branch positions
  const int nB = bl_hi >= bl_lo ? (bl_hi - bl_lo) / kTileKeys + 1 : 0;
  const int n_tiles = nA + nB;                            // >= 1: every row sees itself
  auto tile_at = [&](int i, int& pk0, int& lp0, int& pk_end) {
    if (i < nA) {
      pk0 = a_lo + kTileKeys * i;
      lp0 = pk0;
      pk_end = a_hi + 1;
    } else {
      lp0 = bl_lo + kTileKeys * (i - nA);
      pk0 = off0 + (lp0 - P);
      pk_end = off0 + (bl_hi - P) + 1;
    }
  };
  auto issue_k = [&](int i) {                             // one thread: K rows of tile i
    int pk0, lp0, pk_end;
    tile_at(i, pk0, lp0, pk_end);
    uint64_t* bk = bar_k + (i % KB);
    mbar_arrive_expect_tx(bk, NG * 8192);
#pragma unroll
    for (int g = 0; g < NG; ++g)
      tc::tma_load_3d(sbase + T::K_OFF + ((i % KB) * NG + g) * 8192, &tmk, 64 * g, kvh, pk0, smem_u32(bk));
  };
  auto issue_v = [&](int i) {                             // one thread: V rows (the CTA's dims) of tile i
    int pk0, lp0, pk_end;
    tile_at(i, pk0, lp0, pk_end);
    mbar_arrive_expect_tx(bar_v, NO * 8192);
#pragma unroll
    for (int j = 0; j < NO; ++j)
      tc::tma_load_3d(sbase + (T::VSTAGE ? T::VS_OFF : T::V_OFF) + j * 8192, &tmv, d_base + 64 * j, kvh, pk0,
                      smem_u32(bar_v));
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
  // launched as a programmatic dependent of the q prep grid: q, the donor's
  // keys and values and the status word are touched only after it is complete
  pdl_wait();
  bool dead = false;
  auto wait = [&](uint64_t* bar, int parity) {
    if (!dead && !mbar_wait(bar, parity)) {
      dead = true;
      flag_error(status, KVQ_DEV_TIMEOUT);
    }
  };

  if (warp == kThreads / 32) {
    // ================= the MMA warp: copies of q and K, QK and PV =================
    const bool leader = lane == 0;
    constexpr uint32_t ID_QK = tc::idesc_bf16_f32(128, 64);
    constexpr uint32_t ID_PV = tc::idesc_f16_f32(128, DO);
    if (leader) {
      mbar_arrive_expect_tx(bar_q, NG * 16384);
#pragma unroll
      for (int g = 0; g < NG; ++g)
        tc::tma_load_3d(sbase + T::Q_OFF + g * 16384, &tmq, 64 * g, kvh * G, off0 + t0, smem_u32(bar_q));
      issue_k(0);
      if (KB == 2 && n_tiles > 1) issue_k(1);
      if (!T::VSTAGE) issue_v(0);
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
#pragma unroll
        for (int g = 0; g < NG; ++g)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_f16(tmem + T::C_S + 64 * slot,
                        tc::desc_kmajor_sw128(sbase + T::Q_OFF + g * 16384 + 32 * k, 1024),
                        tc::desc_kmajor_sw128(sbase + T::K_OFF + (kb * NG + g) * 8192 + 32 * k, 1024), ID_QK,
                        (g | k) != 0);
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
      // no V stage: V(ti) replaces V^T(ti-1) once PV(ti-1) is done
      if (!T::VSTAGE && ti > 0) {
        wait(bar_o, (ti - 1) & 1);
        if (leader) issue_v(ti);
        __syncwarp();
      }
    }
    issue_pv(n_tiles - 1);
  } else {
    // ================= the softmax warps =================
    const int r = 32 * (warp & 3) + lane, hf = warp >> 2;
    constexpr int DPT = DO / kNQ;                         // output dims per thread
    const int tq = r / G, h = r % G;
    const int t = t0 + tq;
    const bool row_valid = t < rows_b;
    const int lp_r = base + t;                            // the row's position
    const int lo_r = W > 0 ? lp_r - W + 1 : -(1 << 30);   // its oldest visible position
    const int hq = kvh * G + h;
    const int kk0 = kKPT * hf;
    const int dd0 = DPT * hf;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    if (T::VSTAGE && tid == 0) issue_v(0);
    float m_ref = -INFINITY, l_part = 0.f;
    for (int ti = 0; ti < n_tiles; ++ti) {
      const int slot = ti & 1;
      int pk0, lp0, pk_end;
      tile_at(ti, pk0, lp0, pk_end);
      wait(bar_s + slot, (ti >> 1) & 1);                  // QK(ti) done
      tc::fence_after_sync();
      __syncwarp();
      float S[kKPT];
      tc::ld_x16(lane_base + T::C_S + 64 * slot + kk0, S);
      tc::wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_sfree + slot);       // this warp's share of the slot is read
      const int lpk = lp0 + kk0, pkk = pk0 + kk0;
      float mt = -INFINITY;
      if (__all_sync(0xffffffffu, row_valid && lpk >= lo_r && lpk + kKPT - 1 <= lp_r && pkk + kKPT - 1 < pk_end)) {
#pragma unroll
        for (int j = 0; j < kKPT; ++j) mt = fmaxf(mt, S[j]);
      } else {
#pragma unroll
        for (int j = 0; j < kKPT; ++j) {
          const bool vis = row_valid && lpk + j >= lo_r && lpk + j <= lp_r && pkk + j < pk_end;
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

      // ---- V(ti) -> V^T as f16 ----
      wait(bar_v, ti & 1);
      __syncwarp();
      constexpr int QPK = DO / 32;                        // groups of four 8x8 blocks per 8-key row
      const uint32_t vsrc = sbase + (T::VSTAGE ? T::VS_OFF : T::V_OFF);
      uint32_t vr[NO][4];
#pragma unroll
      for (int i = 0; i < NO; ++i) {
        const int qd = warp * NO + i, kb8 = qd / QPK, db0 = 4 * (qd % QPK);
        const int dch = db0 + (lane >> 3);                // 8-dim chunk of the CTA's dims
        ldsm_x4(vsrc + (dch >> 3) * 8192 + tc::sw128_off(8 * kb8 + (lane & 7), dch & 7), vr[i]);
      }
      if (!T::VSTAGE) softmax_sync();                     // every V row read before any is overwritten
#pragma unroll
      for (int i = 0; i < NO; ++i) {
        const int qd = warp * NO + i, kb8 = qd / QPK, db0 = 4 * (qd % QPK);
        const int dim = 8 * (db0 + (lane >> 3)) + (lane & 7);
        tc::stmatrix_x4_trans(sbase + T::V_OFF + tc::sw128_off(dim, kb8), bf2_to_h2(vr[i][0]),
                              bf2_to_h2(vr[i][1]), bf2_to_h2(vr[i][2]), bf2_to_h2(vr[i][3]));
      }
      fence_proxy_async();
      tc::wait_st();                                      // P and the rescaled output written
      tc::fence_before_sync();
      softmax_sync();
      if (tid == 0) {
        mbar_arrive(bar_pv);                              // PV(ti) may go
        if (T::VSTAGE && ti + 1 < n_tiles) issue_v(ti + 1);   // the stage is read
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
      for (int i = 0; i < 16; ++i) v[i] *= inv;
      if (!row_valid) continue;
      const size_t oi = (((size_t)off0 + t) * a.L.n_q + hq) * D + d_base + dd0 + 16 * cc;
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

// ---- host side ----

// A bf16 tensor [rows][heads][D] read in boxes of (64 dims, box_h heads,
// box_r rows).
bool bf16_rows_map(CUtensorMap* m, const void* base, int D, int heads, int rows, int box_h, int box_r) {
  return rows_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, D, heads, rows, box_h, box_r);
}

template <int D>
int train_launch_smem() {
  // at most 512 / TMEM_COLS CTAs may share an SM's tensor memory: ask for
  // enough shared memory that no more fit
  constexpr int smem = Tr<D>::BYTES;
  const int per_sm = 512 / Tr<D>::TMEM_COLS;
  return per_sm >= 3 ? smem : std::max(smem, (228 * 1024) / (per_sm + 1) + 1024);
}

template <int D>
cudaError_t launch_train_t(const TrainArgs& t, const uint16_t* q_raw, const uint16_t* q_w, const uint16_t* k_hat,
                           const uint16_t* v_hat, uint16_t* q_prepped, void* ws, int max_block_rows,
                           const RopeFreqs& f, cudaStream_t st, const AppendArgs* ap) {
  static_assert(Tr<D>::BYTES <= 227 * 1024, "shared memory");
  cudaError_t e;
  static std::atomic<bool> attr_set[64];
  static std::mutex attr_mu;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const int smem = train_launch_smem<D>();
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(attr_mu);
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(train_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      attr_set[dev].store(true, std::memory_order_release);
    }
  }
  const LayerArgs& L = t.L;
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  uint16_t* qhat = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) + 256);
  CUtensorMap mq, mk, mv;
  const int TQ = kRows / L.G;
  if (!bf16_rows_map(&mq, qhat, D, L.n_q, t.n_rows, L.G, TQ) ||
      !bf16_rows_map(&mk, k_hat, D, L.n_kv, t.n_rows, 1, kTileKeys) ||
      !bf16_rows_map(&mv, v_hat, D, L.n_kv, t.n_rows, 1, kTileKeys))
    return cudaErrorInvalidValue;

  // q prep: q_hat (bf16) into the workspace; it also clears the status word
  DecodeArgs qa = {};
  qa.L = L;
  qa.seqs = nullptr;
  qa.n_seqs = t.n_blocks;
  qa.n_rows = t.n_rows;
  qa.row_offsets = t.off;
  qa.pos = nullptr;
  qa.q_raw = q_raw;
  qa.q_w = q_w;
  qa.q_prepped = q_prepped;
  qa.ws.status = status;
  qa.ws.qhat = qhat;
  if ((e = launch_qprep_rows<D>(qa, f, st, ap)) != cudaSuccess) return e;
  if (t.n_blocks > 65535 || L.n_kv * Tr<D>::NSPLIT > 65535) return cudaErrorInvalidValue;
  const dim3 grid((max_block_rows + TQ - 1) / TQ, t.n_blocks, L.n_kv * Tr<D>::NSPLIT);
  if ((e = prof_before(st)) != cudaSuccess) return e;
  if ((e = launch_pdl(train_tc_kernel<D>, grid, dim3(kThreads + 32), (size_t)smem, st, t, status, mq, mk, mv)) !=
      cudaSuccess)
    return e;
  return prof_after(st);
}

}  // namespace

bool train_supported(const LayerArgs& L) {
  return (L.D == 64 || L.D == 128 || L.D == 256 || L.D == 512) && L.G >= 1 && L.G <= kMaxG &&
         (kRows % L.G) == 0 && L.rot == nullptr;
}

size_t train_ws_bytes(int n_rows, const LayerArgs& L) {
  return 256 + (size_t)n_rows * L.n_q * L.D * 2;          // status word, q_hat rows
}

cudaError_t launch_train(const TrainArgs& t, const uint16_t* q_raw, const uint16_t* q_w, const uint16_t* k_hat,
                         const uint16_t* v_hat, uint16_t* q_prepped, void* ws, int max_block_rows,
                         const RopeFreqs& f, cudaStream_t st, const AppendArgs* ap) {
  if (t.n_rows == 0) return cudaSuccess;
  switch (t.L.D) {
    case 64: return launch_train_t<64>(t, q_raw, q_w, k_hat, v_hat, q_prepped, ws, max_block_rows, f, st, ap);
    case 128: return launch_train_t<128>(t, q_raw, q_w, k_hat, v_hat, q_prepped, ws, max_block_rows, f, st, ap);
    case 256: return launch_train_t<256>(t, q_raw, q_w, k_hat, v_hat, q_prepped, ws, max_block_rows, f, st, ap);
    case 512: return launch_train_t<512>(t, q_raw, q_w, k_hat, v_hat, q_prepped, ws, max_block_rows, f, st, ap);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
