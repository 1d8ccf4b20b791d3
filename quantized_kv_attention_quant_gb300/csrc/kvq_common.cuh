// Device helpers shared by the kvq kernels (sm_103a).
//
// Precision contract of the "prep" steps (q/k RMSNorm, un-scaled v norm,
// RoPE): each prepped element is the bf16 value nearest to the exact real
// result (ties to even).  The arithmetic runs in float-float pairs of fp32
// (~2^-44 relative), which GB300 executes at full fp32 rate, instead of in
// fp64 (a small fraction of that rate on this part).
//
// Model code this implements (pages of the @mlx-bun/inference package):
//   model.ts, "Parity notes" header: SDPA scale 1.0 because q and k are
//     normalized; K = V full layers with un-scaled v norm; proportional RoPE
//     rotating only partial_rotary_factor * dims dims.
//   model.ts, attentionTraining: qNorm/kNorm/vNorm per head, RoPE at the
//     cache offset, appendWindow(k, v), then read.attend(q, 1.0).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "rope_consts.h"

namespace kvq {

// ----------------------------------------------------------------------------
// bf16 bit helpers
// ----------------------------------------------------------------------------
__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }
__device__ __forceinline__ float bf16lo_to_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// IEEE round-to-nearest-even fp32 -> bf16 (finite inputs).
__device__ __forceinline__ uint16_t f_to_bf16_rn(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// ----------------------------------------------------------------------------
// float-float arithmetic.  The _rn intrinsics keep the compiler from fusing
// or reordering the error-free transformations.
// ----------------------------------------------------------------------------
struct ff { float hi, lo; };

__device__ __forceinline__ ff two_sum(float a, float b) {
  float s = __fadd_rn(a, b);
  float bp = __fsub_rn(s, a);
  float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
  return {s, e};
}
// requires |a| >= |b| (or a == 0)
__device__ __forceinline__ ff fast_two_sum(float a, float b) {
  float s = __fadd_rn(a, b);
  float e = __fsub_rn(b, __fsub_rn(s, a));
  return {s, e};
}
__device__ __forceinline__ ff two_prod(float a, float b) {
  float p = __fmul_rn(a, b);
  float e = __fmaf_rn(a, b, -p);
  return {p, e};
}
__device__ __forceinline__ ff ff_add(ff a, ff b) {
  ff s = two_sum(a.hi, b.hi);
  float e = __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo));
  return fast_two_sum(s.hi, e);
}
__device__ __forceinline__ ff ff_neg(ff a) { return {-a.hi, -a.lo}; }
__device__ __forceinline__ ff ff_mul_f(ff a, float b) {
  ff p = two_prod(a.hi, b);
  float e = __fmaf_rn(a.lo, b, p.lo);
  return fast_two_sum(p.hi, e);
}
__device__ __forceinline__ ff ff_mul(ff a, ff b) {
  ff p = two_prod(a.hi, b.hi);
  float e = __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, p.lo));
  return fast_two_sum(p.hi, e);
}

// Correctly rounded bf16 of the real number hi + lo, where (hi, lo) is
// normalised (|lo| <= ulp(hi)/2, as fast_two_sum leaves it).  hi is the fp32
// nearest to hi + lo, so hi + lo lies on the same side of every bf16 rounding
// boundary as hi, except when hi sits exactly on a boundary; then lo decides.
__device__ __forceinline__ uint16_t ff_to_bf16_rn(ff v) {
  uint32_t u = __float_as_uint(v.hi);
  uint32_t low = u & 0xFFFFu;
  uint32_t top = u >> 16;
  if (low > 0x8000u) return uint16_t(top + 1);
  if (low < 0x8000u) return uint16_t(top);
  if (v.lo == 0.f) return uint16_t(top + (top & 1u));
  bool away = (v.lo > 0.f) == (v.hi > 0.f);   // true magnitude above the tie
  return uint16_t(away ? top + 1 : top);
}

// Correctly rounded bf16 of a double (ties to even).  f = d truncated toward
// zero to fp32 and r = d - f (exact, zero or of d's sign): d lies strictly
// above f's magnitude when r != 0, so a low half of f below the midpoint
// 0x8000 rounds down, above it up, and at it up unless r == 0 (a tie).
__device__ __forceinline__ uint16_t d_to_bf16_rn(double d) {
  const float f = __double2float_rz(d);
  const double r = d - (double)f;
  const uint32_t u = __float_as_uint(f);
  const uint32_t low = u & 0xFFFFu;
  uint32_t top = u >> 16;
  if (low > 0x8000u || (low == 0x8000u && (r != 0.0 || (top & 1u)))) ++top;
  return uint16_t(top);
}

// ----------------------------------------------------------------------------
// RMSNorm pieces (reading: y = x / sqrt(mean(x^2) + eps) * w, rounded once)
// ----------------------------------------------------------------------------
// Accumulate x^2 (exact in fp32 for bf16 x) into a float-float sum.
__device__ __forceinline__ void ff_acc_sq(ff& acc, float x) {
  float sq = __fmul_rn(x, x);
  ff s = two_sum(acc.hi, sq);
  acc = fast_two_sum(s.hi, __fadd_rn(s.lo, acc.lo));
}
__device__ __forceinline__ ff ff_shfl_xor(ff v, int m) {
  return {__shfl_xor_sync(0xffffffffu, v.hi, m), __shfl_xor_sync(0xffffffffu, v.lo, m)};
}
// Full-warp float-float sum.
__device__ __forceinline__ ff ff_warp_sum(ff v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = ff_add(v, ff_shfl_xor(v, m));
  return v;
}
// 1 / sqrt(ss / D + eps) as a float-float (~2^-45 relative), in fp32 only
// (fp64 sqrt + divide cost ~1500 cycles of latency on this part):
//   r = ss/D + eps (float-float; /D is exact for a power of two);
//   y0 = 1/sqrt(r.hi), IEEE-rounded sqrt and division (|rel. error| <= 2^-23);
//   one Newton step y = y0 + y0 (1 - r y0^2) / 2 with r y0^2 formed exactly
//   (two_prod; 1 - p.hi is exact by Sterbenz since p.hi ~ 1); the step's
//   error is 1.5 (2^-23)^2 ~ 2^-45.
__device__ __forceinline__ ff rms_inv(ff ss, int D, float eps) {
  const float invD = 1.0f / (float)D;                    // D is a power of two
  ff r = two_sum(__fmul_rn(ss.hi, invD), eps);
  r = fast_two_sum(r.hi, __fadd_rn(r.lo, __fmul_rn(ss.lo, invD)));
  const float y0 = __fdiv_rn(1.0f, __fsqrt_rn(r.hi));
  const ff t = two_prod(y0, y0);                         // y0^2 exactly
  const ff p = two_prod(r.hi, t.hi);                     // r.hi * t.hi exactly
  const float small = __fmaf_rn(r.hi, t.lo, __fmul_rn(r.lo, t.hi));
  const float e = __fsub_rn(__fsub_rn(__fsub_rn(1.0f, p.hi), p.lo), small);
  return fast_two_sum(y0, __fmul_rn(__fmul_rn(y0, e), 0.5f));
}
// x * w * inv, correctly rounded to bf16; x and w are bf16 values so x*w is
// exact in fp32.
//
// Fast path, bit-identical to the float-float result: p = fl(inv.hi * xw).
// The float-float product's leading float hi' differs from p by at most
// 1.5 ulp(p) (|p - inv.hi*xw| <= ulp/2, |inv.lo*xw| <= 2^-24 |p| < ulp(p)),
// i.e. by at most 3 steps of the fp32 bit pattern even where a binade
// boundary halves the ulp.  bf16 rounding of a float looks only at its low 16
// bits (ties at exactly 0x8000), so when p's low half is more than 4 steps
// from 0x8000, hi' and p round alike (a carry across the 16-bit boundary
// keeps the rounded value: p = top|0xFFFF and top+1|0x0002 both give top+1).
__device__ __forceinline__ uint16_t norm_scale_bf16(float x, float w, ff inv) {
  float xw = __fmul_rn(x, w);
  // exact zero keeps its IEEE sign (inv > 0); the float-float sums would drop it
  if (xw == 0.f) return uint16_t(__float_as_uint(xw) >> 16);
  const uint32_t u = __float_as_uint(__fmul_rn(inv.hi, xw));
  const uint32_t low = u & 0xFFFFu;
  if (low - 0x7FFCu > 8u) return uint16_t((u >> 16) + (low > 0x8000u ? 1u : 0u));
  return ff_to_bf16_rn(ff_mul_f(inv, xw));
}

// ----------------------------------------------------------------------------
// Rotary angles.  For position p (integer < 2^24) and frequency f given as an
// exact sum f1 + f2 + f3 of floats (the float64 theta^(-2j/D) split three
// ways), returns cos and sin of p*f as float-float pairs accurate to ~2^-45
// absolute, without fp64 arithmetic:
//   1. p*f1, p*f2 exactly by two_prod (p*f3 is below 2^-33 and rounded once);
//   2. k = rint(p*f * 2/pi); r = p*f - k*pi/2 with pi/2 as a three-float
//      Cody-Waite split, every product exact by two_prod; the leading
//      difference is exact (Sterbenz), the small terms are summed float-float;
//   3. k2 = rint(r * 128/pi); r -= k2*pi/128 the same way, |r| <= ~pi/256;
//   4. cos/sin of r by Taylor series (r^2/2 and r carried float-float);
//   5. rotate by the table entry (cos, sin)((64k + k2) * pi/128).
// ----------------------------------------------------------------------------
__device__ __forceinline__ void ff_accum(ff& acc, float t) {
  ff s = two_sum(acc.hi, t);
  acc = fast_two_sum(s.hi, __fadd_rn(s.lo, acc.lo));
}

__device__ __forceinline__ void rope_cos_sin(int p, float f1, float f2, float f3, ff& c, ff& s) {
  const float P = (float)p;
  ff a1 = two_prod(P, f1);
  ff a2 = two_prod(P, f2);
  float a3 = __fmul_rn(P, f3);
  // first reduction by pi/2
  float k = rintf(__fmul_rn(a1.hi, KVQ_TWO_OVER_PI));
  ff b1 = two_prod(k, KVQ_PIO2_1);
  ff b2 = two_prod(k, KVQ_PIO2_2);
  float b3 = __fmul_rn(k, KVQ_PIO2_3);
  ff r = {__fsub_rn(a1.hi, b1.hi), 0.f};      // exact
  r = fast_two_sum(r.hi, 0.f);
  ff_accum(r, a1.lo);
  ff_accum(r, -b1.lo);
  ff_accum(r, a2.hi);
  ff_accum(r, -b2.hi);
  ff_accum(r, a2.lo);
  ff_accum(r, -b2.lo);
  ff_accum(r, __fsub_rn(a3, b3));
  // second reduction by pi/128
  float k2 = rintf(__fmul_rn(r.hi, KVQ_128_OVER_PI));
  ff c1 = two_prod(k2, KVQ_PIO128_1);
  ff c2 = two_prod(k2, KVQ_PIO128_2);
  float c3 = __fmul_rn(k2, KVQ_PIO128_3);
  ff t = two_sum(r.hi, -c1.hi);
  ff rr = fast_two_sum(t.hi, t.lo);
  ff_accum(rr, r.lo);
  ff_accum(rr, -c1.lo);
  ff_accum(rr, -c2.hi);
  ff_accum(rr, -c2.lo);
  ff_accum(rr, -c3);
  // table index: the angle removed is (64 k + k2) * pi/128
  int ki = (int)k;
  int idx = ((ki & 3) * 64 + (int)k2) & 255;
  // Taylor series of sin / cos at |rr| <= ~0.0123
  float x = rr.hi;
  ff x2 = two_prod(x, x);
  x2.lo = __fmaf_rn(2.f * x, rr.lo, x2.lo);
  x2 = fast_two_sum(x2.hi, x2.lo);
  float z = x2.hi;
  // sin r = r - r^3/6 + r^5/120 - r^7/5040
  float ps = __fmul_rn(z, __fmaf_rn(z, __fmaf_rn(z, -1.f / 5040.f, 1.f / 120.f), -1.f / 6.f));
  ff sr = fast_two_sum(x, __fmaf_rn(x, ps, rr.lo));
  // cos r = 1 - r^2/2 + r^4/24 - r^6/720
  float pc = __fmul_rn(__fmul_rn(z, z), __fmaf_rn(z, -1.f / 720.f, 1.f / 24.f));
  ff half = {__fmul_rn(x2.hi, 0.5f), __fmul_rn(x2.lo, 0.5f)};
  ff cr = two_sum(1.f, -half.hi);
  cr = fast_two_sum(cr.hi, __fadd_rn(cr.lo, __fsub_rn(pc, half.lo)));
  // rotate by the table angle
  float4 tb = __ldg(&kvq_rope_table[idx]);
  ff tc = {tb.x, tb.y}, ts = {tb.z, tb.w};
  c = ff_add(ff_mul(tc, cr), ff_neg(ff_mul(ts, sr)));
  s = ff_add(ff_mul(ts, cr), ff_mul(tc, sr));
}

// Copy rope_dims/2 frequency triples from the kernel-parameter table into
// shared memory (16-byte aligned on both sides), 16 bytes per read.  Every
// read of the parameter block is warp-uniform (a lane index into it would
// serialise on the constant cache) and four are in flight at a time; call
// from all threads of the block, followed by a block barrier.
__device__ __forceinline__ void stage_freqs(const float (*f)[3], int half, float (*dst)[3]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const float4* src4 = reinterpret_cast<const float4*>(&f[0][0]);
  float4* dst4 = reinterpret_cast<float4*>(&dst[0][0]);
  // up to 3 floats past 3*half: still inside the 256-triple table and inside
  // dst, which holds D/2 triples (3*D/2 is a multiple of 4)
  const int n4 = (3 * half + 3) / 4;
#pragma unroll 4
  for (int k = warp; k < n4; k += nw) {
    const float4 v = src4[k];
    if (lane == 0) dst4[k] = v;
  }
}

// x*c - y*s, correctly rounded to bf16 (x, y bf16 values; c, s float-float).
//
// Fast path: r = fl(x*c.hi - fl(y*s.hi)) (one fma).  Against the exact value
// it drops x*c.lo and y*s.lo (each <= 2^-24 of its product) and rounds twice
// (<= 2^-24 of |y*s.hi| and of |r|), so |r - exact| <= 2^-22 B with
// B = |x*c.hi| + |y*s.hi|; the float-float result lies within 2^-44 B of the
// exact value.  bf16 rounding midpoints sit where the fp32 low half is 0x8000
// (mid-binade), so when r is a normal float whose distance to the nearest
// one, |low - 0x8000| * ulp(r), exceeds 2^-21 B, the exact value, the
// float-float result and r all round to the same bf16.
__device__ __forceinline__ uint16_t rot_bf16(float x, float y, ff c, ff s) {
  if (x == 0.f && y == 0.f)   // signed zero as IEEE arithmetic gives it
    return uint16_t(__float_as_uint(__fsub_rn(__fmul_rn(x, c.hi), __fmul_rn(y, s.hi))) >> 16);
  const float ys = __fmul_rn(y, s.hi);
  const float r = __fmaf_rn(x, c.hi, -ys);
  const uint32_t u = __float_as_uint(r);
  const uint32_t ex = u & 0x7F800000u;
  if (ex >= (24u << 23) && ex < 0x7F800000u) {
    const uint32_t low = u & 0xFFFFu;
    const float steps = (float)(low > 0x8000u ? low - 0x8000u : 0x8000u - low);
    const float ulp = __uint_as_float(ex - (23u << 23));               // 2^(e - 23)
    const float bound = __fmul_rn(__fadd_rn(fabsf(__fmul_rn(x, c.hi)), fabsf(ys)), 4.76837158203125e-7f);  // 2^-21
    if (__fmul_rn(steps, ulp) > bound) return uint16_t((u >> 16) + (low > 0x8000u ? 1u : 0u));
  }
  ff a = ff_mul_f(c, x);
  ff b = ff_mul_f(s, y);
  return ff_to_bf16_rn(ff_add(a, ff_neg(b)));
}

// ----------------------------------------------------------------------------
// The rotation of the deferred TurboQuant read: a bf16 row y of D values
// (E per thread, thread t of the row's TH holding elements t*E .. t*E+E-1)
// becomes bf16((y * s) H), H the Sylvester Hadamard matrix (H_ij =
// (-1)^popcount(i & j)): sign flip, then the in-place Walsh-Hadamard butterflies
// (u, v) -> (u + v, u - v) at strides 1, 2, .., D/2 in float64 shared memory,
// then one correct rounding to bf16 (a zero becomes +0).  Every thread of the
// block calls it (block barriers inside); `active` marks threads of real rows.
// ----------------------------------------------------------------------------
template <int D, int E, int TH>
__device__ __forceinline__ void rotate_row_bf16(uint16_t (&y)[E], const int8_t* signs, double* row, int t,
                                                bool active) {
  if (active) {
#pragma unroll
    for (int i = 0; i < E; ++i) row[t * E + i] = (double)bf16_to_f(y[i]) * (double)__ldg(signs + t * E + i);
  }
  __syncthreads();
#pragma unroll 1
  for (int h = 1; h < D; h <<= 1) {
    if (active) {
      for (int p = t; p < D / 2; p += TH) {
        const int i = (p / h) * 2 * h + (p % h);
        const double u = row[i], v = row[i + h];
        row[i] = u + v;
        row[i + h] = u - v;
      }
    }
    __syncthreads();
  }
  if (active) {
#pragma unroll
    for (int i = 0; i < E; ++i) y[i] = d_to_bf16_rn(row[t * E + i] + 0.0);
  }
}

// ----------------------------------------------------------------------------
// Bounded waits.  Every wait in these kernels gives up after kWaitLimitNs of
// wall-clock time (read from %globaltimer), records the fact in a status word
// and lets the kernel run to its end, so a lost arrival can never hang the GPU.
// ----------------------------------------------------------------------------
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

enum : uint32_t { KVQ_DEV_OK = 0, KVQ_DEV_TIMEOUT = 1, KVQ_DEV_BADSEQ = 2 };

__device__ __forceinline__ void flag_error(uint32_t* status, uint32_t code) {
  if (status) atomicOr(status, 1u << code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Returns false if the phase did not complete within kWaitLimitNs.
// Wait for the phase `parity` of `bar` to complete; false when limit_ns of
// wall-clock time pass first.
__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_for(bar, parity, kWaitLimitNs);
}

// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch controls (no-ops without the attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `kernel` as a programmatic dependent of the stream's previous kernel
// (it may start before that grid is complete and waits for it with pdl_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

// ----------------------------------------------------------------------------
// Warp-level tensor-core MMA, m16n8k16, f16 inputs, fp32 accumulate.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
               "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16_zc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
               "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
               : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_u32(p)));
}

// ----------------------------------------------------------------------------
// Code -> f16 conversion with one logic op per pair.  A 16-bit half whose
// exponent field is zero is an f16 subnormal: bits m (m < 1024) in its
// mantissa are the exact value m * 2^-24.  So masking a packed word leaves
// two codes as exact f16 values scaled by 2^-24 (codes taken from bits 4..7
// come out scaled by 2^-20, i.e. 16 times larger).  The tensor cores multiply
// f16 subnormals exactly; the power of two is divided out of the fp32 result.
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ uint32_t h2_mul(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
constexpr float kTwo24 = 16777216.f;            // 2^24

// bits 0..3 of each 16-bit half -> (c, c) * 2^-24
__device__ __forceinline__ uint32_t sub_n0(uint32_t x) { return x & 0x000F000Fu; }
// bits 4..7 of each 16-bit half -> (c, c) * 2^-20
__device__ __forceinline__ uint32_t sub_n1(uint32_t x) { return x & 0x00F000F0u; }
// bits 0..7 of each 16-bit half -> (c, c) * 2^-24
__device__ __forceinline__ uint32_t sub_b0(uint32_t x) { return x & 0x00FF00FFu; }
// bytes 1 and 3 of x moved to bytes 0 and 2, zeros above -> (c, c) * 2^-24
__device__ __forceinline__ uint32_t sub_b1(uint32_t x) { return prmt(x, 0u, 0x4341u); }

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace kvq
