// kv_quant_append: prep (norm, RoPE) and group-quantize new K/V rows into the
// affine cache (model.ts attentionTraining: kNorm, vNorm, RoPE at the cache
// offset, then cache.appendWindow(k, v); gemma4-e4b.ts Gemma4Layer.kv:
// {bits, groupSize 64}).  The same kernel preps the plain keys and values of
// the training read (kvq_train_kv_prep), which are not quantized.
//
// One block handles one row (token) and a block of its (kv head, K-or-V)
// items, TH threads of E contiguous elements per item: the row's RoPE angles
// (the costly float-float sine/cosine) are evaluated once for all its K
// heads, and the float-float norm chains of the items run side by side.  A
// 64-element quantization group spans 64/E threads and is reduced with
// shuffles.
#include "kvq_append.cuh"

namespace kvq {

namespace {

template <int D>
__global__ void __launch_bounds__(1024)
append_kernel(const AppendArgs a, const RopeFreqs freqs, const int ipb) {
  append_block<D>(a, freqs, ipb, blockIdx.x, blockIdx.y);
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, const RopeFreqs& f, cudaStream_t st) {
  if (a.n_rows == 0) return cudaSuccess;
  auto go = [&](auto tag) {
    constexpr int D = decltype(tag)::value;
    const int items = 2 * a.L.n_kv;
    const int ipb = items < App<D>::IPB ? items : App<D>::IPB;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.n_rows, (unsigned)((items + ipb - 1) / ipb));
    cfg.blockDim = dim3(ipb * App<D>::TH);
    cfg.dynamicSmemBytes = a.L.rot ? (size_t)ipb * D * sizeof(double) : 0;   // rotation rows
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, append_kernel<D>, a, f, ipb);
  };
  switch (a.L.D) {
    case 64: return go(std::integral_constant<int, 64>{});
    case 128: return go(std::integral_constant<int, 128>{});
    case 256: return go(std::integral_constant<int, 256>{});
    case 512: return go(std::integral_constant<int, 512>{});
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
