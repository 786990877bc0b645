// Split-KV paged decode attention: the kernel for calls whose rows are all
// decode rows (one query each); the body of a CTA is in decode_core.cuh.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "decode_core.cuh"
#include "kernels.h"
#include "pkv_device.cuh"

namespace pkv {

template <int D, int NT>
__global__ void __launch_bounds__(288, 1)
    decode_splitkv_kernel(const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  decode_cta<D, NT>(kmap, vmap, p, align1024(smem_raw), blockIdx.x, gridDim.x);
}

int decode_grid_size(int device) {
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms <= 0)
    sms = 148;
  return sms;
}

template <int D, int NT>
static cudaError_t launch_decode_t(const DecodeParams& prm, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, int grid, size_t smem,
                                   cudaStream_t stream) {
  auto kern = decode_splitkv_kernel<D, NT>;
  const cudaError_t status = raise_smem_limit_once<decode_splitkv_kernel<D, NT>>(kSmemBudget);
  if (status != cudaSuccess) return status;
  if (smem > kSmemBudget) return cudaErrorNotSupported;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  // a programmatic dependent of the kernel before it in the stream
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>((prm.hkv + 1) * 32));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, kmap, vmap, prm);
}

cudaError_t launch_decode_bf16(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                               const DecodeScratch& ws, int grid, cudaStream_t stream,
                               const CacheWrite* write) {
  if (a.num_reqs == 0) return cudaSuccess;
  DecodeParams prm;
  size_t smem = 0;
  const cudaError_t e = make_decode_params(a, ws, write, kSmemBudget, &prm, &smem);
  if (e != cudaSuccess) return e;
  const bool wide = prm.group > 8;
  if (a.head_dim == 128)
    return wide ? launch_decode_t<128, 2>(prm, kmap, vmap, grid, smem, stream)
                : launch_decode_t<128, 1>(prm, kmap, vmap, grid, smem, stream);
  if (a.head_dim == 64)
    return wide ? launch_decode_t<64, 2>(prm, kmap, vmap, grid, smem, stream)
                : launch_decode_t<64, 1>(prm, kmap, vmap, grid, smem, stream);
  return cudaErrorNotSupported;
}

}  // namespace pkv
