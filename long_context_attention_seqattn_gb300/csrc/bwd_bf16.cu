// bwd_bf16.cu -- placeholder until the tensor-core backward lands.
#include "internal.h"
namespace seqattn {
cudaError_t launch_bwd_bf16(const ChunkGeom&, const Bf16BwdMaps&, const float*, const float*,
                            float*, float*, float*, unsigned int*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace seqattn
