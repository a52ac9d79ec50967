// fwd_bf16.cu -- placeholder until the tensor-core forward lands.
#include "internal.h"
namespace seqattn {
cudaError_t launch_fwd_bf16(const ChunkGeom&, const Bf16FwdMaps&, void*, float*, unsigned int*,
                            cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace seqattn
