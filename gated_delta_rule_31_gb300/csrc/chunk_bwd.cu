// chunk_bwd.cu - backward (VJP) of the chunked gated delta rule.
#include <cuda_runtime.h>

#include "chunk.h"

namespace gdr {

cudaError_t launch_chunk_bwd(const ChunkBwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace gdr
