// Decode attention over KIVI-variant caches (keys in 32-token sub-groups,
// bf16 metadata, values partly in the FIFO ring): the tensor-core decode of
// decode_mma.cuh instantiated with its KIVI paths, in a translation unit of
// its own so the build compiles it in parallel with the other variants.
#include "decode_mma.cuh"

namespace kvq {

cudaError_t launch_decode_kivi(const MmaArgs& a, int nrep, int bits, int warps, cudaStream_t s) {
  if (bits == 2) return launch_rep<2, 2, false, true>(a, nrep, warps, s);
  return launch_rep<4, 4, false, true>(a, nrep, warps, s);
}

}  // namespace kvq
