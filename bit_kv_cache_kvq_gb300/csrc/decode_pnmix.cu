// Decode attention over PN-Mix H3/L1 caches (1-bit LSB plane and 2-bit upper
// plane of the keys, uniform values): the tensor-core decode of
// decode_mma.cuh instantiated with its PN-Mix paths, in a translation unit
// of its own so the build compiles it in parallel with the other variants.
#include "decode_mma.cuh"

namespace kvq {

cudaError_t launch_decode_pnmix(const MmaArgs& a, int nrep, int vbits, int warps, cudaStream_t s) {
  if (vbits == 2) return launch_rep<2, 2, false, false, true>(a, nrep, warps, s);
  return launch_rep<2, 4, false, false, true>(a, nrep, warps, s);
}

}  // namespace kvq
