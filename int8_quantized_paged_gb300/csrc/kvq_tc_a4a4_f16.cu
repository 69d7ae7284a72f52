// Tensor-core decode-kernel instantiations for one K/V kind pair and one
// scale type (a translation unit of its own, so they compile in parallel).
#include "kvq_decode_tc.cuh"

namespace kvq {
kvq_status launch_tc_a4a4_f16(const TcArgs& t, int hd, int nt, int ng, dim3 grid, size_t smem,
                           cudaStream_t s, bool pdl) {
  return launch_tc_pt<KVQ_AFFINE_INT4, KVQ_AFFINE_INT4, KVQ_F16>(t, hd, nt, ng, grid, smem, s, pdl);
}
}  // namespace kvq
