// Decode-kernel instantiations for one K/V kind pair (built as its own
// translation unit so the pairs compile in parallel): the tensor-core kernel
// and the CUDA-core kernel.
#include "kvq_decode_impl.cuh"
#include "kvq_decode_tc.cuh"

namespace kvq {
kvq_status launch_decode_a4a4(const DecodeArgs& a, int hd, int G, dim3 grid, cudaStream_t s) {
  return launch_decode_kinds<KVQ_AFFINE_INT4, KVQ_AFFINE_INT4>(a, hd, G, grid, s);
}
kvq_status launch_tc_a4a4(const TcArgs& t, const CUtensorMap& mk, const CUtensorMap& mv, int hd, bool oneg,
                        int param, dim3 grid, size_t smem, cudaStream_t s, bool pdl) {
  return launch_tc_kinds<KVQ_AFFINE_INT4, KVQ_AFFINE_INT4>(t, mk, mv, hd, oneg, param, grid, smem, s, pdl);
}
}  // namespace kvq
