// CUDA-core decode-kernel instantiations for one K/V kind pair (built as its
// own translation unit so the pairs compile in parallel).
#include "kvq_decode_impl.cuh"

namespace kvq {
kvq_status launch_decode_s8s4(const DecodeArgs& a, int hd, int G, dim3 grid, cudaStream_t s) {
  return launch_decode_kinds<KVQ_SYM_INT8, KVQ_SYM_INT4>(a, hd, G, grid, s);
}
}  // namespace kvq
