// Tensor-core decode-kernel instantiations for one K/V kind pair and one
// scale type (a translation unit of its own, so they compile in parallel).
#include "kvq_decode_tc.cuh"

namespace kvq {
kvq_status launch_tc_s8s8_bf16(const TcArgs& t, int hd, int nt, int ng, const TcLaunchCfg& lc) {
  return launch_tc_pt<KVQ_SYM_INT8, KVQ_SYM_INT8, KVQ_BF16>(t, hd, nt, ng, lc);
}
}  // namespace kvq
